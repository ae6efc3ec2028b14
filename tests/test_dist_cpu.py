"""Multi-process host logic of bench.py on CPU (gloo, world size 2).

The decode path shards into independent units, so N GPUs run N replicas with no data-path
collective; the only exchange is the max over ranks of the timed region.  These tests run
that exchange, the whole-job rate and the reference arm's rank handling as two gloo ranks.
"""
import argparse
import json
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, outdir: str):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch
    import torch.distributed as dist

    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w = bench._dist()
        ms = [10.0, 25.0][rank]                       # rank 1 is the slow one
        ms_max = bench.max_over_ranks(ms, world, torch.device("cpu"))
        rate = bench.whole_job_rate(16 * 4, world, ms_max)
        ref = bench.run_reference(argparse.Namespace(workload="tiny_qevict", steps=1, warmup=3)) if rank else None
        with open(os.path.join(outdir, f"rank{rank}.json"), "w") as f:
            json.dump({"rank": r, "world": w, "ms_max": ms_max, "rate": rate, "ref": ref}, f)
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_rate(tmp_path):
    mp = pytest.importorskip("torch.multiprocessing")
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    res = [json.load(open(tmp_path / f"rank{r}.json")) for r in range(world)]
    for r, x in enumerate(res):
        assert (x["rank"], x["world"]) == (r, world)
        assert x["ms_max"] == 25.0                     # both ranks see the slowest rank's time
        assert x["rate"] == pytest.approx(2 * 64 / 0.025)   # all ranks' tokens / slowest time
    assert res[1]["ref"] is None                       # the reference arm runs on rank 0 only


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1, None) == 3.5
    assert bench.whole_job_rate(64, 1, 32.0) == pytest.approx(2000.0)


def test_reference_line_matches_contract():
    sys.path.insert(0, ROOT)
    import bench
    line = bench.run_reference(argparse.Namespace(workload="tiny_qevict", steps=2, warmup=3))
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC
    assert line["unit"] == "tokens/s" and line["higher_is_better"] is True
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    import qe_inputs as gen
    assert line["config"] == bench.workload_config(gen.WORKLOADS["tiny_qevict"], 1)
