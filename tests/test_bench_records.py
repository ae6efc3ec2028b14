"""bench.py's link between the committed ncu records and the sources (CPU): a record's DRAM
traffic is used only while the sources it was captured on are unchanged.  The joint hash covers
the kernel's translation unit and its local headers; it ignores comments and whitespace, so a
comment edit keeps the record and a code edit, in the .cu or in a header, voids it."""
import json
import os
import shutil

import pytest

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture()
def tree(tmp_path, monkeypatch):
    """A copy of the kernel sources and profile records, with bench.ROOT pointed at it."""
    src = os.path.join(ROOT, "tiered_quantize_evict_gb300", "csrc")
    dst = tmp_path / "tiered_quantize_evict_gb300" / "csrc"
    shutil.copytree(src, dst)
    shutil.copytree(os.path.join(ROOT, "profiles"), tmp_path / "profiles")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    return tmp_path


def _edit(path, old, new):
    s = path.read_text()
    assert old in s
    path.write_text(s.replace(old, new, 1))


@pytest.mark.parametrize("kernel,workload", [("qe_decode_attn", "throughput_32k"), ("tk_attn", "hqe_16k")])
def test_committed_records_match_the_sources(kernel, workload):
    rec = json.load(open(os.path.join(ROOT, "profiles", f"{kernel}_{workload}.json")))
    assert rec["source_files"] == bench.KERNEL_SOURCES[kernel]
    got = bench._traffic(workload, kernel)
    assert got == rec["dram_bytes_read"] + rec["dram_bytes_write"] == rec["dram_bytes_per_launch_full"]


def test_comment_edit_keeps_the_record(tree):
    before = bench._traffic("throughput_32k")
    assert before is not None
    _edit(tree / "tiered_quantize_evict_gb300" / "csrc" / "qe_attn.cu", "// qe_attn.cu --", "// qe_attn.cu  (edited) --")
    assert bench._traffic("throughput_32k") == before


@pytest.mark.parametrize("name", ["qe_attn.cu", "qe_partition.cuh", "qe_common.cuh"])
def test_code_edit_voids_the_record(tree, name):
    assert bench._traffic("throughput_32k") is not None
    path = tree / "tiered_quantize_evict_gb300" / "csrc" / name
    path.write_text(path.read_text() + "\nnamespace qe { constexpr int edited_for_the_test = 1; }\n")
    assert bench._traffic("throughput_32k") is None
