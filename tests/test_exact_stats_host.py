"""The exact row statistics of the 1-bit tier (HqeKV reading notes §2.3 eq. (3): a token's mean
and population standard deviation), as the library computes them, against the oracle, on the
host (no GPU).

The five-tier rebuild kernel takes both statistics from ``qe_exact_stats.cuh``: a fast path in
64/128-bit integers for rows whose nonzero values lie within 2^32 of the largest, and a wide
multi-limb path for the rest.  Its helpers also compile for the host; this test builds a small
host program from that header (``exact_stats_check.cu``), runs both paths on every row, and
requires each path's mean and std to equal the oracle's bit for bit: random rows, rows shaped
like the cache's contents (bf16 values, dequantized 4- and 2-bit values) and adversarial rows
(cancellation, values 2^100 apart, subnormals, a tie, a float32 sum that would overflow)."""
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

from oracle import hqekv as H
from tests.test_oracle_hqekv import _adversarial_rows

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "tiered_quantize_evict_gb300", "csrc")


def _nvcc():
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    return None


@pytest.fixture(scope="module")
def checker():
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not found")
    d = tempfile.mkdtemp(prefix="qe_xs_")
    exe = os.path.join(d, "exact_stats_check")
    subprocess.run([nvcc, "-x", "cu", "-O2", "-std=c++17", "-I", CSRC,
                    os.path.join(ROOT, "tests", "exact_stats_check.cu"), "-o", exe], check=True)
    yield exe, d
    shutil.rmtree(d, ignore_errors=True)


def _run(checker, x):
    exe, d = checker
    x = np.ascontiguousarray(x, np.float32)
    fin, fout = os.path.join(d, "in.bin"), os.path.join(d, "out.bin")
    with open(fin, "wb") as f:
        np.array(x.shape, np.int32).tofile(f)
        x.tofile(f)
    subprocess.run([exe, fin, fout], check=True)
    raw = np.fromfile(fout, np.uint32).reshape(-1, 5)
    return raw[:, 0].astype(bool), raw[:, 1:].view(np.float32)


def _rows(D, rng):
    rows = [(rng.standard_normal((40, D)) * rng.uniform(0.01, 100, (40, 1))).astype(np.float32)]
    bf = rng.standard_normal((40, D)).astype(np.float32)              # bf16 values (8 significant bits)
    rows.append((bf.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32))
    for b in (4, 2):                                                  # dequantized uniform rows
        v = rng.standard_normal((40, D)).astype(np.float32) * 3
        codes, z, s = H.uniform_quantize_rows(v, b)
        rows.append(H.uniform_dequantize_rows(codes, z, s))
    rows.append(_adversarial_rows(D, rng))
    wide = rng.standard_normal((10, D)).astype(np.float32)            # dynamic range past the window
    wide[:, ::5] *= np.float32(2.0 ** -40)
    rows.append(wide)
    return np.concatenate(rows)


@pytest.mark.parametrize("D", [64, 128])
def test_both_paths_equal_the_oracle(checker, D):
    rng = np.random.default_rng(100 + D)
    x = _rows(D, rng)
    used, got = _run(checker, x)
    m, s = H.mean_std_f32(x)
    bits = lambda a: np.asarray(a, np.float32).view(np.uint32)
    assert np.array_equal(bits(got[:, 2]), bits(m)), np.nonzero(bits(got[:, 2]) != bits(m))
    assert np.array_equal(bits(got[:, 3]), bits(s)), np.nonzero(bits(got[:, 3]) != bits(s))
    assert np.array_equal(bits(got[used, 0]), bits(m[used]))
    assert np.array_equal(bits(got[used, 1]), bits(s[used]))
    assert used.sum() > 100 and (~used).sum() >= 10   # both paths exercised
