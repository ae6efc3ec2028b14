"""The integer arithmetic that cuts a layer's unit x tile sequence into the attention launch's
cost-weighted ranges (``qe_partition.cuh``), built for the host and checked against its
definitions: the range ends ceil(w C / NW), the interleaved tile order floor(i nq / n), the
tile's cost position, the interleaved index of a bf16 tile, and the first-tile estimate, which
the kernel refines by testing the 32 tiles around it.  The cases include operands past 2^32,
where the helpers take their 64-bit branches.  Also the five-tier attention's 32-way search for
the unit that holds a cost position (``qe_tok.cuh``), with the lanes' tests run in a loop."""
import os
import random
import shutil
import subprocess
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "tiered_quantize_evict_gb300", "csrc")


def _nvcc():
    for c in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if c and os.path.exists(c):
            return c
    return None


@pytest.fixture(scope="module")
def run():
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not found")
    d = tempfile.mkdtemp(prefix="qe_part_")
    exe = os.path.join(d, "partition_check")
    subprocess.run([nvcc, "-x", "cu", "-O2", "-std=c++17", "-I", CSRC,
                    os.path.join(ROOT, "tests", "partition_check.cu"), "-o", exe], check=True)

    def go(lines):
        fin, fout = os.path.join(d, "in.txt"), os.path.join(d, "out.txt")
        with open(fin, "w") as f:
            f.write("\n".join(lines) + "\n")
        subprocess.run([exe, fin, fout], check=True)
        return [ln.split() for ln in open(fout).read().splitlines()]

    yield go
    shutil.rmtree(d, ignore_errors=True)


def _ceil_div(a, b):
    return -(-a // b)


def _q_before(i, nq, n):
    return i * nq // n


def _start(i, nq, n, cb, cq):
    qb = _q_before(i, nq, n)
    return (i - qb) * cb + qb * cq


def test_range_ends_are_the_exact_ceilings(run):
    rng = random.Random(7)
    cases = []
    for _ in range(4000):
        units = rng.choice([1, 3, 8, 64, 128, 1000, 4096, 70000])
        nw = rng.choice([12, 1824, 1800, 7 * 12, 152 * 12])
        cu = rng.choice([1, rng.randint(1, 5000), rng.randint(1, 10 ** 6), rng.randint(10 ** 9, 10 ** 12)])
        w = rng.randint(0, nw)
        cases.append((cu, nw, units, w))
    got = run([f"R {cu} {nw} {u} {w}" for cu, nw, u, w in cases])
    for (cu, nw, units, w), (x, c, k) in zip(cases, got):
        x, c, k = int(x), int(c), int(k)
        assert x == _ceil_div(w * units * cu, nw)
        assert k == w * units // nw and 0 <= c <= cu and x == k * cu + c
        # the unit holding x and the offset inside it, as the kernel derives them
        u_first = k + (1 if c >= cu else 0)
        assert u_first == x // cu


def test_tile_order_and_cost_positions(run):
    rng = random.Random(8)
    cases = []
    for _ in range(4000):
        nbt = rng.randint(1, 70000)
        nq = rng.choice([0, rng.randint(0, 70000)])
        n = nbt + nq
        i = rng.randint(0, n)
        cb, cq = rng.randint(1, 16), rng.randint(1, 16)
        cases.append((i, nq, n, cb, cq))
    got_q = run([f"Q {i} {nq} {n}" for i, nq, n, _, _ in cases])
    got_s = run([f"S {i} {nq} {n} {cb} {cq}" for i, nq, n, cb, cq in cases])
    for (i, nq, n, cb, cq), (q,), (s,) in zip(cases, got_q, got_s):
        assert int(q) == _q_before(i, nq, n)
        assert int(s) == _start(i, nq, n, cb, cq)
    # past 2^32: i nq = 65536 * 70000
    assert int(run(["Q 65536 70000 135536"])[0][0]) == 65536 * 70000 // 135536


def test_bf16_tile_index_is_the_interleaved_position(run):
    rng = random.Random(9)
    cases = []
    for _ in range(400):
        nbt = rng.randint(1, 600)
        nq = rng.randint(0, 600)
        loc = rng.randint(0, nbt - 1)
        cases.append((loc, nbt + nq, nbt, nq))
    got = run([f"B {loc} {n} {nbt}" for loc, n, nbt, _ in cases])
    for (loc, n, nbt, nq), (t,) in zip(cases, got):
        # brute force: the tile whose position in bf16 order is loc
        seen = -1
        for i in range(n):
            if _q_before(i + 1, nq, n) == _q_before(i, nq, n):   # tile i is bf16
                seen += 1
                if seen == loc:
                    break
        assert int(t) == i


def test_first_tile_lies_in_the_window_the_kernel_tests(run):
    """The kernel tests tiles est - 15 .. est + 16 and falls back to a binary search otherwise;
    with the library's tile costs (16-token bf16 sub-tile 8, 2-bit window 6 w / 32) and any
    costs within a factor 8 of each other, the window always holds the answer."""
    rng = random.Random(10)
    cases = []
    for _ in range(3000):
        nbt, nq = rng.randint(0, 3000), rng.randint(0, 3000)
        if nbt + nq == 0:
            continue
        cb = rng.randint(1, 16)
        cq = rng.choice([6, 3, 12, max(1, cb * rng.randint(1, 8) // 8), rng.randint(1, 16)])
        cu = nbt * cb + nq * cq
        r = rng.randint(0, cu - 1)
        cases.append((r, nbt + nq, cu, nq, cb, cq))
    got = run([f"E {r} {n} {cu}" for r, n, cu, _, _, _ in cases])
    for (r, n, cu, nq, cb, cq), (est,) in zip(cases, got):
        est = int(est)
        assert est == r * n // cu
        lo, hi = 0, n                           # the first tile starting at or after r
        while lo < hi:
            mid = (lo + hi) // 2
            if _start(mid, nq, n, cb, cq) >= r:
                hi = mid
            else:
                lo = mid + 1
        if max(cb, cq) <= 8 * min(cb, cq):
            assert est - 15 <= lo <= est + 16, (r, n, cu, cb, cq, est, lo)


@pytest.fixture(scope="module")
def search32():
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not found")
    d = tempfile.mkdtemp(prefix="qe_s32_")
    exe = os.path.join(d, "search32_check")
    subprocess.run([nvcc, "-x", "cu", "-O2", "-std=c++17", "-I", CSRC,
                    os.path.join(ROOT, "tests", "search32_check.cu"), "-o", exe], check=True)

    def go(cases):
        fin, fout = os.path.join(d, "in.txt"), os.path.join(d, "out.txt")
        with open(fin, "w") as f:
            for X, x in cases:
                f.write(f"{len(X)} {x} " + " ".join(map(str, X)) + "\n")
        subprocess.run([exe, fin, fout], check=True)
        return [tuple(map(int, ln.split())) for ln in open(fout).read().splitlines()]

    yield go
    shutil.rmtree(d, ignore_errors=True)


def test_five_tier_unit_search_finds_the_unit(search32):
    """The five-tier attention finds the unit holding a cost position (the largest u with
    X(u) <= x over the per-unit cost prefix) by rounds of 32 tests; it must equal the
    definition for any nondecreasing prefix, empty units (repeated X) included, in at most
    ceil(log32 n) + 1 rounds."""
    rng = random.Random(11)
    cases = []
    for _ in range(600):
        n = rng.choice([1, 2, 5, 31, 32, 33, 64, 100, 1000, 5000])
        X = [0]
        for _ in range(n - 1):
            X.append(X[-1] + rng.choice([0, rng.randint(1, 100), rng.randint(1, 10 ** 9)]))
        x = rng.choice([0, X[-1], rng.randint(0, X[-1] + 5)])
        cases.append((X, x))
    got = search32(cases)
    for (X, x), (u, rounds) in zip(cases, got):
        want = max(i for i in range(len(X)) if X[i] <= x)
        assert u == want, (len(X), x, u, want)
        bound = 1
        while 32 ** bound < len(X):
            bound += 1
        assert rounds <= bound + 1
