"""Seeded synthetic inputs for the tiered KV-cache decode path.

This module holds no part of the method's arithmetic: it only draws the
key/value/query tensors that both the CPU oracle and the CUDA path consume.
Every number is produced by integer arithmetic (SplitMix64, a published
counter-based mixer by Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014; finaliser constants as popularised by
Vigna) followed by exactly-representable float32 operations and a
round-to-nearest-even cast to bf16, so a second implementation (the CUDA
generator in ``gen.cu``) reproduces every bit.

Normal variates are Irwin-Hall sums of twelve 16-bit uniforms (mean 0,
variance 1 up to 2^-32, support [-6, 6]).  A row of ``d`` channels with
64-bit row key ``k`` draws channel ``c`` from
``splitmix64(k + 3c + j)`` for ``j = 0, 1, 2`` (four 16-bit fields each).

Row keys chain SplitMix64 over (seed, tensor id, batch, layer, head,
position-or-step), see :func:`row_key`.

Workloads (shapes, windows, capacities, value recipes) are defined in
:data:`WORKLOADS`, each with the value recipe of the workload it stands for.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np

__all__ = [
    "GAMMA", "splitmix64", "row_key", "normal_int_sums", "normal_rows_f32",
    "bf16_bits_rne", "bf16_bits_to_f32", "Workload", "WORKLOADS",
    "outlier_channels", "channel_scales", "planted_direction",
    "gen_keys_values", "gen_queries", "drift_window", "drift_mean",
    "T_K", "T_V", "T_Q", "T_OUTLIER", "T_DRIFT", "T_PLANT", "T_SCORE",
]

GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_U64 = np.uint64

# tensor ids mixed into the row key
T_K, T_V, T_Q, T_OUTLIER, T_DRIFT, T_PLANT, T_SCORE = 1, 2, 3, 4, 5, 6, 7

# Irwin-Hall offset: 12 draws of 16 bits, mean 12 * 32767.5
IH_OFFSET = 393210
IH_SCALE = 65536.0


def splitmix64(x):
    """SplitMix64 output function on uint64 (array or scalar), wrapping."""
    x = np.asarray(x, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = x + _U64(GAMMA)
        z = (z ^ (z >> _U64(30))) * _U64(_M1)
        z = (z ^ (z >> _U64(27))) * _U64(_M2)
        return z ^ (z >> _U64(31))


def row_key(seed, tensor, b, layer, head, pos):
    """64-bit key of one d-vector; every argument broadcasts (ints or arrays)."""
    k = splitmix64(_U64(seed))
    for part in (tensor, b, layer, head, pos):
        k = splitmix64(k ^ np.asarray(part, dtype=np.int64).astype(np.uint64))
    return k


def normal_int_sums(keys, d: int):
    """Centred Irwin-Hall integer sums S - 393210 for each key and channel.

    Returns int64 of shape keys.shape + (d,), values in [-393210, 393210].
    """
    keys = np.asarray(keys, dtype=np.uint64)
    c = np.arange(d, dtype=np.uint64)
    with np.errstate(over="ignore"):
        base = keys[..., None] + _U64(3) * c
        s = np.zeros(base.shape, dtype=np.int64)
        for j in range(3):
            r = splitmix64(base + _U64(j))
            for sh in (0, 16, 32, 48):
                s += ((r >> _U64(sh)) & _U64(0xFFFF)).astype(np.int64)
    return s - IH_OFFSET


def normal_rows_f32(keys, d: int, scale_int=None):
    """float32 normal rows; ``scale_int`` (int, broadcast over channels) multiplies exactly."""
    s = normal_int_sums(keys, d)
    if scale_int is not None:
        s = s * np.asarray(scale_int, dtype=np.int64)
    # |s| < 2^22 so the int->float32 conversion and the power-of-two division are exact
    return s.astype(np.float32) / np.float32(IH_SCALE)


def bf16_bits_rne(f32):
    """Round float32 to bf16 (nearest, ties to even); returns uint16 bits.  No NaN inputs."""
    bits = np.ascontiguousarray(f32, dtype=np.float32).view(np.uint32).astype(np.uint64)
    bits = (bits + _U64(0x7FFF) + ((bits >> _U64(16)) & _U64(1))) >> _U64(16)
    return bits.astype(np.uint16)


def bf16_bits_to_f32(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


@dataclasses.dataclass(frozen=True)
class Workload:
    """Shapes, window geometry, capacity rule and value recipe of one workload."""
    name: str
    batch: int
    n_layers: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    prefill: int            # L0 tokens per sequence
    decode_steps: int       # T
    window: int             # w tokens per window
    route_period: int       # Omega
    n_sink: int
    n_recent: int
    cap_mode: int           # 0 fixed counts, 1 token fractions, 2 byte budget
    kf: int = 0
    kq: int = 0
    frac_bf16: float = 0.0
    frac_int2: float = 0.0
    budget_frac: float = 0.0
    seed: int = 20261202
    # value recipe
    outlier_mode: str = "random4x10"   # "fixed" (channels, scale) or "random4x10"
    outlier_fixed: tuple = ()          # ((channel, scale), ...) for mode "fixed"
    plant_tokens: tuple = ()           # (first, last_exclusive) positions planted along u
    plant_step: int = 0                # decode step from which queries carry u
    plant_amp: float = 3.0
    drift_period: int = 0              # 0 = no drift
    # five-tier per-token variant (tiering "tokens"): token fractions of the BF16 / INT4 / INT2 /
    # 1-bit tiers (the rest evicted) and the number of last steps before a re-rank whose
    # attention is counted (0 = every step); route_period is the re-rank period
    tiering: str = "windows"
    frac_int4: float = 0.0
    frac_nq1: float = 0.0
    score_window: int = 0
    # rotary embedding base for keys stored pre-RoPE (0 = keys carry no rotation)
    rope_theta: float = 0.0
    # 2-bit window slots beyond the most K_q (cache setting): 0 automatic, -1 none, n > 0
    int2_slack: int = 0

    @property
    def group(self) -> int:
        return self.n_q_heads // self.n_kv_heads

    @property
    def max_context(self) -> int:
        return self.prefill + self.decode_steps


WORKLOADS = {
    # 1 layer, batch 1, H_q=4/H_kv=1, d=64; 256 + 64; w=16, Omega=8; 4 sink + 16 recent; Kf=3, Kq=4
    "tiny_qevict": Workload(
        name="tiny_qevict", batch=1, n_layers=1, n_q_heads=4, n_kv_heads=1, head_dim=64,
        prefill=256, decode_steps=64, window=16, route_period=8, n_sink=4, n_recent=16,
        cap_mode=0, kf=3, kq=4, seed=20261202 + 1,
        outlier_mode="fixed", outlier_fixed=((3, 8), (17, 8)),
        plant_tokens=(64, 80), plant_step=40, plant_amp=3.0),
    # Llama-3.1-8B-shaped stack, 20% byte budget (10% of tokens BF16, INT2 fills the rest)
    "llama8b_stack": Workload(
        name="llama8b_stack", batch=1, n_layers=32, n_q_heads=32, n_kv_heads=8, head_dim=128,
        prefill=512, decode_steps=256, window=16, route_period=16, n_sink=5, n_recent=32,
        cap_mode=2, frac_bf16=0.10, budget_frac=0.20, seed=20261202 + 2,
        drift_period=64),
    # headline throughput workload
    "throughput_32k": Workload(
        name="throughput_32k", batch=16, n_layers=32, n_q_heads=32, n_kv_heads=8, head_dim=128,
        prefill=32768, decode_steps=128, window=32, route_period=32, n_sink=5, n_recent=32,
        cap_mode=1, frac_bf16=0.08, frac_int2=0.25, seed=20261202 + 3,
        drift_period=64),
    # the throughput workload with keys stored pre-RoPE (rotary base 10000), rotated in the
    # attention at their original positions
    "throughput_32k_rope": Workload(
        name="throughput_32k_rope", batch=16, n_layers=32, n_q_heads=32, n_kv_heads=8, head_dim=128,
        prefill=32768, decode_steps=128, window=32, route_period=32, n_sink=5, n_recent=32,
        cap_mode=1, frac_bf16=0.08, frac_int2=0.25, seed=20261202 + 3,
        drift_period=64, rope_theta=10000.0),
    # five-tier per-token variant: 10 % BF16 / 20 % INT4 / 30 % INT2 / 30 % 1-bit / 10 % evicted,
    # re-ranked every 64 steps over the attention of the last 20 steps (w = 32 is the drift epoch's
    # window grid only)
    "hqe_16k": Workload(
        name="hqe_16k", batch=8, n_layers=32, n_q_heads=32, n_kv_heads=8, head_dim=128,
        prefill=16384, decode_steps=128, window=32, route_period=64, n_sink=5, n_recent=32,
        cap_mode=1, frac_bf16=0.10, frac_int2=0.30, seed=20261202 + 5, drift_period=64,
        tiering="tokens", frac_int4=0.20, frac_nq1=0.30, score_window=20),
    # the same rule at a size the oracle follows through every step
    "tiny_hqe": Workload(
        name="tiny_hqe", batch=2, n_layers=2, n_q_heads=8, n_kv_heads=2, head_dim=128,
        prefill=300, decode_steps=48, window=32, route_period=16, n_sink=5, n_recent=16,
        cap_mode=1, frac_bf16=0.10, frac_int2=0.30, seed=20261202 + 6, drift_period=64,
        tiering="tokens", frac_int4=0.20, frac_nq1=0.30, score_window=6),
    "long_131k": Workload(
        name="long_131k", batch=1, n_layers=32, n_q_heads=32, n_kv_heads=8, head_dim=128,
        prefill=131072, decode_steps=64, window=64, route_period=64, n_sink=5, n_recent=32,
        cap_mode=1, frac_bf16=0.05, frac_int2=0.30, seed=20261202 + 4,
        drift_period=64),
}


def outlier_channels(wl: Workload, layer: int, kvh: int) -> list:
    """[(channel, integer scale)] of the key outlier channels of one KV head."""
    if wl.outlier_mode == "fixed":
        return [tuple(x) for x in wl.outlier_fixed]
    key = row_key(wl.seed, T_OUTLIER, 0, layer, kvh, 0)
    chosen, i = [], 0
    while len(chosen) < 4:
        c = int(splitmix64(key + _U64(i)) % _U64(wl.head_dim))
        i += 1
        if c not in chosen:
            chosen.append(c)
    return [(c, 10) for c in chosen]


def channel_scales(wl: Workload, layer: int, kvh: int) -> np.ndarray:
    s = np.ones(wl.head_dim, dtype=np.int64)
    for c, m in outlier_channels(wl, layer, kvh):
        s[c] = m
    return s


def planted_direction(wl: Workload, layer: int, kvh: int) -> np.ndarray:
    """Unit vector u (float64) of one KV head, from a seeded normal row."""
    n = normal_rows_f32(row_key(wl.seed, T_PLANT, 0, layer, kvh, 0), wl.head_dim).astype(np.float64)
    return n / math.sqrt(float(np.sum(n * n)))


def gen_keys_values(wl: Workload, b: int, layer: int, kvh: int, pos0: int, n: int):
    """bf16 bits of K and V rows for positions [pos0, pos0+n) of one (batch, layer, KV head).

    Returns (k_bits, v_bits), each uint16 [n, d].
    """
    d = wl.head_dim
    pos = np.arange(pos0, pos0 + n, dtype=np.int64)
    kk = row_key(wl.seed, T_K, b, layer, kvh, pos)
    kv = row_key(wl.seed, T_V, b, layer, kvh, pos)
    kf = normal_rows_f32(kk, d, channel_scales(wl, layer, kvh))
    if wl.plant_tokens:
        lo, hi = wl.plant_tokens
        sel = (pos >= lo) & (pos < hi)
        if np.any(sel):
            u = planted_direction(wl, layer, kvh)
            kf[sel] = (kf[sel].astype(np.float64) + wl.plant_amp * u).astype(np.float32)
    vf = normal_rows_f32(kv, d)
    return bf16_bits_rne(kf), bf16_bits_rne(vf)


def drift_window(wl: Workload, b: int, layer: int, kvh: int, step: int) -> int:
    """Window whose mean key the queries of decode step ``step`` (1-based) lean towards.

    Re-drawn at steps 1, 1+P, 1+2P, ... (P = drift period) uniformly among the
    complete windows before the current position of the epoch's first step.
    """
    epoch = (step - 1) // wl.drift_period
    first = epoch * wl.drift_period + 1
    p = wl.prefill + first - 1
    n_complete = p // wl.window
    r = splitmix64(row_key(wl.seed, T_DRIFT, b, layer, kvh, epoch))
    return int(r % _U64(n_complete))


def drift_mean(wl: Workload, b: int, layer: int, kvh: int, step: int) -> np.ndarray:
    """Exact float64 mean of the original bf16 keys of the drift window."""
    j = drift_window(wl, b, layer, kvh, step)
    kb, _ = gen_keys_values(wl, b, layer, kvh, j * wl.window, wl.window)
    return bf16_bits_to_f32(kb).astype(np.float64).sum(axis=0) / wl.window


def gen_queries(wl: Workload, b: int, layer: int, heads: Sequence[int], step: int):
    """bf16 bits of the queries of decode step ``step`` (1-based) for the given query heads: [len(heads), d]."""
    d = wl.head_dim
    heads = np.asarray(list(heads), dtype=np.int64)
    keys = row_key(wl.seed, T_Q, b, layer, heads, step)
    z = normal_rows_f32(keys, d)
    if wl.plant_tokens and step >= wl.plant_step:
        out = np.empty_like(z)
        for i, h in enumerate(heads):
            u = planted_direction(wl, layer, int(h) // wl.group)
            out[i] = (z[i].astype(np.float64) + wl.plant_amp * u).astype(np.float32)
        z = out
    if wl.drift_period:
        out = np.empty_like(z)
        for i, h in enumerate(heads):
            mu = drift_mean(wl, b, layer, int(h) // wl.group, step)
            out[i] = (z[i].astype(np.float64) + mu).astype(np.float32)
        z = out
    return bf16_bits_rne(z)
