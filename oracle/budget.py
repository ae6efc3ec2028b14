"""Byte accounting and tier capacities.

Test infrastructure (see ``oracle/__init__``).

Sources
-------
* QEvict reading notes, §4.1 eq. "budget": sink and local bytes plus
  Full windows at M_f and Quantized windows at M_q must fit B_total.
* QEvict reading notes, §4.3 eq. (3): K_f = floor((1-q) B_hist / M_f),
  K_q = floor(q B_hist / M_q); §4.5 works the example through.
* KV Cache technology evolution, §2: B_KV = 2 N H_kv d b sum_i T_i; §5: KIVI
  payload w/8 + s/g bytes per element; §10.2: a cache holding T-R
  quantized tokens at b_bar bytes and R recent tokens at b bytes occupies
  2 H_kv d ((T-R) b_bar + R b) bytes per layer.
* H2O page, §1 (capacity M_KV = 2 L H_kv D N b).

Capacity rule per workload (the pages leave the mapping of "x % of tokens"
to window counts open; the reading adopted here): at a routing event with
current length L,
* fixed:        K_f, K_q given;
* token shares: K_f = max(0, floor((f_bf16 L - n_sink - n_recent) / w)),
                K_q = floor(f_int2 L / w);
* byte budget:  K_f as above, K_q = floor((budget - f_bf16) L * 4d / M_q(w)),
  where 4d is the bf16 K+V bytes of one token of one KV head.
"""
from __future__ import annotations

import math


def kv_bytes_per_token(n_layers: int, n_kv_heads: int, head_dim: int, elem_bytes: float) -> float:
    """2 (K and V) x layers x KV heads x head dim x bytes per element."""
    return 2 * n_layers * n_kv_heads * head_dim * elem_bytes


def kivi_payload_bytes_per_elem(bits: int, group: int, param_bytes: float) -> float:
    """Average bytes per element of a group-quantized tensor: bits/8 + params/group."""
    return bits / 8 + param_bytes / group


def residual_region_bytes(n_kv_heads: int, head_dim: int, T: int, R: int, b: float, b_bar: float) -> float:
    """Per-layer bytes with T-R quantized tokens (b_bar each) and R full-precision ones (b each)."""
    return 2 * n_kv_heads * head_dim * ((T - R) * b_bar + R * b)


def tier_capacities_eq3(B_hist: float, q: float, M_f: float, M_q: float):
    """eq. (3): (K_f, K_q)."""
    return math.floor((1 - q) * B_hist / M_f), math.floor(q * B_hist / M_q)


def int2_window_bytes(window: int, head_dim: int, v_group: int | None = None) -> int:
    """Device bytes of one INT2 window of one KV head as this build stores it.

    2-bit codes for K and V (2 * w * d / 4 bytes), float32 min + float32 scale
    per key channel (8 d) and per value group of each token (8 w d / v_group).
    """
    g = head_dim if v_group is None else v_group
    return 2 * window * head_dim // 4 + 8 * head_dim + 8 * window * (head_dim // g)


def bf16_token_bytes(head_dim: int) -> int:
    """bf16 K + V bytes of one token of one KV head."""
    return 2 * head_dim * 2


def capacities(wl, L: int):
    """(K_f, K_q) in windows per (layer, KV head) at current length L."""
    if wl.cap_mode == 0:
        return wl.kf, wl.kq
    w = wl.window
    kf = max(0, math.floor((wl.frac_bf16 * L - wl.n_sink - wl.n_recent) / w))
    if wl.cap_mode == 1:
        kq = math.floor(wl.frac_int2 * L / w)
    elif wl.cap_mode == 2:
        kq = math.floor((wl.budget_frac - wl.frac_bf16) * L * bf16_token_bytes(wl.head_dim)
                        / int2_window_bytes(w, wl.head_dim))
    else:
        raise ValueError(f"unknown cap_mode {wl.cap_mode}")
    return kf, max(0, kq)
