"""Oracle pins against values the pages print (no GPU).

Each fixture under tests/golden/ carries its citation.
"""
import json
import math
import os

import numpy as np
import pytest

from conftest import GOLDEN
from oracle import budget
from oracle.h2o import h2o_step


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_h2o_capacity6_worked_step():
    g = _load("h2o_capacity6.json")
    heavy = {int(k): v for k, v in g["heavy_before"].items()}
    recent = {int(k): v for k, v in g["recent_before"].items()}
    S, evicted, cache = h2o_step(heavy, recent, g["new_position"], g["weights_over_candidates"],
                                 n_heavy=len(heavy), n_recent=len(recent))
    got = [round(float(S[p]), g["printed_decimals"]) for p in g["candidate_order"]]
    assert got == g["scores_after"]
    assert evicted == g["evicted"]
    assert cache == g["cache_after"]


def test_h2o_order_matters():
    """The victim is chosen on the updated scores (H2O page, §2.2 figure notes): once the
    current weight lifts position 8's score above position 5's, position 5 is evicted."""
    g = _load("h2o_capacity6.json")
    heavy = {int(k): v for k, v in g["heavy_before"].items()}
    recent = {int(k): v for k, v in g["recent_before"].items()}
    # Give position 8 a weight that lifts it above position 5: it must then survive.
    w = list(g["weights_over_candidates"])
    w[3] = 1.0
    S, evicted, cache = h2o_step(heavy, recent, 11, w, 3, 3)
    assert evicted == [5]
    assert cache == [1, 3, 8, 9, 10, 11]


def test_kivi_payload_formula():
    g = _load("byte_accounting.json")["kivi_payload"]
    b = budget.kivi_payload_bytes_per_elem(g["bits"], g["group"], g["param_bytes"])
    assert b == g["bytes_per_elem"]
    assert round(2 / b, 2) == g["compression_vs_bf16"]


def test_residual_region_ratio():
    g = _load("byte_accounting.json")["residual_region"]
    quant = budget.residual_region_bytes(8, 128, g["T"], g["R"], g["b"], g["b_bar"])
    full = budget.residual_region_bytes(8, 128, g["T"], 0, g["b"], g["b"])
    assert round(100 * quant / full, 1) == g["ratio_vs_bf16_percent_printed"]


def test_per_token_bytes():
    g = _load("byte_accounting.json")["per_token_bytes"]
    assert budget.kv_bytes_per_token(1, g["n_kv_heads"], g["head_dim"], g["elem_bytes"]) == g["per_layer"]
    per_tok = budget.kv_bytes_per_token(g["n_layers"], g["n_kv_heads"], g["head_dim"], g["elem_bytes"])
    assert per_tok == g["all_layers"]
    assert 8192 * per_tok == g["tokens_8k_bytes"]
    assert 8192 * budget.kv_bytes_per_token(g["n_layers"], 32, g["head_dim"], 2) == g["mha_32_kv_heads_8k_bytes"]
    m = _load("byte_accounting.json")["h2o_mha_example"]
    assert budget.kv_bytes_per_token(m["n_layers"], m["n_kv_heads"], m["head_dim"], m["elem_bytes"]) == m["per_token"]


def test_eq3_worked_example():
    g = _load("byte_accounting.json")["eq3_example"]
    kf, kq = budget.tier_capacities_eq3(g["B_hist_MB"], g["q"], g["M_f_MB"], g["M_q_MB"])
    assert (kf, kq) == (g["K_f"], g["K_q"])
    assert kf * g["window_tokens"] == g["full_tokens"]
    assert abs(kq * g["window_tokens"] - g["int2_tokens_approx"]) <= g["window_tokens"]
    m = _load("byte_accounting.json")["eq3_mf"]
    mf = m["window"] * budget.kv_bytes_per_token(32, 8, 128, 2) / 1024
    assert mf == m["M_f_KB"]
    # the page's "~131 KB" takes 1 MB as 1000 KB here (1024 KB would give 134 KB)
    assert round(1000 * 2 / 16 * 1.05) == m["M_q_KB_approx"]


def test_int2_window_bytes_match_kivi_formula():
    """The stored INT2 window (2-bit codes + float32 min and scale) follows the payload formula
    with 8 parameter bytes per group: K groups of w tokens, V groups of d channels."""
    w, d = 32, 128
    k_bytes = w * d * budget.kivi_payload_bytes_per_elem(2, w, 8)
    v_bytes = w * d * budget.kivi_payload_bytes_per_elem(2, d, 8)
    assert budget.int2_window_bytes(w, d) == k_bytes + v_bytes == 3328
