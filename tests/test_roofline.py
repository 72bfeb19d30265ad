"""The algorithmic-bytes/flops arithmetic reproduces the pages' printed roofline figures."""

import json
import os

import pytest

from mla_decode_attention_gqa_gb300 import roofline as R

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "roofline_pages.json")))


@pytest.mark.parametrize("row", GOLDEN["helix"]["rows"])
def test_helix_figure1_kv_read(row):
    p = GOLDEN["helix"]["params"]
    t = R.helix_kv_read_seconds(p["B"], p["K"], row["TPA"], p["Hsz"], p["S"], row["KVP"],
                                p["bytes_param"], p["membw"])
    assert abs(t * 1e6 - row["kv_read_us_approx"]) < 0.5  # the page prints "~128 us", "~16 us"


@pytest.mark.parametrize("row", GOLDEN["dcp_h200"]["rows"])
def test_dcp_h200_kv_scan(row):
    p = GOLDEN["dcp_h200"]["params"]
    t = R.helix_kv_read_seconds(p["B"], p["K"], row["TPA"], p["Hsz"], p["S"], row["KVP"],
                                p["bytes_param"], p["membw"])
    assert abs(t * 1e6 - row["kv_scan_us"]) < 0.005  # printed to two decimals
    # the same bytes through the per-call counter (one KV head, KVP shards as splits)
    S = p["S"]
    kvp = row["KVP"]
    bounds = [[0, S // kvp]] * p["B"]
    b = R.kv_bytes(1, p["Hsz"], p["Hsz"], "bf16", [S] * p["B"], bounds)
    assert b == row["kv_cache_bytes"]


def test_kv_bytes_counts_each_visible_token_once():
    # 2 splits covering 0..100 of a 100-token sequence, 3 KV heads, bf16 d=4
    assert R.kv_bytes(3, 4, 4, "bf16", [100], [[0, 60, 128]]) == 100 * 3 * 8 * 2
    # ragged: a split past seq_len reads nothing
    assert R.kv_bytes(1, 4, 4, "bf16", [50], [[0, 64, 128]]) == 50 * 8 * 2
    # MLA: the latent row is read once (V is part of it)
    assert R.kv_bytes(1, 576, 512, "bf16", [10], [[0, 10]], mla=True) == 10 * 576 * 2
    # fp8: one byte per element plus one fp32 scale per touched 64-token block, K and V
    assert R.kv_bytes(1, 128, 128, "fp8_e4m3", [130], [[0, 130]]) == 130 * 256 + 2 * 4 * 3


def test_flops_count_visible_pairs():
    # decode: Tq=1, no mask
    assert R.attn_flops(1, 2, 8, 8, [10], [[0, 10]]) == 2 * 16 * 2 * 10
    # causal, offset 0, 4 rows over 4 tokens: 1+2+3+4 visible pairs
    assert R.attn_flops(4, 1, 8, 8, [4], [[0, 4]], causal_offset=0) == 2 * 16 * 10
    # ring prefill: last of 8 chunks of 4096 -> 7 full chunks + the diagonal triangle
    T = 4096
    f = R.attn_flops(T, 128, 128, 128, [8 * T], [[j * T for j in range(9)]], causal_offset=7 * T)
    assert f == 2 * 256 * 128 * (7 * T * T + T * (T + 1) // 2)
    assert abs(f - 8.246471426048e12) < 1  # figure in the workload's roofline table
