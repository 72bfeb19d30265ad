"""Pins for the paged block KV cache gather ("Attention DP", section "KV Cache": a rank's
cache is [num_blocks, num_kv_heads/TP, block_len, d_head]; a block table maps each
sequence's logical blocks to physical ones).

The oracle's gather is checked against a hand-worked example, against the seeded input
generator's independent scatter of a logical cache into pages (bf16 and fp8 with block
scales), and for attention invariance under any relabelling of the physical blocks."""

import math

import numpy as np
import torch

import oracle
from oracle import attention as A
from mla_decode_attention_gqa_gb300 import workloads as W


def test_hand_worked_gather():
    # 3 physical blocks of 2 tokens, 1 KV head, d = 1; page p row r holds 10 p + r
    pages = np.array([[[[10 * p + r] for r in range(2)]] for p in range(3)], dtype=np.float64)
    # sequence 0: logical blocks -> physical 2, 0, 1; sequence 1: 1, 1, 0 (shared pages)
    got = oracle.gather_pages(pages, [[2, 0, 1], [1, 1, 0]], 6)
    assert got[0, 0, :, 0].tolist() == [20, 21, 0, 1, 10, 11]
    assert got[1, 0, :, 0].tolist() == [10, 11, 10, 11, 0, 1]


def test_hand_worked_block_scales():
    # 2 physical blocks of 4 tokens with scale blocks of 2 tokens: 2 scales per page
    scales = np.array([[[1.0, 2.0]], [[3.0, 4.0]]])
    got = oracle.gather_block_scales(scales, [[1, 0]], 8, 4, 2)
    assert got[0, 0].tolist() == [3.0, 4.0, 1.0, 2.0]


def _f64(t):
    return oracle.bf16_bits_to_f64(t.contiguous().view(torch.int16).numpy())


def test_gather_inverts_the_generators_scatter_bf16():
    w = W.Workload("pg", B=3, Tq=1, Hq=4, Hkv=2, dk=16, dv=16, S=256, paged=True, block_len=64, seed=17)
    inp = W.make_inputs(w)
    for name, pages in (("k", inp["k_pages"]), ("v", inp["v_pages"])):
        got = oracle.gather_pages(pages.view(torch.int16).numpy(), inp["block_table_host"], w.S)
        assert np.array_equal(got, inp[name].view(torch.int16).numpy()), name


def test_gather_inverts_the_generators_scatter_fp8_with_scales():
    w = W.Workload("pg8", B=2, Tq=1, Hq=4, Hkv=2, dk=16, dv=16, S=512, paged=True, block_len=128,
                   kv_dtype="fp8_e4m3", seed=19)
    inp = W.make_inputs(w)
    got = oracle.gather_pages(inp["k_pages"].numpy(), inp["block_table_host"], w.S)
    assert np.array_equal(got, inp["k"].numpy())
    sc = oracle.gather_block_scales(inp["k_scale_pages"].numpy(), inp["block_table_host"], w.S, w.block_len,
                                    w.scale_block)
    assert np.array_equal(sc, inp["k_scale"].numpy())


def test_attention_is_invariant_under_page_relabelling():
    rng = np.random.default_rng(5)
    B, Hkv, L, d, nb = 2, 2, 4, 8, 3
    Hq = 4
    pages_k = rng.standard_normal((B * nb + 1, Hkv, L, d))
    pages_v = rng.standard_normal((B * nb + 1, Hkv, L, d))
    table = [[0, 1, 2], [3, 4, 5]]
    q = rng.standard_normal((B, 2, Hq, d))
    S = nb * L
    ref = A.full_attention(q, oracle.gather_pages(pages_k, table, S), oracle.gather_pages(pages_v, table, S),
                           [S, S - 3], W.NO_CAUSAL, 1 / math.sqrt(d))
    perm = rng.permutation(B * nb + 1)  # physical block p moves to perm[p]
    pk, pv = np.empty_like(pages_k), np.empty_like(pages_v)
    pk[perm], pv[perm] = pages_k, pages_v
    table2 = [[int(perm[p]) for p in row] for row in table]
    got = A.full_attention(q, oracle.gather_pages(pk, table2, S), oracle.gather_pages(pv, table2, S), [S, S - 3],
                           W.NO_CAUSAL, 1 / math.sqrt(d))
    np.testing.assert_array_equal(got[0], ref[0])
    np.testing.assert_array_equal(got[1], ref[1])
