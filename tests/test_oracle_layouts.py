"""Pins for attention over tokens stored out of sequence order (zigzag and striped layouts).

The layout maps and the causal rule by original position are checked against the worked
examples printed in "现代大模型推理并行策略总览", section "序列布局：Contiguous、Zigzag 与
Striped" and the chunk pairing of "Context Parallelism for Scalable Million-Token
Inference", section "Load-balanced sharding makes causal work and memory land evenly"
(fixture ``tests/golden/sequence_layouts.json``), and the oracle's attention under a
layout against the plain causal attention over the original order (the pages state that
the storage order does not change the result), and against brute force on a tiny case.
"""

import json
import math
import os

import numpy as np
import pytest

from oracle import attention as A
from mla_decode_attention_gqa_gb300 import workloads as W

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "sequence_layouts.json")))


def test_zigzag_rank_blocks_match_the_worked_example():
    g = GOLDEN["zigzag_S32_CP4"]
    for r, want in enumerate(g["rank_positions"]):
        assert W.layout_positions("zigzag", 32, 4, r) == want


def test_zigzag_pairs_chunk_i_with_chunk_2n_minus_1_minus_i():
    # one-token chunks: rank i holds (C_i, C_{2N-i-1})
    for r, want in enumerate(GOLDEN["zigzag_CP2_chunk_pairs"]):
        assert W.layout_positions("zigzag", 4, 2, r) == want


def test_striped_rank_positions_match_the_worked_example():
    for r, want in enumerate(GOLDEN["striped_S8_CP2"]["rank_positions"]):
        assert W.layout_positions("striped", 8, 2, r) == want


def test_every_zigzag_rank_processes_132_kv_positions():
    """S=32, CP=4: each rank's queries see 132 KV positions in total (causal, all 32 KV)."""
    want = GOLDEN["zigzag_S32_CP4"]["kv_positions_processed_per_rank"]
    all_kv = np.arange(32)
    for r in range(4):
        q = W.layout_positions("zigzag", 32, 4, r)
        assert int(A.visible_mask(q, all_kv).sum()) == want
    # the contiguous split of the same sequence is unbalanced (36 ... 228)
    counts = [int(A.visible_mask(W.layout_positions("contiguous", 32, 4, r), all_kv).sum()) for r in range(4)]
    assert counts == [36, 100, 164, 228] and sum(counts) == 4 * want


def test_striped_visibility_example():
    """Rank 0 (Q[0,2,4,6]) against rank 1's K/V[1,3,5,7]: Q2 sees K1 only, Q4 sees K1 and K3."""
    g = GOLDEN["striped_S8_CP2"]
    q = g["rank_positions"][0]
    kv = g["rank_positions"][1]
    mask = A.visible_mask(q, kv)
    for qp, seen in g["rank0_queries_against_rank1_kv"].items():
        i = q.index(int(qp))
        assert [kv[t] for t in np.flatnonzero(mask[i])] == seen
    assert not mask[q.index(0)].any()  # position 0 sees nothing of rank 1


def _contiguous_reference(q_all, k_all, v_all, scale):
    """Plain causal attention over the original order (row i sees t <= i)."""
    B, S = q_all.shape[0], q_all.shape[1]
    return A.full_attention(q_all, k_all, v_all, [S] * B, 0, scale)


@pytest.mark.parametrize("layout,S,cp", [("zigzag", 32, 4), ("striped", 24, 3), ("zigzag", 48, 2), ("striped", 16, 4)])
def test_layout_attention_equals_original_order_attention(layout, S, cp):
    """Storing tokens in a layout and masking by original position reproduces the attention
    of the original order, row by row, for every rank's query chunk and all its splits merged."""
    rng = np.random.default_rng(7)
    B, Hq, Hkv, d = 1, 4, 2, 8
    scale = 1.0 / math.sqrt(d)
    q_all = rng.standard_normal((B, S, Hq, d))
    k_all = rng.standard_normal((B, Hkv, S, d))
    v_all = rng.standard_normal((B, Hkv, S, d))
    ref_o, ref_l = _contiguous_reference(q_all, k_all, v_all, scale)
    k_order = [p for r in range(cp) for p in W.layout_positions(layout, S, cp, r)]
    k_st, v_st = k_all[:, :, k_order], v_all[:, :, k_order]
    m = S // cp
    bounds = [[j * m for j in range(cp + 1)]]
    for r in range(cp):
        q_order = W.layout_positions(layout, S, cp, r)
        o_p, l_p = A.split_attention(q_all[:, q_order], k_st, v_st, [S], bounds, 0, scale,
                                     q_positions=[q_order], k_positions=[k_order])
        o, l = A.merge_lse(o_p, l_p)
        np.testing.assert_allclose(o, ref_o[:, q_order], rtol=0, atol=1e-12)
        np.testing.assert_allclose(l, ref_l[:, q_order], rtol=0, atol=1e-12)


def test_layout_attention_brute_force_tiny():
    """Striped S=8, CP=2, rank 1: every row against every stored token by explicit loops."""
    rng = np.random.default_rng(3)
    d, scale = 4, 0.5
    S, cp, r = 8, 2, 1
    k_order = [p for j in range(cp) for p in W.layout_positions("striped", S, cp, j)]
    q_order = W.layout_positions("striped", S, cp, r)
    q = rng.standard_normal((len(q_order), d))
    k = rng.standard_normal((S, d))
    v = rng.standard_normal((S, d))
    o, l = A.attend(q, k, v, scale, q_order, k_order)
    for i, qp in enumerate(q_order):
        w, acc = [], np.zeros(d)
        for t, kp in enumerate(k_order):
            if kp <= qp:
                w.append((math.exp(scale * float(q[i] @ k[t])), t))
        den = sum(x for x, _ in w)
        for x, t in w:
            acc += x / den * v[t]
        assert abs(l[i] - math.log(den)) < 1e-12
        np.testing.assert_allclose(o[i], acc, rtol=0, atol=1e-12)
