"""Pins for the oracle: closed forms, brute force, invariants and library routines.

These tests never touch a GPU.  Each pin checks the oracle against something other
than itself, chosen so that a plausible slip (a dropped scale, a wrong sign or
index, a transposed operand, a wrong head mapping, an off-by-one causal mask, a
wrong merge weight) fails at least one of them; ``test_oracle_mutations.py`` plants
such slips in the oracle and checks that they are caught.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import attention as A

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _num(x):
    """Evaluate the small symbolic strings used in the golden fixtures."""
    if isinstance(x, (int, float)):
        return float(x)
    env = {"ln2": math.log(2), "ln3": math.log(3), "ln4": math.log(4), "ln5": math.log(5),
           "ln8": math.log(8)}
    return float(eval(x, {"__builtins__": {}}, env))


def _arr(xs):
    return np.array([[_num(v) for v in row] if isinstance(row, list) else _num(row) for row in xs])


# ---------------------------------------------------------------- number formats

def test_e4m3_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_bits_to_f64(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.all(both_nan | (ours == ref))
    assert np.array_equal(np.isnan(ours), np.isnan(ref))


def test_e4m3_spec_values():
    f = lambda c: float(oracle.e4m3_bits_to_f64(np.array([c], dtype=np.uint8))[0])
    assert f(0x7E) == 448.0  # largest finite: 1.75 * 2^8
    assert f(0x01) == 2.0 ** -9  # smallest subnormal
    assert f(0x08) == 2.0 ** -6  # smallest normal
    assert f(0x38) == 1.0
    assert f(0xC0) == -2.0
    assert math.isnan(f(0x7F)) and math.isnan(f(0xFF))
    assert f(0x80) == 0.0 and math.copysign(1.0, f(0x80)) == -1.0


def test_bf16_decode_matches_torch():
    g = torch.Generator().manual_seed(7)
    x = torch.randn(4096, generator=g).to(torch.bfloat16)
    ours = oracle.bf16_bits_to_f64(x.view(torch.int16).numpy())
    assert np.array_equal(ours, x.to(torch.float64).numpy())


def test_dequant_uses_absolute_block_index():
    codes = np.full((6, 2), 0x38, dtype=np.uint8)  # value 1.0
    scales = np.array([1.0, 2.0, 4.0])
    out = oracle.dequant_e4m3_blocks(codes, scales, block=4, t0=2)  # tokens 2..7
    assert np.array_equal(out[:, 0], [1.0, 1.0, 2.0, 2.0, 2.0, 2.0])


# ---------------------------------------------------------------- closed forms

@pytest.mark.parametrize("case", json.load(open(os.path.join(GOLDEN, "closed_form_attention.json")))["cases"],
                         ids=lambda c: c["name"])
def test_golden_closed_forms(case):
    q = np.array([_num(x) for x in case["q"]])[None, :]
    k = _arr(case["k"])
    v = _arr(case["v"])
    o, lse = oracle.attend(q, k, v, case["scale"])
    np.testing.assert_allclose(o[0], [_num(x) for x in case["expect_o"]], rtol=0, atol=1e-12)
    assert abs(lse[0] - _num(case["expect_lse"])) < 1e-12


def test_two_tokens_is_a_logistic_blend():
    rng = np.random.default_rng(1)
    for _ in range(20):
        q, k, v = rng.normal(size=(1, 5)), rng.normal(size=(2, 5)), rng.normal(size=(2, 3))
        sc = rng.uniform(0.1, 2.0)
        s0, s1 = sc * (q[0] @ k[0]), sc * (q[0] @ k[1])
        sig = 1.0 / (1.0 + math.exp(s1 - s0))
        o, lse = oracle.attend(q, k, v, sc)
        np.testing.assert_allclose(o[0], sig * v[0] + (1 - sig) * v[1], atol=1e-13)
        assert abs(lse[0] - np.logaddexp(s0, s1)) < 1e-13


def test_brute_force_without_max_shift():
    """Direct sums of exp(s) on small scores (no stabilisation) agree with the oracle."""
    rng = np.random.default_rng(2)
    R, n, dk, dv = 3, 5, 3, 2  # non-square on purpose: a transposed operand cannot fit
    q, k, v = rng.normal(size=(R, dk)), rng.normal(size=(n, dk)), rng.normal(size=(n, dv))
    sc = 0.7
    o, lse = oracle.attend(q, k, v, sc)
    for r in range(R):
        w = [math.exp(sc * sum(q[r, c] * k[t, c] for c in range(dk))) for t in range(n)]
        den = sum(w)
        for c in range(dv):
            assert abs(o[r, c] - sum(w[t] * v[t, c] for t in range(n)) / den) < 1e-13
        assert abs(lse[r] - math.log(den)) < 1e-13


def test_single_token_identical_keys_zero_query():
    rng = np.random.default_rng(3)
    v = rng.normal(size=(6, 4))
    q = rng.normal(size=(2, 8))
    k1 = rng.normal(size=(1, 8))
    o, lse = oracle.attend(q, k1, v[:1], 0.3)
    np.testing.assert_allclose(o, np.repeat(v[:1], 2, 0), atol=1e-14)
    np.testing.assert_allclose(lse, 0.3 * (q @ k1[0]), atol=1e-14)
    kk = np.repeat(k1, 6, 0)  # identical keys: mean of V, lse = s + ln n
    o, lse = oracle.attend(q, kk, v, 0.3)
    np.testing.assert_allclose(o, np.repeat(v.mean(0, keepdims=True), 2, 0), atol=1e-14)
    np.testing.assert_allclose(lse, 0.3 * (q @ k1[0]) + math.log(6), atol=1e-13)
    o, lse = oracle.attend(np.zeros((1, 8)), rng.normal(size=(6, 8)), v, 0.3)  # zero q
    np.testing.assert_allclose(o[0], v.mean(0), atol=1e-14)
    assert abs(lse[0] - math.log(6)) < 1e-14


def test_permutation_and_scale_invariants():
    rng = np.random.default_rng(4)
    q, k, v = rng.normal(size=(4, 6)), rng.normal(size=(9, 6)), rng.normal(size=(9, 5))
    o, lse = oracle.attend(q, k, v, 0.4)
    p = rng.permutation(9)
    o2, lse2 = oracle.attend(q, k[p], v[p], 0.4)
    np.testing.assert_allclose(o, o2, atol=1e-13)
    np.testing.assert_allclose(lse, lse2, atol=1e-13)
    o3, lse3 = oracle.attend(2.0 * q, k, v, 0.2)  # scale multiplies q.k
    np.testing.assert_allclose(o, o3, atol=1e-13)
    np.testing.assert_allclose(lse, lse3, atol=1e-13)
    o4, lse4 = oracle.attend(q, k, v + 3.0, 0.4)  # softmax weights sum to one
    np.testing.assert_allclose(o4, o + 3.0, atol=1e-13)
    np.testing.assert_allclose(lse4, lse, atol=1e-13)


# ---------------------------------------------------------------- causal mask

def _qkv(rng, B, Tq, Hq, Hkv, S, dk, dv):
    return rng.normal(size=(B, Tq, Hq, dk)), rng.normal(size=(B, Hkv, S, dk)), rng.normal(size=(B, Hkv, S, dv))


def test_causal_offset_zero_is_dense_lower_triangle():
    rng = np.random.default_rng(5)
    S = 7
    q, k, v = _qkv(rng, 1, S, 2, 1, S, 4, 3)
    o, lse = oracle.full_attention(q, k, v, [S], 0, 0.5)
    for i in range(S):  # row i attends to exactly tokens 0..i
        oo, ll = oracle.attend(q[0, i], k[0, 0, : i + 1], v[0, 0, : i + 1], 0.5)
        np.testing.assert_allclose(o[0, i], oo, atol=1e-13)
        np.testing.assert_allclose(lse[0, i], ll, atol=1e-13)
    # row 0 sees one token: its V row
    np.testing.assert_allclose(o[0, 0, 0], v[0, 0, 0], atol=1e-14)


def test_causal_offset_edges():
    rng = np.random.default_rng(6)
    q, k, v = _qkv(rng, 1, 3, 1, 1, 5, 4, 2)
    o_nomask, l_nomask = oracle.full_attention(q, k, v, [5], 1 << 62, 0.5)
    o_big, l_big = oracle.full_attention(q, k, v, [5], 4, 0.5)  # row 0 already sees all 5
    np.testing.assert_allclose(o_big, o_nomask, atol=1e-14)
    o_neg, l_neg = oracle.full_attention(q, k, v, [5], -1, 0.5)  # row 0 sees nothing
    assert np.all(o_neg[0, 0] == 0) and np.all(np.isneginf(l_neg[0, 0]))
    np.testing.assert_allclose(o_neg[0, 1, 0], v[0, 0, 0], atol=1e-14)  # row 1 sees token 0


# ---------------------------------------------------------------- GQA grouping

def test_gqa_contiguous_groups():
    assert [A.kv_head_of(h, 8, 2) for h in range(8)] == [0, 0, 0, 0, 1, 1, 1, 1]
    assert [A.kv_head_of(h, 128, 8) for h in (0, 15, 16, 127)] == [0, 0, 1, 7]
    rng = np.random.default_rng(7)
    q, k, v = _qkv(rng, 1, 1, 4, 2, 6, 3, 2)
    o, _ = oracle.full_attention(q, k, v, [6], 1 << 62, 1.0)
    k2, v2 = k.copy(), v.copy()
    k2[0, 1] += 1.0
    v2[0, 1] *= -2.0
    o2, _ = oracle.full_attention(q, k2, v2, [6], 1 << 62, 1.0)
    np.testing.assert_array_equal(o[0, 0, :2], o2[0, 0, :2])  # heads 0,1 read KV head 0
    assert np.all(np.abs(o[0, 0, 2:] - o2[0, 0, 2:]) > 1e-6)  # heads 2,3 read KV head 1
    for h in range(4):  # each head equals plain single-head attention on its KV head
        oo, _ = oracle.attend(q[0, :, h], k[0, h // 2], v[0, h // 2], 1.0)
        np.testing.assert_allclose(o[0, :, h], oo, atol=1e-14)


# ---------------------------------------------------------------- splits and merge

@pytest.mark.parametrize("seed", range(6))
def test_any_split_merges_to_unsplit(seed):
    rng = np.random.default_rng(100 + seed)
    B, Tq, Hq, Hkv, S = 2, 3, 4, 2, 40
    q, k, v = _qkv(rng, B, Tq, Hq, Hkv, S, 5, 3)
    seq = [int(rng.integers(1, S + 1)) for _ in range(B)]
    n_split = int(rng.integers(1, 6))
    cuts = sorted(int(c) for c in rng.integers(0, S + 1, size=n_split - 1))
    bounds = [[0] + cuts + [S] for _ in range(B)]
    causal = int(rng.choice([1 << 62, S - Tq, 10]))
    o_p, l_p = oracle.split_attention(q, k, v, seq, bounds, causal, 0.6)
    o_m, l_m = oracle.merge_lse(o_p, l_p)
    o_f, l_f = oracle.full_attention(q, k, v, seq, causal, 0.6)
    np.testing.assert_allclose(o_m, o_f, atol=1e-12)
    np.testing.assert_allclose(l_m, l_f, atol=1e-12)
    perm = rng.permutation(n_split)  # order of the fragments does not matter
    o_m2, l_m2 = oracle.merge_lse(o_p[perm], l_p[perm])
    np.testing.assert_allclose(o_m2, o_m, atol=1e-13)


def test_merged_fragments_merge_again():
    """A merged (o, lse) is itself a fragment: merging groups of splits first and then the
    groups' results (what a KVP group's All-to-All and a ring's running output do) gives
    the flat merge and the unsplit attention; a group whose splits are all empty merges to
    (0, -inf) and stays neutral one level up."""
    rng = np.random.default_rng(21)
    B, Tq, Hq, Hkv, S = 2, 2, 4, 2, 48
    q, k, v = _qkv(rng, B, Tq, Hq, Hkv, S, 5, 3)
    seq = [29, 48]  # batch 0: the last two splits lie past its end
    bounds = [[0, 5, 13, 20, 29, 40, 48]] * B
    o_p, l_p = oracle.split_attention(q, k, v, seq, bounds, 1 << 62, 0.7)
    groups = [[0, 1, 2], [3], [4, 5]]  # batch 0's group [4, 5] is empty
    lvl = [oracle.merge_lse(o_p[g], l_p[g]) for g in groups]
    assert np.all(np.isneginf(lvl[2][1][0])) and np.all(lvl[2][0][0] == 0)
    o2, l2 = oracle.merge_lse(np.stack([x[0] for x in lvl]), np.stack([x[1] for x in lvl]))
    o1, l1 = oracle.merge_lse(o_p, l_p)
    o_f, l_f = oracle.full_attention(q, k, v, seq, 1 << 62, 0.7)
    np.testing.assert_allclose(o2, o1, atol=1e-13)
    np.testing.assert_allclose(l2, l1, atol=1e-13)
    np.testing.assert_allclose(o2, o_f, atol=1e-12)
    np.testing.assert_allclose(l2, l_f, atol=1e-12)


def test_merge_two_fragments_closed_form_and_empty_split():
    rng = np.random.default_rng(8)
    o1, o2 = rng.normal(size=(3, 4)), rng.normal(size=(3, 4))
    l1, l2 = rng.normal(size=3) * 3, rng.normal(size=3) * 3
    o, lse = oracle.merge_lse(np.stack([o1, o2]), np.stack([l1, l2]))
    w1 = 1.0 / (1.0 + np.exp(l2 - l1))
    np.testing.assert_allclose(o, w1[:, None] * o1 + (1 - w1)[:, None] * o2, atol=1e-13)
    np.testing.assert_allclose(lse, np.logaddexp(l1, l2), atol=1e-13)
    # an empty fragment (o = 0, lse = -inf) is neutral
    oe, le = oracle.merge_lse(np.stack([o1, np.zeros_like(o1)]), np.stack([l1, np.full(3, -np.inf)]))
    np.testing.assert_allclose(oe, o1, atol=1e-15)
    np.testing.assert_allclose(le, l1, atol=1e-15)
    # all fragments empty -> o = 0, lse = -inf
    oz, lz = oracle.merge_lse(np.zeros((2, 3, 4)), np.full((2, 3), -np.inf))
    assert np.all(oz == 0) and np.all(np.isneginf(lz))


def test_split_past_seq_len_is_empty_and_poison_is_never_read():
    rng = np.random.default_rng(9)
    S = 16
    q, k, v = _qkv(rng, 1, 1, 2, 1, S, 4, 2)
    k[0, 0, 10:] = np.nan
    v[0, 0, 10:] = np.nan
    o, l = oracle.split_attention(q, k, v, [10], [[0, 8, 12, 16]], 1 << 62, 0.5)
    assert np.all(np.isfinite(o)) and np.all(np.isneginf(l[2]))
    assert np.all(o[2] == 0)
    o_t, l_t = oracle.full_attention(q, k[:, :, :10], v[:, :, :10], [10], 1 << 62, 0.5)
    o_m, l_m = oracle.merge_lse(o, l)
    np.testing.assert_allclose(o_m, o_t, atol=1e-13)
    np.testing.assert_allclose(l_m, l_t, atol=1e-13)
