"""GPU parity of the GQA split-KV path (bf16 and fp8 KV) against the fp64 oracle.

Every case runs the CUDA kernels through the C ABI (ctypes binding) on seeded inputs
from ``workloads.make_inputs`` and compares element by element with the oracle on the
same bytes.  Bars: bf16 KV out max-abs <= 1e-2, lse <= 1e-3; fp8 KV <= 4e-2 (both).
"""

import numpy as np
import pytest
import torch

import mla_decode_attention_gqa_gb300 as skv
from mla_decode_attention_gqa_gb300 import workloads as W
import oracle
from tests import oracle_io as io

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _run_all_paths(w, inp, bounds=None, causal=None):
    """Partials, separate merge and fused call for one workload; checked against the oracle."""
    bounds = inp["split_bounds"] if bounds is None else bounds
    causal = w.causal_offset if causal is None else causal
    tol = io.tol_for(w)
    kw = dict(k_scale=inp["k_scale"], v_scale=inp["v_scale"], softmax_scale=w.scale, scale_block=w.scale_block)
    o_p, l_p = skv.attn_partial(inp["q"], inp["k"], inp["v"], inp["seq_lens"], bounds, causal, **kw)
    o_m, l_m = skv.attn_merge_lse(o_p, l_p)
    o_f, l_f = skv.gqa_decode_attn(inp["q"], inp["k"], inp["v"], inp["seq_lens"], bounds, causal, **kw)
    torch.cuda.synchronize()
    assert skv.device_error() == 0
    ro_p, rl_p = io.oracle_all(inp, w, bounds, causal)
    ro, rl = oracle.merge_lse(ro_p, rl_p)
    io.assert_close(o_p, l_p, ro_p, rl_p, tol, "partials")
    io.assert_close(o_m, l_m, ro, rl, tol, "merged")
    io.assert_close(o_f, l_f, ro, rl, tol, "fused")
    return o_f, l_f


def test_tiny_gqa_decode_full():
    """The tiny workload in full: B=1 Hq=8 Hkv=2 d=64 S=1024, 4 splits."""
    w = W.TINY_GQA
    inp = W.make_inputs(w, DEV)
    _run_all_paths(w, inp)


@pytest.mark.parametrize("S,n_split", [(4096, 1), (3000, 3), (1000, 4)])
def test_helix_dense_shape_small_s(S, n_split):
    """Helix dense decode heads (B=2, Hq=128, Hkv=8, d=128) at oracle-friendly S, incl. ragged tails."""
    w = W.scaled(W.HELIX_DENSE_128K, B=2, S=S, n_split=n_split)
    inp = W.make_inputs(w, DEV)
    _run_all_paths(w, inp)


def test_fp8_kvp8_ragged_small_s():
    """fp8-e4m3 KV, 64-token block scales, 8 contiguous shards, ragged seq_lens, NaN past the end."""
    w = W.scaled(W.HELIX_KVP8_FP8_1M, B=3, S=8192)
    inp = W.make_inputs(w, DEV)
    assert min(inp["seq_lens_host"]) < w.S  # ragged: some shards are partly or wholly empty
    _run_all_paths(w, inp)


def test_fp8_unaligned_bounds_and_block_scale_128():
    w = W.scaled(W.HELIX_KVP8_FP8_1M, B=2, S=2048, n_split=3, scale_block=128)
    inp = W.make_inputs(w, DEV)
    bounds = [[5, 700, 701, 2048], [0, 1000, 1500, 1900]]
    _run_all_paths(w, inp, bounds=bounds)


def test_ring_prefill_chunk_small():
    """Ring pass-KV prefill structure: the Q chunk is the last of 8 KV chunks, causal on the diagonal."""
    w = W.scaled(W.RING_PREFILL, Tq=64, S=8 * 64, Hq=32, Hkv=2)
    inp = W.make_inputs(w, DEV)
    o_f, l_f = _run_all_paths(w, inp)
    # per-step form: each ring step on its own KV chunk with causal_offset = (7 - j) * chunk
    T = 64
    kw = dict(softmax_scale=w.scale)
    parts_o, parts_l = [], []
    for j in range(8):
        kj = inp["k"][:, :, j * T : (j + 1) * T]
        vj = inp["v"][:, :, j * T : (j + 1) * T]
        o, l = skv.attn_partial(inp["q"], kj, vj, torch.full((1,), T, dtype=torch.int32, device=DEV),
                                [[0, T]], (7 - j) * T, **kw)
        parts_o.append(o)
        parts_l.append(l)
    o_s, l_s = skv.attn_merge_lse(torch.cat(parts_o), torch.cat(parts_l))
    torch.cuda.synchronize()
    assert (o_s.float() - o_f.float()).abs().max().item() <= 1e-2
    assert (l_s - l_f).abs().max().item() <= 1e-3


def test_prefill_causal_offset_zero_dense_lower_triangle():
    w = W.Workload("causal0", B=1, Tq=100, Hq=8, Hkv=2, dk=64, dv=64, S=100, n_split=2, causal_offset=0,
                   seed=77)
    inp = W.make_inputs(w, DEV)
    _run_all_paths(w, inp)


def test_edge_cases_empty_splits_zero_len_and_negative_offset():
    w = W.Workload("edges", B=3, Tq=2, Hq=8, Hkv=2, dk=64, dv=64, S=300, n_split=4, seed=78)
    inp = W.make_inputs(w, DEV)
    inp["seq_lens"] = torch.tensor([0, 130, 300], dtype=torch.int32, device=DEV)
    inp["seq_lens_host"] = [0, 130, 300]
    bounds = [[0, 0, 64, 200, 300], [0, 100, 100, 129, 300], [10, 11, 12, 13, 299]]
    _run_all_paths(w, inp, bounds=bounds)  # empty splits, a zero-length sequence, tiny splits
    _run_all_paths(w, inp, bounds=bounds, causal=-1)  # row 0 sees nothing, row 1 sees token 0


def test_nan_outside_the_split_is_never_read():
    w = W.scaled(W.HELIX_DENSE_128K, B=1, S=640, n_split=1)
    inp = W.make_inputs(w, DEV)
    bounds = [[100, 500]]
    inp["k"][:, :, :100] = float("nan")
    inp["v"][:, :, :100] = float("nan")
    inp["k"][:, :, 500:] = float("nan")
    inp["v"][:, :, 500:] = float("nan")
    o, l = skv.attn_partial(inp["q"], inp["k"], inp["v"], inp["seq_lens"], bounds, softmax_scale=w.scale)
    torch.cuda.synchronize()
    ro, rl = io.oracle_all(inp, w, bounds)
    io.assert_close(o, l, ro, rl, io.TOL_BF16, "poisoned")


def test_strided_query_and_cache_views():
    """q and K/V given as non-contiguous views (explicit strides go through the ABI)."""
    w = W.Workload("strided", B=2, Tq=1, Hq=16, Hkv=4, dk=128, dv=128, S=512, n_split=2, seed=79)
    inp = W.make_inputs(w, DEV)
    big_q = torch.zeros((2, 3, 24, 128), dtype=torch.bfloat16, device=DEV)
    big_q[:, 1:2, 4:20] = inp["q"]
    q_view = big_q[:, 1:2, 4:20]
    big_k = torch.zeros((2, 6, 512, 128), dtype=torch.bfloat16, device=DEV)
    big_k[:, 1:5] = inp["k"]
    k_view = big_k[:, 1:5]
    o, l = skv.gqa_decode_attn(q_view, k_view, inp["v"], inp["seq_lens"], inp["split_bounds"],
                               softmax_scale=w.scale)
    torch.cuda.synchronize()
    ro_p, rl_p = io.oracle_all(inp, w)
    ro, rl = oracle.merge_lse(ro_p, rl_p)
    io.assert_close(o, l, ro, rl, io.TOL_BF16, "strided")


def test_repeat_calls_are_deterministic():
    w = W.scaled(W.HELIX_DENSE_128K, B=2, S=2048)
    inp = W.make_inputs(w, DEV)
    a = skv.gqa_decode_attn(inp["q"], inp["k"], inp["v"], inp["seq_lens"], inp["split_bounds"])
    b = skv.gqa_decode_attn(inp["q"], inp["k"], inp["v"], inp["seq_lens"], inp["split_bounds"])
    torch.cuda.synchronize()
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


@pytest.mark.parametrize("q_exp", [17, -20], ids=["q_above_fp16_max", "q_below_fp16_normal"])
@pytest.mark.parametrize("Tq", [1, 4], ids=["decode", "prefill_rows"])
def test_fp8_query_outside_the_fp16_range(q_exp, Tq):
    """fp8 KV runs its products in f16, so the bf16 query is converted to fp16.  The kernels
    scale each warp's query rows by a power of two first and fold it back into the score
    scale, so a query far above fp16's largest finite value (2^17 > 65504) or below its
    smallest normal (2^-20 < 2^-14) gives the same result as the oracle's exact product.
    The softmax scale compensates, so the scores stay those of N(0,1) data."""
    w = W.scaled(W.HELIX_KVP8_FP8_1M, B=2, Tq=Tq, S=2048, n_split=2, seed=1700 + q_exp + Tq,
                 softmax_scale=2.0 ** -q_exp / np.sqrt(128.0))
    inp = W.make_inputs(w, DEV)
    inp["q"] = (inp["q"].float() * 2.0 ** q_exp).to(torch.bfloat16)  # a power of two: exact in bf16
    assert inp["q"].float().abs().max().item() > (65504.0 if q_exp > 0 else 0.0)
    _run_all_paths(w, inp)
