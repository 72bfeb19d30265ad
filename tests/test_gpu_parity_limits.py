"""GPU parity at the boundary's size limits: a call whose split-bounds table has exactly the
2048 entries the kernels take by value (B * (n_split + 1) = 2048), on each kernel family,
and a pass-Q call with the largest rank x request count (n_ranks * B = 1024).  Every case
is checked against the fp64 oracle at the bars of test_gpu_parity_gqa.py."""

import numpy as np
import pytest
import torch

import mla_decode_attention_gqa_gb300 as skv
from mla_decode_attention_gqa_gb300 import workloads as W
import oracle
from tests import oracle_io as io

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _ragged_bounds(B, n_split, S, seed):
    """[B][n_split + 1] non-decreasing bounds over [0, S] with empty and one-token splits."""
    rng = np.random.default_rng(seed)
    rows = []
    for _ in range(B):
        cuts = np.sort(rng.integers(0, S + 1, n_split - 1))
        rows.append([0] + [int(c) for c in cuts] + [S])
    return rows


def _check_split_call(w, bounds):
    inp = W.make_inputs(w, DEV)
    kw = dict(k_scale=inp["k_scale"], v_scale=inp["v_scale"], softmax_scale=w.scale, scale_block=w.scale_block)
    po, pl = skv.attn_partial(inp["q"], inp["k"], inp["v"], inp["seq_lens"], bounds, w.causal_offset, **kw)
    out, lse = skv.gqa_decode_attn(inp["q"], inp["k"], inp["v"], inp["seq_lens"], bounds, w.causal_offset, **kw)
    torch.cuda.synchronize()
    assert skv.device_error() == 0
    ro_p, rl_p = io.oracle_all(inp, w, bounds=bounds)
    ro, rl = oracle.merge_lse(ro_p, rl_p)
    tol = io.tol_for(w)
    io.assert_close(po, pl, ro_p, rl_p, tol, "partials")
    io.assert_close(out, lse, ro, rl, tol, "merged")


def test_gqa_decode_2048_bound_entries():
    """B = 128 sequences x 15 splits (16 bounds each): many empty and one-token splits."""
    w = W.Workload("lim_gqa", B=128, Tq=1, Hq=8, Hkv=2, dk=64, dv=64, S=480, n_split=15, ragged=True, seed=601)
    assert w.B * (w.n_split + 1) == 2048
    _check_split_call(w, _ragged_bounds(w.B, w.n_split, w.S, 601))


def test_fp8_decode_2048_bound_entries():
    w = W.Workload("lim_fp8", B=64, Tq=1, Hq=16, Hkv=1, dk=128, dv=128, S=768, n_split=31, ragged=True,
                   kv_dtype="fp8_e4m3", seed=602)
    assert w.B * (w.n_split + 1) == 2048
    _check_split_call(w, _ragged_bounds(w.B, w.n_split, w.S, 602))


def test_tensor_core_chunk_2048_bound_entries():
    """The tcgen05 prefill path (128 rows per KV head) with 127 splits per sequence."""
    w = W.Workload("lim_tc", B=16, Tq=128, Hq=16, Hkv=1, dk=128, dv=128, S=1024, n_split=127,
                   causal_offset=1024 - 128, seed=603)
    assert w.B * (w.n_split + 1) == 2048
    _check_split_call(w, _ragged_bounds(w.B, w.n_split, w.S, 603))


def test_mla_pair_2048_bound_entries():
    """The MLA cluster pair with 63 splits per sequence (most shorter than a tile)."""
    w = W.Workload("lim_mla", B=32, Tq=1, Hq=128, Hkv=1, dk=576, dv=512, S=1024, n_split=63, mla=True,
                   softmax_scale=W.MLA_ABSORBED.softmax_scale, ragged=True, seed=604)
    assert w.B * (w.n_split + 1) == 2048
    _check_split_call(w, _ragged_bounds(w.B, w.n_split, w.S, 604))


def test_passq_1024_rank_request_rows():
    """Pass-Q with 8 ranks x 128 requests (16 queries owned per rank)."""
    w = W.Workload("lim_pq", B=128, Tq=1, Hq=16, Hkv=1, dk=128, dv=128, S=256, ragged=True, passq_ranks=8,
                   passq_decode_tokens=16, seed=605)
    assert w.passq_ranks * w.B == 1024
    inp = W.make_inputs(w, DEV)
    out, lse = skv.gqa_decode_attn_passq(inp["q"], inp["k_shards"], inp["v_shards"], inp["shard_lens"],
                                         softmax_scale=w.scale)
    torch.cuda.synchronize()
    assert skv.device_error() == 0
    G = w.Hq // w.Hkv
    for b in range(w.B):
        ro, rl = io.oracle_passq(inp, w, b, 0)
        io.assert_close(out[b, :, :G], lse[b, :, :G], ro, rl, io.TOL_BF16, f"b={b}")


def test_one_past_the_limit_is_refused():
    w = W.Workload("lim_over", B=128, Tq=1, Hq=8, Hkv=2, dk=64, dv=64, S=256, n_split=16, seed=606)
    inp = W.make_inputs(w, DEV)
    with pytest.raises(skv.SplitKVError):
        skv.gqa_decode_attn(inp["q"], inp["k"], inp["v"], inp["seq_lens"], w.split_bounds(), softmax_scale=w.scale)
