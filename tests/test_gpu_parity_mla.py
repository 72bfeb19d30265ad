"""GPU parity of the MLA latent-cache variant (Hkv = 1, key = 576-dim latent+rope row,
value = its first 512 dims, 128 query heads) against the fp64 oracle.
Bars: bf16 out max-abs <= 1e-2, lse <= 1e-3."""

import numpy as np
import pytest
import torch

import mla_decode_attention_gqa_gb300 as skv
from mla_decode_attention_gqa_gb300 import workloads as W
import oracle
from tests import oracle_io as io

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _all_paths(w, inp, bounds=None):
    bounds = inp["split_bounds"] if bounds is None else bounds
    kw = dict(softmax_scale=w.scale)
    o_p, l_p = skv.attn_partial(inp["q"], inp["k"], inp["v"], inp["seq_lens"], bounds, w.causal_offset, **kw)
    o_m, l_m = skv.attn_merge_lse(o_p, l_p)
    o_f, l_f = skv.gqa_decode_attn(inp["q"], inp["k"], inp["v"], inp["seq_lens"], bounds, w.causal_offset, **kw)
    torch.cuda.synchronize()
    assert skv.device_error() == 0
    ro_p, rl_p = io.oracle_all(inp, w, bounds)
    ro, rl = oracle.merge_lse(ro_p, rl_p)
    io.assert_close(o_p, l_p, ro_p, rl_p, io.TOL_BF16, "partials")
    io.assert_close(o_m, l_m, ro, rl, io.TOL_BF16, "merged")
    io.assert_close(o_f, l_f, ro, rl, io.TOL_BF16, "fused")


def test_mla_absorbed_small_s():
    w = W.scaled(W.MLA_ABSORBED, B=2, S=2048)
    _all_paths(w, W.make_inputs(w, DEV))


def test_mla_ragged_tail_and_odd_splits():
    w = W.scaled(W.MLA_ABSORBED, B=2, S=1000, n_split=3)
    inp = W.make_inputs(w, DEV)
    _all_paths(w, inp, bounds=[[0, 333, 334, 1000], [17, 500, 900, 990]])


def test_mla_fewer_heads_partial_row_tile():
    # 96 heads: the second 64-head tile of each item is half empty
    w = W.scaled(W.MLA_ABSORBED, B=1, Hq=96, S=640, n_split=2)
    _all_paths(w, W.make_inputs(w, DEV))


def test_mla_ragged_lengths_with_nan_past_the_end():
    w = W.scaled(W.MLA_ABSORBED, B=3, S=1500, ragged=True)
    inp = W.make_inputs(w, DEV)
    assert min(inp["seq_lens_host"]) < w.S
    _all_paths(w, inp)


def test_mla_strided_latent_view():
    """The latent as a view into a NaN-filled buffer with padded token rows (640 elements)
    and 64 spare rows per sequence: the tensor maps (the chunked view that lands a whole score
    group or value tile in one copy included) and the L2 prefetch address rows by the cache's
    own strides, so a read outside the view would put NaN into the output."""
    w = W.scaled(W.MLA_ABSORBED, B=2, S=1024, n_split=2)
    inp = W.make_inputs(w, DEV)
    big = torch.full((w.B, 1, w.S + 64, 640), float("nan"), dtype=torch.bfloat16, device=DEV)
    big[:, :, :w.S, :576] = inp["k"]
    view = big[:, :, :w.S, :576]
    assert not view.is_contiguous()
    _all_paths(w, dict(inp, k=view, v=view[..., :512]))


@pytest.mark.slow
def test_mla_absorbed_full_size_sampled():
    w = W.MLA_ABSORBED  # B=16, Hq=128, latent 576 (V 512), S=32768, 4 splits
    inp = W.make_inputs(w, DEV)
    out, lse = skv.gqa_decode_attn(inp["q"], inp["k"], inp["v"], inp["seq_lens"], inp["split_bounds"],
                                   softmax_scale=w.scale)
    torch.cuda.synchronize()
    assert skv.device_error() == 0
    worst = 0.0
    for b in range(w.B):  # every sequence (the chunk planner spreads them over waves)
        ro_p, rl_p = io.oracle_rows(inp, w, b, 0, [0])
        ro, rl = oracle.merge_lse(ro_p, rl_p)
        io.assert_close(out[b, [0]], lse[b, [0]], ro, rl, io.TOL_BF16, f"b={b}")
        rel = io.rel_rms_err(out[b, [0]], ro)
        worst = max(worst, rel)
        assert rel <= io.REL_RMS_BAR, f"b={b}: err / RMS {rel:.3e} > {io.REL_RMS_BAR}"
    print(f"{w.name}: {w.B} sequences checked, largest err / RMS(out) {worst:.3e}")


def test_mla_64_heads_half_row_tile():
    """64 heads: the 128-row tensor-core tile is half empty."""
    w = W.scaled(W.MLA_ABSORBED, B=2, Hq=64, S=700, n_split=2)
    _all_paths(w, W.make_inputs(w, DEV))


def test_mla_two_query_rows_causal():
    """Two query rows per sequence (two 128-row tiles), causal by position."""
    w = W.Workload("mla_tq2", B=2, Tq=2, Hq=128, Hkv=1, dk=576, dv=512, S=500, n_split=3, mla=True,
                   softmax_scale=W.MLA_ABSORBED.softmax_scale, causal_offset=300, seed=1013)
    _all_paths(w, W.make_inputs(w, DEV))


def test_mla_single_split_chunked_long():
    """One long split that the planner cuts into chunks to fill the GPU."""
    w = W.scaled(W.MLA_ABSORBED, B=1, S=9000, n_split=1)
    _all_paths(w, W.make_inputs(w, DEV))


def _shard_bounds(B, S, seed):
    """[B][3] bounds: a random range per sequence (every 7th empty, every 11th one token),
    cut at a random point."""
    rng = np.random.default_rng(seed)
    rows = []
    for b in range(B):
        a = int(rng.integers(0, S + 1))
        c = int(rng.integers(a, S + 1))
        if b % 7 == 0:
            c = a
        if b % 11 == 0:
            c = min(a + 1, S)
        rows.append([a, int(rng.integers(a, c + 1)), c])
    return rows


def test_mla_many_ragged_sequences():
    """160 short sequences whose ranges are empty, one token long or start off a tile
    boundary, with lengths that stop short of the bounds."""
    w = W.Workload("mla_many", B=160, Tq=1, Hq=128, Hkv=1, dk=576, dv=512, S=640, n_split=2, mla=True,
                   softmax_scale=W.MLA_ABSORBED.softmax_scale, ragged=True, seed=1014)
    inp = W.make_inputs(w, DEV)
    _all_paths(w, inp, bounds=_shard_bounds(w.B, w.S, 1014))


def test_mla_six_hundred_sequences():
    """600 two-tile sequences: 600 cluster pairs, eight waves of them."""
    w = W.Workload("mla_b600", B=600, Tq=1, Hq=128, Hkv=1, dk=576, dv=512, S=128, n_split=1, mla=True,
                   softmax_scale=W.MLA_ABSORBED.softmax_scale, ragged=True, seed=1015)
    _all_paths(w, W.make_inputs(w, DEV))
