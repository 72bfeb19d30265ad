"""GPU parity of the tensor-core (tcgen05) attention path: bf16 KV, dk = dv = 128 and at
least 128 (query row, head) rows per KV head -- the ring pass-KV prefill chunk shape.
Checked element by element against the fp64 oracle (out max-abs <= 1e-2, lse <= 1e-3),
both as per-split partials (attn_partial) and fused over all splits (gqa_decode_attn)."""

import pytest
import torch

import mla_decode_attention_gqa_gb300 as skv
from mla_decode_attention_gqa_gb300 import workloads as W
import oracle
from tests import oracle_io as io

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _check(w, inp, bounds=None, causal=None):
    bounds = inp["split_bounds"] if bounds is None else bounds
    causal = w.causal_offset if causal is None else causal
    o_p, l_p = skv.attn_partial(inp["q"], inp["k"], inp["v"], inp["seq_lens"], bounds, causal, softmax_scale=w.scale)
    o_f, l_f = skv.gqa_decode_attn(inp["q"], inp["k"], inp["v"], inp["seq_lens"], bounds, causal,
                                   softmax_scale=w.scale)
    torch.cuda.synchronize()
    assert skv.device_error() == 0
    ro_p, rl_p = io.oracle_all(inp, w, bounds, causal)
    ro, rl = oracle.merge_lse(ro_p, rl_p)
    io.assert_close(o_p, l_p, ro_p, rl_p, io.TOL_BF16, "partials")
    io.assert_close(o_f, l_f, ro, rl, io.TOL_BF16, "fused")


@pytest.mark.parametrize("Hq,Hkv", [(16, 1), (32, 2), (8, 8), (16, 4), (128, 1)])
def test_group_sizes(Hq, Hkv):
    """G = 16, 16, 1, 4, 128 query heads per KV head; ragged number of rows per tile."""
    w = W.Workload("tc_groups", B=2, Tq=40, Hq=Hq, Hkv=Hkv, dk=128, dv=128, S=700, n_split=3, seed=90 + Hq + Hkv)
    _check(w, W.make_inputs(w, DEV))


def test_causal_offset_zero_dense_lower_triangle():
    w = W.Workload("tc_causal0", B=1, Tq=300, Hq=4, Hkv=1, dk=128, dv=128, S=300, n_split=2, causal_offset=0, seed=95)
    _check(w, W.make_inputs(w, DEV))


def test_ring_chunk_last_of_four():
    w = W.scaled(W.RING_PREFILL, Tq=128, S=4 * 128, n_split=4, Hq=64, Hkv=4)
    _check(w, W.make_inputs(w, DEV))


def test_edges_empty_splits_zero_length_negative_offset():
    w = W.Workload("tc_edges", B=3, Tq=20, Hq=32, Hkv=4, dk=128, dv=128, S=400, n_split=4, seed=96)
    inp = W.make_inputs(w, DEV)
    inp["seq_lens"] = torch.tensor([0, 150, 400], dtype=torch.int32, device=DEV)
    inp["seq_lens_host"] = [0, 150, 400]
    bounds = [[0, 0, 64, 200, 400], [0, 100, 100, 149, 400], [10, 11, 12, 13, 399]]
    _check(w, inp, bounds=bounds)
    _check(w, inp, bounds=bounds, causal=-3)  # first rows see nothing


def test_nan_outside_the_range_is_never_read():
    w = W.Workload("tc_nan", B=1, Tq=16, Hq=16, Hkv=1, dk=128, dv=128, S=640, n_split=1, seed=97)
    inp = W.make_inputs(w, DEV)
    bounds = [[100, 500]]
    for t in (inp["k"], inp["v"]):
        t[:, :, :100] = float("nan")
        t[:, :, 500:] = float("nan")
    _check(w, inp, bounds=bounds)


def test_ragged_lengths_with_nan_past_the_end():
    w = W.Workload("tc_ragged", B=3, Tq=24, Hq=32, Hkv=2, dk=128, dv=128, S=1000, n_split=2, ragged=True, seed=98)
    inp = W.make_inputs(w, DEV)
    assert min(inp["seq_lens_host"]) < w.S
    _check(w, inp)
