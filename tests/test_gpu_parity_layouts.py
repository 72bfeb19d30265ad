"""GPU parity for tokens stored out of sequence order: the zigzag and striped layouts of
"现代大模型推理并行策略总览", section "序列布局：Contiguous、Zigzag 与 Striped", through
attn_partial_pos / gqa_decode_attn_pos (causal rule k_pos[t] <= q_pos[i]).  Element by
element against the fp64 oracle run on the same positions, on the tensor-core prefill
path, the mma.sync prefill and decode paths (bf16 d=64, fp8 d=128) and at full size on
sampled rows."""

import numpy as np
import pytest
import torch

import mla_decode_attention_gqa_gb300 as skv
from mla_decode_attention_gqa_gb300 import workloads as W
import oracle
from tests import oracle_io as io

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _layout(layout, S, cp, rank, **kw):
    base = dict(B=1, Hq=32, Hkv=2, dk=128, dv=128, seed=300 + S + cp + rank)
    base.update(kw)
    return W.Workload(f"{layout}_{S}_{cp}_{rank}", Tq=S // cp, S=S, n_split=cp, layout=layout, cp_rank=rank, **base)


def _check(w, inp):
    kw = dict(k_scale=inp["k_scale"], v_scale=inp["v_scale"], softmax_scale=w.scale, scale_block=w.scale_block)
    o_p, l_p = skv.attn_partial_pos(inp["q"], inp["k"], inp["v"], inp["seq_lens"], inp["split_bounds"], inp["q_pos"],
                                    inp["k_pos"], **kw)
    o_f, l_f = skv.gqa_decode_attn_pos(inp["q"], inp["k"], inp["v"], inp["seq_lens"], inp["split_bounds"],
                                       inp["q_pos"], inp["k_pos"], **kw)
    torch.cuda.synchronize()
    assert skv.device_error() == 0
    ro_p, rl_p = io.oracle_all(inp, w)
    ro, rl = oracle.merge_lse(ro_p, rl_p)
    tol = io.tol_for(w)
    io.assert_close(o_p, l_p, ro_p, rl_p, tol, "partials")
    io.assert_close(o_f, l_f, ro, rl, tol, "fused")


@pytest.mark.parametrize("layout,rank", [("zigzag", 0), ("zigzag", 3), ("striped", 0), ("striped", 2)])
def test_tensor_core_path(layout, rank):
    """bf16 d=128, 16 heads per KV head: the tcgen05 prefill kernel."""
    w = _layout(layout, 4 * 256, 4, rank)
    _check(w, W.make_inputs(w, DEV))


@pytest.mark.parametrize("layout", ["zigzag", "striped"])
def test_mma_sync_prefill_bf16_d64(layout):
    w = _layout(layout, 4 * 128, 4, 1, Hq=8, Hkv=2, dk=64, dv=64)
    _check(w, W.make_inputs(w, DEV))


@pytest.mark.parametrize("layout", ["zigzag", "striped"])
def test_mma_sync_prefill_fp8(layout):
    w = _layout(layout, 4 * 128, 4, 2, Hq=8, Hkv=2, kv_dtype="fp8_e4m3")
    _check(w, W.make_inputs(w, DEV))


def test_decode_single_row_mid_sequence():
    """One query row (Tq=1) at an interior position of a striped KV: later tokens masked."""
    w = W.Workload("pos_decode", B=2, Tq=1, Hq=16, Hkv=2, dk=128, dv=128, S=640, n_split=3, seed=331)
    inp = W.make_inputs(w, DEV)
    k_row = [p for r in range(4) for p in W.layout_positions("striped", 640, 4, r)]
    inp["k_pos_host"] = [list(k_row), list(k_row)]
    inp["q_pos_host"] = [[400], [77]]
    inp["k_pos"] = torch.tensor(inp["k_pos_host"], dtype=torch.int32, device=DEV)
    inp["q_pos"] = torch.tensor(inp["q_pos_host"], dtype=torch.int32, device=DEV)
    _check(w, inp)


def test_contiguous_positions_equal_the_causal_offset_call():
    """Positions i + offset / t reproduce gqa_decode_attn with that causal_offset bit for bit."""
    w = W.scaled(W.RING_PREFILL, Tq=256, S=4 * 256, n_split=4, Hq=32, Hkv=2)
    inp = W.make_inputs(w, DEV)
    q_pos = (w.causal_offset + torch.arange(w.Tq, dtype=torch.int32, device=DEV))[None]
    k_pos = torch.arange(w.S, dtype=torch.int32, device=DEV)[None]
    a_o, a_l = skv.gqa_decode_attn(inp["q"], inp["k"], inp["v"], inp["seq_lens"], inp["split_bounds"],
                                   w.causal_offset, softmax_scale=w.scale)
    b_o, b_l = skv.gqa_decode_attn_pos(inp["q"], inp["k"], inp["v"], inp["seq_lens"], inp["split_bounds"], q_pos,
                                       k_pos, softmax_scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(a_o.view(torch.int16), b_o.view(torch.int16))
    assert torch.equal(a_l.view(torch.int32), b_l.view(torch.int32))


@pytest.mark.slow
@pytest.mark.parametrize("w", [W.RING_PREFILL_ZIGZAG, W.RING_PREFILL_STRIPED], ids=lambda w: w.name)
def test_full_size_ring_chunk_sampled_rows(w):
    """The bench workloads (rank 0's 4096 queries against 8 x 4096 KV): every split fused,
    checked on sampled query rows of both KV heads 0 and 7."""
    inp = W.make_inputs(w, DEV)
    out, lse = skv.gqa_decode_attn_pos(inp["q"], inp["k"], inp["v"], inp["seq_lens"], inp["split_bounds"],
                                       inp["q_pos"], inp["k_pos"], softmax_scale=w.scale)
    torch.cuda.synchronize()
    assert skv.device_error() == 0
    G = w.Hq // w.Hkv
    rows = [0, 1, 2047, 2048, 3000, 4095]
    for g in (0, w.Hkv - 1):
        ro_p, rl_p = io.oracle_rows(inp, w, 0, g, rows)
        ro, rl = oracle.merge_lse(ro_p, rl_p)
        io.assert_close(out[0, rows, g * G:(g + 1) * G], lse[0, rows, g * G:(g + 1) * G], ro, rl, io.TOL_BF16,
                        f"g={g}")
