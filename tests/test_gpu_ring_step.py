"""GPU parity of attn_ring_step: a pass-KV ring ("Context Parallelism for Scalable
Million-Token Inference", section "Pass-KV keeps queries local and circulates keys and
values") emulated step by step, every KV block in its own buffer, merged in place into a
running (o, lse).  The result must equal the oracle's unsplit causal attention of the
local query chunk over all blocks (fp32 output: the bare 1e-2 / 1e-3 bar)."""

import numpy as np
import pytest
import torch

import mla_decode_attention_gqa_gb300 as skv
from mla_decode_attention_gqa_gb300 import workloads as W
import oracle
from tests import oracle_io as io

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _ring(w, inp, n_blocks, order, first_q_block):
    """Run the ring over blocks in `order`; the query chunk is block `first_q_block`."""
    C = w.S // n_blocks
    B = w.B
    o_acc = torch.empty((B, w.Tq, w.Hq, w.dv), dtype=torch.float32, device=DEV)
    lse_acc = torch.empty((B, w.Tq, w.Hq), dtype=torch.float32, device=DEV)
    q_start = first_q_block * C
    for step, j in enumerate(order):
        kb = inp["k"][:, :, j * C:(j + 1) * C].contiguous()  # the received block, its own buffer
        vb = inp["v"][:, :, j * C:(j + 1) * C].contiguous()
        ks = vs = None
        if inp["k_scale"] is not None:
            per = C // w.scale_block
            ks = inp["k_scale"][:, :, j * per:(j + 1) * per].contiguous()
            vs = inp["v_scale"][:, :, j * per:(j + 1) * per].contiguous()
        seq = torch.clamp(inp["seq_lens"] - j * C, 0, C).to(torch.int32)
        off = q_start - j * C if w.causal_offset != W.NO_CAUSAL else W.NO_CAUSAL
        skv.attn_ring_step(inp["q"], kb, vb, seq, o_acc, lse_acc, off, first=(step == 0), k_scale=ks, v_scale=vs,
                           softmax_scale=w.scale, scale_block=w.scale_block)
    torch.cuda.synchronize()
    assert skv.device_error() == 0
    return o_acc, lse_acc


def _oracle(inp, w, causal):
    ro, rl = oracle.full_attention(io.q_f64(inp["q"]), np.stack([np.stack([io.kv_f64(inp, w, "k", b, g)
                                                                           for g in range(w.Hkv)]) for b in range(w.B)]),
                                   np.stack([np.stack([io.kv_f64(inp, w, "v", b, g) for g in range(w.Hkv)])
                                             for b in range(w.B)]), inp["seq_lens_host"], causal, w.scale)
    return ro, rl


@pytest.mark.parametrize("order", [[0, 1, 2, 3], [3, 0, 2, 1]])
def test_prefill_ring_tensor_core(order):
    """The last of 4 chunks (512 rows x 16 heads per KV head) against all 4 blocks."""
    w = W.Workload("ring_tc", B=1, Tq=512, Hq=32, Hkv=2, dk=128, dv=128, S=4 * 512, causal_offset=3 * 512, seed=500)
    inp = W.make_inputs(w, DEV)
    o, l = _ring(w, inp, 4, order, 3)
    ro, rl = _oracle(inp, w, w.causal_offset)
    io.assert_close(o, l, ro, rl, io.TOL_BF16, "ring")


def test_prefill_ring_middle_chunk_has_invisible_blocks():
    """Query chunk 1 of 4: blocks 2 and 3 are entirely in its future (lse = -inf partials)."""
    w = W.Workload("ring_mid", B=2, Tq=256, Hq=16, Hkv=1, dk=128, dv=128, S=4 * 256, causal_offset=256, seed=501)
    inp = W.make_inputs(w, DEV)
    o, l = _ring(w, inp, 4, [1, 2, 3, 0], 1)
    ro, rl = _oracle(inp, w, w.causal_offset)
    io.assert_close(o, l, ro, rl, io.TOL_BF16, "ring middle")


def test_decode_ring_ragged_with_empty_blocks():
    """Decode (one row per sequence), ragged lengths: later blocks are empty for short sequences."""
    w = W.Workload("ring_dec", B=4, Tq=1, Hq=32, Hkv=4, dk=128, dv=128, S=4 * 1024, ragged=True, seed=502)
    inp = W.make_inputs(w, DEV)
    inp["seq_lens"][0] = 700  # blocks 1..3 empty for sequence 0
    inp["seq_lens_host"][0] = 700
    o, l = _ring(w, inp, 4, [2, 0, 3, 1], 0)
    ro, rl = _oracle(inp, w, W.NO_CAUSAL)
    io.assert_close(o, l, ro, rl, io.TOL_BF16, "ring decode")


def test_fp8_decode_ring():
    w = W.Workload("ring_fp8", B=2, Tq=1, Hq=16, Hkv=2, dk=128, dv=128, S=4 * 512, kv_dtype="fp8_e4m3", seed=503)
    inp = W.make_inputs(w, DEV)
    o, l = _ring(w, inp, 4, [1, 3, 0, 2], 0)
    ro, rl = _oracle(inp, w, W.NO_CAUSAL)
    io.assert_close(o, l, ro, rl, io.TOL_FP8, "ring fp8")


@pytest.mark.slow
def test_full_size_ring_steps_sampled_rows():
    """The ring-step workload bench.py times, at full size (8 steps of 4096-token blocks for
    the last 4096-query chunk): equal to the single fused call over the same cache within
    the bar, and sampled rows (edges of the diagonal block included) against the oracle."""
    w = W.RING_PREFILL_STEPS
    inp = W.make_inputs(w, DEV)
    o_acc, lse_acc = _ring(w, inp, w.n_split, list(range(w.n_split)), w.n_split - 1)
    out, lse = skv.gqa_decode_attn(inp["q"], inp["k"], inp["v"], inp["seq_lens"], inp["split_bounds"],
                                   w.causal_offset, softmax_scale=w.scale)
    torch.cuda.synchronize()
    assert skv.device_error() == 0
    # the fused call's output is a bf16 value v: its rounding is at most half an ulp of v,
    # at most 2^-8 |v|, on top of the bar
    ref = out.float()
    assert torch.all((o_acc - ref).abs() <= io.TOL_BF16["out"] + 2.0 ** -8 * ref.abs())
    assert (lse_acc - lse).abs().max().item() <= io.TOL_BF16["lse"]
    G = w.Hq // w.Hkv
    rows = [0, 1, 127, 128, 2047, 4094, 4095]
    for g in (0, 7):
        ro_p, rl_p = io.oracle_rows(inp, w, 0, g, rows)
        ro, rl = oracle.merge_lse(ro_p, rl_p)
        io.assert_close(o_acc[0, rows, g * G:(g + 1) * G], lse_acc[0, rows, g * G:(g + 1) * G], ro, rl, io.TOL_BF16,
                        f"g={g}")
