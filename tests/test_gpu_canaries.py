"""Guard canaries around every output and workspace a call writes (GPU).

A write outside a buffer would otherwise go unseen by the parity tests (it lands in
memory nobody compares), and no memory checker runs here.  So each output tensor, and
each caller workspace, is a view into a larger buffer: GUARD elements on each side hold
a NaN bit pattern that no kernel writes, and the output itself is pre-filled with it.
After the call the guards must be intact (nothing written outside the buffer) and no
output element may still hold the pattern (every element was written).  Workspaces only
need intact guards.  One small case per kernel and mode: GQA decode bf16 and fp8
(partials, merge, fused call), the tensor-core prefill chunk (partials and the fused
in-kernel merge), the MLA cluster pair and its mma.sync fallback, the position-masked
and paged variants, pass-KV ring steps (tensor-core and decode shapes) and pass-Q decode.
"""

import ctypes
import math

import pytest
import torch

import mla_decode_attention_gqa_gb300 as skv
from mla_decode_attention_gqa_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
GUARD = 4096  # elements each side; keeps every view 256-byte aligned

# canary bit patterns (NaN payloads for the float types)
_BITS = {torch.float32: (torch.int32, 0x7FBADBAD), torch.bfloat16: (torch.int16, 0x7FBD),
         torch.uint8: (torch.uint8, 0xA5)}


class Guarded:
    """A tensor of `shape` inside a buffer with GUARD canary elements on each side."""

    def __init__(self, shape, dtype):
        self.n = math.prod(shape)
        self.buf = torch.empty(GUARD + self.n + GUARD, dtype=dtype, device=DEV)
        self.ibits, self.pat = _BITS[dtype]
        self.bits().fill_(self.pat)
        self.t = self.buf[GUARD:GUARD + self.n].view(shape)

    def bits(self):
        return self.buf.view(self.ibits)

    def check(self, name, written=True):
        b = self.bits()
        assert bool((b[:GUARD] == self.pat).all()), f"{name}: write before the buffer"
        assert bool((b[GUARD + self.n:] == self.pat).all()), f"{name}: write past the end of the buffer"
        if written:
            left = int((b[GUARD:GUARD + self.n] == self.pat).sum())
            assert left == 0, f"{name}: {left} element(s) never written"


def _outs(w, n_split=None):
    """Guarded (out bf16, lse fp32) of a merged call, or fp32 partials when n_split is given."""
    if n_split is None:
        return Guarded((w.B, w.Tq, w.Hq, w.dv), torch.bfloat16), Guarded((w.B, w.Tq, w.Hq), torch.float32)
    return (Guarded((n_split, w.B, w.Tq, w.Hq, w.dv), torch.float32),
            Guarded((n_split, w.B, w.Tq, w.Hq), torch.float32))


def _done():
    torch.cuda.synchronize()
    assert skv.device_error() == 0


def _decode_family(w):
    """attn_partial, attn_merge_lse and gqa_decode_attn (with a guarded workspace)."""
    inp = W.make_inputs(w, DEV)
    bounds = inp["split_bounds"]
    n_split = len(bounds[0]) - 1
    kw = dict(k_scale=inp["k_scale"], v_scale=inp["v_scale"], softmax_scale=w.scale, scale_block=w.scale_block)
    op, lp = _outs(w, n_split)
    skv.attn_partial(inp["q"], inp["k"], inp["v"], inp["seq_lens"], bounds, w.causal_offset, out_partial=op.t,
                     lse_partial=lp.t, **kw)
    _done()
    op.check("out_partial")
    lp.check("lse_partial")
    om, lm = _outs(w)
    skv.attn_merge_lse(op.t, lp.t, out=om.t, lse=lm.t)
    _done()
    om.check("merged out")
    lm.check("merged lse")
    d = skv.make_desc(inp["q"], inp["k"], inp["v"], w.scale, w.scale_block)
    nbytes = skv.gqa_decode_attn_workspace_size(d, len(bounds[0]) - 1)
    ws = Guarded((max(nbytes, 1),), torch.uint8)
    of, lf = _outs(w)
    skv.gqa_decode_attn(inp["q"], inp["k"], inp["v"], inp["seq_lens"], bounds, w.causal_offset, out=of.t, lse=lf.t,
                        workspace=ws.t, **kw)
    _done()
    of.check("fused out")
    lf.check("fused lse")
    ws.check("workspace", written=False)


@pytest.mark.parametrize("w", [
    W.scaled(W.HELIX_DENSE_128K, B=3, S=1000, n_split=3, ragged=True),         # gqa_partial, bf16 decode
    W.scaled(W.HELIX_KVP8_FP8_1M, B=2, S=2048),                                # gqa_partial, fp8, 8 shards
    W.scaled(W.RING_PREFILL, Tq=256, S=1024, n_split=4, Hq=32, Hkv=2),          # tc_attn partials / fused
    W.Workload("cn_pre_d64", B=2, Tq=20, Hq=8, Hkv=2, dk=64, dv=64, S=300, n_split=2, seed=700),  # mma.sync prefill
    W.scaled(W.MLA_ABSORBED, B=2, S=1000, n_split=3),                          # mla_tc cluster pair
    W.scaled(W.MLA_ABSORBED, B=1, Hq=96, S=640, n_split=2),                    # mla_partial (96 heads)
], ids=lambda w: w.name + f"_B{w.B}_Tq{w.Tq}_Hq{w.Hq}_S{w.S}")
def test_partial_merge_and_fused_calls_write_only_their_outputs(w):
    _decode_family(w)


def test_position_mode_writes_only_its_outputs():
    w = W.Workload("cn_zigzag", B=1, Tq=128, Hq=32, Hkv=2, dk=128, dv=128, S=1024, n_split=8, layout="zigzag",
                   cp_rank=2, seed=701)
    inp = W.make_inputs(w, DEV)
    op, lp = _outs(w, w.n_split)
    skv.attn_partial_pos(inp["q"], inp["k"], inp["v"], inp["seq_lens"], inp["split_bounds"], inp["q_pos"],
                         inp["k_pos"], softmax_scale=w.scale, out_partial=op.t, lse_partial=lp.t)
    of, lf = _outs(w)
    skv.gqa_decode_attn_pos(inp["q"], inp["k"], inp["v"], inp["seq_lens"], inp["split_bounds"], inp["q_pos"],
                            inp["k_pos"], softmax_scale=w.scale, out=of.t, lse=lf.t)
    _done()
    for g, name in ((op, "out_partial"), (lp, "lse_partial"), (of, "out"), (lf, "lse")):
        g.check(name)


@pytest.mark.parametrize("w", [
    W.Workload("cn_pg_dec", B=3, Tq=1, Hq=32, Hkv=4, dk=128, dv=128, S=1024, n_split=3, ragged=True, paged=True,
               block_len=64, seed=702),
    W.Workload("cn_pg_mla", B=2, Tq=1, Hq=128, Hkv=1, dk=576, dv=512, S=1024, n_split=2, mla=True, ragged=True,
               paged=True, block_len=64, seed=703),
], ids=lambda w: w.name)
def test_paged_calls_write_only_their_outputs(w):
    inp = W.make_inputs(w, DEV)
    kw = dict(k_scale=inp.get("k_scale_pages"), v_scale=inp.get("v_scale_pages"), softmax_scale=w.scale,
              scale_block=w.scale_block)
    op, lp = _outs(w, w.n_split)
    skv.attn_partial_paged(inp["q"], inp["k_pages"], inp["v_pages"], inp["seq_lens"], inp["split_bounds"],
                           inp["block_table"], w.causal_offset, out_partial=op.t, lse_partial=lp.t, **kw)
    of, lf = _outs(w)
    skv.gqa_decode_attn_paged(inp["q"], inp["k_pages"], inp["v_pages"], inp["seq_lens"], inp["split_bounds"],
                              inp["block_table"], w.causal_offset, out=of.t, lse=lf.t, **kw)
    _done()
    for g, name in ((op, "out_partial"), (lp, "lse_partial"), (of, "out"), (lf, "lse")):
        g.check(name)


@pytest.mark.parametrize("w", [
    W.scaled(W.RING_PREFILL, Tq=256, S=1024, n_split=4, Hq=32, Hkv=2),   # tensor core: merge in the epilogue
    W.scaled(W.HELIX_DENSE_128K, B=2, Hq=32, Hkv=4, S=1024, n_split=4),   # decode: partial + two-way merge
], ids=lambda w: f"Tq{w.Tq}")
def test_ring_steps_write_only_the_running_output(w):
    inp = W.make_inputs(w, DEV)
    C = w.S // w.n_split
    o_acc = Guarded((w.B, w.Tq, w.Hq, w.dv), torch.float32)
    l_acc = Guarded((w.B, w.Tq, w.Hq), torch.float32)
    q_start = w.S - w.Tq
    for j in range(w.n_split):
        kb = inp["k"][:, :, j * C:(j + 1) * C].contiguous()
        vb = inp["v"][:, :, j * C:(j + 1) * C].contiguous()
        seq = torch.clamp(inp["seq_lens"] - j * C, 0, C).to(torch.int32)
        off = q_start - j * C if w.causal_offset != W.NO_CAUSAL else W.NO_CAUSAL
        skv.attn_ring_step(inp["q"], kb, vb, seq, o_acc.t, l_acc.t, off, first=(j == 0), softmax_scale=w.scale)
    _done()
    o_acc.check("o_acc")
    l_acc.check("lse_acc")


def test_passq_writes_only_its_outputs_and_workspace():
    w = W.Workload("cn_passq", B=8, Tq=1, Hq=32, Hkv=4, dk=128, dv=128, S=2048, ragged=True, passq_ranks=4,
                   passq_decode_tokens=64, seed=704)
    inp = W.make_inputs(w, DEV)
    B, N = w.B, w.passq_ranks
    d = skv.make_desc(inp["q"], inp["k_shards"][:B], inp["v_shards"][:B], w.scale, w.scale_block)
    n = ctypes.c_size_t(0)
    assert skv.load_library().gqa_decode_attn_passq_workspace_size(ctypes.byref(d), N, ctypes.byref(n)) == 0
    ws = Guarded((max(int(n.value), 1),), torch.uint8)
    of, lf = _outs(w)
    skv.gqa_decode_attn_passq(inp["q"], inp["k_shards"], inp["v_shards"], inp["shard_lens"],
                              k_scale=inp["k_shard_scale"], v_scale=inp["v_shard_scale"], softmax_scale=w.scale,
                              scale_block=w.scale_block, out=of.t, lse=lf.t, workspace=ws.t)
    _done()
    of.check("out")
    lf.check("lse")
    ws.check("workspace", written=False)
