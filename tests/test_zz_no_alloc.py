"""GPU tests of gqa_decode_attn_noalloc, the fused decode entry point that allocates nothing.

Who needs it: callers that may not allocate device memory or pass a workspace -- for
example a plugin inside a host runtime that owns all device allocations, a latency-critical
path that cannot afford an allocation's possible device-wide synchronisation, or a
foreign-language caller that reaches the library only through its C ABI.  The entry point
runs the same kernels as gqa_decode_attn: the tensor-core shapes need no scratch at all,
every other shape keeps its partials in a fixed 32 MiB scratch array compiled into the
library.

Each case calls it through the C ABI twice in a row, with different inputs (so the second
call cannot pass by reusing the first call's scratch contents), and checks both results
against the fp64 oracle at the GPU parity tolerances (bf16 KV: out 1e-2, lse 1e-3; fp8:
4e-2), and against the regular gqa_decode_attn (caller workspace).  The cases cover the
bf16 GQA decode, the fp8 KVP shards with ragged lengths, the MLA latent, a tensor-core
shape, and a problem whose regular plan needs more partials than the scratch holds (it
is planned again with fewer chunks and still accepted).  A problem too large even with one
chunk per split is refused before anything is launched.  This file is named so that pytest
runs it last.
"""

import ctypes

import numpy as np
import pytest
import torch

import mla_decode_attention_gqa_gb300 as skv
from mla_decode_attention_gqa_gb300 import workloads as W
from tests.oracle_io import assert_close, oracle_all, oracle_rows, tol_for
import oracle

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
SCRATCH_BYTES = 32 << 20


def _noalloc_fn():
    lib = skv.load_library()
    f = lib.gqa_decode_attn_noalloc
    P = ctypes.c_void_p
    f.argtypes = [ctypes.POINTER(skv.SkvDesc), P, P, P, P, P, P, P, ctypes.c_int32, ctypes.c_int64, P, P, P]
    f.restype = ctypes.c_int32
    return f


def _call_noalloc(w, inp, bounds_dev):
    f = _noalloc_fn()
    d = skv.make_desc(inp["q"], inp["k"], inp["v"], w.scale, w.scale_block)
    out = torch.empty((w.B, w.Tq, w.Hq, w.dv), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((w.B, w.Tq, w.Hq), dtype=torch.float32, device=DEV)
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    st = f(ctypes.byref(d), ptr(inp["q"]), ptr(inp["k"]), ptr(inp["v"]), ptr(inp["k_scale"]), ptr(inp["v_scale"]),
           ptr(inp["seq_lens"]), ptr(bounds_dev), bounds_dev.shape[1] - 1, int(w.causal_offset), ptr(out), ptr(lse),
           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, out, lse


def _regular_ws_bytes(w, inp):
    d = skv.make_desc(inp["q"], inp["k"], inp["v"], w.scale, w.scale_block)
    return skv.gqa_decode_attn_workspace_size(d, w.n_split)


CASES = [
    # bf16 GQA decode, group 16, three splits (partial kernel + merge, partials in the scratch)
    ("bf16_decode", W.scaled(W.HELIX_DENSE_128K, B=2, S=6000, n_split=3), None),
    # fp8 e4m3 KV with 64-token block scales, 8 KVP shards over ragged lengths
    ("fp8_kvp_shards", W.scaled(W.HELIX_KVP8_FP8_1M, B=2, S=8192), None),
    # MLA latent (128 heads, 576/512 dims), four splits: the tensor-core cluster kernel's partials
    ("mla_latent", W.scaled(W.MLA_ABSORBED, B=2, S=4096), None),
    # bf16 d = 128 with 64 x 16 rows per KV head: the fused tensor-core kernel, no scratch
    ("tensor_core_chunk", W.scaled(W.RING_PREFILL, Tq=64, S=1024, n_split=4), None),
    # MLA B = 16, S = 32768, one split: the regular plan cuts it into more chunks than the
    # scratch holds partials for; planned again with fewer chunks (rows 0 of sequences 0, 7, 15)
    ("replanned_mla", W.scaled(W.MLA_ABSORBED, n_split=1), [0, 7, 15]),
]


@pytest.mark.parametrize("name,w,sample_b", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_the_oracle_on_two_calls_in_a_row(name, w, sample_b):
    for call, seed in enumerate((w.seed + 501, w.seed + 502)):
        wc = W.scaled(w, seed=seed)
        inp = W.make_inputs(wc, DEV)
        bounds_dev = torch.tensor(inp["split_bounds"], dtype=torch.int32, device=DEV)
        if name == "replanned_mla":
            assert _regular_ws_bytes(wc, inp) > SCRATCH_BYTES  # the regular plan would not fit
        if name == "tensor_core_chunk":
            assert _regular_ws_bytes(wc, inp) == 0
        st, out, lse = _call_noalloc(wc, inp, bounds_dev)
        assert st == skv.SKV_OK, skv.last_error()
        torch.cuda.synchronize()
        assert skv.device_error() == 0
        # the same problem through the regular entry point (caller workspace)
        ref_o, ref_l = skv.gqa_decode_attn(inp["q"], inp["k"], inp["v"], inp["seq_lens"], bounds_dev,
                                           wc.causal_offset, k_scale=inp["k_scale"], v_scale=inp["v_scale"],
                                           softmax_scale=wc.scale, scale_block=wc.scale_block)
        torch.cuda.synchronize()
        tol = tol_for(wc)
        assert (out.float() - ref_o.float()).abs().max().item() <= tol["out"]
        fin = torch.isfinite(ref_l)
        assert torch.equal(fin, torch.isfinite(lse))
        assert (lse[fin] - ref_l[fin]).abs().max().item() <= tol["lse"]
        # the fp64 oracle on the same bytes
        if sample_b is None:
            o, l = oracle_all(inp, wc)
            mo, ml = oracle.merge_lse(o, l)
            assert_close(out, lse, mo, ml, tol, f"{name} call {call}")
        else:
            for b in sample_b:
                o, l = oracle_rows(inp, wc, b, 0, [0])
                mo, ml = oracle.merge_lse(o, l)
                assert_close(out[b], lse[b], mo, ml, tol, f"{name} call {call} sequence {b}")


def test_noalloc_refuses_problems_larger_than_its_scratch():
    # 64 sequences x 4 rows x 64 heads x 129 floats x 30 splits: far above 32 MiB of partials
    # even with one chunk per split
    w = W.Workload("too_big", B=64, Tq=4, Hq=64, Hkv=4, dk=128, dv=128, S=64, n_split=30, seed=503)
    q = torch.zeros((w.B, w.Tq, w.Hq, w.dk), dtype=torch.bfloat16, device=DEV)
    k = torch.zeros((w.B, w.Hkv, w.S, w.dk), dtype=torch.bfloat16, device=DEV)
    inp = {"q": q, "k": k, "v": k, "k_scale": None, "v_scale": None,
           "seq_lens": torch.full((w.B,), w.S, dtype=torch.int32, device=DEV)}
    bounds_dev = torch.tensor(w.split_bounds(), dtype=torch.int32, device=DEV)
    st, _, _ = _call_noalloc(w, inp, bounds_dev)
    assert st == skv.SKV_EWORKSPACE
    assert "built-in scratch" in skv.last_error()
