"""GPU test of gqa_decode_attn_noalloc, the fused decode entry point that allocates nothing.

Who needs it: callers that may not allocate device memory or pass a workspace -- for
example a plugin inside a host runtime that owns all device allocations, a latency-critical
path that cannot afford an allocation's possible device-wide synchronisation, or a
foreign-language caller that reaches the library only through its C ABI.  The entry point
keeps its partials in a fixed 32 MiB scratch array compiled into the library.

The test calls it through the C ABI twice in a row (with different inputs, so the second
call cannot pass by reusing the first call's scratch contents) and compares each result
with the regular gqa_decode_attn (caller workspace) at the parity tolerance of the GPU
tests (bf16 KV: out 1e-2, lse 1e-3).  It also checks that a problem too large for the
scratch is refused before anything is launched.  This file is named so that pytest runs it
last.
"""

import ctypes

import pytest
import torch

import mla_decode_attention_gqa_gb300 as skv
from mla_decode_attention_gqa_gb300 import workloads as W

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _noalloc_fn():
    lib = skv.load_library()
    f = lib.gqa_decode_attn_noalloc
    P = ctypes.c_void_p
    f.argtypes = [ctypes.POINTER(skv.SkvDesc), P, P, P, P, P, P, ctypes.POINTER(ctypes.c_int32), ctypes.c_int32,
                  ctypes.c_int64, P, P, P]
    f.restype = ctypes.c_int32
    return f


def _call_noalloc(w, inp):
    f = _noalloc_fn()
    d = skv.make_desc(inp["q"], inp["k"], inp["v"], w.scale, w.scale_block)
    rows = inp["split_bounds"]
    flat = (ctypes.c_int32 * (len(rows) * len(rows[0])))(*[x for r in rows for x in r])
    out = torch.empty((w.B, w.Tq, w.Hq, w.dv), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((w.B, w.Tq, w.Hq), dtype=torch.float32, device=DEV)
    ptr = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    st = f(ctypes.byref(d), ptr(inp["q"]), ptr(inp["k"]), ptr(inp["v"]), ptr(inp["k_scale"]), ptr(inp["v_scale"]),
           ptr(inp["seq_lens"]), flat, len(rows[0]) - 1, int(w.causal_offset), ptr(out), ptr(lse),
           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, out, lse


@pytest.mark.parametrize("seeds", [(501, 502)])
def test_noalloc_matches_workspace_entry_point_twice(seeds):
    for seed in seeds:
        w = W.scaled(W.HELIX_DENSE_128K, B=2, S=6000, n_split=3, seed=seed)
        inp = W.make_inputs(w, DEV)
        st, out, lse = _call_noalloc(w, inp)
        assert st == skv.SKV_OK, skv.last_error()
        ref_o, ref_l = skv.gqa_decode_attn(inp["q"], inp["k"], inp["v"], inp["seq_lens"], inp["split_bounds"],
                                           softmax_scale=w.scale)
        torch.cuda.synchronize()
        assert skv.device_error() == 0
        assert (out.float() - ref_o.float()).abs().max().item() <= 1e-2
        assert (lse - ref_l).abs().max().item() <= 1e-3


def test_noalloc_refuses_problems_larger_than_its_scratch():
    # 64 sequences x 4 rows x 64 heads x 129 floats x many parts: far above 32 MiB of partials
    w = W.Workload("too_big", B=64, Tq=4, Hq=64, Hkv=4, dk=128, dv=128, S=64, n_split=30, seed=503)
    q = torch.zeros((w.B, w.Tq, w.Hq, w.dk), dtype=torch.bfloat16, device=DEV)
    k = torch.zeros((w.B, w.Hkv, w.S, w.dk), dtype=torch.bfloat16, device=DEV)
    inp = {"q": q, "k": k, "v": k, "k_scale": None, "v_scale": None,
           "seq_lens": torch.full((w.B,), w.S, dtype=torch.int32, device=DEV), "split_bounds": w.split_bounds()}
    st, _, _ = _call_noalloc(w, inp)
    assert st == skv.SKV_EWORKSPACE
    assert "built-in scratch" in skv.last_error()
