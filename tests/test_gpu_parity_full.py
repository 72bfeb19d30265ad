"""GPU parity at the workloads' full sizes: every (batch, KV head) group of the decode
workloads and every KV head of the prefill chunk, at sampled query rows, computed by the
oracle one group at a time, in the launch configuration bench.py times (the fused
gqa_decode_attn call) and through attn_partial + attn_merge_lse.  Bars as in
test_gpu_parity_gqa.py, plus one on the largest merged-output error relative to the
outputs' RMS (oracle_io.REL_RMS_BAR).  Each test prints the oracle's host time."""

import time

import numpy as np
import pytest
import torch

import mla_decode_attention_gqa_gb300 as skv
from mla_decode_attention_gqa_gb300 import workloads as W
import oracle
from tests import oracle_io as io

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

DEV = "cuda:0"


def _all_groups(w):
    return [(b, g) for b in range(w.B) for g in range(w.Hkv)]


def _check_groups(w, inp, out, lse, groups, t_rows, parts=None):
    tol = io.tol_for(w)
    G = w.Hq // w.Hkv
    t0 = time.perf_counter()
    worst = 0.0
    for b, g in groups:
        ro_p, rl_p = io.oracle_rows(inp, w, b, g, t_rows)
        ro, rl = oracle.merge_lse(ro_p, rl_p)
        got_o = out[b, t_rows, g * G : (g + 1) * G]
        got_l = lse[b, t_rows, g * G : (g + 1) * G]
        io.assert_close(got_o, got_l, ro, rl, tol, f"merged b={b} g={g}")
        rel = io.rel_rms_err(got_o, ro)
        worst = max(worst, rel)
        assert rel <= io.REL_RMS_BAR, f"merged b={b} g={g}: err / RMS {rel:.3e} > {io.REL_RMS_BAR}"
        if parts is not None:
            po, pl = parts
            io.assert_close(po[:, b, t_rows, g * G : (g + 1) * G], pl[:, b, t_rows, g * G : (g + 1) * G], ro_p, rl_p,
                            tol, f"partials b={b} g={g}")
    print(f"{w.name}: {len(groups)} groups x {len(t_rows)} row(s) checked, largest err / RMS(out) {worst:.3e}, "
          f"oracle host time {time.perf_counter() - t0:.1f} s")


def test_helix_dense_decode_full_size():
    w = W.HELIX_DENSE_128K  # B=8 Hq=128 Hkv=8 d=128 S=131072 bf16
    inp = W.make_inputs(w, DEV)
    out, lse = skv.gqa_decode_attn(inp["q"], inp["k"], inp["v"], inp["seq_lens"], inp["split_bounds"],
                                   softmax_scale=w.scale)
    torch.cuda.synchronize()
    assert skv.device_error() == 0
    _check_groups(w, inp, out, lse, _all_groups(w), [0])


def test_helix_kvp8_fp8_full_size():
    w = W.HELIX_KVP8_FP8_1M  # fp8, S=2^20, 8 shards, ragged
    inp = W.make_inputs(w, DEV)
    kw = dict(k_scale=inp["k_scale"], v_scale=inp["v_scale"], softmax_scale=w.scale, scale_block=w.scale_block)
    out, lse = skv.gqa_decode_attn(inp["q"], inp["k"], inp["v"], inp["seq_lens"], inp["split_bounds"], **kw)
    po, pl = skv.attn_partial(inp["q"], inp["k"], inp["v"], inp["seq_lens"], inp["split_bounds"], **kw)
    mo, ml = skv.attn_merge_lse(po, pl)
    torch.cuda.synchronize()
    assert skv.device_error() == 0
    assert (mo.float() - out.float()).abs().max().item() <= 1e-2
    _check_groups(w, inp, out, lse, _all_groups(w), [0], parts=(po, pl))


def test_ring_prefill_full_size_sampled_rows():
    w = W.RING_PREFILL  # Tq=4096 over 8 x 4096 KV, causal on the diagonal
    inp = W.make_inputs(w, DEV)
    out, lse = skv.gqa_decode_attn(inp["q"], inp["k"], inp["v"], inp["seq_lens"], inp["split_bounds"],
                                   w.causal_offset, softmax_scale=w.scale)
    # the eight ring steps' own partials too (2 GiB of fp32), compared split by split
    po, pl = skv.attn_partial(inp["q"], inp["k"], inp["v"], inp["seq_lens"], inp["split_bounds"], w.causal_offset,
                              softmax_scale=w.scale)
    torch.cuda.synchronize()
    assert skv.device_error() == 0
    rows = [0, 1, 63, 64, 2047, 4094, 4095]
    _check_groups(w, inp, out, lse, _all_groups(w), rows, parts=(po, pl))
