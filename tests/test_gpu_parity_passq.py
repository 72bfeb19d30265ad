"""GPU parity of pass-Q decode (gqa_decode_attn_passq): the context-parallel group's ring
of query blocks, the return of the partials to their owners and the merge ("Context
Parallelism for Scalable Million-Token Inference", sections "Pass-Q keeps KV stationary
for cache-heavy turns" and "Pass-Q decode protects capacity but can hurt TTIT"), all
ranks emulated on one GPU.  Every case is checked against the fp64 oracle's attention
over the union of each request's shards, at the bars of test_gpu_parity_gqa.py."""

import numpy as np
import pytest
import torch

import mla_decode_attention_gqa_gb300 as skv
from mla_decode_attention_gqa_gb300 import workloads as W
from tests import oracle_io as io

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _call(w, inp, **kw):
    out, lse = skv.gqa_decode_attn_passq(inp["q"], inp["k_shards"], inp["v_shards"], inp["shard_lens"],
                                         k_scale=inp["k_shard_scale"], v_scale=inp["v_shard_scale"],
                                         softmax_scale=w.scale, scale_block=w.scale_block, **kw)
    torch.cuda.synchronize()
    assert skv.device_error() == 0
    return out, lse


def _check(w, inp, out, lse, pairs=None):
    G = w.Hq // w.Hkv
    tol = io.tol_for(w)
    pairs = [(b, g) for b in range(w.B) for g in range(w.Hkv)] if pairs is None else pairs
    for b, g in pairs:
        ro, rl = io.oracle_passq(inp, w, b, g)
        io.assert_close(out[b, :, g * G:(g + 1) * G], lse[b, :, g * G:(g + 1) * G], ro, rl, tol, f"b={b} g={g}")


def _w(name, **kw):
    base = dict(B=8, Tq=1, Hq=32, Hkv=4, dk=128, dv=128, S=2048, ragged=True, passq_ranks=4,
                passq_decode_tokens=64, seed=500)
    base.update(kw)
    return W.Workload(name, **base)


@pytest.mark.parametrize("w", [
    _w("pq_bf16_d128_n4"),
    _w("pq_bf16_d128_g16", Hq=128, Hkv=8, S=4096, seed=501),  # the bench shape, small
    _w("pq_bf16_d64_n2", B=4, Hq=8, Hkv=2, dk=64, dv=64, S=1024, passq_ranks=2, seed=502),
    _w("pq_bf16_n3", B=6, Hq=16, Hkv=2, passq_ranks=3, seed=503),
    _w("pq_fp8_n4", B=4, Hq=16, Hkv=2, kv_dtype="fp8_e4m3", seed=504),
    _w("pq_fp8_n2", B=6, Hq=32, Hkv=2, kv_dtype="fp8_e4m3", S=3000, passq_ranks=2, seed=505),
], ids=lambda w: w.name)
def test_passq_matches_the_oracle(w):
    inp = W.make_inputs(w, DEV)
    out, lse = _call(w, inp)
    _check(w, inp, out, lse)


def test_single_rank_is_the_plain_decode_bit_for_bit():
    """With one rank the ring is the identity: the same kernels over the same bytes as
    gqa_decode_attn over that rank's shard."""
    w = _w("pq_n1", B=3, passq_ranks=1, seed=510)
    inp = W.make_inputs(w, DEV)
    out, lse = _call(w, inp)
    S_loc = inp["k_shards"].shape[2]
    ref_o, ref_l = skv.gqa_decode_attn(inp["q"], inp["k_shards"], inp["v_shards"], inp["shard_lens"][0].contiguous(),
                                       [[0, S_loc]], softmax_scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), ref_o.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), ref_l.view(torch.int32))
    _check(w, inp, out, lse)


def test_empty_shards_and_a_request_resident_nowhere():
    """Request 0 has no token on any rank (out 0, lse -inf); request 1 lives on the last
    rank only; request 2 on the first only; shorter lengths never read the tokens behind."""
    w = _w("pq_empty", seed=520)
    inp = W.make_inputs(w, DEV)
    lens = inp["shard_lens_host"]
    N = w.passq_ranks
    for r in range(N):
        lens[r][0] = 0
        if r != N - 1:
            lens[r][1] = 0
        if r != 0:
            lens[r][2] = 0
    lens[1][3] = 1  # a single resident token
    inp["shard_lens"] = torch.tensor(lens, dtype=torch.int32, device=DEV)
    out, lse = _call(w, inp)
    assert torch.all(out[0] == 0) and torch.all(torch.isneginf(lse[0]))
    _check(w, inp, out, lse)


def test_caller_workspace_and_outputs():
    w = _w("pq_ws", seed=530)
    inp = W.make_inputs(w, DEV)
    out0, lse0 = _call(w, inp)
    ws = torch.empty(64 << 20, dtype=torch.uint8, device=DEV)
    out = torch.full_like(out0, float("nan"))
    lse = torch.full_like(lse0, float("nan"))
    out1, lse1 = _call(w, inp, out=out, lse=lse, workspace=ws)
    assert out1.data_ptr() == out.data_ptr()
    assert torch.equal(out0.view(torch.int16), out.view(torch.int16)) and torch.equal(lse0, lse)


@pytest.mark.slow
def test_full_size_cp4_sampled():
    """The bench workload (CP4, 8 requests of 64K..128K tokens) in the launch bench.py
    times; the shortest and the longest request, two KV heads each, against the oracle."""
    w = W.PASSQ_DECODE_CP4
    inp = W.make_inputs(w, DEV)
    out, lse = _call(w, inp)
    seq = inp["seq_lens_host"]
    bs = sorted(range(w.B), key=lambda b: seq[b])
    pairs = [(bs[0], 0), (bs[0], 7), (bs[-1], 3), (bs[-1], 4)]
    _check(w, inp, out, lse, pairs)
    G = w.Hq // w.Hkv
    for b, g in pairs:
        ro, _ = io.oracle_passq(inp, w, b, g)
        rel = io.rel_rms_err(out[b, :, g * G:(g + 1) * G], ro)
        print(f"{w.name} b={b} g={g}: max-abs err / RMS(out) = {rel:.3e}")
        assert rel <= io.REL_RMS_BAR, f"b={b} g={g}: err / RMS {rel:.3e} > {io.REL_RMS_BAR}"
    assert torch.isfinite(out.float()).all()
