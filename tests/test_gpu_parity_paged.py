"""GPU parity over a paged block KV cache (pages [num_blocks, Hkv, block_len, d] and a
per-sequence block table; the layout of "Attention DP", section "KV Cache") through
attn_partial_paged / gqa_decode_attn_paged.  Each case is checked against the fp64
oracle and, bit for bit, against the contiguous call on the same logical cache (the
kernels read the same bytes in the same order)."""

import numpy as np
import pytest
import torch

import mla_decode_attention_gqa_gb300 as skv
from mla_decode_attention_gqa_gb300 import workloads as W
import oracle
from tests import oracle_io as io

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _run(w, inp, fn_paged, fn_contig, **extra):
    scales = dict(k_scale=inp.get("k_scale_pages"), v_scale=inp.get("v_scale_pages"))
    common = dict(softmax_scale=w.scale, scale_block=w.scale_block, **extra)
    a = fn_paged(inp["q"], inp["k_pages"], inp["v_pages"], inp["seq_lens"], inp["split_bounds"], inp["block_table"],
                 w.causal_offset, **scales, **common)
    b = fn_contig(inp["q"], inp["k"], inp["v"], inp["seq_lens"], inp["split_bounds"], w.causal_offset,
                  k_scale=inp["k_scale"], v_scale=inp["v_scale"], **common)
    torch.cuda.synchronize()
    assert skv.device_error() == 0
    return a, b


def _bitwise(x, y):
    for s, t in zip(x, y):
        assert torch.equal(s.contiguous().view(torch.int8), t.contiguous().view(torch.int8))


def _check(w, inp=None):
    inp = W.make_inputs(w, DEV) if inp is None else inp
    (o_p, l_p), (c_p, cl_p) = _run(w, inp, skv.attn_partial_paged, skv.attn_partial)
    (o_f, l_f), (c_f, cl_f) = _run(w, inp, skv.gqa_decode_attn_paged, skv.gqa_decode_attn)
    _bitwise((o_p, l_p, o_f, l_f), (c_p, cl_p, c_f, cl_f))
    ro_p, rl_p = io.oracle_all(inp, w)
    ro, rl = oracle.merge_lse(ro_p, rl_p)
    tol = io.tol_for(w)
    io.assert_close(o_p, l_p, ro_p, rl_p, tol, "partials")
    io.assert_close(o_f, l_f, ro, rl, tol, "fused")


@pytest.mark.parametrize("block_len", [64, 128, 512])
def test_decode_bf16_d128_ragged(block_len):
    w = W.Workload("pg_dec", B=3, Tq=1, Hq=32, Hkv=4, dk=128, dv=128, S=2048, n_split=3, ragged=True, paged=True,
                   block_len=block_len, seed=400 + block_len)
    _check(w)


def test_decode_bf16_d64():
    w = W.Workload("pg_d64", B=2, Tq=1, Hq=8, Hkv=2, dk=64, dv=64, S=1024, n_split=4, paged=True, block_len=64,
                   seed=411)
    _check(w)


@pytest.mark.parametrize("block_len", [64, 256])
def test_decode_fp8_page_scales(block_len):
    w = W.Workload("pg_fp8", B=2, Tq=1, Hq=16, Hkv=2, dk=128, dv=128, S=2048, kv_dtype="fp8_e4m3", n_split=2,
                   ragged=True, paged=True, block_len=block_len, seed=420 + block_len)
    _check(w)


@pytest.mark.parametrize("block_len", [64, 256])
def test_tensor_core_prefill_pages(block_len):
    """128-token tiles read as two 64-token halves, possibly from two pages."""
    w = W.Workload("pg_tc", B=2, Tq=64, Hq=32, Hkv=2, dk=128, dv=128, S=1024, n_split=2, causal_offset=1024 - 64,
                   paged=True, block_len=block_len, seed=430 + block_len)
    _check(w)


@pytest.mark.parametrize("Hq", [128, 96])
def test_mla_pages(Hq):
    """Hq=128: the tcgen05 cluster-pair kernel; Hq=96: the mma.sync kernel."""
    w = W.Workload("pg_mla", B=2, Tq=1, Hq=Hq, Hkv=1, dk=576, dv=512, S=1024, n_split=2, mla=True, ragged=True,
                   softmax_scale=W.MLA_ABSORBED.softmax_scale, paged=True, block_len=128, seed=440 + Hq)
    _check(w)


def test_shared_pages_between_sequences():
    """Two sequences whose tables point at the same pages (a shared prefix) give identical
    results for the shared part."""
    w = W.Workload("pg_share", B=2, Tq=1, Hq=16, Hkv=2, dk=128, dv=128, S=512, n_split=1, paged=True, block_len=64,
                   seed=450)
    inp = W.make_inputs(w, DEV)
    inp["block_table"][1] = inp["block_table"][0]  # sequence 1 reads sequence 0's pages
    inp["block_table_host"][1] = list(inp["block_table_host"][0])
    inp["q"][1] = inp["q"][0]
    out, lse = skv.gqa_decode_attn_paged(inp["q"], inp["k_pages"], inp["v_pages"], inp["seq_lens"],
                                         inp["split_bounds"], inp["block_table"], softmax_scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(out[0], out[1]) and torch.equal(lse[0], lse[1])
    # and both equal the oracle over the gathered pages
    kf = oracle.gather_pages(oracle.bf16_bits_to_f64(inp["k_pages"].view(torch.int16).cpu().numpy()),
                             inp["block_table_host"], w.S)
    vf = oracle.gather_pages(oracle.bf16_bits_to_f64(inp["v_pages"].view(torch.int16).cpu().numpy()),
                             inp["block_table_host"], w.S)
    ro, rl = oracle.full_attention(io.q_f64(inp["q"]), kf, vf, [w.S, w.S], w.causal_offset, w.scale)
    io.assert_close(out, lse, ro, rl, io.TOL_BF16, "shared")


@pytest.mark.slow
@pytest.mark.parametrize("w", [W.HELIX_DENSE_128K_PAGED, W.MLA_ABSORBED_PAGED], ids=lambda w: w.name)
def test_full_size_paged_equals_contiguous(w):
    inp = W.make_inputs(w, DEV)
    (o_f, l_f), (c_f, cl_f) = _run(w, inp, skv.gqa_decode_attn_paged, skv.gqa_decode_attn)
    _bitwise((o_f, l_f), (c_f, cl_f))
