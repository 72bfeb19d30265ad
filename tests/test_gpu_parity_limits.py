"""GPU parity at the boundary's limits.  The split-bounds table is a device array that the
host never reads, so batch size and split count are not capped by it:

* B = 512 sequences x 8 splits (4,608 bounds) on the bf16 decode, the fp8 decode and the
  MLA latent paths, with ragged lengths;
* many splits per sequence (most empty or shorter than a tile) on every kernel family;
* pass-Q with 8 ranks x 256 requests and a ring step over 1,100 sequences (both once
  capped at 1,024 rows);
* bound rows the host does not check (decreasing, negative, past the end): each split is
  clipped on the device exactly as the oracle clips it.

Every case is checked against the fp64 oracle at the bars of test_gpu_parity_gqa.py."""

import numpy as np
import pytest
import torch

import mla_decode_attention_gqa_gb300 as skv
from mla_decode_attention_gqa_gb300 import workloads as W
import oracle
from tests import oracle_io as io

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def _ragged_bounds(B, n_split, S, seed):
    """[B][n_split + 1] non-decreasing bounds over [0, S] with empty and one-token splits."""
    rng = np.random.default_rng(seed)
    rows = []
    for _ in range(B):
        cuts = np.sort(rng.integers(0, S + 1, n_split - 1))
        rows.append([0] + [int(c) for c in cuts] + [S])
    return rows


def _check_split_call(w, bounds, fused_too=True):
    inp = W.make_inputs(w, DEV)
    bounds_dev = torch.tensor(bounds, dtype=torch.int32, device=DEV)
    kw = dict(k_scale=inp["k_scale"], v_scale=inp["v_scale"], softmax_scale=w.scale, scale_block=w.scale_block)
    po, pl = skv.attn_partial(inp["q"], inp["k"], inp["v"], inp["seq_lens"], bounds_dev, w.causal_offset, **kw)
    if fused_too:
        out, lse = skv.gqa_decode_attn(inp["q"], inp["k"], inp["v"], inp["seq_lens"], bounds_dev, w.causal_offset,
                                       **kw)
    else:  # the merge of the partials
        out, lse = skv.attn_merge_lse(po, pl)
    torch.cuda.synchronize()
    assert skv.device_error() == 0
    ro_p, rl_p = io.oracle_all(inp, w, bounds=bounds)
    ro, rl = oracle.merge_lse(ro_p, rl_p)
    tol = io.tol_for(w)
    io.assert_close(po, pl, ro_p, rl_p, tol, "partials")
    io.assert_close(out, lse, ro, rl, tol, "merged")


@pytest.mark.parametrize("w", [
    W.Workload("b512_bf16", B=512, Tq=1, Hq=4, Hkv=1, dk=128, dv=128, S=512, n_split=8, ragged=True, seed=611),
    W.Workload("b512_fp8", B=512, Tq=1, Hq=16, Hkv=1, dk=128, dv=128, S=512, n_split=8, ragged=True,
               kv_dtype="fp8_e4m3", seed=612),
    W.Workload("b512_mla", B=512, Tq=1, Hq=16, Hkv=1, dk=576, dv=512, S=256, n_split=8, mla=True,
               softmax_scale=W.MLA_ABSORBED.softmax_scale, ragged=True, seed=613),
], ids=lambda w: w.name)
def test_serving_batch_4608_device_bounds(w):
    """512 sequences x 8 KVP shards: 4,608 bounds in device memory."""
    assert w.B * (w.n_split + 1) == 4608
    _check_split_call(w, w.split_bounds())


def test_gqa_decode_many_ragged_splits():
    """B = 128 sequences x 15 splits: many empty and one-token splits."""
    w = W.Workload("lim_gqa", B=128, Tq=1, Hq=8, Hkv=2, dk=64, dv=64, S=480, n_split=15, ragged=True, seed=601)
    _check_split_call(w, _ragged_bounds(w.B, w.n_split, w.S, 601))


def test_fp8_decode_many_ragged_splits():
    w = W.Workload("lim_fp8", B=64, Tq=1, Hq=16, Hkv=1, dk=128, dv=128, S=768, n_split=31, ragged=True,
                   kv_dtype="fp8_e4m3", seed=602)
    _check_split_call(w, _ragged_bounds(w.B, w.n_split, w.S, 602))


def test_tensor_core_chunk_many_splits():
    """The tcgen05 prefill path (128 rows per KV head) with 127 splits per sequence."""
    w = W.Workload("lim_tc", B=16, Tq=128, Hq=16, Hkv=1, dk=128, dv=128, S=1024, n_split=127,
                   causal_offset=1024 - 128, seed=603)
    _check_split_call(w, _ragged_bounds(w.B, w.n_split, w.S, 603))


def test_mla_pair_many_splits():
    """The MLA cluster pair with 63 splits per sequence (most shorter than a tile)."""
    w = W.Workload("lim_mla", B=32, Tq=1, Hq=128, Hkv=1, dk=576, dv=512, S=1024, n_split=63, mla=True,
                   softmax_scale=W.MLA_ABSORBED.softmax_scale, ragged=True, seed=604)
    _check_split_call(w, _ragged_bounds(w.B, w.n_split, w.S, 604))


@pytest.mark.parametrize("kind", ["bf16", "fp8", "mla"])
def test_bound_rows_the_host_never_checks(kind):
    """Decreasing, negative and past-the-end bounds: every split is clipped to [0, seq_len)
    and a split whose upper bound does not exceed its lower one is empty, on the device as
    in the oracle (partials and their merge)."""
    if kind == "mla":
        w = W.Workload("odd_mla", B=4, Tq=1, Hq=32, Hkv=1, dk=576, dv=512, S=640, n_split=4, mla=True,
                       softmax_scale=W.MLA_ABSORBED.softmax_scale, ragged=True, seed=621)
    else:
        w = W.Workload(f"odd_{kind}", B=4, Tq=1, Hq=16, Hkv=2, dk=128, dv=128, S=640, n_split=4, ragged=True,
                       kv_dtype="fp8_e4m3" if kind == "fp8" else "bf16", seed=622)
    rows = [[-50, 100, 60, 300, 640],     # negative start, a decreasing pair (an empty split)
            [0, 200, 200, 9999, 1 << 30],  # an empty split, bounds past S_max
            [640, 0, 640, 0, 640],        # every other split inverted
            [-7, -3, 10, 10, 65]]         # a negative split, a short tail
    _check_split_call(w, rows, fused_too=False)


def test_passq_2048_rank_request_rows():
    """Pass-Q with 8 ranks x 256 requests (32 queries owned per rank)."""
    w = W.Workload("lim_pq", B=256, Tq=1, Hq=16, Hkv=1, dk=128, dv=128, S=256, ragged=True, passq_ranks=8,
                   passq_decode_tokens=16, seed=605)
    assert w.passq_ranks * w.B == 2048
    inp = W.make_inputs(w, DEV)
    out, lse = skv.gqa_decode_attn_passq(inp["q"], inp["k_shards"], inp["v_shards"], inp["shard_lens"],
                                         softmax_scale=w.scale)
    torch.cuda.synchronize()
    assert skv.device_error() == 0
    G = w.Hq // w.Hkv
    for b in range(w.B):
        ro, rl = io.oracle_passq(inp, w, b, 0)
        io.assert_close(out[b, :, :G], lse[b, :, :G], ro, rl, io.TOL_BF16, f"b={b}")


def test_ring_steps_over_1100_sequences():
    """Two pass-KV ring steps over 1,100 sequences, each block in its own buffer: the running
    output equals the oracle's attention over both blocks."""
    w = W.Workload("ring_b1100", B=1100, Tq=1, Hq=4, Hkv=1, dk=64, dv=64, S=256, n_split=2, ragged=True, seed=631)
    inp = W.make_inputs(w, DEV)
    C = w.S // 2
    o_acc = torch.empty((w.B, 1, w.Hq, w.dv), dtype=torch.float32, device=DEV)
    l_acc = torch.empty((w.B, 1, w.Hq), dtype=torch.float32, device=DEV)
    for j in range(2):
        kb = inp["k"][:, :, j * C:(j + 1) * C].contiguous()
        vb = inp["v"][:, :, j * C:(j + 1) * C].contiguous()
        sl = torch.clamp(inp["seq_lens"] - j * C, 0, C).to(torch.int32)
        skv.attn_ring_step(inp["q"], kb, vb, sl, o_acc, l_acc, first=(j == 0), softmax_scale=w.scale)
    torch.cuda.synchronize()
    assert skv.device_error() == 0
    ro_p, rl_p = io.oracle_all(inp, w)
    ro, rl = oracle.merge_lse(ro_p, rl_p)
    io.assert_close(o_acc, l_acc, ro, rl, io.TOL_BF16, "ring steps")
