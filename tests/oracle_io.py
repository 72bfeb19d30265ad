"""Test helpers: turn a workload's torch tensors into the oracle's float64 inputs and
compare GPU results with the oracle's.  (Test code: may import the oracle.)"""

import numpy as np
import torch

import oracle

# Parity bars (written in the tests): max-abs error of the output and of the LSE.
TOL_BF16 = {"out": 1e-2, "lse": 1e-3}
TOL_FP8 = {"out": 4e-2, "lse": 4e-2}
# The bars apply to the computed output.  An output stored in bf16 is further rounded to
# nearest, by up to half an ulp (0.0156 for |o| in [4, 8): a weighted mean of a few V rows
# can land there), so a bf16 output element may also differ from the reference by the
# reference's own bf16 rounding |bf16(o_ref) - o_ref|.  Where the GPU's value rounds to the
# other neighbour the two sit on either side of a rounding midpoint within the computation
# error e of each other, so the excess over that allowance is at most 2e: the bar still
# bounds the computation.  fp32 outputs (the partials) are held to the bare bar.


def bf16_round(x):
    """Nearest bfloat16 value of float64 x (ties to even), as float64: 8 significant bits."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)  # x = m * 2^e, 0.5 <= |m| < 1
    return np.ldexp(np.rint(m * 256.0) / 256.0, e)  # np.rint rounds halves to even


def tol_for(w):
    return TOL_FP8 if w.kv_dtype == "fp8_e4m3" else TOL_BF16


def q_f64(q):
    return oracle.bf16_bits_to_f64(q.contiguous().view(torch.int16).cpu().numpy())


_E4M3_TABLE = None


def e4m3_table():
    """The oracle's value of every e4m3 code (its bit-layout decoder applied to all 256)."""
    global _E4M3_TABLE
    if _E4M3_TABLE is None:
        _E4M3_TABLE = oracle.e4m3_bits_to_f64(np.arange(256, dtype=np.uint8))
    return _E4M3_TABLE


def dequant_fp8_rows(codes, scales, block):
    """oracle.dequant_e4m3_blocks for rows 0.. of a (batch, KV head), through the oracle's
    code table (one gather instead of the bit decoding of every element: the full-size
    caches hold 2^27 codes per group)."""
    codes = np.asarray(codes)
    s = np.asarray(scales, dtype=np.float64)[np.arange(codes.shape[0]) // block]
    return e4m3_table()[codes] * s[:, None]


def kv_f64(inp, w, which, b, g, n_tok=None):
    """Dequantised K or V rows [n_tok, d] (default: all S) of (batch b, KV head g) as float64."""
    t = inp[which][b, g]
    if n_tok is not None:
        t = t[:n_tok]
    if w.kv_dtype == "bf16":
        return oracle.bf16_bits_to_f64(t.contiguous().view(torch.int16).cpu().numpy())
    scales = inp["k_scale" if which == "k" else "v_scale"][b, g].cpu().numpy()
    return dequant_fp8_rows(t.contiguous().cpu().numpy(), scales, w.scale_block)


def oracle_group(inp, w, b, g, bounds=None, causal_offset=None):
    """Oracle partials of one (batch, KV head): o [n_split, Tq, G, dv], lse [n_split, Tq, G]."""
    G = w.Hq // w.Hkv
    bounds = inp["split_bounds"] if bounds is None else bounds
    causal = w.causal_offset if causal_offset is None else causal_offset
    qb = q_f64(inp["q"][b : b + 1, :, g * G : (g + 1) * G])
    kb = kv_f64(inp, w, "k", b, g)[None, None]
    vb = kv_f64(inp, w, "v", b, g)[None, None]
    pos = {}
    if inp.get("q_pos_host") is not None:  # tokens stored out of sequence order
        pos = {"q_positions": [inp["q_pos_host"][b]], "k_positions": [inp["k_pos_host"][b]]}
    o, lse = oracle.split_attention(qb, kb, vb, [inp["seq_lens_host"][b]], [bounds[b]], causal, w.scale, **pos)
    return o[:, 0], lse[:, 0]


def oracle_all(inp, w, bounds=None, causal_offset=None):
    """Oracle partials of every (batch, KV head): o [n_split,B,Tq,Hq,dv], lse [n_split,B,Tq,Hq]."""
    G = w.Hq // w.Hkv
    bounds = inp["split_bounds"] if bounds is None else bounds
    n_split = len(bounds[0]) - 1
    o = np.zeros((n_split, w.B, w.Tq, w.Hq, w.dv))
    lse = np.zeros((n_split, w.B, w.Tq, w.Hq))
    for b in range(w.B):
        for g in range(w.Hkv):
            og, lg = oracle_group(inp, w, b, g, bounds, causal_offset)
            o[:, b, :, g * G : (g + 1) * G] = og
            lse[:, b, :, g * G : (g + 1) * G] = lg
    return o, lse


def assert_close(got_o, got_lse, ref_o, ref_lse, tol, what=""):
    """Element-wise parity: |o - o_ref| <= tol['out'], |lse - lse_ref| <= tol['lse'];
    rows with lse_ref = -inf must have lse = -inf and o = 0."""
    stored_bf16 = got_o.dtype == torch.bfloat16
    go = got_o.detach().float().cpu().numpy().astype(np.float64)
    gl = got_lse.detach().float().cpu().numpy().astype(np.float64)
    assert go.shape == ref_o.shape, (what, go.shape, ref_o.shape)
    assert gl.shape == ref_lse.shape, (what, gl.shape, ref_lse.shape)
    assert np.all(np.isfinite(go)), f"{what}: non-finite output"
    empty = np.isneginf(ref_lse)
    assert np.array_equal(np.isneginf(gl), empty), f"{what}: empty-row pattern differs"
    if empty.any():
        assert np.all(go[empty] == 0.0), f"{what}: empty rows must be 0"
    full = ~empty
    err_o = float(np.max(np.abs(go - ref_o))) if go.size else 0.0
    err_l = float(np.max(np.abs(gl[full] - ref_lse[full]))) if full.any() else 0.0
    if stored_bf16:
        # element-wise: |o - o_ref| <= bar + |bf16(o_ref) - o_ref|; report the excess over the bar
        allow = np.abs(bf16_round(ref_o) - ref_o)
        excess = float(np.max(np.abs(go - ref_o) - allow)) if go.size else 0.0
        assert excess <= tol["out"], (f"{what}: out err beyond bf16 storage rounding {excess:.3e} > {tol['out']} "
                                      f"(max-abs {err_o:.3e})")
    else:
        assert err_o <= tol["out"], f"{what}: out max-abs err {err_o:.3e} > {tol['out']}"
    assert err_l <= tol["lse"], f"{what}: lse max-abs err {err_l:.3e} > {tol['lse']}"
    return err_o, err_l


# Bar on the largest output error relative to the RMS of the reference outputs, for the
# full-size cases: there the outputs are averages over up to 2^20 value rows (magnitude
# ~1/sqrt(tokens)), so an absolute bar of 1e-2 (4e-2 for fp8) says little.  The expected
# error is dominated by the bf16 rounding of the stored output, at most 2^-9 of an element
# that is a few times the RMS (~1 % of the RMS); P's rounding averages out over the tokens.
# The bar, 2^-5 of the RMS, leaves a factor of ~3.
REL_RMS_BAR = 2.0 ** -5


def rel_rms_err(got_o, ref_o):
    """max |o - o_ref| / RMS(o_ref) over a set of output rows."""
    go = got_o.detach().float().cpu().numpy().astype(np.float64)
    ref = np.asarray(ref_o, dtype=np.float64)
    rms = float(np.sqrt(np.mean(ref * ref)))
    return float(np.max(np.abs(go - ref))) / rms if rms > 0 else 0.0


def oracle_rows(inp, w, b, g, t_rows, bounds=None, causal_offset=None):
    """Oracle partials of selected query rows of one (batch, KV head):
    o [n_split, len(t_rows), G, dv], lse [n_split, len(t_rows), G].  Used at full size,
    where computing every row would be too slow on the host."""
    G = w.Hq // w.Hkv
    bounds = inp["split_bounds"] if bounds is None else bounds
    causal = w.causal_offset if causal_offset is None else causal_offset
    n_split = len(bounds[b]) - 1
    seq = inp["seq_lens_host"][b]
    t_rows = list(t_rows)
    qb = q_f64(inp["q"][b, t_rows, g * G : (g + 1) * G])  # [R, G, dk]
    n_tok = min(seq, w.S)  # tokens at or past seq_len are never visible
    kf = kv_f64(inp, w, "k", b, g, n_tok)
    vf = kv_f64(inp, w, "v", b, g, n_tok)
    R = len(t_rows)
    o = np.zeros((n_split, R, G, w.dv))
    lse = np.full((n_split, R, G), -np.inf)
    if inp.get("q_pos_host") is not None:  # tokens stored out of sequence order
        q_pos = np.repeat(np.asarray(inp["q_pos_host"][b], dtype=np.int64)[t_rows], G)
        k_pos = np.asarray(inp["k_pos_host"][b], dtype=np.int64)
    else:
        q_pos = np.repeat(causal + np.asarray(t_rows, dtype=np.int64), G)
        k_pos = np.arange(w.S)
    for j in range(n_split):
        lo, hi = max(bounds[b][j], 0), min(bounds[b][j + 1], seq, w.S)
        if hi <= lo:
            continue
        oo, ll = oracle.attend(qb.reshape(R * G, w.dk), kf[lo:hi], vf[lo:hi], w.scale, q_pos, k_pos[lo:hi])
        o[j] = oo.reshape(R, G, w.dv)
        lse[j] = ll.reshape(R, G)
    return o, lse


def oracle_passq(inp, w, b, g):
    """Oracle of one (request b, KV head g) of a pass-Q workload: attention of the request's
    query heads over the union of its shards on every rank.  Returns (o [1, G, dv], lse [1, G])."""
    G = w.Hq // w.Hkv
    N = w.passq_ranks
    lens = inp["shard_lens_host"]
    ks, vs = [], []
    for r in range(N):
        row = r * w.B + b
        for which, acc in (("k", ks), ("v", vs)):
            t = inp[f"{which}_shards"][row, g]
            if w.kv_dtype == "bf16":
                f = oracle.bf16_bits_to_f64(t.contiguous().view(torch.int16).cpu().numpy())
            else:
                sc = inp[f"{which}_shard_scale"][row, g].cpu().numpy()
                f = oracle.dequant_e4m3_blocks(t.contiguous().cpu().numpy(), sc, w.scale_block)
            acc.append(f[None, None, None])  # [1 rank, 1 request, 1 head, S_loc, d]
    sl = [[lens[r][b]] for r in range(N)]
    ku, tot = oracle.gather_shards(np.concatenate(ks), sl)
    vu, _ = oracle.gather_shards(np.concatenate(vs), sl)
    qb = q_f64(inp["q"][b : b + 1, :, g * G : (g + 1) * G])
    o, lse = oracle.full_attention(qb, ku, vu, tot, w.causal_offset, w.scale)
    return o[0], lse[0]
