"""The seeded input generator follows its stated recipe (CPU, small sizes).

Both the CUDA path's tests and the oracle's read their inputs from
``mla_decode_attention_gqa_gb300.workloads``; these checks pin what that module promises:
the same seed gives the same bytes, ragged lengths stay in {S/2, ..., S}, every K/V row
past a sequence's end is NaN (bf16 0x7FC0, e4m3 0x7F) and no row before it is, fp8 blocks
are scaled by amax / 448 per (batch, KV head, block), an MLA workload's V is a view of the
latent's first dv columns, and the KVP shards cut the allocated S into equal parts."""

import math

import torch

from mla_decode_attention_gqa_gb300 import workloads as W


def _small(w, **kw):
    return W.scaled(w, **kw)


def _bits(t):
    """A tensor's bytes for exact comparison (bf16 NaNs compare unequal as values)."""
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t


def test_same_seed_same_bytes_and_seeds_differ_between_workloads():
    w = _small(W.HELIX_KVP8_FP8_1M, B=2, Hq=16, Hkv=2, S=512)
    a, b = W.make_inputs(w), W.make_inputs(w)
    for key in ("q", "k", "v", "k_scale", "v_scale", "seq_lens"):
        assert torch.equal(_bits(a[key]), _bits(b[key])), key
    assert len({x.seed for x in W.WORKLOADS}) == len(W.WORKLOADS)


def test_ragged_lengths_and_nan_poison_past_the_end_bf16():
    w = _small(W.HELIX_DENSE_128K, B=6, Hq=16, Hkv=2, S=256, ragged=True)
    inp = W.make_inputs(w)
    for b, n in enumerate(inp["seq_lens_host"]):
        assert w.S // 2 <= n <= w.S
        for x in (inp["k"], inp["v"]):
            assert torch.isnan(x[b, :, n:].float()).all()
            assert torch.isfinite(x[b, :, :n].float()).all()
    assert inp["seq_lens"].tolist() == inp["seq_lens_host"]


def test_fp8_blocks_scaled_by_amax_over_448_and_poisoned_with_nan_codes():
    w = _small(W.HELIX_KVP8_FP8_1M, B=3, Hq=16, Hkv=2, S=640)
    inp = W.make_inputs(w)
    k, ks = inp["k"], inp["k_scale"]
    assert ks.shape == (w.B, w.Hkv, math.ceil(w.S / w.scale_block))
    deq = k.view(torch.float8_e4m3fn).float()  # codes in units of the block scale
    for b, n in enumerate(inp["seq_lens_host"]):
        assert (k[b, :, n:] == 0x7F).all() and torch.isnan(deq[b, :, n:]).all()
        for g in range(w.Hkv):
            for blk in range(n // w.scale_block):  # whole blocks below the end
                codes = deq[b, g, blk * w.scale_block:(blk + 1) * w.scale_block]
                # the block's largest |x| maps to the largest finite e4m3 value
                assert float(codes.abs().max()) == W.E4M3_MAX
                assert float(ks[b, g, blk]) > 0
    # the scale is amax / 448 of the values it was drawn from: redraw block 0 of (0, 0)
    gen = torch.Generator().manual_seed(w.seed)
    W._randn((w.B, w.Tq, w.Hq, w.dk), gen, torch.device("cpu"))  # q is drawn first
    torch.randint(w.S // 2, w.S + 1, (w.B,), generator=gen)      # then the ragged lengths
    x = W._randn((w.S, w.dk), gen, torch.device("cpu"))          # then K of (b=0, g=0)
    amax = float(x[:w.scale_block].abs().max())
    assert math.isclose(float(ks[0, 0, 0]), amax / W.E4M3_MAX, rel_tol=1e-6)


def test_mla_value_is_a_view_of_the_latent():
    w = _small(W.MLA_ABSORBED, B=2, S=128)
    inp = W.make_inputs(w)
    k, v = inp["k"], inp["v"]
    assert k.shape == (w.B, 1, w.S, w.dk) and v.shape == (w.B, 1, w.S, w.dv)
    assert v.data_ptr() == k.data_ptr() and v.stride() == k.stride()
    assert torch.equal(_bits(v), _bits(k[..., : w.dv]))


def test_kvp_shards_cut_the_allocated_length_into_equal_parts():
    w = W.HELIX_KVP8_FP8_1M
    bounds = w.split_bounds()
    assert len(bounds) == w.B and all(row == bounds[0] for row in bounds)
    assert bounds[0] == [j * w.S // w.n_split for j in range(w.n_split + 1)]
    assert w.n_split == 8 and w.S == 1 << 20


def test_table_dequantiser_of_the_parity_helpers_equals_the_oracle():
    """tests/oracle_io.dequant_fp8_rows (the oracle's 256 code values, gathered) gives the
    same float64 values as oracle.dequant_e4m3_blocks, NaN codes included."""
    import numpy as np

    import oracle
    from tests import oracle_io as io

    rng = np.random.default_rng(5)
    codes = rng.integers(0, 256, size=(1000, 64), dtype=np.uint8)
    scales = rng.random(1000 // 64 + 1) * 3
    a = io.dequant_fp8_rows(codes, scales, 64)
    b = oracle.dequant_e4m3_blocks(codes, scales, 64)
    assert np.array_equal(np.isnan(a), np.isnan(b))
    assert np.array_equal(a[~np.isnan(a)], b[~np.isnan(b)])
