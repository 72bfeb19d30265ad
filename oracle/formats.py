"""Number formats read by the oracle, decoded from their bit layouts in float64.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``).

* bfloat16: the upper 16 bits of an IEEE-754 binary32 value, so a bf16 code ``c``
  is the binary32 whose bit pattern is ``c << 16``.
* fp8 E4M3 (the OCP 8-bit floating-point format, "E4M3" encoding): 1 sign bit,
  4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 is subnormal
  (value ``m/8 * 2**-6``); the all-ones pattern ``S.1111.111`` is NaN; there are no
  infinities, so the largest finite magnitude is ``1.75 * 2**8 = 448``.

The KV-cache quantisation that uses E4M3 (one fp32 scale per block of 64 tokens and
per KV head, dequantised value = code value x scale) is the long-context KVP
workload's cache format; the Helix page ("Helix Parallelism: Why Tensor
Parallelism Hits a Wall at Million-Token Context", section "The ceiling, in
algebra") only names low-precision (FP4) KV, so the block-scale format (one fp32
scale per block of 64 tokens and KV head, value = code x scale) is this project's reading.
"""

import numpy as np


def bf16_bits_to_f64(bits):
    """bfloat16 codes (uint16 / int16 array) -> exact float64 values."""
    u = np.asarray(bits).astype(np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def e4m3_bits_to_f64(codes):
    """fp8 E4M3 codes (uint8 array) -> exact float64 values (NaN for S.1111.111)."""
    c = np.asarray(codes).astype(np.uint8).astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    exp_field = (c >> 3) & 0xF
    mant = (c & 0x7).astype(np.float64)
    normal = (1.0 + mant / 8.0) * np.exp2(exp_field.astype(np.float64) - 7.0)
    subnormal = (mant / 8.0) * 2.0 ** -6
    mag = np.where(exp_field == 0, subnormal, normal)
    mag = np.where((exp_field == 0xF) & ((c & 0x7) == 0x7), np.nan, mag)
    return sign * mag


def dequant_e4m3_blocks(codes, scales, block, t0=0):
    """Dequantise a run of E4M3 KV rows of one (batch, KV head).

    codes  : uint8 [n_tok, d] holding tokens t0 .. t0+n_tok-1
    scales : float32/64 [n_blocks] for that (batch, KV head); token t uses
             scales[t // block] (block index by absolute token position)
    returns float64 [n_tok, d] = value(code) * scale
    """
    codes = np.asarray(codes)
    t = np.arange(t0, t0 + codes.shape[0])
    s = np.asarray(scales, dtype=np.float64)[t // block]
    return e4m3_bits_to_f64(codes) * s[:, None]
