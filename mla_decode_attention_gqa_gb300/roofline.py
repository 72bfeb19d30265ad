"""Algorithmic bytes and flops of split-KV attention, and the pages' KV-read roofline.

Host-side arithmetic only (no device work).  ``bench.py`` divides these algorithmic
figures by measured kernel durations to report achieved GB/s or TFLOP/s.

* KV bytes: every visible (token, KV head) pair is read exactly once - K row plus V
  row (an MLA latent row is read once and serves as both), plus the fp32 block
  scales of fp8 caches.  This is the Helix page's KV-read term
  t_kv = B * 2 * ceil(K/TPA) * Hsz * (S/KVP) * bytes / MemBW with TPA = KVP = 1
  ("Helix Parallelism: Why Tensor Parallelism Hits a Wall at Million-Token
  Context", section "The ceiling, in algebra").
* Flops: 2 * (dk + dv) per visible (query row, query head, token) triple (QK^T and
  PV multiply-adds); masked pairs are not counted.
"""

import math

NO_CAUSAL = 1 << 62


def helix_kv_read_seconds(B, K, TPA, Hsz, S, KVP, bytes_param, membw_bytes_per_s):
    """Per-layer KV read time of one GPU, the Helix page's formula."""
    return B * 2 * math.ceil(K / TPA) * Hsz * (S / KVP) * bytes_param / membw_bytes_per_s


def _visible_per_row(lo, hi, seq_len, causal_offset, i):
    hi = min(hi, seq_len, causal_offset + i + 1)
    return max(0, hi - max(lo, 0))


def visible_tokens(split_bounds_b, seq_len, n_split):
    """Number of distinct existing tokens covered by the splits of one sequence."""
    total = 0
    for j in range(n_split):
        lo, hi = split_bounds_b[j], min(split_bounds_b[j + 1], seq_len)
        total += max(0, hi - lo)
    return total


def kv_bytes(Hkv, dk, dv, kv_dtype, seq_lens, split_bounds, mla=False, scale_block=64):
    """Algorithmic KV-cache bytes of one call (each visible token x KV head once)."""
    elem = 1 if kv_dtype == "fp8_e4m3" else 2
    n_split = len(split_bounds[0]) - 1
    total = 0
    for b, L in enumerate(seq_lens):
        n_tok = visible_tokens(split_bounds[b], L, n_split)
        row = dk * elem if mla else (dk + dv) * elem
        total += n_tok * Hkv * row
        if kv_dtype == "fp8_e4m3":
            # one fp32 scale per touched block for K and for V
            blocks = set()
            for j in range(n_split):
                lo, hi = split_bounds[b][j], min(split_bounds[b][j + 1], L)
                if hi > lo:
                    blocks.update(range(lo // scale_block, (hi - 1) // scale_block + 1))
            total += 2 * 4 * len(blocks) * Hkv
    return total


def attn_flops(Tq, Hq, dk, dv, seq_lens, split_bounds, causal_offset=NO_CAUSAL):
    """Algorithmic flops: 2*(dk+dv) per visible (row, head, token) triple."""
    n_split = len(split_bounds[0]) - 1
    pairs = 0
    for b, L in enumerate(seq_lens):
        for j in range(n_split):
            lo, hi = split_bounds[b][j], split_bounds[b][j + 1]
            if causal_offset >= NO_CAUSAL // 2:
                pairs += Tq * max(0, min(hi, L) - lo)
            else:
                # row i sees tokens t <= causal_offset + i
                pairs += sum(_visible_per_row(lo, hi, L, causal_offset, i) for i in range(Tq))
    return 2 * (dk + dv) * Hq * pairs


def attn_flops_positions(Hq, dk, dv, seq_lens, split_bounds, q_positions, k_positions):
    """Algorithmic flops when the causal rule comes from original positions (zigzag /
    striped storage): 2*(dk+dv) per (row, head, token) with k_pos[t] <= q_pos[row]."""
    import numpy as np

    n_split = len(split_bounds[0]) - 1
    pairs = 0
    for b, L in enumerate(seq_lens):
        qp = np.asarray(q_positions[b], dtype=np.int64)
        kp = np.asarray(k_positions[b], dtype=np.int64)
        for j in range(n_split):
            lo, hi = max(split_bounds[b][j], 0), min(split_bounds[b][j + 1], L)
            if hi <= lo:
                continue
            ks = np.sort(kp[lo:hi])
            pairs += int(np.searchsorted(ks, qp, side="right").sum())
    return 2 * (dk + dv) * Hq * pairs
