"""Paged block KV cache: the logical cache of every sequence gathered from physical blocks.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``).

Source: "Attention DP", section "KV Cache": each rank keeps its cache as
[num_blocks, num_kv_heads / TP, block_len, d_head].  Reading (where the page is silent):
a per-sequence block table maps logical block i of sequence b to
the physical block that holds its tokens [i * block_len, (i + 1) * block_len), so token t
of sequence b, KV head g is row t mod block_len of block table[b][t // block_len], head g.
Per-block fp8 scales follow the block: scales[phys, g, (t mod block_len) // scale_block].
"""

import numpy as np


def gather_pages(pages, block_table, n_tokens):
    """Logical cache [B, Hkv, n_tokens, d] from pages [num_blocks, Hkv, block_len, d].

    block_table : [B][max_blocks] physical block of each logical block
    n_tokens : tokens per sequence to gather (a multiple of block_len)
    """
    pages = np.asarray(pages)
    nb, Hkv, L, d = pages.shape
    table = np.asarray(block_table, dtype=np.int64)
    B = table.shape[0]
    if n_tokens % L:
        raise ValueError("n_tokens must be a multiple of block_len")
    out = np.empty((B, Hkv, n_tokens, d), dtype=pages.dtype)
    for b in range(B):
        for i in range(n_tokens // L):
            out[b, :, i * L:(i + 1) * L, :] = pages[table[b, i]]
    return out


def gather_block_scales(scales, block_table, n_tokens, block_len, scale_block):
    """Logical fp8 block scales [B, Hkv, n_tokens / scale_block] from per-page scales
    [num_blocks, Hkv, block_len / scale_block]."""
    scales = np.asarray(scales)
    table = np.asarray(block_table, dtype=np.int64)
    B = table.shape[0]
    per = block_len // scale_block
    out = np.empty((B, scales.shape[1], n_tokens // scale_block), dtype=scales.dtype)
    for b in range(B):
        for i in range(n_tokens // block_len):
            out[b, :, i * per:(i + 1) * per] = scales[table[b, i]]
    return out
