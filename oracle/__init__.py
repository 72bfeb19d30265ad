"""Oracle for split-KV exact attention with a log-sum-exp merge.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, ``__graft_entry__.smoke()``
and ``bench.py`` (its ``cpu_baseline`` leg and its ``--impl reference`` arm) may
import anything here.  The CUDA library and its Python binding
(``mla_decode_attention_gqa_gb300``) never import this package and share no code,
table or helper with it; the only thing both sides consume is the seeded input
generator in ``mla_decode_attention_gqa_gb300/workloads.py``, which holds none of
the method's arithmetic.

Everything is plain float64 numpy, written from the pages' statement of the
method (cited per function).  Each function is pinned by ``tests/test_oracle_*``
against closed forms, brute force on tiny inputs, invariants and a library
routine (torch's float8/bfloat16 casts); no function here is "parity unpinned".
"""

from .formats import bf16_bits_to_f64, e4m3_bits_to_f64, dequant_e4m3_blocks
from .attention import (
    kv_head_of,
    attend,
    split_attention,
    merge_lse,
    full_attention,
)
from .paged import gather_pages, gather_block_scales
from .passq import passq_decode, gather_shards

__all__ = [
    "bf16_bits_to_f64",
    "e4m3_bits_to_f64",
    "dequant_e4m3_blocks",
    "kv_head_of",
    "attend",
    "split_attention",
    "merge_lse",
    "full_attention",
    "gather_pages",
    "gather_block_scales",
    "passq_decode",
    "gather_shards",
]
