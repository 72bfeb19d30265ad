"""Seeded synthetic workloads for split-KV attention (shapes, seeds and input tensors).

This module only *draws* inputs: it holds none of the attention or merge
arithmetic.  It is the one module that both the CUDA path's callers (tests,
``bench.py``) and the oracle's callers use, so both sides see the same bytes.

Input recipe (per workload, seed = 1000 + index):
  * Q, K, V ~ N(0, 1) drawn in float32 with ``torch.Generator(device).manual_seed``
    and rounded to bfloat16.
  * fp8 workloads quantise K and V per (batch, KV head, block of ``scale_block``
    tokens): scale = amax(|x|) / 448, code = e4m3(clamp(x / scale, +-448)) with
    torch's round-to-nearest-even cast; the fp32 scales are stored [B, Hkv, n_blocks].
  * Ragged workloads draw seq_len_b uniformly from {S/2, ..., S}; every other
    workload uses seq_len_b = S.
  * Every K/V row at a position >= seq_len_b is poisoned with NaN (bf16 0x7FC0,
    e4m3 0x7F) so that any read past the end of a sequence shows up in the output.
  * MLA workloads hold one latent buffer [B, 1, S, dk]; V is the view of its first
    ``dv`` columns (same storage, row stride dk).
  * Paged workloads also scatter that same logical cache into pages
    [num_blocks, Hkv, block_len, d]: logical block i of sequence b goes to physical block
    perm[b * S / block_len + i] of a seeded permutation of all blocks (B spare blocks,
    NaN-poisoned, are never referenced); the block table [B, S / block_len] records it.
    fp8 scales move with their block: [num_blocks, Hkv, block_len / scale_block].
  * Zigzag / striped ring-prefill workloads store each of the n_split ranks' tokens in
    the rank's layout order (``layout_positions``); the KV cache is the ranks' shards
    one after another and the query chunk is rank ``cp_rank``'s tokens.  The original
    positions go with them as int32 arrays q_pos [B, Tq] and k_pos [B, S].
  * Pass-Q decode workloads spread each request's seq_len_b tokens over ``passq_ranks``
    ranks (``passq_shard_lens``) and draw every rank's resident shard directly:
    k_shards / v_shards [N * B, Hkv, S_loc, d] (row r * B + b: rank r's shard of request
    b; S_loc = the longest shard rounded up to 64), N(0, 1) like the other caches, NaN
    past each shard's length; fp8 shards are quantised per shard block of scale_block
    tokens.  No logical cache is drawn: attention without a causal cut does not depend on
    the order of the tokens, only on which tokens exist.

Shapes follow the pages' workloads: Llama-405B-like GQA heads (Hq=128, Hkv=8,
d=128) from the Helix and context-parallel pages, a DeepSeek-style absorbed MLA
latent (512 + 64 RoPE dims), and the 8-step ring pass-KV prefill chunk.
"""

from dataclasses import dataclass, replace
import math

import torch

NO_CAUSAL = 1 << 62  # causal_offset that masks nothing (decode)
E4M3_MAX = 448.0


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Tq: int
    Hq: int
    Hkv: int
    dk: int
    dv: int
    S: int  # KV positions allocated per (batch, KV head)
    kv_dtype: str = "bf16"  # "bf16" | "fp8_e4m3"
    scale_block: int = 64
    n_split: int = 1
    ragged: bool = False
    causal_offset: int = NO_CAUSAL
    softmax_scale: float = 0.0  # 0 -> 1/sqrt(dk)
    mla: bool = False
    seed: int = 1000
    layout: str = "contiguous"  # "contiguous" | "zigzag" | "striped" (position-array workloads)
    cp_rank: int = 0            # the emulated rank whose query chunk is computed
    paged: bool = False         # also store the cache as pages with a block table
    block_len: int = 64         # tokens per page
    ring_steps: bool = False    # run as n_split pass-KV ring steps, one KV block per call
    passq_ranks: int = 0        # pass-Q decode over this many emulated CP ranks (0: off)
    passq_decode_tokens: int = 0  # tokens each request has decoded since its prompt

    @property
    def scale(self) -> float:
        return self.softmax_scale if self.softmax_scale > 0 else 1.0 / math.sqrt(self.dk)

    @property
    def group(self) -> int:
        return self.Hq // self.Hkv

    def split_bounds(self):
        """[B][n_split+1] contiguous, equal sequence shards of the allocated S."""
        row = [(j * self.S) // self.n_split for j in range(self.n_split + 1)]
        return [list(row) for _ in range(self.B)]


def layout_positions(layout, S, cp, rank):
    """Original positions of the tokens that rank ``rank`` of ``cp`` stores, in storage
    order ("现代大模型推理并行策略总览", section "序列布局：Contiguous、Zigzag 与 Striped";
    "Context Parallelism for Scalable Million-Token Inference", section "Load-balanced
    sharding makes causal work and memory land evenly"):
      contiguous: [r m, (r + 1) m) with m = S / cp;
      zigzag:     2 cp blocks of S / (2 cp); rank r holds block r, then block 2 cp - 1 - r;
      striped:    positions r, r + cp, r + 2 cp, ...
    """
    if S % cp:
        raise ValueError("S must be a multiple of cp")
    if layout == "contiguous":
        m = S // cp
        return list(range(rank * m, (rank + 1) * m))
    if layout == "zigzag":
        if S % (2 * cp):
            raise ValueError("zigzag needs S to be a multiple of 2 cp")
        blk = S // (2 * cp)
        late = 2 * cp - 1 - rank
        return list(range(rank * blk, (rank + 1) * blk)) + list(range(late * blk, (late + 1) * blk))
    if layout == "striped":
        return list(range(rank, S, cp))
    raise ValueError(f"unknown layout {layout}")


# The five workloads, in the order they are numbered (0..4).
TINY_GQA = Workload("tiny_gqa_decode", B=1, Tq=1, Hq=8, Hkv=2, dk=64, dv=64, S=1024,
                    n_split=4, seed=1000)
HELIX_DENSE_128K = Workload("helix_dense_decode_s128k", B=8, Tq=1, Hq=128, Hkv=8, dk=128,
                            dv=128, S=131072, n_split=1, seed=1001)
HELIX_KVP8_FP8_1M = Workload("helix_kvp8_fp8_decode_s1m", B=8, Tq=1, Hq=128, Hkv=8, dk=128,
                             dv=128, S=1 << 20, kv_dtype="fp8_e4m3", scale_block=64,
                             n_split=8, ragged=True, seed=1002)
MLA_ABSORBED = Workload("mla_absorbed_decode_s32k", B=16, Tq=1, Hq=128, Hkv=1, dk=576, dv=512,
                        S=32768, n_split=4, softmax_scale=1.0 / math.sqrt(192.0), mla=True,
                        seed=1003)
RING_PREFILL = Workload("ring_prefill_chunk_8x4096", B=1, Tq=4096, Hq=128, Hkv=8, dk=128,
                        dv=128, S=8 * 4096, n_split=8, causal_offset=7 * 4096, seed=1004)

# The ring prefill chunk with load-balanced layouts: rank 0's 4096 query tokens (zigzag:
# blocks 0 and 15 of 16; striped: every 8th token) against all 8 ranks' shards.
RING_PREFILL_ZIGZAG = Workload("ring_prefill_zigzag_8x4096", B=1, Tq=4096, Hq=128, Hkv=8, dk=128, dv=128,
                               S=8 * 4096, n_split=8, layout="zigzag", cp_rank=0, seed=1005)
RING_PREFILL_STRIPED = Workload("ring_prefill_striped_8x4096", B=1, Tq=4096, Hq=128, Hkv=8, dk=128, dv=128,
                                S=8 * 4096, n_split=8, layout="striped", cp_rank=0, seed=1006)

# The Helix dense decode and the MLA decode with their caches in 64-token pages at a
# seeded permutation of physical blocks.
HELIX_DENSE_128K_PAGED = replace(HELIX_DENSE_128K, name="helix_dense_decode_s128k_paged64", paged=True,
                                 block_len=64, seed=1007)
MLA_ABSORBED_PAGED = replace(MLA_ABSORBED, name="mla_absorbed_decode_s32k_paged64", paged=True, block_len=64,
                             seed=1008)

# The ring prefill chunk as 8 pass-KV ring steps: each step's 4096-token KV block in its
# own buffer, merged into a running output (attn_ring_step).
RING_PREFILL_STEPS = replace(RING_PREFILL, name="ring_prefill_steps_8x4096", ring_steps=True, seed=1009)

# Pass-Q decode on a CP4 group: 8 one-token queries (2 owned by each rank) of requests with
# 64K..128K tokens of context, each request's cache spread over the 4 ranks (load-balanced
# prompt chunks plus 1024 decoded tokens on a rotating owner); Llama-405B-like GQA heads.
PASSQ_DECODE_CP4 = Workload("passq_decode_cp4_s128k", B=8, Tq=1, Hq=128, Hkv=8, dk=128, dv=128, S=131072,
                            ragged=True, passq_ranks=4, passq_decode_tokens=1024, seed=1010)

WORKLOADS = [TINY_GQA, HELIX_DENSE_128K, HELIX_KVP8_FP8_1M, MLA_ABSORBED, RING_PREFILL, RING_PREFILL_ZIGZAG,
             RING_PREFILL_STRIPED, HELIX_DENSE_128K_PAGED, MLA_ABSORBED_PAGED, RING_PREFILL_STEPS, PASSQ_DECODE_CP4]


def passq_shard_lens(w, seq_lens):
    """[N][B] tokens of each request resident on each of the w.passq_ranks ranks.

    A request of L tokens is a prompt of P = L - D tokens followed by D = min(L,
    passq_decode_tokens) decoded ones.  The prompt is cut into 2N chunks of ceil(P / 2N)
    tokens (the last ones shorter or empty) and rank r keeps chunks r and 2N - 1 - r, the
    load-balanced pairing of "Context Parallelism for Scalable Million-Token Inference",
    section "Load-balanced sharding makes causal work and memory land evenly"; decoded
    token t of request b was stored on rank (b + t) mod N, the owner moving on every
    decode iteration (same page, section "Pass-Q decode protects capacity but can hurt
    TTIT").
    """
    N = w.passq_ranks
    lens = [[0] * len(seq_lens) for _ in range(N)]
    for b, L in enumerate(seq_lens):
        D = min(w.passq_decode_tokens, L)
        P = L - D
        c = -(-P // (2 * N))
        for r in range(N):
            for ch in (r, 2 * N - 1 - r):
                lens[r][b] += max(0, min(P, (ch + 1) * c) - ch * c)
            # decoded tokens t with (b + t) mod N == r: t = (r - b) mod N, then every N-th
            first = (r - b) % N
            lens[r][b] += 0 if first >= D else (D - 1 - first) // N + 1
    return lens


def scaled(w: Workload, **kw) -> Workload:
    """A smaller workload of the same structure (for parity at oracle-friendly sizes)."""
    if ("S" in kw or "Tq" in kw) and "causal_offset" not in kw and w.causal_offset != NO_CAUSAL:
        # keep the Q chunk at the end of the KV so the last split is the diagonal
        kw["causal_offset"] = kw.get("S", w.S) - kw.get("Tq", w.Tq)
    return replace(w, **kw)


def _randn(shape, gen, device):
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)


def _quantize_e4m3_blocks(x, block):
    """x [n_tok, d] float32 -> (codes uint8 [n_tok, d], scales float32 [ceil(n_tok/block)])."""
    n_tok, d = x.shape
    nb = (n_tok + block - 1) // block
    pad = nb * block - n_tok
    xp = torch.nn.functional.pad(x, (0, 0, 0, pad)) if pad else x
    xb = xp.view(nb, block, d)
    amax = xb.abs().amax(dim=(1, 2))
    scales = torch.where(amax > 0, amax / E4M3_MAX, torch.ones_like(amax))
    y = (xb / scales[:, None, None]).clamp(-E4M3_MAX, E4M3_MAX)
    codes = y.to(torch.float8_e4m3fn).view(torch.uint8).reshape(nb * block, d)[:n_tok]
    return codes.contiguous(), scales.float()


def make_inputs(w: Workload, device="cpu", poison=True):
    """Draw every input of a workload on ``device``.

    Returns a dict with
      q        bf16  [B, Tq, Hq, dk]
      k, v     bf16  [B, Hkv, S, dk|dv]  or uint8 e4m3 codes of that shape
               (MLA: k is the latent [B, 1, S, dk] and v a view of its first dv columns)
      k_scale, v_scale  float32 [B, Hkv, ceil(S/scale_block)] or None
      seq_lens int32 [B] (on ``device``)
      seq_lens_host  list[int]
      split_bounds   list[list[int]]  ([B][n_split+1])
      q_pos, k_pos   int32 [B, Tq], [B, S] original positions (layout workloads), else None
      q_pos_host, k_pos_host  the same as lists, or None
      paged workloads also: k_pages, v_pages [num_blocks, Hkv, block_len, d] (MLA: v_pages
        a view of k_pages), k_scale_pages / v_scale_pages (fp8), block_table int32 [B, S /
        block_len] and block_table_host
    """
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed)
    B, Hkv, S = w.B, w.Hkv, w.S
    q = _randn((B, w.Tq, w.Hq, w.dk), gen, dev).to(torch.bfloat16)
    if w.ragged:
        seq = torch.randint(S // 2, S + 1, (B,), generator=gen, device=dev)
    else:
        seq = torch.full((B,), S, dtype=torch.int64, device=dev)
    seq_host = [int(x) for x in seq.cpu().tolist()]

    k_scale = v_scale = None
    if w.mla:
        if w.kv_dtype != "bf16":
            raise ValueError("MLA workloads are bf16")
        lat = torch.empty((B, 1, S, w.dk), dtype=torch.bfloat16, device=dev)
        for b in range(B):
            lat[b, 0] = _randn((S, w.dk), gen, dev).to(torch.bfloat16)
            if poison and seq_host[b] < S:
                lat[b, 0, seq_host[b]:] = float("nan")
        k = lat
        v = lat[..., : w.dv]
    elif w.kv_dtype == "bf16":
        k = torch.empty((B, Hkv, S, w.dk), dtype=torch.bfloat16, device=dev)
        v = torch.empty((B, Hkv, S, w.dv), dtype=torch.bfloat16, device=dev)
        for b in range(B):
            for g in range(Hkv):
                k[b, g] = _randn((S, w.dk), gen, dev).to(torch.bfloat16)
                v[b, g] = _randn((S, w.dv), gen, dev).to(torch.bfloat16)
            if poison and seq_host[b] < S:
                k[b, :, seq_host[b]:] = float("nan")
                v[b, :, seq_host[b]:] = float("nan")
    elif w.kv_dtype == "fp8_e4m3":
        nb = (S + w.scale_block - 1) // w.scale_block
        k = torch.empty((B, Hkv, S, w.dk), dtype=torch.uint8, device=dev)
        v = torch.empty((B, Hkv, S, w.dv), dtype=torch.uint8, device=dev)
        k_scale = torch.empty((B, Hkv, nb), dtype=torch.float32, device=dev)
        v_scale = torch.empty((B, Hkv, nb), dtype=torch.float32, device=dev)
        for b in range(B):
            for g in range(Hkv):
                k[b, g], k_scale[b, g] = _quantize_e4m3_blocks(_randn((S, w.dk), gen, dev), w.scale_block)
                v[b, g], v_scale[b, g] = _quantize_e4m3_blocks(_randn((S, w.dv), gen, dev), w.scale_block)
            if poison and seq_host[b] < S:
                k[b, :, seq_host[b]:] = 0x7F
                v[b, :, seq_host[b]:] = 0x7F
    else:
        raise ValueError(f"unknown kv dtype {w.kv_dtype}")

    if w.passq_ranks:
        return _make_passq(w, q, seq, seq_host, gen, dev, poison)

    pages = {}
    if w.paged:
        pages = _make_pages(w, k, v, k_scale, v_scale, gen, dev)

    q_pos = k_pos = None
    q_pos_host = k_pos_host = None
    if w.layout != "contiguous":
        if w.S % w.n_split or w.Tq != w.S // w.n_split:
            raise ValueError("a layout workload holds one rank's chunk: Tq = S / n_split")
        k_row = [p for r in range(w.n_split) for p in layout_positions(w.layout, w.S, w.n_split, r)]
        q_row = layout_positions(w.layout, w.S, w.n_split, w.cp_rank)
        q_pos_host = [list(q_row) for _ in range(B)]
        k_pos_host = [list(k_row) for _ in range(B)]
        q_pos = torch.tensor(q_pos_host, dtype=torch.int32, device=dev)
        k_pos = torch.tensor(k_pos_host, dtype=torch.int32, device=dev)

    return {
        "q": q,
        "k": k,
        "v": v,
        "k_scale": k_scale,
        "v_scale": v_scale,
        "seq_lens": seq.to(torch.int32),
        "seq_lens_host": seq_host,
        "split_bounds": w.split_bounds(),
        "q_pos": q_pos,
        "k_pos": k_pos,
        "q_pos_host": q_pos_host,
        "k_pos_host": k_pos_host,
        **pages,
    }


def _make_pages(w, k, v, k_scale, v_scale, gen, dev):
    """Scatter the logical cache into pages (see the module docstring)."""
    L = w.block_len
    if w.S % L:
        raise ValueError("S must be a multiple of block_len")
    nb = w.S // L
    n_blocks = w.B * nb + w.B  # B spare blocks nobody references
    perm = torch.randperm(n_blocks, generator=gen, device=dev)
    phys = perm[: w.B * nb]

    def scatter(x):  # [B, H, S, d] -> [n_blocks, H, L, d]
        B, H, S, d = x.shape
        blocks = x.reshape(B, H, nb, L, d).permute(0, 2, 1, 3, 4).reshape(B * nb, H, L, d)
        out = torch.empty((n_blocks, H, L, d), dtype=x.dtype, device=dev)
        if x.dtype == torch.uint8:
            out.fill_(0x7F)  # e4m3 NaN
        else:
            out.fill_(float("nan"))
        out[phys] = blocks
        return out

    res = {"block_table": phys.reshape(w.B, nb).to(torch.int32).contiguous(),
           "block_table_host": phys.reshape(w.B, nb).cpu().tolist()}
    if w.mla:
        lat = scatter(k)
        res["k_pages"] = lat
        res["v_pages"] = lat[..., : w.dv]
    else:
        res["k_pages"] = scatter(k)
        res["v_pages"] = scatter(v)
    if k_scale is not None:
        per = L // w.scale_block

        def scatter_s(sc):  # [B, H, S / sb] -> [n_blocks, H, L / sb]
            B, H, _ = sc.shape
            blocks = sc.reshape(B, H, nb, per).permute(0, 2, 1, 3).reshape(B * nb, H, per)
            out = torch.ones((n_blocks, H, per), dtype=sc.dtype, device=dev)
            out[phys] = blocks
            return out

        res["k_scale_pages"] = scatter_s(k_scale)
        res["v_scale_pages"] = scatter_s(v_scale)
    return res


def _make_passq(w, q, seq, seq_host, gen, dev, poison):
    """Inputs of a pass-Q decode workload (see the module docstring)."""
    N, B, Hkv = w.passq_ranks, w.B, w.Hkv
    if B % N or w.Tq != 1:
        raise ValueError("pass-Q decode: one query token per request, B a multiple of passq_ranks")
    lens = passq_shard_lens(w, seq_host)
    S_loc = max(64, -(-max(max(r) for r in lens) // 64) * 64)
    fp8 = w.kv_dtype == "fp8_e4m3"
    if not fp8 and w.kv_dtype != "bf16":
        raise ValueError(f"unknown kv dtype {w.kv_dtype}")
    dt = torch.uint8 if fp8 else torch.bfloat16
    k = torch.empty((N * B, Hkv, S_loc, w.dk), dtype=dt, device=dev)
    v = torch.empty((N * B, Hkv, S_loc, w.dv), dtype=dt, device=dev)
    ks = vs = None
    if fp8:
        nb = S_loc // w.scale_block if S_loc % w.scale_block == 0 else S_loc // w.scale_block + 1
        ks = torch.empty((N * B, Hkv, nb), dtype=torch.float32, device=dev)
        vs = torch.empty((N * B, Hkv, nb), dtype=torch.float32, device=dev)
    for r in range(N):
        for b in range(B):
            row, n = r * B + b, lens[r][b]
            for g in range(Hkv):
                if fp8:
                    k[row, g], ks[row, g] = _quantize_e4m3_blocks(_randn((S_loc, w.dk), gen, dev), w.scale_block)
                    v[row, g], vs[row, g] = _quantize_e4m3_blocks(_randn((S_loc, w.dv), gen, dev), w.scale_block)
                else:
                    k[row, g] = _randn((S_loc, w.dk), gen, dev).to(torch.bfloat16)
                    v[row, g] = _randn((S_loc, w.dv), gen, dev).to(torch.bfloat16)
            if poison and n < S_loc:
                if fp8:
                    k[row, :, n:] = 0x7F
                    v[row, :, n:] = 0x7F
                else:
                    k[row, :, n:] = float("nan")
                    v[row, :, n:] = float("nan")
    return {
        "q": q, "k": None, "v": None, "k_scale": None, "v_scale": None,
        "seq_lens": seq.to(torch.int32), "seq_lens_host": seq_host, "split_bounds": [[0, w.S]] * B,
        "q_pos": None, "k_pos": None, "q_pos_host": None, "k_pos_host": None,
        "k_shards": k, "v_shards": v, "k_shard_scale": ks, "v_shard_scale": vs,
        "shard_lens": torch.tensor(lens, dtype=torch.int32, device=dev), "shard_lens_host": lens,
    }
