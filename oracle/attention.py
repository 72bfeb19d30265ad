"""Exact attention over a sequence-split KV cache, and the exact LSE merge, in float64.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``).

Sources (web pages; cited by title and section):

* [Helix] "Helix Parallelism: Why Tensor Parallelism Hits a Wall at Million-Token
  Context", section "Sharding the sequence instead": every KVP rank runs
  attention over its own KV shard and emits a partial output plus a log-sum-exp
  per token and query head; the fragments are merged with m = max lse,
  den = sum exp(lse - m), o = sum o * exp(lse - m) / den.
* [CP] "Context Parallelism for Scalable Million-Token Inference" (knowledge
  note), section "Pass-KV keeps queries local and circulates keys and values": the
  same merge as a closed-form equation over the N ring steps, and section "A
  runtime heuristic chooses the ring direction": shape(Q) = [T, N_H, D_H],
  shape(K) = shape(V) = [T+P, N_KV, D_H].
* [Overview] "现代大模型推理并行策略总览", section "Transformer 的工程实践": rank r of a
  head-aligned split holds query heads [r*h_q_local, (r+1)*h_q_local) and KV heads
  [r*h_kv_local, ...), i.e. query heads map to KV heads in contiguous groups;
  section "Decode CP：固定 KV Cache 分片，归并局部结果": each shard keeps one LSE per
  query head and the shards are merged by their share of the softmax
  denominator; section "序列布局": a causal mask is decided by a token's original
  position.

Readings where the pages are silent: the LSE is the
natural log of the softmax denominator over *scaled* scores; a partial output is
normalised by its own denominator; the merged LSE is m + ln(den); a split with no
visible token has o = 0 and lse = -inf and weight 0 in the merge; query row i of a
chunk sits at global position causal_offset + i and sees KV position t iff
t <= causal_offset + i.  When the tokens are stored out of sequence order (the
zigzag and striped layouts of [Overview] section "序列布局：Contiguous、Zigzag 与
Striped"), every stored query row and KV token carries its original position and the
same rule applies to those positions: a token is visible iff its position is at most
the row's.
"""

import numpy as np


def kv_head_of(h, Hq, Hkv):
    """KV head read by query head h: contiguous groups of Hq/Hkv heads ([Overview])."""
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    return h // (Hq // Hkv)


def visible_mask(q_pos, kv_pos):
    """[R, n] bool: KV token t is visible to query row i iff kv_pos[t] <= q_pos[i]
    (causal mask by original position, [Overview] section "序列布局")."""
    return np.asarray(kv_pos)[None, :] <= np.asarray(q_pos)[:, None]


def attend(q, k, v, scale, q_pos=None, kv_pos=None):
    """Exact softmax attention of query rows over a set of tokens.

    q : [R, dk] float64   query rows
    k : [n, dk] float64   key rows of the candidate tokens
    v : [n, dv] float64   value rows of the candidate tokens
    scale : softmax scale applied to q.k
    q_pos, kv_pos : optional global positions ([R], [n]); when both are given a
        token is visible to a row only if kv_pos <= q_pos (causal mask by original
        position, [Overview] "序列布局").

    Returns (o [R, dv], lse [R]):  o = sum_t e^{s_t - M} v_t / sum_t e^{s_t - M},
    lse = M + ln sum_t e^{s_t - M}, s_t = scale * q.k_t over the visible t, M their
    max.  A row with no visible token gets o = 0, lse = -inf.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    R, n, dv = q.shape[0], k.shape[0], v.shape[1]
    o = np.zeros((R, dv))
    lse = np.full(R, -np.inf)
    if n == 0 or R == 0:
        return o, lse
    s = scale * (q @ k.T)  # [R, n] scores
    if q_pos is not None and kv_pos is not None:
        s = np.where(visible_mask(q_pos, kv_pos), s, -np.inf)  # invisible tokens take no part
    m = s.max(axis=1)
    has = np.isfinite(m)  # rows with at least one visible token
    m_safe = np.where(has, m, 0.0)
    e = np.exp(s - m_safe[:, None])  # exactly 0 for invisible tokens
    den = e.sum(axis=1)
    num = e @ v
    o[has] = num[has] / den[has, None]
    lse[has] = m[has] + np.log(den[has])
    return o, lse


def _visible_range(lo, hi, seq_len):
    """Tokens of a split [lo, hi) that exist in a sequence of length seq_len."""
    return max(lo, 0), min(hi, seq_len)


def split_attention(q, k, v, seq_lens, split_bounds, causal_offset, scale, q_positions=None, k_positions=None):
    """Partial attention of every split of the KV cache ([Helix], [CP]).

    q : [B, Tq, Hq, dk] float64
    k : [B, Hkv, S, dk] float64 (dequantised)
    v : [B, Hkv, S, dv] float64
    seq_lens : [B] ints; tokens t >= seq_lens[b] do not exist
    split_bounds : [B][n_split + 1] ints; split j of batch b is [b_j, b_{j+1})
    causal_offset : query row i sits at global position causal_offset + i
    scale : softmax scale
    q_positions, k_positions : optional [B][Tq] and [B][S] original positions of the
        stored query rows and KV tokens (zigzag / striped storage); when given they
        replace causal_offset + i and t in the causal rule.

    Returns (o [n_split, B, Tq, Hq, dv], lse [n_split, B, Tq, Hq]).
    """
    B, Tq, Hq, dk = q.shape
    _, Hkv, S, dv = v.shape
    bounds = np.asarray(split_bounds, dtype=np.int64).reshape(B, -1)
    n_split = bounds.shape[1] - 1
    o = np.zeros((n_split, B, Tq, Hq, dv))
    lse = np.full((n_split, B, Tq, Hq), -np.inf)
    positional = q_positions is not None and k_positions is not None
    for b in range(B):
        q_pos = np.asarray(q_positions[b], dtype=np.int64) if positional else causal_offset + np.arange(Tq)
        for j in range(n_split):
            lo, hi = _visible_range(int(bounds[b, j]), int(bounds[b, j + 1]), int(seq_lens[b]))
            if hi <= lo:
                continue
            kv_pos = np.asarray(k_positions[b], dtype=np.int64)[lo:hi] if positional else np.arange(lo, hi)
            for h in range(Hq):
                g = kv_head_of(h, Hq, Hkv)
                oo, ll = attend(q[b, :, h, :], k[b, g, lo:hi], v[b, g, lo:hi], scale, q_pos, kv_pos)
                o[j, b, :, h, :] = oo
                lse[j, b, :, h] = ll
    return o, lse


def full_attention(q, k, v, seq_lens, causal_offset, scale, q_positions=None, k_positions=None):
    """Unsplit attention over every existing token: the result the merge must equal."""
    B = q.shape[0]
    bounds = [[0, int(seq_lens[b])] for b in range(B)]
    o, lse = split_attention(q, k, v, seq_lens, bounds, causal_offset, scale, q_positions, k_positions)
    return o[0], lse[0]


def merge_lse(o_parts, lse_parts):
    """Exact merge of partial outputs by their log-sum-exp ([Helix], [CP]).

    o_parts : [n, ..., dv], lse_parts : [n, ...]
    m = max_s lse_s;  w_s = exp(lse_s - m);  o = sum_s w_s o_s / sum_s w_s;
    lse = m + ln sum_s w_s.  Where every lse_s is -inf the result is o = 0, lse = -inf.
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    m = lse_parts.max(axis=0)
    empty = np.isneginf(m)
    m_safe = np.where(empty, 0.0, m)
    w = np.exp(lse_parts - m_safe[None])  # exp(-inf) = 0 for empty parts
    den = w.sum(axis=0)
    num = (w[..., None] * o_parts).sum(axis=0)
    with np.errstate(invalid="ignore", divide="ignore"):
        o = np.where(empty[..., None], 0.0, num / np.where(empty, 1.0, den)[..., None])
        lse = np.where(empty, -np.inf, m_safe + np.log(np.where(empty, 1.0, den)))
    return o, lse
