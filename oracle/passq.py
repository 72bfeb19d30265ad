"""Pass-Q decode over a context-parallel group: the ring of query blocks, the return of the
partials to their owners and the exact merge, in float64.

TEST INFRASTRUCTURE (see ``oracle/__init__.py``).

Source: "Context Parallelism for Scalable Million-Token Inference" (knowledge note),
sections "Pass-Q keeps KV stationary for cache-heavy turns" and "Pass-Q decode protects
capacity but can hurt TTIT".  Every rank keeps its own KV shard of each request where it
is; the query blocks travel around the ring together with the batch ids of their
requests; a rank computes partial attention for whatever block is with it, against its
resident entry for each of those requests; after the ring the partials are permuted and
returned to the ranks the queries came from by an All-to-All, and merged there exactly
by their log-sum-exp (the merge of section "Pass-KV keeps queries local and circulates
keys and values").  The decode batch is padded to a multiple of the group size.

Readings where the pages are silent: rank r owns the queries of
requests [r * B/N, (r + 1) * B/N); at ring step s rank k holds the block that started on
rank (k - s) mod N (each rank passes its block to rank k + 1); a decode token follows
every token of its request's cache, so it sees every resident token on every rank, in
any order.  The plain definition of the result is attention over the union of a
request's shards (``gather_shards`` + ``full_attention``); ``passq_decode`` takes the
pages' steps and is pinned to that definition.
"""

import numpy as np

from . import attention as A


def owned_requests(r, B, n_ranks):
    """Requests whose one-token queries start on rank r: a contiguous block of B / N."""
    if B % n_ranks:
        raise ValueError("the decode batch must be padded to a multiple of the group size")
    bq = B // n_ranks
    return list(range(r * bq, (r + 1) * bq))


def ring_source(k, s, n_ranks):
    """Rank whose query block is on rank k at ring step s (blocks move to rank + 1)."""
    return (k - s) % n_ranks


def rank_partial(q_block, batch_ids, k_local, v_local, lens_local, scale):
    """One rank's partial attention for the query block it holds.

    q_block : [Bq, Tq, Hq, dk] float64, the arriving queries
    batch_ids : [Bq] request of each arriving query (travels with the block)
    k_local, v_local : [B, Hkv, S_loc, d] float64, this rank's resident shard of every request
    lens_local : [B] resident tokens of each request on this rank

    Returns (o [Bq, Tq, Hq, dv], lse [Bq, Tq, Hq]).
    """
    ids = list(batch_ids)
    kb = np.asarray(k_local)[ids]
    vb = np.asarray(v_local)[ids]
    lens = [int(lens_local[b]) for b in ids]
    # the decode token sits after every cached token: no causal cut
    return A.full_attention(q_block, kb, vb, lens, 1 << 62, scale)


def return_to_owners(arrived):
    """The permutation and All-to-All after the ring: rank k's partial from step s belongs
    to the queries of rank (k - s) mod N, which files it under the sending rank k.

    arrived : [N ranks][N steps] partials in arrival order.  Returns [N owners][N senders].
    """
    N = len(arrived)
    received = [[None] * N for _ in range(N)]
    for k in range(N):
        for s in range(N):
            received[ring_source(k, s, N)][k] = arrived[k][s]
    return received


def passq_decode(q, k_shards, v_shards, shard_lens, scale):
    """Pass-Q decode of every request, in the pages' steps.

    q : [B, Tq, Hq, dk] float64 (Tq = 1 for decode)
    k_shards, v_shards : [N, B, Hkv, S_loc, d] float64: rank r's resident shard of request b
    shard_lens : [N][B] resident tokens

    Returns (o [B, Tq, Hq, dv], lse [B, Tq, Hq]).
    """
    q = np.asarray(q, dtype=np.float64)
    N = len(shard_lens)
    B, Tq, Hq, _ = q.shape
    dv = np.asarray(v_shards).shape[-1]
    blocks = [owned_requests(r, B, N) for r in range(N)]
    bq = B // N
    # 1. the ring: at step s rank k holds the block of rank (k - s) mod N and its batch ids;
    #    its partials are kept in arrival order
    arrived = [[None] * N for _ in range(N)]  # [rank][step] -> (o, lse)
    for s in range(N):
        for k in range(N):
            src = ring_source(k, s, N)
            ids = blocks[src]
            arrived[k][s] = rank_partial(q[ids], ids, k_shards[k], v_shards[k], shard_lens[k], scale)
    # 2. permutation + All-to-All
    received = return_to_owners(arrived)
    # 3. every owner merges the N partials of each of its queries
    o = np.zeros((B, Tq, Hq, dv))
    lse = np.full((B, Tq, Hq), -np.inf)
    for r in range(N):
        parts_o = np.stack([received[r][k][0] for k in range(N)])
        parts_l = np.stack([received[r][k][1] for k in range(N)])
        mo, ml = A.merge_lse(parts_o, parts_l)
        o[r * bq:(r + 1) * bq] = mo
        lse[r * bq:(r + 1) * bq] = ml
    return o, lse


def gather_shards(shards, shard_lens):
    """The union of each request's shards: [B, Hkv, max_b sum_r len, d] (rank order, each
    shard's resident tokens in their stored order; zeros past a request's total) and the
    per-request token counts [B].

    shards : [N, B, Hkv, S_loc, d]; shard_lens : [N][B]
    """
    shards = np.asarray(shards)
    N, B, Hkv, _, d = shards.shape
    lens = np.asarray(shard_lens, dtype=np.int64).reshape(N, B)
    total = lens.sum(axis=0)
    out = np.zeros((B, Hkv, max(int(total.max()), 1), d), dtype=shards.dtype)
    for b in range(B):
        t = 0
        for r in range(N):
            n = int(lens[r, b])
            out[b, :, t:t + n] = shards[r, b, :, :n]
            t += n
    return out, [int(x) for x in total]
