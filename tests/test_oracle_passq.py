"""Pins of the pass-Q decode oracle ("Context Parallelism for Scalable Million-Token
Inference", sections "Pass-Q keeps KV stationary for cache-heavy turns" and "Pass-Q decode
protects capacity but can hurt TTIT") and of the shard placement the generator draws.

The ring, the return of the partials and the merge must reach exactly the attention of
each request's query over the union of its shards; the pins below check that against a
closed form, a hand-worked gather, invariances and the unsplit oracle, each chosen so
that a routing slip (a query attending the wrong request's shard, a partial filed under
the wrong owner, a block that never reaches some rank) fails at least one of them."""

import numpy as np
import pytest

import oracle
from oracle import passq as PQ
from mla_decode_attention_gqa_gb300 import workloads as W


def _shards(seed, N, B, Hkv, S_loc, d, lens):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((N, B, Hkv, S_loc, d))
    v = rng.standard_normal((N, B, Hkv, S_loc, d))
    for r in range(N):
        for b in range(B):
            k[r, b, :, lens[r][b]:] = np.nan  # never read
            v[r, b, :, lens[r][b]:] = np.nan
    return k, v


def _definition(q, k, v, lens, scale):
    """Attention over the union of each request's shards (no causal cut)."""
    ku, tot = oracle.gather_shards(k, lens)
    vu, _ = oracle.gather_shards(v, lens)
    return oracle.full_attention(q, ku, vu, tot, 1 << 62, scale)


@pytest.mark.parametrize("N,B", [(1, 3), (2, 4), (3, 6), (4, 4)])
def test_passq_equals_attention_over_the_union(N, B):
    rng = np.random.default_rng(10 + N)
    Hkv, G, d, S_loc = 2, 3, 8, 7
    lens = [[int(x) for x in rng.integers(0, S_loc + 1, B)] for _ in range(N)]
    lens[0][0] = max(lens[0][0], 1)
    k, v = _shards(N, N, B, Hkv, S_loc, d, lens)
    q = rng.standard_normal((B, 1, Hkv * G, d))
    o, lse = oracle.passq_decode(q, k, v, lens, 0.35)
    ro, rl = _definition(q, k, v, lens, 0.35)
    assert np.array_equal(np.isneginf(lse), np.isneginf(rl))
    assert np.allclose(o, ro, atol=1e-12, rtol=0) and np.allclose(lse[np.isfinite(rl)], rl[np.isfinite(rl)],
                                                                  atol=1e-12, rtol=0)


def test_zero_query_is_the_mean_value_over_every_rank_and_log_count():
    """q = 0: every resident token scores 0, so o is the plain mean of all resident V rows
    of the request on all ranks and lse = ln(count) -- computed here straight from the
    shards, without the gather."""
    N, B, Hkv, G, d, S_loc = 3, 3, 1, 2, 4, 5
    lens = [[2, 0, 5], [1, 3, 5], [4, 0, 1]]
    k, v = _shards(3, N, B, Hkv, S_loc, d, lens)
    q = np.zeros((B, 1, Hkv * G, d))
    o, lse = oracle.passq_decode(q, k, v, lens, 0.5)
    for b in range(B):
        rows = np.concatenate([v[r, b, 0, :lens[r][b]] for r in range(N)])
        for h in range(G):
            assert np.allclose(o[b, 0, h], rows.mean(axis=0), atol=1e-13)
            assert abs(lse[b, 0, h] - np.log(len(rows))) < 1e-13


def test_one_token_per_request_returns_its_value_row():
    """A request whose only resident token sits on the last rank gets that token's V row
    and lse = its score, whichever rank owns the query."""
    N, B, d = 2, 2, 3
    lens = [[0, 0], [1, 1]]
    k = np.zeros((N, B, 1, 1, d))
    v = np.zeros((N, B, 1, 1, d))
    k[1, 0, 0, 0] = [1.0, 0.0, 0.0]
    k[1, 1, 0, 0] = [0.0, 2.0, 0.0]
    v[1, 0, 0, 0] = [3.0, 4.0, 5.0]
    v[1, 1, 0, 0] = [-1.0, 0.5, 7.0]
    q = np.zeros((B, 1, 1, d))
    q[0, 0, 0] = [2.0, 0.0, 0.0]
    q[1, 0, 0] = [0.0, 3.0, 0.0]
    o, lse = oracle.passq_decode(q, k, v, lens, 0.5)
    assert np.array_equal(o[0, 0, 0], [3.0, 4.0, 5.0]) and lse[0, 0, 0] == 0.5 * 2.0
    assert np.array_equal(o[1, 0, 0], [-1.0, 0.5, 7.0]) and lse[1, 0, 0] == 0.5 * 6.0


def test_resharding_leaves_the_result_unchanged():
    """The same tokens spread differently over the ranks give the same attention."""
    rng = np.random.default_rng(7)
    B, Hkv, G, d, n = 3, 1, 2, 6, 9
    kt = rng.standard_normal((B, Hkv, n, d))
    vt = rng.standard_normal((B, Hkv, n, d))
    q = rng.standard_normal((B, 1, G, d))
    results = []
    for cuts in ([3, 6], [0, 9], [8, 8], [1, 2]):
        N = 3
        lens = [[0] * B for _ in range(N)]
        k = np.full((N, B, Hkv, n, d), np.nan)
        v = np.full((N, B, Hkv, n, d), np.nan)
        edges = [0] + cuts + [n]
        for b in range(B):
            for r in range(N):
                a, e = edges[r], edges[r + 1]
                lens[r][b] = e - a
                k[r, b, :, : e - a] = kt[b, :, a:e]
                v[r, b, :, : e - a] = vt[b, :, a:e]
        results.append(oracle.passq_decode(q, k, v, lens, 0.4))
    for o, lse in results[1:]:
        assert np.allclose(o, results[0][0], atol=1e-13) and np.allclose(lse, results[0][1], atol=1e-13)


def test_request_resident_nowhere_is_empty():
    N, B, Hkv, G, d, S_loc = 2, 2, 1, 1, 4, 3
    lens = [[0, 2], [0, 1]]
    k, v = _shards(5, N, B, Hkv, S_loc, d, lens)
    q = np.ones((B, 1, G, d))
    o, lse = oracle.passq_decode(q, k, v, lens, 1.0)
    assert np.all(o[0] == 0.0) and np.all(np.isneginf(lse[0]))
    assert np.all(np.isfinite(lse[1]))


def test_ring_schedule_visits_every_block_once():
    """At every step the blocks sit on distinct ranks, and over the N steps every rank
    holds every block exactly once."""
    for N in range(1, 9):
        for s in range(N):
            assert sorted(PQ.ring_source(k, s, N) for k in range(N)) == list(range(N))
        for k in range(N):
            assert sorted(PQ.ring_source(k, s, N) for s in range(N)) == list(range(N))
        assert [PQ.ring_source(k, 0, N) for k in range(N)] == list(range(N))  # step 0: its own block


def test_owned_requests_need_a_padded_batch():
    assert PQ.owned_requests(1, 6, 3) == [2, 3]
    with pytest.raises(ValueError):
        PQ.owned_requests(0, 5, 2)


def test_hand_worked_gather():
    """Two ranks, two requests, one head, d = 1: the union keeps rank order."""
    sh = np.array([[[[[1.0], [2.0], [-9.0]]], [[[3.0], [-9.0], [-9.0]]]],
                   [[[[4.0], [-9.0], [-9.0]]], [[[5.0], [6.0], [7.0]]]]])  # [N=2, B=2, Hkv=1, S=3, d=1]
    out, tot = oracle.gather_shards(sh, [[2, 1], [1, 3]])
    assert tot == [3, 4]
    assert out.shape == (2, 1, 4, 1)
    assert out[0, 0, :3, 0].tolist() == [1.0, 2.0, 4.0]
    assert out[1, 0, :, 0].tolist() == [3.0, 5.0, 6.0, 7.0]


def test_shard_lens_hand_worked_and_complete():
    """L = 16, N = 2, 4 decoded tokens: the prompt of 12 is cut into chunks of 3; rank 0
    keeps chunks 0 and 3, rank 1 chunks 1 and 2 (6 each); decoded tokens of request 0 go
    to ranks 0, 1, 0, 1 and those of request 1 to ranks 1, 0, 1, 0."""
    w = W.Workload("pq", B=2, Tq=1, Hq=2, Hkv=1, dk=64, dv=64, S=16, passq_ranks=2, passq_decode_tokens=4)
    assert W.passq_shard_lens(w, [16, 16]) == [[8, 8], [8, 8]]
    assert W.passq_shard_lens(w, [15, 3]) == [[5 + 2, 1], [6 + 2, 2]]
    w4 = W.PASSQ_DECODE_CP4
    rng = np.random.default_rng(0)
    seq = [int(x) for x in rng.integers(0, 200000, 8)] + [0, 1, 1023, 1024, 1025]
    lens = W.passq_shard_lens(w4, seq)
    assert [sum(lens[r][b] for r in range(4)) for b in range(len(seq))] == seq
    # load balance: only the rounding of the chunk size (under 2N tokens, all short on the
    # last chunk) and one decoded token separate the shards of a long request
    long = W.passq_shard_lens(w4, [131072 - 5])
    assert max(r[0] for r in long) - min(r[0] for r in long) <= 2 * 4
