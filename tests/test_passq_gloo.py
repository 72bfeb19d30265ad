"""Pass-Q decode as a real two-rank ring on the CPU (gloo, world_size 2, 127.0.0.1).

Each process is one rank of the context-parallel group of "Context Parallelism for
Scalable Million-Token Inference" (sections "Pass-Q keeps KV stationary for cache-heavy
turns" and "Pass-Q decode protects capacity but can hurt TTIT"): it keeps its own KV
shard of every request, passes the query block it holds (with the block's batch ids) to
rank + 1 at every step, computes the held block's partials with the fp64 oracle, returns
them to the queries' owners with a pairwise exchange (the All-to-All of two ranks) and
merges what it receives.  The test checks the message schedule against the one the
single-GPU kernel decodes (at step s rank k holds the block of rank (k - s) mod N) and
the merged result against the oracle's definition (attention over the union of shards).
"""

import os
import socket
import sys

import numpy as np
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
N_RANKS, B, HKV, G, D, S_LOC, SCALE = 2, 4, 2, 2, 8, 6, 0.3


def _problem():
    rng = np.random.default_rng(2024)
    lens = [[int(x) for x in rng.integers(0, S_LOC + 1, B)] for _ in range(N_RANKS)]
    lens[0][1], lens[1][1] = 0, 0  # one request resident nowhere
    lens[0][2], lens[1][2] = max(lens[0][2], 1), 0  # one resident on rank 0 only
    k = rng.standard_normal((N_RANKS, B, HKV, S_LOC, D))
    v = rng.standard_normal((N_RANKS, B, HKV, S_LOC, D))
    q = rng.standard_normal((B, 1, HKV * G, D))
    return q, k, v, lens


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, port, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    from oracle import attention as A
    from oracle import passq as PQ

    dist.init_process_group("gloo", rank=rank, world_size=N_RANKS)
    q, k, v, lens = _problem()
    N = N_RANKS
    nxt, prv = (rank + 1) % N, (rank - 1) % N
    held_ids = torch.tensor(PQ.owned_requests(rank, B, N), dtype=torch.int64)
    held_q = torch.from_numpy(q[held_ids.numpy()].copy())
    schedule, arrived = [], []
    for s in range(N):
        schedule.append(held_ids.tolist())
        arrived.append(PQ.rank_partial(held_q.numpy(), held_ids.tolist(), k[rank], v[rank], lens[rank], SCALE))
        if s + 1 < N:  # the ring hop: send the held block on, receive the previous rank's
            rq, ri = torch.empty_like(held_q), torch.empty_like(held_ids)
            reqs = [dist.isend(held_q, nxt), dist.isend(held_ids, nxt), dist.irecv(rq, prv), dist.irecv(ri, prv)]
            for r in reqs:
                r.wait()
            held_q, held_ids = rq, ri
    # return the partials: the one from step s belongs to the owner of that block
    received = [None] * N
    for s in range(N):
        owner = PQ.ring_source(rank, s, N)
        if owner == rank:
            received[rank] = arrived[s]
            continue
        o_s, l_s = (torch.from_numpy(np.ascontiguousarray(x)) for x in arrived[s])
        ro, rl = torch.empty_like(o_s), torch.empty_like(l_s)
        reqs = [dist.isend(o_s, owner), dist.isend(l_s, owner), dist.irecv(ro, owner), dist.irecv(rl, owner)]
        for r in reqs:
            r.wait()
        received[owner] = (ro.numpy(), rl.numpy())
    o, lse = A.merge_lse(np.stack([received[j][0] for j in range(N)]), np.stack([received[j][1] for j in range(N)]))
    dist.barrier()
    dist.destroy_process_group()
    out_q.put((rank, schedule, o, lse))


def test_two_rank_passq_ring_matches_the_schedule_and_the_union_attention():
    sys.path.insert(0, ROOT)
    import oracle
    from oracle import passq as PQ

    ctx = mp.get_context("spawn")
    out_q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, out_q)) for r in range(N_RANKS)]
    for p in procs:
        p.start()
    res = sorted((out_q.get(timeout=240) for _ in procs), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0

    q, k, v, lens = _problem()
    ku, tot = oracle.gather_shards(k, lens)
    vu, _ = oracle.gather_shards(v, lens)
    ro, rl = oracle.full_attention(q, ku, vu, tot, 1 << 62, SCALE)
    po, pl = oracle.passq_decode(q, k, v, lens, SCALE)
    bq = B // N_RANKS
    for rank, schedule, o, lse in res:
        # the block held at step s is the one the kernel's ring decoding assigns
        assert schedule == [PQ.owned_requests(PQ.ring_source(rank, s, N_RANKS), B, N_RANKS) for s in range(N_RANKS)]
        mine = slice(rank * bq, (rank + 1) * bq)
        assert np.array_equal(np.isneginf(lse), np.isneginf(rl[mine]))
        fin = np.isfinite(rl[mine])
        assert np.allclose(o, ro[mine], atol=1e-12, rtol=0)
        assert np.allclose(lse[fin], rl[mine][fin], atol=1e-12, rtol=0)
        assert np.allclose(o, po[mine], atol=1e-13, rtol=0)
    assert np.all(np.isneginf(rl[1])) and np.all(np.isfinite(rl[2]))
