"""The two context-parallel exchanges whose single-GPU form is a split of one call, run as
real two-rank groups on the CPU (gloo, world_size 2, 127.0.0.1), with the fp64 oracle as
each rank's attention.

KVP decode ("Helix Parallelism: Why Tensor Parallelism Hits a Wall at Million-Token
Context", section "Sharding the sequence instead"): every rank holds one contiguous shard
of every sequence's KV, computes the partial of all query heads over it, and one
All-to-All over the query-head axis gives each rank every shard's partial for its own
slab of heads, which it merges exactly by the lse.  The ranks run the package's exchange
step (mla_decode_attention_gqa_gb300.kvp.kvp_decode_step, the function bench.py's KVP mode
runs over NCCL) with the oracle as the attention and the merge.  The test also checks that
a rank's send buffer, slabs side by side, is its split of the single-GPU partial layout
[split][B][Tq][Hq][dv], the layout attn_partial writes.

Pass-KV prefill ("Context Parallelism for Scalable Million-Token Inference", section
"Pass-KV keeps queries local and circulates keys and values"): every rank keeps its query
chunk, the KV chunks travel the ring (each rank passes the block it holds to rank + 1),
and the partial of every step is merged into a running (o, lse), as attn_ring_step does;
masked by original position, in the contiguous and the zigzag layout.
"""

import os
import socket
import sys

import numpy as np
import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
N_RANKS = 2
NO_CAUSAL = 1 << 62

# KVP decode problem: B sequences, one decode row each, S tokens in N contiguous shards
B, HQ, HKV, D, S, SCALE = 3, 8, 2, 8, 12, 0.35
# pass-KV problem: one sequence of S_P tokens in N_RANKS chunks (contiguous) or 2 N blocks (zigzag)
S_P, HQ_P, HKV_P = 16, 4, 2


def _kvp_problem():
    rng = np.random.default_rng(7)
    q = rng.standard_normal((B, 1, HQ, D))
    k = rng.standard_normal((B, HKV, S, D))
    v = rng.standard_normal((B, HKV, S, D))
    lens = [S, 4, 9]  # sequence 1 ends inside shard 0: shard 1 holds nothing of it
    return q, k, v, lens


def _passkv_problem():
    rng = np.random.default_rng(11)
    q = rng.standard_normal((1, S_P, HQ_P, D))
    k = rng.standard_normal((1, HKV_P, S_P, D))
    v = rng.standard_normal((1, HKV_P, S_P, D))
    return q, k, v


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _kvp_worker(rank, port, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import oracle
    from mla_decode_attention_gqa_gb300 import kvp

    dist.init_process_group("gloo", rank=rank, world_size=N_RANKS)
    q, k, v, lens = _kvp_problem()
    m = S // N_RANKS
    lo = rank * m
    # this rank's shard: tokens [lo, lo + m) of every sequence, and how many of them exist
    k_loc, v_loc = k[:, :, lo:lo + m], v[:, :, lo:lo + m]
    lens_loc = [min(max(n - lo, 0), m) for n in lens]

    def partial(qs, ks, vs, sl, k_scale, v_scale, scale, scale_block, out_o, out_l):  # the oracle as the attention
        o, lse = oracle.split_attention(qs.numpy(), ks.numpy(), vs.numpy(), sl.tolist(), [[0, m]] * B, NO_CAUSAL,
                                        scale)
        out_o.copy_(torch.from_numpy(o))
        out_l.copy_(torch.from_numpy(lse))

    def merge(o, lse):
        mo, ml = oracle.merge_lse(o.numpy(), lse.numpy())
        return torch.from_numpy(mo), torch.from_numpy(ml)

    # the package's exchange step: partials straight into the All-to-All send buffer, one
    # slab per destination rank, then the exchange and the merge of this rank's heads
    mo, ml, (send_o, send_l, _, _) = kvp.kvp_decode_step(
        torch.from_numpy(q), torch.from_numpy(np.ascontiguousarray(k_loc)), torch.from_numpy(np.ascontiguousarray(v_loc)),
        torch.tensor(lens_loc, dtype=torch.int32), softmax_scale=SCALE, partial=partial, merge=merge)
    # the send buffer's slabs side by side over the head axis: this rank's partial of every head
    o = np.concatenate([send_o[s].numpy() for s in range(N_RANKS)], axis=2)
    lse = np.concatenate([send_l[s].numpy() for s in range(N_RANKS)], axis=2)
    dist.barrier()
    dist.destroy_process_group()
    out_q.put((rank, o, lse, mo.numpy(), ml.numpy()))


def _passkv_worker(rank, port, layout, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist

    import oracle
    from mla_decode_attention_gqa_gb300 import workloads as W

    dist.init_process_group("gloo", rank=rank, world_size=N_RANKS)
    q, k, v = _passkv_problem()
    N = N_RANKS
    nxt, prv = (rank + 1) % N, (rank - 1) % N
    my_pos = W.layout_positions(layout, S_P, N, rank)
    q_loc = q[:, my_pos]
    held_src = rank
    held_k = torch.from_numpy(np.ascontiguousarray(k[:, :, my_pos]))
    held_v = torch.from_numpy(np.ascontiguousarray(v[:, :, my_pos]))
    n_loc = len(my_pos)
    o_acc = lse_acc = None
    sources = []
    for s in range(N):
        sources.append(held_src)
        kv_pos = W.layout_positions(layout, S_P, N, held_src)
        o, lse = oracle.split_attention(q_loc, held_k.numpy(), held_v.numpy(), [n_loc], [[0, n_loc]], 0, SCALE,
                                        q_positions=[my_pos], k_positions=[kv_pos])
        if o_acc is None:
            o_acc, lse_acc = o[0], lse[0]
        else:  # the online merge of the running output with this step's partial
            o_acc, lse_acc = oracle.merge_lse(np.stack([o_acc, o[0]]), np.stack([lse_acc, lse[0]]))
        if s + 1 < N:  # the ring hop: pass the held block on, take the previous rank's
            rk, rv = torch.empty_like(held_k), torch.empty_like(held_v)
            src = torch.tensor([held_src], dtype=torch.int64)
            rsrc = torch.empty_like(src)
            reqs = [dist.isend(held_k, nxt), dist.isend(held_v, nxt), dist.isend(src, nxt),
                    dist.irecv(rk, prv), dist.irecv(rv, prv), dist.irecv(rsrc, prv)]
            for r in reqs:
                r.wait()
            held_k, held_v, held_src = rk, rv, int(rsrc.item())
    dist.barrier()
    dist.destroy_process_group()
    out_q.put((rank, sources, my_pos, o_acc, lse_acc))


def _run(target, *args):
    ctx = mp.get_context("spawn")
    out_q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=target, args=(r, port, *args, out_q)) for r in range(N_RANKS)]
    for p in procs:
        p.start()
    res = sorted((out_q.get(timeout=240) for _ in procs), key=lambda x: x[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return res


def test_two_rank_kvp_decode_all_to_all_over_heads():
    sys.path.insert(0, ROOT)
    import oracle

    res = _run(_kvp_worker)
    q, k, v, lens = _kvp_problem()
    ro, rl = oracle.full_attention(q, k, v, lens, NO_CAUSAL, SCALE)
    # the single-GPU form: one call with one split per shard
    m = S // N_RANKS
    po, pl = oracle.split_attention(q, k, v, lens, [[0, m, S]] * B, NO_CAUSAL, SCALE)
    hs = HQ // N_RANKS
    for rank, o, lse, mo, ml in res:
        # the rank's send buffer is split `rank` of the [split][B][Tq][Hq][dv] layout
        assert np.allclose(o, po[rank], atol=1e-13, rtol=0)
        assert np.array_equal(np.isneginf(lse), np.isneginf(pl[rank]))
        heads = slice(rank * hs, (rank + 1) * hs)
        assert np.allclose(mo, ro[:, :, heads], atol=1e-12, rtol=0)
        assert np.allclose(ml, rl[:, :, heads], atol=1e-12, rtol=0)
    # sequence 1 lies wholly in shard 0: shard 1's partial is empty and neutral
    assert np.all(np.isneginf(res[1][2][1]))


@pytest.mark.parametrize("layout", ["contiguous", "zigzag"])
def test_two_rank_passkv_ring_prefill(layout):
    sys.path.insert(0, ROOT)
    import oracle

    res = _run(_passkv_worker, layout)
    q, k, v = _passkv_problem()
    ro, rl = oracle.full_attention(q, k, v, [S_P], 0, SCALE)  # causal over original positions
    for rank, sources, my_pos, o, lse in res:
        # the block held at ring step s started on rank (rank - s) mod N
        assert sources == [(rank - s) % N_RANKS for s in range(N_RANKS)]
        assert np.allclose(o, ro[:, my_pos], atol=1e-12, rtol=0)
        assert np.allclose(lse, rl[:, my_pos], atol=1e-12, rtol=0)


def test_head_slabs_cover_whole_groups_or_lie_inside_one():
    sys.path.insert(0, ROOT)
    from mla_decode_attention_gqa_gb300 import kvp

    # Helix dense decode on 8 ranks: one KV head (16 query heads) per rank
    assert kvp.head_slabs(128, 8, 8) == [((16 * s, 16 * s + 16), (s, s + 1)) for s in range(8)]
    # 2 ranks: four KV heads per slab
    assert kvp.head_slabs(128, 8, 2) == [((0, 64), (0, 4)), ((64, 128), (4, 8))]
    # the MLA latent (one KV head) on 8 ranks: every slab inside the one group
    assert kvp.head_slabs(128, 1, 8)[3] == ((48, 64), (0, 1))
    with pytest.raises(ValueError):
        kvp.head_slabs(24, 8, 12)  # groups of 3 heads, slabs of 2: a slab would straddle two groups
