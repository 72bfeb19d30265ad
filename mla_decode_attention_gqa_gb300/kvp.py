"""KV parallelism (KVP) across ranks: the exchange step of a sequence-sharded decode.

"Helix Parallelism: Why Tensor Parallelism Hits a Wall at Million-Token Context", section
"Sharding the sequence instead": each of N ranks holds one contiguous shard of every
sequence's KV cache, computes the partial attention (normalised output plus log-sum-exp)
of every query head over its shard, and one All-to-All over the query-head axis hands each
rank every shard's partial for its own slab of Hq / N heads, which it merges exactly by
the lse ("现代大模型推理并行策略总览", section "Decode CP：固定 KV Cache 分片，归并局部结果").

``kvp_decode_step`` is that step for one rank.  The partials go straight into the
All-to-All send buffer [N][B][Tq][Hq/N][dv]: slab s (the heads rank s owns) is computed by
its own call over the KV heads those query heads read, so no permutation copy is needed and,
when every slab covers whole KV groups, every KV byte of the shard is read once.  The
attention and the merge are arguments: on GPUs they default to this library's
``attn_partial`` and ``attn_merge_lse`` over ``torch.distributed`` (NCCL); a caller may pass
other implementations (the CPU tests run the same exchange over gloo with the fp64 oracle).
With a world of one rank the All-to-All is the identity and no process group is needed.
"""

import torch


def head_slabs(Hq, Hkv, n_ranks):
    """[(query heads [lo, hi), KV heads [lo, hi))] of the slab each rank owns.

    The query heads are split into n_ranks equal contiguous slabs; slab s reads the KV heads
    its query heads map to (contiguous groups of G = Hq / Hkv).  A slab must cover whole
    groups (G divides Hq / n_ranks) or lie inside one group (Hq / n_ranks divides G)."""
    if Hq % n_ranks:
        raise ValueError("Hq must be a multiple of the number of KVP ranks")
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    G, hs = Hq // Hkv, Hq // n_ranks
    if hs % G and G % hs:
        raise ValueError("each rank's head slab must cover whole KV groups or lie inside one")
    return [((s * hs, (s + 1) * hs), ((s * hs) // G, ((s + 1) * hs - 1) // G + 1)) for s in range(n_ranks)]


def _library_partial(q, k, v, seq_lens, k_scale, v_scale, softmax_scale, scale_block, out_o, out_l):
    from . import attn_partial

    S = k.shape[2]
    bounds = torch.tensor([[0, S]] * q.shape[0], dtype=torch.int32, device=q.device)
    attn_partial(q, k, v, seq_lens, bounds, k_scale=k_scale, v_scale=v_scale, softmax_scale=softmax_scale,
                 scale_block=scale_block, out_partial=out_o, lse_partial=out_l)


def _library_merge(o_parts, l_parts):
    from . import attn_merge_lse

    return attn_merge_lse(o_parts, l_parts)


def slab_scales(k_scale, v_scale, Hq, Hkv, n_ranks):
    """fp8 block scales [B, Hkv, n_blk] cut into the contiguous per-slab pieces the partial
    calls take (once per cache, not per step)."""
    return [(k_scale[:, g0:g1].contiguous(), v_scale[:, g0:g1].contiguous())
            for _, (g0, g1) in head_slabs(Hq, Hkv, n_ranks)]


def kvp_decode_step(q, k_shard, v_shard, seq_lens, *, group=None, k_scale=None, v_scale=None, softmax_scale=None,
                    scale_block=64, partial=None, merge=None, buffers=None, scales=None):
    """One KVP decode step on this rank.

    q        [B, Tq, Hq, dk]: every query head of every sequence (the same on every rank)
    k_shard, v_shard  [B, Hkv, S_loc, d]: this rank's shard of every sequence's cache
    seq_lens [B] int32: tokens of each sequence held in this shard (0 allowed)
    group    torch.distributed process group (None: the default group, or a world of one)
    partial  fn(q, k, v, seq_lens, k_scale, v_scale, softmax_scale, scale_block, out_o, out_l)
             writing the partial of q over (k, v) into out_o [1, B, Tq, h, dv] and out_l
             [1, B, Tq, h] (default: this library's attn_partial, one split over the shard)
    merge    fn(o_parts [N, B, Tq, h, dv], l_parts [N, B, Tq, h]) -> (out, lse) (default:
             this library's attn_merge_lse)
    buffers  optional (send_o, send_l, recv_o, recv_l) to reuse across steps
    scales   fp8: optional slab_scales(k_scale, v_scale, ...) made once, instead of cutting
             k_scale / v_scale per step

    Returns (out [B, Tq, Hq/N, dv], lse [B, Tq, Hq/N]) for the heads this rank owns (slab
    rank), and the send / receive buffers."""
    import torch.distributed as dist

    world = dist.get_world_size(group) if dist.is_available() and dist.is_initialized() else 1
    rank = dist.get_rank(group) if world > 1 else 0
    B, Tq, Hq, _ = q.shape
    Hkv, dv = k_shard.shape[1], v_shard.shape[3]
    slabs = head_slabs(Hq, Hkv, world)
    hs = Hq // world
    if buffers is None:
        pdt = torch.float64 if q.dtype == torch.float64 else torch.float32  # fp32 partials; fp64 for an fp64 oracle
        send_o = torch.empty((world, B, Tq, hs, dv), dtype=pdt, device=q.device)
        send_l = torch.empty((world, B, Tq, hs), dtype=pdt, device=q.device)
        recv_o, recv_l = torch.empty_like(send_o), torch.empty_like(send_l)
    else:
        send_o, send_l, recv_o, recv_l = buffers
    partial = partial or _library_partial
    merge = merge or _library_merge
    if scales is None and k_scale is not None:
        scales = slab_scales(k_scale, v_scale, Hq, Hkv, world)
    for s, ((h0, h1), (g0, g1)) in enumerate(slabs):
        ks, vs = scales[s] if scales is not None else (None, None)
        partial(q[:, :, h0:h1], k_shard[:, g0:g1], v_shard[:, g0:g1], seq_lens, ks, vs, softmax_scale, scale_block,
                send_o[s:s + 1], send_l[s:s + 1])
    if world > 1:
        dist.all_to_all_single(recv_o, send_o, group=group)
        dist.all_to_all_single(recv_l, send_l, group=group)
    else:
        recv_o, recv_l = send_o, send_l
    out, lse = merge(recv_o, recv_l)
    return out, lse, (send_o, send_l, recv_o, recv_l)
