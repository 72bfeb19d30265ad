"""bench.py's multi-rank host logic on CPU: two gloo ranks (world_size 2) on 127.0.0.1.

Every rank runs an independent replica; the timed region is bracketed by barriers, the
step time is the max over ranks and the KV bytes are summed over ranks; the reference
arm prints its line on rank 0 only."""

import io
import contextlib
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import argparse

    import torch.distributed as dist

    import bench
    from mla_decode_attention_gqa_gb300 import workloads as W

    ws_, r, _ = bench.dist_setup()
    mx = bench.max_over_ranks(float(10 * (rank + 1)), ws_)
    sm = bench.sum_over_ranks(float(rank + 1), ws_)
    bench.barrier(ws_)
    args = argparse.Namespace(steps=1, warmup=1)
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.reference_arm(args, W.TINY_GQA, ws_, r)
    dist.destroy_process_group()
    q.put((r, ws_, mx, sm, buf.getvalue()))


def test_two_gloo_ranks_max_sum_and_rank0_output():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(rk, 2, port, q)) for rk in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=240) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, ws0, mx0, sm0, out0), (r1, ws1, mx1, sm1, out1) = res
    assert (r0, r1) == (0, 1) and ws0 == ws1 == 2
    assert mx0 == mx1 == 20.0  # max over ranks of 10, 20
    assert sm0 == sm1 == 3.0  # sum over ranks of 1, 2
    assert '"impl": "reference"' in out0 and out1 == ""
