#!/usr/bin/env python3
"""Benchmark: split-KV decode attention on GB300 (one JSON line on stdout, rank 0).

Default workload: the Helix dense-model decode layer -- B=8, Hq=128, Hkv=8 (group 16),
d=128, S=131072 bf16 KV per sequence, one new token per sequence, no split (KVP=1),
bf16 output + fp32 LSE.  One step = one gqa_decode_attn call (split-KV partial kernel
+ LSE merge) over the resident KV cache.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--config NAME]
                  [--extras auto|none|NAME,...]

On one GPU the default run then measures, each in its own timed region with its own clock
record and oracle parity sample, the other workloads the metric is quoted on: the
long-context KVP=8 decode at S=2^20 with fp8-e4m3 KV, the MLA absorbed decode, and the
ring pass-KV prefill chunk as one fused call and as eight ring steps.  They are reported
under "workloads" in the same JSON line (time per layer, the dominant kernel's time, its
HBM and bf16-tensor fractions of the measured peaks).

Multi-GPU (torchrun): every rank runs an independent replica of the workload (the
attention of a layer shards into independent problems; no data-path collective), the
timed region is bracketed by barriers, the max time over ranks is taken, and value is
the KV bytes of all ranks over that time ("scaling": "weak").

The reference arm (--impl reference) times the fp64 CPU oracle on a bounded sample of
the same workload on this host's cores; it is a deliberately slow correctness
baseline, not a competitor.
"""

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

# the oracle's BLAS uses every core this process may run on; state it explicitly
_CORES = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
os.environ.setdefault("OPENBLAS_NUM_THREADS", str(_CORES))
os.environ.setdefault("OMP_NUM_THREADS", str(_CORES))

import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from mla_decode_attention_gqa_gb300 import workloads as W  # noqa: E402
from mla_decode_attention_gqa_gb300 import roofline as RL  # noqa: E402

METRIC = "decode attn µs/layer & KV-read HBM GB/s (fraction of GB300 peak) at S=128K/1M"
PEAKS_PATH = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_PATH = os.path.join(ROOT, "profiles", "traffic.json")
# sources a traffic record was measured with, when the record does not list its own
KERNEL_SOURCES = ["mla_decode_attention_gqa_gb300/csrc/gqa_partial.cu", "mla_decode_attention_gqa_gb300/csrc/skv_common.cuh"]


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def config_of(w, ws=1):
    """The `config` object both arms print: the workload by name and sizes."""
    esz = 1 if w.kv_dtype == "fp8_e4m3" else 2
    alloc = w.B * w.Hkv * w.S * (w.dk if w.mla else w.dk + w.dv) * esz
    return {"workload": w.name, "B": w.B, "Tq": w.Tq, "Hq": w.Hq, "Hkv": w.Hkv, "dk": w.dk, "dv": w.dv, "S": w.S,
            "kv_dtype": w.kv_dtype, "n_split": w.n_split, "ragged": w.ragged,
            "l2": ("no flush: a tensor-bound prefill chunk (%.2f GB of KV, re-read from L2 per query tile by "
                   "design)" % (alloc / 1e9)) if w.Tq > 1 else
                  ("no flush: each step streams the resident KV cache (%.2f GB allocated), far above the 129 MB L2"
                   % (alloc / 1e9)) if alloc > 4 * 129e6 else
                  ("KV (%.4f GB) fits in L2: a parity-size workload, not a bench line" % (alloc / 1e9)),
            "parallelism": f"replicas x{ws}",
            **({"layout": w.layout, "query_rank": w.cp_rank} if w.layout != "contiguous" else {}),
            **({"paged": True, "block_len": w.block_len} if w.paged else {}),
            **({"ring_steps": w.n_split, "step_api": "attn_ring_step"} if w.ring_steps else {}),
            **({"passq_ranks": w.passq_ranks, "decode_tokens": w.passq_decode_tokens,
                "step_api": "gqa_decode_attn_passq"} if w.passq_ranks else {})}


def workload_by_name(name):
    for w in W.WORKLOADS:
        if w.name == name:
            return w
    raise SystemExit(f"unknown workload {name}; choose from {[w.name for w in W.WORKLOADS]}")


FALLBACK_BF16_TFLOPS = 1900.0


def hbm_peak():
    try:
        with open(PEAKS_PATH) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def bf16_peak():
    """Dense bf16 tensor peak (burst: the kernel is timed on its own, not in a long loop)."""
    try:
        with open(PEAKS_PATH) as f:
            return float(json.load(f)["bf16_tflops"]), "measured (burst)"
    except Exception:
        return FALLBACK_BF16_TFLOPS, "fallback"


def kernel_source_sha(sources=None):
    h = hashlib.sha256()
    for rel in sources or KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload_name):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary, if the
    kernel sources still match the ones that were profiled (else None)."""
    try:
        with open(TRAFFIC_PATH) as f:
            rec = json.load(f)
        e = rec[workload_name]
        if e.get("kernel_source_sha") != kernel_source_sha(e.get("kernel_sources")):
            return None
        v = e.get("dram_bytes_per_launch")
        return None if v is None else float(v)
    except Exception:
        return None


class ClockSampler:
    """Samples nvidia-smi SM clocks and throttle reasons while the timed region runs."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu_index = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=2)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(x, ws):
    if ws == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, ws):
    if ws == 1:
        return x
    import torch.distributed as dist

    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# --------------------------------------------------------------------------- CPU oracle leg

def launches_per_step(w):
    """This library's kernel launches in one timed step of a workload (its routing):
    the tensor-core shapes (bf16, d = 128, the group dividing 128, >= 128 rows per KV
    head) run one fused kernel; every other call is a partial kernel plus the merge."""
    G = w.Hq // w.Hkv
    tensor_core = (not w.mla and w.kv_dtype == "bf16" and w.dk == 128 and w.dv == 128 and 128 % G == 0
                   and w.Tq * G >= 128)
    if w.ring_steps:  # tensor core: one kernel per step, merging in its epilogue; otherwise the
        # block's partial per step and a two-way merge after the first
        return w.n_split if tensor_core else 2 * w.n_split - 1
    return 1 if tensor_core else 2


# Bounds on one oracle sample, so that a sample takes seconds rather than minutes: a decode
# group longer than ORACLE_MAX_TOKENS tokens is cut to its first ones (time and bytes both
# scale with the tokens), and a query chunk of more than ORACLE_MAX_ROWS rows computes every
# (Tq / ORACLE_MAX_ROWS)-th row, its KV bytes credited in proportion to the rows computed.
ORACLE_MAX_TOKENS = 131072
ORACLE_MAX_ROWS = 256


def oracle_sample(w, budget_s=12.0, max_groups=None):
    """Time the fp64 oracle on bounded samples of (batch, KV head) groups of the workload
    until the budget is spent; returns (KV bytes credited, seconds, groups, tokens per
    group, query rows computed per group)."""
    import numpy as np
    import oracle

    gen = torch.Generator().manual_seed(w.seed)
    G = w.Hq // w.Hkv
    if w.passq_ranks:
        return _oracle_sample_passq(w, gen, budget_s, max_groups)
    S = min(w.S, ORACLE_MAX_TOKENS) if w.Tq == 1 else w.S
    bounds = [min(x, S) for x in w.split_bounds()[0]]
    rows = np.arange(w.Tq) if w.Tq <= ORACLE_MAX_ROWS else np.arange(0, w.Tq, w.Tq // ORACLE_MAX_ROWS)
    pos = {}
    if w.layout != "contiguous":  # tokens stored in a zigzag / striped layout
        pos = {"q_positions": [np.asarray(W.layout_positions(w.layout, w.S, w.n_split, w.cp_rank))[rows]],
               "k_positions": [[p for r in range(w.n_split) for p in W.layout_positions(w.layout, w.S, w.n_split, r)]]}
    elif len(rows) < w.Tq:  # a subset of the chunk's rows: give their positions explicitly
        pos = {"q_positions": [w.causal_offset + rows], "k_positions": [np.arange(S)]}
    done_bytes, elapsed, groups = 0.0, 0.0, 0
    while elapsed < budget_s and (max_groups is None or groups < max_groups):
        q = torch.randn((1, w.Tq, G, w.dk), generator=gen).to(torch.bfloat16)
        k = torch.randn((S, w.dk), generator=gen).to(torch.bfloat16)
        v = torch.randn((S, w.dv), generator=gen).to(torch.bfloat16)
        if w.kv_dtype == "fp8_e4m3":
            kc, ks = W._quantize_e4m3_blocks(k.float(), w.scale_block)
            vc, vs = W._quantize_e4m3_blocks(v.float(), w.scale_block)
        t0 = time.perf_counter()
        qf = oracle.bf16_bits_to_f64(q.view(torch.int16).numpy())[:, rows]
        if w.kv_dtype == "fp8_e4m3":
            kf = oracle.dequant_e4m3_blocks(kc.numpy(), ks.numpy(), w.scale_block)
            vf = oracle.dequant_e4m3_blocks(vc.numpy(), vs.numpy(), w.scale_block)
        else:
            kf = oracle.bf16_bits_to_f64(k.view(torch.int16).numpy())
            vf = oracle.bf16_bits_to_f64(v.view(torch.int16).numpy())
        o, lse = oracle.split_attention(qf, kf[None, None], vf[None, None], [S], [bounds], w.causal_offset, w.scale,
                                        **pos)
        oracle.merge_lse(o, lse)
        elapsed += time.perf_counter() - t0
        done_bytes += (RL.kv_bytes(1, w.dk, w.dv, w.kv_dtype, [S], [bounds], mla=w.mla, scale_block=w.scale_block)
                       * len(rows) / w.Tq)
        groups += 1
    return done_bytes, elapsed, groups, S, len(rows)


def oracle_sample_text(w, groups, tokens, rows):
    """What one oracle sample covered, in words."""
    tok = f"{tokens} tokens" + (f" (the first {tokens} of {w.S})" if tokens < w.S else "")
    row = f"{rows} row(s)" if rows == w.Tq else f"{rows} of {w.Tq} rows (every {w.Tq // rows}th)"
    ring = f", through the {w.passq_ranks}-rank pass-Q ring" if w.passq_ranks else ""
    return f"{groups} (batch, KV head) group(s) of {tok} x {row} x {w.Hq // w.Hkv} heads{ring}"


def _oracle_sample_passq(w, gen, budget_s, max_groups):
    """Pass-Q: one (request, KV head) group of S tokens spread over the N ranks as the
    workload spreads them, its query block padded with N - 1 empty requests (the padding
    of a batch of one to the group size), run through the oracle's ring, return and merge;
    returns like oracle_sample."""
    import numpy as np
    import oracle

    N, G = w.passq_ranks, w.Hq // w.Hkv
    lens = W.passq_shard_lens(W.scaled(w, B=N), [w.S] + [0] * (N - 1))
    S_loc = max(lens[r][0] for r in range(N))
    done_bytes, elapsed, groups = 0, 0.0, 0
    while elapsed < budget_s and (max_groups is None or groups < max_groups):
        q = torch.randn((N, 1, G, w.dk), generator=gen).to(torch.bfloat16)
        k = torch.randn((N, 1, S_loc, w.dk), generator=gen).to(torch.bfloat16)  # request 0 on each rank
        v = torch.randn((N, 1, S_loc, w.dv), generator=gen).to(torch.bfloat16)
        t0 = time.perf_counter()
        qf = oracle.bf16_bits_to_f64(q.view(torch.int16).numpy())
        kf = np.zeros((N, N, 1, S_loc, w.dk))  # the empty requests' rows are never touched
        vf = np.zeros((N, N, 1, S_loc, w.dv))
        kf[:, 0] = oracle.bf16_bits_to_f64(k.view(torch.int16).numpy())
        vf[:, 0] = oracle.bf16_bits_to_f64(v.view(torch.int16).numpy())
        oracle.passq_decode(qf, kf, vf, lens, w.scale)
        elapsed += time.perf_counter() - t0
        done_bytes += RL.kv_bytes(1, w.dk, w.dv, "bf16", [w.S], [[0, w.S]])
        groups += 1
    return done_bytes, elapsed, groups, w.S, 1


def oracle_parity(w, par):
    """Max-abs error of the timed steps' output and lse for batch 0, KV head 0 against the
    fp64 oracle on the same bytes (the parity sample of the bench's own result).  The
    oracle walks the group one split at a time (attention of the sampled rows over the
    split's tokens, then the exact merge of the splits), so that a group of 2^20 tokens
    needs one split's rows in float64 at a time."""
    if "error" in par:
        return par
    try:
        import numpy as np
        import oracle

        n_tok, rows = par["n_tok"], np.asarray(par["rows"])
        qf = oracle.bf16_bits_to_f64(par["q"].view(torch.int16).numpy())  # [R, G, dk]
        R, G, dk = qf.shape
        bounds = [min(x, n_tok) for x in w.split_bounds()[0]]
        q_pos = np.repeat(w.causal_offset + rows.astype(np.int64), G) if w.causal_offset != W.NO_CAUSAL else None
        o_parts, l_parts = [], []
        for j in range(len(bounds) - 1):
            lo, hi = max(bounds[j], 0), bounds[j + 1]
            if hi <= lo:
                continue
            if par["ks"] is not None:
                kf = oracle.dequant_e4m3_blocks(par["k"][lo:hi].numpy(), par["ks"].numpy(), w.scale_block, t0=lo)
                vf = oracle.dequant_e4m3_blocks(par["v"][lo:hi].numpy(), par["vs"].numpy(), w.scale_block, t0=lo)
            else:
                kf = oracle.bf16_bits_to_f64(par["k"][lo:hi].view(torch.int16).numpy())
                vf = oracle.bf16_bits_to_f64(par["v"][lo:hi].view(torch.int16).numpy())
            kv_pos = np.arange(lo, hi) if q_pos is not None else None
            o, l = oracle.attend(qf.reshape(R * G, dk), kf, vf, w.scale, q_pos, kv_pos)
            o_parts.append(o)
            l_parts.append(l)
        if o_parts:
            mo, ml = oracle.merge_lse(np.stack(o_parts), np.stack(l_parts))
        else:
            mo, ml = np.zeros((R * G, w.dv)), np.full(R * G, -np.inf)
        mo, ml = mo.reshape(R, G, w.dv), ml.reshape(R, G)
        got_l = par["lse"].numpy().astype(np.float64)
        fin = np.isfinite(ml)
        return {"sample": f"batch 0, KV head 0: {R} of {w.Tq} row(s) x {G} heads, {n_tok} tokens",
                "out_max_abs_err": float(np.max(np.abs(par["out"].numpy() - mo))),
                "lse_max_abs_err": float(np.max(np.abs(got_l[fin] - ml[fin]))) if fin.any() else 0.0,
                "empty_rows_match": bool(np.array_equal(np.isneginf(got_l), ~fin))}
    except Exception as e:  # the parity sample must never cost the bench line
        return {"error": f"{type(e).__name__}: {e}"[:200]}


def reference_arm(args, w, ws, rank):
    if rank != 0:
        return
    steps = []
    bytes_total, secs_total = 0, 0.0
    sample = None
    for i in range(args.warmup + args.steps):
        b, s, g, t, r = oracle_sample(w, budget_s=float("inf"), max_groups=1)
        if i >= args.warmup:
            steps.append(s)
            bytes_total += b
            secs_total += s
            sample = oracle_sample_text(w, g, t, r) + " per step"
    gbs = bytes_total / secs_total / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * secs_total / len(steps), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, ws),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": _CORES, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- GPU arm

# Workloads measured after the main one in the default run (one GPU): the long-context KVP
# decode at S = 2^20 (fp8), the MLA absorbed decode, and the ring-prefill chunk both as one
# fused call and as eight pass-KV ring steps.  Each gets its own timed region, clock record
# and parity sample, reported under "workloads" in the same JSON line.
EXTRA_WORKLOADS = (W.HELIX_KVP8_FP8_1M.name, W.MLA_ABSORBED.name, W.RING_PREFILL.name, W.RING_PREFILL_STEPS.name)

# The parity sample of a decode group holds its whole sequence up to this many tokens (the
# oracle then walks it one split at a time, so host memory stays at one split's rows).
PARITY_MAX_TOKENS = 1 << 20


def measure(args, w, ws, rank, local, want_e2e, want_parity):
    """One workload on this rank's GPU: warm-up, the two timed passes (pass 1 gives value
    and ms_per_step, pass 2 the per-step spread and the library's own kernel times), the
    clocks sampled during both, and optionally the
    end-to-end run from pinned host buffers and one (batch, KV head) group's inputs and
    result for the oracle parity sample.  Returns a dict; time is the max over ranks."""
    import mla_decode_attention_gqa_gb300 as skv

    dev = torch.device("cuda", local)
    t0 = time.time()
    inp = W.make_inputs(w, dev)
    torch.cuda.synchronize()
    log(f"[rank {rank}] {w.name}: inputs ready in {time.time() - t0:.1f}s")
    kw = dict(k_scale=inp["k_scale"], v_scale=inp["v_scale"], softmax_scale=w.scale, scale_block=w.scale_block)
    bounds = inp["split_bounds"]  # host copy: the algorithmic byte and flop counts
    # the library reads the split bounds in device memory: uploaded once, outside the timed region
    inp["split_bounds_dev"] = bounds_dev = torch.tensor(bounds, dtype=torch.int32, device=dev)
    kv_bytes = RL.kv_bytes(w.Hkv, w.dk, w.dv, w.kv_dtype, inp["seq_lens_host"], bounds, mla=w.mla,
                           scale_block=w.scale_block)
    positional = inp["q_pos"] is not None  # zigzag / striped storage: the *_pos entry point
    if w.passq_ranks:  # pass-Q: every rank's resident shard of every request, once
        flat = [n for r in inp["shard_lens_host"] for n in r]
        S_loc = inp["k_shards"].shape[2]
        kv_bytes = RL.kv_bytes(w.Hkv, w.dk, w.dv, w.kv_dtype, flat, [[0, S_loc]] * len(flat),
                               scale_block=w.scale_block)
        flops = RL.attn_flops(1, w.Hq, w.dk, w.dv, flat, [[0, S_loc]] * len(flat))
    elif positional:
        flops = RL.attn_flops_positions(w.Hq, w.dk, w.dv, inp["seq_lens_host"], bounds, inp["q_pos_host"],
                                        inp["k_pos_host"])
    else:
        flops = RL.attn_flops(w.Tq, w.Hq, w.dk, w.dv, inp["seq_lens_host"], bounds, w.causal_offset)
    out = torch.empty((w.B, w.Tq, w.Hq, w.dv), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.Tq, w.Hq), dtype=torch.float32, device=dev)

    if w.paged:  # the pages are the cache; the logical copy is not needed here
        for key in ("k", "v", "k_scale", "v_scale"):
            inp[key] = None
        torch.cuda.empty_cache()
        kw = dict(k_scale=inp.get("k_scale_pages"), v_scale=inp.get("v_scale_pages"), softmax_scale=w.scale,
                  scale_block=w.scale_block)

    o_acc = lse_acc = None
    if w.ring_steps:  # pass-KV ring: every step's KV block in its own buffer
        C = w.S // w.n_split
        ring_blocks = [(inp["k"][:, :, j * C:(j + 1) * C].contiguous(), inp["v"][:, :, j * C:(j + 1) * C].contiguous(),
                        torch.clamp(inp["seq_lens"] - j * C, 0, C).to(torch.int32)) for j in range(w.n_split)]
        o_acc = torch.empty((w.B, w.Tq, w.Hq, w.dv), dtype=torch.float32, device=dev)
        lse_acc = torch.empty((w.B, w.Tq, w.Hq), dtype=torch.float32, device=dev)

    def ring_run(q, blocks):
        C = w.S // w.n_split
        for j, (kb, vb, sl) in enumerate(blocks):
            skv.attn_ring_step(q, kb, vb, sl, o_acc, lse_acc, w.causal_offset - j * C, first=(j == 0),
                               softmax_scale=w.scale)

    def step():
        if w.passq_ranks:
            skv.gqa_decode_attn_passq(inp["q"], inp["k_shards"], inp["v_shards"], inp["shard_lens"],
                                      k_scale=inp["k_shard_scale"], v_scale=inp["v_shard_scale"],
                                      softmax_scale=w.scale, scale_block=w.scale_block, out=out, lse=lse)
        elif w.ring_steps:
            ring_run(inp["q"], ring_blocks)
        elif w.paged:
            skv.gqa_decode_attn_paged(inp["q"], inp["k_pages"], inp["v_pages"], inp["seq_lens"], bounds_dev,
                                      inp["block_table"], w.causal_offset, out=out, lse=lse, **kw)
        elif positional:
            skv.gqa_decode_attn_pos(inp["q"], inp["k"], inp["v"], inp["seq_lens"], bounds_dev, inp["q_pos"],
                                    inp["k_pos"], out=out, lse=lse, **kw)
        else:
            skv.gqa_decode_attn(inp["q"], inp["k"], inp["v"], inp["seq_lens"], bounds_dev, w.causal_offset, out=out,
                                lse=lse, **kw)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if skv.device_error() != 0:
        raise RuntimeError(f"{w.name}: a kernel reported a timed-out wait during warm-up")

    stream = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    sampler = ClockSampler(local)
    barrier(ws)
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)  # let the sampler start before the timed region
    start_all = torch.cuda.Event(enable_timing=True)
    end_all = torch.cuda.Event(enable_timing=True)
    # pass 1 (value, ms_per_step): the K steps bracketed by one event pair and nothing else
    start_all.record(stream)
    for i in range(args.steps):
        step()
    end_all.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    # pass 2 (roofline, per-step spread): the same K steps with an event pair around every
    # step and the library's own event pair around each attention kernel, on the launch
    # stream.  These events lengthen a step by ~15 us, so they stay out of pass 1.
    skv.kernel_timing(True)
    for i in range(args.steps):
        ev[i][0].record(stream)
        step()
        ev[i][1].record(stream)
    skv.kernel_timing(False)
    torch.cuda.synchronize()
    barrier(ws)
    clocks = sampler.stop()
    total_ms = start_all.elapsed_time(end_all)
    kernel_ms, kernel_launches = skv.kernel_timing_read()
    step_ms = [a.elapsed_time(b) for a, b in ev]
    if skv.device_error() != 0:
        raise RuntimeError(f"{w.name}: a kernel reported a timed-out wait in the timed region")

    max_total_ms = max_over_ranks(total_ms, ws)
    all_bytes = sum_over_ranks(float(kv_bytes) * args.steps, ws)
    res = {"kv_bytes": kv_bytes, "flops": flops, "ms_per_step": max_total_ms / args.steps,
           "value_gbs": all_bytes / (max_total_ms * 1e-3) / 1e9, "kernel_ms": kernel_ms,
           "kernel_launches": kernel_launches, "step_ms": step_ms, "clocks": clocks, "par": None, "e2e": None}

    # one (batch, KV head) group's inputs and the timed steps' result for it, kept on the host
    # for the oracle parity sample (plain caches with at most PARITY_MAX_TOKENS tokens in the
    # group; a long query chunk keeps every (Tq / ORACLE_MAX_ROWS)-th row)
    if want_parity and not (w.paged or w.passq_ranks or positional):
        try:
            G = w.Hq // w.Hkv
            n_tok = inp["seq_lens_host"][0]
            rows = list(range(w.Tq)) if w.Tq <= ORACLE_MAX_ROWS else list(range(0, w.Tq, w.Tq // ORACLE_MAX_ROWS))
            if n_tok <= PARITY_MAX_TOKENS:
                fp8 = w.kv_dtype == "fp8_e4m3"
                res_o, res_l = (o_acc, lse_acc) if w.ring_steps else (out, lse)
                res["par"] = {"n_tok": n_tok, "rows": rows,
                              "q": inp["q"][0, rows, :G].contiguous().cpu(),
                              "k": inp["k"][0, 0, :n_tok].contiguous().cpu(),
                              "v": inp["v"][0, 0, :n_tok].contiguous().cpu(),
                              "ks": inp["k_scale"][0, 0].cpu() if fp8 else None,
                              "vs": inp["v_scale"][0, 0].cpu() if fp8 else None,
                              "out": res_o[0, rows, :G].float().cpu(), "lse": res_l[0, rows, :G].cpu()}
        except Exception as e:  # the parity sample must never cost the bench line
            res["par"] = {"error": f"{type(e).__name__}: {e}"[:200]}

    # e2e: the public call with host (pinned) inputs; copies in and the result back every step
    if want_e2e:
        host = {}
        # the MLA value cache is a view of the latent (k): it is copied once, as k
        if w.ring_steps:
            keys = ("q",)
        elif w.passq_ranks:
            keys = ("q", "k_shards", "v_shards", "k_shard_scale", "v_shard_scale", "shard_lens")
        elif w.paged:
            keys = ("q", "k_pages", "seq_lens", "split_bounds_dev", "block_table") + (() if w.mla else ("v_pages",)) + (
                ("k_scale_pages", "v_scale_pages") if w.kv_dtype != "bf16" else ())
        elif w.mla:
            keys = ("q", "k", "k_scale", "v_scale", "seq_lens", "split_bounds_dev")
        else:
            keys = ("q", "k", "v", "k_scale", "v_scale", "seq_lens", "split_bounds_dev", "q_pos", "k_pos")
        for key in keys:
            t = inp.get(key)
            host[key] = None if t is None else t.cpu().pin_memory()
        if w.ring_steps:  # each step's block arrives from the host into its own buffer
            for j, (kb, vb, sl) in enumerate(ring_blocks):
                host[f"k{j}"], host[f"v{j}"], host[f"s{j}"] = kb.cpu().pin_memory(), vb.cpu().pin_memory(), sl.cpu().pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host.values() if t is not None)
        out_h = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        lse_h = torch.empty(lse.shape, dtype=lse.dtype).pin_memory()
        d2h = out_h.numel() * out_h.element_size() + lse_h.numel() * lse_h.element_size()
        dev_bufs = {k2: (None if t is None else torch.empty_like(t, device=dev)) for k2, t in host.items()}
        if w.mla and w.paged:
            dev_bufs["v_pages"] = dev_bufs["k_pages"][..., : w.dv]
            dev_bufs["v_scale_pages"] = None
        elif w.mla:
            dev_bufs["v"] = dev_bufs["k"][..., : w.dv]
        del inp
        torch.cuda.empty_cache()

        def e2e_step():
            for k2, t in host.items():
                if t is not None:
                    dev_bufs[k2].copy_(t, non_blocking=True)
            e2e_kw = dict(k_scale=dev_bufs.get("k_scale"), v_scale=dev_bufs.get("v_scale"), softmax_scale=w.scale,
                          scale_block=w.scale_block, out=out, lse=lse)
            if w.passq_ranks:
                skv.gqa_decode_attn_passq(dev_bufs["q"], dev_bufs["k_shards"], dev_bufs["v_shards"],
                                          dev_bufs["shard_lens"], k_scale=dev_bufs["k_shard_scale"],
                                          v_scale=dev_bufs["v_shard_scale"], softmax_scale=w.scale,
                                          scale_block=w.scale_block, out=out, lse=lse)
            elif w.ring_steps:
                ring_run(dev_bufs["q"], [(dev_bufs[f"k{j}"], dev_bufs[f"v{j}"], dev_bufs[f"s{j}"])
                                         for j in range(w.n_split)])
                out.copy_(o_acc)  # the final output (bf16) read back like the other workloads'
                lse.copy_(lse_acc)
            elif w.paged:
                e2e_kw.update(k_scale=dev_bufs.get("k_scale_pages"), v_scale=dev_bufs.get("v_scale_pages"))
                skv.gqa_decode_attn_paged(dev_bufs["q"], dev_bufs["k_pages"], dev_bufs["v_pages"], dev_bufs["seq_lens"],
                                          dev_bufs["split_bounds_dev"], dev_bufs["block_table"], w.causal_offset,
                                          **e2e_kw)
            elif positional:
                skv.gqa_decode_attn_pos(dev_bufs["q"], dev_bufs["k"], dev_bufs["v"], dev_bufs["seq_lens"],
                                        dev_bufs["split_bounds_dev"], dev_bufs["q_pos"], dev_bufs["k_pos"], **e2e_kw)
            else:
                skv.gqa_decode_attn(dev_bufs["q"], dev_bufs["k"], dev_bufs["v"], dev_bufs["seq_lens"],
                                    dev_bufs["split_bounds_dev"], w.causal_offset, **e2e_kw)
            out_h.copy_(out, non_blocking=True)
            lse_h.copy_(lse, non_blocking=True)

        e2e_steps = max(1, min(args.steps, 5))
        e2e_step()
        torch.cuda.synchronize()
        barrier(ws)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        barrier(ws)
        e2e_ms = max_over_ranks(a.elapsed_time(b), ws)
        e2e_bytes = sum_over_ranks(float(kv_bytes) * e2e_steps, ws)
        res["e2e"] = {"value": round(e2e_bytes / (e2e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                      "ms_per_step": round(e2e_ms / e2e_steps, 3)}
    return res


def roofline_of(w, m, steps):
    """The dominant kernel's roofline: algorithmic bytes (decode: HBM-bound) or flops (a
    query chunk: tensor-bound) over its own device time from the library's events in pass
    2 (a ring step workload holds several launches per step, each over 1/n of the work)."""
    step_ms = m["step_ms"]
    kernel_ms, kernel_launches = m["kernel_ms"], m["kernel_launches"]
    kv_bytes, flops = m["kv_bytes"], m["flops"]
    step_s = (kernel_ms / steps) * 1e-3 if kernel_launches > 0 else statistics.mean(step_ms) * 1e-3
    hbm, hbm_kind = hbm_peak()
    tc, tc_kind = bf16_peak()
    tensor_bound = w.Tq > 1  # the prefill chunk is a dense contraction; decode streams KV
    if tensor_bound:
        roof = {"bound": "tensor", "achieved": round(flops / step_s / 1e12, 2), "peak": tc, "unit": "TFLOP/s",
                "frac": round(flops / step_s / 1e12 / tc, 4), "peak_kind": tc_kind}
    else:
        roof = {"bound": "hbm", "achieved": round(kv_bytes / step_s / 1e9, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(kv_bytes / step_s / 1e9 / hbm, 4), "peak_kind": hbm_kind}
    roof.update({"kernel_ms_per_step": round(kernel_ms / steps, 4), "kernel_launches": kernel_launches,
                 "step_frac": round((flops / (statistics.mean(step_ms) * 1e-3) / 1e12 / tc) if tensor_bound else
                                    (kv_bytes / (statistics.mean(step_ms) * 1e-3) / 1e9 / hbm), 4),
                 "traffic": ncu_traffic(w.name),
                 "algorithmic_bytes_per_launch": round(kv_bytes / max(1, kernel_launches // steps)),
                 "flops_per_launch": round(flops / max(1, kernel_launches // steps)),
                 "hbm_gbs": round(kv_bytes / step_s / 1e9, 1),
                 "hbm_frac_of_nominal_8tbs": round(kv_bytes / step_s / 1e9 / 8000.0, 4),
                 "tflops": round(flops / step_s / 1e12, 2), "tensor_frac": round(flops / step_s / 1e12 / tc, 4)})
    return roof


def workload_summary(w, m, steps, parity):
    """Compact record of one extra workload for the "workloads" block: time per layer, the
    dominant kernel's time and roofline fractions (HBM and bf16 tensor, of the measured
    peaks), the clocks sampled during its timed region and the oracle parity sample."""
    r = roofline_of(w, m, steps)
    c = m["clocks"]
    return {"ms_per_step": round(m["ms_per_step"], 4), "us_per_layer": round(m["ms_per_step"] * 1e3, 2),
            "kernel_ms_per_step": r["kernel_ms_per_step"], "bound": r["bound"], "frac": r["frac"],
            "step_frac": r["step_frac"], "hbm_gbs": r["hbm_gbs"], "hbm_frac": round(r["hbm_gbs"] / hbm_peak()[0], 4),
            "tflops": r["tflops"], "tensor_frac": r["tensor_frac"], "traffic": r["traffic"],
            "gpu_launches": launches_per_step(w) * steps,
            "clocks": {"sm_mhz": c.get("sm_mhz"), "sm_max_mhz": c.get("sm_max_mhz"), "reasons": c.get("reasons")},
            "parity": parity}


def kvp_arm(args, w, ws, rank, local):
    """KVP decode across ranks (--mode kvp): rank r holds shard r (tokens [r S/N, (r+1) S/N))
    of every sequence of the workload, runs its partials into the All-to-All send buffer,
    exchanges them over the query-head axis (NCCL all_to_all_single; identity on one rank)
    and merges the received partials of its own Hq/N heads: the step of
    mla_decode_attention_gqa_gb300.kvp.kvp_decode_step.  value = the KV bytes of all shards
    over the slowest rank's step time ("scaling": "strong": the problem is fixed)."""
    import mla_decode_attention_gqa_gb300 as skv  # noqa: F401 - loads the library
    from mla_decode_attention_gqa_gb300 import kvp

    dev = torch.device("cuda", local)
    S_loc = w.S // ws
    gen = torch.Generator().manual_seed(w.seed)
    seq = (torch.randint(w.S // 2, w.S + 1, (w.B,), generator=gen) if w.ragged else torch.full((w.B,), w.S)).tolist()
    lens = [min(max(n - rank * S_loc, 0), S_loc) for n in seq]
    shard = W.scaled(w, S=S_loc, ragged=False, n_split=1, seed=w.seed + 1 + rank)
    inp = W.make_inputs(shard, dev, poison=False)
    seq_lens = torch.tensor(lens, dtype=torch.int32, device=dev)
    scales = (kvp.slab_scales(inp["k_scale"], inp["v_scale"], w.Hq, w.Hkv, ws) if w.kv_dtype == "fp8_e4m3" else None)
    all_lens = [min(max(n - r * S_loc, 0), S_loc) for r in range(ws) for n in seq]
    kv_bytes = RL.kv_bytes(w.Hkv, w.dk, w.dv, w.kv_dtype, all_lens, [[0, S_loc]] * len(all_lens),
                           scale_block=w.scale_block)
    bufs = None

    def step():
        nonlocal bufs
        _, _, bufs = kvp.kvp_decode_step(inp["q"], inp["k"], inp["v"], seq_lens, softmax_scale=w.scale,
                                         scale_block=w.scale_block, scales=scales, buffers=bufs)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    sampler = ClockSampler(local)
    barrier(ws)
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(args.steps):
        step()
    b.record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    clocks = sampler.stop()
    ms = max_over_ranks(a.elapsed_time(b), ws) / args.steps
    if rank != 0:
        return
    line = {"metric": METRIC, "value": round(kv_bytes / (ms * 1e-3) / 1e9, 2), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 4), "us_per_layer": round(ms * 1e3, 2),
            "higher_is_better": True, "scaling": "strong", "vs_baseline": None,
            "dtype": "bf16" if w.kv_dtype == "bf16" else "fp8_e4m3 KV, bf16 q", "data": "synthetic (seeded N(0,1))",
            "config": dict(config_of(w, ws), parallelism=f"kvp{ws}", kvp_shard_tokens=S_loc),
            "mode": "kvp", "clocks": clocks,
            "gpu_launches": (ws + 1) * args.steps}
    print(json.dumps(line), flush=True)


def ours_arm(args, w, ws, rank, local):
    want_par = not args.no_cpu_baseline
    m = measure(args, w, ws, rank, local, want_e2e=not args.no_e2e, want_parity=want_par)
    torch.cuda.empty_cache()
    extras = {}
    for name in args.extra_names:
        we = workload_by_name(name)
        me = measure(args, we, ws, rank, local, want_e2e=False, want_parity=want_par)
        torch.cuda.empty_cache()
        if rank == 0:
            par = oracle_parity(we, me["par"]) if me["par"] is not None else None
            extras[name] = workload_summary(we, me, args.steps, par)
    if rank != 0:
        return
    roof = roofline_of(w, m, args.steps)
    cpu = None
    if not args.no_cpu_baseline:
        b, s, g, t, r = oracle_sample(w, budget_s=args.cpu_budget)
        cpu = {"value": round(b / s / 1e9, 4), "unit": "GB/s", "cores": _CORES, "kind": "oracle",
               "sample": oracle_sample_text(w, g, t, r) + f", {s:.1f} s"}
        if m["par"] is not None:
            cpu["parity"] = oracle_parity(w, m["par"])
    step_ms = m["step_ms"]
    line = {
        "metric": METRIC,
        "value": round(m["value_gbs"], 2),
        "unit": "GB/s",
        "n_gpus": ws,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(m["ms_per_step"], 4),
        "us_per_layer": round(m["ms_per_step"] * 1e3, 2),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.kv_dtype == "bf16" else "fp8_e4m3 KV, bf16 q",
        "data": "synthetic (seeded N(0,1) bf16 Q/K/V)",
        "config": config_of(w, ws),
        "roofline": roof,
        "clocks": m["clocks"],
        "gpu_launches": launches_per_step(w) * args.steps,
        "e2e": m["e2e"],
        "cpu_baseline": cpu,
        "step_ms_min_median_max": [round(min(step_ms), 4), round(statistics.median(step_ms), 4),
                                   round(max(step_ms), 4)],
    }
    if extras:
        line["workloads"] = extras
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=W.HELIX_DENSE_128K.name)
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--S", type=int, default=None, help="smaller KV length of the same workload (profiling)")
    ap.add_argument("--B", type=int, default=None, help="smaller batch of the same workload (profiling)")
    ap.add_argument("--Tq", type=int, default=None, help="fewer query rows of the same workload (profiling)")
    ap.add_argument("--mode", choices=["replicas", "kvp"], default="replicas",
                    help="replicas: every rank runs the whole workload (default); kvp: the workload's sequence is "
                         "sharded over the ranks and one All-to-All over the query heads exchanges the partials")
    ap.add_argument("--extras", default="auto",
                    help="workloads measured after the main one: 'auto' (the long-context fp8 decode, the MLA "
                         "decode and the ring-prefill chunk fused and as ring steps, when the default workload runs "
                         "unscaled on one GPU), 'none', or a comma-separated list of workload names")
    args = ap.parse_args()
    if args.warmup < 3:
        raise SystemExit("--warmup must be >= 3")
    w = workload_by_name(args.config)
    over = {k: v for k, v in (("S", args.S), ("B", args.B), ("Tq", args.Tq)) if v is not None}
    if over:
        w = W.scaled(w, **over)
    ws, rank, local = dist_setup()
    if args.mode == "kvp" and args.config == W.HELIX_DENSE_128K.name:
        w = W.HELIX_KVP8_FP8_1M  # the KVP mode's workload: the long-context fp8 decode
    if args.extras == "auto":
        args.extra_names = list(EXTRA_WORKLOADS) if (ws == 1 and not over and w.name == W.HELIX_DENSE_128K.name) else []
    elif args.extras == "none":
        args.extra_names = []
    else:
        args.extra_names = [workload_by_name(n).name for n in args.extras.split(",") if n]
    if args.impl == "reference":
        reference_arm(args, w, ws, rank)
    elif args.mode == "kvp":
        kvp_arm(args, w, ws, rank, local)
    else:
        ours_arm(args, w, ws, rank, local)
    if ws > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
