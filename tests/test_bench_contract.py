"""bench.py's output contract, checked on the CPU.

* `config` names a workload by what it is (sizes, dtype, layout, L2 policy) and carries
  no model keys;
* a DRAM-traffic record is reported only while the kernel sources it was measured on
  still hash to the recorded value, and never for a workload it does not cover;
* the reference arm (the fp64 oracle on host cores) prints one JSON line with the
  contract's keys, its `cpu_baseline` and a host-only `e2e` (no device copies);
* the cpu_baseline leg's parity sample reports the error of the result it is given."""

import argparse
import contextlib
import io
import json
import os
import shutil
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from mla_decode_attention_gqa_gb300 import workloads as W  # noqa: E402


@pytest.mark.parametrize("w", W.WORKLOADS, ids=lambda w: w.name)
def test_config_names_the_workload_only(w):
    c = bench.config_of(w)
    assert c["workload"] == w.name
    for k in ("B", "Tq", "Hq", "Hkv", "dk", "dv", "S", "kv_dtype", "n_split", "l2", "parallelism"):
        assert k in c, k
    assert not {"model", "global_batch", "seq_len"} & set(c)
    assert json.loads(json.dumps(c)) == c  # plain JSON


def _records():
    with open(os.path.join(ROOT, "profiles", "traffic.json")) as f:
        return json.load(f)


def test_traffic_records_name_existing_sources_and_a_dominant_kernel():
    for name, rec in _records().items():
        assert any(w.name == name for w in W.WORKLOADS), name
        assert rec["kernel"] and rec["dram_bytes_per_launch"] > 0
        for rel in rec["kernel_sources"]:
            assert os.path.isfile(os.path.join(ROOT, rel)), rel


def test_traffic_is_dropped_once_a_kernel_source_changes(tmp_path, monkeypatch):
    recs = _records()
    name = next(iter(recs))
    rec = recs[name]
    # a private copy of the record and of its sources, so that a source can be edited
    for rel in rec["kernel_sources"]:
        dst = tmp_path / rel
        dst.parent.mkdir(parents=True, exist_ok=True)
        shutil.copyfile(os.path.join(ROOT, rel), dst)
    path = tmp_path / "traffic.json"
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "TRAFFIC_PATH", str(path))
    sha = bench.kernel_source_sha(rec["kernel_sources"])
    rec2 = dict(rec, kernel_source_sha=sha)
    path.write_text(json.dumps({name: rec2}))
    assert bench.ncu_traffic(name) == float(rec["dram_bytes_per_launch"])
    assert bench.ncu_traffic("no_such_workload") is None
    with open(tmp_path / rec["kernel_sources"][0], "a") as f:
        f.write("\n// edited\n")
    assert bench.ncu_traffic(name) is None


def test_reference_arm_prints_one_contract_line():
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.reference_arm(argparse.Namespace(steps=1, warmup=3), W.TINY_GQA, 1, 0)
    lines = [l for l in buf.getvalue().splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
              "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert k in d, k
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    assert d["value"] > 0 and d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["config"] == bench.config_of(W.TINY_GQA, 1)
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_is_silent_off_rank_zero():
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        bench.reference_arm(argparse.Namespace(steps=1, warmup=3), W.TINY_GQA, 2, 1)
    assert buf.getvalue() == ""


def test_parity_sample_reports_the_error_of_the_given_result():
    """oracle_parity compares a stored result with the oracle on the same bytes: an exact
    result (the oracle's own, rounded to bf16) gives errors at rounding level, and a planted
    error in one output element shows up in full."""
    import numpy as np

    import oracle

    w = W.scaled(W.HELIX_DENSE_128K, B=1, Hq=16, Hkv=1, S=512)
    inp = W.make_inputs(w)
    G, n = w.Hq // w.Hkv, inp["seq_lens_host"][0]
    qf = oracle.bf16_bits_to_f64(inp["q"][0:1, :, :G].contiguous().view(torch.int16).numpy())
    kf = oracle.bf16_bits_to_f64(inp["k"][0, 0, :n].contiguous().view(torch.int16).numpy())
    vf = oracle.bf16_bits_to_f64(inp["v"][0, 0, :n].contiguous().view(torch.int16).numpy())
    o, l = oracle.split_attention(qf, kf[None, None], vf[None, None], [n], [w.split_bounds()[0]], w.causal_offset,
                                  w.scale)
    mo, ml = oracle.merge_lse(o, l)
    par = {"n_tok": n, "rows": [0], "q": inp["q"][0, [0], :G].contiguous(), "k": inp["k"][0, 0, :n].contiguous(),
           "v": inp["v"][0, 0, :n].contiguous(), "ks": None, "vs": None,
           "out": torch.from_numpy(mo[0]).to(torch.bfloat16).float(), "lse": torch.from_numpy(ml[0]).float()}
    good = bench.oracle_parity(w, par)
    assert good["out_max_abs_err"] < 2 ** -8 * float(np.abs(mo).max()) + 1e-6 and good["lse_max_abs_err"] < 1e-6
    par["out"] = par["out"].clone()
    par["out"][0, 3, 5] += 0.5
    bad = bench.oracle_parity(w, par)
    assert bad["out_max_abs_err"] > 0.49
    assert "error" in bench.oracle_parity(w, {"error": "x"})


@pytest.mark.parametrize("kind", ["fp8_ragged", "causal_rows"])
def test_parity_sample_walks_splits_like_the_whole_group(kind):
    """oracle_parity takes the group one split at a time (dequantising each split's rows by
    absolute position, masking rows by their chunk position); fed the whole-group oracle
    result it reports rounding-level errors, for fp8 block-scaled KV with ragged splits and
    for a causal query chunk sampled every few rows."""
    import numpy as np

    import oracle

    if kind == "fp8_ragged":
        w = W.scaled(W.HELIX_KVP8_FP8_1M, B=1, Hq=16, Hkv=1, S=1024, seed=77)
        rows = [0]
    else:
        w = W.scaled(W.RING_PREFILL, B=1, Hq=16, Hkv=1, Tq=64, S=512, seed=78)
        rows = list(range(0, 64, 4))
    inp = W.make_inputs(w)
    G, n = w.Hq // w.Hkv, inp["seq_lens_host"][0]
    qf = oracle.bf16_bits_to_f64(inp["q"][0:1, rows, :G].contiguous().view(torch.int16).numpy())
    if w.kv_dtype == "fp8_e4m3":
        kf = oracle.dequant_e4m3_blocks(inp["k"][0, 0, :n].numpy(), inp["k_scale"][0, 0].numpy(), w.scale_block)
        vf = oracle.dequant_e4m3_blocks(inp["v"][0, 0, :n].numpy(), inp["v_scale"][0, 0].numpy(), w.scale_block)
    else:
        kf = oracle.bf16_bits_to_f64(inp["k"][0, 0, :n].contiguous().view(torch.int16).numpy())
        vf = oracle.bf16_bits_to_f64(inp["v"][0, 0, :n].contiguous().view(torch.int16).numpy())
    pos = {}
    if w.causal_offset != W.NO_CAUSAL:
        pos = {"q_positions": [w.causal_offset + np.asarray(rows)], "k_positions": [np.arange(n)]}
    o, l = oracle.split_attention(qf, kf[None, None], vf[None, None], [n], [w.split_bounds()[0]], w.causal_offset,
                                  w.scale, **pos)
    mo, ml = oracle.merge_lse(o, l)
    fp8 = w.kv_dtype == "fp8_e4m3"
    par = {"n_tok": n, "rows": rows, "q": inp["q"][0, rows, :G].contiguous(), "k": inp["k"][0, 0, :n].contiguous(),
           "v": inp["v"][0, 0, :n].contiguous(), "ks": inp["k_scale"][0, 0] if fp8 else None,
           "vs": inp["v_scale"][0, 0] if fp8 else None,
           "out": torch.from_numpy(mo[0]).float(), "lse": torch.from_numpy(ml[0]).float()}
    res = bench.oracle_parity(w, par)
    assert "error" not in res, res
    assert res["out_max_abs_err"] < 1e-6 and res["lse_max_abs_err"] < 1e-5 and res["empty_rows_match"], res
