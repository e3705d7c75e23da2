"""The reference arm's JSON line (the CPU oracle timed on the host cores), on
small workloads of the same structure as the bench's: the keys and units the
line must carry, and that its three figures are the one timed value."""
import argparse
import os
import json

import pytest

import bench

SMALL = dict(layers=2, H=2, Hq=8, d=64, P=32, rk=8, rv=8, sink=4, W=64, B=1, T=1024, rope=1e4, k=6, n_out=2,
             desc="small reference-arm check: 2 layers, 2 KV / 8 query heads, d=64, T=1024, P=32, r=8")


@pytest.mark.parametrize("extra", [{}, {"int4": True}, {"rope": None, "rope_theta": 1e4}],
                         ids=["bf16", "int4", "prerope"])
def test_reference_arm_line(monkeypatch, extra):
    wl = {**SMALL, **extra}
    monkeypatch.setitem(bench.WORKLOADS, "small-check", wl)
    args = argparse.Namespace(workload="small-check", steps=2, warmup=1)
    res = bench.reference_arm(args, 0, 1)
    line = json.loads(json.dumps(res))  # the printed line round-trips
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e", "gpu_launches"):
        assert key in line, key
    assert line["impl"] == "reference" and line["n_gpus"] == 1
    assert (line["steps"], line["warmup"]) == (2, 1)
    assert line["unit"] == "us/step" and line["higher_is_better"] is False
    assert line["value"] > 0 and line["ms_per_step"] == pytest.approx(line["value"] / 1000.0, abs=1e-3)
    assert line["config"]["workload"] == wl["desc"] and line["config"]["seq_len"] == wl["T"]
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["unit"] == line["unit"]
    assert cb["cores"] >= 1 and cb["pages_cores"] >= 1 and cb["sample"] and cb["cpu_model"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert line["gpu_launches"] == 0 and line["vs_baseline"] is None


def test_reference_arm_other_ranks_do_no_work(monkeypatch):
    monkeypatch.setitem(bench.WORKLOADS, "small-check", SMALL)
    args = argparse.Namespace(workload="small-check", steps=1, warmup=0)
    assert bench.reference_arm(args, 1, 2) is None


def test_gpu_arm_cpu_baseline_fields():
    """The cpu_baseline object of the GPU arm's line (host work only)."""
    cb = bench.cpu_baseline_sample(SMALL)
    assert cb["kind"] == "oracle" and cb["unit"] == "us/step" and cb["value"] > 0
    assert cb["cores"] == cb["nproc"] == (os.cpu_count() or 1) and cb["pages_cores"] >= 1 and cb["pages_sample"] > 0
    assert cb["pages_factorized_per_s"] > 0 and cb["sample"] and cb["cpu_model"]
    # decode timed on one core and on all of them; the whole tiny workload through the oracle
    rates = cb["decode_pairs_per_s"]
    assert rates["1_core"] > 0 and rates[f"{cb['nproc']}_cores"] > 0 and cb["decode_us_per_step_1_core"] > 0
    assert cb["tiny_workload_full_oracle_s"] > 0
