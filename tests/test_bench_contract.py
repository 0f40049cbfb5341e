"""bench.py's JSON line and roofline arithmetic, on a fake timing result (no GPU)."""
import json
import os
import sys
import types

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from sparse_top_mla_gb300 import synth  # noqa: E402

REQUIRED = ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
            "vs_baseline", "dtype", "data", "config", "roofline", "clocks", "e2e", "gpu_launches")


def _fake(kind, w):
    return {"label": "fake " + kind, "w0": w, "value": 1000.0, "total_ms": 7.5, "steps": 100, "l2_flush": False,
            "ms_per_step": 0.075, "kern_avg_ms": 0.0675, "kern_samples": 25, "gathered": w.gathered_bytes(),
            "flops": w.flops(), "idx_bytes": 524288, "q_bytes": w.T * w.H * 576 * 2,
            "alg_bytes": w.algorithmic_bytes(),
            "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 3},
            "e2e": {"value": 500.0, "unit": "GB/s", "h2d_bytes_per_step": 1, "d2h_bytes_per_step": 1},
            "launches": 200, "peaks": {"hbm_gbs": 6680.5, "bf16_tflops": 1943.9, "bf16_tflops_sustained": 1700.0,
                                       "source": "of measured"}}


def test_decode_line_has_the_contract_keys():
    w = synth.config(1)
    r = _fake("decode", w)
    args = types.SimpleNamespace(warmup=5)
    d = bench.line_for("decode", r, args, 1, {"value": 0.2, "unit": "GB/s", "cores": 16, "kind": "oracle",
                                              "sample": "x"})
    for k in REQUIRED:
        assert k in d, k
    json.dumps(d)
    assert d["higher_is_better"] is True and d["scaling"] == "weak" and d["n_gpus"] == 1
    rl = d["roofline"]
    # valid gathered rows + indices + q + O + LSE, per the measurement definition
    kset = w.main.topk + (w.extra.topk if w.extra is not None else 0)
    alg = w.gathered_bytes() + w.T * kset * 4 + w.T * w.H * 576 * 2 + w.T * w.H * 512 * 2 + w.T * w.H * 4
    assert rl["bound"] == "hbm" and rl["unit"] == "GB/s"
    assert rl["algorithmic_bytes_per_launch"] == alg
    assert abs(rl["achieved"] - alg / 0.0675e-3 / 1e9) < 1e-6
    assert abs(rl["frac"] - rl["achieved"] / 6680.5) < 1e-12
    assert abs(rl["frac_gathered"] - w.gathered_bytes() / 0.0675e-3 / 1e9 / 6680.5) < 1e-12
    assert abs(rl["frac_call"] - alg / 0.075e-3 / 1e9 / 6680.5) < 1e-12
    assert d["cpu_baseline"]["kind"] == "oracle"


def test_prefill_roofline_is_tensor_flops():
    w = synth.config(1)
    r = _fake("prefill", w)
    rl = bench.roofline_for("prefill", r)
    assert rl["bound"] == "tensor" and rl["unit"] == "TFLOP/s"
    assert abs(rl["achieved"] - w.flops() / 0.0675e-3 / 1e12) < 1e-9
    assert abs(rl["frac"] - rl["achieved"] / 1943.9) < 1e-12


def test_traffic_only_for_the_captured_source(monkeypatch):
    d = json.load(open(os.path.join(ROOT, "profiles", "traffic.json")))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda key="decode": d["decode"]["kernel_source_hash"])
    assert bench.ncu_traffic("decode") == d["decode"]["dram_bytes_per_launch"]
    monkeypatch.setattr(bench, "kernel_source_hash", lambda key="decode": "0" * 16)
    assert bench.ncu_traffic("decode") is None


def test_l2_rule_is_stated():
    assert bench.input_mb(synth.config(1)) < bench.L2_MB
    assert bench.l2_note(synth.config(1), True).startswith("L2 flushed")
    assert "larger than L2" in bench.l2_note(synth.config(1), False)


def test_clock_summary_uses_the_timed_window():
    row = "0, {sm}, 2070, 900, 0x0, Not Active, Not Active, Not Active, {cap}"
    lines = [(10.0, row.format(sm=1200, cap="Not Active")), (10.4, row.format(sm=2070, cap="Active")),
             (10.5, row.format(sm=2040, cap="Not Active")), (11.0, row.format(sm=1100, cap="Not Active"))]
    c = bench.ClockSampler.summarise(lines, 10.3, 10.6)
    assert c["samples_in_region"] == 2 and c["sm_mhz"] == 2055.0 and c["reasons"] == ["sw_power_cap"]
    c = bench.ClockSampler.summarise(lines, 10.6, 10.7)  # nothing inside: the nearest sample
    assert c["samples_in_region"] == 0 and c["samples"] == 1 and c["sm_mhz"] == 2040.0
    # a short region: the one-shot samples just before and after it are its record
    edge = ((10.59, row.format(sm=2070, cap="Not Active")), (10.71, row.format(sm=2060, cap="Active")))
    c = bench.ClockSampler.summarise(lines, 10.6, 10.7, edge)
    assert c["samples_in_region"] == 0 and c["bracket_samples"] == 2 and c["sm_mhz"] == 2065.0
    assert c["reasons"] == ["sw_power_cap"]


def test_secondary_workload_sub_object():
    w = synth.config(1)
    r = _fake("prefill", w)
    cpu = {"value": 0.01, "unit": "TFLOP/s", "cores": 16, "kind": "oracle", "sample": "x"}
    d = bench.secondary_for("prefill", r, cpu)
    json.dumps(d)
    assert d["unit"] == "TFLOP/s" and abs(d["value"] - w.flops() / 0.075e-3 / 1e12) < 1e-9
    assert d["roofline"]["bound"] == "tensor" and d["cpu_baseline"]["unit"] == "TFLOP/s"
    assert abs(d["roofline"]["frac_sustained"] - d["roofline"]["achieved"] / 1700.0) < 1e-12
    for k in ("us_per_call", "kernel_avg_us", "l2", "clocks", "steps"):
        assert k in d


def test_default_steps_give_a_long_enough_timed_region(monkeypatch):
    monkeypatch.setattr(sys, "argv", ["bench.py"])
    assert bench.parse().steps == bench.DEFAULT_STEPS["decode"]
    monkeypatch.setattr(sys, "argv", ["bench.py", "--steps", "7"])
    assert bench.parse().steps == 7
