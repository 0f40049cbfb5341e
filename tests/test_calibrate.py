"""Host logic of the decode/prefill crossover calibration (no GPU).

The rule follows flashinfer PR "fix(sm120): explain sparse-MLA decode dispatch misses; add
config query API", merged body, "Dispatch: cpb model + crossover": decode serves a token count
only where it takes at most 0.95x the prefill schedule's time.
"""
import json
import os

import pytest

from sparse_top_mla_gb300 import binding, calibrate, synth


def test_crossover_rule():
    pts = [(1, 5.0, 10.0), (16, 9.5, 10.0), (64, 9.6, 10.0), (256, 1.0, 10.0)]
    # 16 is the last T of the leading run that meets the 0.95x rule; 256 does not count
    assert calibrate.crossover(pts) == 16
    assert calibrate.crossover(list(reversed(pts))) == 16      # order of the list does not matter
    assert calibrate.crossover([(1, 11.0, 10.0), (16, 1.0, 10.0)]) == 0
    assert calibrate.crossover([(1, 1.0, 10.0), (1024, 1.0, 10.0)]) == 1024
    assert calibrate.crossover([(1, float("nan"), 10.0)]) == 0  # a failed timing never selects decode
    assert calibrate.crossover([(8, 9.0, 10.0)], ratio=0.9) == 8
    assert calibrate.crossover([(8, 9.1, 10.0)], ratio=0.9) == 0


def test_table_round_trip(tmp_path):
    lib = binding.load()
    entries = [(1, 64, 1, 1024), (64, 2048, 1, 96), (128, 2048, 1, 24), (64, 2048, 0, 48)]
    text = calibrate.table_json(entries, {"device": "test", "timings_us_T_decode_prefill":
                                          {"H=64 topk=2048 format=1": [[1, 10.0, 40.0], [96, 50.5, 60.1]]}})
    d = json.loads(text)
    assert d["version"] == 1 and [tuple(e) for e in d["entries"]] == entries
    path = tmp_path / "table.json"
    path.write_text(text)
    try:
        assert binding.load_crossover(str(path)) == binding.SMLA_OK
        assert binding.decode_max_tokens(64, 2048, 1) == 96
        assert binding.decode_max_tokens(64, 2048, 0) == 48
        assert binding.decode_max_tokens(128, 2048, 1) == 24
        assert binding.decode_max_tokens(2, 64, 1) == 1024      # nearest entry in log2 (H, topk)
    finally:
        binding.set_crossover([])
        if os.path.exists(binding.CROSSOVER_TABLE):
            assert lib.smla_load_crossover(binding.CROSSOVER_TABLE.encode()) == binding.SMLA_OK


def test_packaged_table_covers_the_sweep():
    if not os.path.exists(binding.CROSSOVER_TABLE):
        pytest.skip("no calibration table has been measured yet")
    d = json.load(open(binding.CROSSOVER_TABLE))
    assert d["version"] == 1
    got = {(H, k, f): m for H, k, f, m in d["entries"]}
    for H in synth.SWEEP_H:
        for k in synth.SWEEP_TOPK:
            assert (H, k, 1) in got, (H, k)
            assert 0 <= got[(H, k, 1)] <= max(d["t_grid"])
    # each entry is the rule applied to the timings stored beside it
    for (H, k, f), m in got.items():
        pts = d["timings_us_T_decode_prefill"][f"H={H} topk={k} format={f}"]
        assert calibrate.crossover([tuple(p) for p in pts]) == m
