"""Decode/prefill crossover calibration for smla_forward.

flashinfer PR "fix(sm120): explain sparse-MLA decode dispatch misses; add config query API",
merged body, section "Dispatch: cpb model + crossover": the token count up to which the split-K
decode schedule serves a configuration (decode_max_tokens) is picked from measurements, and
decode is chosen only where it takes at most 0.95x the time of the prefill schedule.

For every (H, topk) of the envelope sweep (a paged context of 64 sequences x 16384 tokens,
random distinct indices with 5% masked, per-head sink) this script times smla_decode and
smla_prefill at every T of a grid, each on `rotations` independent query/index sets called
back to back (so successive calls gather different rows), and writes the table that
smla_load_crossover reads:

    {"version": 1, "entries": [[H, topk, format, decode_max_tokens], ...], ...timings...}

decode_max_tokens is the largest grid T such that decode met the rule at that T and at every
smaller grid T (0 when it loses already at the smallest). Run on the GPU the table is for:

    python -m sparse_top_mla_gb300.calibrate --out sparse_top_mla_gb300/crossover_gb300.json
"""
from __future__ import annotations

import argparse
import json
import math
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
DEFAULT_TABLE = os.path.join(HERE, "crossover_gb300.json")
T_GRID = (1, 2, 4, 8, 16, 24, 32, 48, 64, 65, 96, 128, 192, 256, 384, 512, 1024)
RATIO = 0.95


def crossover(points, ratio: float = RATIO) -> int:
    """points: [(T, decode_us, prefill_us), ...]. Largest T of the leading run of grid points
    (ascending T) where decode_us <= ratio * prefill_us; 0 if the smallest T already fails."""
    best = 0
    for T, dec, pre in sorted(points):
        if not (dec <= ratio * pre):
            break
        best = T
    return best


def table_json(entries, meta: dict) -> str:
    """The table in the layout smla_load_crossover parses ("version" and "entries" first)."""
    head = '{\n "version": 1,\n "entries": [\n' + ",\n".join(
        "  [%d, %d, %d, %d]" % tuple(int(v) for v in e) for e in entries) + "\n ]"
    lines = []
    for k, v in meta.items():
        if isinstance(v, dict):
            body = ",\n".join(f"  {json.dumps(kk)}: {json.dumps(vv)}" for kk, vv in v.items())
            lines.append(f" {json.dumps(k)}: {{\n{body}\n }}")
        else:
            lines.append(f" {json.dumps(k)}: {json.dumps(v)}")
    return head + "".join(",\n" + l for l in lines) + "\n}\n"


def graph_time_us(fn, calls, stream, reps: int, inner: int = 4) -> float:
    """GPU time per call, from a CUDA graph replaying `inner` rounds of the rotating calls (the
    pages' protocol times graph replays, GPU-only): host submission is then not part of the
    number, which matters at small T where a call is a few microseconds of GPU work."""
    import torch
    for c in calls:
        fn(c, stream)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(inner):
            for c in calls:
                fn(c, None)  # None: torch's current stream, the capture stream here
    g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    best = math.inf
    for _ in range(reps):
        e0.record(stream)
        g.replay()
        e1.record(stream)
        e1.synchronize()
        best = min(best, e0.elapsed_time(e1) * 1e3 / (inner * len(calls)))
    return best


def calibrate(formats=(1,), heads=None, topks=None, t_grid=T_GRID, rotations: int = 4, reps: int = 3,
              ratio: float = RATIO, device: str = "cuda:0", log=print) -> dict:
    import torch
    from . import binding, synth
    heads = heads or synth.SWEEP_H
    topks = topks or synth.SWEEP_TOPK
    dev = torch.device(device)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    tmax = max(t_grid)
    props = torch.cuda.get_device_properties(dev)
    entries, timings = [], {}
    workspace = [torch.empty(0, dtype=torch.uint8, device=dev)]

    def ws_for(calls):
        need = max(binding.workspace_size(c) for c in calls)
        if need > workspace[0].numel():
            workspace[0] = torch.empty(need, dtype=torch.uint8, device=dev)
        for c in calls:
            c.set_workspace(workspace[0] if need else None)

    for fmt in formats:
        t0 = time.time()
        pool = synth.SweepPool(fmt=fmt)
        cache = torch.from_numpy(pool.cache).to(dev)
        bt = torch.from_numpy(pool.block_table).to(dev)
        sl = torch.from_numpy(pool.seq_lens).to(dev)
        token_seq = torch.from_numpy((np.arange(tmax) % pool.num_seqs).astype(np.int32)).to(dev)
        rng = np.random.default_rng(7000 + fmt)
        idx = {k: [torch.from_numpy(synth.mask_random(rng, synth.distinct_indices(
            rng, np.full(tmax, pool.ctx - 1), k), 0.05)).to(dev) for _ in range(rotations)] for k in topks}
        log(f"format {fmt}: context and index sets ready in {time.time() - t0:.1f} s")
        for H in heads:
            qs = [torch.from_numpy(synth.make_q(rng, tmax, H).view(np.int16)).to(dev).view(torch.bfloat16)
                  for _ in range(rotations)]
            sink = torch.from_numpy(synth.normal_f32(rng, (H,))).to(dev)
            out = torch.empty((tmax, H, 512), dtype=torch.bfloat16, device=dev)
            lse = torch.empty((tmax, H), dtype=torch.float32, device=dev)
            for k in topks:
                pts = []
                for T in t_grid:
                    calls = []
                    for r in range(rotations):
                        main = binding.DeviceSet(cache, fmt, pool.row_stride, pool.page_stride, pool.num_pages, bt,
                                                 sl, idx[k][r][:T], k)
                        calls.append(binding.Call(qs[r][:T], token_seq[:T], main, out[:T], lse[:T], None, sink,
                                                  np.float32(1.0 / math.sqrt(576)), None, num_seqs=pool.num_seqs))
                    ws_for(calls)
                    dec = graph_time_us(binding.decode, calls, stream, reps)
                    pre = graph_time_us(binding.prefill, calls, stream, reps)
                    pts.append((T, dec, pre))
                mt = crossover(pts, ratio)
                entries.append((H, k, fmt, mt))
                timings[f"H={H} topk={k} format={fmt}"] = [[T, round(d, 2), round(p, 2)] for T, d, p in pts]
                log(f"H={H:3d} topk={k:4d} format={fmt}: decode_max_tokens={mt:4d}  " +
                    " ".join(f"T{T}:{d:.1f}/{p:.1f}" for T, d, p in pts if T in (1, 16, 64, 256, 1024)))
        del cache
        assert binding.device_error() == 0
    meta = {"device": props.name, "sm_count": props.multi_processor_count,
            "rule": f"decode iff t_decode <= {ratio} t_prefill at T and every smaller grid T",
            "t_grid": list(t_grid), "rotations": rotations,
            "timing": "CUDA-graph replay of 4 rounds of the rotating calls, best of reps, GPU time per call",
            "context": "64 sequences x 16384 tokens, random distinct indices, 5% masked, per-head sink",
            "timings_us_T_decode_prefill": timings}
    return {"entries": entries, "meta": meta}


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--out", default=DEFAULT_TABLE)
    ap.add_argument("--formats", default="1", help="comma-separated cache formats (0 = bf16, 1 = fp8)")
    ap.add_argument("--heads", default="", help="comma-separated H values (default: the sweep's)")
    ap.add_argument("--topks", default="", help="comma-separated topk values (default: the sweep's)")
    ap.add_argument("--rotations", type=int, default=4)
    ap.add_argument("--reps", type=int, default=3)
    a = ap.parse_args(argv)
    ints = lambda s: tuple(int(v) for v in s.split(",") if v)  # noqa: E731
    from . import build
    build.build()
    r = calibrate(formats=ints(a.formats), heads=ints(a.heads) or None, topks=ints(a.topks) or None,
                  rotations=a.rotations, reps=a.reps)
    with open(a.out, "w") as f:
        f.write(table_json(r["entries"], r["meta"]))
    from . import binding
    st = binding.load_crossover(a.out)
    if st != binding.SMLA_OK:
        print(f"the written table does not load: {binding.status_string(st)}", file=sys.stderr)
        return 1
    print(f"wrote {len(r['entries'])} entries to {a.out}")
    return 0


if __name__ == "__main__":
    sys.exit(main())
