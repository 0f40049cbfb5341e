"""Per-CTA event timelines of the attention kernel (developer tool).

Builds a second copy of the library with -DSMLA_TRACE (every CTA records global-timer
timestamps of its pipeline events in a device array; the copy is not the product library and
is never loaded by it), runs one workload a few times, and prints, per event, the minimum /
median / maximum over CTAs of the last run, the per-tile medians of the pipeline events, and
the CTAs' exit times grouped by their share of the work (tiles and item segments).

    python -m sparse_top_mla_gb300.timeline decode|prefill|large|t1 [prefill|decode|forward]

Event slots (as the kernel records them): 0 entry, 1 after the dependency wait, 2 exit, 3 the
resolution prologue done (tiles 0-2 published), 4 the first gathers issued; tile j < 10 at
8 + 24 j + k with k: 0 S^T ready, 1 fast softmax pass done, 2 P^T final (decision barrier),
3 PV and row sums issued, 4 / 10 / 5 the issuer past the waits for blocks 0-3 / 4-7 / 8,
6 / 7 / 11 the loaders' arrivals for them, 8 / 9 epilogue start / end, 12..15 a loader past
the release of block pair 0..3, 16..19 that pair stored, 20..23 its refill issued; 248..254
steps of the CTA's first epilogue.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import sys

import numpy as np

from . import binding, build, synth

HERE = os.path.dirname(os.path.abspath(__file__))
OUT = os.path.join(HERE, "_build", "trace")
TILE_EVENTS = ["Sready", "fast", "decis", "PViss", "A(iss)", "R(iss)", "A(ld)", "B(ld)", "epi0", "epi1", "B(iss)",
               "R(ld)", "pv0", "pv1", "pv2", "pv3", "st0", "st1", "st2", "st3", "is0", "is1", "is2", "is3"]
# print order: the loaders' pairs, the issuer's waits, the softmax, the epilogue
TILE_ORDER = [12, 16, 20, 13, 17, 21, 6, 4, 14, 18, 22, 15, 19, 23, 7, 10, 11, 5, 0, 1, 2, 3, 8, 9]
CTA_EVENTS = {0: "entry", 1: "dependency wait done", 3: "resolution prologue done", 4: "first gathers issued",
              2: "exit", 248: "epilogue 1: row sums loaded", 249: "epilogue 1: factors",
              250: "epilogue 1: O^T block 0 loaded", 251: "epilogue 1: block 0 stored", 252: "epilogue 1: block 1 stored",
              253: "epilogue 1: block 3 stored", 254: "epilogue 1: end"}


def build_traced() -> str:
    """Compile the library sources with -DSMLA_TRACE into _build/trace; returns the .so path."""
    os.makedirs(OUT, exist_ok=True)
    cc = build.nvcc()
    objs, procs = [], []
    for src in build.SOURCES:
        obj = os.path.join(OUT, src.replace(".cu", ".o"))
        objs.append(obj)
        procs.append(subprocess.Popen([cc, *build.ARCH, *build.FLAGS, "-DSMLA_TRACE", "-c",
                                       os.path.join(build.CSRC, src), "-o", obj]))
    if any(p.wait() != 0 for p in procs):
        raise RuntimeError("trace build failed")
    lib = os.path.join(OUT, "libsmla_trace.so")
    subprocess.check_call([cc, *build.ARCH, "-shared", "-o", lib, *objs])
    return lib


def workload(kind: str):
    return {"decode": lambda: synth.config(2), "prefill": lambda: synth.config(3),
            "large": lambda: synth.config(4, T=1024),
            "t1": lambda: synth.SweepPool().point(64, 512, 1, True)}[kind]()


def capture(w, mode: str = "forward", runs: int = 8) -> np.ndarray:
    """Event times (microseconds from the first CTA's entry; NaN = not recorded) of the last
    of `runs` calls of workload w, [CTAs, 256]."""
    import torch
    lib = binding.use_library(build_traced())
    lib.smla_trace_read.argtypes = [ctypes.c_void_p, ctypes.c_size_t]
    dp = binding.DeviceProblem(w, device="cuda:0")
    for _ in range(runs):
        dp.run(mode)
    torch.cuda.synchronize()
    if binding.device_error() != 0:
        raise RuntimeError("device error during the traced runs")
    buf = np.zeros((1024, 256), dtype=np.uint64)
    if lib.smla_trace_read(buf.ctypes.data, buf.nbytes) != 0:
        raise RuntimeError("smla_trace_read failed")
    n = int(np.count_nonzero(buf[:, 0]))
    raw = buf[:n].astype(np.int64)
    rel = (raw - raw[:, 0].min()) / 1000.0
    rel[raw == 0] = np.nan
    return rel


def report(rel: np.ndarray, total_tiles: int = 0, tiles_per_item: int = 0) -> str:
    lines = [f"{rel.shape[0]} CTAs; event times in us from the first CTA's entry: min / median / max"]
    for slot, name in CTA_EVENTS.items():
        col = rel[:, slot]
        if np.all(np.isnan(col)):
            continue
        lines.append(f"  {name:34s} {np.nanmin(col):8.2f} {np.nanmedian(col):8.2f} {np.nanmax(col):8.2f}")
    for j in range(10):
        cols = rel[:, 8 + 24 * j: 32 + 24 * j]
        if np.all(np.isnan(cols)):
            continue
        cells = [f"{TILE_EVENTS[k]}={np.nanmedian(cols[:, k]):6.2f}" for k in TILE_ORDER
                 if not np.all(np.isnan(cols[:, k]))]
        lines.append(f"  tile {j}: " + " ".join(cells))
    sready = rel[:, 8:248:24]
    period = np.array([np.nanmean(np.diff(r[~np.isnan(r)])) if np.count_nonzero(~np.isnan(r)) > 1 else np.nan
                       for r in sready])
    lines.append(f"  mean S^T-ready period per CTA: min {np.nanmin(period):.2f} median {np.nanmedian(period):.2f} "
                 f"max {np.nanmax(period):.2f} us")
    if total_tiles and tiles_per_item:
        n = rel.shape[0]
        lo = [c * total_tiles // n for c in range(n + 1)]
        ntile = np.array([lo[c + 1] - lo[c] for c in range(n)])
        nseg = np.array([(lo[c + 1] - 1) // tiles_per_item - lo[c] // tiles_per_item + 1 for c in range(n)])
        for t in sorted(set(ntile)):
            for s in sorted(set(nseg)):
                m = (ntile == t) & (nseg == s)
                if m.any():
                    ex = rel[m, 2]
                    lines.append(f"  exit, {t} tiles in {s} item segment(s), {m.sum()} CTAs: "
                                 f"{np.nanmin(ex):.2f} / {np.nanmedian(ex):.2f} / {np.nanmax(ex):.2f}")
    return "\n".join(lines)


def main(argv=None) -> int:
    argv = sys.argv[1:] if argv is None else argv
    kind = argv[0] if argv else "decode"
    mode = argv[1] if len(argv) > 1 else "forward"
    w = workload(kind)
    rel = capture(w, mode)
    total = tpi = 0
    if kind == "decode" and mode in ("decode", "forward"):
        # one head group per token at this size: items are tokens
        tpi = (w.main.topk + 127) // 128
        total = w.T * tpi
    print(f"{kind} ({mode})")
    print(report(rel, total, tpi))
    return 0


if __name__ == "__main__":
    sys.exit(main())
