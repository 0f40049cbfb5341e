"""Benchmark: sparse top-k MLA attention on one GB300 (or N independent replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl smla|reference]
                    [--workload decode|prefill|large_prefill|tiny|quantize|small_t] [--no-secondary]

The headline step is one smla_forward call (index resolve, gather + FP8 dequant, QK^T,
softmax with sink, PV, split-K partials, combine) over the decode workload: 64 sequences x
16384 cached tokens, T = 64 query tokens, H = 64 heads, top-k 2048 (5% masked), FP8 KV,
per-head sink. Eight index sets (and query sets) rotate between steps so that every call
gathers its rows from HBM (8 x 81.7 MB of distinct rows > the 129 MB L2); the cache itself is
688 MB.

One JSON line is printed by rank 0. `value` is gathered-KV GB/s over all ranks; `e2e`
repeats the measurement with the step's inputs copied from pinned host memory and the
outputs copied back inside the timed region. With the default decode workload the same line
also carries the prefill (T=4096, H=32, topk=512, bf16) and large-prefill (T=8192, H=128,
topk=2048+128, FP8 + bf16 extra cache) workloads under config.prefill and
config.large_prefill, each timed for K steps with its own TFLOP/s roofline and an oracle
CPU baseline on a token sample. `--impl reference` times the fp64 CPU oracle (the only
other implementation this project has) on the same workload and metric.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-MLA prefill TFLOP/s & decode µs/call + GB/s, as % of roofline"
ROTATIONS = 8
# about half a second of timed GPU work per workload
DEFAULT_STEPS = {"decode": 6000, "prefill": 800, "large_prefill": 40, "tiny": 8000, "quantize": 200, "small_t": 1}


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0,
                    help="timed steps (default: the workload's, about half a second of GPU time, so the "
                         "20 ms clock samples fall inside the timed region)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="smla", choices=["smla", "reference"])
    ap.add_argument("--workload", default="decode", choices=["decode", "prefill", "large_prefill", "tiny", "quantize", "small_t"])
    ap.add_argument("--no-secondary", action="store_true",
                    help="decode only: leave the prefill, large-prefill and cache-writer workloads out of the line")
    ap.add_argument("--tokens", type=int, default=0,
                    help="prefill / large_prefill: time only the first N query tokens (smaller profiler captures)")
    args = ap.parse_args()
    args.steps_given = args.steps > 0
    if args.steps <= 0:
        args.steps = 50 if args.impl == "reference" else DEFAULT_STEPS[args.workload]
    return args


# ----------------------------------------------------------------------------- distributed
def dist_init(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl"
        try:
            import torch
            if not torch.cuda.is_available():
                backend = "gloo"
        except Exception:
            backend = "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- workloads
def workload_label(kind, T=0):
    """The workload's name in `config.workload`, the same for both arms (T: query tokens timed)."""
    return {"decode": "decode fp8: 64 seqs x 16384 ctx (688 MB cache), T=64, H=64, topk=2048 (5% -1), sink",
            "prefill": f"prefill bf16: 1 seq x 32768 ctx, T={T or 4096}, H=32, topk=512 causal, sink",
            "tiny": "tiny bf16: 1 seq x 256 ctx, T=4, H=16, topk=128, no sink",
            "large_prefill": (f"large prefill: 1 seq x 65536 ctx fp8 main + bf16 extra, T={T or 8192}, H=128, "
                              "topk=2048 causal + 128-token window, sink")}[kind]


def build_workloads(kind, tokens=0):
    from sparse_top_mla_gb300 import synth
    T = tokens if tokens > 0 else None
    if kind == "decode":
        base = synth.config(2)
        rots = [base]
        for r in range(1, ROTATIONS):
            rng = np.random.default_rng(2000 + r)
            idx = synth.mask_random(rng, synth.distinct_indices(rng, np.full(base.T, 16383), 2048), 0.05)
            q = synth.make_q(rng, base.T, base.H)
            rots.append(synth.replace(base, q=q, main=synth.replace(base.main, indices=idx)))
        return rots, workload_label("decode")
    if kind == "prefill":
        w = synth.config(3, T=T)
        return [w], workload_label("prefill", w.T)
    if kind == "tiny":
        return [synth.config(1)], workload_label("tiny")
    w = synth.config(4, T=T)
    return [w], workload_label("large_prefill", w.T)


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks/throttle reasons sampled every 20 ms; only the samples taken while the
    timed region ran (host wall-clock window) are summarised."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    @classmethod
    def once(cls, gpu_index):
        """One read-only sample (host time, csv line), or None without nvidia-smi."""
        try:
            r = subprocess.run(["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={cls.FIELDS}",
                                "--format=csv,noheader,nounits"], capture_output=True, text=True, timeout=10)
            return (time.time(), r.stdout.strip()) if r.returncode == 0 else None
        except (FileNotFoundError, subprocess.TimeoutExpired):
            return None

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []  # (host time, csv line)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "20"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except FileNotFoundError:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self, t0=None, t1=None, bracket=()):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.05)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        return self.summarise(self.lines, t0, t1, bracket)

    @classmethod
    def summarise(cls, lines, t0=None, t1=None, bracket=()):
        """Median SM clock and the throttle reasons seen in [t0, t1]. `bracket` holds the one-shot
        samples taken just before the timed region started and just after it ended; they are
        always summarised with the samples inside the window, so a region shorter than the
        20 ms sampling period still has a clock record next to it."""
        inside = [ln for t, ln in lines if (t0 is None or t >= t0) and (t1 is None or t <= t1)]
        edge = [b[1] for b in bracket if b is not None]
        use = inside + edge
        if not use and lines and t0 is not None:
            mid = (t0 + (t1 if t1 is not None else t0)) / 2
            use = [min(lines, key=lambda x: abs(x[0] - mid))[1]]
        sm, smax, reasons = [], None, set()
        for ln in use:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(cls.REASONS, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm), "samples_in_region": len(inside), "bracket_samples": len(edge)}


# ----------------------------------------------------------------------------- helpers
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "of measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "of fallback"}


# Source files that define or launch each workload's dominant kernel: a traffic figure stays
# valid while these are unchanged.
KERNEL_SOURCES = {
    "attention": ("smla_kernels.cu", "smla_ptx.cuh", "smla_internal.h", "smla_api.cu"),
    "quantize_kv": ("smla_quant.cu", "smla_ptx.cuh", "smla_internal.h"),
}


def kernel_source_hash(workload_key="decode"):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "sparse_top_mla_gb300", "csrc")
    for f in KERNEL_SOURCES["quantize_kv" if workload_key == "quantize_kv" else "attention"]:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(workload_key):
    """DRAM bytes per launch of the dominant kernel from the committed ncu summary, or None
    when that kernel's sources changed since the capture."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    d = json.load(open(path))
    e = d.get(workload_key)
    if not e or e.get("kernel_source_hash") != kernel_source_hash(workload_key):
        return None
    return e.get("dram_bytes_per_launch")


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ----------------------------------------------------------------------------- reference arm
def run_reference(args, world, rank):
    if rank != 0:
        return 0
    import oracle
    from sparse_top_mla_gb300 import synth
    oracle.build()
    if args.workload == "quantize":
        rng = np.random.default_rng(3000)
        x = synth.f32_to_bf16_bits(synth.normal_f32(rng, (65536, 576)))
        times = []
        for s in range(args.warmup + args.steps):
            t0 = time.perf_counter()
            oracle.pack_rows(x, 1)
            if s >= args.warmup:
                times.append(time.perf_counter() - t0)
        gbs = x.shape[0] * (1152 + 656 + 8) * len(times) / sum(times) / 1e9
        sample = "65536 bf16 latent rows per step (of the 1,048,576-row cache), fp64 oracle cache writer"
        print(json.dumps({"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
                          "steps": args.steps, "warmup": args.warmup, "ms_per_step": sum(times) / len(times) * 1e3,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
                          "data": "synthetic", "config": {"workload": "cache writer", "sample": sample},
                          "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": oracle.threads(0), "kind": "oracle",
                                           "sample": sample},
                          "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
                          "gpu_launches": 0}), flush=True)
        return 0
    w = {"decode": lambda: synth.config(2), "prefill": lambda: synth.config(3), "tiny": lambda: synth.config(1),
         "large_prefill": lambda: synth.config(4, T=64)}[args.workload]()
    per_tok = w.gathered_bytes() / w.T
    n_tok = {"decode": 64, "prefill": 256, "large_prefill": 16, "tiny": 4}[args.workload]
    threads = oracle.threads(0)
    times = []
    for s in range(args.warmup + args.steps):
        tok = (np.arange(n_tok) + s * n_tok) % w.T
        t0 = time.perf_counter()
        oracle.attention(w, tokens=tok, nthreads=threads)
        dt = time.perf_counter() - t0
        if s >= args.warmup:
            times.append(dt)
    total = sum(times)
    gbs = per_tok * n_tok * len(times) / total / 1e9
    sample = f"{n_tok} query tokens of the workload per step (of {w.T}); fp64 oracle"
    line = {"impl": "reference", "metric": METRIC, "value": gbs, "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / len(times) * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": workload_label(args.workload, args.tokens), "sample": sample},
            "cpu_baseline": {"value": gbs, "unit": "GB/s", "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": gbs, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- smla arm
def time_workload(kind, steps, warmup, world, rank, local, with_e2e=True, tokens=0):
    import torch
    from sparse_top_mla_gb300 import binding
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    rots, label = build_workloads(kind, tokens)
    probs = [binding.DeviceProblem(rots[0], device=dev)]
    # the other rotations share the first rotation's device cache (only q and indices differ)
    for w in rots[1:]:
        probs.append(binding.DeviceProblem(w, device=dev, share_caches_with=probs[0]))
    for p in probs:
        p.ensure_workspace()
    w0 = rots[0]
    gathered = [w.gathered_bytes() for w in rots]
    flops = w0.flops()
    idx_bytes = sum(w0.main.indices[:, :w0.main.topk].nbytes for _ in [0]) + (
        w0.extra.indices[:, :w0.extra.topk].nbytes if w0.extra is not None else 0)
    q_bytes = w0.T * w0.H * 576 * 2
    stream = torch.cuda.current_stream()
    # warm-up
    for s in range(warmup):
        binding.forward(probs[s % len(probs)].call, stream)
    torch.cuda.synchronize()
    assert binding.device_error() == 0
    # timed region. The dominant kernel is timed with events on every KSAMPLE-th step only: an
    # event recorded between two kernels stops the second from launching programmatically (early)
    # behind the first, so the other steps run as a plain stream of calls.
    # every k-th step, k odd (coprime with the 8 rotations, so the samples cover every index set)
    # and at least 7; long runs take ~200 samples, so the events perturb few calls
    ksample = max(7, steps // 200) | 1
    sampled = [s for s in range(steps) if s % ksample == 0]
    kev = {s: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for s in sampled}
    for a, b in kev.values():  # torch creates CUDA events lazily: record once so the handles exist
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.2)
    barrier(world)
    torch.cuda.synchronize()
    # inputs that fit in L2 are evicted before every timed step by a write larger than L2; each
    # step is then timed on its own and the flushes stay outside the sum
    flush = sum(input_mb(w) for w in rots) <= L2_MB
    scratch = torch.empty(2 * int(L2_MB) << 20, dtype=torch.uint8, device=dev) if flush else None
    sev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)] \
        if flush else []
    t_start = torch.cuda.Event(enable_timing=True)
    t_stop = torch.cuda.Event(enable_timing=True)
    before = ClockSampler.once(local)
    wall0 = time.time()
    t_start.record(stream)
    for s in range(steps):
        p = probs[s % len(probs)]
        if flush:
            scratch.fill_(s & 0xFF)
            sev[s][0].record(stream)
        if s in kev:
            binding.set_timing_events(kev[s][0], kev[s][1])
            binding.forward(p.call, stream)
            binding.set_timing_events(None, None)
        else:
            binding.forward(p.call, stream)
        if flush:
            sev[s][1].record(stream)
    t_stop.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    after = ClockSampler.once(local)
    barrier(world)
    binding.set_timing_events(None, None)
    clk = clocks.stop(wall0, wall1, (before, after))
    assert binding.device_error() == 0
    elapsed = sum(a.elapsed_time(b) for a, b in sev) if flush else t_start.elapsed_time(t_stop)
    total_ms = max_over_ranks(elapsed, world)
    kern_ms = [kev[s][0].elapsed_time(kev[s][1]) for s in sampled]
    bytes_steps = sum(gathered[s % len(probs)] for s in range(steps))
    value = bytes_steps * world / (total_ms * 1e-3) / 1e9
    # launches per step: attention kernel + combine when split-K is used
    splits_used = probs[0].workspace is not None and binding.workspace_size(probs[0].call) > 0
    decode_route = w0.T <= binding.decode_max_tokens(w0.H, w0.main.topk + (w0.extra.topk if w0.extra else 0),
                                                      w0.main.fmt)
    launches_per_step = 2 if (decode_route and splits_used) else 1

    peaks = measured_peaks()
    kern_avg_ms = sum(kern_ms) / len(kern_ms)
    res = {"label": label, "w0": w0, "value": value, "total_ms": total_ms, "steps": steps, "l2_flush": flush,
           "ms_per_step": total_ms / steps, "kern_avg_ms": kern_avg_ms, "kern_samples": len(kern_ms),
           "gathered": gathered[0], "flops": flops, "idx_bytes": idx_bytes, "q_bytes": q_bytes,
           "alg_bytes": w0.algorithmic_bytes(), "clocks": clk, "launches": launches_per_step * steps,
           "peaks": peaks, "probs": probs}
    if not with_e2e:
        return res

    # e2e: pinned host inputs -> device, forward, outputs -> pinned host, every step. Each
    # step's inputs (q, indices, token_seq, seq_lens, block table, sink) sit packed in one pinned
    # host buffer and are uploaded with one copy into one device buffer the call's tensors view;
    # O and LSE come back with one copy. The copies run on their own streams so they overlap the
    # kernels of neighbouring steps, as in a serving loop: uploads on the input stream, the
    # forwards on the compute stream once their inputs have landed, the downloads on the output
    # stream once the forwards are done (synchronised per group of steps, below). Every rotation
    # has its own device buffers, rewritten only after its previous forward and download
    # completed; host output buffers alternate between two groups.
    def packed(parts):
        offs, n = [], 0
        for a in parts:
            offs.append(n)
            n += (a.nbytes + 255) // 256 * 256
        return offs, n

    T, S = w0.T, w0.num_seqs
    e_calls, d_in, h_in, d_out = [], [], [], []
    for r, w in enumerate(rots):
        ex = w.extra
        arrs = [np.ascontiguousarray(w.q), np.ascontiguousarray(w.main.indices),
                np.ascontiguousarray(w.token_seq, dtype=np.int32), np.ascontiguousarray(w.main.seq_lens),
                np.ascontiguousarray(w.main.block_table),
                np.ascontiguousarray(w.sink) if w.sink is not None else np.zeros(0, np.float32)]
        if ex is not None:
            arrs += [np.ascontiguousarray(ex.indices), np.ascontiguousarray(ex.seq_lens),
                     np.ascontiguousarray(ex.block_table)]
        offs, n = packed(arrs)
        host = torch.zeros(n, dtype=torch.uint8).pin_memory()
        for a, o in zip(arrs, offs):
            host[o:o + a.nbytes].copy_(torch.from_numpy(a.view(np.uint8).reshape(-1)))
        dbuf = torch.empty(n, dtype=torch.uint8, device=dev)

        def view(i, dtype, shape):
            return dbuf[offs[i]:offs[i] + arrs[i].nbytes].view(dtype).view(shape)

        oo, on = packed([np.empty((T, w.H, 512), np.uint16), np.empty((T, w.H), np.float32)])
        obuf = torch.empty(on, dtype=torch.uint8, device=dev)
        main = binding.DeviceSet(probs[0].main.cache, w.main.fmt, w.main.row_stride, w.main.page_stride,
                                 w.main.num_pages, view(4, torch.int32, w.main.block_table.shape),
                                 view(3, torch.int32, w.main.seq_lens.shape), view(1, torch.int32, w.main.indices.shape),
                                 w.main.topk)
        extra = None
        if ex is not None:
            extra = binding.DeviceSet(probs[0].extra.cache, ex.fmt, ex.row_stride, ex.page_stride, ex.num_pages,
                                      view(8, torch.int32, ex.block_table.shape), view(7, torch.int32, ex.seq_lens.shape),
                                      view(6, torch.int32, ex.indices.shape), ex.topk)
        call = binding.Call(view(0, torch.bfloat16, w.q.shape), view(2, torch.int32, (T,)), main,
                            obuf[oo[0]:oo[0] + T * w.H * 1024].view(torch.bfloat16).view(T, w.H, 512),
                            obuf[oo[1]:oo[1] + T * w.H * 4].view(torch.float32).view(T, w.H), extra,
                            view(5, torch.float32, w.sink.shape) if w.sink is not None else None,
                            np.float32(w.sm_scale), None, num_seqs=w.num_seqs)
        call.set_workspace(probs[0].workspace)
        e_calls.append(call)
        d_in.append(dbuf)
        h_in.append(host)
        d_out.append(obuf)
    h2d = h_in[0].numel()
    d2h = d_out[0].numel()
    # steps go in groups of G: one event per group orders the group's uploads before its
    # forwards, the forwards before the group's downloads, and a rotation's reuse after its
    # previous group; inside a group the forwards follow each other directly, so each call's
    # kernels launch behind the previous call's without a synchronisation between them
    nrot = len(e_calls)
    G = 4 if nrot % 4 == 0 and nrot >= 8 else 1  # single-rotation workloads: a group per step
    # up to 400 steps (~24 ms at decode), so filling and draining the copy pipeline (the first
    # group's uploads, the last group's downloads) is a small part of the timed region
    e2e_steps = max(G, (min(steps, 400) // G) * G)
    ngroups = e2e_steps // G
    h_out = [torch.empty(d_out[0].numel(), dtype=torch.uint8).pin_memory() for _ in range(2 * G)]
    s_in = torch.cuda.Stream(device=dev)
    s_out = torch.cuda.Stream(device=dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    up_done = [ev() for _ in range(ngroups)]
    fwd_done = [ev() for _ in range(ngroups)]
    down_done = [ev() for _ in range(ngroups)]
    for c in e_calls[:1]:  # one untimed pass through this path
        d_in[0].copy_(h_in[0])
        binding.forward(c, stream)
    barrier(world)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    gpr = nrot // G  # groups per rotation cycle
    for g in range(ngroups):
        with torch.cuda.stream(s_in):
            if g >= gpr:
                s_in.wait_event(fwd_done[g - gpr])  # these rotations' previous forwards read their inputs
            for k in range(G):
                r = (g * G + k) % nrot
                d_in[r].copy_(h_in[r], non_blocking=True)
            up_done[g].record(s_in)
        stream.wait_event(up_done[g])
        if g >= gpr:
            stream.wait_event(down_done[g - gpr])  # these rotations' previous outputs were read back
        for k in range(G):
            binding.forward(e_calls[(g * G + k) % nrot], stream)
        fwd_done[g].record(stream)
        with torch.cuda.stream(s_out):
            s_out.wait_event(fwd_done[g])
            for k in range(G):
                r = (g * G + k) % nrot
                h_out[(g & 1) * G + k].copy_(d_out[r], non_blocking=True)
            down_done[g].record(s_out)
    stream.wait_event(down_done[ngroups - 1])
    stream.wait_event(up_done[ngroups - 1])
    e1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    e2e_value = sum(gathered[s % len(probs)] for s in range(e2e_steps)) * world / (e2e_ms * 1e-3) / 1e9

    res["e2e"] = {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                  "steps": e2e_steps}
    return res


def cpu_baseline_tokens(kind, n_tok):
    """The oracle on a seeded sample of n_tok query tokens of a prefill workload, scaled to
    TFLOP/s (tokens are independent, so work is proportional to the tokens computed)."""
    import oracle
    from sparse_top_mla_gb300 import synth
    oracle.build()
    w = synth.config(3) if kind == "prefill" else synth.config(4)
    tok = np.sort(np.random.default_rng(99).choice(w.T, size=n_tok, replace=False))
    threads = oracle.threads(0)
    t0 = time.perf_counter()
    oracle.attention(w, tokens=tok, nthreads=threads)
    dt = time.perf_counter() - t0
    flops = w.flops() * n_tok / w.T
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{n_tok} of {w.T} query tokens (seeded), all heads and entries, fp64 oracle",
            "seconds": dt}


def cpu_baseline_decode():
    import oracle
    from sparse_top_mla_gb300 import synth
    oracle.build()
    w = synth.config(2)
    threads = oracle.threads(0)
    t0 = time.perf_counter()
    oracle.attention(w, nthreads=threads)
    dt = time.perf_counter() - t0
    return {"value": w.gathered_bytes() / dt / 1e9, "unit": "GB/s", "cores": threads, "kind": "oracle",
            "sample": "the whole decode batch (64 tokens x 64 heads x 2048 entries), one pass, fp64 oracle",
            "seconds": dt}


def roofline_for(kind, r):
    peaks = r["peaks"]
    if kind in ("decode", "tiny"):
        # algorithmic bytes of one call (valid gathered rows, indices, q, O, LSE) over the
        # dominant kernel's time; the gathered-rows-only fraction is reported beside it
        alg = r["alg_bytes"]
        ks = r["kern_avg_ms"] * 1e-3
        achieved = alg / ks / 1e9
        return {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"], "traffic": ncu_traffic(kind),
                "algorithmic_bytes_per_launch": alg,
                "frac_gathered": r["gathered"] / ks / 1e9 / peaks["hbm_gbs"],
                "frac_call": alg / (r["ms_per_step"] * 1e-3) / 1e9 / peaks["hbm_gbs"],
                "kernel": "sparse_mla_kernel<%d> (split-K partials)" % (64 if kind == "decode" else 16),
                "peak_source": peaks["source"] + " (hbm_gbs, STREAM-style copy)"}
    achieved = r["flops"] / (r["kern_avg_ms"] * 1e-3) / 1e12
    pk = peaks["bf16_tflops"]
    return {"bound": "tensor", "achieved": achieved, "peak": pk, "unit": "TFLOP/s", "frac": achieved / pk,
            "traffic": ncu_traffic(kind), "algorithmic_flops_per_launch": r["flops"],
            "frac_sustained": achieved / peaks["bf16_tflops_sustained"] if peaks.get("bf16_tflops_sustained")
            else None,
            "peak_source": peaks["source"] + " (bf16_tflops burst, cuBLAS; frac_sustained against the "
                                             "sustained figure)"}


L2_MB = 129.0


def input_mb(w):
    """MB of one input set: q, the caches and the index lists."""
    sets = [w.main] + ([w.extra] if w.extra is not None else [])
    return (w.q.nbytes + sum(st.cache.nbytes + st.indices.nbytes for st in sets)) / 1e6


def l2_note(w, flushed):
    """How the timed steps relate to the 129 MB L2."""
    sets = [w.main] + ([w.extra] if w.extra is not None else [])
    q_mb = w.q.nbytes / 1e6
    cache_mb = sum(st.cache.nbytes for st in sets) / 1e6
    idx_mb = sum(st.indices.nbytes for st in sets) / 1e6
    parts = f"q {q_mb:.1f} MB + cache {cache_mb:.1f} MB + indices {idx_mb:.1f} MB"
    if flushed:
        return (f"L2 flushed before every timed step (a {2 * int(L2_MB)} MB write, outside the timed sum): "
                f"inputs ({parts}) fit in L2")
    return f"inputs larger than L2: {parts}, one input set; cache rows are reused within a call, as in serving"


def line_for(kind, r, args, world, cpu):
    w0 = r["w0"]
    us = r["ms_per_step"] * 1e3
    rl = roofline_for(kind, r)
    d = {"metric": METRIC, "value": r["value"], "unit": "GB/s", "n_gpus": world, "steps": r["steps"],
         "warmup": args.warmup, "ms_per_step": r["ms_per_step"], "higher_is_better": True,
         "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
         "config": {"workload": r["label"], "l2": ("inputs larger than L2: 8 rotating index/query sets over a "
                                                   "688 MB cache (654 MB of distinct gathered rows)")
                    if kind == "decode" else l2_note(w0, r["l2_flush"]),
                    "us_per_call": us, "tflops": r["flops"] / (r["ms_per_step"] * 1e-3) / 1e12,
                    "kernel_avg_us": r["kern_avg_ms"] * 1e3, "kernel_timed_steps": r["kern_samples"],
                    "gathered_bytes_per_call": r["gathered"]},
         "roofline": rl, "clocks": r["clocks"], "e2e": r["e2e"], "gpu_launches": r["launches"]}
    if cpu is not None:
        d["cpu_baseline"] = cpu
    return d


def time_quantize(steps, warmup, world, local):
    """The device cache writer over the decode cache: 64 x 16384 rows of bf16 latents (1.2 GB)
    packed into FP8 rows (688 MB) at shuffled physical slots. HBM-bound: every row reads 1152
    bytes and writes 656."""
    import torch
    from sparse_top_mla_gb300 import binding, synth
    dev = torch.device(f"cuda:{local}")
    n = 64 * 16384
    rng = np.random.default_rng(3000)
    # bf16 latents ~N(0,1), drawn in chunks by the seeded generator
    kv = torch.empty((n, 576), dtype=torch.bfloat16, device=dev)
    chunk = 65536
    for c0 in range(0, n, chunk):
        x = synth.normal_f32(rng, (chunk, 576))
        kv[c0:c0 + chunk].view(torch.int16).copy_(torch.from_numpy(synth.f32_to_bf16_bits(x).view(np.int16)))
    slots = torch.from_numpy(rng.permutation(n).astype(np.int64)).to(dev)
    cache = torch.empty(n * 656, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        binding.quantize_kv(kv, slots, cache, 1, 656, 64 * 656, n // 64, stream)
    torch.cuda.synchronize()
    barrier(world)
    before = ClockSampler.once(local)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        binding.quantize_kv(kv, slots, cache, 1, 656, 64 * 656, n // 64, stream)
    e1.record(stream)
    torch.cuda.synchronize()
    after = ClockSampler.once(local)
    barrier(world)
    ms = max_over_ranks(e0.elapsed_time(e1), world) / steps
    peaks = measured_peaks()
    alg = n * (1152 + 656 + 8)  # bf16 row in, fp8 row out, slot id
    gbs = alg / (ms * 1e-3) / 1e9
    return {"workload": "cache writer: 1,048,576 bf16 latent rows -> FP8 rows (656 B) at shuffled slots",
            "value": gbs * world, "unit": "GB/s", "us_per_call": ms * 1e3, "steps": steps,
            "rows_per_call": n, "l2": "inputs larger than L2: 1.2 GB of bf16 rows in, 688 MB of FP8 rows out",
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "traffic": ncu_traffic("quantize_kv"),
                         "algorithmic_bytes_per_launch": alg, "kernel": "quantize_kv_kernel",
                         "peak_source": peaks["source"] + " (hbm_gbs, STREAM-style copy)"},
            "clocks": ClockSampler.summarise([], None, None, (before, after)), "gpu_launches": steps}


def time_small_t(probs):
    """Small-T latency on the decode workload's cache and queries: T = 1, 16, 64 query tokens,
    H = 64, the first 512 of each token's entries (topk = 512, FP8), one call per rotation, through
    the crossover dispatch. us_per_call: GPU time per call from a CUDA-graph replay of the rotating
    calls (host submission excluded, best of 5); attention_launch_us: CUDA events recorded on the
    stream around the attention kernel's launch alone (median of 32 calls): the kernel and its launch
    latency, without the overlap with the neighbouring calls that the replay has, and without the
    combine. The kernels' own durations come from a profiler's launch list of --workload small_t."""
    import statistics
    import numpy as np
    import torch
    from sparse_top_mla_gb300 import binding, calibrate
    stream = torch.cuda.current_stream()
    res, launches = {}, 0
    for T in (1, 16, 64):
        calls = []
        for p in probs[:4]:
            m = p.main
            main = binding.DeviceSet(m.cache, m.format, m.row_stride, m.page_stride, m.num_pages, m.block_table,
                                     m.seq_lens, m.indices[:T, :512], 512)
            calls.append(binding.Call(p.q[:T], p.token_seq[:T], main, p.out[:T], p.lse[:T], None, p.sink,
                                      np.float32(p.w.sm_scale), None, num_seqs=p.w.num_seqs))
        need = max(binding.workspace_size(c) for c in calls)
        ws = torch.empty(need, dtype=torch.uint8, device=probs[0].device) if need else None
        for c in calls:
            c.set_workspace(ws)
        split = T <= binding.decode_max_tokens(64, 512, probs[0].main.format)
        reps, inner = 5, 4
        us = calibrate.graph_time_us(binding.forward, calls, stream, reps, inner)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(32)]
        for a, b in evs:
            a.record(stream)
            b.record(stream)
        torch.cuda.synchronize()
        for i, (a, b) in enumerate(evs):
            binding.set_timing_events(a, b)
            binding.forward(calls[i % len(calls)], stream)
        binding.set_timing_events(None, None)
        torch.cuda.synchronize()
        assert binding.device_error() == 0
        ker = statistics.median(a.elapsed_time(b) * 1e3 for a, b in evs)
        res[f"T={T}"] = {"us_per_call": round(us, 2), "attention_launch_us": round(ker, 2),
                         "schedule": "split-K + combine" if split else "whole items"}
        ncalls = len(calls) * (1 + inner * (1 + reps)) + len(evs)
        launches += ncalls * (2 if split else 1)
    res["workload"] = ("decode cache (64 seqs x 16384 ctx, FP8), H=64, first 512 entries of each token "
                       "(5% -1), sink; 4 rotating query/index sets")
    return res, launches


def secondary_for(kind, r, cpu):
    """The prefill-type workload as a sub-object of the decode line (TFLOP/s headline)."""
    us = r["ms_per_step"] * 1e3
    d = {"workload": r["label"], "value": r["flops"] / (r["ms_per_step"] * 1e-3) / 1e12, "unit": "TFLOP/s",
         "us_per_call": us, "kernel_avg_us": r["kern_avg_ms"] * 1e3, "kernel_timed_steps": r["kern_samples"],
         "steps": r["steps"], "gathered_bytes_per_call": r["gathered"],
         "gathered_gbs": r["gathered"] / (r["ms_per_step"] * 1e-3) / 1e9,
         "l2": l2_note(r["w0"], r["l2_flush"]), "roofline": roofline_for(kind, r), "clocks": r["clocks"],
         "gpu_launches": r["launches"]}
    if cpu is not None:
        d["cpu_baseline"] = cpu
    return d


def main():
    args = parse()
    world, rank, local = dist_init(args.gpus)
    if args.impl == "reference":
        rc = run_reference(args, world, rank)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return rc
    from sparse_top_mla_gb300 import build as smla_build
    if rank == 0:
        smla_build.build()
    barrier(world)
    if args.workload == "small_t":
        import torch
        from sparse_top_mla_gb300 import binding
        dev = torch.device(f"cuda:{local}")
        torch.cuda.set_device(dev)
        rots, _ = build_workloads("decode")
        probs = [binding.DeviceProblem(rots[0], device=dev)]
        probs += [binding.DeviceProblem(w, device=dev, share_caches_with=probs[0]) for w in rots[1:4]]
        st, n = time_small_t(probs)
        if rank == 0:
            line = {"metric": METRIC, "value": st["T=1"]["us_per_call"], "unit": "us/call", "n_gpus": world,
                    "steps": args.steps, "warmup": args.warmup, "ms_per_step": st["T=1"]["us_per_call"] / 1e3,
                    "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                    "data": "synthetic", "config": {"workload": "small T (value: T=1): " + st["workload"],
                                                    "small_t": st}, "gpu_launches": n}
            print(json.dumps(line), flush=True)
        return 0
    if args.workload == "quantize":
        qr = time_quantize(args.steps, args.warmup, world, local)
        if rank == 0:
            line = {"metric": METRIC, "value": qr["value"], "unit": "GB/s", "n_gpus": world, "steps": args.steps,
                    "warmup": args.warmup, "ms_per_step": qr["us_per_call"] / 1e3, "higher_is_better": True,
                    "scaling": "weak", "vs_baseline": None, "dtype": "bf16->e4m3", "data": "synthetic",
                    "config": {"workload": qr["workload"], "l2": qr["l2"]}, "roofline": qr["roofline"],
                    "clocks": qr["clocks"], "gpu_launches": qr["gpu_launches"]}
            print(json.dumps(line), flush=True)
        return 0
    r = time_workload(args.workload, args.steps, args.warmup, world, rank, local, True, args.tokens)
    cpu = cpu_baseline_decode() if (rank == 0 and world == 1 and args.workload == "decode") else None
    line = line_for(args.workload, r, args, world, cpu)
    if args.workload == "decode" and not args.no_secondary:
        line["config"]["small_t"], n_small = time_small_t(r.pop("probs"))
        line["gpu_launches"] += n_small
        # the prefill half of the metric, in the same line: each workload timed for the same
        # number of steps when --steps is given, else for its own default (about half a second)
        for kind, n_tok in (("prefill", 256), ("large_prefill", 16)):
            steps = args.steps if args.steps_given else DEFAULT_STEPS[kind]
            rr = time_workload(kind, steps, args.warmup, world, rank, local, False, args.tokens)
            cpu_k = cpu_baseline_tokens(kind, n_tok) if (rank == 0 and world == 1) else None
            rr.pop("probs", None)
            line["config"][kind] = secondary_for(kind, rr, cpu_k)
            line["gpu_launches"] += rr["launches"]
            import torch
            torch.cuda.empty_cache()
        qsteps = args.steps if args.steps_given else 200
        line["config"]["quantize_kv"] = time_quantize(qsteps, args.warmup, world, local)
        line["gpu_launches"] += qsteps
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
