"""ctypes binding of libsmla (include/smla.h): argument marshalling only.

Every step of the computation runs in the CUDA library; this module fills the C structs
from torch CUDA tensors (device memory and streams are torch's) and calls the entry
points with the same names. If the library has not been built it raises: there is no
CPU fallback.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsmla.so")
CROSSOVER_TABLE = os.path.join(HERE, "crossover_gb300.json")

SMLA_OK, SMLA_ERR_INVALID, SMLA_ERR_UNSUPPORTED, SMLA_ERR_WORKSPACE, SMLA_ERR_CUDA, SMLA_ERR_DEVICE = range(6)
KV_BF16, KV_FP8 = 0, 1

EXPORTS = ("smla_supported", "smla_workspace_size", "smla_prefill", "smla_decode", "smla_decode_static",
           "smla_forward", "smla_quantize_kv",
           "smla_decode_max_tokens", "smla_set_crossover", "smla_load_crossover", "smla_status_string",
           "smla_device_error", "smla_last_error", "smla_set_timing_events", "smla_struct_size", "smla_version")


class SmlaError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: status {status}")
        self.status = status


class KvSet(ctypes.Structure):
    _fields_ = [("cache", ctypes.c_void_p), ("format", ctypes.c_int32), ("row_stride_bytes", ctypes.c_int64),
                ("page_stride_bytes", ctypes.c_int64), ("page_size", ctypes.c_int32),
                ("num_pages", ctypes.c_int32), ("block_table", ctypes.c_void_p), ("bt_stride", ctypes.c_int32),
                ("seq_lens", ctypes.c_void_p), ("indices", ctypes.c_void_p), ("idx_stride", ctypes.c_int64),
                ("topk", ctypes.c_int32), ("topk_length", ctypes.c_void_p)]


class Params(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("d_qk", ctypes.c_int32), ("d_v", ctypes.c_int32),
                ("num_seqs", ctypes.c_int32), ("q", ctypes.c_void_p), ("q_stride_t", ctypes.c_int64),
                ("q_stride_h", ctypes.c_int64), ("token_seq", ctypes.c_void_p), ("main", KvSet),
                ("extra", ctypes.c_void_p), ("sink", ctypes.c_void_p), ("sm_scale", ctypes.c_float),
                ("out", ctypes.c_void_p), ("out_stride_t", ctypes.c_int64), ("out_stride_h", ctypes.c_int64),
                ("lse", ctypes.c_void_p), ("lse_stride_t", ctypes.c_int64), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t)]


_lib = None


def load(path: Optional[str] = None):
    """Load libsmla.so (built by sparse_top_mla_gb300.build). Raises if it is missing."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with `python -m sparse_top_mla_gb300.build` "
                           "(nvcc, sm_103a). There is no CPU fallback.")
    lib = ctypes.CDLL(p)
    P = ctypes.POINTER(Params)
    vp = ctypes.c_void_p
    sig = {
        "smla_supported": ([P, ctypes.c_char_p, ctypes.c_size_t], ctypes.c_int),
        "smla_workspace_size": ([P], ctypes.c_size_t),
        "smla_prefill": ([P, vp], ctypes.c_int),
        "smla_decode": ([P, vp], ctypes.c_int),
        "smla_decode_static": ([P, vp], ctypes.c_int),
        "smla_forward": ([P, vp], ctypes.c_int),
        "smla_quantize_kv": ([vp, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, vp, vp, ctypes.c_int32,
                              ctypes.c_int64, ctypes.c_int64, ctypes.c_int32, vp], ctypes.c_int),
        "smla_decode_max_tokens": ([ctypes.c_int32, ctypes.c_int32, ctypes.c_int32], ctypes.c_int32),
        "smla_set_crossover": ([ctypes.POINTER(ctypes.c_int32), ctypes.c_int32], ctypes.c_int),
        "smla_load_crossover": ([ctypes.c_char_p], ctypes.c_int),
        "smla_status_string": ([ctypes.c_int], ctypes.c_char_p),
        "smla_device_error": ([ctypes.POINTER(ctypes.c_int32)], ctypes.c_int),
        "smla_last_error": ([], ctypes.c_char_p),
        "smla_set_timing_events": ([vp, vp], ctypes.c_int),
        "smla_struct_size": ([ctypes.c_int32], ctypes.c_size_t),
        "smla_version": ([], ctypes.c_int32),
    }
    for name, (args, res) in sig.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    if lib.smla_struct_size(0) != ctypes.sizeof(Params) or lib.smla_struct_size(1) != ctypes.sizeof(KvSet):
        raise RuntimeError("libsmla ABI mismatch: struct sizes differ from this binding")
    if path is None:
        _lib = lib
        # the decode/prefill crossover measured on this GPU model by sparse_top_mla_gb300.calibrate
        # (smla_forward falls back to the library's analytical default without it)
        if os.path.exists(CROSSOVER_TABLE):
            lib.smla_load_crossover(CROSSOVER_TABLE.encode())
    return lib


def use_library(path: str):
    """Load the library at `path` (an instrumented build, for instance) and make it the one every
    call of this module uses, with this GPU model's crossover table."""
    global _lib
    lib = load(path)
    _lib = lib
    if os.path.exists(CROSSOVER_TABLE):
        lib.smla_load_crossover(CROSSOVER_TABLE.encode())
    return lib


def status_string(st: int) -> str:
    return load().smla_status_string(st).decode()


def _check(st: int, what: str, call=None):
    if st != SMLA_OK:
        reason = ""
        if call is not None and st in (SMLA_ERR_INVALID, SMLA_ERR_UNSUPPORTED):
            reason = " (" + supported(call)[1] + ")"
        elif st == SMLA_ERR_CUDA:
            reason = " (" + load().smla_last_error().decode() + ")"
        raise SmlaError(st, f"{what} failed: {status_string(st)}{reason}")


@dataclass
class DeviceSet:
    """Device tensors of one cache + index set (torch tensors on one CUDA device)."""
    cache: "object"
    format: int
    row_stride: int
    page_stride: int
    num_pages: int
    block_table: "object"
    seq_lens: "object"
    indices: "object"
    topk: int
    topk_length: "object" = None

    def struct(self) -> KvSet:
        return KvSet(self.cache.data_ptr(), self.format, self.row_stride, self.page_stride, 64, self.num_pages,
                     self.block_table.data_ptr(), row_stride(self.block_table), self.seq_lens.data_ptr(),
                     self.indices.data_ptr(), row_stride(self.indices), self.topk,
                     None if self.topk_length is None else self.topk_length.data_ptr())


def row_stride(t, dim: int = 0) -> int:
    """Stride of dim in elements; a size-1 dim reports the dense extent of the dims after it
    (torch keeps arbitrary strides, even 0, on size-1 dims)."""
    if t.shape[dim] > 1:
        return t.stride(dim)
    n = 1
    for d in range(dim + 1, t.dim()):
        n = max(n, t.stride(d) * t.shape[d])
    return n


class Call:
    """Holds a filled smla_params struct plus references to everything it points at."""

    def __init__(self, q, token_seq, main: DeviceSet, out, lse=None, extra: Optional[DeviceSet] = None,
                 sink=None, sm_scale: float = 576 ** -0.5, workspace=None, num_seqs: Optional[int] = None):
        import torch
        assert q.dtype == torch.bfloat16 and q.stride(2) == 1
        assert out.dtype == torch.bfloat16 and out.stride(2) == 1
        T, H = q.shape[0], q.shape[1]
        self.keep = [q, token_seq, main, out, lse, extra, sink, workspace]
        self.extra_struct = extra.struct() if extra is not None else None
        ns = num_seqs if num_seqs is not None else main.seq_lens.shape[0]
        self.p = Params(T, H, 576, 512, ns, q.data_ptr(), row_stride(q, 0), row_stride(q, 1), token_seq.data_ptr(),
                        main.struct(),
                        ctypes.addressof(self.extra_struct) if self.extra_struct is not None else None,
                        None if sink is None else sink.data_ptr(), float(sm_scale), out.data_ptr(),
                        row_stride(out, 0), row_stride(out, 1), None if lse is None else lse.data_ptr(),
                        0 if lse is None else row_stride(lse, 0),
                        None if workspace is None else workspace.data_ptr(),
                        0 if workspace is None else workspace.numel() * workspace.element_size())

    def set_workspace(self, ws):
        self.keep[7] = ws
        self.p.workspace = None if ws is None else ws.data_ptr()
        self.p.workspace_bytes = 0 if ws is None else ws.numel() * ws.element_size()

    def ref(self):
        return ctypes.byref(self.p)


def supported(call: Call) -> tuple[bool, str]:
    buf = ctypes.create_string_buffer(512)
    ok = load().smla_supported(call.ref(), buf, 512)
    return bool(ok), buf.value.decode()


def workspace_size(call: Call) -> int:
    return int(load().smla_workspace_size(call.ref()))


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def prefill(call: Call, stream=None, check: bool = True) -> int:
    st = load().smla_prefill(call.ref(), _stream(stream))
    if check:
        _check(st, "smla_prefill", call)
    return st


def decode(call: Call, stream=None, check: bool = True) -> int:
    st = load().smla_decode(call.ref(), _stream(stream))
    if check:
        _check(st, "smla_decode", call)
    return st


def decode_static(call: Call, stream=None, check: bool = True) -> int:
    """smla_decode_static: split-K decode with the library's own fixed scratch (no workspace)."""
    st = load().smla_decode_static(call.ref(), _stream(stream))
    if check:
        _check(st, "smla_decode_static", call)
    return st


def forward(call: Call, stream=None, check: bool = True) -> int:
    st = load().smla_forward(call.ref(), _stream(stream))
    if check:
        _check(st, "smla_forward", call)
    return st


def quantize_kv(kv, slots, cache, fmt: int, row_stride: int, page_stride: int, num_pages: int, stream=None,
                check: bool = True) -> int:
    """smla_quantize_kv: pack rows of kv (torch bf16 or float32 [n, 576], row stride >= 576) into
    the device cache (uint8 tensor) at physical slots (int64 [n], page * 64 + row)."""
    import torch
    assert kv.dim() == 2 and kv.shape[1] == 576 and kv.stride(1) == 1
    assert kv.dtype in (torch.bfloat16, torch.float32) and slots.dtype == torch.int64
    dtype = 1 if kv.dtype == torch.float32 else 0
    st = load().smla_quantize_kv(kv.data_ptr(), dtype, row_stride_of(kv), kv.shape[0], slots.data_ptr(),
                                 cache.data_ptr(), fmt, row_stride, page_stride, num_pages, _stream(stream))
    if check:
        _check(st, "smla_quantize_kv")
    return st


def row_stride_of(t) -> int:
    return row_stride(t, 0)


def decode_max_tokens(H: int, topk_total: int, fmt: int) -> int:
    return int(load().smla_decode_max_tokens(H, topk_total, fmt))


def set_crossover(entries) -> None:
    flat = [int(v) for e in entries for v in e]
    arr = (ctypes.c_int32 * max(1, len(flat)))(*flat)
    _check(load().smla_set_crossover(arr, len(flat) // 4), "smla_set_crossover")


def load_crossover(path: str) -> int:
    return load().smla_load_crossover(path.encode())


def device_error() -> int:
    code = ctypes.c_int32(0)
    st = load().smla_device_error(ctypes.byref(code))
    if st not in (SMLA_OK, SMLA_ERR_DEVICE):
        _check(st, "smla_device_error")
    return int(code.value)


def set_timing_events(start=None, stop=None) -> None:
    """Hand two recorded torch.cuda.Event objects to the library's measurement hook."""
    a = None if start is None else ctypes.c_void_p(start.cuda_event)
    b = None if stop is None else ctypes.c_void_p(stop.cuda_event)
    if (start is not None and not a.value) or (stop is not None and not b.value):
        raise ValueError("timing events must have been recorded once (torch creates them lazily)")
    _check(load().smla_set_timing_events(a, b), "smla_set_timing_events")


# ---------------------------------------------------------------------------------------
# host workload -> device tensors (byte copies only)
# ---------------------------------------------------------------------------------------
def upload_set(s, device, cache=None) -> DeviceSet:
    """Copy one set's arrays to the device (reusing `cache`, a device tensor, when given)."""
    import torch
    t = lambda a: torch.from_numpy(a).to(device)  # noqa: E731
    return DeviceSet(t(s.cache) if cache is None else cache, s.fmt, s.row_stride, s.page_stride, s.num_pages, t(s.block_table),
                     t(s.seq_lens), t(s.indices), s.topk, None if s.topk_length is None else t(s.topk_length))


class DeviceProblem:
    """A synth.Workload copied to one GPU, with output buffers and a ready Call."""

    def __init__(self, w, device="cuda", lse: bool = True, out_pad: int = 0, lse_pad: int = 0,
                 q_pad: tuple = (0, 0), share_caches_with: "Optional[DeviceProblem]" = None):
        import numpy as np
        import torch
        self.w = w
        self.device = torch.device(device)
        qc = np.ascontiguousarray(w.q).view(np.int16)
        hp, cp = q_pad
        q_full = torch.zeros((w.T, w.H + hp, 576 + cp), dtype=torch.int16, device=self.device)
        q_full[:, :w.H, :576] = torch.from_numpy(qc).to(self.device)
        self.q = q_full.view(torch.bfloat16)[:, :w.H, :576]
        self.token_seq = torch.from_numpy(np.ascontiguousarray(w.token_seq, dtype=np.int32)).to(self.device)
        src = share_caches_with
        self.main = upload_set(w.main, self.device, None if src is None else src.main.cache)
        self.extra = (upload_set(w.extra, self.device, None if src is None or src.extra is None else src.extra.cache)
                      if w.extra is not None else None)
        self.sink = torch.from_numpy(w.sink).to(self.device) if w.sink is not None else None
        self.out_full = torch.full((w.T, w.H, 512 + out_pad), float("nan"), dtype=torch.bfloat16, device=self.device)
        self.out = self.out_full[:, :, :512]
        self.lse_full = torch.full((w.T, w.H + lse_pad), float("nan"), dtype=torch.float32,
                                   device=self.device) if lse else None
        self.lse = self.lse_full[:, :w.H] if lse else None
        self.call = Call(self.q, self.token_seq, self.main, self.out, self.lse, self.extra, self.sink,
                         np.float32(w.sm_scale), None, num_seqs=w.num_seqs)
        self.workspace = None

    def ensure_workspace(self):
        import torch
        n = workspace_size(self.call)
        if n and (self.workspace is None or self.workspace.numel() < n):
            self.workspace = torch.empty(n, dtype=torch.uint8, device=self.device)
            self.call.set_workspace(self.workspace)
        return n

    def run(self, mode: str = "forward", stream=None):
        if mode in ("decode", "forward"):
            self.ensure_workspace()
        fn = {"forward": forward, "prefill": prefill, "decode": decode}[mode]
        return fn(self.call, stream)

    def results(self):
        """(O float64 [T,H,512], LSE float64 [T,H]) copied back to the host."""
        import torch
        torch.cuda.synchronize(self.device)
        O = self.out.float().cpu().double().numpy()
        L = self.lse.cpu().double().numpy() if self.lse is not None else None
        return O, L
