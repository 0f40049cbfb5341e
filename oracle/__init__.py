"""CPU fp64 oracle for sparse top-k MLA attention — TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import this package. The CUDA library never loads it and shares no code with it.
The arithmetic lives in ``smla_oracle.cpp`` (plain C++17, fp64); this module builds it
with g++ and marshals numpy arrays into its C ABI.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "smla_oracle.cpp")
_LIB = os.path.join(_HERE, "libsmla_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (no fast-math, no FMA contraction: same results on x86 and Arm)."""
    with _lock:
        fresh = os.path.exists(_LIB) and os.path.getmtime(_LIB) >= max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "smla_oracle.h")))
        if force or not fresh:
            tmp = _LIB + f".tmp{os.getpid()}"
            cmd = ["g++", "-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
                   "-pthread", _SRC, "-o", tmp]
            subprocess.run(cmd, check=True)
            os.replace(tmp, _LIB)
    return _LIB


class _KVSet(ctypes.Structure):
    _fields_ = [("cache", ctypes.c_void_p), ("fmt", ctypes.c_int32), ("row_stride", ctypes.c_int64),
                ("page_stride", ctypes.c_int64), ("num_pages", ctypes.c_int32),
                ("block_table", ctypes.c_void_p), ("bt_stride", ctypes.c_int32),
                ("seq_lens", ctypes.c_void_p), ("indices", ctypes.c_void_p),
                ("idx_stride", ctypes.c_int64), ("topk", ctypes.c_int32),
                ("topk_length", ctypes.c_void_p)]


class _Problem(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("num_seqs", ctypes.c_int32),
                ("q", ctypes.c_void_p), ("q_stride_t", ctypes.c_int64), ("q_stride_h", ctypes.c_int64),
                ("token_seq", ctypes.c_void_p), ("main", _KVSet), ("extra", ctypes.c_void_p),
                ("sink", ctypes.c_void_p), ("sm_scale", ctypes.c_float)]


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        lib.oracle_attention.argtypes = [ctypes.POINTER(_Problem), ctypes.c_void_p, ctypes.c_int32,
                                         ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int32]
        lib.oracle_attention.restype = ctypes.c_int
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_value.restype = ctypes.c_double
        lib.oracle_bf16_value.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_value.restype = ctypes.c_double
        lib.oracle_pack_rows.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32,
                                         ctypes.c_int32, ctypes.c_void_p]
        lib.oracle_pack_rows.restype = ctypes.c_int
        lib.oracle_threads.argtypes = [ctypes.c_int32]
        lib.oracle_threads.restype = ctypes.c_int32
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _kvset(s, keep):
    for a in (s.cache, s.block_table, s.seq_lens, s.indices):
        assert a.flags["C_CONTIGUOUS"]
    tl = None if s.topk_length is None else np.ascontiguousarray(s.topk_length, dtype=np.int32)
    keep.append(tl)
    return _KVSet(_ptr(s.cache), s.fmt, s.row_stride, s.page_stride, s.num_pages, _ptr(s.block_table),
                  s.block_table.shape[1], _ptr(s.seq_lens), _ptr(s.indices), s.indices.shape[1], s.topk,
                  _ptr(tl))


def attention(w, tokens=None, nthreads: int = 0):
    """Run the oracle on workload ``w`` (see sparse_top_mla_gb300.synth.Workload).

    Returns (O [n, H, 512] float64, LSE [n, H] float64) for the requested tokens
    (all T tokens when ``tokens`` is None)."""
    lib = _load()
    keep = []
    q = w.q
    assert q.dtype == np.uint16 and q.strides[2] == 2
    main = _kvset(w.main, keep)
    extra = None
    if w.extra is not None:
        extra = _kvset(w.extra, keep)
        keep.append(extra)
    sink = None if w.sink is None else np.ascontiguousarray(w.sink, dtype=np.float32)
    token_seq = np.ascontiguousarray(w.token_seq, dtype=np.int32)
    prob = _Problem(w.T, w.H, w.main.seq_lens.shape[0], q.ctypes.data, q.strides[0] // 2, q.strides[1] // 2,
                    _ptr(token_seq), main, ctypes.addressof(extra) if extra is not None else None,
                    _ptr(sink), np.float32(w.sm_scale))
    if tokens is None:
        tok = None
        n = w.T
    else:
        tok = np.ascontiguousarray(tokens, dtype=np.int32)
        assert tok.size == 0 or (tok.min() >= 0 and tok.max() < w.T)
        n = tok.shape[0]
    O = np.zeros((n, w.H, 512), dtype=np.float64)
    lse = np.zeros((n, w.H), dtype=np.float64)
    rc = lib.oracle_attention(ctypes.byref(prob), _ptr(tok), n, O.ctypes.data, lse.ctypes.data, nthreads)
    if rc != 0:
        raise ValueError("oracle rejected the problem")
    return O, lse


def pack_rows(x, fmt: int):
    """Cache writer: rows of 576 values (float32 array, or uint16 bf16 bits) -> row bytes
    [n, 1152] (fmt 0, bf16) or [n, 656] (fmt 1, FP8 with per-128-channel scales)."""
    lib = _load()
    x = np.ascontiguousarray(x)
    assert x.ndim == 2 and x.shape[1] == 576 and x.dtype in (np.float32, np.uint16)
    dtype = 1 if x.dtype == np.float32 else 0
    rb = 1152 if fmt == 0 else 656
    out = np.zeros((x.shape[0], rb), dtype=np.uint8)
    if lib.oracle_pack_rows(_ptr(x), dtype, 576, x.shape[0], fmt, _ptr(out)) != 0:
        raise ValueError("oracle rejected the rows")
    return out


def e4m3_value(code: int) -> float:
    return _load().oracle_e4m3_value(code)


def bf16_value(bits: int) -> float:
    return _load().oracle_bf16_value(bits)


def threads(requested: int = 0) -> int:
    return _load().oracle_threads(requested)
