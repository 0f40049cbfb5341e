"""Seeded synthetic workloads for sparse top-k MLA attention (DSv4 family).

This module draws inputs only. It holds none of the attention arithmetic: it
produces the query tensor, the paged latent caches in their byte formats, the
block tables, the top-k index lists, the optional per-token widths and the
per-head sink logits, with the shapes and value distributions of the workloads
described on the pages ("[SM12x] Drop the 64-head TP pad on the DSv4 MLA
prefill path", Problem and Measurements sections: 64 or 32 local heads sharing
one latent KV; "fix(sparse-mla-sm120): add topk=256 prefill-dsv4 dispatch",
Description: 64-token pages, top-k widths that are multiples of the 64-row
index tile, -1 for a masked slot). Both the CPU oracle and the CUDA library
consume the exact bytes produced here.

Cache row formats (one row per cached token, d_qk = 576 = 512 latent + 64 rope):
  * bf16  : 576 x bf16 = 1152 bytes.
  * fp8   : 656 bytes = [512 x e4m3 latent][4 x fp32 scale, one per 128 latent
            channels][64 x bf16 rope]. The pages name FP8 caches with per-token
            scales but print no byte layout; this layout is our own reading.
Rows may be padded (row_stride > row bytes); padding bytes are 0xFF, which
decodes to NaN in both formats, so a kernel that reads padding is caught.
"""
from __future__ import annotations

import math
import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field, replace
from typing import Optional

import numpy as np

D_QK = 576
D_V = 512
D_ROPE = 64
PAGE = 64
ROW_BYTES_BF16 = D_QK * 2
ROW_BYTES_FP8 = D_V + 16 + D_ROPE * 2
FMT_BF16 = 0
FMT_FP8 = 1
E4M3_MAX = 448.0


# ----------------------------------------------------------------------------
# number formats (encoders only; decoding is the consumers' business)
# ----------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (round to nearest even); return the uint16 bits."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return (rounded >> np.uint32(16)).astype(np.uint16)


def e4m3_encode(v: np.ndarray) -> np.ndarray:
    """Encode float32 values to OCP FP8 E4M3FN codes: saturate to +-448, round to nearest even.

    E4M3FN: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, no infinities,
    NaN = S.1111.111, largest finite 448 = 1.75 * 2^8, subnormal quantum 2^-9.
    Works on the float32 bit pattern: normal results keep the top 3 mantissa bits
    after round-to-nearest-even and rebias the exponent (127 -> 7); results below
    2^-6 are multiples of 2^-9 and are rounded with np.rint (half to even).
    """
    f = np.ascontiguousarray(v, dtype=np.float32)
    u = f.view(np.uint32)
    sign = (u >> np.uint32(31)).astype(np.uint8) << np.uint8(7)
    a = np.minimum(u & np.uint32(0x7FFFFFFF), np.uint32(0x43E00000))  # |v| clamped to 448
    r = (a + np.uint32(0x7FFFF) + ((a >> np.uint32(20)) & np.uint32(1))) >> np.uint32(20)
    normal_code = (r.astype(np.int32) - (120 << 3)).astype(np.int32)
    small = a < np.uint32(0x3C800000)  # |v| < 2^-6
    sub_code = np.rint(a.view(np.float32) * np.float32(512.0)).astype(np.int32)
    code = np.where(small, sub_code, normal_code).astype(np.uint8)
    return code | sign


def encode_rows(x: np.ndarray, fmt: int) -> np.ndarray:
    """Encode float32 latent rows [n, 576] into cache row bytes [n, row_bytes]."""
    n = x.shape[0]
    if fmt == FMT_BF16:
        return f32_to_bf16_bits(x).view(np.uint8).reshape(n, ROW_BYTES_BF16)
    out = np.empty((n, ROW_BYTES_FP8), dtype=np.uint8)
    lat = x[:, :D_V].reshape(n, 4, 128)
    amax = np.max(np.abs(lat), axis=2)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    scaled = (lat / scale[:, :, None]).astype(np.float32)
    out[:, :D_V] = e4m3_encode(scaled).reshape(n, D_V)
    out[:, D_V:D_V + 16] = scale.view(np.uint8).reshape(n, 16)
    out[:, D_V + 16:] = f32_to_bf16_bits(np.ascontiguousarray(x[:, D_V:])).view(np.uint8).reshape(n, 128)
    return out


# ----------------------------------------------------------------------------
# workload containers
# ----------------------------------------------------------------------------
@dataclass
class KVSet:
    """One paged cache plus the index set that reads it (main or extra)."""
    cache: np.ndarray          # uint8, flat, num_pages * page_stride bytes
    fmt: int                   # FMT_BF16 or FMT_FP8
    row_stride: int            # bytes between consecutive rows of a page
    page_stride: int           # bytes between consecutive physical pages
    num_pages: int
    block_table: np.ndarray    # int32 [num_seqs, bt_stride]: logical page -> physical page
    seq_lens: np.ndarray       # int32 [num_seqs]
    indices: np.ndarray        # int32 [T, idx_stride]; first topk columns are used
    topk: int
    topk_length: Optional[np.ndarray] = None  # int32 [T] or None

    @property
    def row_bytes(self) -> int:
        return ROW_BYTES_BF16 if self.fmt == FMT_BF16 else ROW_BYTES_FP8


@dataclass
class Workload:
    name: str
    T: int
    H: int
    q: np.ndarray              # uint16 bf16 bits [T, H, 576] (rows may be strided)
    token_seq: np.ndarray      # int32 [T]: sequence of each query token
    main: KVSet
    extra: Optional[KVSet]
    sink: Optional[np.ndarray]  # float32 [H] or None
    sm_scale: float
    meta: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.main.seq_lens.shape[0])

    def valid_rows(self) -> int:
        """Number of (token, slot) pairs that reference a real cache row."""
        return count_valid(self)

    def gathered_bytes(self) -> int:
        n = count_valid_set(self, self.main) * self.main.row_bytes
        if self.extra is not None:
            n += count_valid_set(self, self.extra) * self.extra.row_bytes
        return n

    def algorithmic_bytes(self) -> int:
        """Valid gathered rows + indices + q + O + LSE (bytes moved by an ideal kernel)."""
        kset = self.main.topk + (self.extra.topk if self.extra is not None else 0)
        return (self.gathered_bytes() + self.T * kset * 4 + self.T * self.H * D_QK * 2
                + self.T * self.H * D_V * 2 + self.T * self.H * 4)

    def flops(self) -> int:
        """2 * T * H * (topk + topk_extra) * (576 + 512), masked slots included."""
        kset = self.main.topk + (self.extra.topk if self.extra is not None else 0)
        return 2 * self.T * self.H * kset * (D_QK + D_V)


def count_valid_set(w: Workload, s: KVSet) -> int:
    idx = s.indices[:, :s.topk]
    seq = w.token_seq.astype(np.int64)
    ok_seq = (seq >= 0) & (seq < s.seq_lens.shape[0])
    seqc = np.clip(seq, 0, s.seq_lens.shape[0] - 1)
    lens = s.seq_lens[seqc][:, None]
    valid = (idx >= 0) & (idx < lens) & ok_seq[:, None]
    if s.topk_length is not None:
        valid &= np.arange(s.topk)[None, :] < s.topk_length[:, None]
    ip = np.where(valid, idx, 0) // PAGE
    page = s.block_table[seqc[:, None], np.minimum(ip, s.block_table.shape[1] - 1)]
    valid &= ip < s.block_table.shape[1]
    valid &= (page >= 0) & (page < s.num_pages)
    return int(valid.sum())


def count_valid(w: Workload) -> int:
    n = count_valid_set(w, w.main)
    if w.extra is not None:
        n += count_valid_set(w, w.extra)
    return n


# ----------------------------------------------------------------------------
# generators
# ----------------------------------------------------------------------------
def normal_f32(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(size=shape, dtype=np.float32)


def _chunk_rng(base: int, tag: int, chunk: int) -> np.random.Generator:
    """Independent PCG64 stream for one chunk: the values depend only on (base, tag, chunk),
    never on how many threads fill the chunks."""
    return np.random.default_rng(np.random.SeedSequence(entropy=base, spawn_key=(tag, chunk)))


def _parallel(fn, n_chunks: int) -> None:
    workers = max(1, min(n_chunks, os.cpu_count() or 1))
    if workers == 1:
        for c in range(n_chunks):
            fn(c)
        return
    with ThreadPoolExecutor(max_workers=workers) as ex:
        list(ex.map(fn, range(n_chunks)))


def make_cache(rng: np.random.Generator, num_pages: int, fmt: int, row_pad: int = 0,
               page_pad: int = 0, chunk_rows: int = 4096) -> tuple[np.ndarray, int, int]:
    """Draw num_pages*64 latent rows ~N(0,1) and encode them; return (bytes, row_stride, page_stride)."""
    row_bytes = ROW_BYTES_BF16 if fmt == FMT_BF16 else ROW_BYTES_FP8
    row_stride = row_bytes + row_pad
    page_stride = PAGE * row_stride + page_pad
    buf = np.full(num_pages * page_stride, 0xFF, dtype=np.uint8)
    # [page, row, byte] view (a view even when pages are padded)
    rows3 = buf.reshape(num_pages, page_stride)[:, :PAGE * row_stride].reshape(num_pages, PAGE, row_stride)
    assert np.shares_memory(rows3, buf)
    chunk_pages = max(1, chunk_rows // PAGE)
    base = int(rng.integers(0, 2 ** 63))

    def fill(c):
        p0 = c * chunk_pages
        p1 = min(num_pages, p0 + chunk_pages)
        x = normal_f32(_chunk_rng(base, 1, c), ((p1 - p0) * PAGE, D_QK))
        rows3[p0:p1, :, :row_bytes] = encode_rows(x, fmt).reshape(p1 - p0, PAGE, row_bytes)

    _parallel(fill, (num_pages + chunk_pages - 1) // chunk_pages)
    return buf, row_stride, page_stride


def make_q(rng: np.random.Generator, T: int, H: int, chunk_tokens: int = 64) -> np.ndarray:
    q = np.empty((T, H, D_QK), dtype=np.uint16)
    base = int(rng.integers(0, 2 ** 63))

    def fill(c):
        t0 = c * chunk_tokens
        t1 = min(T, t0 + chunk_tokens)
        q[t0:t1] = f32_to_bf16_bits(normal_f32(_chunk_rng(base, 2, c), (t1 - t0, H, D_QK)))

    _parallel(fill, (T + chunk_tokens - 1) // chunk_tokens)
    return q


def shuffled_block_table(rng: np.random.Generator, num_seqs: int, pages_per_seq: int) -> np.ndarray:
    perm = rng.permutation(num_seqs * pages_per_seq).astype(np.int32)
    return perm.reshape(num_seqs, pages_per_seq)


def distinct_indices(rng: np.random.Generator, hi: np.ndarray, topk: int) -> np.ndarray:
    """Row t holds min(topk, hi[t]+1) distinct positions drawn uniformly from [0, hi[t]],
    in random order, padded with -1 on the right when fewer positions exist."""
    hi = np.asarray(hi, dtype=np.int64)
    T = hi.shape[0]
    out = np.full((T, topk), -1, dtype=np.int32)
    small = (hi + 1) <= 4 * topk
    # small populations: a random permutation of the whole range, truncated
    for t in np.nonzero(small)[0]:
        n = int(hi[t]) + 1
        p = rng.permutation(n)[:topk]
        out[t, :p.shape[0]] = p
    big = np.nonzero(~small)[0]
    if big.size:
        draw = topk + max(16, topk // 4)
        pending = big
        while pending.size:
            r = rng.integers(0, hi[pending][:, None] + 1, size=(pending.size, draw), dtype=np.int64)
            r.sort(axis=1)
            dup = np.zeros_like(r, dtype=bool)
            dup[:, 1:] = r[:, 1:] == r[:, :-1]
            enough = (~dup).sum(axis=1) >= topk
            ok_rows = pending[enough]
            if ok_rows.size:
                rr = r[enough]
                dd = dup[enough]
                order = np.argsort(dd, axis=1, kind="stable")
                uniq = np.take_along_axis(rr, order, axis=1)[:, :topk]
                shuf = np.argsort(rng.random(uniq.shape), axis=1)
                out[ok_rows] = np.take_along_axis(uniq, shuf, axis=1).astype(np.int32)
            pending = pending[~enough]
    return out


def mask_random(rng: np.random.Generator, idx: np.ndarray, p: float) -> np.ndarray:
    out = idx.copy()
    out[rng.random(idx.shape) < p] = -1
    return out


def _kvset(cache, fmt, row_stride, page_stride, num_pages, bt, seq_lens, idx, topk, topk_length=None):
    return KVSet(cache=cache, fmt=fmt, row_stride=row_stride, page_stride=page_stride,
                 num_pages=num_pages, block_table=np.ascontiguousarray(bt, dtype=np.int32),
                 seq_lens=np.ascontiguousarray(seq_lens, dtype=np.int32),
                 indices=np.ascontiguousarray(idx, dtype=np.int32), topk=topk,
                 topk_length=topk_length)


# ----------------------------------------------------------------------------
# the five workloads
# ----------------------------------------------------------------------------
CONFIG_NAMES = {
    1: "tiny bf16: 1 seq x 256 ctx, T=4, H=16, topk=128",
    2: "decode fp8: 64 seqs x 16384 ctx, T=64, H=64, topk=2048 (5% -1), sink",
    3: "prefill bf16: 1 seq x 32768 ctx, T=4096, H=32, topk=512 causal, sink",
    4: "large prefill fp8 + bf16 extra: 1 seq x 65536 ctx, T=8192, H=128, topk=2048 causal + 128 window, sink",
    5: "envelope sweep point over a 16384-token fp8 context",
}


def config(n: int, T: Optional[int] = None, seed: Optional[int] = None) -> Workload:
    """Build workload n (1..4). T may be reduced (a prefix of the query tokens) for tests."""
    rng = np.random.default_rng(1000 + n if seed is None else seed)
    if n == 1:
        ctx, H, topk, Tf = 256, 16, 128, 4
        T = Tf if T is None else T
        cache, rs, ps = make_cache(rng, ctx // PAGE, FMT_BF16)
        bt = np.arange(ctx // PAGE, dtype=np.int32)[None, :]
        q = make_q(rng, T, H)
        idx = distinct_indices(rng, np.full(T, ctx - 1), topk)
        main = _kvset(cache, FMT_BF16, rs, ps, ctx // PAGE, bt, [ctx], idx, topk)
        return Workload(CONFIG_NAMES[1], T, H, q, np.zeros(T, np.int32), main, None, None,
                        1.0 / math.sqrt(D_QK), meta={"config": 1, "ctx": ctx})
    if n == 2:
        S, ctx, H, topk = 64, 16384, 64, 2048
        T = S if T is None else T
        pps = ctx // PAGE
        cache, rs, ps = make_cache(rng, S * pps, FMT_FP8)
        bt = shuffled_block_table(rng, S, pps)
        q = make_q(rng, T, H)
        idx = mask_random(rng, distinct_indices(rng, np.full(T, ctx - 1), topk), 0.05)
        sink = normal_f32(rng, (H,))
        main = _kvset(cache, FMT_FP8, rs, ps, S * pps, bt, np.full(S, ctx), idx, topk)
        return Workload(CONFIG_NAMES[2], T, H, q, (np.arange(T) % S).astype(np.int32), main, None, sink,
                        1.0 / math.sqrt(D_QK), meta={"config": 2, "ctx": ctx})
    if n == 3:
        ctx, H, topk, Tf = 32768, 32, 512, 4096
        T = Tf if T is None else T
        cache, rs, ps = make_cache(rng, ctx // PAGE, FMT_BF16)
        bt = shuffled_block_table(rng, 1, ctx // PAGE)
        q = make_q(rng, T, H)
        pos = ctx - Tf + np.arange(T)
        idx = distinct_indices(rng, pos, topk)
        sink = normal_f32(rng, (H,))
        main = _kvset(cache, FMT_BF16, rs, ps, ctx // PAGE, bt, [ctx], idx, topk)
        return Workload(CONFIG_NAMES[3], T, H, q, np.zeros(T, np.int32), main, None, sink,
                        1.0 / math.sqrt(D_QK), meta={"config": 3, "ctx": ctx})
    if n == 4:
        ctx, H, topk, topk_x, Tf = 65536, 128, 2048, 128, 8192
        T = Tf if T is None else T
        pages = ctx // PAGE
        cache, rs, ps = make_cache(rng, pages, FMT_FP8)
        bt = shuffled_block_table(rng, 1, pages)
        xcache, xrs, xps = make_cache(rng, pages, FMT_BF16)
        xbt = shuffled_block_table(rng, 1, pages)
        q = make_q(rng, T, H)
        pos = ctx - Tf + np.arange(T)
        idx = distinct_indices(rng, pos, topk)
        win = pos[:, None] - np.arange(topk_x)[None, ::-1]  # [p-127, p]
        xidx = np.where(win >= 0, win, -1).astype(np.int32)
        sink = normal_f32(rng, (H,))
        main = _kvset(cache, FMT_FP8, rs, ps, pages, bt, [ctx], idx, topk)
        extra = _kvset(xcache, FMT_BF16, xrs, xps, pages, xbt, [ctx], xidx, topk_x)
        return Workload(CONFIG_NAMES[4], T, H, q, np.zeros(T, np.int32), main, extra, sink,
                        1.0 / math.sqrt(D_QK), meta={"config": 4, "ctx": ctx})
    raise ValueError(f"unknown config {n}")


class SweepPool:
    """Config 5: one 16384-token paged context (64 sequences; FP8 by default, bf16 with
    fmt=FMT_BF16) shared by every sweep point.

    Each point draws its own queries and index sets (random distinct positions over
    the context, 5% set to -1). `rotations` independent index sets per point let a
    timing loop touch different rows on successive calls so that each call reads
    its rows from HBM rather than L2.
    """

    def __init__(self, ctx: int = 16384, num_seqs: int = 64, seed: int = 1005, fmt: int = FMT_FP8):
        self.ctx = ctx
        self.num_seqs = num_seqs
        self.fmt = fmt
        rng = np.random.default_rng(seed)
        pps = ctx // PAGE
        self.cache, self.row_stride, self.page_stride = make_cache(rng, num_seqs * pps, fmt)
        self.num_pages = num_seqs * pps
        self.block_table = shuffled_block_table(rng, num_seqs, pps)
        self.seq_lens = np.full(num_seqs, ctx, dtype=np.int32)

    def point(self, H: int, topk: int, T: int, sink: bool, rotation: int = 0) -> Workload:
        seed = (1005 * 1_000_003 + H * 10007 + topk * 101 + T * 7 + int(sink)) * 31 + rotation
        rng = np.random.default_rng(seed & 0x7FFFFFFFFFFFFFFF)
        q = make_q(rng, T, H)
        idx = mask_random(rng, distinct_indices(rng, np.full(T, self.ctx - 1), topk), 0.05)
        snk = normal_f32(rng, (H,)) if sink else None
        token_seq = (np.arange(T) % self.num_seqs).astype(np.int32)
        main = _kvset(self.cache, self.fmt, self.row_stride, self.page_stride, self.num_pages,
                      self.block_table, self.seq_lens, idx, topk)
        return Workload(f"sweep H={H} topk={topk} T={T} sink={int(sink)}", T, H, q, token_seq, main,
                        None, snk, 1.0 / math.sqrt(D_QK),
                        meta={"config": 5, "ctx": self.ctx, "rotation": rotation})


SWEEP_H = (1, 8, 16, 32, 64, 128)
SWEEP_TOPK = (64, 128, 256, 512, 1024, 2048)
SWEEP_T = (1, 16, 64, 65, 256, 1024)


def small_case(seed: int, T: int, H: int, topk: int, ctx: int, fmt: int = FMT_BF16,
               num_seqs: int = 1, sink: bool = False, mask_p: float = 0.0, causal: bool = False,
               extra_topk: int = 0, extra_fmt: int = FMT_BF16, row_pad: int = 0, page_pad: int = 0,
               idx_pad: int = 0, shuffle_pages: bool = True, spare_pages: int = 0,
               topk_length: bool = False, sm_scale: Optional[float] = None) -> Workload:
    """A small seeded workload for parity tests (any H, topk, T, formats, strides)."""
    rng = np.random.default_rng(seed)
    pps = (ctx + PAGE - 1) // PAGE
    num_pages = num_seqs * pps + spare_pages
    cache, rs, ps = make_cache(rng, num_pages, fmt, row_pad, page_pad)
    if shuffle_pages:
        bt = rng.permutation(num_pages)[:num_seqs * pps].astype(np.int32).reshape(num_seqs, pps)
    else:
        bt = np.arange(num_seqs * pps, dtype=np.int32).reshape(num_seqs, pps)
    q = make_q(rng, T, H)
    token_seq = (np.arange(T) % num_seqs).astype(np.int32)
    if causal:
        hi = np.minimum(ctx - 1, np.arange(T) + max(0, ctx - T))
    else:
        hi = np.full(T, ctx - 1)
    idx = distinct_indices(rng, hi, topk)
    if mask_p > 0:
        idx = mask_random(rng, idx, mask_p)
    if idx_pad:
        wide = np.full((T, topk + idx_pad), -5, dtype=np.int32)
        wide[:, :topk] = idx
        idx = wide
    tl = None
    if topk_length:
        tl = rng.integers(0, topk + 1, size=T).astype(np.int32)
    main = _kvset(cache, fmt, rs, ps, num_pages, bt, np.full(num_seqs, ctx), idx, topk, tl)
    extra = None
    if extra_topk:
        xcache, xrs, xps = make_cache(rng, num_pages, extra_fmt)
        xbt = rng.permutation(num_pages)[:num_seqs * pps].astype(np.int32).reshape(num_seqs, pps)
        xidx = distinct_indices(rng, hi, extra_topk)
        if mask_p > 0:
            xidx = mask_random(rng, xidx, mask_p)
        extra = _kvset(xcache, extra_fmt, xrs, xps, num_pages, xbt, np.full(num_seqs, ctx), xidx, extra_topk)
    snk = normal_f32(rng, (H,)) if sink else None
    scale = 1.0 / math.sqrt(D_QK) if sm_scale is None else sm_scale
    return Workload(f"small seed={seed} T={T} H={H} topk={topk}", T, H, q, token_seq, main, extra, snk,
                    scale, meta={"ctx": ctx})


def with_indices(w: Workload, idx: np.ndarray, which: str = "main") -> Workload:
    """Return a copy of w whose main (or extra) index set is replaced."""
    s = getattr(w, which)
    s2 = replace(s, indices=np.ascontiguousarray(idx, dtype=np.int32), topk=idx.shape[1])
    return replace(w, **{which: s2})
