// Sparse top-k MLA attention kernels for GB300 (sm_103a).
//
// Persistent, warp-specialised kernel. Each CTA (one per SM) walks a stream of tiles; a tile
// is 128 gathered cache rows of one work item (query token t, head group g). Roles:
//   warps 0-3   softmax + epilogue (thread i owns gathered row i = TMEM lane i); lane 0 of
//               warp 3 also issues every tcgen05 MMA and commit, at fixed points of the
//               softmax program (a separate issue warp would push the block past the
//               register budget of 640 threads x 96 registers)
//   warps 4-19  loaders: resolve indices -> cache rows, keep the next tile's raw rows in
//               registers, and store each 128-channel block pair into shared memory as
//               soon as the previous tile's PV has released it (FP8 rows are dequantised
//               to bf16 on the way: e4m3 * per-128-channel scale)
// Per tile the tensor core computes
//   S^T[128 x NH]  = K_tile[128 x 576] . Q^T          (M = gathered rows, N = heads)
//   O^T[512 x NH] += V^T[512 x 128] . P^T[128 x NH]  (M = value channels, 4 blocks)
//   L[128 x NH]   += 1[128 x 128] . P^T[128 x NH]    (row sums of P, every lane equal)
// with S^T, L and O^T in TMEM. V is the first 512 channels of the same gathered tile (the
// tile is read K-major for QK^T and MN-major for PV). The issuing thread interleaves PV of
// tile j with QK^T of tile j+1 block by block, so the loaders refill the blocks PV has
// finished with while the tensor core keeps working.
//
// Schedules: whole items per CTA (prefill; the epilogue writes O and LSE), or contiguous
// flat tile ranges per CTA (split-K decode; every item segment writes a normalised partial
// O in bf16 and a base-2 partial LSE, merged by combine_kernel with warp shuffles).
//
// Heads ride in the MMA N dimension (16, 32 or 64 per group), so every head count runs
// without padding memory traffic or outputs; unused N columns are zero Q rows.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "smla_internal.h"
#include "smla_ptx.cuh"

namespace smla {

__device__ int g_device_error;

namespace {

using namespace ptx;

constexpr int kSmWarps = 4;
constexpr int kLdWarps = 16;
constexpr int kLdThreads = kLdWarps * 32;
constexpr int kThreads = (kSmWarps + kLdWarps) * 32;  // 640
constexpr int kIssueWarp = kSmWarps - 1;               // its lane 0 issues the MMAs
constexpr int kKBlocks = 9;                            // 576 channels / 64 per 128-byte row
constexpr int kBlockBytes = kTile * 128;               // one 64-channel block of the tile: 16 KB
constexpr int kTileBytes = kKBlocks * kBlockBytes;
constexpr float kLazyRescaleLog2 = 8.0f;               // raise the running max only past 2^8
constexpr long long kSpinCycles = 4000000000LL;        // bounded waits (~2 s)
constexpr uint32_t kSleepHintNs = 20000;
constexpr int kErrTimeout = 1;

template <int NH>
struct Smem {
  static constexpr int kQOff = kTileBytes;
  static constexpr int kRedOff = kQOff + kKBlocks * NH * 128;  // float [4][64]
  static constexpr int kMOff = kRedOff + 4 * 64 * 4;            // float [64] running max (base 2)
  static constexpr int kAlphaOff = kMOff + 64 * 4;              // float [64]
  static constexpr int kFinOff = kAlphaOff + 64 * 4;            // float [64] output factor per head
  static constexpr int kRowOff = kFinOff + 64 * 4;              // int64 [4][128] row byte offsets (-1 = masked)
  static constexpr int kBarOff = kRowOff + 4 * 128 * 8;         // mbarriers
  static constexpr int kNumBars = 20;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;       // tmem base, flags, votes
  static constexpr int kOnesOff = kMiscOff + 128;               // 128 B of bf16 1.0 (row-sum operand)
  static constexpr int kBytes = kOnesOff + 128;
  static constexpr int kAlloc = kBytes + 1024;                  // + alignment slack
};
static_assert(Smem<64>::kAlloc <= 232448, "shared memory budget");

// barrier indices
constexpr int kBarFull = 0;     // [9] tile block kb stored (16 loader warps arrive)
constexpr int kBarSFull = 9;    // S^T of the tile is in TMEM (tcgen05.commit)
constexpr int kBarPReady = 10;  // P^T in smem, O/L rescaled (4 softmax warps arrive)
constexpr int kBarPvDone = 11;  // [4] PV block pair done (tcgen05.commit)
constexpr int kBarRow = 15;     // [4] row offsets of tile j in slot j&3 (16 loader warps arrive)
constexpr int kBarSm = 19;      // barrier among the 128 softmax threads (every thread arrives)

template <int NH>
struct TmemCols {
  static constexpr int kS = 0;
  static constexpr int kL = 64;   // row sums of P per head, accumulated by the tensor core (all lanes equal)
  static constexpr int kO = 128;  // O^T block b at kO + b*NH
  static constexpr int kAlloc = (kO + 4 * NH) <= 256 ? 256 : 512;
};

struct Shared {
  uint8_t* base;
  uint32_t tile, q;
  float *red, *m_run, *alpha, *fin;
  int64_t* rowoff;
  uint32_t bars;
  uint32_t* tmem_slot;
  volatile int* abort_flag;
  volatile int* rescale_flag;
  volatile int* vote;  // [2] per-tile "a max must move" flags
  uint32_t ones;       // 128 B of bf16 1.0
  __device__ uint32_t bar(int i) const { return bars + 8u * i; }
};

// Bounded wait on an mbarrier phase. The thread sleeps in hardware between checks; only after
// a sleep ends without the phase does it look at the abort flag and the clock.
__device__ __forceinline__ bool wait_bar(const Shared& sh, uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
    if (*sh.abort_flag) return false;
    if (clock64() - t0 > kSpinCycles) {
      atomicExch(&g_device_error, kErrTimeout);
      *sh.abort_flag = 1;
      return false;
    }
  }
}

// Warp-uniform wait: the warp proceeds only if all lanes saw the phase (a lane that gave up
// makes the whole warp give up, so no lane runs a warp-collective instruction alone). Every
// lane waits on the mbarrier itself: one lane waiting and the others following through
// __syncwarp gave stale reads.
__device__ __forceinline__ bool wait_bar_w(const Shared& sh, uint32_t bar, uint32_t parity) {
  const bool ok = wait_bar(sh, bar, parity);
  return __all_sync(0xffffffffu, ok);
}

// Barrier among the 128 softmax threads, built on an mbarrier so the wait is bounded.
__device__ __forceinline__ bool sm_sync(const Shared& sh, uint32_t& phase) {
  mbar_arrive(sh.bar(kBarSm));
  const bool ok = wait_bar_w(sh, sh.bar(kBarSm), phase & 1);
  ++phase;
  return ok;
}

// ------------------------------------------------------------------ tile stream
struct TileRef {
  long long item;
  int tile;
  bool first, last;
};

__device__ __forceinline__ TileRef tile_ref(const AttnArgs& a, long long lo, int n, int j) {
  TileRef r;
  if (a.split) {
    const long long x = lo + j;
    r.item = x / a.tiles_per_item;
    r.tile = static_cast<int>(x - r.item * a.tiles_per_item);
  } else {
    const int k = j / a.tiles_per_item;
    r.item = blockIdx.x + static_cast<long long>(k) * a.nctas;
    r.tile = j - k * a.tiles_per_item;
  }
  r.first = r.tile == 0 || j == 0;
  r.last = r.tile == a.tiles_per_item - 1 || j == n - 1;
  return r;
}

__device__ __forceinline__ int set_of(const AttnArgs& a, int tile) {
  return (a.nsets > 1 && tile >= a.set[0].ntiles) ? 1 : 0;
}

// Fields of set 0 or 1, selected field by field (a runtime index into the kernel-parameter
// array would force a local-memory copy of the parameters).
#define SET_FIELD(a, sid, f) ((sid) ? (a).set[1].f : (a).set[0].f)

// Index resolution (entry -> cache row byte offset, -1 when masked), split into three phases
// whose loads only depend on the previous phase, so the loaders can issue each phase right
// after a tile store and consume it a tile later.
struct Resolve {
  int seq, seqlen, idx[2], page[2];
};

__device__ __forceinline__ void resolve_a(const AttnArgs& a, long long item, int tile, int rg, Resolve& R) {
  const int t = static_cast<int>(item / a.groups);
  const int sid = set_of(a, tile);
  const int base = (tile - (sid ? a.set[0].ntiles : 0)) * kTile + rg;
  int width = SET_FIELD(a, sid, topk);
  const int32_t* tl = SET_FIELD(a, sid, topk_length);
  if (tl != nullptr) width = min(width, max(0, __ldg(tl + t)));
  R.seq = __ldg(a.token_seq + t);
  const int32_t* ip = SET_FIELD(a, sid, indices) + static_cast<int64_t>(t) * SET_FIELD(a, sid, idx_stride);
#pragma unroll
  for (int k = 0; k < 2; ++k) R.idx[k] = (base + 64 * k < width) ? __ldg(ip + base + 64 * k) : -1;
}

__device__ __forceinline__ void resolve_b(const AttnArgs& a, int tile, Resolve& R) {
  const int sid = set_of(a, tile);
  const bool seq_ok = R.seq >= 0 && R.seq < a.num_seqs;
  const int32_t bts = SET_FIELD(a, sid, bt_stride);
  R.seqlen = seq_ok ? __ldg(SET_FIELD(a, sid, seq_lens) + R.seq) : 0;
  const int32_t* bt = SET_FIELD(a, sid, block_table) + static_cast<int64_t>(seq_ok ? R.seq : 0) * bts;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i = R.idx[k];
    R.page[k] = (seq_ok && i >= 0 && (i >> 6) < bts) ? __ldg(bt + (i >> 6)) : -1;
  }
}

__device__ __forceinline__ void resolve_c(const AttnArgs& a, int tile, const Resolve& R, int64_t* off) {
  const int sid = set_of(a, tile);
  const int32_t np = SET_FIELD(a, sid, num_pages);
  const int64_t ps = SET_FIELD(a, sid, page_stride);
  const int64_t rs = SET_FIELD(a, sid, row_stride);
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int i = R.idx[k];
    const int p = R.page[k];
    off[k] = (i >= 0 && i < R.seqlen && p >= 0 && p < np)
                 ? static_cast<int64_t>(p) * ps + static_cast<int64_t>(i & 63) * rs
                 : -1;
  }
}

// ------------------------------------------------------------------ helpers
template <int CNT, int OFF, bool kMax>
__device__ __forceinline__ void col_reduce_step(float* v, int lane) {
  if constexpr (OFF > 0) {
    if constexpr (CNT > 1) {
      constexpr int half = CNT / 2;
      const bool upper = (lane & OFF) != 0;
#pragma unroll
      for (int k = 0; k < half; ++k) {
        const float send = upper ? v[k] : v[k + half];
        const float keep = upper ? v[k + half] : v[k];
        const float recv = __shfl_xor_sync(0xffffffffu, send, OFF);
        v[k] = kMax ? fmaxf(keep, recv) : keep + recv;
      }
      col_reduce_step<half, OFF / 2, kMax>(v, lane);
    } else {
      const float recv = __shfl_xor_sync(0xffffffffu, v[0], OFF);
      v[0] = kMax ? fmaxf(v[0], recv) : v[0] + recv;
      col_reduce_step<1, OFF / 2, kMax>(v, lane);
    }
  }
}

// Column reduction of N (16 or 32) values per lane across the warp ("transpose reduce":
// each step halves the values a lane holds and exchanges the other half with its partner,
// N-1 shuffles in total). Writes the warp's column results to red_w[0..N).
template <int N, bool kMax>
__device__ __forceinline__ void warp_col_reduce_store(float* v, int lane, float* red_w) {
  col_reduce_step<N, 16, kMax>(v, lane);
  if (N == 32) {
    red_w[lane] = v[0];
  } else if ((lane & 1) == 0) {
    red_w[lane >> 1] = v[0];
  }
}

__device__ __forceinline__ void dequant16(const uint4 raw, float scale, uint4& lo, uint4& hi) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const __nv_fp8x2_storage_t pair = static_cast<__nv_fp8x2_storage_t>((w[i] >> (16 * h)) & 0xFFFFu);
      const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
      const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * scale, f.y * scale);
      o[2 * i + h] = *reinterpret_cast<const uint32_t*>(&b);
    }
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

__device__ __forceinline__ uint32_t swz(int row, int chunk) {  // 128-byte swizzle inside a 1 KB atom
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// ------------------------------------------------------------------ loader role
// Thread u (0..511) owns rows rg and rg+64 (rg = u/8) and the 16-byte chunk lane8 = u%8
// of every 128-byte row segment, so 8 consecutive threads read 128 contiguous bytes.
//
// Register staging (4 slots of one 16-byte chunk per row): an FP8 block pair needs one slot,
// so FP8 tiles are loaded a whole tile ahead (block pair bp of tile j+1 is issued as soon as
// block pair bp of tile j is stored); a bf16 block pair needs two slots, so bf16 tiles are
// loaded half a tile ahead (block pair bp+2 after bp is stored). Index resolution runs in
// three phases one tile apart (A: index and sequence loads, B: block-table and length loads,
// C: offsets), finishing two tiles ahead of use.
struct LdData {
  uint4 d[4][2];   // [slot][row k]
  float sc[4][2];  // fp8 scale of the block pair held in slot [s][row k]
  uint4 rope[2];
};

template <int S>  // fp8 block pair -> slot S
__device__ __forceinline__ void ld_issue_fp8(const uint8_t* cache, const int64_t* off, int lane8, int bp, LdData& D) {
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    D.d[S][k] = make_uint4(0, 0, 0, 0);
    D.sc[S][k] = 0.f;
    if (off[k] >= 0) {
      const uint8_t* row = cache + off[k];
      D.d[S][k] = ldg_nc_v4(row + 128 * bp + 16 * lane8);
      D.sc[S][k] = __ldg(reinterpret_cast<const float*>(row + 512) + bp);
    }
  }
}

template <int P>  // bf16 block pair -> slots 2P, 2P+1
__device__ __forceinline__ void ld_issue_bf16(const uint8_t* cache, const int64_t* off, int lane8, int bp, LdData& D) {
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    D.d[2 * P][k] = make_uint4(0, 0, 0, 0);
    D.d[2 * P + 1][k] = make_uint4(0, 0, 0, 0);
    if (off[k] >= 0) {
      const uint8_t* row = cache + off[k];
      D.d[2 * P][k] = ldg_nc_v4(row + 256 * bp + 16 * lane8);
      D.d[2 * P + 1][k] = ldg_nc_v4(row + 256 * bp + 128 + 16 * lane8);
    }
  }
}

__device__ __forceinline__ void ld_issue_rope(int fmt, const uint8_t* cache, const int64_t* off, int lane8,
                                              LdData& D) {
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    D.rope[k] = make_uint4(0, 0, 0, 0);
    if (off[k] >= 0) D.rope[k] = ldg_nc_v4(cache + off[k] + (fmt == 0 ? 1024 : 528) + 16 * lane8);
  }
}

template <int S>
__device__ __forceinline__ void ld_store_fp8(const Shared& sh, int rg, int lane8, int bp, const LdData& D) {
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int r = rg + 64 * k;
    uint4 lo, hi;
    dequant16(D.d[S][k], D.sc[S][k], lo, hi);
    const int kb = 2 * bp + (lane8 >> 2);
    const int c0 = (lane8 & 3) * 2;
    sts_v4(sh.tile + kb * kBlockBytes + swz(r, c0), lo);
    sts_v4(sh.tile + kb * kBlockBytes + swz(r, c0 + 1), hi);
  }
}

template <int P>
__device__ __forceinline__ void ld_store_bf16(const Shared& sh, int rg, int lane8, int bp, const LdData& D) {
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int r = rg + 64 * k;
    sts_v4(sh.tile + (2 * bp) * kBlockBytes + swz(r, lane8), D.d[2 * P][k]);
    sts_v4(sh.tile + (2 * bp + 1) * kBlockBytes + swz(r, lane8), D.d[2 * P + 1][k]);
  }
}

// fp8 block pair bp (runtime) -> its slot
__device__ __forceinline__ void ld_issue_fp8_rt(const uint8_t* cache, const int64_t* off, int lane8, int bp,
                                                LdData& D) {
  switch (bp) {
    case 0: ld_issue_fp8<0>(cache, off, lane8, 0, D); break;
    case 1: ld_issue_fp8<1>(cache, off, lane8, 1, D); break;
    case 2: ld_issue_fp8<2>(cache, off, lane8, 2, D); break;
    default: ld_issue_fp8<3>(cache, off, lane8, 3, D); break;
  }
}

template <int NH>
__device__ __forceinline__ void loader_role(const AttnArgs& a, const Shared& sh, long long lo, int n) {
  const int u = threadIdx.x - kSmWarps * 32;
  const int lane = threadIdx.x & 31;
  const int lane8 = u & 7;
  const int rg = u >> 3;
  if (n <= 0) return;

  auto load_q = [&](long long item) {
    const int t = static_cast<int>(item / a.groups);
    const int h0 = static_cast<int>(item - static_cast<long long>(t) * a.groups) * a.heads_per_group;
    const int hg = min(a.heads_per_group, a.H - h0);
    const uint16_t* qb = a.q + static_cast<int64_t>(t) * a.q_stride_t;
    for (int e = u; e < NH * 72; e += kLdThreads) {
      const int nrow = e / 72;
      const int c = e - nrow * 72;
      const bool live = nrow < hg;
      const uint16_t* src =
          qb + (live ? static_cast<int64_t>(h0 + nrow) * a.q_stride_h + (c >> 3) * 64 + (c & 7) * 8 : 0);
      cp_async16(sh.q + (c >> 3) * NH * 128 + swz(nrow, c & 7), src, live ? 16u : 0u);
    }
    cp_async_commit();
  };
  auto prefetch_q = [&](long long item) {
    const int t = static_cast<int>(item / a.groups);
    const int h0 = static_cast<int>(item - static_cast<long long>(t) * a.groups) * a.heads_per_group;
    const int hg = min(a.heads_per_group, a.H - h0);
    for (int e = u; e < hg * 9; e += kLdThreads) {
      const uint16_t* p = a.q + static_cast<int64_t>(t) * a.q_stride_t +
                          static_cast<int64_t>(h0 + e / 9) * a.q_stride_h + (e % 9) * 64;
      asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
    }
  };
  auto publish = [&](int jt, const int64_t* off) {  // row validity for the softmax warps
    if (lane8 == 0) {
      sh.rowoff[(jt & 3) * 128 + rg] = off[0];
      sh.rowoff[(jt & 3) * 128 + rg + 64] = off[1];
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(sh.bar(kBarRow + (jt & 3)));
  };
  auto fmt_of = [&](int jt) { return SET_FIELD(a, set_of(a, tile_ref(a, lo, n, jt).tile), format); };
  auto cache_of = [&](int jt) { return SET_FIELD(a, set_of(a, tile_ref(a, lo, n, jt).tile), cache); };

  // resolution pipeline: tile 0 now (its loads go out at once), then tile 1, then tile 2
  // through phase A
  int64_t off_cur[2], off_nxt[2] = {-1, -1};
  Resolve RA, RB;
  LdData D;
  int fmt_cur = fmt_of(0);
  const uint8_t* cache_cur = cache_of(0);
  int fmt_nxt = n > 1 ? fmt_of(1) : 0;
  const uint8_t* cache_nxt = n > 1 ? cache_of(1) : nullptr;
  {
    TileRef r = tile_ref(a, lo, n, 0);
    resolve_a(a, r.item, r.tile, rg, RB);
    if (r.first) prefetch_q(r.item);
    resolve_b(a, r.tile, RB);
    resolve_c(a, r.tile, RB, off_cur);
    publish(0, off_cur);
    if (fmt_cur == 1) {
      ld_issue_fp8<0>(cache_cur, off_cur, lane8, 0, D);
      ld_issue_fp8<1>(cache_cur, off_cur, lane8, 1, D);
      ld_issue_fp8<2>(cache_cur, off_cur, lane8, 2, D);
      ld_issue_fp8<3>(cache_cur, off_cur, lane8, 3, D);
      ld_issue_rope(1, cache_cur, off_cur, lane8, D);
    } else {
      ld_issue_bf16<0>(cache_cur, off_cur, lane8, 0, D);
      ld_issue_bf16<1>(cache_cur, off_cur, lane8, 1, D);
    }
    if (n > 1) {
      r = tile_ref(a, lo, n, 1);
      resolve_a(a, r.item, r.tile, rg, RB);
      resolve_b(a, r.tile, RB);
      resolve_c(a, r.tile, RB, off_nxt);
      publish(1, off_nxt);
    }
    if (n > 2) {
      r = tile_ref(a, lo, n, 2);
      resolve_a(a, r.item, r.tile, rg, RA);
    }
  }

  for (int j = 0; j < n; ++j) {
    const TileRef tr = tile_ref(a, lo, n, j);
    const bool has1 = j + 1 < n;
    const bool has2 = j + 2 < n;
    if (has1 && tile_ref(a, lo, n, j + 1).first) prefetch_q(tile_ref(a, lo, n, j + 1).item);
    int64_t off2[2] = {-1, -1};
    auto step = [&](auto bpc) -> bool {
      constexpr int bp = decltype(bpc)::value;
      if (j > 0 && !wait_bar_w(sh, sh.bar(kBarPvDone + bp), (j - 1) & 1)) return false;
      if (bp == 0 && tr.first) load_q(tr.item);
      if (fmt_cur == 1) {
        ld_store_fp8<bp>(sh, rg, lane8, bp, D);
      } else {
        ld_store_bf16<(bp & 1)>(sh, rg, lane8, bp, D);
      }
      if (bp == 3) {
#pragma unroll
        for (int k = 0; k < 2; ++k) sts_v4(sh.tile + 8 * kBlockBytes + swz(rg + 64 * k, lane8), D.rope[k]);
      }
      if (bp == 0 && tr.first) cp_async_wait_all();
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(sh.bar(kBarFull + 2 * bp));
        mbar_arrive(sh.bar(kBarFull + 2 * bp + 1));
        if (bp == 3) mbar_arrive(sh.bar(kBarFull + 8));
      }
      // ---- refill the slots this store freed
      if (fmt_cur == 1) {
        if (has1) {
          if (fmt_nxt == 1) {
            ld_issue_fp8<bp>(cache_nxt, off_nxt, lane8, bp, D);
            if (bp == 3) ld_issue_rope(1, cache_nxt, off_nxt, lane8, D);
          } else if (bp == 1) {
            ld_issue_bf16<0>(cache_nxt, off_nxt, lane8, 0, D);
          } else if (bp == 3) {
            ld_issue_bf16<1>(cache_nxt, off_nxt, lane8, 1, D);
          }
        }
      } else {
        if (bp == 0) {
          ld_issue_bf16<0>(cache_cur, off_cur, lane8, 2, D);
        } else if (bp == 1) {
          ld_issue_bf16<1>(cache_cur, off_cur, lane8, 3, D);
          ld_issue_rope(0, cache_cur, off_cur, lane8, D);
        } else if (has1) {
          if (fmt_nxt == 0) {
            ld_issue_bf16<(bp & 1)>(cache_nxt, off_nxt, lane8, bp - 2, D);
          } else {
            ld_issue_fp8_rt(cache_nxt, off_nxt, lane8, 2 * (bp - 2), D);
            ld_issue_fp8_rt(cache_nxt, off_nxt, lane8, 2 * (bp - 2) + 1, D);
            if (bp == 3) ld_issue_rope(1, cache_nxt, off_nxt, lane8, D);
          }
        }
      }
      // ---- index resolution pipeline
      if (bp == 0 && has2) {
        RB = RA;  // phase A of tile j+2 was issued a tile ago
        resolve_b(a, tile_ref(a, lo, n, j + 2).tile, RB);
        if (j + 3 < n) {
          const TileRef r3 = tile_ref(a, lo, n, j + 3);
          resolve_a(a, r3.item, r3.tile, rg, RA);
        }
      }
      if (bp == 3 && has2) {
        resolve_c(a, tile_ref(a, lo, n, j + 2).tile, RB, off2);
        publish(j + 2, off2);
      }
      return true;
    };
    if (!step(std::integral_constant<int, 0>{}) || !step(std::integral_constant<int, 1>{}) ||
        !step(std::integral_constant<int, 2>{}) || !step(std::integral_constant<int, 3>{}))
      return;
    off_cur[0] = off_nxt[0];
    off_cur[1] = off_nxt[1];
    fmt_cur = fmt_nxt;
    cache_cur = cache_nxt;
    if (has2) {
      off_nxt[0] = off2[0];
      off_nxt[1] = off2[1];
      fmt_nxt = fmt_of(j + 2);
      cache_nxt = cache_of(j + 2);
    }
  }
}

// ------------------------------------------------------------------ MMA issue (one thread)
// Descriptors are built once; each MMA adds a compile-time byte offset (>> 4) to the start
// address field, so issuing costs a few instructions per MMA.
struct MmaDesc {
  uint64_t qk_a, qk_b, pv_a, pv_b, ones;
};

template <int NH>
__device__ __forceinline__ MmaDesc make_descs(const Shared& sh) {
  MmaDesc d;
  d.qk_a = smem_desc(sh.tile, 16, 1024, kSwizzle128B);
  d.qk_b = smem_desc(sh.q, 16, 1024, kSwizzle128B);
  d.pv_a = smem_desc(sh.tile, kBlockBytes, 1024, kSwizzle128B);
  d.pv_b = smem_desc(sh.tile + 8 * kBlockBytes, 128, 2048, kSwizzleNone);
  d.ones = smem_desc(sh.ones, 0, 0, kSwizzleNone);  // every row and K step reads the same ones
  return d;
}

template <int NH, int KB0, int KB1>
__device__ __forceinline__ bool mma_qk(const Shared& sh, const MmaDesc& d, uint32_t tmem, int j) {
  constexpr uint32_t idesc = idesc_bf16(128, NH, 0, 0);
#pragma unroll
  for (int kb = KB0; kb < KB1; ++kb) {
    if (!wait_bar(sh, sh.bar(kBarFull + kb), j & 1)) return false;
    tc_fence_after();
#pragma unroll
    for (int ks = 0; ks < 4; ++ks) {
      mma_bf16_ss(tmem + TmemCols<NH>::kS, d.qk_a + static_cast<uint64_t>((kb * kBlockBytes + ks * 32) >> 4),
                  d.qk_b + static_cast<uint64_t>((kb * NH * 128 + ks * 32) >> 4), idesc, (kb | ks) != 0);
    }
  }
  return true;
}

template <int NH, int BP>
__device__ __forceinline__ void mma_pv(const Shared& sh, const MmaDesc& d, uint32_t tmem, bool first) {
  constexpr uint32_t idesc = idesc_bf16(128, NH, 1, 1);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    mma_bf16_ss(tmem + TmemCols<NH>::kO + BP * NH,
                d.pv_a + static_cast<uint64_t>((2 * BP * kBlockBytes + ks * 2048) >> 4),
                d.pv_b + static_cast<uint64_t>((ks * 256) >> 4), idesc, (first && ks == 0) ? 0u : 1u);
  }
  mma_commit(sh.bar(kBarPvDone + BP));
}

// Row sums of P for every head: L[m, h] += sum_k 1 * P^T[k, h] (all 128 lanes get the same
// sums). Same B operand and accumulate rule as PV, so the normalisation uses exactly the bf16
// P that multiplied V.
template <int NH>
__device__ __forceinline__ void mma_rowsum(const MmaDesc& d, uint32_t tmem, bool first) {
  constexpr uint32_t idesc = idesc_bf16(128, NH, 0, 1);
#pragma unroll
  for (int ks = 0; ks < 8; ++ks)
    mma_bf16_ss(tmem + TmemCols<NH>::kL, d.ones, d.pv_b + static_cast<uint64_t>((ks * 256) >> 4), idesc,
                (first && ks == 0) ? 0u : 1u);
}

// QK^T of the first tile of the stream.
template <int NH>
__device__ __forceinline__ bool mma_issue_first(const Shared& sh, const MmaDesc& d, uint32_t tmem) {
  if (!mma_qk<NH, 0, kKBlocks>(sh, d, tmem, 0)) return false;
  mma_commit(sh.bar(kBarSFull));
  return true;
}

// After the softmax of tile j: PV of tile j block pair by block pair, interleaved with QK^T of
// tile j+1 as its blocks arrive (the loaders refill a block pair once its PV has finished).
template <int NH>
__device__ __forceinline__ bool mma_issue_after(const AttnArgs& a, const Shared& sh, const MmaDesc& d, uint32_t tmem,
                                                long long lo, int n, int j) {
  if (!wait_bar(sh, sh.bar(kBarPReady), j & 1)) return false;
  tc_fence_after();
  const bool first = tile_ref(a, lo, n, j).first;
  mma_pv<NH, 0>(sh, d, tmem, first);
  mma_pv<NH, 1>(sh, d, tmem, first);
  if (j + 1 >= n) {
    mma_pv<NH, 2>(sh, d, tmem, first);
    mma_rowsum<NH>(d, tmem, first);
    mma_pv<NH, 3>(sh, d, tmem, first);
    return true;
  }
  if (!mma_qk<NH, 0, 2>(sh, d, tmem, j + 1)) return false;
  mma_pv<NH, 2>(sh, d, tmem, first);
  if (!mma_qk<NH, 2, 4>(sh, d, tmem, j + 1)) return false;
  mma_rowsum<NH>(d, tmem, first);
  mma_pv<NH, 3>(sh, d, tmem, first);
  if (!mma_qk<NH, 4, kKBlocks>(sh, d, tmem, j + 1)) return false;
  mma_commit(sh.bar(kBarSFull));
  return true;
}

// ------------------------------------------------------------------ softmax / epilogue role
// P^T (bf16) for 16 heads from S^T chunk c0, using the running maxima; returns whether any score
// exceeds its head's maximum by more than 2^8 (then the maxima have to move).
template <int NH>
__device__ __forceinline__ bool softmax_chunk(const AttnArgs& a, const Shared& sh, uint32_t s_addr, uint32_t pt, int c0,
                                              bool valid, int tid) {
  float s[16];
  tmem_ld16(s_addr, s);
  bool over = false;
  uint32_t w[8];
  const float4* m4 = reinterpret_cast<const float4*>(sh.m_run + c0);
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const float4 m = m4[q];
    const float mv[4] = {m.x, m.y, m.z, m.w};
    float p[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float x = valid ? s[4 * q + e] * a.scale_log2 : -INFINITY;
      over |= x > mv[e] + kLazyRescaleLog2;
      p[e] = ex2(x - (mv[e] == -INFINITY ? 0.f : mv[e]));
    }
    const __nv_bfloat162 b0 = __floats2bfloat162_rn(p[0], p[1]);
    const __nv_bfloat162 b1 = __floats2bfloat162_rn(p[2], p[3]);
    w[2 * q] = *reinterpret_cast<const uint32_t*>(&b0);
    w[2 * q + 1] = *reinterpret_cast<const uint32_t*>(&b1);
  }
  // P^T in the no-swizzle MN-major layout: [head/8][row/8][row%8][head%8]
  const uint32_t dst = pt + (c0 >> 3) * 2048 + (tid >> 3) * 128 + (tid & 7) * 16;
  sts_v4(dst, make_uint4(w[0], w[1], w[2], w[3]));
  sts_v4(dst + 2048, make_uint4(w[4], w[5], w[6], w[7]));
  return over;
}

template <int NH>
__device__ __forceinline__ void softmax_role(const AttnArgs& a, const Shared& sh, uint32_t tmem, long long lo, int n) {
  constexpr int CW = NH < 32 ? NH : 32;  // columns per reduction pass
  using TC = TmemCols<NH>;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t lb = static_cast<uint32_t>(warp * 32) << 16;
  const uint32_t pt = sh.tile + 8 * kBlockBytes;

  const bool issuer = warp == kIssueWarp && lane == 0;
  const MmaDesc md = make_descs<NH>(sh);
  uint32_t smph = 0;
  if (warp == kIssueWarp) {
    bool ok = true;
    if (issuer && n > 0) ok = mma_issue_first<NH>(sh, md, tmem);
    __syncwarp();
    if (!__shfl_sync(0xffffffffu, ok, 0)) return;
  }

  for (int j = 0; j < n; ++j) {
    const TileRef tr = tile_ref(a, lo, n, j);
    if (!wait_bar_w(sh, sh.bar(kBarRow + (j & 3)), (j >> 2) & 1)) return;
    const bool valid = sh.rowoff[(j & 3) * 128 + tid] >= 0;
    if (!wait_bar_w(sh, sh.bar(kBarSFull), j & 1)) return;
    tc_fence_after();
    if (tr.first && tid < 64) sh.m_run[tid] = -INFINITY;
    // vote slot of the next tile: every read of it (tile j-1) happened before this tile began
    if (tid == 0) sh.vote[(j + 1) & 1] = 0;

    // ---- optimistic pass: P with the running maxima. Needs a redo only when some score
    // exceeds its head's maximum by more than 2^8 (always on the first tile of an item).
    bool need_max = tr.first;
    if (!need_max) {
      bool over = false;
#pragma unroll 1
      for (int c0 = 0; c0 < NH; c0 += 16) over |= softmax_chunk<NH>(a, sh, tmem + lb + TC::kS + c0, pt, c0, valid, tid);
      if (__any_sync(0xffffffffu, over) && lane == 0) sh.vote[j & 1] = 1;
      if (!sm_sync(sh, smph)) return;
      need_max = sh.vote[j & 1] != 0;
    }
    if (need_max) {
      // ---- per-head maximum of the tile, new running maxima and rescale factors
#pragma unroll 1
      for (int c0 = 0; c0 < NH; c0 += CW) {
        float s[CW];
#pragma unroll
        for (int c = 0; c < CW; c += 16) tmem_ld16(tmem + lb + TC::kS + c0 + c, s + c);
#pragma unroll
        for (int h = 0; h < CW; ++h) s[h] = valid ? s[h] * a.scale_log2 : -INFINITY;
        warp_col_reduce_store<CW, true>(s, lane, sh.red + warp * 64 + c0);
      }
      if (!sm_sync(sh, smph)) return;
      if (warp == 0) {
        bool raised = false;
        for (int h = lane; h < NH; h += 32) {
          const float tmax = fmaxf(fmaxf(sh.red[h], sh.red[64 + h]), fmaxf(sh.red[128 + h], sh.red[192 + h]));
          const float mo = sh.m_run[h];
          float al = 1.f;
          if (tmax > mo + kLazyRescaleLog2) {
            al = (mo == -INFINITY) ? 0.f : ex2(mo - tmax);
            sh.m_run[h] = tmax;
            raised = true;
          }
          sh.alpha[h] = al;
        }
        raised = __any_sync(0xffffffffu, raised);
        if (lane == 0) *sh.rescale_flag = raised ? 1 : 0;
      }
      if (!sm_sync(sh, smph)) return;
#pragma unroll 1
      for (int c0 = 0; c0 < NH; c0 += 16) softmax_chunk<NH>(a, sh, tmem + lb + TC::kS + c0, pt, c0, valid, tid);
      // O^T and the row sums *= alpha when a running max moved (the previous PV is complete:
      // S^T of this tile was committed after it)
      if (!tr.first && *sh.rescale_flag != 0) {
#pragma unroll 1
        for (int b = 0; b <= 4; ++b) {
          const uint32_t col = b < 4 ? TC::kO + b * NH : TC::kL;
#pragma unroll 1
          for (int c0 = 0; c0 < NH; c0 += 16) {
            float o[16];
            const uint32_t addr = tmem + lb + col + c0;
            tmem_ld16(addr, o);
#pragma unroll
            for (int i = 0; i < 16; ++i) o[i] *= sh.alpha[c0 + i];
            tmem_st16(addr, o);
          }
        }
        tmem_st_wait();
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(sh.bar(kBarPReady));
    if (warp == kIssueWarp) {
      bool ok = true;
      if (issuer) ok = mma_issue_after<NH>(a, sh, md, tmem, lo, n, j);
      __syncwarp();
      if (!__shfl_sync(0xffffffffu, ok, 0)) return;
    }

    if (!tr.last) continue;
    // ---- epilogue of the item segment: wait for its last PV (and row sums)
    if (!wait_bar_w(sh, sh.bar(kBarPvDone + 3), j & 1)) return;
    tc_fence_after();
    const long long item = tr.item;
    const int t = static_cast<int>(item / a.groups);
    const int h0 = static_cast<int>(item - static_cast<long long>(t) * a.groups) * a.heads_per_group;
    const int hg = min(a.heads_per_group, a.H - h0);
    const int slot =
        a.split ? static_cast<int>(blockIdx.x - split_owner(item * a.tiles_per_item, a.total_tiles, a.nctas)) : 0;
    // thread h (< NH) turns the row sum of head h into the output factor and the LSE
#pragma unroll 1
    for (int c0 = 0; c0 < NH; c0 += 16) {
      float l[16];
      tmem_ld16(tmem + lb + TC::kL + c0, l);
      if (tid >= c0 && tid < c0 + 16) {
        const int h = tid;
        float lh = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) lh = (i == tid - c0) ? l[i] : lh;
        const float m = sh.m_run[h];
        float factor = 0.f, lse2 = -INFINITY;
        if (lh > 0.f) {
          lse2 = m + log2f(lh);
          float denom = lh;
          if (!a.split && a.sink != nullptr && h < hg) denom += exp2f(a.sink[h0 + h] * 1.4426950408889634f - m);
          factor = 1.f / denom;
        }
        sh.fin[h] = factor;
        if (h < hg) {
          if (a.split) {
            a.part_lse[(static_cast<int64_t>(slot) * a.T + t) * a.H + h0 + h] = lse2;
          } else if (a.lse != nullptr) {
            a.lse[static_cast<int64_t>(t) * a.lse_stride_t + h0 + h] = lse2 * 0.6931471805599453f;
          }
        }
      }
    }
    if (!sm_sync(sh, smph)) return;
    // O^T: thread tid holds channel 128b + tid of every head; warps write 64-byte runs
    uint16_t* obase = a.split ? static_cast<uint16_t*>(a.part_o) +
                                    ((static_cast<int64_t>(slot) * a.T + t) * a.H + h0) * kDv
                              : a.out + static_cast<int64_t>(t) * a.out_stride_t +
                                    static_cast<int64_t>(h0) * a.out_stride_h;
    const int64_t hstride = a.split ? kDv : a.out_stride_h;
#pragma unroll 1
    for (int b = 0; b < 4; ++b) {
#pragma unroll 1
      for (int c0 = 0; c0 < NH; c0 += 16) {
        float o[16], f[16];
        tmem_ld16(tmem + lb + TC::kO + b * NH + c0, o);
#pragma unroll
        for (int i = 0; i < 16; ++i) f[i] = sh.fin[c0 + i];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int h = c0 + i;
          if (h < hg) {
            const __nv_bfloat16 v = __float2bfloat16_rn(f[i] != 0.f ? o[i] * f[i] : 0.f);
            obase[h * hstride + b * 128 + tid] = *reinterpret_cast<const uint16_t*>(&v);
          }
        }
      }
    }
    tc_fence_before();
    if (!sm_sync(sh, smph)) return;
  }
}

template <int NH>
__global__ void __maxnreg__(96) sparse_mla_kernel(const AttnArgs a) {
  using L = Smem<NH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Shared sh;
  sh.base = base;
  sh.tile = smem_u32(base);
  sh.q = smem_u32(base + L::kQOff);
  sh.red = reinterpret_cast<float*>(base + L::kRedOff);
  sh.m_run = reinterpret_cast<float*>(base + L::kMOff);
  sh.alpha = reinterpret_cast<float*>(base + L::kAlphaOff);
  sh.fin = reinterpret_cast<float*>(base + L::kFinOff);
  sh.rowoff = reinterpret_cast<int64_t*>(base + L::kRowOff);
  sh.bars = smem_u32(base + L::kBarOff);
  sh.tmem_slot = reinterpret_cast<uint32_t*>(base + L::kMiscOff);
  sh.abort_flag = reinterpret_cast<volatile int*>(base + L::kMiscOff + 4);
  sh.rescale_flag = reinterpret_cast<volatile int*>(base + L::kMiscOff + 8);
  sh.vote = reinterpret_cast<volatile int*>(base + L::kMiscOff + 16);
  sh.ones = smem_u32(base + L::kOnesOff);

  const int warp = threadIdx.x >> 5;
  long long lo = 0;
  int n = 0;
  if (a.split) {
    lo = split_lo(blockIdx.x, a.total_tiles, a.nctas);
    n = static_cast<int>(split_lo(blockIdx.x + 1, a.total_tiles, a.nctas) - lo);
  } else {
    const long long k = (a.n_items - blockIdx.x + a.nctas - 1) / a.nctas;
    n = static_cast<int>(k * a.tiles_per_item);
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < 9; ++i) mbar_init(sh.bar(kBarFull + i), kLdWarps);
    mbar_init(sh.bar(kBarSFull), 1);
    mbar_init(sh.bar(kBarPReady), kSmWarps);
    mbar_init(sh.bar(kBarSm), kSmWarps * 32);
    for (int i = 0; i < 4; ++i) mbar_init(sh.bar(kBarPvDone + i), 1);
    for (int i = 0; i < 4; ++i) mbar_init(sh.bar(kBarRow + i), kLdWarps);
    *sh.abort_flag = 0;
    *sh.rescale_flag = 0;
    sh.vote[0] = 0;
    sh.vote[1] = 0;
    fence_mbar_init();
  }
  if (threadIdx.x < 32) reinterpret_cast<uint32_t*>(base + L::kOnesOff)[threadIdx.x] = 0x3F803F80u;
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(smem_u32(sh.tmem_slot), TmemCols<NH>::kAlloc);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sh.tmem_slot;

  if (warp < kSmWarps) {
    softmax_role<NH>(a, sh, tmem, lo, n);
  } else {
    loader_role<NH>(a, sh, lo, n);
    cp_async_wait_all();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TmemCols<NH>::kAlloc);
  }
}

// Split-K combine: one warp per (token, head). Lanes hold the partials' base-2 LSEs; the
// max and the sum of weights are warp-shuffle reductions; each lane then accumulates 16 of
// the 512 channels over the partials, applies the sink and writes bf16 O and natural-log LSE.
__global__ void __launch_bounds__(256) combine_kernel(const AttnArgs a) {
  const int wg = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (wg >= a.T * a.H) return;
  const int t = wg / a.H;
  const int h = wg - t * a.H;
  const long long item = static_cast<long long>(t) * a.groups + h / a.heads_per_group;
  const long long x0 = item * a.tiles_per_item;
  const int c0 = static_cast<int>(split_owner(x0, a.total_tiles, a.nctas));
  const int ns = static_cast<int>(split_owner(x0 + a.tiles_per_item - 1, a.total_tiles, a.nctas)) - c0 + 1;
  auto lse_at = [&](int s) { return a.part_lse[(static_cast<int64_t>(s) * a.T + t) * a.H + h]; };
  float M = -INFINITY;
  for (int s = lane; s < ns; s += 32) M = fmaxf(M, lse_at(s));
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  uint16_t* orow = a.out + static_cast<int64_t>(t) * a.out_stride_t + static_cast<int64_t>(h) * a.out_stride_h;
  if (M == -INFINITY) {
    reinterpret_cast<uint4*>(orow + lane * 16)[0] = make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4*>(orow + lane * 16)[1] = make_uint4(0, 0, 0, 0);
    if (lane == 0 && a.lse != nullptr) a.lse[static_cast<int64_t>(t) * a.lse_stride_t + h] = -INFINITY;
    return;
  }
  float W = 0.f;
  for (int s = lane; s < ns; s += 32) W += exp2f(lse_at(s) - M);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) W += __shfl_xor_sync(0xffffffffu, W, off);
  const float L2 = M + log2f(W);
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  const uint16_t* part = static_cast<const uint16_t*>(a.part_o);
  for (int s0 = 0; s0 < ns; s0 += 32) {
    const int s = s0 + lane;
    const float wl = s < ns ? exp2f(lse_at(s) - L2) : 0.f;
    const int cnt = min(32, ns - s0);
    for (int k = 0; k < cnt; ++k) {
      const float w = __shfl_sync(0xffffffffu, wl, k);
      if (w == 0.f) continue;
      const uint4* src = reinterpret_cast<const uint4*>(
          part + ((static_cast<int64_t>(s0 + k) * a.T + t) * a.H + h) * kDv + lane * 16);
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const uint4 v = src[q];
        const uint32_t wv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv[e]));
          acc[8 * q + 2 * e] += w * f.x;
          acc[8 * q + 2 * e + 1] += w * f.y;
        }
      }
    }
  }
  float f = 1.f;
  if (a.sink != nullptr) f = 1.f / (1.f + exp2f(a.sink[h] * 1.4426950408889634f - L2));
  uint32_t w32[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * k] * f, acc[2 * k + 1] * f);
    w32[k] = *reinterpret_cast<const uint32_t*>(&b);
  }
  reinterpret_cast<uint4*>(orow + lane * 16)[0] = make_uint4(w32[0], w32[1], w32[2], w32[3]);
  reinterpret_cast<uint4*>(orow + lane * 16)[1] = make_uint4(w32[4], w32[5], w32[6], w32[7]);
  if (lane == 0 && a.lse != nullptr) a.lse[static_cast<int64_t>(t) * a.lse_stride_t + h] = L2 * 0.6931471805599453f;
}

template <int NH>
cudaError_t launch_nh(const AttnArgs& a, const Plan& plan, cudaStream_t stream, cudaEvent_t ev0, cudaEvent_t ev1) {
  const int smem = Smem<NH>::kAlloc;
  cudaError_t e = cudaFuncSetAttribute(sparse_mla_kernel<NH>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) {
    note_cuda_error(e, "cudaFuncSetAttribute(sparse_mla_kernel, max dynamic shared memory)");
    return e;
  }
  if (ev0) cudaEventRecord(ev0, stream);
  sparse_mla_kernel<NH><<<plan.nctas, kThreads, smem, stream>>>(a);
  e = cudaGetLastError();
  if (ev1) cudaEventRecord(ev1, stream);
  if (e != cudaSuccess) {
    note_cuda_error(e, "launch of sparse_mla_kernel");
    return e;
  }
  if (plan.split) {
    const long long warps = static_cast<long long>(a.T) * a.H;
    combine_kernel<<<static_cast<unsigned>((warps + 7) / 8), 256, 0, stream>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) note_cuda_error(e, "launch of combine_kernel");
  }
  return e;
}

}  // namespace

cudaError_t launch_attention(const AttnArgs& args, const Plan& plan, cudaStream_t stream, cudaEvent_t ev0,
                             cudaEvent_t ev1) {
  switch (plan.nh) {
    case 16: return launch_nh<16>(args, plan, stream, ev0, ev1);
    case 32: return launch_nh<32>(args, plan, stream, ev0, ev1);
    case 64: return launch_nh<64>(args, plan, stream, ev0, ev1);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t read_and_clear_device_error(int* code) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(code, g_device_error, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
}

}  // namespace smla
