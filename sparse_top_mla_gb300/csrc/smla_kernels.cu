// Sparse top-k MLA attention kernels for GB300 (sm_103a).
//
// Persistent, warp-specialised kernel. Each CTA (one per SM) walks a stream of tiles; a tile
// is 128 gathered cache rows of one work item (query token t, head group g). Roles:
//   warps 0-3   softmax + epilogue; thread i owns gathered row i of every tile (= TMEM lane i)
//               and also resolves that row's index -> cache row offset three tiles ahead
//               (index, then block table and sequence length, then the byte offset), so the
//               loaders only read finished offsets from shared memory. Warp 3 runs the MMA
//               issue stream; its lane 0 issues every tcgen05 MMA and commit.
//   warps 4-11  loaders: keep the next tile's raw rows in registers and store each 128-channel
//               block pair into shared memory as soon as the previous tile's PV has released it
//               (FP8 rows are dequantised to bf16 on the way: e4m3 * per-128-channel scale)
// Per tile the tensor core computes
//   S^T[128 x NH]  = K_tile[128 x 576] . Q^T          (M = gathered rows, N = heads)
//   O^T[512 x NH] += V^T[512 x 128] . P^T[128 x NH]  (M = value channels, 4 blocks)
//   L[128 x NH]   += 1[128 x 128] . P^T[128 x NH]    (row sums of P, every lane equal)
// with S^T, L and O^T in TMEM. V is the first 512 channels of the same gathered tile (the
// tile is read K-major for QK^T and MN-major for PV). For tile j the issuing thread queues PV
// of all four block pairs (one commit each) and the row sums, then QK^T of tile j+1 block by
// block as the loaders refill the blocks PV has finished with.
//
// Softmax: P = 2^(s*scale*log2e - m) against per-head running maxima m. A tile whose scores
// stay within 2^8 of the maxima (the common case) needs one barrier among the softmax warps,
// on which they learn whether any row overflowed; only then do they run the rescale pass (new
// maxima, O^T and L rescaled, P recomputed) before PV is issued. The first tile of an item
// always takes the max pass.
//
// Schedules: whole items per CTA (prefill; the epilogue writes O and LSE), or contiguous
// flat tile ranges per CTA (split-K decode; every item segment writes a normalised partial
// O in bf16 and a base-2 partial LSE, merged by combine_kernel).
//
// Heads ride in the MMA N dimension (16, 32 or 64 per group), so every head count runs
// without padding memory traffic or outputs; unused N columns are zero Q rows.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <type_traits>

#include "smla_internal.h"
#include "smla_ptx.cuh"

namespace smla {

__device__ int g_device_error;

// Event timestamps (global timer, ns) per CTA for timeline analysis; compiled in only with
// -DSMLA_TRACE. Slot layout: 0 entry, 1 after the dependency wait, 2 exit, 3 first rows
// published, 4 first loads issued; tile j < 10 at 8 + 24j: +0 S^T ready, +1 fast pass done,
// +2 P^T final (issuer), +3 PV issued, +4 / +10 / +5 blocks 0-3 / 4-7 / 8 stored (issuer),
// +6 / +7 / +11 the loaders' arrivals for them, +8/+9 epilogue start/end, +12..15 the loaders
// past the release of block pair 0..3, +16..19 block pair 0..3 stored, +20..23 its refill
// issued.
#ifdef SMLA_TRACE
__device__ unsigned long long g_trace[1024][256];
#define SMLA_TRACE_AT(slot)                                                  \
  do {                                                                       \
    unsigned long long t_;                                                   \
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                  \
    if (blockIdx.x < 1024 && (slot) < 256) g_trace[blockIdx.x][(slot)] = t_; \
  } while (0)
#define SMLA_TRACE_TILE(j, k) SMLA_TRACE_AT(((j) < 10 ? 8 + 24 * (j) + (k) : 255))
#else
#define SMLA_TRACE_AT(slot) \
  do {                      \
  } while (0)
#define SMLA_TRACE_TILE(j, k) \
  do {                        \
  } while (0)
#endif

namespace {

using namespace ptx;

constexpr int kSmWarps = 4;
constexpr int kLdWarps = 8;
constexpr int kLdThreads = kLdWarps * 32;
constexpr int kThreads = (kSmWarps + kLdWarps) * 32;  // 384
constexpr int kLdRows = kTile / (kLdThreads / 8);      // rows per loader thread: 4
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
  static constexpr int kRedOff = kQOff + kKBlocks * NH * 128;  // float [4][64] per-warp column maxima
  static constexpr int kMOff = kRedOff + 4 * 64 * 4;            // float [64] running max (base 2)
  static constexpr int kMUseOff = kMOff + 64 * 4;               // float [64] exponent offset (0 while max = -inf)
  static constexpr int kThrOff = kMUseOff + 64 * 4;             // float [64] s*scale - m_use above this: rescale
  static constexpr int kAlphaOff = kThrOff + 64 * 4;            // float [64] rescale factor
  static constexpr int kFinOff = kAlphaOff + 64 * 4;            // float [64] output factor per head
  static constexpr int kRowOff = kFinOff + 64 * 4;              // int32 [4][128] rows: page << 6 | row (-1 = masked)
  static constexpr int kResOff = kRowOff + 4 * kTile * 4;       // int32 [2][5][128] index-resolution staging
  static constexpr int kBarOff = kResOff + 2 * 5 * kTile * 4;   // mbarriers
  static constexpr int kNumBars = 24;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;       // tmem base, flags
  static constexpr int kBytes = kMiscOff + 128;
  static constexpr int kAlloc = kBytes + 1024;                  // + alignment slack
};
static_assert(Smem<64>::kAlloc <= 232448, "shared memory budget");

// barrier indices
constexpr int kBarFullA = 0;      // tile blocks 0-3 stored (8 loader warps arrive)
constexpr int kBarFullB = 1;      // tile blocks 4-7 stored (8 loader warps arrive)
constexpr int kBarFullR = 2;      // tile block 8 (rope) stored (8 loader warps arrive)
constexpr int kBarSFull = 9;      // S^T of the tile is in TMEM (tcgen05.commit)
constexpr int kBarPvDone = 11;    // [4] PV block pair done (tcgen05.commit)
constexpr int kBarRow = 15;       // [4] rows of tile j in slot j&3 (softmax warps 0-2 arrive)
constexpr int kBarSm = 19;        // barrier among the 128 softmax threads (every thread arrives)
constexpr int kBarPFixed = 21;    // rescale pass done, P^T rewritten (4 softmax warps arrive)
constexpr int kBarRowsum = 22;    // row sums (issued after the last PV block pair) done (tcgen05.commit)

template <int NH>
struct TmemCols {
  static constexpr int kS = 0;
  static constexpr int kL = 64;   // row sums of P per head, accumulated by the tensor core (all lanes equal)
  static constexpr int kO = 128;  // O^T block b at kO + b*NH
  static constexpr int kAlloc = (kO + 4 * NH) <= 256 ? 256 : 512;
  // bf16 1.0 in 16 columns, the A operand of the row sums (read from TMEM, so the row sums
  // take no shared-memory bandwidth for it): past O^T, or in the gap after S^T when O^T fills
  // the allocation
  static constexpr int kOnes = (kO + 4 * NH + 16) <= kAlloc ? kO + 4 * NH : 32;
  static_assert((kOnes >= kO + 4 * NH && kOnes + 16 <= kAlloc) || (kOnes >= NH && kOnes + 16 <= kL),
                "ones columns overlap another TMEM region");
};

struct Shared {
  uint8_t* base;
  uint32_t tile, q;
  float *red, *m_run, *m_use, *thr, *alpha, *fin;
  int32_t* rowoff;
  uint32_t res;     // staging of the index-resolution loads (cp.async destination)
  int32_t* resp;    // the same staging, generic pointer
  uint32_t bars;
  uint32_t* tmem_slot;
  volatile int* abort_flag;
  volatile int* rescale_flag;
  volatile int* overflow;  // [2] tag j+1: a score of tile j passed its threshold (by tile parity)
  __device__ uint32_t bar(int i) const { return bars + 8u * i; }
};

// Bounded wait on an mbarrier phase. The common case (phase already complete) is inline; the
// waiting loop is one out-of-line copy: the thread sleeps in hardware between checks, and only
// after a sleep ends without the phase does it look at the abort flag and the clock.
__device__ __noinline__ bool wait_bar_slow(volatile int* abort_flag, uint32_t bar, uint32_t parity) {
  const long long t0 = clock64();
  for (;;) {
    if (mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > kSpinCycles) {
      atomicExch(&g_device_error, kErrTimeout);
      *abort_flag = 1;
      return false;
    }
  }
}
__device__ __forceinline__ bool wait_bar(const Shared& sh, uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_bar_slow(sh.abort_flag, bar, parity);
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
// Position in the CTA's tile stream: work item and tile within the item. Whole-item schedule:
// items blockIdx.x, blockIdx.x + nctas, ...; split schedule: consecutive flat tiles from lo.
struct Cursor {
  uint32_t item;
  int tile;
  __device__ __forceinline__ void init(const AttnArgs& a, long long lo) {
    if (a.split) {
      item = static_cast<uint32_t>(lo / a.tiles_per_item);
      tile = static_cast<int>(lo - static_cast<long long>(item) * a.tiles_per_item);
    } else {
      item = blockIdx.x;
      tile = 0;
    }
  }
  __device__ __forceinline__ void next(const AttnArgs& a) {
    if (++tile == a.tiles_per_item) {
      tile = 0;
      item += a.split ? 1u : static_cast<uint32_t>(a.nctas);
    }
  }
};

// Head groups per token: 1, 2 or 4 (a power of two); item = token * groups + group.
__device__ __forceinline__ uint32_t item_token(const AttnArgs& a, uint32_t item) {
  return item >> (31 - __clz(a.groups));
}
__device__ __forceinline__ int item_head0(const AttnArgs& a, uint32_t item) {
  return static_cast<int>(item & static_cast<uint32_t>(a.groups - 1)) * a.heads_per_group;
}

__device__ __forceinline__ int set_of(const AttnArgs& a, int tile) {
  return (a.nsets > 1 && tile >= a.set[0].ntiles) ? 1 : 0;
}

// Fields of set 0 or 1, selected field by field (a runtime index into the kernel-parameter
// array would force a local-memory copy of the parameters).
#define SET_FIELD(a, sid, f) ((sid) ? (a).set[1].f : (a).set[0].f)

// ------------------------------------------------------------------ index resolution
// Entry -> cache row (page << 6 | row in page, -1 when masked) in three phases whose loads only
// depend on the previous phase; a softmax thread runs each phase one tile after the previous
// one. The loads are asynchronous copies into a shared staging area (double-buffered by tile
// parity), so no load result waits in a register for a tile.
constexpr int kResIdx = 0, kResTl = 1, kResSeq = 2, kResPage = 3, kResLen = 4;
__device__ __forceinline__ int res_slot(int jt, int field, int r) { return ((jt & 1) * 5 + field) * kTile + r; }

struct ResA {  // phase A issued: entry number, set, which copies were made (1 index, 2 length limit)
  int e, sid, flags;
};
struct ResB {  // phase B issued: index, set, which copies were made (1 page, 2 sequence length)
  int idx, sid, flags;
};

__device__ __forceinline__ void res_a(const AttnArgs& a, const Shared& sh, const Cursor& c, int jt, int r, ResA& R) {
  const uint32_t t = item_token(a, c.item);
  const int sid = set_of(a, c.tile);
  R.sid = sid;
  R.e = (c.tile - (sid ? a.set[0].ntiles : 0)) * kTile + r;
  R.flags = 0;
  if (R.e < SET_FIELD(a, sid, topk)) {
    const int32_t* ip = SET_FIELD(a, sid, indices) + static_cast<int64_t>(t) * SET_FIELD(a, sid, idx_stride);
    cp_async4(sh.res + 4 * res_slot(jt, kResIdx, r), ip + R.e);
    R.flags |= 1;
  }
  const int32_t* tl = SET_FIELD(a, sid, topk_length);
  if (tl != nullptr) {
    cp_async4(sh.res + 4 * res_slot(jt, kResTl, r), tl + t);
    R.flags |= 2;
  }
  cp_async4(sh.res + 4 * res_slot(jt, kResSeq, r), a.token_seq + t);
}

// Needs phase A's copies complete.
__device__ __forceinline__ void res_b(const AttnArgs& a, const Shared& sh, const ResA& A, int jt, int r, ResB& B) {
  const int sid = A.sid;
  const int tl = (A.flags & 2) ? sh.resp[res_slot(jt, kResTl, r)] : 0x7fffffff;
  const int seq = sh.resp[res_slot(jt, kResSeq, r)];
  B.sid = sid;
  B.idx = ((A.flags & 1) && A.e < tl) ? sh.resp[res_slot(jt, kResIdx, r)] : -1;
  B.flags = 0;
  if (seq >= 0 && seq < a.num_seqs) {
    cp_async4(sh.res + 4 * res_slot(jt, kResLen, r), SET_FIELD(a, sid, seq_lens) + seq);
    B.flags |= 2;
    const int32_t bts = SET_FIELD(a, sid, bt_stride);
    if (B.idx >= 0 && (B.idx >> 6) < bts) {
      cp_async4(sh.res + 4 * res_slot(jt, kResPage, r),
                SET_FIELD(a, sid, block_table) + static_cast<int64_t>(seq) * bts + (B.idx >> 6));
      B.flags |= 1;
    }
  }
}

// Needs phase B's copies complete.
__device__ __forceinline__ int32_t res_c(const AttnArgs& a, const Shared& sh, const ResB& B, int jt, int r) {
  const int seqlen = (B.flags & 2) ? sh.resp[res_slot(jt, kResLen, r)] : 0;
  const int page = (B.flags & 1) ? sh.resp[res_slot(jt, kResPage, r)] : -1;
  return (B.idx >= 0 && B.idx < seqlen && page >= 0 && page < SET_FIELD(a, B.sid, num_pages))
             ? (page << 6) | (B.idx & 63)
             : -1;
}

// Row r of tile jt -> shared slot jt&3, read by the loaders and by the softmax thread of row r.
__device__ __forceinline__ void publish_row(const Shared& sh, int jt, int r, int32_t row) {
  sh.rowoff[(jt & 3) * kTile + r] = row;
}
// The warp's rows of tile jt are published: one arrival per warp.
__device__ __forceinline__ void publish_done(const Shared& sh, int jt, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(sh.bar(kBarRow + (jt & 3)));
}

// ------------------------------------------------------------------ helpers
// Column maxima of N (16 or 32) values per lane across the warp: one warp-wide float max
// reduction (`redux.sync.max.f32`, every lane receives the result) per column; lane c keeps
// column c's and writes it to red_w[c].
template <int N>
__device__ __forceinline__ void warp_col_max_store(const float* v, int lane, float* red_w) {
  float mine = -INFINITY;
#pragma unroll
  for (int c = 0; c < N; ++c) {
    float r;
    asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v[c]));
    mine = lane == c ? r : mine;
  }
  if (lane < N) red_w[lane] = mine;
}

// One e4m3 pair -> bf16x2: exact conversion to f16x2 and then to two fp32 values, one packed
// fp32x2 multiply by {scale, scale} (round to nearest), one rounding to bf16 (RNE).
__device__ __forceinline__ uint32_t dequant_pair(uint16_t pair, uint64_t scale2) {
  uint32_t out;
  asm("{\n .reg .b16 lo, hi;\n .reg .b32 h2;\n .reg .f32 a, b;\n .reg .b64 f, r;\n"
      " cvt.rn.f16x2.e4m3x2 h2, %1;\n mov.b32 {lo, hi}, h2;\n"
      " cvt.f32.f16 a, lo;\n cvt.f32.f16 b, hi;\n mov.b64 f, {a, b};\n"
      " mul.rn.f32x2 r, f, %2;\n mov.b64 {a, b}, r;\n cvt.rn.bf16x2.f32 %0, b, a;\n}\n"
      : "=r"(out)
      : "h"(pair), "l"(scale2));
  return out;
}

__device__ __forceinline__ void dequant16(const uint4 raw, float scale, uint4& lo, uint4& hi) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  uint64_t scale2;
  asm("mov.b64 %0, {%1, %1};" : "=l"(scale2) : "f"(scale));
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    o[2 * i] = dequant_pair(static_cast<uint16_t>(w[i] & 0xFFFFu), scale2);
    o[2 * i + 1] = dequant_pair(static_cast<uint16_t>(w[i] >> 16), scale2);
  }
  lo = make_uint4(o[0], o[1], o[2], o[3]);
  hi = make_uint4(o[4], o[5], o[6], o[7]);
}

__device__ __forceinline__ uint32_t swz(int row, int chunk) {  // 128-byte swizzle inside a 1 KB atom
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// TMEM columns [c, c+W) of this warp's lanes into v (W = 16 or 32): issue, and the wait that
// makes v usable (it waits for every earlier load of the thread).
template <int W>
__device__ __forceinline__ void tmem_load_nw(uint32_t addr, float* v) {
  if constexpr (W == 32) {
    tmem_ld32_nw(addr, v);
  } else {
    tmem_ld16_nw(addr, v);
  }
}
template <int W>
__device__ __forceinline__ void tmem_load_wait(float* v) {
  if constexpr (W == 32) {
    tmem_ld_wait32(v);
  } else {
    tmem_ld_wait16(v);
  }
}

// TMEM columns [c, c+W) of this warp's lanes into v (W = 16 or 32), waited.
template <int W>
__device__ __forceinline__ void tmem_load(uint32_t addr, float* v) {
  if constexpr (W == 32) {
    tmem_ld32_nw(addr, v);
    tmem_ld_wait32(v);
  } else {
    tmem_ld16_nw(addr, v);
    tmem_ld_wait16(v);
  }
}

// ------------------------------------------------------------------ loader role
// Thread u (0..255) owns rows rg + 32k, k < 4 (rg = u/8) and the 16-byte chunk lane8 = u%8
// of every 128-byte row segment, so 8 consecutive threads read 128 contiguous bytes.
//
// Register staging (4 slots of one 16-byte chunk per row): an FP8 block pair needs one slot,
// so FP8 tiles are loaded a whole tile ahead (block pair bp of tile j+1 is issued as soon as
// block pair bp of tile j is stored); a bf16 block pair needs two slots, so bf16 tiles are
// loaded half a tile ahead (block pair bp+2 after bp is stored).
struct LdData {
  uint4 d[4][kLdRows];   // [slot][row k]
  float sc[4][kLdRows];  // fp8 scale of the block pair held in slot [s][row k]
  uint4 rope[kLdRows];
};

template <int S>  // fp8 block pair -> slot S
__device__ __forceinline__ void ld_issue_fp8(const uint8_t* cache, const int64_t* off, int lane8, int bp, LdData& D) {
#pragma unroll
  for (int k = 0; k < kLdRows; ++k) {
    D.d[S][k] = make_uint4(0, 0, 0, 0);
    D.sc[S][k] = 0.f;
    if (off[k] >= 0) {
      const uint8_t* row = cache + off[k];
      D.d[S][k] = ldg_nc_v4(row + 128 * bp + 16 * lane8);
      D.sc[S][k] = ldg_nc_f32(row + 512 + 4 * bp);
    }
  }
}

template <int P>  // bf16 block pair -> slots 2P, 2P+1
__device__ __forceinline__ void ld_issue_bf16(const uint8_t* cache, const int64_t* off, int lane8, int bp, LdData& D) {
#pragma unroll
  for (int k = 0; k < kLdRows; ++k) {
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
  for (int k = 0; k < kLdRows; ++k) {
    D.rope[k] = make_uint4(0, 0, 0, 0);
    if (off[k] >= 0) D.rope[k] = ldg_nc_v4(cache + off[k] + (fmt == 0 ? 1024 : 528) + 16 * lane8);
  }
}

// Rows k < kDqAhead of the fp8 block pair in slot S, dequantised into registers ahead of the
// wait for their store (the other rows are converted after it: registers do not allow more).
constexpr int kDqAhead = 2;
template <int S>
__device__ __forceinline__ void ld_dequant_fp8(const LdData& D, uint4 (&dq)[kDqAhead][2]) {
#pragma unroll
  for (int k = 0; k < kDqAhead; ++k) dequant16(D.d[S][k], D.sc[S][k], dq[k][0], dq[k][1]);
}

// An fp8 chunk of 16 channels becomes two bf16 chunks of block 2bp + lane8/4. The threads
// of the second block store their two chunks in the opposite order, so the 8 threads of a
// store phase always hit 8 different 16-byte bank groups.
template <int S>
__device__ __forceinline__ void ld_store_fp8(const Shared& sh, int rg, int lane8, int bp, const LdData& D,
                                             const uint4 (&dq)[kDqAhead][2]) {
  const bool second = (lane8 >> 2) != 0;
  const uint32_t blk = sh.tile + (2 * bp + (lane8 >> 2)) * kBlockBytes;
  const int c0 = (lane8 & 3) * 2;
#pragma unroll
  for (int k = 0; k < kLdRows; ++k) {
    const int r = rg + 32 * k;
    uint4 lo, hi;
    if (k < kDqAhead) {
      lo = dq[k < kDqAhead ? k : 0][0];
      hi = dq[k < kDqAhead ? k : 0][1];
    } else {
      dequant16(D.d[S][k], D.sc[S][k], lo, hi);
    }
    sts_v4(blk + swz(r, c0 + (second ? 1 : 0)), second ? hi : lo);
    sts_v4(blk + swz(r, c0 + (second ? 0 : 1)), second ? lo : hi);
  }
}

template <int P>
__device__ __forceinline__ void ld_store_bf16(const Shared& sh, int rg, int lane8, int bp, const LdData& D) {
#pragma unroll
  for (int k = 0; k < kLdRows; ++k) {
    const int r = rg + 32 * k;
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

// Q of one work item (NH heads x 576 channels, zero rows past the group's heads) -> shared
// memory in the 128-byte-swizzled K-major layout, by the 256 loader threads (cp.async).
template <int NH>
__device__ __forceinline__ void load_q_tile(const AttnArgs& a, const Shared& sh, uint32_t item, int u) {
  const uint32_t t = item_token(a, item);
  const int h0 = item_head0(a, item);
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
}

// F0, F1: cache formats of the main and the extra set (compile-time, so each kernel carries only
// the load paths it uses).
template <int NH, int F0, int F1>
__device__ __forceinline__ void loader_role(const AttnArgs& a, const Shared& sh, long long lo, int n) {
  const int u = threadIdx.x - kSmWarps * 32;
  const int lane = threadIdx.x & 31;
  const int lane8 = u & 7;
  const int rg = u >> 3;
  if (n <= 0) return;

  auto load_q = [&](uint32_t item) { load_q_tile<NH>(a, sh, item, u); };
  auto prefetch_q = [&](uint32_t item) {
    const uint32_t t = item_token(a, item);
    const int h0 = item_head0(a, item);
    const int hg = min(a.heads_per_group, a.H - h0);
    for (int e = u; e < hg * 9; e += kLdThreads) {
      const uint16_t* p = a.q + static_cast<int64_t>(t) * a.q_stride_t +
                          static_cast<int64_t>(h0 + e / 9) * a.q_stride_h + (e % 9) * 64;
      asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
    }
  };
  // byte offsets of this thread's rows of tile jt (published by the softmax threads three
  // tiles ahead of their use); one barrier wait per tile
  auto get_off = [&](int jt, const Cursor& c, int64_t* off) -> bool {
    if (!wait_bar_w(sh, sh.bar(kBarRow + (jt & 3)), (jt >> 2) & 1)) return false;
    const int sid = set_of(a, c.tile);
    const int64_t ps = SET_FIELD(a, sid, page_stride);
    const int64_t rs = SET_FIELD(a, sid, row_stride);
#pragma unroll
    for (int k = 0; k < kLdRows; ++k) {
      const int32_t p = sh.rowoff[(jt & 3) * kTile + rg + 32 * k];
      off[k] = p < 0 ? -1 : static_cast<int64_t>(p >> 6) * ps + static_cast<int64_t>(p & 63) * rs;
    }
    return true;
  };

  auto fmt_of = [&](const Cursor& c) { return F0 == F1 ? F0 : (set_of(a, c.tile) ? F1 : F0); };
  auto cache_of = [&](const Cursor& c) { return SET_FIELD(a, set_of(a, c.tile), cache); };
  // Whole rows of tile jt into L2, one bulk prefetch per row, two tiles ahead of their loads:
  // the loads then hit L2, and DRAM serves each gathered row as one contiguous read instead of
  // one access per 128-byte block pair. Called for tiles 3 on: at kernel start every CTA's first
  // loads already saturate DRAM.
  auto prefetch_rows = [&](int jt, const Cursor& c) -> bool {
    int64_t off[kLdRows];
    if (!get_off(jt, c, off)) return false;
    if (lane8 == 0) {
      const uint8_t* cache = cache_of(c);
      const uint32_t bytes = fmt_of(c) == 1 ? kRowFp8 : kRowBf16;
#pragma unroll
      for (int k = 0; k < kLdRows; ++k)
        if (off[k] >= 0) prefetch_l2_bulk(cache + off[k], bytes);
    }
    return true;
  };

  Cursor cur;
  cur.init(a, lo);
  LdData D;
  int64_t off_cur[kLdRows], off_nxt[kLdRows];
  load_q(cur.item);  // the first item's Q, while the first row offsets are being resolved
  if (!get_off(0, cur, off_cur)) return;
  {
    const uint8_t* cache = cache_of(cur);
    if (fmt_of(cur) == 1) {
      ld_issue_fp8<0>(cache, off_cur, lane8, 0, D);
      ld_issue_fp8<1>(cache, off_cur, lane8, 1, D);
      ld_issue_fp8<2>(cache, off_cur, lane8, 2, D);
      ld_issue_fp8<3>(cache, off_cur, lane8, 3, D);
      ld_issue_rope(1, cache, off_cur, lane8, D);
    } else {
      ld_issue_bf16<0>(cache, off_cur, lane8, 0, D);
      ld_issue_bf16<1>(cache, off_cur, lane8, 1, D);
    }
  }
  if (u == 0) SMLA_TRACE_AT(4);

  for (int j = 0; j < n; ++j) {
    const bool first = cur.tile == 0 || j == 0;
    const bool has1 = j + 1 < n;
    Cursor nxt = cur;
    nxt.next(a);
    auto next_rows = [&]() -> bool {
      if (nxt.tile == 0) prefetch_q(nxt.item);
      return get_off(j + 1, nxt, off_nxt);
    };
    // rows of the next two tiles, while the tensor core still works on the previous tile; on the
    // first tile the next rows are taken after its first store instead (at the start of the stream
    // tile 1 is still being resolved while tile 0 is stored), and tiles 1 and 2 are not prefetched
    if (j > 0 && has1 && !next_rows()) return;
    if (j > 0 && j + 2 < n) {
      Cursor c2 = nxt;
      c2.next(a);
      if (!prefetch_rows(j + 2, c2)) return;
    }
    const int fmt_cur = fmt_of(cur);
    const int fmt_nxt = has1 ? fmt_of(nxt) : 0;
    const uint8_t* cache_cur = cache_of(cur);
    const uint8_t* cache_nxt = has1 ? cache_of(nxt) : cache_cur;
    // fp8: each block pair is dequantised before the wait for its PV release, so only the
    // shared-memory stores remain on the path from that release to the tensor core
    uint4 dq[kDqAhead][2];
    if (fmt_cur == 1) ld_dequant_fp8<0>(D, dq);
    auto step = [&](auto bpc) -> bool {
      constexpr int bp = decltype(bpc)::value;
      if (j > 0 && !wait_bar_w(sh, sh.bar(kBarPvDone + bp), (j - 1) & 1)) return false;
      if (u == 0) SMLA_TRACE_TILE(j, 12 + bp);
      if (bp == 0 && first && j > 0) load_q(cur.item);
      if (fmt_cur == 1) {
        ld_store_fp8<bp>(sh, rg, lane8, bp, D, dq);
      } else {
        ld_store_bf16<(bp & 1)>(sh, rg, lane8, bp, D);
      }
      if (u == 0) SMLA_TRACE_TILE(j, 16 + bp);
      if (bp == 0 && first) cp_async_wait_all();
      if (bp & 1) {  // blocks 0-3 (after bp 1) or 4-7 (after bp 3) complete
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(sh.bar(bp == 1 ? kBarFullA : kBarFullB));
        if (u == 0) SMLA_TRACE_TILE(j, bp == 1 ? 6 : 7);
      }
      if (bp == 3) {
        // the rope block holds the previous tile's P^T until its row sums (issued after the
        // last PV block pair) have read it
        if (j > 0 && !wait_bar_w(sh, sh.bar(kBarRowsum), (j - 1) & 1)) return false;
#pragma unroll
        for (int k = 0; k < kLdRows; ++k) sts_v4(sh.tile + 8 * kBlockBytes + swz(rg + 32 * k, lane8), D.rope[k]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(sh.bar(kBarFullR));
        if (u == 0) SMLA_TRACE_TILE(j, 11);
      }
      // first tile: an fp8 tile's first refill already needs the next rows; a bf16 tile's
      // first refills still read the current tile
      if (j == 0 && bp == 0 && has1 && fmt_cur == 1 && !next_rows()) return false;
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
      } else if (bp == 0) {
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
      if (u == 0) SMLA_TRACE_TILE(j, 20 + bp);
      if (j == 0 && bp == 0 && has1 && fmt_cur != 1 && !next_rows()) return false;
      if (fmt_cur == 1 && bp < 3) ld_dequant_fp8<(bp < 3 ? bp + 1 : 3)>(D, dq);
      return true;
    };
    if (!step(std::integral_constant<int, 0>{}) || !step(std::integral_constant<int, 1>{}) ||
        !step(std::integral_constant<int, 2>{}) || !step(std::integral_constant<int, 3>{}))
      return;
    cur = nxt;
#pragma unroll
    for (int k = 0; k < kLdRows; ++k) off_cur[k] = off_nxt[k];
  }
}

// ------------------------------------------------------------------ MMA issue (one thread)
// Descriptor low words are built once per call; each MMA adds a compile-time byte offset (>> 4)
// to the start address field. The high words are constants of the operand layouts.
struct MmaDesc {
  uint32_t qk_a, qk_b, pv_a, pv_b;
};
constexpr uint32_t kHiK128 = smem_desc_hi(1024, kSwizzle128B);  // K-major, 128B swizzle, 8-row groups 1 KB apart
constexpr uint32_t kHiP = smem_desc_hi(2048, kSwizzleNone);     // P^T: 8x8 core matrices, N groups 2 KB apart

template <int NH>
__device__ __forceinline__ MmaDesc make_descs(const Shared& sh) {
  MmaDesc d;
  d.qk_a = smem_desc_lo(sh.tile, 16);
  d.qk_b = smem_desc_lo(sh.q, 16);
  d.pv_a = smem_desc_lo(sh.tile, kBlockBytes);
  d.pv_b = smem_desc_lo(sh.tile + 8 * kBlockBytes, 128);
  return d;
}

// The whole issuing warp runs the issue code (waits are warp-wide); elect.sync inside each MMA
// and commit picks the one lane that issues. A warp whose lanes stay diverged for the length
// of an issue sequence pays several hundred cycles to reconverge afterwards.
//
// QK^T of tile j, waiting once for blocks 0-3 and once for blocks 4-8 (every mbarrier wait in
// the issue stream lets the tensor pipe run dry for a few hundred cycles). Fully unrolled: in
// a loop the advancing descriptors cost ~40 cycles per MMA.
template <int NH>
__device__ __forceinline__ bool mma_qk(const Shared& sh, const MmaDesc& d, uint32_t tmem, int j) {
  constexpr uint32_t idesc = idesc_bf16(128, NH, 0, 0);
#pragma unroll
  for (int kb = 0; kb < kKBlocks; ++kb) {
    if (kb == 0 || kb == 4 || kb == 8) {
      if (!wait_bar_w(sh, sh.bar(kb == 0 ? kBarFullA : (kb == 4 ? kBarFullB : kBarFullR)), j & 1)) return false;
      tc_fence_after();
      if (threadIdx.x == kIssueWarp * 32) SMLA_TRACE_TILE(j, kb == 0 ? 4 : (kb == 4 ? 10 : 5));
    }
    // four K steps of 16 channels: 32 bytes along the swizzled row of block kb
    mma_bf16_x4<2, 2>(tmem + TmemCols<NH>::kS, d.qk_a + static_cast<uint32_t>((kb * kBlockBytes) >> 4), kHiK128,
                      d.qk_b + static_cast<uint32_t>((kb * NH * 128) >> 4), kHiK128, idesc, kb != 0);
  }
  return true;
}

// O^T block pair bp (value channels 128bp..128bp+127) += V^T . P^T, then a commit that releases
// the tile's blocks 2bp, 2bp+1 to the loaders.
template <int NH>
__device__ __forceinline__ void mma_pv(const Shared& sh, const MmaDesc& d, uint32_t tmem, int bp, bool first) {
  constexpr uint32_t idesc = idesc_bf16(128, NH, 1, 1);
  const uint32_t da = d.pv_a + static_cast<uint32_t>((2 * bp * kBlockBytes) >> 4);
  // eight K steps of 16 tokens: 2 KB of V^T rows, 256 B of P^T core matrices per step
  mma_bf16_x4<128, 16>(tmem + TmemCols<NH>::kO + bp * NH, da, kHiK128, d.pv_b, kHiP, idesc, first ? 0u : 1u);
  mma_bf16_x4<128, 16>(tmem + TmemCols<NH>::kO + bp * NH, da + 512, kHiK128, d.pv_b + 64, kHiP, idesc, 1u);
  mma_commit_warp(sh.bar(kBarPvDone + bp));
}

// Row sums of P for every head: L[m, h] += sum_k 1 * P^T[k, h] (all 128 lanes get the same
// sums). Same B operand and accumulate rule as PV, so the normalisation uses exactly the bf16
// P that multiplied V.
template <int NH>
__device__ __forceinline__ void mma_rowsum(const MmaDesc& d, uint32_t tmem, bool first) {
  constexpr uint32_t idesc = idesc_bf16(128, NH, 0, 1);
  const uint32_t ones = tmem + TmemCols<NH>::kOnes;
  mma_bf16_ts_x4<16>(tmem + TmemCols<NH>::kL, ones, d.pv_b, kHiP, idesc, first ? 0u : 1u);
  mma_bf16_ts_x4<16>(tmem + TmemCols<NH>::kL, ones, d.pv_b + 64, kHiP, idesc, 1u);
}

// QK^T of tile j as its blocks arrive, then the commit that tells the softmax warps S^T is ready.
template <int NH>
__device__ __forceinline__ bool mma_issue_qk(const Shared& sh, uint32_t tmem, int j) {
  const MmaDesc d = make_descs<NH>(sh);
  if (!mma_qk<NH>(sh, d, tmem, j)) return false;
  mma_commit_warp(sh.bar(kBarSFull));
  return true;
}

// After the softmax of tile j: PV of all four block pairs (each with its own commit, so the
// loaders refill a block pair as soon as it is released), then the row sums with their own
// commit (the loaders store the next rope block, where this tile's P^T lives, after it). QK^T of
// tile j+1 follows at the top of the next iteration of the tile loop; when tile j ends an item
// the issuing warp first writes its share of the outputs (waiting for tile j+1's blocks first
// would hold back the next softmax, which needs every warp).
template <int NH>
__device__ __forceinline__ void mma_issue_pv(const Shared& sh, uint32_t tmem, int j, bool first) {
  const MmaDesc d = make_descs<NH>(sh);
  tc_fence_after();
#pragma unroll 1
  for (int bp = 0; bp < 4; ++bp) mma_pv<NH>(sh, d, tmem, bp, first);
  mma_rowsum<NH>(d, tmem, first);
  mma_commit_warp(sh.bar(kBarRowsum));
  if (threadIdx.x == kIssueWarp * 32) SMLA_TRACE_TILE(j, 3);
}

// ------------------------------------------------------------------ softmax / epilogue role
// P^T (bf16) of this thread's row from S^T: p = 2^(s*scale - m_use) per head. Returns whether
// the row is valid and some head's score passed its threshold (the running max must move).
// Invalid rows write zeros.
template <int NH>
__device__ __forceinline__ bool p_pass(const AttnArgs& a, const Shared& sh, uint32_t s_addr, uint32_t pt, bool valid,
                                       int tid) {
  constexpr int CW = NH < 32 ? NH : 32;
  bool over = false;
#pragma unroll 1
  for (int c0 = 0; c0 < NH; c0 += CW) {
    float s[CW];
    tmem_load<CW>(s_addr + c0, s);
    uint32_t w[CW / 2];
#pragma unroll
    for (int q = 0; q < CW / 4; ++q) {
      const float4 mu = reinterpret_cast<const float4*>(sh.m_use)[(c0 >> 2) + q];
      const float4 th = reinterpret_cast<const float4*>(sh.thr)[(c0 >> 2) + q];
      const float d0 = fmaf(s[4 * q + 0], a.scale_log2, -mu.x);
      const float d1 = fmaf(s[4 * q + 1], a.scale_log2, -mu.y);
      const float d2 = fmaf(s[4 * q + 2], a.scale_log2, -mu.z);
      const float d3 = fmaf(s[4 * q + 3], a.scale_log2, -mu.w);
      over |= (d0 > th.x) | (d1 > th.y) | (d2 > th.z) | (d3 > th.w);
      const __nv_bfloat162 b0 = __floats2bfloat162_rn(ex2(d0), ex2(d1));
      const __nv_bfloat162 b1 = __floats2bfloat162_rn(ex2(d2), ex2(d3));
      w[2 * q] = valid ? *reinterpret_cast<const uint32_t*>(&b0) : 0u;
      w[2 * q + 1] = valid ? *reinterpret_cast<const uint32_t*>(&b1) : 0u;
    }
    // P^T in the no-swizzle MN-major layout: [head/8][row/8][row%8][head%8]
#pragma unroll
    for (int g = 0; g < CW / 8; ++g)
      sts_v4(pt + ((c0 >> 3) + g) * 2048 + (tid >> 3) * 128 + (tid & 7) * 16,
             make_uint4(w[4 * g], w[4 * g + 1], w[4 * g + 2], w[4 * g + 3]));
  }
  return over && valid;
}

// Max pass: per-head maximum of the tile over valid rows, new running maxima (always on the
// first tile of an item; otherwise only where a maximum passed its threshold), O^T and L
// rescaled where a maximum moved, then P^T recomputed.
template <int NH>
__device__ __forceinline__ bool max_pass(const AttnArgs& a, const Shared& sh, uint32_t tmem_lane, uint32_t pt,
                                         bool valid, bool first, uint32_t& smph, int tid) {
  constexpr int CW = NH < 32 ? NH : 32;
  using TC = TmemCols<NH>;
  const int warp = tid >> 5;
  const int lane = tid & 31;
#pragma unroll 1
  for (int c0 = 0; c0 < NH; c0 += CW) {
    float s[CW];
    tmem_load<CW>(tmem_lane + TC::kS + c0, s);
#pragma unroll
    for (int h = 0; h < CW; ++h) s[h] = valid ? s[h] * a.scale_log2 : -INFINITY;
    warp_col_max_store<CW>(s, lane, sh.red + warp * 64 + c0);
  }
  if (!sm_sync(sh, smph)) return false;
  if (warp == 0) {
    bool raised = false;
    for (int h = lane; h < NH; h += 32) {
      const float tmax = fmaxf(fmaxf(sh.red[h], sh.red[64 + h]), fmaxf(sh.red[128 + h], sh.red[192 + h]));
      const float mo = first ? -INFINITY : sh.m_run[h];
      float m = mo, al = 1.f;
      if (first || tmax > mo + kLazyRescaleLog2) {
        m = tmax;
        al = (mo == -INFINITY) ? 0.f : ex2(mo - tmax);
        raised = true;
      }
      sh.m_run[h] = m;
      sh.m_use[h] = m == -INFINITY ? 0.f : m;
      sh.thr[h] = m == -INFINITY ? -INFINITY : kLazyRescaleLog2;
      sh.alpha[h] = al;
    }
    raised = __any_sync(0xffffffffu, raised);
    if (lane == 0) *sh.rescale_flag = raised ? 1 : 0;
  }
  if (!sm_sync(sh, smph)) return false;
  p_pass<NH>(a, sh, tmem_lane + TC::kS, pt, valid, tid);
  // O^T and the row sums *= alpha where a running max moved (the previous PV is complete:
  // S^T of this tile was committed after it)
  if (!first && *sh.rescale_flag != 0) {
#pragma unroll 1
    for (int b = 0; b <= 4; ++b) {
      const uint32_t col = b < 4 ? TC::kO + b * NH : TC::kL;
#pragma unroll 1
      for (int c0 = 0; c0 < NH; c0 += 16) {
        float o[16];
        const uint32_t addr = tmem_lane + col + c0;
        tmem_load<16>(addr, o);
#pragma unroll
        for (int i = 0; i < 16; ++i) o[i] *= sh.alpha[c0 + i];
        tmem_st16(addr, o);
      }
    }
    tmem_st_wait();
  }
  return true;
}

template <int NH>
__device__ __forceinline__ void softmax_role(const AttnArgs& a, const Shared& sh, uint32_t tmem, long long lo, int n) {
  constexpr int CW = NH < 32 ? NH : 32;
  using TC = TmemCols<NH>;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const uint32_t tl = tmem + (static_cast<uint32_t>(warp * 32) << 16);  // this warp's TMEM lanes
  const uint32_t pt = sh.tile + 8 * kBlockBytes;
  uint32_t smph = 0;
  bool tr_first = true;  // first epilogue of the CTA (event timestamps only)
  (void)tr_first;
  int nfix = 0;  // rescale passes so far (phase of PFixed)
  if (n <= 0) return;
  {
    // the row sums' A operand (bf16 1.0 pairs) in this warp's TMEM lanes; the issuer first reads
    // it after the PFixed barrier of the stream's first tile, which every warp reaches with a
    // fence after this store
    float ones[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) ones[i] = __uint_as_float(0x3F803F80u);
    tmem_st16(tl + TC::kOnes, ones);
    tmem_st_wait();
  }

  // ---- index resolution, by warps 0-2 (warp 0 also takes rows 96-127, so the issuing warp
  // stays free)
  const int nres = warp == 0 ? 2 : (warp < kIssueWarp ? 1 : 0);
  const int rrow[2] = {tid, 3 * 32 + lane};
  // both rows' state stays in registers: the calls below index it with constants
  auto each = [&](auto&& f) {
    f(std::integral_constant<int, 0>{});
    if (nres > 1) f(std::integral_constant<int, 1>{});
  };
  Cursor rc;
  rc.init(a, lo);
  ResA ra[2] = {{0, 0, 0}, {0, 0, 0}};
  ResB rb[2] = {{-1, 0, 0}, {-1, 0, 0}};
  // step j: publish tile j+3 (phase C), phase B of tile j+4, phase A of tile j+5; the copies it
  // waits for were issued by the previous step
  auto resolve_step = [&](int j) {
    cp_async_wait_all();
    if (j + 3 >= 0 && j + 3 < n) {
      each([&](auto q) { publish_row(sh, j + 3, rrow[q], res_c(a, sh, rb[q], j + 3, rrow[q])); });
      publish_done(sh, j + 3, lane);
    }
    if (j + 4 >= 0 && j + 4 < n) each([&](auto q) { res_b(a, sh, ra[q], j + 4, rrow[q], rb[q]); });
    if (j + 5 >= 0 && j + 5 < n) {
      each([&](auto q) { res_a(a, sh, rc, j + 5, rrow[q], ra[q]); });
      rc.next(a);
    }
    cp_async_commit();
  };
  // prologue: tiles 0-2 published, phase B of tile 3 and phase A of tile 4 issued
  if (nres > 0) {
#pragma unroll 1
    for (int j = -5; j < 0; ++j) resolve_step(j);
  }
  if (tid == 0) SMLA_TRACE_AT(3);


  Cursor cur;
  cur.init(a, lo);
  for (int j = 0; j < n; ++j, cur.next(a)) {
    const bool first = cur.tile == 0 || j == 0;
    const bool last = cur.tile == a.tiles_per_item - 1 || j == n - 1;
    if (warp == kIssueWarp) {
      tc_fence_after();
      if (!mma_issue_qk<NH>(sh, tmem, j)) return;
    }
    // resolution runs while QK^T of tile j is in flight, so tile j+3's rows are published before
    // the loaders look for them at the start of their next tile. It reuses the row slot of tile
    // j-1, whose readers (the loaders, two and three tiles earlier) finished before that tile's
    // S^T was ready.
    if (warp != kIssueWarp) resolve_step(j);
    const bool valid = sh.rowoff[(j & 3) * kTile + tid] >= 0;
    if (!wait_bar_w(sh, sh.bar(kBarSFull), j & 1)) return;
    tc_fence_after();
    if (tid == 0) SMLA_TRACE_TILE(j, 0);
    // the first tile of an item has no running maxima yet: it always takes the max pass, which
    // every warp knows, so it skips the fast pass and the decision barrier
    bool fix = true;
    if (!first) {
      const bool over = p_pass<NH>(a, sh, tl + TC::kS, pt, valid, tid);
      if (tid == 0) SMLA_TRACE_TILE(j, 1);
      // decision among the four softmax warps: a warp with an overflowing row tags the tile's
      // flag slot with j+1 (a tag, so no slot is ever reset); after the barrier every warp reads
      // the same decision. A slot is written again two tiles later, after every warp has passed
      // the next tile's barrier and therefore finished reading it.
      if (__any_sync(0xffffffffu, over) && lane == 0) sh.overflow[j & 1] = j + 1;
      fence_proxy_async_smem();
      tc_fence_before();
      if (!sm_sync(sh, smph)) return;
      fix = sh.overflow[j & 1] == j + 1;
    }
    if (fix) {
      if (!max_pass<NH>(a, sh, tl, pt, valid, first, smph, tid)) return;
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sh.bar(kBarPFixed));
    }
    if (warp == kIssueWarp) {
      if (fix && !wait_bar_w(sh, sh.bar(kBarPFixed), nfix & 1)) return;
      if (lane == 0) SMLA_TRACE_TILE(j, 2);
      tc_fence_after();
      mma_issue_pv<NH>(sh, tmem, j, first);
    }
    if (fix) ++nfix;

    if (!last) continue;
    // ---- epilogue of the item segment: wait for its last PV (and row sums). Every TMEM lane of
    // L holds the same row sums, so each warp derives the output factors of the heads it writes
    // from its own lanes: no step across warps (each warp moves on to the next tile as soon as
    // its own share is written; the issuing warp then issues the next tile's QK^T). Warp 0 also
    // writes the LSEs.
    if (!wait_bar_w(sh, sh.bar(kBarRowsum), j & 1)) return;
    tc_fence_after();
    if (tid == 0) SMLA_TRACE_TILE(j, 8);
    const uint32_t t = item_token(a, cur.item);
    const int h0 = item_head0(a, cur.item);
    const int hg = min(a.heads_per_group, a.H - h0);
    const int slot = a.split ? static_cast<int>(blockIdx.x - split_owner(static_cast<long long>(cur.item) *
                                                                                 a.tiles_per_item,
                                                                             a.total_tiles, a.nctas))
                             : 0;
#pragma unroll 1
    for (int c0 = 0; c0 < NH; c0 += CW) {
      if (c0 >= hg) break;
      // output factor 1 / (row sum + e^(sink - m)) of heads c0 .. c0+CW-1 (sink only for final
      // outputs; the combine applies it to split partials); 0 for an empty head. Lane i works
      // out head c0+i's factor (and warp 0 its LSE) into this warp's row of the reduction
      // area, which the max pass does not use until every warp has left its epilogue.
      float* fw = sh.red + warp * 64;
      // O^T blocks 0..3 of these heads: block 0's load is in flight while the factors are worked
      // out; for NH <= 32 two register buffers also keep each later block's load in flight while
      // the previous one is converted and stored
      float oa[CW], ob[CW];
      (void)ob;
      tmem_load_nw<CW>(tl + TC::kO + c0, oa);
      {
        float l[CW];
        tmem_load<CW>(tl + TC::kL + c0, l);
        if (tid == 0 && tr_first && c0 == 0) SMLA_TRACE_AT(248);
        // lane i takes column c0+i (every lane holds the same sums): a select tree on the lane's
        // bits, log2(CW) levels
#pragma unroll
        for (int w = CW / 2, bit = 0; w >= 1; w /= 2, ++bit) {
          const bool hi = ((lane >> bit) & 1) != 0;
#pragma unroll
          for (int i = 0; i < w; ++i) l[i] = hi ? l[2 * i + 1] : l[2 * i];
        }
        const float lsel = l[0];
        if (lane < CW) {
          const int h = c0 + lane;
          const float m = sh.m_run[h];
          float denom = lsel;
          if (!a.split && a.sink != nullptr && h < hg) denom += exp2f(a.sink[h0 + h] * 1.4426950408889634f - m);
          fw[h] = lsel > 0.f ? __frcp_rn(denom) : 0.f;
          if (warp == 0 && h < hg) {
            const float lse2 = lsel > 0.f ? m + log2f(lsel) : -INFINITY;
            if (a.split) {
              a.part_lse[(static_cast<int64_t>(slot) * a.T + t) * a.H + h0 + h] = lse2;
            } else if (a.lse != nullptr) {
              a.lse[static_cast<int64_t>(t) * a.lse_stride_t + h0 + h] = lse2 * 0.6931471805599453f;
            }
          }
        }
        __syncwarp();
      }
      // factors of head pairs, packed for the paired fp32 multiply (an empty head's factor is 0
      // and its O^T column is 0, so its outputs are 0)
      uint64_t f2[CW / 2];
#pragma unroll
      for (int i = 0; i < CW; i += 4) {
        const float4 v = *reinterpret_cast<const float4*>(fw + c0 + i);
        f2[i / 2] = pack_f32x2(v.x, v.y);
        f2[i / 2 + 1] = pack_f32x2(v.z, v.w);
      }
      if (tid == 0 && tr_first && c0 == 0) SMLA_TRACE_AT(249);
      auto emit_blocks = [&](auto&& emit) {
        if constexpr (NH <= 32) {
#pragma unroll 1
          for (int b = 0; b < 4; b += 2) {
            tmem_load_wait<CW>(oa);
            if (tid == 0 && tr_first && c0 == 0 && b == 0) SMLA_TRACE_AT(250);
            tmem_load_nw<CW>(tl + TC::kO + (b + 1) * NH + c0, ob);
            emit(oa, b);
            tmem_load_wait<CW>(ob);
            if (b + 2 < 4) tmem_load_nw<CW>(tl + TC::kO + (b + 2) * NH + c0, oa);
            emit(ob, b + 1);
          }
        } else {
          // one buffer: the second copy of the conversion code costs the larger kernels more in
          // instruction fetch than the overlap gains
#pragma unroll 1
          for (int b = 0; b < 4; ++b) {
            if (b > 0) tmem_load_nw<CW>(tl + TC::kO + b * NH + c0, oa);
            tmem_load_wait<CW>(oa);
            if (tid == 0 && tr_first && c0 == 0 && b == 0) SMLA_TRACE_AT(250);
            emit(oa, b);
          }
        }
      };
      if (a.split) {
        // partial O^T in head chunks of 8: entry (channel, 8 heads) of chunk k is 16 bytes at
        // ((slot*T + t)*nchunks + k)*512 + channel, so a warp's 32 channels are 512 contiguous
        // bytes per store
        uint4* pbase = reinterpret_cast<uint4*>(a.part_o) +
                       ((static_cast<int64_t>(slot) * a.T + t) * a.nchunks + ((h0 + c0) >> 3)) * kDv + tid;
        auto emit = [&](const float* o, int b) {
#pragma unroll
          for (int g8 = 0; g8 < CW / 8; ++g8) {
            if (c0 + 8 * g8 < hg) {
              uint32_t w4[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int i = 8 * g8 + 2 * e;
                w4[e] = mul_pack_bf16x2(o[i], o[i + 1], f2[i / 2]);
              }
              pbase[static_cast<int64_t>(g8) * kDv + 128 * b] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
            }
          }
          if (tid == 0 && tr_first && c0 == 0) SMLA_TRACE_AT(251 + (b < 2 ? b : (b == 3 ? 2 : 5)));
        };
        emit_blocks(emit);
      } else {
        // final O: thread tid holds channel 128b + tid of every head. Within each group of 8
        // lanes an 8x8 transpose of the bf16 values (three exchange stages on pairs packed two
        // to a word) gives every lane 8 consecutive channels of one head, stored as one 16-byte
        // write (rows 16-byte aligned, strides multiples of 8).
        uint16_t* obase =
            a.out + static_cast<int64_t>(t) * a.out_stride_t + static_cast<int64_t>(h0) * a.out_stride_h;
        const int64_t hstride = a.out_stride_h;
        const int k8 = lane & 7;
        auto emit = [&](const float* o, int b) {
#pragma unroll
          for (int q = 0; q < CW / 8; ++q) {
            // heads c0+8q .. c0+8q+7 of this lane's channel, as bf16 pairs (p[m] = heads 2m, 2m+1)
            uint32_t p[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) p[m] = mul_pack_bf16x2(o[8 * q + 2 * m], o[8 * q + 2 * m + 1], f2[4 * q + m]);
            // 8x8 transpose of bf16 elements across the 8 lanes of the group, in three exchange
            // stages: lane pairs k, k^4 swap whole words 2,3 <-> 0,1; k, k^2 swap words 1,3 <->
            // 0,2; k, k^1 swap the odd <-> even halves of every word (packed two to a word)
            {
              const bool up = (k8 & 4) != 0;
              const uint32_t r0 = __shfl_xor_sync(0xffffffffu, up ? p[0] : p[2], 4);
              const uint32_t r1 = __shfl_xor_sync(0xffffffffu, up ? p[1] : p[3], 4);
              if (up) {
                p[0] = r0;
                p[1] = r1;
              } else {
                p[2] = r0;
                p[3] = r1;
              }
            }
            {
              const bool up = (k8 & 2) != 0;
              const uint32_t r0 = __shfl_xor_sync(0xffffffffu, up ? p[0] : p[1], 2);
              const uint32_t r1 = __shfl_xor_sync(0xffffffffu, up ? p[2] : p[3], 2);
              if (up) {
                p[0] = r0;
                p[2] = r1;
              } else {
                p[1] = r0;
                p[3] = r1;
              }
            }
            {
              const bool up = (k8 & 1) != 0;
              const uint32_t sel = up ? 0x5410u : 0x7632u;  // the halves this lane gives away
              const uint32_t q0 = __shfl_xor_sync(0xffffffffu, __byte_perm(p[0], p[1], sel), 1);
              const uint32_t q1 = __shfl_xor_sync(0xffffffffu, __byte_perm(p[2], p[3], sel), 1);
              const uint32_t s_lo = up ? 0x3254u : 0x5410u, s_hi = up ? 0x3276u : 0x7610u;
              p[0] = __byte_perm(p[0], q0, s_lo);
              p[1] = __byte_perm(p[1], q0, s_hi);
              p[2] = __byte_perm(p[2], q1, s_lo);
              p[3] = __byte_perm(p[3], q1, s_hi);
            }
            // lane 8g+k now holds head c0+8q+k for channels 32w+8g .. 32w+8g+7
            const int h = c0 + 8 * q + k8;
            if (h < hg)
              *reinterpret_cast<uint4*>(obase + h * hstride + b * 128 + (tid & ~7)) = make_uint4(p[0], p[1], p[2], p[3]);
          }
          if (tid == 0 && tr_first && c0 == 0) SMLA_TRACE_AT(251 + (b < 2 ? b : (b == 3 ? 2 : 5)));
        };
        emit_blocks(emit);
      }
      if (tid == 0 && tr_first) SMLA_TRACE_AT(254);
    }
    tr_first = false;
    if (tid == 0) SMLA_TRACE_TILE(j, 9);
    tc_fence_before();
  }
}

template <int NH, int F0, int F1>
__global__ void __launch_bounds__(kThreads, 1) sparse_mla_kernel(const __grid_constant__ AttnArgs a) {
  using L = Smem<NH>;
  extern __shared__ uint8_t smem_raw[];
  if (threadIdx.x == 0) SMLA_TRACE_AT(0);
  // 1 KB alignment computed on the 32-bit shared address (the MMA descriptors derive from it)
  const uint32_t sraw = smem_u32(smem_raw);
  const uint32_t s0 = (sraw + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (s0 - sraw);
  Shared sh;
  sh.base = base;
  sh.tile = s0;
  sh.q = s0 + L::kQOff;
  sh.red = reinterpret_cast<float*>(base + L::kRedOff);
  sh.m_run = reinterpret_cast<float*>(base + L::kMOff);
  sh.m_use = reinterpret_cast<float*>(base + L::kMUseOff);
  sh.thr = reinterpret_cast<float*>(base + L::kThrOff);
  sh.alpha = reinterpret_cast<float*>(base + L::kAlphaOff);
  sh.fin = reinterpret_cast<float*>(base + L::kFinOff);
  sh.rowoff = reinterpret_cast<int32_t*>(base + L::kRowOff);
  sh.res = s0 + L::kResOff;
  sh.resp = reinterpret_cast<int32_t*>(base + L::kResOff);
  sh.bars = s0 + L::kBarOff;
  sh.tmem_slot = reinterpret_cast<uint32_t*>(base + L::kMiscOff);
  sh.abort_flag = reinterpret_cast<volatile int*>(base + L::kMiscOff + 4);
  sh.rescale_flag = reinterpret_cast<volatile int*>(base + L::kMiscOff + 8);
  sh.overflow = reinterpret_cast<volatile int*>(base + L::kMiscOff + 16);

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
    mbar_init(sh.bar(kBarFullA), kLdWarps);
    mbar_init(sh.bar(kBarFullB), kLdWarps);
    mbar_init(sh.bar(kBarFullR), kLdWarps);
    mbar_init(sh.bar(kBarRowsum), 1);
    mbar_init(sh.bar(kBarSFull), 1);
    mbar_init(sh.bar(kBarSm), kSmWarps * 32);
    mbar_init(sh.bar(kBarPFixed), kSmWarps);
    for (int i = 0; i < 4; ++i) mbar_init(sh.bar(kBarPvDone + i), 1);
    for (int i = 0; i < 4; ++i) mbar_init(sh.bar(kBarRow + i), kIssueWarp);
    *sh.abort_flag = 0;
    *sh.rescale_flag = 0;
    sh.overflow[0] = sh.overflow[1] = 0;
    fence_mbar_init();
  }
  fence_proxy_async_smem();
  if (warp == 0) {
    tmem_alloc(smem_u32(sh.tmem_slot), TmemCols<NH>::kAlloc);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sh.tmem_slot;
  // launched as a programmatic dependent of the previous kernel on the stream: the set-up above
  // overlaps its tail; nothing in global memory is read or written before it has completed
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) SMLA_TRACE_AT(1);

  if (warp < kSmWarps) {
    softmax_role<NH>(a, sh, tmem, lo, n);
  } else {
    loader_role<NH, F0, F1>(a, sh, lo, n);
  }
  cp_async_wait_all();
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, TmemCols<NH>::kAlloc);
  }
  if (threadIdx.x == 0) SMLA_TRACE_AT(2);
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Split-K combine, one CTA per (token, 32-head chunk, part of the 512 channels). Each thread
// owns an 8-head subgroup and 4 channels of a 256-channel part (2 of a 128-channel part); it
// issues the loads of its first four partial slots before anything else, so they are in
// flight while threads 0..31 merge the
// heads' partial base-2 LSEs into the final LSE, the sink factor and the per-slot weights
// 2^(lse_s - lse) (shared memory). The weighted sums are transposed through shared memory and
// written as bf16 O with 16-byte stores.
constexpr int kCombineThreads = 256;
constexpr int kCombineHeads = 32;
constexpr int kCombineSlots = 4;  // partial slots loaded per round
// The 512 channels are split over kParts CTAs: 2 when T x head chunks already fill the GPU, 4
// when they leave SMs idle (more CTAs, half the loads per thread, for small T).
constexpr int kCombineFewCtas = 128;

__device__ __forceinline__ void item_slots(const AttnArgs& a, int t, int h, int& c0, int& ns) {
  const long long item = static_cast<long long>(t) * a.groups + h / a.heads_per_group;
  const long long x0 = item * a.tiles_per_item;
  const long long x1 = x0 + a.tiles_per_item - 1;
  if ((a.total_tiles + 1) * a.nctas < (1ll << 32)) {  // 32-bit divisions (every realistic size)
    const uint32_t tot = static_cast<uint32_t>(a.total_tiles), nc = static_cast<uint32_t>(a.nctas);
    c0 = static_cast<int>((static_cast<uint32_t>(x0 + 1) * nc - 1u) / tot);
    ns = static_cast<int>((static_cast<uint32_t>(x1 + 1) * nc - 1u) / tot) - c0 + 1;
  } else {
    c0 = static_cast<int>(split_owner(x0, a.total_tiles, a.nctas));
    ns = static_cast<int>(split_owner(x1, a.total_tiles, a.nctas)) - c0 + 1;
  }
}

template <int kParts>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const __grid_constant__ AttnArgs a) {
  constexpr int kCombineCh = kDv / kParts;  // channels per CTA
  extern __shared__ float wts[];  // [max_slots][kCombineHeads]
  __shared__ float fac[kCombineHeads];
  __shared__ __align__(16) uint16_t ot[kCombineHeads][kCombineCh];
  // launched as a programmatic dependent of the attention kernel: wait for its partials. The
  // next kernel on the stream may be scheduled at once (it waits for this grid's completion
  // before its own first global access), so its set-up overlaps this grid's tail.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int t = blockIdx.x;
  const int hbase = blockIdx.y * kCombineHeads;
  const int cbase = blockIdx.z * kCombineCh;
  const int tid = threadIdx.x;
  const int H = a.H;

  // 16-byte chunk (channel cbase + tid/4 + 64q, heads hbase + 8g .. +7) of every slot's
  // partial block: four consecutive threads read one channel's 64 contiguous bytes
  constexpr int kChunks = kCombineCh * (kCombineHeads / 8) / kCombineThreads;  // 4 or 2
  constexpr int kChStep = kCombineThreads / 4;
  const int g = tid & 3;
  int ns = 0;  // slots of this thread's 8 heads (heads_per_group is a multiple of 8)
  if (hbase + 8 * g < H) {
    int c0;
    item_slots(a, t, hbase + 8 * g, c0, ns);
  }
  // partial entry (channel, 8 heads) of head chunk k: 16 bytes at ((slot*T + t)*nchunks + k)*512 + channel
  const int64_t sstride = static_cast<int64_t>(a.T) * a.nchunks * kDv;  // in 16-byte entries
  const uint4* col = reinterpret_cast<const uint4*>(a.part_o) +
                     (static_cast<int64_t>(t) * a.nchunks + ((hbase >> 3) + g)) * kDv + cbase + (tid >> 2);
  uint4 v[kCombineSlots][kChunks];
  auto issue = [&](int s0) {
#pragma unroll
    for (int s = 0; s < kCombineSlots; ++s)
#pragma unroll
      for (int q = 0; q < kChunks; ++q)
        v[s][q] = s0 + s < ns ? col[(s0 + s) * sstride + q * kChStep] : make_uint4(0, 0, 0, 0);
  };
  issue(0);

  if (tid < kCombineHeads) {
    const int h = hbase + tid;
    int nh = 0;
    float f = 0.f;
    if (h < H) {
      int c0;
      item_slots(a, t, h, c0, nh);
      const float* lp = a.part_lse + static_cast<int64_t>(t) * H + h;
      const int64_t lstride = static_cast<int64_t>(a.T) * H;
      // the sink and the first slots' partial LSEs are loaded together (one round trip), the
      // LSEs go to shared memory, and the max, the sum and the weights are computed from there
      const float sk = a.sink != nullptr ? a.sink[h] : 0.f;
      float l0[kCombineSlots];
#pragma unroll
      for (int s = 0; s < kCombineSlots; ++s) l0[s] = s < nh ? lp[s * lstride] : 0.f;
      for (int s = kCombineSlots; s < nh; ++s) wts[s * kCombineHeads + tid] = lp[s * lstride];
#pragma unroll
      for (int s = 0; s < kCombineSlots; ++s)
        if (s < nh) wts[s * kCombineHeads + tid] = l0[s];
      float M = -INFINITY;
      for (int s = 0; s < nh; ++s) M = fmaxf(M, wts[s * kCombineHeads + tid]);
      float L2 = -INFINITY;
      if (M != -INFINITY) {
        float W = 0.f;
        for (int s = 0; s < nh; ++s) W += exp2f(wts[s * kCombineHeads + tid] - M);
        L2 = M + log2f(W);
      }
      for (int s = 0; s < nh; ++s)
        wts[s * kCombineHeads + tid] = L2 == -INFINITY ? 0.f : exp2f(wts[s * kCombineHeads + tid] - L2);
      if (L2 != -INFINITY) f = a.sink != nullptr ? 1.f / (1.f + exp2f(sk * 1.4426950408889634f - L2)) : 1.f;
      if (a.lse != nullptr && blockIdx.z == 0)
        a.lse[static_cast<int64_t>(t) * a.lse_stride_t + h] = L2 * 0.6931471805599453f;
    }
    for (int s = nh; s < a.max_slots; ++s) wts[s * kCombineHeads + tid] = 0.f;
    fac[tid] = f;
  }
  __syncthreads();

  float acc[kChunks][8];
#pragma unroll
  for (int q = 0; q < kChunks; ++q)
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[q][i] = 0.f;
#pragma unroll 1
  for (int s0 = 0; s0 < ns; s0 += kCombineSlots) {
    if (s0 > 0) issue(s0);
#pragma unroll
    for (int s = 0; s < kCombineSlots; ++s) {
      if (s0 + s >= ns) break;
      float w[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) w[i] = wts[(s0 + s) * kCombineHeads + 8 * g + i];
#pragma unroll
      for (int q = 0; q < kChunks; ++q) {
        const uint32_t wv[4] = {v[s][q].x, v[s][q].y, v[s][q].z, v[s][q].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          // a slot past one head's own range (weight 0) may hold unrelated data: select, not
          // multiply
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv[e]));
          acc[q][2 * e] += w[2 * e] != 0.f ? w[2 * e] * f.x : 0.f;
          acc[q][2 * e + 1] += w[2 * e + 1] != 0.f ? w[2 * e + 1] * f.y : 0.f;
        }
      }
    }
  }
  // transpose through shared memory (bf16 [32 heads][256 channels]), then coalesced stores
#pragma unroll
  for (int q = 0; q < kChunks; ++q) {
    const int c = (tid >> 2) + q * kChStep;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const __nv_bfloat16 b = __float2bfloat16_rn(acc[q][i] * fac[8 * g + i]);
      ot[8 * g + i][c] = *reinterpret_cast<const uint16_t*>(&b);
    }
  }
  __syncthreads();
  uint16_t* obase = a.out + static_cast<int64_t>(t) * a.out_stride_t + cbase;
#pragma unroll
  for (int e = tid; e < kCombineHeads * (kCombineCh / 8); e += kCombineThreads) {
    const int hh = e / (kCombineCh / 8), c8 = (e - hh * (kCombineCh / 8)) * 8;
    if (hbase + hh < H)
      *reinterpret_cast<uint4*>(obase + static_cast<int64_t>(hbase + hh) * a.out_stride_h + c8) =
          *reinterpret_cast<const uint4*>(&ot[hh][c8]);
  }
}

// Dynamic shared memory above 48 KB is enabled once per kernel and device (a bit per device in
// `done`, for up to 64 devices; beyond that it is set on every call). `bytes_done` remembers the
// largest size enabled so far for kernels whose request varies.
template <typename K>
cudaError_t enable_smem(K kernel, int bytes, std::atomic<uint64_t>& done, std::atomic<int>& bytes_done,
                        const char* what) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 64;
  const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0 && bytes <= bytes_done.load()) return cudaSuccess;
  const int want = bytes > bytes_done.load() ? bytes : bytes_done.load();
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, want);
  if (e != cudaSuccess) {
    note_cuda_error(e, what);
    return e;
  }
  int prev = bytes_done.load();
  while (want > prev && !bytes_done.compare_exchange_weak(prev, want)) {
  }
  if (bit != 0) done.fetch_or(bit, std::memory_order_acq_rel);
  return cudaSuccess;
}

// one record for the combine kernel, which every attention instantiation launches
std::atomic<uint64_t> g_combine_attr_done[2] = {};
std::atomic<int> g_combine_attr_bytes[2] = {};

template <int NH, int F0, int F1>
cudaError_t launch_nh(const AttnArgs& a, const Plan& plan, cudaStream_t stream, cudaEvent_t ev0, cudaEvent_t ev1) {
  static std::atomic<uint64_t> attr_done{0};
  static std::atomic<int> attr_bytes{0};
  const int smem = Smem<NH>::kAlloc;
  cudaError_t e = enable_smem(sparse_mla_kernel<NH, F0, F1>, smem, attr_done, attr_bytes,
                              "cudaFuncSetAttribute(sparse_mla_kernel, max dynamic shared memory)");
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute pdl;
  pdl.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  pdl.val.programmaticStreamSerializationAllowed = 1;
  if (ev0) cudaEventRecord(ev0, stream);
  {
    // programmatic dependent launch: the grid is scheduled while the previous kernel on the
    // stream drains; the kernel waits for it (griddepcontrol.wait) before touching memory
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(plan.nctas));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = stream;
    cfg.attrs = &pdl;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, sparse_mla_kernel<NH, F0, F1>, a);
    if (e == cudaSuccess) e = cudaGetLastError();
  }
  if (ev1) cudaEventRecord(ev1, stream);
  if (e != cudaSuccess) {
    note_cuda_error(e, "launch of sparse_mla_kernel");
    return e;
  }
  if (plan.split) {
    // programmatic dependent launch: the combine grid is scheduled while the attention kernel
    // drains and waits (griddepcontrol.wait) for its results
    const unsigned chunks = static_cast<unsigned>((a.H + kCombineHeads - 1) / kCombineHeads);
    const bool few = static_cast<long long>(a.T) * chunks * 2 < kCombineFewCtas;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.T), chunks, few ? 4 : 2);
    cfg.blockDim = dim3(kCombineThreads);
    cfg.dynamicSmemBytes = static_cast<size_t>(a.max_slots) * kCombineHeads * sizeof(float);
    e = few ? enable_smem(combine_kernel<4>, static_cast<int>(cfg.dynamicSmemBytes), g_combine_attr_done[1],
                          g_combine_attr_bytes[1], "cudaFuncSetAttribute(combine_kernel, max dynamic shared memory)")
            : enable_smem(combine_kernel<2>, static_cast<int>(cfg.dynamicSmemBytes), g_combine_attr_done[0],
                          g_combine_attr_bytes[0], "cudaFuncSetAttribute(combine_kernel, max dynamic shared memory)");
    if (e != cudaSuccess) return e;
    cfg.stream = stream;
    cfg.attrs = &pdl;
    cfg.numAttrs = 1;
    e = few ? cudaLaunchKernelEx(&cfg, combine_kernel<4>, a) : cudaLaunchKernelEx(&cfg, combine_kernel<2>, a);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) note_cuda_error(e, "launch of combine_kernel");
  }
  return e;
}

template <int NH>
cudaError_t launch_fmt(const AttnArgs& a, const Plan& plan, cudaStream_t stream, cudaEvent_t ev0, cudaEvent_t ev1) {
  const int f0 = a.set[0].format;
  const int f1 = a.nsets > 1 ? a.set[1].format : f0;
  switch (f0 * 2 + f1) {
    case 0: return launch_nh<NH, 0, 0>(a, plan, stream, ev0, ev1);
    case 1: return launch_nh<NH, 0, 1>(a, plan, stream, ev0, ev1);
    case 2: return launch_nh<NH, 1, 0>(a, plan, stream, ev0, ev1);
    default: return launch_nh<NH, 1, 1>(a, plan, stream, ev0, ev1);
  }
}

}  // namespace

cudaError_t launch_attention(const AttnArgs& args, const Plan& plan, cudaStream_t stream, cudaEvent_t ev0,
                             cudaEvent_t ev1) {
  switch (plan.nh) {
    case 16: return launch_fmt<16>(args, plan, stream, ev0, ev1);
    case 32: return launch_fmt<32>(args, plan, stream, ev0, ev1);
    case 64: return launch_fmt<64>(args, plan, stream, ev0, ev1);
    default: return cudaErrorInvalidValue;
  }
}

#ifdef SMLA_TRACE
extern "C" int smla_trace_read(void* host, size_t bytes) {
  return static_cast<int>(cudaMemcpyFromSymbol(host, g_trace, bytes < sizeof(g_trace) ? bytes : sizeof(g_trace)));
}
#endif

cudaError_t read_and_clear_device_error(int* code) {
  int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(code, g_device_error, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
}

}  // namespace smla
