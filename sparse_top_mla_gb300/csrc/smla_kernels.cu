// Sparse top-k MLA attention kernels for GB300 (sm_103a).
//
// One CTA handles one (query token t, head group g, split s). It walks its share of the
// token's index list in tiles of 128 gathered rows:
//   1. index resolve  — each thread turns one index into a cache row address (or a mask),
//   2. gather         — the 128 rows (576 channels) land in shared memory as a bf16 tile in
//                       the 128-byte-swizzled layout the tensor core reads; FP8 rows are
//                       dequantised on the way (e4m3 * per-128-channel scale -> bf16),
//   3. S^T = K_tile Q^T on tcgen05 (M = 128 gathered rows, N = heads of the group, K = 576),
//      accumulated in TMEM,
//   4. online softmax with the sink handled at the end; running max per head is kept in
//      shared memory and only raised when a tile exceeds it by more than 2^8 (lazy rescale),
//   5. O^T += V^T P^T on tcgen05 (M = 128 value channels x 4 blocks, N = heads, K = 128 rows),
//      accumulated in TMEM; V is the first 512 channels of the same gathered tile.
// The epilogue either writes the final O (bf16) and LSE, or — for the split-K decode
// schedule — a normalised fp32 partial O and a base-2 partial LSE that the combine kernel
// merges with warp shuffles.
//
// Head-as-N ("swapAB") orientation: the gathered rows fill the 128-row MMA M dimension and
// the heads of the group are N (16, 32 or 64), so any head count runs without padding the
// problem: unused N columns are MMA-internal zeros, never memory traffic or extra outputs.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "smla_internal.h"
#include "smla_ptx.cuh"

namespace smla {

__device__ int g_device_error;

namespace {

using namespace ptx;

constexpr int kThreads = 128;
constexpr int kKBlocks = 9;                    // 576 channels / 64 channels per 128-byte row
constexpr int kTileBlockBytes = kTile * 128;   // one 64-channel block of the tile: 16 KB
constexpr int kTileBytes = kKBlocks * kTileBlockBytes;
constexpr float kLazyRescaleLog2 = 8.0f;       // raise the running max only past 2^8
constexpr long long kSpinLimit = 1LL << 26;    // bounded waits
constexpr int kErrTimeout = 1;

template <int NH>
struct Smem {
  static constexpr int kQBytes = kKBlocks * NH * 128;
  static constexpr int kTileOff = 0;
  static constexpr int kQOff = kTileBytes;
  static constexpr int kRowOff = kQOff + kQBytes;          // int64 [128]
  static constexpr int kRedOff = kRowOff + kTile * 8;      // float [4][64]
  static constexpr int kMOff = kRedOff + 4 * 64 * 4;       // float [64] running max (base 2)
  static constexpr int kAlphaOff = kMOff + 64 * 4;         // float [64]
  static constexpr int kFinOff = kAlphaOff + 64 * 4;       // float [64] per-head output factor
  static constexpr int kMiscOff = kFinOff + 64 * 4;        // bars, tmem base, flags
  static constexpr int kBytes = kMiscOff + 64;
  static constexpr int kAlloc = kBytes + 1024;             // + alignment slack
};

template <int NH>
struct TmemCols {
  static constexpr int kS = 0;
  static constexpr int kO = 64;  // O^T block b at kO + b*NH
  static constexpr int kUsed = kO + 4 * NH;
  static constexpr int kAlloc = kUsed <= 128 ? 128 : (kUsed <= 256 ? 256 : 512);
};

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity) {
  for (long long it = 0; it < kSpinLimit; ++it)
    if (mbar_try_wait(bar, parity)) return true;
  atomicExch(&g_device_error, kErrTimeout);
  return false;
}

// Column reduction across the 32 lanes of a warp for N values per lane ("transpose
// reduce"): each step halves the values a lane holds while exchanging the other half
// with its partner, so the warp does N-1 shuffles instead of 5N. Afterwards lane l holds
//   N = 64: heads 2l, 2l+1 in v[0], v[1];  N = 32: head l in v[0];  N = 16: head l/2 in v[0].
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

template <int N, bool kMax>
__device__ __forceinline__ void warp_col_reduce(float* v, int lane) {
  col_reduce_step<N, 16, kMax>(v, lane);
}

// Store the per-warp column results into red[warp][head].
template <int N>
__device__ __forceinline__ void store_col_result(float* red_w, const float* v, int lane) {
  if (N == 64) {
    red_w[2 * lane] = v[0];
    red_w[2 * lane + 1] = v[1];
  } else if (N == 32) {
    red_w[lane] = v[0];
  } else {
    if ((lane & 1) == 0) red_w[lane >> 1] = v[0];
  }
}

// 16 e4m3 bytes * scale -> 16 bf16 (two 16-byte chunks).
__device__ __forceinline__ void dequant16(const uint4 raw, float scale, uint4& lo, uint4& hi) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  uint32_t outw[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const __nv_fp8x2_storage_t pair = static_cast<__nv_fp8x2_storage_t>((w[i] >> (16 * half)) & 0xFFFFu);
      const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&hr));
      const __nv_bfloat162 b = __floats2bfloat162_rn(f.x * scale, f.y * scale);
      outw[2 * i + half] = *reinterpret_cast<const uint32_t*>(&b);
    }
  }
  lo = make_uint4(outw[0], outw[1], outw[2], outw[3]);
  hi = make_uint4(outw[4], outw[5], outw[6], outw[7]);
}

__device__ __forceinline__ uint32_t swz(int row, int chunk) {  // 128-byte swizzle inside a 1 KB atom
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

template <int NH>
__global__ void __launch_bounds__(kThreads, 1) sparse_mla_kernel(const AttnArgs args) {
  using L = Smem<NH>;
  using TC = TmemCols<NH>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t s_tile = smem_u32(smem + L::kTileOff);
  const uint32_t s_q = smem_u32(smem + L::kQOff);
  const uint32_t s_pt = s_tile + 8 * kTileBlockBytes;  // P^T lives in the rope block after QK^T
  int64_t* rowoff = reinterpret_cast<int64_t*>(smem + L::kRowOff);
  float* red = reinterpret_cast<float*>(smem + L::kRedOff);
  float* m_run = reinterpret_cast<float*>(smem + L::kMOff);
  float* alpha = reinterpret_cast<float*>(smem + L::kAlphaOff);
  float* fin = reinterpret_cast<float*>(smem + L::kFinOff);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kMiscOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff + 16);
  int* flags = reinterpret_cast<int*>(smem + L::kMiscOff + 32);
  const uint32_t bar_qk = smem_u32(&bars[0]);
  const uint32_t bar_pv = smem_u32(&bars[1]);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;

  // ---- work decomposition: blockIdx.x = (t * groups + g) * splits + s
  const int s_idx = blockIdx.x % args.splits;
  const int tg = blockIdx.x / args.splits;
  const int g = tg % args.groups;
  const int t = tg / args.groups;
  const int h0 = g * args.heads_per_group;
  const int hg = min(args.heads_per_group, args.H - h0);
  const int tile_begin = s_idx * args.tiles_per_split;
  const int tile_end = min(args.total_tiles, tile_begin + args.tiles_per_split);
  const int seq = args.token_seq[t];
  const bool seq_ok = seq >= 0 && seq < args.num_seqs;

  // ---- setup: barriers, TMEM, Q tile (zero rows for heads past the group)
  if (tid == 0) {
    mbar_init(bar_qk, 1);
    mbar_init(bar_pv, 1);
    fence_mbar_init();
    flags[0] = 0;
    flags[1] = 0;
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), TC::kAlloc);
    tmem_relinquish();
  }
  {
    const uint16_t* qbase = args.q + static_cast<int64_t>(t) * args.q_stride_t;
    for (int e = tid; e < NH * 72; e += kThreads) {
      const int n = e / 72;
      const int c = e - n * 72;
      const int kb = c >> 3;
      const int ch = c & 7;
      const bool live = n < hg;
      const uint16_t* src = qbase + (live ? static_cast<int64_t>(h0 + n) * args.q_stride_h + kb * 64 + ch * 8 : 0);
      cp_async16(s_q + kb * NH * 128 + swz(n, ch), src, live ? 16u : 0u);
    }
    cp_async_commit();
  }
  if (tid < 64) m_run[tid] = -INFINITY;
  float l_part[NH];
#pragma unroll
  for (int i = 0; i < NH; ++i) l_part[i] = 0.f;

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  constexpr uint32_t idesc_qk = idesc_bf16(128, NH, 0, 0);
  constexpr uint32_t idesc_pv = idesc_bf16(128, NH, 1, 1);

  uint32_t phase_qk = 0, phase_pv = 0;
  bool first_pv = true;
  bool failed = false;

  for (int u = tile_begin; u < tile_end && !failed; ++u) {
    const int set_id = (args.nsets > 1 && u >= args.set[0].ntiles) ? 1 : 0;
    const KvSetDev& S = args.set[set_id];
    const int lt = u - (set_id ? args.set[0].ntiles : 0);

    // ---- 1. index resolve: thread tid owns gathered row tid of this tile
    bool valid = false;
    int64_t off = 0;
    {
      const int j = lt * kTile + tid;
      int width = S.topk;
      if (S.topk_length != nullptr) width = min(width, max(0, S.topk_length[t]));
      if (seq_ok && j < width) {
        const int32_t i = S.indices[static_cast<int64_t>(t) * S.idx_stride + j];
        if (i >= 0 && i < S.seq_lens[seq]) {
          const int32_t lp = i >> 6;
          if (lp < S.bt_stride) {
            const int32_t p = S.block_table[static_cast<int64_t>(seq) * S.bt_stride + lp];
            if (p >= 0 && p < S.num_pages) {
              valid = true;
              off = static_cast<int64_t>(p) * S.page_stride + static_cast<int64_t>(i & 63) * S.row_stride;
            }
          }
        }
      }
      rowoff[tid] = valid ? off : -1;
    }
    __syncthreads();

    // ---- 2. gather into the swizzled bf16 tile (masked rows become zeros)
    if (S.format == 0) {
#pragma unroll 2
      for (int it = 0; it < 8; ++it) {
        const int r = warp * 32 + it * 4 + (lane >> 3);
        const int c = lane & 7;
        const int64_t ro = rowoff[r];
        const uint8_t* src = S.cache + (ro >= 0 ? ro : 0) + c * 16;
        const uint32_t nbytes = ro >= 0 ? 16u : 0u;
#pragma unroll
        for (int kb = 0; kb < kKBlocks; ++kb)
          cp_async16(s_tile + kb * kTileBlockBytes + swz(r, c), src + kb * 128, nbytes);
      }
      cp_async_commit();
    } else {
      // fp8 row: lane l converts latent bytes [16l, 16l+16) with scale l/8; lanes 0-7 copy the rope
#pragma unroll 1
      for (int it = 0; it < 32; it += 4) {
        uint4 lat[4], rope[4];
        float sc[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int r = warp * 32 + it + k;
          const int64_t ro = rowoff[r];
          lat[k] = make_uint4(0, 0, 0, 0);
          rope[k] = make_uint4(0, 0, 0, 0);
          sc[k] = 0.f;
          if (ro >= 0) {
            const uint8_t* row = S.cache + ro;
            lat[k] = ldg_nc_v4(row + lane * 16);
            sc[k] = __ldg(reinterpret_cast<const float*>(row + 512) + (lane >> 3));
            if (lane < 8) rope[k] = ldg_nc_v4(row + 528 + lane * 16);
          }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int r = warp * 32 + it + k;
          uint4 lo, hi;
          dequant16(lat[k], sc[k], lo, hi);
          const int kb = lane >> 2;
          const int c0 = (lane & 3) * 2;
          sts_v4(s_tile + kb * kTileBlockBytes + swz(r, c0), lo);
          sts_v4(s_tile + kb * kTileBlockBytes + swz(r, c0 + 1), hi);
          if (lane < 8) sts_v4(s_tile + 8 * kTileBlockBytes + swz(r, lane), rope[k]);
        }
      }
    }
    cp_async_wait_all();
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- 3. S^T[128 x NH] = K_tile[128 x 576] . Q^T
    if (tid == 0) {
      tc_fence_after();
#pragma unroll 1
      for (int kb = 0; kb < kKBlocks; ++kb) {
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t a = smem_desc(s_tile + kb * kTileBlockBytes + ks * 32, 16, 1024, kSwizzle128B);
          const uint64_t b = smem_desc(s_q + kb * NH * 128 + ks * 32, 16, 1024, kSwizzle128B);
          mma_bf16_ss(tmem + TC::kS, a, b, idesc_qk, (kb | ks) != 0);
        }
      }
      mma_commit(bar_qk);
    }
    __syncwarp();
    const bool ok_qk = wait_bar(bar_qk, phase_qk);
    phase_qk ^= 1;
    tc_fence_after();
    if (__syncthreads_or(!ok_qk)) {
      failed = true;
      break;
    }

    // ---- 4. softmax (base 2); thread tid = gathered row tid = TMEM lane tid
    float s[NH];
#pragma unroll
    for (int c = 0; c < NH; c += 16) tmem_ld16(tmem + lane_base + TC::kS + c, s + c);
#pragma unroll
    for (int h = 0; h < NH; ++h) s[h] = valid ? s[h] * args.scale_log2 : -INFINITY;
    warp_col_reduce<NH, true>(s, lane);  // destroys s; S is re-read from TMEM below
    store_col_result<NH>(red + warp * 64, s, lane);
    __syncthreads();
    if (warp == 0) {
      bool raised = false;
      for (int h = lane; h < NH; h += 32) {
        const float tmax = fmaxf(fmaxf(red[h], red[64 + h]), fmaxf(red[128 + h], red[192 + h]));
        const float mo = m_run[h];
        float a = 1.f;
        if (tmax > mo + kLazyRescaleLog2) {
          a = (mo == -INFINITY) ? 0.f : ex2(mo - tmax);
          m_run[h] = tmax;
          raised = true;
        }
        alpha[h] = a;
      }
      raised = __any_sync(0xffffffffu, raised);
      if (lane == 0) flags[0] = raised ? 1 : 0;
    }
    __syncthreads();
    const bool rescale = flags[0] != 0;
#pragma unroll
    for (int c = 0; c < NH; c += 16) tmem_ld16(tmem + lane_base + TC::kS + c, s + c);
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      const float mh = m_run[h];
      const float x = valid ? s[h] * args.scale_log2 : -INFINITY;
      const float p = ex2(x - (mh == -INFINITY ? 0.f : mh));
      if (rescale) l_part[h] *= alpha[h];
      l_part[h] += p;
      s[h] = p;
    }
    // P^T (bf16) in the no-swizzle MN-major layout: [head/8][row/8][row%8][head%8]
#pragma unroll
    for (int a8 = 0; a8 < NH / 8; ++a8) {
      uint32_t w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(s[a8 * 8 + 2 * k], s[a8 * 8 + 2 * k + 1]);
        w[k] = *reinterpret_cast<const uint32_t*>(&b);
      }
      sts_v4(s_pt + a8 * 2048 + (tid >> 3) * 128 + (tid & 7) * 16, make_uint4(w[0], w[1], w[2], w[3]));
    }
    // O^T *= alpha (only when a running max moved and O already holds earlier tiles)
    if (rescale && !first_pv) {
#pragma unroll 1
      for (int b = 0; b < 4; ++b) {
#pragma unroll
        for (int c = 0; c < NH; c += 16) {
          float o[16];
          const uint32_t addr = tmem + lane_base + TC::kO + b * NH + c;
          tmem_ld16(addr, o);
#pragma unroll
          for (int i = 0; i < 16; ++i) o[i] *= alpha[c + i];
          tmem_st16(addr, o);
        }
      }
      tmem_st_wait();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- 5. O^T[512 x NH] += V^T[512 x 128] . P^T[128 x NH]
    if (tid == 0) {
      tc_fence_after();
#pragma unroll 1
      for (int b = 0; b < 4; ++b) {
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t a = smem_desc(s_tile + 2 * b * kTileBlockBytes + ks * 2048, kTileBlockBytes, 1024, kSwizzle128B);
          const uint64_t bd = smem_desc(s_pt + ks * 256, 128, 2048, kSwizzleNone);
          mma_bf16_ss(tmem + TC::kO + b * NH, a, bd, idesc_pv, (first_pv && ks == 0) ? 0u : 1u);
        }
      }
      mma_commit(bar_pv);
    }
    __syncwarp();
    first_pv = false;
    const bool ok_pv = wait_bar(bar_pv, phase_pv);
    phase_pv ^= 1;
    tc_fence_after();
    if (__syncthreads_or(!ok_pv)) {
      failed = true;
      break;
    }
  }

  // ---- epilogue
  if (!failed) {
    // row sums: reduce l_part over the 128 rows
    warp_col_reduce<NH, false>(l_part, lane);
    store_col_result<NH>(red + warp * 64, l_part, lane);
    __syncthreads();
    const bool partial = args.part_o != nullptr;
    if (tid < NH) {
      const int h = tid;
      const float l = red[h] + red[64 + h] + red[128 + h] + red[192 + h];
      const float m = m_run[h];
      float factor = 0.f;
      float lse2 = -INFINITY;
      if (l > 0.f) {
        lse2 = m + log2f(l);
        float denom = l;
        if (!partial && args.sink != nullptr && h < hg) denom += exp2f(args.sink[h0 + h] * 1.4426950408889634f - m);
        factor = 1.f / denom;
      }
      fin[h] = factor;
      if (h < hg) {
        if (partial) {
          args.part_lse[(static_cast<int64_t>(s_idx) * args.T + t) * args.H + h0 + h] = lse2;
        } else if (args.lse != nullptr) {
          args.lse[static_cast<int64_t>(t) * args.lse_stride_t + h0 + h] = lse2 * 0.6931471805599453f;
        }
      }
    }
    __syncthreads();
    // O^T (TMEM) -> scaled rows in shared memory (reusing the tile) -> global
    if (partial) {
      float* stage = reinterpret_cast<float*>(smem + L::kTileOff);  // [NH][512] fp32
#pragma unroll 1
      for (int b = 0; b < 4; ++b) {
#pragma unroll
        for (int c = 0; c < NH; c += 16) {
          float o[16];
          tmem_ld16(tmem + lane_base + TC::kO + b * NH + c, o);
#pragma unroll
          for (int i = 0; i < 16; ++i) stage[(c + i) * kDv + b * 128 + tid] = fin[c + i] != 0.f ? o[i] * fin[c + i] : 0.f;
        }
      }
      __syncthreads();
      float* dst = args.part_o + ((static_cast<int64_t>(s_idx) * args.T + t) * args.H + h0) * kDv;
      const uint4* src4 = reinterpret_cast<const uint4*>(stage);
      uint4* dst4 = reinterpret_cast<uint4*>(dst);
      for (int e = tid; e < hg * (kDv / 4); e += kThreads) dst4[e] = src4[e];
    } else {
      __nv_bfloat16* stage = reinterpret_cast<__nv_bfloat16*>(smem + L::kTileOff);  // [NH][512] bf16
#pragma unroll 1
      for (int b = 0; b < 4; ++b) {
#pragma unroll
        for (int c = 0; c < NH; c += 16) {
          float o[16];
          tmem_ld16(tmem + lane_base + TC::kO + b * NH + c, o);
#pragma unroll
          for (int i = 0; i < 16; ++i) stage[(c + i) * kDv + b * 128 + tid] = __float2bfloat16_rn(fin[c + i] != 0.f ? o[i] * fin[c + i] : 0.f);
        }
      }
      __syncthreads();
      const uint4* src4 = reinterpret_cast<const uint4*>(stage);
      uint16_t* obase = args.out + static_cast<int64_t>(t) * args.out_stride_t;
      for (int e = tid; e < hg * (kDv / 8); e += kThreads) {
        const int h = e / (kDv / 8);
        const int c8 = e - h * (kDv / 8);
        *reinterpret_cast<uint4*>(obase + static_cast<int64_t>(h0 + h) * args.out_stride_h + c8 * 8) = src4[e];
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, TC::kAlloc);
}

// Split-K combine: one warp per (token, head). Lanes hold the splits' base-2 LSEs; the
// max and the sum of weights are warp-shuffle reductions; each lane then accumulates 16 of
// the 512 channels over the splits, applies the sink and writes bf16 O and natural-log LSE.
__global__ void __launch_bounds__(256) combine_kernel(const AttnArgs args) {
  const int warp_global = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (warp_global >= args.T * args.H) return;
  const int t = warp_global / args.H;
  const int h = warp_global - t * args.H;
  const int S = args.splits;
  float M = -INFINITY;
  for (int s = lane; s < S; s += 32) M = fmaxf(M, args.part_lse[(static_cast<int64_t>(s) * args.T + t) * args.H + h]);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  uint16_t* orow = args.out + static_cast<int64_t>(t) * args.out_stride_t + static_cast<int64_t>(h) * args.out_stride_h;
  if (M == -INFINITY) {
    reinterpret_cast<uint4*>(orow + lane * 16)[0] = make_uint4(0, 0, 0, 0);
    reinterpret_cast<uint4*>(orow + lane * 16)[1] = make_uint4(0, 0, 0, 0);
    if (lane == 0 && args.lse != nullptr) args.lse[static_cast<int64_t>(t) * args.lse_stride_t + h] = -INFINITY;
    return;
  }
  float W = 0.f;
  for (int s = lane; s < S; s += 32) W += exp2f(args.part_lse[(static_cast<int64_t>(s) * args.T + t) * args.H + h] - M);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) W += __shfl_xor_sync(0xffffffffu, W, off);
  const float L2 = M + log2f(W);
  float acc[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) acc[i] = 0.f;
  for (int s0 = 0; s0 < S; s0 += 32) {
    const int s = s0 + lane;
    const float wl = s < S ? exp2f(args.part_lse[(static_cast<int64_t>(s) * args.T + t) * args.H + h] - L2) : 0.f;
    const int n = min(32, S - s0);
    for (int k = 0; k < n; ++k) {
      const float w = __shfl_sync(0xffffffffu, wl, k);
      if (w == 0.f) continue;
      const float4* src = reinterpret_cast<const float4*>(
          args.part_o + ((static_cast<int64_t>(s0 + k) * args.T + t) * args.H + h) * kDv + lane * 16);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 v = src[q];
        acc[4 * q + 0] += w * v.x;
        acc[4 * q + 1] += w * v.y;
        acc[4 * q + 2] += w * v.z;
        acc[4 * q + 3] += w * v.w;
      }
    }
  }
  float f = 1.f;
  if (args.sink != nullptr) f = 1.f / (1.f + exp2f(args.sink[h] * 1.4426950408889634f - L2));
  uint32_t w32[8];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * k] * f, acc[2 * k + 1] * f);
    w32[k] = *reinterpret_cast<const uint32_t*>(&b);
  }
  reinterpret_cast<uint4*>(orow + lane * 16)[0] = make_uint4(w32[0], w32[1], w32[2], w32[3]);
  reinterpret_cast<uint4*>(orow + lane * 16)[1] = make_uint4(w32[4], w32[5], w32[6], w32[7]);
  if (lane == 0 && args.lse != nullptr) args.lse[static_cast<int64_t>(t) * args.lse_stride_t + h] = L2 * 0.6931471805599453f;
}

template <int NH>
cudaError_t launch_nh(const AttnArgs& a, const Plan& plan, cudaStream_t stream, cudaEvent_t ev0, cudaEvent_t ev1) {
  const int smem = Smem<NH>::kAlloc;
  cudaError_t e = cudaFuncSetAttribute(sparse_mla_kernel<NH>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const long long nblocks = static_cast<long long>(a.T) * plan.groups * plan.splits;
  if (ev0) cudaEventRecord(ev0, stream);
  sparse_mla_kernel<NH><<<static_cast<unsigned>(nblocks), kThreads, smem, stream>>>(a);
  e = cudaGetLastError();
  if (ev1) cudaEventRecord(ev1, stream);
  if (e != cudaSuccess) return e;
  if (plan.splits > 1) {
    const long long warps = static_cast<long long>(a.T) * a.H;
    combine_kernel<<<static_cast<unsigned>((warps + 7) / 8), 256, 0, stream>>>(a);
    e = cudaGetLastError();
  }
  return e;
}

static_assert(Smem<64>::kAlloc <= 232448, "shared memory budget");

}  // namespace

cudaError_t launch_attention(const AttnArgs& args, const Plan& plan, cudaStream_t stream, cudaEvent_t ev0,
                             cudaEvent_t ev1) {
  AttnArgs a = args;
  int* err = nullptr;
  cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&err), g_device_error);
  if (e != cudaSuccess) return e;
  a.err = err;
  switch (plan.nh) {
    case 16: return launch_nh<16>(a, plan, stream, ev0, ev1);
    case 32: return launch_nh<32>(a, plan, stream, ev0, ev1);
    case 64: return launch_nh<64>(a, plan, stream, ev0, ev1);
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
