// Cache writer: packs new latent rows (512 latent + 64 rope values, bf16 or fp32) into the
// paged cache in either row format, quantising to FP8 E4M3 with one fp32 scale per 128
// latent channels. The pages name this step as the packing of their benchmark inputs
// (flashinfer PR "add topk=256 prefill-dsv4 dispatch", conversation, GB10 benchmark "Method"
// paragraph) without its arithmetic; per 128-channel block this kernel computes
//   scale = amax / 448 (fp32, correctly rounded; 1 for an all-zero block)
//   code  = E4M3FN(x / scale)  (fp32 quotient, round to nearest even, saturate to +-448)
// and rounds rope channels (every channel of a bf16 row) to bf16, nearest even.
//
// One warp per row; lane l owns latent channels 16l..16l+15, so the eight lanes of a
// 128-channel block find its amax with three shuffles and every store is a coalesced
// 16-byte write. HBM-bound: a row reads 1152 (bf16) or 2304 (fp32) bytes and writes 656
// (FP8) or 1152 (bf16) bytes.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>

#include "smla.h"
#include "smla_internal.h"
#include "smla_ptx.cuh"

namespace smla {
namespace {

using namespace ptx;

// Bounded waits of the cache writer (~2 s), reported through smla_device_error.
__device__ int g_quant_error;
constexpr long long kQuantSpinCycles = 4000000000LL;

constexpr int kQuantWarps = 8;

struct QuantArgs {
  const uint8_t* kv;
  int64_t kv_stride_bytes;  // bytes between consecutive input rows
  int32_t in_f32;           // 0: bf16 input, 1: fp32 input
  int32_t n;
  const int64_t* slots;
  uint8_t* cache;
  int64_t row_stride, page_stride;
  int64_t num_slots;        // num_pages * 64
  int32_t fp8;
};

__device__ __forceinline__ uint4 ldg_v4(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Two fp32 values -> two E4M3FN codes (round to nearest even, saturating), a in the low byte.
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(b), "f"(a));
  return r;
}

// Two fp32 values -> two bf16 (round to nearest even), a in the low half.
__device__ __forceinline__ uint32_t bf16x2(float a, float b) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
  return r;
}

// This lane's 16 consecutive input values starting at channel c0, as fp32.
__device__ __forceinline__ void load16(const QuantArgs& q, const uint8_t* row, int c0, float* x) {
  if (q.in_f32) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 v = ldg_v4(row + 4 * (c0 + 4 * k));
      x[4 * k] = __uint_as_float(v.x);
      x[4 * k + 1] = __uint_as_float(v.y);
      x[4 * k + 2] = __uint_as_float(v.z);
      x[4 * k + 3] = __uint_as_float(v.w);
    }
  } else {
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const uint4 v = ldg_v4(row + 2 * (c0 + 8 * k));
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        x[8 * k + 2 * i] = bf16_lo(w[i]);
        x[8 * k + 2 * i + 1] = bf16_hi(w[i]);
      }
    }
  }
}

// One row from `in` (the row's 576 input values; shared memory here) to cache slot `slot`.
__device__ __forceinline__ void quantize_row(const QuantArgs& q, const uint8_t* in, long long slot, int lane) {
  if (!q.fp8) {
    // bf16 row: 576 channels = 72 chunks of 8 values; every load is issued before the slot is
    // known (they do not depend on it)
    uint4 o[3];
#pragma unroll
    for (int r = 0; r < 3; ++r) {
      const int ch = lane + 32 * r;
      o[r] = make_uint4(0, 0, 0, 0);
      if (ch < 72) {
        if (q.in_f32) {
          const uint4 a = ldg_v4(in + 32 * ch);
          const uint4 b = ldg_v4(in + 32 * ch + 16);
          o[r] = make_uint4(bf16x2(__uint_as_float(a.x), __uint_as_float(a.y)),
                            bf16x2(__uint_as_float(a.z), __uint_as_float(a.w)),
                            bf16x2(__uint_as_float(b.x), __uint_as_float(b.y)),
                            bf16x2(__uint_as_float(b.z), __uint_as_float(b.w)));
        } else {
          o[r] = ldg_v4(in + 16 * ch);
        }
      }
    }
    if (slot < 0 || slot >= q.num_slots) return;
    uint8_t* out = q.cache + (slot >> 6) * q.page_stride + (slot & 63) * q.row_stride;
#pragma unroll
    for (int r = 0; r < 3; ++r)
      if (lane + 32 * r < 72) *reinterpret_cast<uint4*>(out + 16 * (lane + 32 * r)) = o[r];
    return;
  }

  // FP8 row: latent channels 16*lane .. 16*lane+15 belong to block lane/8; the latent, rope and
  // slot loads are all issued before any of them is used
  float x[16];
  load16(q, in, 16 * lane, x);
  uint4 ra = make_uint4(0, 0, 0, 0), rb = make_uint4(0, 0, 0, 0);
  if (lane < 8) {
    if (q.in_f32) {
      const uint8_t* r = in + 4 * (kDv + 8 * lane);
      ra = ldg_v4(r);
      rb = ldg_v4(r + 16);
    } else {
      ra = ldg_v4(in + 2 * (kDv + 8 * lane));
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(x[k]));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
  amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
  const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 1.f;
  // x / scale rounded to nearest, sixteen times with one divisor: Markstein's correction of
  // x * RN(1/scale) (P. Markstein, "Computation of elementary functions on the IBM RISC
  // System/6000 processor", IBM J. Res. Dev. 34(1), 1990): with y = RN(1/b) and q = RN(a*y),
  // the remainder a - b*q is exact in one fma and RN(q + (a - b*q)*y) = RN(a/b) whenever the
  // quotient is a normal number. Quotients below the normal range all encode to E4M3 +-0,
  // which the sign (kept by working on |x|) decides. A block scale below the normal range
  // (amax < 448 * 2^-126) has no finite reciprocal: such blocks divide directly.
  const bool direct = scale < 1.17549435e-38f;
  const float ys = __frcp_rn(scale);
  auto quot = [&](float v) {
    if (direct) return __fdiv_rn(v, scale);
    const float a = fabsf(v);
    const float q0 = __fmul_rn(a, ys);
    const float r = __fmaf_rn(-scale, q0, a);
    return copysignf(__fmaf_rn(r, ys, q0), v);
  };
  uint32_t w[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint32_t lo = e4m3x2(quot(x[4 * k]), quot(x[4 * k + 1]));
    const uint32_t hi = e4m3x2(quot(x[4 * k + 2]), quot(x[4 * k + 3]));
    w[k] = lo | (hi << 16);
  }
  // the four block scales, gathered into lane 0
  const float s1 = __shfl_sync(0xffffffffu, scale, 8);
  const float s2 = __shfl_sync(0xffffffffu, scale, 16);
  const float s3 = __shfl_sync(0xffffffffu, scale, 24);
  if (slot < 0 || slot >= q.num_slots) return;
  uint8_t* out = q.cache + (slot >> 6) * q.page_stride + (slot & 63) * q.row_stride;
  *reinterpret_cast<uint4*>(out + 16 * lane) = make_uint4(w[0], w[1], w[2], w[3]);
  if (lane == 0)
    *reinterpret_cast<uint4*>(out + kDv) =
        make_uint4(__float_as_uint(scale), __float_as_uint(s1), __float_as_uint(s2), __float_as_uint(s3));
  // rope: 64 channels -> bf16, 8 lanes x 8 channels
  if (lane < 8) {
    const uint4 o = q.in_f32 ? make_uint4(bf16x2(__uint_as_float(ra.x), __uint_as_float(ra.y)),
                                          bf16x2(__uint_as_float(ra.z), __uint_as_float(ra.w)),
                                          bf16x2(__uint_as_float(rb.x), __uint_as_float(rb.y)),
                                          bf16x2(__uint_as_float(rb.z), __uint_as_float(rb.w)))
                             : ra;
    *reinterpret_cast<uint4*>(out + kDv + 16 + 16 * lane) = o;
  }
}

// Persistent: as many CTAs as fit on every SM at once, each warp walking the rows with the
// grid's warp count as stride. A warp keeps two rows in flight: lane 0 bulk-copies the next
// row into the warp's other shared-memory buffer (completion on that buffer's mbarrier) while
// the warp converts the current one; the slot word is also loaded a row ahead.
__device__ __forceinline__ bool quant_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait_sleep(bar, parity, 20000)) {
    if (clock64() - t0 > kQuantSpinCycles) return false;
  }
  return true;
}

__global__ void __launch_bounds__(kQuantWarps * 32) quantize_kv_kernel(const __grid_constant__ QuantArgs q) {
  __shared__ __align__(128) uint8_t rows[kQuantWarps][2][kDqk * 4];
  __shared__ __align__(8) uint64_t bars[kQuantWarps][2];
  const int lane = threadIdx.x & 31;
  const int w = threadIdx.x >> 5;
  const uint32_t bytes = q.in_f32 ? kDqk * 4 : kDqk * 2;
  const long long stride = static_cast<long long>(gridDim.x) * kQuantWarps;
  long long i = static_cast<long long>(blockIdx.x) * kQuantWarps + w;
  const uint32_t bar0 = smem_u32(&bars[w][0]), bar1 = smem_u32(&bars[w][1]);
  auto bar = [&](int b) { return b ? bar1 : bar0; };
  if (lane == 0) {
    mbar_init(bar0, 1);
    mbar_init(bar1, 1);
    fence_mbar_init();
  }
  __syncwarp();
  if (i >= q.n) return;
  auto issue = [&](long long r, int b) {
    if (lane == 0) {
      mbar_arrive_expect_tx(bar(b), bytes);
      cp_async_bulk_g2s(smem_u32(rows[w][b]), q.kv + r * q.kv_stride_bytes, bytes, bar(b));
    }
  };
  issue(i, 0);
  long long slot = q.slots[i];
  uint32_t phase = 0;  // bit b: parity of buffer b's next completion
#pragma unroll 1
  for (int k = 0; i < q.n; ++k, i += stride) {
    const int b = k & 1;
    const long long nx = i + stride;
    long long slot_nx = -1;
    if (nx < q.n) {
      // buffer b^1 was read in iteration k-1 (every lane finished before its __syncwarp): order
      // those reads before the copy that refills it
      fence_proxy_async_smem();
      issue(nx, b ^ 1);
      slot_nx = q.slots[nx];
    }
    if (!quant_wait(bar(b), (phase >> b) & 1u)) {
      // a copy that never lands: report it, give the other buffer's copy a bounded wait, stop
      if (lane == 0) atomicExch(&g_quant_error, 1);
      if (nx < q.n) quant_wait(bar(b ^ 1), (phase >> (b ^ 1)) & 1u);
      return;
    }
    phase ^= 1u << b;
    quantize_row(q, rows[w][b], slot, lane);
    __syncwarp();
    slot = slot_nx;
  }
}

// Resident CTAs of quantize_kv_kernel on the current device (SMs x CTAs per SM), cached per
// device.
int quant_resident_ctas() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 148;
  if (dev < 64) {
    const int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
  }
  int sms = 0, per_sm = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 148;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, quantize_kv_kernel, kQuantWarps * 32, 0) !=
          cudaSuccess ||
      per_sm <= 0)
    per_sm = 1;
  const int n = sms * per_sm;
  if (dev < 64) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

}  // namespace

// Reads and clears the cache writer's device error word.
cudaError_t read_and_clear_quant_error(int* code) {
  cudaError_t e = cudaMemcpyFromSymbol(code, g_quant_error, sizeof(int));
  if (e != cudaSuccess) return e;
  const int zero = 0;
  return cudaMemcpyToSymbol(g_quant_error, &zero, sizeof(int));
}

}  // namespace smla

using namespace smla;

extern "C" smla_status smla_quantize_kv(const void* kv, int32_t kv_dtype, int64_t kv_stride, int32_t n,
                                        const int64_t* slots, void* cache, int32_t format,
                                        int64_t row_stride_bytes, int64_t page_stride_bytes, int32_t num_pages,
                                        smla_stream_t stream) {
  if (n < 0 || (kv_dtype != SMLA_IN_BF16 && kv_dtype != SMLA_IN_F32)) return SMLA_ERR_INVALID;
  if (format != SMLA_KV_BF16 && format != SMLA_KV_FP8_E4M3_S128) return SMLA_ERR_UNSUPPORTED;
  if (n == 0) return SMLA_OK;
  const int64_t esize = kv_dtype == SMLA_IN_F32 ? 4 : 2;
  const int64_t row_bytes = format == SMLA_KV_BF16 ? kRowBf16 : kRowFp8;
  if (kv == nullptr || slots == nullptr || cache == nullptr || num_pages < 1 || num_pages > kMaxPages)
    return SMLA_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(kv) & 15u) != 0 || (reinterpret_cast<uintptr_t>(cache) & 15u) != 0 ||
      kv_stride < kDqk || ((kv_stride * esize) & 15) != 0)
    return SMLA_ERR_INVALID;
  if (row_stride_bytes < row_bytes || (row_stride_bytes & 15) != 0 || page_stride_bytes < kPage * row_stride_bytes ||
      (page_stride_bytes & 15) != 0)
    return SMLA_ERR_INVALID;
  QuantArgs q{};
  q.kv = static_cast<const uint8_t*>(kv);
  q.kv_stride_bytes = kv_stride * esize;
  q.in_f32 = kv_dtype == SMLA_IN_F32 ? 1 : 0;
  q.n = n;
  q.slots = slots;
  q.cache = static_cast<uint8_t*>(cache);
  q.row_stride = row_stride_bytes;
  q.page_stride = page_stride_bytes;
  q.num_slots = static_cast<int64_t>(num_pages) * kPage;
  q.fp8 = format == SMLA_KV_FP8_E4M3_S128 ? 1 : 0;
  const long long want = (static_cast<long long>(n) + kQuantWarps - 1) / kQuantWarps;
  const unsigned grid = static_cast<unsigned>(std::min<long long>(want, quant_resident_ctas()));
  quantize_kv_kernel<<<grid, kQuantWarps * 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(q);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    note_cuda_error(e, "launch of quantize_kv_kernel");
    return SMLA_ERR_CUDA;
  }
  return SMLA_OK;
}
