// Thin inline-PTX wrappers for sm_103a: mbarrier, cp.async, tcgen05 (TMEM alloc, MMA,
// commit, TMEM load/store, fences) and the UMMA shared-memory / instruction descriptors.
#pragma once
#include <cstdint>

namespace smla {
namespace ptx {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.b32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Like mbar_try_wait, but the thread may sleep in hardware (up to hint_ns) until the phase
// completes instead of returning at once, so waiting threads do not poll shared memory.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.b32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Arrive on the mbarrier and raise its expected transaction bytes by `bytes` (the phase then
// completes once that many bytes of asynchronous copies have landed).
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// Bulk copy of `bytes` (multiple of 16; both addresses 16-byte aligned) global -> this CTA's
// shared memory, completing as transaction bytes on the mbarrier.
__device__ __forceinline__ void cp_async_bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// ------------------------------------------------------------------ cp.async (16 B, L2 only)
// src_bytes = 16 copies, 0 zero-fills the destination without reading the source.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
// Bulk prefetch of `bytes` (multiple of 16, 16-byte aligned source) from global memory into L2.
__device__ __forceinline__ void prefetch_l2_bulk(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
// 4-byte asynchronous copy global -> shared (through L1).
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait_group() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Make generic-proxy writes to shared memory visible to the async proxy (tensor core).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ global loads
__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}
// Scalar read-only loads kept in program order (volatile): a load issued ahead of its use must
// stay where it is written, not be sunk to (or re-issued at) the point of use.
__device__ __forceinline__ int32_t ldg_nc_s32(const void* p) {
  int32_t r;
  asm volatile("ld.global.nc.b32 %0, [%1];" : "=r"(r) : "l"(p));
  return r;
}
__device__ __forceinline__ float ldg_nc_f32(const void* p) {
  float r;
  asm volatile("ld.global.nc.f32 %0, [%1];" : "=f"(r) : "l"(p));
  return r;
}
__device__ __forceinline__ void sts_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D(tmem) (+)= A(smem desc) * B(smem desc), bf16 inputs, fp32 accumulate, one CTA: four MMAs
// along K in one warp-collective block. Every lane of the converged warp executes it and
// elect.sync picks the issuing lane (the same lane for every call of a converged warp, so a
// commit tracks the MMAs issued before it); the MMAs are predicated, so the warp never
// diverges around the issue stream. A descriptor is passed as its two 32-bit words: the low
// word carries the start address (and the leading byte offset), the high word is constant per
// operand layout; step k adds k * SA (k * SB) to the low word, i.e. 16 * SA bytes to A's start
// address. Only the first MMA takes `accumulate`; the other three accumulate.
//
// Keeping the address arithmetic in 32 bits, with the per-step offsets as immediates and one
// elect per group, shrinks an MMA from ~450 to ~125 bytes of code (the attention kernel
// issues 112 of them per tile in straight-line code; with 64-bit descriptor adds it was
// dominated by them).
template <int SA, int SB>
__device__ __forceinline__ void mma_bf16_x4(uint32_t d_tmem, uint32_t a_lo, uint32_t a_hi, uint32_t b_lo, uint32_t b_hi,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p, q;\n .reg .b32 r, a1, b1;\n .reg .b64 da, db;\n"
      " elect.sync r|q, 0xffffffff;\n setp.ne.b32 p, %6, 0;\n"
      " mov.b64 da, {%1, %2};\n mov.b64 db, {%3, %4};\n"
      " @q tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n"
      " setp.eq.b32 p, 0, 0;\n"
      " add.u32 a1, %1, %7;\n add.u32 b1, %3, %8;\n mov.b64 da, {a1, %2};\n mov.b64 db, {b1, %4};\n"
      " @q tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n"
      " add.u32 a1, %1, %9;\n add.u32 b1, %3, %10;\n mov.b64 da, {a1, %2};\n mov.b64 db, {b1, %4};\n"
      " @q tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n"
      " add.u32 a1, %1, %11;\n add.u32 b1, %3, %12;\n mov.b64 da, {a1, %2};\n mov.b64 db, {b1, %4};\n"
      " @q tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %5, p;\n}\n" ::"r"(d_tmem),
      "r"(a_lo), "r"(a_hi), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate), "n"(SA), "n"(SB), "n"(2 * SA),
      "n"(2 * SB), "n"(3 * SA), "n"(3 * SB)
      : "memory");
}
// The same with A read from TMEM (tcgen05 "A in tensor memory" form): a_tmem is the TMEM
// address of A's 128 lanes x 16 bf16 (8 columns); every K step reads the same A, and B advances
// by SB per step.
template <int SB>
__device__ __forceinline__ void mma_bf16_ts_x4(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                               uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p, q;\n .reg .b32 r, b1;\n .reg .b64 db;\n"
      " elect.sync r|q, 0xffffffff;\n setp.ne.b32 p, %5, 0;\n"
      " mov.b64 db, {%2, %3};\n"
      " @q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p;\n"
      " setp.eq.b32 p, 0, 0;\n"
      " add.u32 b1, %2, %6;\n mov.b64 db, {b1, %3};\n"
      " @q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p;\n"
      " add.u32 b1, %2, %7;\n mov.b64 db, {b1, %3};\n"
      " @q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p;\n"
      " add.u32 b1, %2, %8;\n mov.b64 db, {b1, %3};\n"
      " @q tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %4, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate), "n"(SB), "n"(2 * SB), "n"(3 * SB)
      : "memory");
}
// Arrive once on the mbarrier when every MMA previously issued by the warp's elected lane has
// completed (warp-collective, like the MMAs).
__device__ __forceinline__ void mma_commit_warp(uint32_t bar) {
  asm volatile(
      "{\n .reg .pred q;\n .reg .b32 r;\n elect.sync r|q, 0xffffffff;\n"
      " @q tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n" ::"r"(bar)
      : "memory");
}

// 32 lanes x 16 columns of 32-bit (each thread: its lane, 16 consecutive columns), then wait.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// Loads without the wait, so several can be in flight before one tmem_ld_wait().
__device__ __forceinline__ void tmem_ld16_nw(uint32_t taddr, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld32_nw(uint32_t taddr, float* v) {
  uint32_t* r = reinterpret_cast<uint32_t*>(v);
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}
// The wait names the loaded registers as in/out operands, so no use of them can be scheduled
// before it.
__device__ __forceinline__ void tmem_ld_wait16(float* v) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+f"(v[0]), "+f"(v[1]), "+f"(v[2]), "+f"(v[3]), "+f"(v[4]), "+f"(v[5]), "+f"(v[6]), "+f"(v[7]),
                 "+f"(v[8]), "+f"(v[9]), "+f"(v[10]), "+f"(v[11]), "+f"(v[12]), "+f"(v[13]), "+f"(v[14]),
                 "+f"(v[15])
               :
               : "memory");
}
__device__ __forceinline__ void tmem_ld_wait32(float* v) {
  tmem_ld_wait16(v);
  asm volatile(""
               : "+f"(v[16]), "+f"(v[17]), "+f"(v[18]), "+f"(v[19]), "+f"(v[20]), "+f"(v[21]), "+f"(v[22]),
                 "+f"(v[23]), "+f"(v[24]), "+f"(v[25]), "+f"(v[26]), "+f"(v[27]), "+f"(v[28]), "+f"(v[29]),
                 "+f"(v[30]), "+f"(v[31])
               :
               : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(
          taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ------------------------------------------------------------------ UMMA descriptors
// Shared-memory matrix descriptor (tcgen05), as two 32-bit words. Low word: start address >> 4
// (bits 0-13) and leading-dimension byte offset >> 4 (bits 16-29). High word: stride-dimension
// byte offset >> 4 (bits 32-45 of the descriptor), descriptor version 1 (bit 46), swizzle mode
// (bits 61-63). A shared address is below 2^18, so adding a byte offset >> 4 that stays inside
// the shared window to the low word never carries out of the start-address field.
enum : uint32_t { kSwizzleNone = 0, kSwizzle128B = 2, kSwizzle64B = 4, kSwizzle32B = 6 };

__device__ __forceinline__ uint32_t smem_desc_lo(uint32_t saddr, uint32_t lbo) {
  return ((saddr & 0x3FFFFu) >> 4) | (((lbo >> 4) & 0x3FFFu) << 16);
}
__host__ __device__ constexpr uint32_t smem_desc_hi(uint32_t sbo, uint32_t swz) {
  return ((sbo >> 4) & 0x3FFFu) | (1u << 14) | (swz << 29);
}

// Instruction descriptor for kind::f16 with bf16 A/B and fp32 D.
// a_mn / b_mn: 0 = K-major operand, 1 = MN-major operand.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4)                                 // D format: f32
         | (1u << 7)                               // A format: bf16
         | (1u << 10)                              // B format: bf16
         | (static_cast<uint32_t>(a_mn) << 15)     // A major
         | (static_cast<uint32_t>(b_mn) << 16)     // B major
         | (static_cast<uint32_t>(N >> 3) << 17)   // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);  // M / 16
}

// ------------------------------------------------------------------ math helpers
__device__ __forceinline__ uint64_t pack_f32x2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
// bf16x2 of (a * f.lo, b * f.hi): one paired fp32 multiply (round to nearest), one rounding to
// bf16 (RNE); a's result in the low half.
__device__ __forceinline__ uint32_t mul_pack_bf16x2(float a, float b, uint64_t f) {
  uint32_t out;
  asm("{\n .reg .b64 x;\n .reg .f32 lo, hi;\n mov.b64 x, {%1, %2};\n mul.rn.f32x2 x, x, %3;\n"
      " mov.b64 {lo, hi}, x;\n cvt.rn.bf16x2.f32 %0, hi, lo;\n}\n"
      : "=r"(out)
      : "f"(a), "f"(b), "l"(f));
  return out;
}
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace ptx
}  // namespace smla
