// sm103_primitives.cuh -- inline-PTX building blocks for the sm_103a
// attention forward: mbarriers with bounded waits, TMA tile loads and
// stores, and the fifth-generation tensor core (tcgen05.mma with TMEM
// accumulators).
//
// Everything here is written from the PTX ISA's descriptions of these
// instructions.  The encodings used:
//
// * Shared-memory matrix descriptor (64 bit) for tcgen05.mma operands:
//     bits  0-13  start address >> 4
//     bits 16-29  leading-dimension byte offset >> 4
//     bits 32-45  stride-dimension byte offset >> 4
//     bits 46-48  fixed 0b001
//     bits 49-51  base offset (0: every tile here is 1024-byte aligned)
//     bit  52     LBO mode (0: relative)
//     bits 61-63  swizzle mode (2 = 128-byte swizzle)
//   With the 128-byte swizzle a K-major operand is rows of 128 bytes (64
//   fp16) in 8-row / 1024-byte atoms: SBO = 1024, LBO unused.  An MN-major
//   operand is K-rows of 128 bytes of MN in the same atoms: SBO = 1024 is the
//   step between 8-deep K groups and LBO the step between 64-wide MN chunks.
//
// * Instruction descriptor (32 bit) of tcgen05.mma.kind::f16:
//     bits 4-5 D format (1 = f32), bits 7-9 A format and 10-12 B format
//     (0 = f16), bit 15 A major and bit 16 B major (0 = K, 1 = MN),
//     bits 17-22 N >> 3, bits 24-28 M >> 4.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>

namespace attn_sm103 {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.release.cta.shared::cta.b64 st, [%0];\n\t}"
      ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .b64 st;\n\t"
      "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 st, [%0], %1;\n\t}"
      ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Shared state of the bounded waits of one CTA.  Every wait gives up after
// `timeout_ns` of global time, raises the CTA's abort flag and records
// `code` in the device status word and in its host copy (page-locked host
// memory mapped into the device, or null); a wait that sees the abort flag
// raised by another role gives up at once.  No wait in the kernel is
// unbounded.
struct WaitCtl {
  volatile int* abort_flag;  // shared memory
  int* status;               // global memory, first error wins
  volatile int* status_host; // host copy, read by the host before each call
  uint64_t timeout_ns;
};

__device__ __forceinline__ void record_error(const WaitCtl& w, int code) {
  atomicCAS(w.status, 0, code);
  if (w.status_host != nullptr) {
    *w.status_host = code;
    __threadfence_system();
  }
}

__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, const WaitCtl& w,
                                          int code, bool honor_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (honor_abort && *w.abort_flag) return false;
    if (globaltimer_ns() - t0 > w.timeout_ns) {
      *w.abort_flag = 1;
      record_error(w, code);
      return false;
    }
  }
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_map(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 3-D tiled load of one box into shared memory; completion is signalled on
// `bar` as transaction bytes.  c0 is the innermost (element) coordinate.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2),
        "r"(smem_u32(bar))
      : "memory");
}

// 3-D tiled store of one box from shared memory (bulk async-group
// completion).  Elements of the box outside the tensor are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, const void* src, int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%2, %3, %4}], [%1];"
      ::"l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Waits until every committed bulk group of this thread has finished
// reading its shared-memory source, so the CTA may exit and its shared
// memory go; the global writes complete on their own.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Orders this thread's earlier generic-proxy shared-memory writes before
// later async-proxy (TMA) reads of them.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- TMEM
// Allocation is warp-collective; the TMEM address is written to `slot`.
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               ::"r"(smem_u32(slot)), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

#define ATTN_R8(b) "=r"(r[b + 0]), "=r"(r[b + 1]), "=r"(r[b + 2]), "=r"(r[b + 3]), \
                   "=r"(r[b + 4]), "=r"(r[b + 5]), "=r"(r[b + 6]), "=r"(r[b + 7])
#define ATTN_W8(b) "+r"(r[b + 0]), "+r"(r[b + 1]), "+r"(r[b + 2]), "+r"(r[b + 3]), \
                   "+r"(r[b + 4]), "+r"(r[b + 5]), "+r"(r[b + 6]), "+r"(r[b + 7])
#define ATTN_S8(b) "r"(r[b + 0]), "r"(r[b + 1]), "r"(r[b + 2]), "r"(r[b + 3]), \
                   "r"(r[b + 4]), "r"(r[b + 5]), "r"(r[b + 6]), "r"(r[b + 7])

// Thread t of the warp reads lane (taddr.lane + t), 32 consecutive 32-bit
// columns starting at taddr.col.  The values are valid only after
// tmem_ld_wait on the same array.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : ATTN_R8(0), ATTN_R8(8), ATTN_R8(16), ATTN_R8(24)
      : "r"(taddr));
}

// Waits for every outstanding tcgen05.ld of the thread.  The registers are
// routed through the asm so that no use of them is scheduled before it.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : ATTN_W8(0), ATTN_W8(8), ATTN_W8(16), ATTN_W8(24)
               :
               : "memory");
}

// tmem_ld32 that also returns, per thread, the maximum of the 32 values it
// loads (tcgen05.ld.red, sm_103a).  Valid after tmem_ld_wait_max.
__device__ __forceinline__ void tmem_ld32_max(uint32_t taddr, uint32_t (&r)[32], float& mx) {
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x32.max.f32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, %32, [%33];"
      : ATTN_R8(0), ATTN_R8(8), ATTN_R8(16), ATTN_R8(24), "=f"(mx)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait_max(uint32_t (&r)[32], float& mx) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : ATTN_W8(0), ATTN_W8(8), ATTN_W8(16), ATTN_W8(24), "+f"(mx)
               :
               : "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      ::"r"(taddr), ATTN_S8(0), ATTN_S8(8), ATTN_S8(16), ATTN_S8(24)
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      ::"r"(taddr), ATTN_S8(0), ATTN_S8(8)
      : "memory");
}

#undef ATTN_R8
#undef ATTN_W8
#undef ATTN_S8

// ---------------------------------------------------------------- UMMA
constexpr uint64_t kSwizzle128B = 2;

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= kSwizzle128B << 61;
  return d;
}

__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4)                                    // D: f32
         | (0u << 7) | (0u << 10)                     // A, B: f16
         | (static_cast<uint32_t>(a_mn_major) << 15)  // A major
         | (static_cast<uint32_t>(b_mn_major) << 16)  // B major
         | (static_cast<uint32_t>(N >> 3) << 17)      // N
         | (static_cast<uint32_t>(M >> 4) << 24);     // M
}

// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void umma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void umma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Warp-wide forms of the three ops above: every lane of a converged warp
// calls them with the same operands and lane 0 alone issues the instruction
// (always the same lane, so that a commit tracks the products it follows).
// Keeping the issuing code warp-uniform lets the operands stay in uniform
// registers; measured on GB300, this issues the products of a fused
// attention step about 5 % faster than a branch on lane 0 around the
// single-thread forms, and faster than predicating on elect.sync.
__device__ __forceinline__ void umma_ss_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t.reg .u32 l;\n\t"
      "mov.u32 l, %%laneid;\n\t"
      "setp.eq.u32 e, l, 0;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_ts_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t.reg .u32 l;\n\t"
      "mov.u32 l, %%laneid;\n\t"
      "setp.eq.u32 e, l, 0;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same two products with 8-bit operands (tcgen05.mma.kind::f8f6f4;
// with A and B format code 0 in the instruction descriptor both are E4M3,
// and one instruction reduces over 32 elements of K, still 32 bytes).
__device__ __forceinline__ void umma_ss_f8_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t.reg .u32 l;\n\t"
      "mov.u32 l, %%laneid;\n\t"
      "setp.eq.u32 e, l, 0;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_ts_f8_warp(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t.reg .u32 l;\n\t"
      "mov.u32 l, %%laneid;\n\t"
      "setp.eq.u32 e, l, 0;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}"
      ::"r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void umma_commit_warp(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t.reg .u32 l;\n\t"
      "mov.u32 l, %%laneid;\n\t"
      "setp.eq.u32 e, l, 0;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}"
      ::"r"(smem_u32(bar)) : "memory");
}

// One arrive on `bar` once every tcgen05 op issued so far by this thread
// has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(smem_u32(bar)) : "memory");
}

// ---------------------------------------------------------------- math
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Four floats rounded to OCP FP8 E4M3 (round to nearest even, saturating
// to +-448), packed little-endian: a in bits 0-7, b in 8-15, c in 16-23, d
// in 24-31 -- the order of consecutive elements in memory and in TMEM.
// cvt.rn.satfinite.e4m3x2.f32 puts its first source in the upper byte.
__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// 2^x for a pair of floats on the FMA pipe instead of the MUFU unit.
// Argument reduction after Cody and Waite ("Software Manual for the
// Elementary Functions", 1980): n = round(x) by adding 1.5 * 2^23, f = x - n
// in [-1/2, 1/2]; 2^f by the degree-4 polynomial with constant term 1 that
// minimises the maximum relative error on [-1/2, 1/2] (Remez exchange;
// fit_exp2_poly.py next to this file reproduces the coefficients); 2^n by
// adding n to the exponent field.  Valid for x <= 127; x below -126 (and NaN)
// is clamped to -126, giving 2^-126 instead of a smaller number or zero.
// Measured maximum relative error of the fp32 evaluation on [-126, 8]:
// 3.7e-6.
__device__ __forceinline__ float2 exp2_poly2(float2 x) {
  constexpr float kShift = 12582912.0f;  // 1.5 * 2^23: adding it rounds to an integer
  const float2 xc = make_float2(fmaxf(x.x, -126.0f), fmaxf(x.y, -126.0f));
  const float2 t = __fadd2_rn(xc, make_float2(kShift, kShift));
  const float2 n = __fadd2_rn(t, make_float2(-kShift, -kShift));
  const float2 f = __ffma2_rn(n, make_float2(-1.0f, -1.0f), xc);
  float2 p = __ffma2_rn(make_float2(0.009782912209630013f, 0.009782912209630013f), f,
                        make_float2(0.055976882576942444f, 0.055976882576942444f));
  p = __ffma2_rn(p, f, make_float2(0.24020710587501526f, 0.24020710587501526f));
  p = __ffma2_rn(p, f, make_float2(0.6931136250495911f, 0.6931136250495911f));
  p = __ffma2_rn(p, f, make_float2(1.0f, 1.0f));
  return make_float2(__int_as_float(__float_as_int(p.x) + (__float_as_int(t.x) << 23)),
                     __int_as_float(__float_as_int(p.y) + (__float_as_int(t.y) << 23)));
}

}  // namespace attn_sm103
