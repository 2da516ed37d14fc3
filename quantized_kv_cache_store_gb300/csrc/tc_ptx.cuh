// tc_ptx.cuh -- thin inline-PTX wrappers for the sm_103a tensor-core path of
// libtqkv: mbarriers, bulk global->shared copies, tcgen05 (TMEM allocation,
// MMA with A in tensor memory, commit, loads and stores), proxy fences and
// named barriers.  Internal header.
#pragma once

#include <stdint.h>

namespace tq {
namespace ptx {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

// ------------------------------------------------------------- mbarriers
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}
// Tests the phase with the given parity; the thread may be suspended for up to
// `suspend_ns` nanoseconds while the phase is still pending (it resumes as soon
// as the phase completes), so waiting warps do not occupy issue slots.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity, uint32_t suspend_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(suspend_ns)
      : "memory");
  return ok != 0;
}
// Non-blocking test of the phase with the given parity.
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// ------------------------------------------------ bulk copy (non-tensor TMA)
// dst, src 16-byte aligned, bytes a multiple of 16; completes tx on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

// L2 eviction policy for data read once per call (the cache pages): evicted
// first, so that the small inputs every CTA re-reads (block table, queries)
// and the partial rows stay in L2.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(pol));
  return pol;
}
// bulk copy with an L2 cache policy
__device__ __forceinline__ void bulk_g2s_hint(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                              uint64_t pol) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;\n" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar), "l"(pol)
      : "memory");
}

// tiled tensor copy (TMA), 3-D box at coordinates {x, y, z}; completes tx on `bar`
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, int x, int y, int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];\n" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// as tma_load_3d, with an L2 cache policy
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const void* tmap, int x, int y, int z, uint32_t bar,
                                                 uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, %3, "
      "%4}], [%5], %6;\n" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(pol)
      : "memory");
}

// ----------------------------------------------------------------- fences
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
// Named barriers in their non-aligned form: a warp may arrive diverged (for
// example after a lane-0-only branch); every thread is counted on arrival.
__device__ __forceinline__ void named_bar(uint32_t id, uint32_t n) {
  asm volatile("barrier.sync %0, %1;\n" ::"r"(id), "r"(n) : "memory");
}
// all threads of the CTA (barrier 0)
__device__ __forceinline__ void cta_bar() { asm volatile("barrier.sync 0;\n" ::: "memory"); }
// barrier over n threads with an OR-reduction of `pred`
__device__ __forceinline__ bool bar_red_or(uint32_t id, uint32_t n, bool pred) {
  uint32_t out;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n barrier.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(out)
      : "r"((uint32_t)pred), "r"(id), "r"(n)
      : "memory");
  return out != 0;
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar) : "memory");
}
// Eight MMAs D (+)= A_k * B_k (kind::f16, A in tensor memory, B by shared-
// memory descriptor, fp32 accumulate), k = 0..7, into the same accumulator, issued
// back to back: A_k at tensor-memory column a + 8 k, B_k's descriptor =
// bdesc + boff[k] (start-address units of 16 bytes).  The first MMA
// accumulates iff acc0; the others always do.
template <uint32_t O1, uint32_t O2, uint32_t O3, uint32_t O4, uint32_t O5, uint32_t O6, uint32_t O7>
__device__ __forceinline__ void mma_ts_x8(uint32_t d, uint32_t a, uint64_t bdesc, uint32_t idesc, uint32_t acc0) {
  asm volatile(
      "{\n .reg .pred p, t;\n .reg .b64 b1, b2, b3, b4, b5, b6, b7;\n .reg .b32 a1, a2, a3, a4, a5, a6, a7;\n"
      " setp.ne.b32 p, %4, 0;\n setp.eq.b32 t, %4, %4;\n"
      " add.u64 b1, %2, %5;\n add.u64 b2, %2, %6;\n add.u64 b3, %2, %7;\n add.u64 b4, %2, %8;\n"
      " add.u64 b5, %2, %9;\n add.u64 b6, %2, %10;\n add.u64 b7, %2, %11;\n"
      " add.u32 a1, %1, 8;\n add.u32 a2, %1, 16;\n add.u32 a3, %1, 24;\n add.u32 a4, %1, 32;\n"
      " add.u32 a5, %1, 40;\n add.u32 a6, %1, 48;\n add.u32 a7, %1, 56;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %3, t;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %3, t;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %3, t;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [a4], b4, %3, t;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [a5], b5, %3, t;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [a6], b6, %3, t;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [a7], b7, %3, t;\n}\n" ::"r"(d),
      "r"(a), "l"(bdesc), "r"(idesc), "r"(acc0), "n"((uint64_t)O1), "n"((uint64_t)O2), "n"((uint64_t)O3),
      "n"((uint64_t)O4), "n"((uint64_t)O5), "n"((uint64_t)O6), "n"((uint64_t)O7)
      : "memory");
}

// Instruction descriptor, kind::f16: A, B f16; D f32; M = 128; N; operand majors.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int a_mn_major, int b_mn_major) {
  return (1u << 4) | ((uint32_t)a_mn_major << 15) | ((uint32_t)b_mn_major << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
// Shared-memory matrix descriptor: start address, leading / stride byte
// offsets, layout (2 = 128B swizzle, 4 = 64B, 6 = 32B).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)layout << 61;
  return d;
}

// 32 lanes x 32b shape: thread i of the warp reaches TMEM lane (quadrant + i),
// N consecutive 32-bit columns.
#define TQ_R8(b) "r"(r[b + 0]), "r"(r[b + 1]), "r"(r[b + 2]), "r"(r[b + 3]), "r"(r[b + 4]), "r"(r[b + 5]), "r"(r[b + 6]), "r"(r[b + 7])
#define TQ_W8(b) "=r"(r[b + 0]), "=r"(r[b + 1]), "=r"(r[b + 2]), "=r"(r[b + 3]), "=r"(r[b + 4]), "=r"(r[b + 5]), "=r"(r[b + 6]), "=r"(r[b + 7])

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
      TQ_R8(0), TQ_R8(8), TQ_R8(16), TQ_R8(24)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(
          taddr),
      TQ_R8(0), TQ_R8(8)
      : "memory");
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      : TQ_W8(0), TQ_W8(8), TQ_W8(16), TQ_W8(24)
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
               : TQ_W8(0)
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n" ::"r"(taddr), TQ_R8(0)
               : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
      : TQ_W8(0), TQ_W8(8)
      : "r"(taddr)
      : "memory");
}
#undef TQ_R8
#undef TQ_W8

template <int N>
__device__ __forceinline__ void tmem_st(uint32_t taddr, const uint32_t (&r)[N]);
template <>
__device__ __forceinline__ void tmem_st<32>(uint32_t taddr, const uint32_t (&r)[32]) {
  tmem_st32(taddr, r);
}
template <>
__device__ __forceinline__ void tmem_st<16>(uint32_t taddr, const uint32_t (&r)[16]) {
  tmem_st16(taddr, r);
}
template <int N>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&r)[N]);
template <>
__device__ __forceinline__ void tmem_ld<32>(uint32_t taddr, uint32_t (&r)[32]) {
  tmem_ld32(taddr, r);
}
template <>
__device__ __forceinline__ void tmem_ld<16>(uint32_t taddr, uint32_t (&r)[16]) {
  tmem_ld16(taddr, r);
}
template <>
__device__ __forceinline__ void tmem_ld<8>(uint32_t taddr, uint32_t (&r)[8]) {
  tmem_ld8(taddr, r);
}

template <uint32_t R>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(R));
}
template <uint32_t R>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(R));
}
// from the launch's per-thread register count L to R: an increase, a
// decrease or nothing (setmaxnreg.dec may only lower, .inc only raise)
template <int R, int L>
__device__ __forceinline__ void regs_to() {
  static_assert(R % 8 == 0 && R >= 24 && R <= 256, "setmaxnreg count");
  if constexpr (R > L) regs_inc<R>();
  else if constexpr (R < L) regs_dec<R>();
}

}  // namespace ptx
}  // namespace tq
