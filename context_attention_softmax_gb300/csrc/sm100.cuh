// Thin inline-PTX wrappers for the Blackwell (sm_100 family, here sm_103a)
// asynchronous machinery: mbarriers, TMA tensor loads, tensor memory (TMEM)
// allocation and access, and tcgen05 MMA with shared-memory descriptors.
// Every wait is bounded: it gives up after a time limit, raises a shared
// abort flag and lets the caller wind down (no trap, no endless spin).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace cpattn {
namespace sm100 {

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
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Arrives on the barrier once every cp.async issued so far by this thread has
// landed; the arrival is counted in the barrier's expected count.
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, but a thread whose phase is still open is suspended
// until the phase completes or about hint_ns have passed, so a waiting
// warp takes no issue slots from the warps that share its sub-partition.
__device__ __forceinline__ bool mbar_try_wait_suspend(uint64_t* bar, uint32_t parity,
                                                      uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Wait until the phase with the given parity has completed.  Returns false
// (and sets *abort) when the wait exceeds limit_ns or another role aborted.
// A thread is suspended for at most min(limit_ns, 1 ms) at a time.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint64_t limit_ns = 2000000000ull) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  const uint32_t hint = limit_ns < 1000000ull ? (uint32_t)limit_ns : 1000000u;
  while (!mbar_try_wait_suspend(bar, parity, hint)) {
    if (*abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      *abort = 1;
      return false;
    }
  }
  return true;
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}
// 3-D tiled load into shared memory; completion is counted on `bar` in bytes.
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int32_t c0, int32_t c1, int32_t c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// L2 cache policies: keep a line (data that every CTA re-reads) or let it go
// first (a result written once and not read again by this kernel).
__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
// tma_load_3d with an L2 cache policy for the copied lines.
__device__ __forceinline__ void tma_load_3d_hint(void* dst, const CUtensorMap* map, uint64_t* bar,
                                                 int32_t c0, int32_t c1, int32_t c2, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "l"(pol)
      : "memory");
}
// 16-byte global store with an L2 cache policy.
__device__ __forceinline__ void st_global_v4_hint(void* ptr, uint4 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(ptr), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
               : "memory");
}

// 3-D tiled store from shared memory (the layout a tma_load_3d of the same
// box would produce) to global memory, with an L2 cache policy; rows outside
// the tensor are not written.  Completion is tracked by bulk groups.
__device__ __forceinline__ void tma_store_3d_hint(const CUtensorMap* map, const void* src, int32_t c0,
                                                  int32_t c1, int32_t c2, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group.L2::cache_hint"
      " [%0, {%2, %3, %4}], [%1], %5;" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(c0), "r"(c1), "r"(c2), "l"(pol)
      : "memory");
}
__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Wait until at most N committed bulk groups still read shared memory.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
// Wait until every committed bulk group has completed (writes included).
__device__ __forceinline__ void bulk_wait_group_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Writes by ordinary stores to shared memory become visible to the tensor
// core (async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- TMEM
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
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

// 32 lanes x 32 consecutive 32-bit columns: thread t of the warp receives
// lane (taddr.lane + t), r[i] = column taddr.col + i.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
      "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
      "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
      "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
// Named barrier over `count` threads (ids 1..15; 0 is __syncthreads).
__device__ __forceinline__ void named_bar_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Named barrier over `count` threads that also ANDs a predicate across them:
// every participant receives the same result.
__device__ __forceinline__ bool named_bar_and(uint32_t id, uint32_t count, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %3, 0;\n\t"
      "bar.red.and.pred q, %1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(id), "r"(count), "r"((uint32_t)pred)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ---------------------------------------------------------------- UMMA
// Shared-memory matrix descriptor (tcgen05 format): start address,
// leading/stride byte offsets (all >> 4), descriptor version 1 (bits 46-47),
// base offset 0, swizzle mode in bits 61-63 (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes,
                                              uint32_t sbo_bytes, uint32_t swizzle) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)(swizzle & 0x7u) << 61;
  return d;
}
constexpr uint32_t kSwizzle128B = 2;

// Instruction descriptor of kind::f16 with bf16 A/B and fp32 accumulation.
// a_mn / b_mn: operand stored MN-major (1) or K-major (0).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int a_mn, int b_mn) {
  return (1u << 4)                       // D format: f32
         | (1u << 7)                     // A format: bf16
         | (1u << 10)                    // B format: bf16
         | ((uint32_t)a_mn << 15)        // A major
         | ((uint32_t)b_mn << 16)        // B major
         | ((uint32_t)(N >> 3) << 17)    // N / 8
         | ((uint32_t)(M >> 4) << 24);   // M / 16
}

// D[tmem] (+)= A[smem] * B[smem]; issued by one thread.
__device__ __forceinline__ void umma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Split form of a shared-memory descriptor for the issue loop: the high word
// (stride byte offset 1024, version 1, 128-byte swizzle) is the same for
// every operand here; the low word carries start address and leading byte
// offset, so stepping along K is one 32-bit add.
constexpr uint32_t kDescHiSw128 = (1024u >> 4) | (1u << 14) | (kSwizzle128B << 29);
__device__ __forceinline__ uint32_t desc_lo(uint32_t saddr, uint32_t lbo_bytes) {
  return ((saddr >> 4) & 0x3FFFu) | (((lbo_bytes >> 4) & 0x3FFFu) << 16);
}
template <bool W = false>
__device__ __forceinline__ void umma_ss_lo(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo,
                                           uint32_t idesc, uint32_t accumulate) {
  if constexpr (W)
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t.reg .b64 da, db;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "mov.b64 da, {%1, %5};\n\t"
        "mov.b64 db, {%2, %5};\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_lo), "r"(b_lo), "r"(idesc), "r"(accumulate), "n"(kDescHiSw128));
  else
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "mov.b64 da, {%1, %5};\n\t"
        "mov.b64 db, {%2, %5};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], da, db, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_lo), "r"(b_lo), "r"(idesc), "r"(accumulate), "n"(kDescHiSw128));
}
__device__ __forceinline__ void umma_ts_lo(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 db;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "mov.b64 db, {%2, %5};\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], db, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(idesc), "r"(accumulate), "n"(kDescHiSw128));
}

// The grouped MMA helpers below come in two issue forms.  W = false: the
// caller is a single thread (a divergent branch of its warp).  W = true: the
// whole warp calls with identical arguments and one lane, picked by
// elect.sync, issues; a converged issuing warp loses fewer issue slots to
// busy warps of its sub-partition.
#define CPATTN_ELECT_DECL ".reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"

// Eight MMAs along K = 128 (16 per instruction) in one PTX block, both
// operands K-major in 64-column 128-byte-swizzled boxes: step k reads the
// descriptors lo + (k / 4) * 1024 + (k % 4) * 2 (16 KiB per box, 32 B per
// step).  The first MMA overwrites D, the rest accumulate.
#define CPATTN_UMMA8_SS_TEXT(DECL, P)                                   \
  "{\n\t.reg .b32 a<8>, b<8>;\n\t.reg .b64 da<8>, db<8>;\n\t" DECL     \
  "add.u32 a0, %1, 0;    add.u32 b0, %2, 0;\n\t"                       \
  "add.u32 a1, %1, 2;    add.u32 b1, %2, 2;\n\t"                       \
  "add.u32 a2, %1, 4;    add.u32 b2, %2, 4;\n\t"                       \
  "add.u32 a3, %1, 6;    add.u32 b3, %2, 6;\n\t"                       \
  "add.u32 a4, %1, 1024; add.u32 b4, %2, 1024;\n\t"                    \
  "add.u32 a5, %1, 1026; add.u32 b5, %2, 1026;\n\t"                    \
  "add.u32 a6, %1, 1028; add.u32 b6, %2, 1028;\n\t"                    \
  "add.u32 a7, %1, 1030; add.u32 b7, %2, 1030;\n\t"                    \
  "mov.b64 da0, {a0, %4}; mov.b64 db0, {b0, %4};\n\t"                  \
  "mov.b64 da1, {a1, %4}; mov.b64 db1, {b1, %4};\n\t"                  \
  "mov.b64 da2, {a2, %4}; mov.b64 db2, {b2, %4};\n\t"                  \
  "mov.b64 da3, {a3, %4}; mov.b64 db3, {b3, %4};\n\t"                  \
  "mov.b64 da4, {a4, %4}; mov.b64 db4, {b4, %4};\n\t"                  \
  "mov.b64 da5, {a5, %4}; mov.b64 db5, {b5, %4};\n\t"                  \
  "mov.b64 da6, {a6, %4}; mov.b64 db6, {b6, %4};\n\t"                  \
  "mov.b64 da7, {a7, %4}; mov.b64 db7, {b7, %4};\n\t"                  \
  P "tcgen05.mma.cta_group::1.kind::f16 [%0], da0, db0, %3, 0;\n\t"    \
  P "tcgen05.mma.cta_group::1.kind::f16 [%0], da1, db1, %3, 1;\n\t"    \
  P "tcgen05.mma.cta_group::1.kind::f16 [%0], da2, db2, %3, 1;\n\t"    \
  P "tcgen05.mma.cta_group::1.kind::f16 [%0], da3, db3, %3, 1;\n\t"    \
  P "tcgen05.mma.cta_group::1.kind::f16 [%0], da4, db4, %3, 1;\n\t"    \
  P "tcgen05.mma.cta_group::1.kind::f16 [%0], da5, db5, %3, 1;\n\t"    \
  P "tcgen05.mma.cta_group::1.kind::f16 [%0], da6, db6, %3, 1;\n\t"    \
  P "tcgen05.mma.cta_group::1.kind::f16 [%0], da7, db7, %3, 1;\n\t}"
template <bool W = false>
__device__ __forceinline__ void umma8_ss_kmajor(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo,
                                                uint32_t idesc) {
  if constexpr (W)
    asm volatile(CPATTN_UMMA8_SS_TEXT(CPATTN_ELECT_DECL, "@e ") ::"r"(d_tmem), "r"(a_lo),
                 "r"(b_lo), "r"(idesc), "n"(kDescHiSw128));
  else
    asm volatile(CPATTN_UMMA8_SS_TEXT("", "") ::"r"(d_tmem), "r"(a_lo), "r"(b_lo), "r"(idesc),
                 "n"(kDescHiSw128));
}

// Eight MMAs along K = 128 with A (16-bit, M x K) in tensor memory at column
// a_tmem + 8 k and B MN-major in shared memory, stepping b_lo by 128 (2 KiB,
// 16 K-rows) per MMA.  acc0 = 0: the first MMA overwrites D.
#define CPATTN_UMMA8_TS_MN_TEXT(DECL, P)                                \
  "{\n\t.reg .b32 b<8>, t<8>;\n\t.reg .b64 db<8>;\n\t" DECL            \
  "add.u32 b0, %2, 0;   add.u32 t0, %1, 0;\n\t"                        \
  "add.u32 b1, %2, 128; add.u32 t1, %1, 8;\n\t"                        \
  "add.u32 b2, %2, 256; add.u32 t2, %1, 16;\n\t"                       \
  "add.u32 b3, %2, 384; add.u32 t3, %1, 24;\n\t"                       \
  "add.u32 b4, %2, 512; add.u32 t4, %1, 32;\n\t"                       \
  "add.u32 b5, %2, 640; add.u32 t5, %1, 40;\n\t"                       \
  "add.u32 b6, %2, 768; add.u32 t6, %1, 48;\n\t"                       \
  "add.u32 b7, %2, 896; add.u32 t7, %1, 56;\n\t"                       \
  "mov.b64 db0, {b0, %4}; mov.b64 db1, {b1, %4};\n\t"                  \
  "mov.b64 db2, {b2, %4}; mov.b64 db3, {b3, %4};\n\t"                  \
  "mov.b64 db4, {b4, %4}; mov.b64 db5, {b5, %4};\n\t"                  \
  "mov.b64 db6, {b6, %4}; mov.b64 db7, {b7, %4};\n\t"                  \
  P "tcgen05.mma.cta_group::1.kind::f16 [%0], [t0], db0, %3, %5;\n\t"  \
  P "tcgen05.mma.cta_group::1.kind::f16 [%0], [t1], db1, %3, 1;\n\t"   \
  P "tcgen05.mma.cta_group::1.kind::f16 [%0], [t2], db2, %3, 1;\n\t"   \
  P "tcgen05.mma.cta_group::1.kind::f16 [%0], [t3], db3, %3, 1;\n\t"   \
  P "tcgen05.mma.cta_group::1.kind::f16 [%0], [t4], db4, %3, 1;\n\t"   \
  P "tcgen05.mma.cta_group::1.kind::f16 [%0], [t5], db5, %3, 1;\n\t"   \
  P "tcgen05.mma.cta_group::1.kind::f16 [%0], [t6], db6, %3, 1;\n\t"   \
  P "tcgen05.mma.cta_group::1.kind::f16 [%0], [t7], db7, %3, 1;\n\t}"
template <int ACC0, bool W = false>
__device__ __forceinline__ void umma8_ts_mnmajor(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo,
                                                 uint32_t idesc) {
  if constexpr (W)
    asm volatile(CPATTN_UMMA8_TS_MN_TEXT(CPATTN_ELECT_DECL, "@e ") ::"r"(d_tmem), "r"(a_tmem),
                 "r"(b_lo), "r"(idesc), "n"(kDescHiSw128), "n"(ACC0));
  else
    asm volatile(CPATTN_UMMA8_TS_MN_TEXT("", "") ::"r"(d_tmem), "r"(a_tmem), "r"(b_lo),
                 "r"(idesc), "n"(kDescHiSw128), "n"(ACC0));
}

// Four MMAs (K = 64) with both operands K-major in one 128-byte-swizzled
// 64-column box: steps advance both descriptors by 32 B (2 in >> 4 units).
#define CPATTN_UMMA4_SS_K_TEXT(DECL, P)                                 \
  "{\n\t.reg .b32 a<4>, b<4>;\n\t.reg .b64 da<4>, db<4>;\n\t" DECL     \
  "add.u32 a0, %1, 0; add.u32 b0, %2, 0;\n\t"                          \
  "add.u32 a1, %1, 2; add.u32 b1, %2, 2;\n\t"                          \
  "add.u32 a2, %1, 4; add.u32 b2, %2, 4;\n\t"                          \
  "add.u32 a3, %1, 6; add.u32 b3, %2, 6;\n\t"                          \
  "mov.b64 da0, {a0, %4}; mov.b64 db0, {b0, %4};\n\t"                  \
  "mov.b64 da1, {a1, %4}; mov.b64 db1, {b1, %4};\n\t"                  \
  "mov.b64 da2, {a2, %4}; mov.b64 db2, {b2, %4};\n\t"                  \
  "mov.b64 da3, {a3, %4}; mov.b64 db3, {b3, %4};\n\t"                  \
  P "tcgen05.mma.cta_group::1.kind::f16 [%0], da0, db0, %3, %5;\n\t"   \
  P "tcgen05.mma.cta_group::1.kind::f16 [%0], da1, db1, %3, 1;\n\t"    \
  P "tcgen05.mma.cta_group::1.kind::f16 [%0], da2, db2, %3, 1;\n\t"    \
  P "tcgen05.mma.cta_group::1.kind::f16 [%0], da3, db3, %3, 1;\n\t}"
template <int ACC0, bool W = false>
__device__ __forceinline__ void umma4_ss_k(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo,
                                           uint32_t idesc) {
  if constexpr (W)
    asm volatile(CPATTN_UMMA4_SS_K_TEXT(CPATTN_ELECT_DECL, "@e ") ::"r"(d_tmem), "r"(a_lo),
                 "r"(b_lo), "r"(idesc), "n"(kDescHiSw128), "n"(ACC0));
  else
    asm volatile(CPATTN_UMMA4_SS_K_TEXT("", "") ::"r"(d_tmem), "r"(a_lo), "r"(b_lo), "r"(idesc),
                 "n"(kDescHiSw128), "n"(ACC0));
}
// Four MMAs (K = 64) with A in tensor memory (columns a_tmem + 8 k) and B
// K-major in one swizzled box (b_lo + 2 k).
#define CPATTN_UMMA4_TS_K_TEXT(DECL, P)                                 \
  "{\n\t.reg .b32 b<4>, t<4>;\n\t.reg .b64 db<4>;\n\t" DECL            \
  "add.u32 b0, %2, 0; add.u32 t0, %1, 0;\n\t"                          \
  "add.u32 b1, %2, 2; add.u32 t1, %1, 8;\n\t"                          \
  "add.u32 b2, %2, 4; add.u32 t2, %1, 16;\n\t"                         \
  "add.u32 b3, %2, 6; add.u32 t3, %1, 24;\n\t"                         \
  "mov.b64 db0, {b0, %4}; mov.b64 db1, {b1, %4};\n\t"                  \
  "mov.b64 db2, {b2, %4}; mov.b64 db3, {b3, %4};\n\t"                  \
  P "tcgen05.mma.cta_group::1.kind::f16 [%0], [t0], db0, %3, %5;\n\t"  \
  P "tcgen05.mma.cta_group::1.kind::f16 [%0], [t1], db1, %3, 1;\n\t"   \
  P "tcgen05.mma.cta_group::1.kind::f16 [%0], [t2], db2, %3, 1;\n\t"   \
  P "tcgen05.mma.cta_group::1.kind::f16 [%0], [t3], db3, %3, 1;\n\t}"
template <int ACC0, bool W = false>
__device__ __forceinline__ void umma4_ts_k(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo,
                                           uint32_t idesc) {
  if constexpr (W)
    asm volatile(CPATTN_UMMA4_TS_K_TEXT(CPATTN_ELECT_DECL, "@e ") ::"r"(d_tmem), "r"(a_tmem),
                 "r"(b_lo), "r"(idesc), "n"(kDescHiSw128), "n"(ACC0));
  else
    asm volatile(CPATTN_UMMA4_TS_K_TEXT("", "") ::"r"(d_tmem), "r"(a_tmem), "r"(b_lo),
                 "r"(idesc), "n"(kDescHiSw128), "n"(ACC0));
}
// Four MMAs (K = 64) with A in tensor memory and B MN-major (16 K-rows =
// 2 KiB per step, b_lo + 128 k; leading offset carried in b_lo).
#define CPATTN_UMMA4_TS_MN_TEXT(DECL, P)                                \
  "{\n\t.reg .b32 b<4>, t<4>;\n\t.reg .b64 db<4>;\n\t" DECL            \
  "add.u32 b0, %2, 0;   add.u32 t0, %1, 0;\n\t"                        \
  "add.u32 b1, %2, 128; add.u32 t1, %1, 8;\n\t"                        \
  "add.u32 b2, %2, 256; add.u32 t2, %1, 16;\n\t"                       \
  "add.u32 b3, %2, 384; add.u32 t3, %1, 24;\n\t"                       \
  "mov.b64 db0, {b0, %4}; mov.b64 db1, {b1, %4};\n\t"                  \
  "mov.b64 db2, {b2, %4}; mov.b64 db3, {b3, %4};\n\t"                  \
  P "tcgen05.mma.cta_group::1.kind::f16 [%0], [t0], db0, %3, %5;\n\t"  \
  P "tcgen05.mma.cta_group::1.kind::f16 [%0], [t1], db1, %3, 1;\n\t"   \
  P "tcgen05.mma.cta_group::1.kind::f16 [%0], [t2], db2, %3, 1;\n\t"   \
  P "tcgen05.mma.cta_group::1.kind::f16 [%0], [t3], db3, %3, 1;\n\t}"
template <int ACC0, bool W = false>
__device__ __forceinline__ void umma4_ts_mn(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo,
                                            uint32_t idesc) {
  if constexpr (W)
    asm volatile(CPATTN_UMMA4_TS_MN_TEXT(CPATTN_ELECT_DECL, "@e ") ::"r"(d_tmem), "r"(a_tmem),
                 "r"(b_lo), "r"(idesc), "n"(kDescHiSw128), "n"(ACC0));
  else
    asm volatile(CPATTN_UMMA4_TS_MN_TEXT("", "") ::"r"(d_tmem), "r"(a_tmem), "r"(b_lo),
                 "r"(idesc), "n"(kDescHiSw128), "n"(ACC0));
}

// D[tmem] (+)= A[tmem] * B[smem]; A (M x K, 16-bit, two elements per 32-bit
// column, lane = row) is read from tensor memory.
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Per-warpgroup register budget (all four warps of a warpgroup execute it).
template <uint32_t N>
__device__ __forceinline__ void regs_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}
template <uint32_t N>
__device__ __forceinline__ void regs_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}

// Packed fp32 pairs (Blackwell f32x2 arithmetic) and the 3-input max.
__device__ __forceinline__ uint64_t f2_pack(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void f2_unpack(uint64_t r, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}
__device__ __forceinline__ uint64_t f2_fma(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t f2_add(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Hardware base-2 exponential (PTX ex2.approx.ftz.f32; -inf -> +0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Arrive once on `bar` when every tcgen05 op issued so far by this thread
// has completed.  W = true: the whole warp calls, the elected lane commits.
template <bool W = false>
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  if constexpr (W)
    asm volatile(
        "{\n\t" CPATTN_ELECT_DECL
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
            smem_u32(bar))
        : "memory");
  else
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

}  // namespace sm100
}  // namespace cpattn
