// Hand-written PTX wrappers for sm_103a: mbarrier, bulk/tensor async copies (TMA),
// tcgen05 (tensor memory allocation, MMA, loads/stores) and a few scalar helpers.
// Every wait loop is bounded: it gives up after a time limit read from %globaltimer and
// reports failure to the caller, which records QGEMM_ERR_TIMEOUT and winds down.
#pragma once

#include <stdint.h>

namespace qgemm {
namespace ptx {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t elect_one_sync() {
  uint32_t pred = 0;
  asm volatile(
      "{\n .reg .pred P;\n elect.sync _|P, %1;\n selp.b32 %0, 1, 0, P;\n}\n"
      : "=r"(pred) : "r"(0xffffffffu));
  return pred;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
               :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred P;\n mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n"
      " selp.b32 %0, 1, 0, P;\n}\n"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}

// try_wait that may suspend the thread for up to `hint_ns` while the phase is incomplete
// (it resumes as soon as the phase completes), so waiting warps do not take issue slots.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred P;\n mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2, %3;\n"
      " selp.b32 %0, 1, 0, P;\n}\n"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns) : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Returns false if the
// shared abort flag was raised or `limit_ns` elapsed; in the latter case raises the flag.
// Between polls the warp sleeps `sleep_ns`, so that waiting warps leave the issue slots
// to the warps doing arithmetic on the same sub-partition.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          volatile int* abort_flag, uint64_t limit_ns,
                                          uint32_t sleep_ns = 0) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  uint32_t spins = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (sleep_ns) __nanosleep(sleep_ns);
    if ((++spins & 15u) == 0) {
      if (*abort_flag) return false;
      if (globaltimer() - t0 > limit_ns) { *abort_flag = 1; return false; }
    }
  }
}

// ---------------------------------------------------------------- async copies
// 1-D bulk copy global -> shared, completion counted on `bar` (bytes % 16 == 0).
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;"
      :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy) : "memory");
}

// 16 bytes global -> shared through L2 only (cp.async.cg): the first src_bytes (0 or 16)
// come from src and the rest is zero-filled.  The bytes land in the generic proxy.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes,
                                            uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;"
               :: "r"(dst), "l"(src), "r"(src_bytes), "l"(policy) : "memory");
}

// The same with the shared and global addresses offset by compile-time byte counts (folded
// into the instruction), all 16 bytes from src.
template <int DOFF, int SOFF>
__device__ __forceinline__ void cp_async_16_at(uint32_t dst, const void* src, uint64_t policy) {
  asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0+%3], [%1+%4], 16, %2;"
               :: "r"(dst), "l"(src), "l"(policy), "n"(DOFF), "n"(SOFF) : "memory");
}

// Wait for every cp.async this thread has issued, committed or not.
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.wait_all;" ::: "memory");
}

// Arrive on bar once every cp.async this thread has issued so far has completed; the
// barrier's expected count includes this arrival (noinc).
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(smem_u32(bar)) : "memory");
}

// 2-D tiled tensor copy global -> shared (coordinates: c0 innermost, in elements).
__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, int32_t c0, int32_t c1,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;"
      :: "r"(smem_u32(dst)), "l"(tmap), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// 3-D tiled tensor copy global -> shared (coordinates innermost first, in elements).
__device__ __forceinline__ void tma_load_3d(void* dst, const void* tmap, int32_t c0, int32_t c1,
                                            int32_t c2, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;"
      :: "r"(smem_u32(dst)), "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)),
         "l"(policy) : "memory");
}

// 4-D tiled tensor copy global -> shared.
__device__ __forceinline__ void tma_load_4d(void* dst, const void* tmap, int32_t c0, int32_t c1,
                                            int32_t c2, int32_t c3, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;"
      :: "r"(smem_u32(dst)), "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(smem_u32(bar)),
         "l"(policy) : "memory");
}

__device__ __forceinline__ void prefetch_tmap(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" :: "l"(tmap) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_normal() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------- tcgen05
// Allocation (whole warp).  Writes the TMEM base address to *dst_smem.
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
               :: "r"(smem_u32(dst_smem)), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
               :: "r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T, BF16 inputs, FP32 accumulate (kind::f16).
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred P;\n setp.ne.b32 P, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, P;\n}\n"
      :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// Block-scaled FP8/FP6/FP4 MMA with A from tensor memory, one scale per 32 K (1X).
__device__ __forceinline__ void mma_mxf8f6f4_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc, uint32_t sfa_tmem,
                                                uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred P;\n setp.ne.b32 P, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], [%1], %2, %3, [%4], [%5], P;\n}\n"
      :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem),
         "r"(accumulate) : "memory");
}

// The same two MMAs and the commit below, executed by a whole converged warp: one lane
// (elect.sync) issues, the others only take part in the election.
__device__ __forceinline__ void mma_f16_ts_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                 uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred P, E;\n setp.ne.b32 P, %4, 0;\n elect.sync _|E, 0xffffffff;\n"
      " @E tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, P;\n}\n"
      :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}

// Four kind::f16 MMAs into one accumulator under a single election (the first accumulates
// when `accumulate` is non-zero, the other three always): one elect.sync instead of four.
__device__ __forceinline__ void mma4_f16_ts_elect(uint32_t d_tmem, uint32_t a0, uint32_t a1,
                                                  uint32_t a2, uint32_t a3, uint64_t b0,
                                                  uint64_t b1, uint64_t b2, uint64_t b3,
                                                  uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred P, Q, E;\n setp.ne.b32 P, %10, 0;\n setp.eq.b32 Q, %10, %10;\n"
      " elect.sync _|E, 0xffffffff;\n"
      " @E tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %5, %9, P;\n"
      " @E tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], %6, %9, Q;\n"
      " @E tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %7, %9, Q;\n"
      " @E tcgen05.mma.cta_group::1.kind::f16 [%0], [%4], %8, %9, Q;\n}\n"
      :: "r"(d_tmem), "r"(a0), "r"(a1), "r"(a2), "r"(a3), "l"(b0), "l"(b1), "l"(b2), "l"(b3),
         "r"(idesc), "r"(accumulate) : "memory");
}

__device__ __forceinline__ void mma_mxf8f6f4_ts_elect(uint32_t d_tmem, uint32_t a_tmem,
                                                      uint64_t b_desc, uint32_t idesc,
                                                      uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                      uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred P, E;\n setp.ne.b32 P, %6, 0;\n elect.sync _|E, 0xffffffff;\n"
      " @E tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], [%1], %2, %3, [%4], [%5], P;\n}\n"
      :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem),
         "r"(accumulate) : "memory");
}

// Block-scaled FP4 x FP4 MMA (kind::mxf4, one E8M0 scale per 32 K: scale_vec::2X with K = 64
// per instruction), A and B from shared memory, under one election of a converged warp.
__device__ __forceinline__ void mma_mxf4_ss_elect(uint32_t d_tmem, uint64_t a_desc,
                                                  uint64_t b_desc, uint32_t idesc,
                                                  uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                  uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred P, E;\n setp.ne.b32 P, %6, 0;\n elect.sync _|E, 0xffffffff;\n"
      " @E tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X"
      " [%0], %1, %2, %3, [%4], [%5], P;\n}\n"
      :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem),
         "r"(accumulate) : "memory");
}

// Block-scaled FP8/FP6/FP4 MMA (kind::mxf8f6f4, one E8M0 scale per 32 K) with A and B from
// shared memory, under one election of a converged warp.
__device__ __forceinline__ void mma_mxf8f6f4_ss_elect(uint32_t d_tmem, uint64_t a_desc,
                                                      uint64_t b_desc, uint32_t idesc,
                                                      uint32_t sfa_tmem, uint32_t sfb_tmem,
                                                      uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred P, E;\n setp.ne.b32 P, %6, 0;\n elect.sync _|E, 0xffffffff;\n"
      " @E tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X"
      " [%0], %1, %2, %3, [%4], [%5], P;\n}\n"
      :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem),
         "r"(accumulate) : "memory");
}

__device__ __forceinline__ void mma_commit_elect(uint64_t* bar) {
  asm volatile(
      "{\n .reg .pred E;\n elect.sync _|E, 0xffffffff;\n"
      " @E tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n"
      :: "r"(smem_u32(bar)) : "memory");
}

// Arrive on `bar` once every previously issued tcgen05.mma of this thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
      :: "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 bits, 32 consecutive columns per thread.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10,"
      " %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27,"
      " %28, %29, %30, %31, %32};"
      :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
         "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
         "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]),
         "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
         "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" :: "r"(taddr), "r"(v)
               : "memory");
}

__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c,
                                         uint32_t d) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};"
               :: "r"(taddr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10,"
      " %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27,"
      " %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
        "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
        "=r"(r[31])
      : "r"(taddr) : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10,"
      " %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr) : "memory");
}

// Shared-memory matrix descriptor for tcgen05.mma: K-major operand, 128-byte swizzle,
// 8-row core groups 1024 bytes apart.  `smem_addr` must lie in a 1024-byte aligned atom
// (a K offset inside the 128-byte row is added to the start address).
__device__ __forceinline__ uint64_t desc_kmajor_sw128(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= uint64_t((smem_addr & 0x3FFFFu) >> 4);        // start address, 16-byte units
  d |= uint64_t(1) << 16;                            // leading byte offset (unused here)
  d |= uint64_t(1024 >> 4) << 32;                    // stride byte offset: 8 rows x 128 B
  d |= uint64_t(1) << 46;                            // descriptor version for tcgen05
  d |= uint64_t(2) << 61;                            // swizzle: 128-byte
  return d;
}

// Shared-memory matrix descriptor: K-major operand, 64-byte swizzle (rows of 64 bytes,
// 8-row atoms of 512 bytes at 512-byte strides); `smem_addr` in a 512-byte aligned atom plus
// a K offset inside the row.
__device__ __forceinline__ uint64_t desc_kmajor_sw64(uint32_t smem_addr) {
  uint64_t d = 0;
  d |= uint64_t((smem_addr & 0x3FFFFu) >> 4);        // start address, 16-byte units
  d |= uint64_t(1) << 16;                            // leading byte offset (unused here)
  d |= uint64_t(512 >> 4) << 32;                     // stride byte offset: 8 rows x 64 B
  d |= uint64_t(1) << 46;                            // descriptor version for tcgen05
  d |= uint64_t(4) << 61;                            // swizzle: 64-byte
  return d;
}

// Instruction descriptor, kind::mxf4: D=F32, A=B=E2M1 (format code 1), K-major, scale
// factors UE8M0 with selectors sfa_id / sfb_id (0 or 2: the byte pair of each 64-K step).
__host__ __device__ constexpr uint32_t idesc_mxf4(int M, int N, int sfa_id, int sfb_id) {
  return (uint32_t(sfb_id & 3) << 4) | (1u << 7) | (1u << 10) | (uint32_t(N >> 3) << 17) |
         (1u << 23) | (uint32_t(M >> 4) << 24) | (uint32_t(sfa_id & 3) << 29);
}

// Instruction descriptor, kind::f16: D=F32, A=B=BF16, both K-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// Instruction descriptor, kind::f16: D=F32, A=B=FP16, both K-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N) {
  return (1u << 4) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// Instruction descriptor, kind::mxf8f6f4: D=F32, A=B=E4M3, scale factors UE8M0 with byte
// selectors sfa_id / sfb_id, shape M x N.
__host__ __device__ constexpr uint32_t idesc_mxf8_e4m3(int M, int N, int sfa_id, int sfb_id) {
  return (uint32_t(sfb_id & 3) << 4) | (0u << 7) | (0u << 10) | (uint32_t(N >> 3) << 17) |
         (1u << 23) | (uint32_t(M >> 4) << 24) | (uint32_t(sfa_id & 3) << 29);
}

// Instruction descriptor, kind::mxf8f6f4: D=F32, A=E2M1 (format code 5), B=E4M3 (0), scale
// factors UE8M0 with byte selectors sfa_id / sfb_id, shape M x N.  The e2m1 operand sits in
// shared memory in the padded form (16 elements in the first 8 of every 16 bytes).
__host__ __device__ constexpr uint32_t idesc_mxf8_e2m1_e4m3(int M, int N, int sfa_id, int sfb_id) {
  return (uint32_t(sfb_id & 3) << 4) | (5u << 7) | (0u << 10) | (uint32_t(N >> 3) << 17) |
         (1u << 23) | (uint32_t(M >> 4) << 24) | (uint32_t(sfa_id & 3) << 29);
}

// ---------------------------------------------------------------- scalar helpers
// Two floats rounded to the nearest BF16 (ties to even), `lo` in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

// prmt.b32 (default mode): result byte i is byte (c >> 4i) & 7 of {b, a} (a the low word);
// when bit 3 of that selector nibble is set, the byte is replaced by copies of its sign bit.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// Two E4M3 codes (the low byte first) -> f16x2 (exact), by the hardware conversion.
__device__ __forceinline__ uint32_t cvt_f16x2_e4m3x2(uint32_t pair) {
  uint32_t r;
  const unsigned short p16 = static_cast<unsigned short>(pair & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(p16));
  return r;
}

// Byte B of w (two e2m1 codes, the low nibble first) -> f16x2 (exact), by the hardware
// conversion.
template <int B>
__device__ __forceinline__ uint32_t cvt_f16x2_e2m1x2(uint32_t w) {
  static_assert(B >= 0 && B < 4, "byte index");
  uint32_t r;
  if constexpr (B == 0)
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b0;\n}\n" : "=r"(r) : "r"(w));
  else if constexpr (B == 1)
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b1;\n}\n" : "=r"(r) : "r"(w));
  else if constexpr (B == 2)
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b2;\n}\n" : "=r"(r) : "r"(w));
  else
    asm("{\n .reg .b8 b0, b1, b2, b3;\n mov.b32 {b0, b1, b2, b3}, %1;\n cvt.rn.f16x2.e2m1x2 %0, b3;\n}\n" : "=r"(r) : "r"(w));
  return r;
}

__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t f16x2_sub(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t f16x2_mul(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// Two floats rounded to the nearest FP16 (ties to even), `lo` in the low half.
__device__ __forceinline__ uint32_t cvt_f16x2_f32(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
// Wait until the grids this launch depends on (programmatic dependent launch) have
// completed and their memory is visible; returns at once when there are none.
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t mask, uint32_t orv) {
  // (a & mask) | orv in one LOP3 (immediate truth table 0xEA = (A & B) | C).
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(mask), "r"(orv));
  return d;
}
__device__ __forceinline__ uint32_t cvt_bf16x2_f32(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
// Two floats rounded to e2m1 (nearest even, saturating at +-6): `lo` in the low nibble.
__device__ __forceinline__ uint32_t cvt_e2m1x2_f32(float lo, float hi) {
  uint32_t d;
  asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n cvt.u32.u8 %0, t;\n}\n"
      : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ uint16_t cvt_e4m3x2_f32(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

}  // namespace ptx
}  // namespace qgemm
