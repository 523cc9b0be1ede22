// tc.cuh -- Blackwell (sm_103a) building blocks: mbarriers with bounded waits,
// tensor memory (TMEM) allocation and loads/stores, tcgen05.mma on operands
// in shared memory, and distributed shared memory within a CTA cluster.
#pragma once

#include "common.cuh"

namespace skv {
namespace tc {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---- mbarriers ----------------------------------------------------------------
__device__ __forceinline__ void bar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

__device__ __forceinline__ void bar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Arrive on the barrier at the same offset in the shared memory of CTA `rank`
// of the cluster (release at cluster scope: earlier remote stores are visible
// to a thread that observes the phase flip with cluster-scope acquire).
__device__ __forceinline__ void bar_arrive_remote(uint64_t* bar, uint32_t rank) {
  asm volatile(
      "{\n.reg .b32 ra;\nmapa.shared::cluster.u32 ra, %0, %1;\n"
      "mbarrier.arrive.release.cluster.shared::cluster.b64 _, [ra];\n}\n" ::"r"(smem_addr(bar)),
      "r"(rank)
      : "memory");
}

// Relaxed variant: only signals, orders nothing (for "buffer consumed" notes
// whose reads have already completed).
__device__ __forceinline__ void bar_arrive_remote_relaxed(uint64_t* bar, uint32_t rank) {
  asm volatile(
      "{\n.reg .b32 ra;\nmapa.shared::cluster.u32 ra, %0, %1;\n"
      "mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [ra];\n}\n" ::"r"(smem_addr(bar)),
      "r"(rank)
      : "memory");
}

__device__ __forceinline__ bool bar_test(uint64_t* bar, uint32_t parity, bool cluster_scope) {
  uint32_t ok;
  if (cluster_scope)
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
  else
    asm volatile(
        "{\n.reg .pred p;\nmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity to complete.  Gives up
// after `limit_ns` of wall time (or at once when *abort is set), sets *abort
// and returns false; the caller then skips its remaining work.
__device__ __forceinline__ bool bar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                         bool cluster_scope = false, uint64_t limit_ns = 2000000000ull) {
  if (bar_test(bar, parity, cluster_scope)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t it = 1;; it++) {
    if (bar_test(bar, parity, cluster_scope)) return true;
    if ((it & 63) == 0) {
      if (*abort) return false;
      if (global_ns() - t0 > limit_ns) {
        *abort = 1;
        return false;
      }
    }
  }
}

// Bounded wait that ignores the abort flag (used to drain in-flight work).
__device__ __forceinline__ bool bar_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = global_ns();
  for (uint32_t it = 0;; it++) {
    if (bar_test(bar, parity, false)) return true;
    if ((it & 63) == 63 && global_ns() - t0 > limit_ns) return false;
  }
}

// Generic-proxy shared-memory writes -> visible to the tensor core's async proxy.
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// ---- cluster ------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\nbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// 16-byte store into the shared memory of CTA `rank` (same offset as `local`).
__device__ __forceinline__ void st_remote16(const void* local, uint32_t rank, float4 v) {
  asm volatile(
      "{\n.reg .b32 ra;\nmapa.shared::cluster.u32 ra, %0, %1;\n"
      "st.shared::cluster.v4.f32 [ra], {%2, %3, %4, %5};\n}\n" ::"r"(smem_addr(local)),
      "r"(rank), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
      : "memory");
}

// Loads from CTA `rank`'s shared memory at the same offset as `local`.
__device__ __forceinline__ float4 ld_remote16(const void* local, uint32_t rank) {
  float4 v;
  asm volatile(
      "{\n.reg .b32 ra;\nmapa.shared::cluster.u32 ra, %4, %5;\n"
      "ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [ra];\n}\n"
      : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
      : "r"(smem_addr(local)), "r"(rank)
      : "memory");
  return v;
}
__device__ __forceinline__ float ld_remote_f32(const void* local, uint32_t rank) {
  float v;
  asm volatile("{\n.reg .b32 ra;\nmapa.shared::cluster.u32 ra, %1, %2;\nld.shared::cluster.f32 %0, [ra];\n}\n"
               : "=f"(v)
               : "r"(smem_addr(local)), "r"(rank)
               : "memory");
  return v;
}

// Asynchronous 16-byte store into CTA `rank`'s shared memory (same offset as
// `local`); on arrival it completes 16 bytes of transaction count on that
// CTA's barrier at the offset of `local_bar`.  No fence is needed: the data is
// visible to threads that observe the barrier's phase completion.
__device__ __forceinline__ void st_async_remote16(const void* local, const uint64_t* local_bar, uint32_t rank,
                                                  float4 v) {
  asm volatile(
      "{\n.reg .b32 ra, rb;\nmapa.shared::cluster.u32 ra, %0, %2;\nmapa.shared::cluster.u32 rb, %1, %2;\n"
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [ra], {%3, %4, %5, %6}, [rb];\n}\n" ::"r"(
          smem_addr(local)),
      "r"(smem_addr(local_bar)), "r"(rank), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
      : "memory");
}

// Bulk copy of `bytes` (multiple of 16) from this CTA's shared memory at
// `src` to the same offset as `dst_local` in CTA `rank`'s shared memory; on
// arrival it completes `bytes` of transaction count on that CTA's barrier at
// the offset of `bar_local`.  Issued by one thread; commit_bulk() closes the
// group and wait_bulk_read() waits until the source may be overwritten.
__device__ __forceinline__ void bulk_copy_to_peer(const void* dst_local, const void* src, uint32_t bytes,
                                                  const uint64_t* bar_local, uint32_t rank) {
  asm volatile(
      "{\n.reg .b32 rd, rb;\nmapa.shared::cluster.u32 rd, %0, %3;\nmapa.shared::cluster.u32 rb, %2, %3;\n"
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [rd], [%1], %4, [rb];\n}\n" ::"r"(
          smem_addr(dst_local)),
      "r"(smem_addr(src)), "r"(smem_addr(bar_local)), "r"(rank), "r"(bytes)
      : "memory");
}
// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// global memory into this CTA's shared memory, completion counted on `bar`.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned) from
// this CTA's shared memory to global memory (bulk-group completion).
__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_addr(src)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void commit_bulk() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void wait_bulk_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void wait_bulk_done() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Arrive on a local barrier and add `bytes` to the transaction count its
// current phase waits for.
__device__ __forceinline__ void bar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

// ---- tensor memory ------------------------------------------------------------
// Whole warp: allocate `ncols` columns (power of two >= 32); the base address is
// written to *dst (shared memory).
template <int NCOLS>
__device__ __forceinline__ void tmem_alloc(uint32_t* dst) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)),
               "n"(NCOLS));
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}

template <int NCOLS>
__device__ __forceinline__ void tmem_dealloc(uint32_t base) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(base), "n"(NCOLS));
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive 32-bit columns of this thread's lane (warp w reads lanes
// 32*(w%4) .. +31; `taddr` carries that lane base in bits 31:16).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
      "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
      "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---- tcgen05.mma ----------------------------------------------------------------
// Shared-memory matrix descriptor, 128-byte swizzle: rows of 128 bytes, the
// 16-byte chunk c of row r stored at chunk c ^ (r % 8), 8-row groups of 1024
// bytes (1024-byte aligned).  K-major operands: `sbo` = 8-row group stride
// (lbo unused).  MN-major operands: `lbo` = stride between 64-element column
// blocks, `sbo` = stride between 8-row (K) groups.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;  // descriptor version
  d |= 2ull << 61;  // 128-byte swizzle
  return d;
}

// Instruction descriptor, kind::f16: fp16 A and B, fp32 accumulator, A
// K-major, B K-major (b_mn = 0) or MN-major (b_mn = 1), M x N.
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, int b_mn) {
  return (1u << 4) | (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// One elected thread: D[tmem] (+)= A[smem] . B[smem].
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                        bool accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1 : 0));
}

// One elected thread: D[tmem] (+)= A[tmem] . B[smem].  A in tensor memory:
// lane i holds row i, 32-bit column c holds elements 2c (low half) and 2c + 1
// (high half) of the K dimension.
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           bool accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate ? 1 : 0));
}

// The barrier's phase completes when every earlier tcgen05 operation of this
// thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}

// 2^x on the special-function unit (approximate, flushes subnormals; 2^-inf = 0).
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two fp8 e4m3 values (a 16-bit pair) -> two fp16 values, exact.
__device__ __forceinline__ uint2 e4m3x4_to_f16x4(uint32_t x) {
  uint32_t lo, hi;
  asm("{\n.reg .b16 a, b;\nmov.b32 {a, b}, %2;\ncvt.rn.f16x2.e4m3x2 %0, a;\ncvt.rn.f16x2.e4m3x2 %1, b;\n}\n"
      : "=r"(lo), "=r"(hi)
      : "r"(x));
  return make_uint2(lo, hi);
}

}  // namespace tc
}  // namespace skv
