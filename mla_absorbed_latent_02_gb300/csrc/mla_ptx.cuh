// Inline-PTX building blocks for the sm_103a kernels: mbarriers with bounded
// waits, TMA tensor loads, and the tcgen05 (5th-generation tensor core) MMA,
// TMEM allocation and TMEM load/store instructions.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#define MLA_DEV __device__ __forceinline__

// Device status bits (OR-ed into the context's status word).
#define MLA_DEVERR_BOUNDS 1
#define MLA_DEVERR_TIMEOUT 2
#define MLA_DEVERR_LENGTH 4

// Every spin on an mbarrier gives up after this many nanoseconds.
#ifndef MLA_WAIT_TIMEOUT_NS
#define MLA_WAIT_TIMEOUT_NS 2000000000ull
#endif

namespace mla {

MLA_DEV uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

MLA_DEV uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
MLA_DEV void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
MLA_DEV void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
MLA_DEV void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
MLA_DEV void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
MLA_DEV bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking probe (mbarrier.test_wait): never suspends the thread, for
// loops that poll several barriers and act on whichever is ready. (try_wait,
// above, may park the thread for a while when the phase is incomplete.)
MLA_DEV bool mbar_probe(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with parity `parity` to complete. `abort` is a
// CTA-shared flag: once any waiter of the CTA gives up, every other waiter
// stops too. On timeout the status word gets MLA_DEVERR_TIMEOUT.
MLA_DEV bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort, int* status) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_test(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > MLA_WAIT_TIMEOUT_NS) {
      *abort = 1;
      atomicOr(status, MLA_DEVERR_TIMEOUT);
      return false;
    }
  }
}

// Same, with an explicit limit (used to drain in-flight copies on abort).
MLA_DEV bool mbar_wait_ns(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer();
  while (!mbar_test(bar, parity))
    if (globaltimer() - t0 > limit_ns) return false;
  return true;
}

// ---------------------------------------------------------------------------
// fences
// ---------------------------------------------------------------------------
// Generic-proxy shared-memory writes -> visible to the async proxy (TMA, MMA).
MLA_DEV void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
MLA_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
MLA_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

MLA_DEV void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor), completion counted on an mbarrier
// ---------------------------------------------------------------------------
MLA_DEV void tma_prefetch_desc(const void* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}
MLA_DEV void tma_load_2d(uint32_t dst, const void* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
MLA_DEV void tma_load_2d_hint(uint32_t dst, const void* map, uint32_t bar, int x, int y,
                              uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(map), "r"(bar), "r"(x), "r"(y), "l"(policy)
      : "memory");
}
MLA_DEV void tma_load_3d(uint32_t dst, const void* map, uint32_t bar, int x, int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(x), "r"(y), "r"(z)
      : "memory");
}
// ---------------------------------------------------------------------------
// thread-block clusters: rank, distributed shared memory, cluster barrier
// ---------------------------------------------------------------------------
// Address of the same shared-memory location in CTA `rank` of the cluster.
MLA_DEV uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// Bulk copy of `bytes` from this CTA's shared memory to `dst` in a CTA of the
// cluster; the bytes are counted on the mbarrier `bar` of that CTA.
MLA_DEV void bulk_copy_to_cluster(uint32_t dst, uint32_t src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "r"(src), "r"(bytes), "r"(bar)
      : "memory");
}
MLA_DEV void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Waits until the committed bulk copies have read their source.
MLA_DEV void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Every thread of every CTA of the cluster; shared-memory writes before it are
// visible to the cluster's reads after it.
MLA_DEV void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Bulk prefetch of [src, src + bytes) into L2 (a hint: no shared memory, no completion).
MLA_DEV void prefetch_l2_bulk(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
MLA_DEV uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
MLA_DEV uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ---------------------------------------------------------------------------
// tcgen05: TMEM allocation, MMA, commit, TMEM <-> registers
// ---------------------------------------------------------------------------
// Whole warp; writes the TMEM base address to shared memory at `dst`.
MLA_DEV void tmem_alloc(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst),
               "r"(ncols)
               : "memory");
}
MLA_DEV void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
MLA_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading and
// stride byte offsets (16-byte units), version 1 at bit 46, layout at bits 61-63.
enum : uint32_t { SMEM_SWIZZLE_NONE = 0, SMEM_SWIZZLE_128B = 2, SMEM_SWIZZLE_64B = 4, SMEM_SWIZZLE_32B = 6 };

MLA_DEV uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes,
                           uint32_t layout) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(layout & 7u) << 61;
  return d;
}

// Instruction descriptor for kind::f16 with bf16 A/B and fp32 accumulation.
// a_mn / b_mn: 1 when that operand is MN-major in shared memory.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N, uint32_t a_mn,
                                                      uint32_t b_mn) {
  return (1u << 4)              // D = f32
         | (1u << 7)            // A = bf16
         | (1u << 10)           // B = bf16
         | (a_mn << 15) | (b_mn << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
MLA_DEV void mma_bf16_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// kind::f8f6f4 with both operands e4m3 (type fields 0) and an f32 accumulator;
// one MMA covers K = 32 (32 bytes of a K-major row, as K = 16 does for bf16).
__host__ __device__ constexpr uint32_t idesc_e4m3_f32(uint32_t M, uint32_t N, uint32_t a_mn,
                                                      uint32_t b_mn) {
  return (1u << 4)              // D = f32
         | (0u << 7)            // A = e4m3
         | (0u << 10)           // B = e4m3
         | (a_mn << 15) | (b_mn << 16) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

MLA_DEV void mma_e4m3_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The mbarrier receives one arrival when every tcgen05 operation this thread
// issued before has completed.
MLA_DEV void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns: thread i of the warp gets lane
// (32*(warp%4) + i) of the TMEM address's lane quarter, columns col..col+15.
MLA_DEV void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
MLA_DEV void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}
MLA_DEV void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}
MLA_DEV void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
MLA_DEV void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
MLA_DEV void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Pins registers written by tcgen05.ld after the wait: uses cannot move above.
MLA_DEV void reg_fence16(uint32_t (&r)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) asm volatile("" : "+r"(r[i]));
}
// W (8 or 16) consecutive 32-bit columns of this thread's TMEM lane.
template <int W>
MLA_DEV void tmem_ld_w(uint32_t taddr, uint32_t* r) {
  static_assert(W == 8 || W == 16, "8 or 16 columns");
  if constexpr (W == 16) tmem_ld16(taddr, *reinterpret_cast<uint32_t(*)[16]>(r));
  else tmem_ld8(taddr, *reinterpret_cast<uint32_t(*)[8]>(r));
}
template <int W>
MLA_DEV void tmem_st_w(uint32_t taddr, const uint32_t* r) {
  static_assert(W == 8 || W == 16, "8 or 16 columns");
  if constexpr (W == 16) tmem_st16(taddr, *reinterpret_cast<const uint32_t(*)[16]>(r));
  else tmem_st8(taddr, *reinterpret_cast<const uint32_t(*)[8]>(r));
}
template <int W>
MLA_DEV void reg_fence_w(uint32_t* r) {
#pragma unroll
  for (int i = 0; i < W; ++i) asm volatile("" : "+r"(r[i]));
}

// ---------------------------------------------------------------------------
// CTA pairs (tcgen05 .cta_group::2): two CTAs of a cluster share one MMA. The
// even CTA of the pair issues it; A rows 0..127 come from its shared memory and
// rows 128..255 from the peer's, at the same offset; B's N columns are split in
// halves the same way; D rows land in each CTA's own tensor memory. Every
// tcgen05 instruction of a kernel that uses pairs carries .cta_group::2.
// ---------------------------------------------------------------------------
MLA_DEV uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// One warp of each CTA of the pair, together: the same columns in both CTAs.
MLA_DEV void tmem_alloc_pair(uint32_t dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst), "r"(ncols)
               : "memory");
}
MLA_DEV void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
MLA_DEV void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
MLA_DEV void mma_bf16_ss_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                              uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// One arrival on the mbarrier at offset `bar` of every CTA in `mask` once the
// pair MMAs issued so far have completed.
MLA_DEV void mma_commit_pair(uint32_t bar, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(mask)
      : "memory");
}
// TMA load into this CTA's shared memory whose bytes are counted on an mbarrier
// of either CTA of the pair (`bar` a shared::cluster address).
MLA_DEV void tma_load_2d_pair(uint32_t dst, const void* map, uint32_t bar, int x, int y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(map), "r"(bar), "r"(x), "r"(y)
      : "memory");
}
// Asynchronous stores into another CTA's shared memory (`cluster_addr`); the
// bytes are counted (complete_tx) on that CTA's mbarrier `cluster_bar`. The
// issuing thread does not wait for them.
MLA_DEV void st_async_v4(uint32_t cluster_addr, uint32_t cluster_bar, uint32_t a, uint32_t b, uint32_t c,
                         uint32_t d) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1,%2,%3,%4}, [%5];" ::"r"(
                   cluster_addr),
               "r"(a), "r"(b), "r"(c), "r"(d), "r"(cluster_bar)
               : "memory");
}
MLA_DEV void st_async_u32(uint32_t cluster_addr, uint32_t cluster_bar, uint32_t v) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(cluster_addr), "r"(v),
               "r"(cluster_bar)
               : "memory");
}
// try_wait with acquire at cluster scope: the phase was completed by arrivals
// of another CTA whose earlier writes must be visible here.
MLA_DEV bool mbar_test_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
MLA_DEV bool mbar_wait_cluster(uint32_t bar, uint32_t parity, volatile int* abort, int* status) {
  if (mbar_test_cluster(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_test_cluster(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > MLA_WAIT_TIMEOUT_NS) {
      *abort = 1;
      atomicOr(status, MLA_DEVERR_TIMEOUT);
      return false;
    }
  }
}

// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialization attribute may start while the previous kernel in the
// stream is still running. pdl_wait() blocks until that kernel has completed and
// its memory is visible; every kernel calls it before its first global-memory
// access. pdl_trigger() lets the next kernel start its own set-up early.
MLA_DEV void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
MLA_DEV void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

MLA_DEV uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t v;
  asm("cvt.rn.bf16x2.f32 %0, %2, %1;" : "=r"(v) : "f"(lo), "f"(hi));
  return v;
}

MLA_DEV float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace mla
