// tc_ptx.cuh -- inline-PTX wrappers shared by the tensor-core kernels:
// mbarriers with bounded waits, TMA tensor loads, tcgen05 MMA / commit /
// TMEM load and store, the 128-byte-swizzle shared-memory descriptor and the
// kind::f16 instruction descriptor, and packed f32x2 arithmetic.
#pragma once
#include <stdint.h>

#include <cuda.h>

#include "common.cuh"

namespace attn {
namespace tc {

constexpr uint64_t kTimeoutNs = 2000000000ull;

// ---- PTX wrappers ------------------------------------------------------------------

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the phase with parity `parity` (acquire on success).
// Its result returns after the shared-memory round trip (~200 cycles), so a
// test issued a batch of MMAs ahead of its use costs no wait at the use.
__device__ __forceinline__ bool mbar_test(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase of `b` with parity `parity`.
__device__ __forceinline__ bool wait_bar(uint64_t* b, uint32_t parity, int* abort_flag, int* status) {
  if (mbar_try(b, parity)) return true;
  const uint64_t t0 = gtimer();
  while (!mbar_try(b, parity)) {
    if (*(volatile int*)abort_flag) return false;
    if (gtimer() - t0 > kTimeoutNs) {
      *(volatile int*)abort_flag = 1;
      atomicExch(status, ATTN_ERR_DEVICE_TIMEOUT);
      return false;
    }
  }
  return true;
}

// Teardown wait: bounded, does not look at the abort flag.
__device__ __forceinline__ bool drain_bar(uint64_t* b, uint32_t parity, int* status) {
  const uint64_t t0 = gtimer();
  while (!mbar_try(b, parity)) {
    if (gtimer() - t0 > kTimeoutNs) {
      atomicExch(status, ATTN_ERR_DEVICE_TIMEOUT);
      return false;
    }
  }
  return true;
}

// Warp-uniform bounded wait: every lane waits, and the warp proceeds only if
// all lanes saw the phase complete, so warp-collective TMEM instructions that
// follow never run with part of the warp.
__device__ __forceinline__ bool wait_warp(uint64_t* b, uint32_t parity, int* abort_flag, int* status) {
  const bool ok = wait_bar(b, parity, abort_flag, status);
  return __all_sync(0xffffffffu, ok);
}

// Warp-uniform bounded wait that skips the barrier round trip when an earlier
// non-blocking test (`ready`) already saw the phase complete in every lane.
__device__ __forceinline__ bool wait_ready(bool ready, uint64_t* b, uint32_t parity, int* abort_flag, int* status) {
  if (__all_sync(0xffffffffu, ready)) return true;
  return wait_warp(b, parity, abort_flag, status);
}

// ---- CTA pairs (a 2-CTA cluster sharing tcgen05 work, cta_group::2) ----

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of both CTAs: arrive, then wait for the whole cluster.
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// The same with a relaxed arrival: it orders none of the thread's earlier
// memory operations (nor waits for its loads in flight).
__device__ __forceinline__ void cluster_sync_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive (release at cluster scope) on the barrier at the same offset in CTA `rank` of the cluster.
__device__ __forceinline__ void mbar_arrive_remote(uint64_t* local_bar, uint32_t rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(su32(local_bar)), "r"(rank));
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(ra) : "memory");
}
// The same arrival without release semantics: it orders nothing by itself.
__device__ __forceinline__ void mbar_arrive_remote_relaxed(uint64_t* local_bar, uint32_t rank) {
  uint32_t ra;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(su32(local_bar)), "r"(rank));
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(ra) : "memory");
}
// Phase tests with acquire at cluster scope: for barriers that other CTAs
// of the cluster (or their tensor cores) arrive on.
__device__ __forceinline__ bool mbar_try_cl(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool mbar_test_cl(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool wait_bar_cl(uint64_t* b, uint32_t parity, int* abort_flag, int* status) {
  if (mbar_try_cl(b, parity)) return true;
  const uint64_t t0 = gtimer();
  while (!mbar_try_cl(b, parity)) {
    if (*(volatile int*)abort_flag) return false;
    if (gtimer() - t0 > kTimeoutNs) {
      *(volatile int*)abort_flag = 1;
      atomicExch(status, ATTN_ERR_DEVICE_TIMEOUT);
      return false;
    }
  }
  return true;
}
__device__ __forceinline__ bool drain_bar_cl(uint64_t* b, uint32_t parity, int* status) {
  const uint64_t t0 = gtimer();
  while (!mbar_try_cl(b, parity)) {
    if (gtimer() - t0 > kTimeoutNs) {
      atomicExch(status, ATTN_ERR_DEVICE_TIMEOUT);
      return false;
    }
  }
  return true;
}
__device__ __forceinline__ bool wait_warp_cl(uint64_t* b, uint32_t parity, int* abort_flag, int* status) {
  const bool ok = wait_bar_cl(b, parity, abort_flag, status);
  return __all_sync(0xffffffffu, ok);
}
__device__ __forceinline__ bool wait_ready_cl(bool ready, uint64_t* b, uint32_t parity, int* abort_flag,
                                              int* status) {
  if (__all_sync(0xffffffffu, ready)) return true;
  return wait_warp_cl(b, parity, abort_flag, status);
}

// Contiguous bulk copy global -> shared, completing on `bar` (both addresses
// 16-byte aligned, `bytes` a multiple of 16).
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   su32(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(su32(bar))
               : "memory");
}

// Fetch a tensor map (a __grid_constant__ kernel parameter) ahead of its first copy.
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1, int c2,
                                            int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], "
      "[%6];" ::"r"(su32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(su32(bar))
      : "memory");
}

// Tiled store of one tensor-map box from shared memory to global memory,
// tracked by the issuing thread's bulk async-group.  Elements of the box
// outside the tensor's extent are not written.
__device__ __forceinline__ void tma_store_4d(const CUtensorMap* map, const void* src, int c0, int c1, int c2, int c3) {
  asm volatile("cp.async.bulk.tensor.4d.global.shared::cta.bulk_group [%0, {%2, %3, %4, %5}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(su32(src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}
// Close the issuing thread's bulk group and wait until its stores have read
// their shared-memory source (the writes to global memory complete on their own).
__device__ __forceinline__ void bulk_store_commit_wait_read() {
  asm volatile("cp.async.bulk.commit_group;\n\tcp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Prefetch of one tensor-map box into L2 (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_4d(const CUtensorMap* map, int c0, int c1, int c2, int c3) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(c0), "r"(c1), "r"(c2), "r"(c3)
               : "memory");
}

__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// Warp-wide forms: every lane of a converged warp executes the statement and
// elect.sync picks the one lane that issues.  The operands are warp-uniform,
// and the issuing thread is not a divergent branch of its warp; measured on
// GB300 this issues a tcgen05.mma in ~35-44 cycles against ~48-54 for the
// same instruction under `if (lane == 0)`.
__device__ __forceinline__ void mma_ss_w(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_ts_w(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma_commit_w(uint64_t* b) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(su32(b))
      : "memory");
}

// Pair forms, issued by one elected lane of the leader CTA's warp: A rows
// 0-127 come from the leader's operand and 128-255 from the follower's at the
// same shared-memory (or TMEM) address, each CTA holds N/2 columns of B at the
// same address, and each CTA's TMEM receives its own 128 rows of D.
__device__ __forceinline__ void mma2_ss_w(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
__device__ __forceinline__ void mma2_ts_w(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
// Completion of the pair MMAs issued so far arrives on the barrier at the
// same offset in both CTAs.
__device__ __forceinline__ void mma2_commit_both_w(uint64_t* b) {
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}" ::"r"(
          su32(b)),
      "h"((uint16_t)3)
      : "memory");
}

__device__ __forceinline__ void mma_commit(uint64_t* b) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(b))
               : "memory");
}

#define ATTN_R32(r)                                                                                                 \
  "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),       \
      "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),        \
      "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),       \
      "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
#define ATTN_W32(r)                                                                                                 \
  "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),    \
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),   \
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),   \
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])

// 32 consecutive 32-bit TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : ATTN_R32(r)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
      "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      ATTN_W32(r)
      : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

#define ATTN_RW32(r)                                                                                                \
  "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]), "+r"(r[8]),       \
      "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]),        \
      "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]),       \
      "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])

// A tcgen05.ld writes its registers asynchronously; they hold the loaded
// values only after tcgen05.wait::ld.  The compiler sees the load's outputs
// as ready at once and may schedule arithmetic on them above the wait, so
// the wait is followed by an empty volatile statement that takes and
// returns every loaded register: each later use then depends on it, and it
// stays after the wait (volatile statements keep their order).
template <int N32>
__device__ __forceinline__ void tmem_ld_wait_regs(uint32_t* r) {
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < N32; ++i) asm volatile("" : ATTN_RW32((r + 32 * i)));
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Shared-memory matrix descriptor, 128-byte swizzle (tcgen05 format: start,
// leading and stride byte offsets in 16-byte units, descriptor version 1).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = (uint64_t)((saddr >> 4) & 0x3FFFu);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// The descriptor of the operand `bytes` further on (a multiple of 16): the
// start address is the low 14 bits in 16-byte units and every shared address
// of a CTA stays below 256 KB, so a 32-bit add on the low word cannot carry
// out of that field.  One add per MMA instead of rebuilding the descriptor.
__device__ __forceinline__ uint64_t sdesc_add(uint64_t d, uint32_t bytes) {
  const uint32_t lo = (uint32_t)d + (bytes >> 4), hi = (uint32_t)(d >> 32);
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
  return r;
}

// Instruction descriptor, kind::f16 with f32 accumulation.
__host__ __device__ constexpr uint32_t idesc_f16(bool bf16, bool b_mn_major, int M, int N) {
  return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

// Packed pair arithmetic (f32x2) and a three-input maximum: half the issue
// slots of the scalar forms for the softmax's per-element work.
__device__ __forceinline__ uint64_t f2u(float lo, float hi) {
  return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32);
}
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(f2u(a0, a1)), "l"(b), "l"(c));
  d0 = __uint_as_float((uint32_t)d);
  d1 = __uint_as_float((uint32_t)(d >> 32));
}
__device__ __forceinline__ void add2(float& a0, float& a1, float b0, float b1) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2u(a0, a1)), "l"(f2u(b0, b1)));
  a0 = __uint_as_float((uint32_t)d);
  a1 = __uint_as_float((uint32_t)(d >> 32));
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

}  // namespace tc
}  // namespace attn
