// Inline-PTX helpers for the sm_103a tensor-core path: mbarriers, TMA tile
// loads, tensor-memory allocation, tcgen05 MMA / load / store and fences.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace nf4 {
namespace tc {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier --
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Bounded wait: gives up after `limit` clock cycles (about a second at the
// GB300's clocks) and returns false; it never traps.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          long long limit = (1ll << 31)) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > limit) return false;
  }
}

// Non-blocking probe of a phase. Unlike try_wait, it never suspends the thread,
// and on the tcgen05 issuing thread it does not hold back the MMAs already
// queued (a try_wait there was measured to let the tensor pipe drain).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// The same probe with acquire semantics at cluster scope, for a barrier that
// threads of the peer CTA arrive on.
__device__ __forceinline__ bool mbar_test_wait_cluster(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Outcome of a wait that also watches a CTA's abort flag.
enum WaitResult { kWaitDone = 0, kWaitAborted = 1, kWaitTimeout = 2 };

// A wait that has lasted this many cycles starts to look at the abort flag.
// Stage waits normally end within a few hundred cycles, so the flag's
// shared-memory load stays off their path.
constexpr long long kAbortCheckAfter = 4096;

// Bounded wait on a phase that gives up early once *abort becomes nonzero
// (another role of the CTA, or the peer CTA of a pair, has failed).
__device__ __forceinline__ int mbar_wait_abortable(uint32_t bar, uint32_t parity,
                                                   const volatile int* abort,
                                                   long long limit = (1ll << 31)) {
  if (mbar_try_wait(bar, parity)) return kWaitDone;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return kWaitDone;
    const long long dt = clock64() - t0;
    if (dt > kAbortCheckAfter && *abort) return kWaitAborted;
    if (dt > limit) return kWaitTimeout;
  }
}

// The same on the non-blocking probe (kCluster: cluster-scope acquire), for
// the tcgen05 issuing warp, which must not suspend.
template <bool kCluster>
__device__ __forceinline__ int mbar_spin_abortable(uint32_t bar, uint32_t parity,
                                                   const volatile int* abort, long long limit) {
  auto probe = [&] {
    return kCluster ? mbar_test_wait_cluster(bar, parity) : mbar_test_wait(bar, parity);
  };
  if (probe()) return kWaitDone;
  const long long t0 = clock64();
  while (true) {
    if (probe()) return kWaitDone;
    const long long dt = clock64() - t0;
    if (dt > kAbortCheckAfter && *abort) return kWaitAborted;
    if (dt > limit) return kWaitTimeout;
  }
}

// Bounded spin on mbar_test_wait, for a thread with nothing else to do;
// kCluster selects the cluster-scope acquire.
template <bool kCluster = false>
__device__ __forceinline__ bool mbar_wait_spin(uint32_t bar, uint32_t parity,
                                               long long limit = (1ll << 31)) {
  auto probe = [&] {
    return kCluster ? mbar_test_wait_cluster(bar, parity) : mbar_test_wait(bar, parity);
  };
  if (probe()) return true;
  const long long t0 = clock64();
  while (true) {
    if (probe()) return true;
    if (clock64() - t0 > limit) return false;
  }
}

// One lane of the (converged) warp gets true. A loop that the whole warp runs
// on warp-uniform operands, issuing its tcgen05 instructions from the elected
// lane, was measured to issue an MMA in ~70 cycles against ~116 from a loop
// inside a one-thread branch.
__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .pred P1;\n\t"
      "elect.sync _|P1, 0xffffffff;\n\t"
      "selp.b32 %0, 1, 0, P1;\n\t}"
      : "+r"(pred));
  return pred != 0;
}

// ----------------------------------------------------------------- cluster --
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// All threads of all CTAs of the cluster; orders shared-memory writes before
// it (release) against reads after it (acquire) across the cluster.
__device__ __forceinline__ void cluster_sync() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::
          : "memory");
}

// Shared::cluster address of the variable at the same offset in CTA `rank`.
__device__ __forceinline__ uint32_t mapa(uint32_t local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local), "r"(rank));
  return r;
}

// Arrive on an mbarrier given by its shared::cluster address (possibly in
// another CTA of the cluster), with the instruction's default semantics
// (release at CTA scope). Measured on a busy SM, a release at cluster scope
// instead waits for the thread's (or, cumulatively, the SM's) memory traffic
// in flight: 1-2.5K cycles.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar) : "memory");
}

// --------------------------------------------------------------------- TMA --
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int32_t x,
                                            int32_t y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// A 2-D box from this CTA's shared memory to global memory (bulk-group
// completion: commit, then wait for the group's reads or writes).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int32_t x,
                                             int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(x), "r"(y)
               : "memory");
}

// The same box added element-wise to global memory (the tensor map's type,
// fp32 here); each element's add is atomic.
__device__ __forceinline__ void tma_reduce_add_2d(const CUtensorMap* map, uint32_t src, int32_t x,
                                                  int32_t y) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.2d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(x), "r"(y)
      : "memory");
}

__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Waits until the shared memory of this thread's committed bulk groups has
// been read (the source may be overwritten).
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Waits until this thread's committed bulk groups have completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------------ tcgen05 --
// Allocation is warp-wide; the base address is written to shared memory.
// With kCg = 2 one warp of each CTA of the pair allocates collectively, the
// same columns in both tensor memories.
template <int kCg = 1>
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  if constexpr (kCg == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     dst_smem),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  } else {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     dst_smem),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
}

template <int kCg = 1>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  if constexpr (kCg == 1) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
  } else {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
  }
}

__device__ __forceinline__ void fence_before_sync() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after_sync() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[tmem] * B[smem descriptor]^T, bf16 inputs, fp32 accumulate.
// With kCg = 2 the instruction is issued by one lane of the even CTA of a
// pair and spans both SMs: each CTA holds half of the M rows of A and D in its
// own tensor memory and half of the N rows of B at the same shared-memory
// offset, and each SM's accumulator receives all N columns.
template <int kCg = 1>
__device__ __forceinline__ void mma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc, uint32_t accumulate) {
  if constexpr (kCg == 1) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}

// D[tmem] (+)= A[smem descriptor] * B[smem descriptor]^T, bf16 inputs, fp32
// accumulate; kCg as for mma_bf16_tmem_a.
template <int kCg = 1>
__device__ __forceinline__ void mma_bf16_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  if constexpr (kCg == 1) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
  }
}

// Makes this thread's generic-proxy shared-memory stores visible to the async
// proxy (TMA, tensor cores) before a later synchronisation.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Arrive on an mbarrier once every tcgen05 operation issued so far by this
// thread has completed. With kCg = 2 the arrival goes to the barrier at the
// same offset in both CTAs of the pair.
template <int kCg = 1>
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  if constexpr (kCg == 1) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
  } else {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(bar),
        "h"(static_cast<uint16_t>(0x3))
        : "memory");
  }
}

// Thread i of the warp writes / reads lane (taddr.lane + i), 16 consecutive
// 32-bit columns from taddr.column. A warp may only touch its lane quarter.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]),
        "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]),
        "=r"(v[14]), "=r"(v[15])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major operand tile laid out as TMA
// writes it with 128-byte swizzling: rows of 128 bytes (64 bf16 along K),
// 8-row groups 1024 bytes apart, tile base 1024-byte aligned.
//   bits  0-13 start address >> 4      bits 16-29 leading byte offset >> 4
//   bits 32-45 stride byte offset >> 4 bits 46-47 descriptor version (1)
//   bits 61-63 swizzle mode (2 = 128-byte swizzle)
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t smem_byte_addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_byte_addr >> 4) & 0x3fffu);
  d |= static_cast<uint64_t>(1u) << 16;            // leading byte offset (unused by SW128 K-major)
  d |= static_cast<uint64_t>(1024u >> 4) << 32;    // stride byte offset: 8 rows x 128 B
  d |= static_cast<uint64_t>(1u) << 46;            // version
  d |= static_cast<uint64_t>(2u) << 61;            // 128-byte swizzle
  return d;
}

// Shared-memory matrix descriptor of an MN-major operand in 128-byte-swizzled
// atoms: an atom is 8 rows of K, each 128 bytes holding 64 consecutive bf16
// along M (N), 1024-byte aligned, 16-byte chunks XOR-permuted by the row.
// `lbo` is the byte distance between atoms adjacent along M, `sbo` between
// atoms adjacent along K.
__device__ __forceinline__ uint64_t sw128_mnmajor_desc(uint32_t smem_byte_addr, uint32_t lbo,
                                                       uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((smem_byte_addr >> 4) & 0x3fffu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3fffu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3fffu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;            // version
  d |= static_cast<uint64_t>(2u) << 61;            // 128-byte swizzle
  return d;
}

// Instruction descriptor for kind::f16 with A and B both bf16 (or both fp16),
// fp32 D, B K-major, shape M x N:
//   bits 4-5 D format (1 = f32)   bits 7-9 A format (0 = f16, 1 = bf16)
//   bits 10-12 B format (as A)     bit 15/16 A/B major (0 = K)
//   bits 17-22 N >> 3              bits 24-28 M >> 4
__host__ __device__ constexpr uint32_t idesc_f16kind_f32(uint32_t m, uint32_t n, bool a_mn_major,
                                                         bool f16) {
  return (1u << 4) | (f16 ? 0u : (1u << 7)) | (f16 ? 0u : (1u << 10)) |
         (a_mn_major ? (1u << 15) : 0u) | ((n >> 3) << 17) | ((m >> 4) << 24);
}

}  // namespace tc
}  // namespace nf4
