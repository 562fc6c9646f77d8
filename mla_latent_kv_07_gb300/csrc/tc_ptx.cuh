// tc_ptx.cuh -- inline PTX wrappers shared by the tensor-core kernels:
// mbarriers, cluster shared memory, tcgen05 (MMA, tensor-memory loads and
// stores, fences), TMA tensor and bulk copies, and the 128-byte swizzle.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace mla {
namespace ptx {

constexpr int kSwBlk = 128 * 128;   // one 128-row x 128-byte swizzled block: 16 KB

__device__ __forceinline__ uint32_t sa(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void bar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(sa(b)), "r"(count));
}
__device__ __forceinline__ void bar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(sa(b)) : "memory");
}
__device__ __forceinline__ void bar_arrive_remote(uint32_t remote_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_addr)
               : "memory");
}
// Remote arrive without release semantics: for signals whose only ordering
// requirement is on loads whose values are already consumed in registers.
__device__ __forceinline__ void bar_arrive_remote_relaxed(uint32_t remote_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote_addr)
               : "memory");
}
// arrive on a peer CTA's barrier, adding `bytes` to the transaction count its
// phase waits for
__device__ __forceinline__ void bar_arrive_expect_tx_remote(uint32_t remote_addr, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.relaxed.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(remote_addr),
               "r"(bytes)
               : "memory");
}
// 16 bytes into a peer CTA's shared memory, counted on the peer's barrier when
// they land (no acknowledgement travels back to this thread)
__device__ __forceinline__ void st_async_v4(uint32_t remote_addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d,
                                            uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(
                   remote_addr),
               "r"(a), "r"(b), "r"(c), "r"(d), "r"(remote_bar)
               : "memory");
}
// 8 bytes into a peer CTA's shared memory, counted on the peer's barrier when
// they land
__device__ __forceinline__ void st_async_v2(uint32_t remote_addr, uint32_t a, uint32_t b, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.b32 [%0], {%1, %2}, [%3];" ::"r"(
                   remote_addr),
               "r"(a), "r"(b), "r"(remote_bar)
               : "memory");
}
// 4 bytes into a peer CTA's shared memory, counted on the peer's barrier when
// they land
__device__ __forceinline__ void st_async_b32(uint32_t remote_addr, uint32_t v, uint32_t remote_bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(remote_addr),
               "r"(v), "r"(remote_bar)
               : "memory");
}
// `count` arrivals at once on a peer CTA's barrier (release: this thread's
// earlier memory accesses are ordered before them)
__device__ __forceinline__ void bar_arrive_remote_n(uint32_t remote_addr, uint32_t count) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(remote_addr), "r"(count)
               : "memory");
}
__device__ __forceinline__ void bar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(sa(b)), "r"(bytes)
               : "memory");
}
// Non-suspending probe of a barrier phase.  (A suspending try_wait was seen to
// return up to microseconds after phases completed by tcgen05.commit or by
// remote arrivals, which serialised the pipeline; a polling test_wait notices
// them at once.)  Cluster-scope acquire: for barriers that the peer CTA's
// stores, copies or commits complete.
__device__ __forceinline__ bool bar_try(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2; "
      "selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(sa(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// The same probe with CTA-scope acquire, for barriers that only this CTA's
// threads, tensor-core commits and tensor copies complete.  It is measurably
// cheaper inside the decode kernel's per-tile hand-offs.
__device__ __forceinline__ bool bar_try_local(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2; "
      "selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(sa(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// 16-byte asynchronous copy, global -> this CTA's shared memory (through L2)
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(sa(dst)), "l"(src) : "memory");
}
// one arrival on b once the thread's earlier cp.async copies have landed
// (counted in the barrier's expected arrivals)
__device__ __forceinline__ void cp_async_arrive(uint64_t* b) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(sa(b)) : "memory");
}
__device__ __forceinline__ uint32_t mapa(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(sa(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned; barrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// generic-proxy global writes of this thread -> later tensor copies (async proxy)
__device__ __forceinline__ void fence_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}
__device__ __forceinline__ void tc_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// smem matrix descriptor: 128-byte swizzle, version 1
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}
// smem matrix descriptor without swizzle (8-row x 16-byte core matrices):
// lbo = bytes between core matrices along K, sbo = along M/N; version 1
__device__ __forceinline__ uint64_t sdesc_plain(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFF) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | (1ull << 46);
}
// instruction descriptor, kind::f16: bf16 x bf16 -> fp32
__host__ __device__ constexpr uint32_t idesc(int M, int N, bool b_mn_major, bool a_mn_major = false) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) |
         ((b_mn_major ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id, int acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; "
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d),
      "l"(a), "l"(b), "r"(id), "r"(acc));
}
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t id, int acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0; "
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }" ::"r"(d),
      "r"(a), "l"(b), "r"(id), "r"(acc));
}
// Descriptor of a tile `bytes` further into shared memory: the start-address
// field is the low 14 bits (address >> 4, shared addresses below 256 KB), so
// the offset adds without a carry into the other fields.  A descriptor built
// once per stage plus a constant offset keeps the issuing thread's work per
// MMA at one add.
__device__ __forceinline__ uint64_t sdesc_at(uint64_t desc, uint32_t bytes) { return desc + (bytes >> 4); }
// MMA with a compile-time accumulate flag (kAcc = false overwrites D)
template <bool kAcc>
__device__ __forceinline__ void mma_ss_c(uint32_t d, uint64_t a, uint64_t b, uint32_t id) {
  if constexpr (kAcc)
    asm volatile("{ .reg .pred p; setp.ne.b32 p, 1, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }"
                 ::"r"(d), "l"(a), "l"(b), "r"(id));
  else
    asm volatile("{ .reg .pred p; setp.ne.b32 p, 0, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }"
                 ::"r"(d), "l"(a), "l"(b), "r"(id));
}
template <bool kAcc>
__device__ __forceinline__ void mma_ts_c(uint32_t d, uint32_t a, uint64_t b, uint32_t id) {
  if constexpr (kAcc)
    asm volatile("{ .reg .pred p; setp.ne.b32 p, 1, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }"
                 ::"r"(d), "r"(a), "l"(b), "r"(id));
  else
    asm volatile("{ .reg .pred p; setp.ne.b32 p, 0, 0; tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p; }"
                 ::"r"(d), "r"(a), "l"(b), "r"(id));
}
__device__ __forceinline__ void mma_commit(uint64_t* b) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   sa(b))
               : "memory");
}
// the MMAs issued so far arrive, once complete, on the barrier at the same
// shared-memory offset in every CTA of the cluster named by `mask`
__device__ __forceinline__ void mma_commit_mc(uint64_t* b, uint16_t mask) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          sa(b)),
      "h"(mask)
      : "memory");
}
#define TC_LD16(taddr, r)                                                                       \
  asm volatile(                                                                                 \
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13," \
      "%14,%15}, [%16];"                                                                        \
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),     \
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), \
        "=r"(r[14]), "=r"(r[15])                                                                \
      : "r"(taddr))
#define TC_LD8(taddr, r)                                                                   \
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"    \
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),    \
                 "=r"(r[6]), "=r"(r[7])                                                    \
               : "r"(taddr))
// 16 lanes (the lane field of taddr onwards) x 32 / 16 fp32 columns: thread
// t holds lanes t/4 and t/4 + 8 at columns 8k + 2 (t%4) and 8k + 2 (t%4) + 1,
// r[4k .. 4k+3] = (lane t/4: both columns, then lane t/4 + 8: both columns)
#define TC_LD16L_X4(taddr, r)                                                                    \
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12," \
               "%13,%14,%15}, [%16];"                                                            \
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),         \
                 "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),       \
                 "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])                              \
               : "r"(taddr))
#define TC_LD16L_X2(taddr, r)                                                                  \
  asm volatile("tcgen05.ld.sync.aligned.16x256b.x2.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"       \
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),       \
                 "=r"(r[6]), "=r"(r[7])                                                        \
               : "r"(taddr))
// the store counterpart of TC_LD16L_X4 (same thread / register layout)
#define TC_ST16L_X4(taddr, r)                                                                          \
  asm volatile("tcgen05.st.sync.aligned.16x256b.x4.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13," \
               "%14,%15,%16};" ::"r"(taddr),                                                           \
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),  \
               "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),       \
               "r"(r[15])                                                                              \
               : "memory")
#define TC_ST16(taddr, r)                                                                     \
  asm volatile(                                                                               \
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12," \
      "%13,%14,%15,%16};" ::"r"(taddr),                                                       \
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), \
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),       \
      "r"(r[15])                                                                              \
      : "memory")
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tma3(void* dst, const CUtensorMap* m, int c0, int c1, int c2,
                                     uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3, %4}], [%5];" ::"r"(sa(dst)),
      "l"(m), "r"(c0), "r"(c1), "r"(c2), "r"(sa(bar))
      : "memory");
}
__device__ __forceinline__ void tma3_store(const CUtensorMap* m, int c0, int c1, int c2,
                                           const void* src) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(m),
      "r"(c0), "r"(c1), "r"(c2), "r"(sa(src))
      : "memory");
}

// Four rows r0..r3 of a 2D tensor map (box: one row high), columns from c0,
// stacked at dst; completes on bar.
__device__ __forceinline__ void tma_gather4(void* dst, const CUtensorMap* m, int c0, int r0, int r1,
                                            int r2, int r3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4, %5, %6}], [%7];" ::"r"(sa(dst)),
      "l"(m), "r"(c0), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(sa(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_store(void* gdst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst),
               "r"(sa(src)), "r"(bytes)
               : "memory");
}
// shared::cta -> a cluster peer's shared memory, completing bytes on the
// peer's mbarrier (remote addresses from mapa)
__device__ __forceinline__ void bulk_s2c(uint32_t remote_dst, const void* src, uint32_t bytes, uint32_t remote_bar) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(remote_dst), "r"(sa(src)), "r"(bytes), "r"(remote_bar) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the bulk stores of this thread have read their shared-memory sources (their
// global writes complete with the grid)
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// byte offset of 16-byte chunk `chunk` of row `row` in a 128-byte-swizzled block
__device__ __forceinline__ uint32_t swz_chunk(int row, int chunk) {
  return (row >> 3) * 1024 + (row & 7) * 128 + (((chunk ^ row) & 7) << 4);
}

}  // namespace ptx
}  // namespace mla
