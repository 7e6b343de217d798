// Inline-PTX wrappers shared by the kernels that stage tiles with TMA:
// mbarriers (init, arrive, expect-tx, bounded waits) and tiled bulk-tensor
// loads into shared memory.
#pragma once
#include <cuda.h>
#include <stdint.h>

#include "common.cuh"

namespace moe {

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0u;
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}

// Bounded wait.  Returns false if `abort` is set or the limit ran out (which
// sets `abort` and records kErrTimeout at `where`).
static __device__ __noinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort, uint64_t limit_ns,
                                       uint32_t* err, uint32_t where) {
  if (mbar_try(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0;; ++i) {
    if (mbar_try(bar, parity)) return true;
    if (*abort) return false;
    if ((i & 7u) == 0u && globaltimer_ns() - t0 > limit_ns) {
      *abort = 1u;
      record_error(err, kErrTimeout, where);
      return false;
    }
  }
}
// mbar_wait with its first poll inlined (the common case: already complete).
__device__ __forceinline__ bool mbar_wait_i(uint32_t bar, uint32_t parity, volatile uint32_t* abort, uint64_t limit_ns,
                                            uint32_t* err, uint32_t where) {
  if (mbar_try(bar, parity)) return true;
  return mbar_wait(bar, parity, abort, limit_ns, err, where);
}
// Bounded wait used while tearing down: ignores any abort flag.
static __device__ __noinline__ bool mbar_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(map), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(dst),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

// ---- L2 eviction policy for data that is read or written once ---------------------
// Lines touched with this policy are the first to be replaced, so a stream
// recycles its own lines instead of evicting (and forcing the write-back of)
// what earlier kernels left in L2.
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void tma_load_2d_hint(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3}], [%4], %5;" ::"r"(dst),
      "l"(map), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ uint4 ld_stream_u4(const void* p, uint64_t policy) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(policy));
  return v;
}
__device__ __forceinline__ void st_stream_u4(void* p, uint4 v, uint64_t policy) {
  asm volatile("st.global.L1::no_allocate.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "r"(v.x),
               "r"(v.y), "r"(v.z), "r"(v.w), "l"(policy)
               : "memory");
}

// ---- thread-block clusters (pairs of CTAs) ----------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Shared::cluster address of the variable at local shared address `a` in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t a, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(rank));
  return r;
}
// Every thread of every CTA of the cluster arrives, then waits (release / acquire).
// After an abort in a CTA pair, a copy the peer issued before it stopped may
// still be landing in this CTA's shared memory or on its barriers (the pair's
// copies complete on the leader's barriers, which only the leader drains).
// A CTA that sees the status word set waits this long (bounded) before its
// shared memory and TMEM are released; copies land within microseconds.
__device__ __forceinline__ void abort_grace(const uint32_t* err) {
  if (*(volatile const uint32_t*)err == 0u) return;
  const uint64_t t0 = globaltimer_ns();
  while (globaltimer_ns() - t0 < 50000ull) __nanosleep(1000);
}

__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive on an mbarrier that may live in another CTA of the cluster.
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// TMA tile loads of a CTA pair: the data lands in this CTA's shared memory,
// the completion is signalled on `bar`, which may be the peer CTA's mbarrier
// (a shared::cluster address).
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                                 uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3}], [%4];" ::"r"(dst),
      "l"(map), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d_pair(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                                 uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, "
      "%3, %4}], [%5];" ::"r"(dst),
      "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}

// ---- host: tensor maps (cuTensorMapEncodeTiled through the runtime's driver entry point) ----
// Row-major bf16 matrix [rows, cols] (cols contiguous), box box_cols x box_rows,
// 128-byte swizzle, zero fill outside the matrix.  False if it cannot be encoded
// (unaligned base or stride, or no driver entry point).
// TMA store of a box from this CTA's shared memory to global memory, tracked by
// the issuing thread's bulk-async groups.  The source follows the tensor map's
// swizzle; the generic-proxy writes that filled it must be fenced first.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(map), "r"(c0),
               "r"(c1), "r"(src)
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// The source shared memory of every committed group has been read.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// Every committed group has completed its writes.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

bool tmap_bf16_2d(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int box_cols, int box_rows);
// Row-major fp32 [rows, cols] (cols a multiple of 4), box 32 columns (128
// bytes) x box_rows, 128-byte swizzle: the layout of an fp32 epilogue tile.
bool tmap_f32_2d(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int box_rows);
// As tmap_bf16_2d with the swizzle chosen by the box row size: 16 bytes none,
// 32 / 64 / 128 bytes the matching swizzle mode.
bool tmap_bf16_2d_swizzle(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int box_cols, int box_rows,
                          int row_bytes);
// Stacked bf16 matrices [G, rows, cols], box box_cols x box_rows x 1, 128-byte swizzle.
bool tmap_bf16_3d(CUtensorMap* m, const void* ptr, int G, int64_t rows, int64_t cols, int box_cols, int box_rows);
// Byte matrices (E4M3 codes): row-major [rows, cols] and stacked [G, rows, cols],
// box 128 bytes x box_rows (x 1), 128-byte swizzle.
bool tmap_u8_2d(CUtensorMap* m, const void* ptr, int64_t rows, int64_t cols, int box_rows);
bool tmap_u8_3d(CUtensorMap* m, const void* ptr, int G, int64_t rows, int64_t cols, int box_rows);

}  // namespace moe
