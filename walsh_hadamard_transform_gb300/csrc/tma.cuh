// Tensor-memory-accelerator (TMA) staging for the strided column tiles.
//
// A column tile is 2^K rows, 2^L elements apart, of one 32/64/128-byte segment
// each.  Seen as a 2-D tensor (rows of 2^L elements), it is a box of CW columns
// by 2^K rows, so a handful of cp.async.bulk.tensor.2d copies (up to 256 rows
// each) move it between HBM and shared memory without occupying the load/store
// units; one mbarrier tracks the arrival of the bytes.  The tile lands in shared
// memory in natural order (row-major, CW elements a row), where the threads read
// their layout-L1 vectors; after the transform they write layout L3 back in
// natural order and TMA stores the box.
#pragma once

#include <cstdint>

#include <cuda.h>  // CUtensorMap (type only; the encoder is fetched at run time)
#include <cuda_runtime.h>

namespace fwt {

// Set (bitwise OR) by a kernel whose bounded wait on a TMA copy gave up.  Each
// translation unit (one per element type) has its own copy; the host reads and
// clears them through read_device_error_*() (fwt_device_status()).
static __device__ unsigned int g_device_error;
constexpr unsigned int kErrTmaTimeout = 1u;

// Programmatic dependent launch: the pass kernels are launched so that they may
// start while the previous kernel on their stream is still draining.  Each waits
// here, before its first global-memory access, until that kernel has completed and
// its writes are visible, and then lets the next kernel on the stream be scheduled
// (it starts once every CTA of this grid has started, so nothing of this grid can
// be left unscheduled behind it).  Without the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_begin() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 1000;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for phase `parity` of the barrier for at most about one second (global
// timer, with an iteration cap as a backstop).  On give-up it records
// kErrTmaTimeout and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t i = 1; i < (1u << 26); ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0 && global_ns() - t0 > 1000000000ull) break;
  }
  atomicOr(&g_device_error, kErrTmaTimeout);
  return false;
}


__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar, unsigned long long policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, const void* src,
                                             unsigned long long policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group.L2::cache_hint"
      " [%0, {%1, %2}], [%3], %4;" ::"l"(map),
      "r"(x), "r"(y), "r"(smem_u32(src)), "l"(policy)
      : "memory");
}

// Untiled bulk copies of a contiguous byte range (16-byte aligned, a multiple of
// 16 bytes long) between global and shared memory.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes,
                                          uint64_t* bar, unsigned long long policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void bulk_store(void* dst, const void* src, uint32_t bytes,
                                           unsigned long long policy) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group.L2::cache_hint [%0], [%1], %2, %3;" ::"l"(
                   dst),
               "r"(smem_u32(src)), "r"(bytes), "l"(policy)
               : "memory");
}

// L2 prefetches (no shared memory, no completion to wait for): a box of a tensor
// map, or a contiguous range (16-byte aligned, a multiple of 16 bytes).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(map), "r"(x),
               "r"(y)
               : "memory");
}
__device__ __forceinline__ void bulk_prefetch(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void tma_store_commit_and_wait() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Generic-proxy writes to shared memory become visible to the TMA (async proxy).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

}  // namespace fwt
