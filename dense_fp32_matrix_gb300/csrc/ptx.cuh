// Inline-PTX building blocks for sm_103a: mbarriers, TMA tile loads,
// 4-byte asynchronous copies, packed fp32x2 FMA and bounded waits.
//
// Every wait in this library is bounded. A wait that runs past its limit
// records (code, site, block) in the per-device status word passed to each
// kernel and returns false; the caller then abandons its work uniformly
// across the block and exits. Nothing here traps.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dfm {

// Default limit of one bounded wait: about one second of wall time.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

// Status word layout (int[4] in device memory): [0] error code (0 = none),
// [1] wait-site id of the first failure, [2] block id, [3] count of failures.
constexpr int kStatusWatchdog = 1;

// Wait-site ids reported by sgemm_watchdog_status().
enum WaitSite : int {
  kSiteSelftest = 1,
  kSiteTiledFull = 2,
  kSiteTiledDrain = 3,
  kSiteGemvRow = 4,
  kSiteGemvCol = 5,
  kSiteTf32Full = 6,
  kSiteTf32Conv = 7,
  kSiteTf32Empty = 8,
  kSiteTf32Acc = 9,
  kSiteTf32Peer = 10,
  kSiteTf32Fix = 11,
  kSiteTiledEmpty = 12,
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void record_timeout(int* status, int site) {
  if (status == nullptr) return;
  if (atomicCAS(&status[0], 0, kStatusWatchdog) == 0) {
    status[1] = site;
    status[2] = static_cast<int>(blockIdx.x + gridDim.x * blockIdx.y);
  }
  atomicAdd(&status[3], 1);
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count)
               : "memory");
}

// Make mbarrier initialisation visible to the other threads and to the
// asynchronous (TMA) proxy.
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar,
                                                      uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
      "r"(bytes)
      : "memory");
}

// kCluster: acquire at cluster scope, for a barrier that blocks of the
// cluster arrive on with release.cluster (their writes become visible).
template <bool kCluster = false>
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  if (kCluster) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], "
        "%2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
  } else {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
  }
  return ok != 0;
}

// Wait until phase `parity` of the mbarrier completes, for at most
// `limit_ns` nanoseconds (and at most 2^31 polls as a second bound). Returns
// false on timeout after recording it.
template <bool kCluster = false>
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  int* status, int site,
                                                  uint64_t limit_ns) {
  if (mbar_try_wait<kCluster>(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1; it < (1u << 31); ++it) {
    if (mbar_try_wait<kCluster>(bar, parity)) return true;
    if ((it & 15u) == 0 && global_timer_ns() - t0 > limit_ns) break;
  }
  record_timeout(status, site);
  return false;
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map))
               : "memory");
}

// 3-D tiled bulk tensor load (z: the batch index of a batched operand).
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map,
                                            int32_t x, int32_t y, int32_t z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap* map,
                                                   int32_t x, int32_t y,
                                                   int32_t z) {
  asm volatile(
      "cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(x), "r"(y), "r"(z)
      : "memory");
}

// 3-D tiled bulk tensor store shared -> global (bulk-group completion);
// elements outside the tensor's extents are not written.
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map,
                                             uint32_t src, int32_t x,
                                             int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, "
      "%4}], [%1];" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(x), "r"(y), "r"(z)
      : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N of this thread's bulk groups still read shared
// memory (their sources may then be overwritten).
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

// Wait until all of this thread's bulk groups have completed.
__device__ __forceinline__ void bulk_wait_group_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// 2-D tiled bulk tensor load global -> shared, completion signalled on the
// mbarrier as transaction bytes. x is the innermost coordinate (elements),
// y the outer one. Out-of-bounds box elements are filled with zero.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map,
                                            int32_t x, int32_t y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

// 1-D tiled bulk tensor load (rank-1 tensor map), zero fill past the end.
__device__ __forceinline__ void tma_load_1d(uint32_t dst, const CUtensorMap* map,
                                            int32_t x, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.1d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2}], [%3];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(bar)
      : "memory");
}

// ---------------------------------------------------------------- clusters

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Every thread of every block of the cluster arrives and waits (release /
// acquire): shared-memory writes before it are visible to all blocks of the
// cluster after it. Hardware barrier; the blocks of a cluster are scheduled
// together, so it completes once all of them reach it.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile(
      "barrier.cluster.arrive.release.aligned;\n\t"
      "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory location in block `rank` of the cluster.
__device__ __forceinline__ uint32_t cluster_map(uint32_t smem_addr,
                                                uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(r)
               : "r"(smem_addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v)
               : "memory");
}

// ---------------------------------------------------------------- cp.async

// 4-byte global -> shared asynchronous copy; copies `src_bytes` (0 or 4)
// bytes and zero-fills the rest, so src_bytes = 0 writes a zero without
// reading global memory.
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src,
                                           uint32_t src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst),
               "l"(src), "r"(src_bytes)
               : "memory");
}

// Bulk copy of `bytes` (a multiple of 16, both addresses 16-byte aligned)
// global -> this CTA's shared memory, completion as transaction bytes on
// the mbarrier.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src,
                                          uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void mbar_inval(uint32_t bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// ---------------------------------------------------------------- fp32x2

// Packed pair of fp32 values in one 64-bit register pair.
struct f2 {
  unsigned long long v;
};

__device__ __forceinline__ f2 f2_pack(float lo, float hi) {
  f2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r.v) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ void f2_unpack(f2 x, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(x.v));
}

// d = a * b + d, elementwise on both halves, each an IEEE fp32 fused
// multiply-add rounded to nearest even.
__device__ __forceinline__ void f2_fma(f2& d, f2 a, f2 b) {
  asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d.v) : "l"(a.v), "l"(b.v));
}

}  // namespace dfm
