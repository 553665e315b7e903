// TMA-staged bandwidth kernels for the vector shapes of the product.
//
// With M = 1 (c = a B) or N = 1 (c = A b) every element of the matrix is used
// once: the product is a stream over it at 2 flops per 4 bytes ("GEMM from
// naive to tiled", section 十.2; "如何让计算受限问题真正达到计算受限",
// section 7), so the only goal is to keep HBM busy. Both kernels stage the
// matrix through a 4-deep ring of 16 KiB TMA tiles per block (up to 64 KiB
// in flight per block whatever the thread count; the N = 1 kernel takes a
// 3-deep ring when that fits its whole grid on the GPU at once), and add
// partial sums in a fixed order, so results are deterministic. The prologue
// fills every stage; after step t the stage it read is refilled with step
// t + (number of stages).
//
//   * k_gemv_row_tma (M = 1): a block owns 64 columns of B and one of S
//     k-ranges; each stage brings 64 rows of B and the 64 matching entries of
//     a. The S blocks of a column strip form a thread-block cluster and add
//     their 64 partial sums in rank order through distributed shared memory
//     (no global scratch, no atomics).
//   * k_gemv_col_tma (N = 1): a block owns 16 rows of A and all of K, b is
//     staged beside A in the same ring; 16 lanes per row, shuffle tree.
//
// Layouts that TMA cannot describe (16-byte misaligned bases or row strides)
// use the plain kernels in sgemm_small.cu.
#include "kernels.h"
#include "ptx.cuh"

namespace dfm {
namespace {

constexpr int kThreads = 256;
constexpr int kStages = 4;

// ---------------------------------------------------------------- M == 1

constexpr int GR_COLS = 64;                       // columns per block
constexpr int GR_ROWS = 64;                       // k rows per stage
constexpr int GR_GROUPS = kThreads / GR_COLS;     // 4 row groups
constexpr int GR_STAGE = GR_COLS * GR_ROWS * 4;   // 16 KiB of B
constexpr int GR_A_STAGE = GR_ROWS * 4;           // 256 B of a
constexpr int GR_MAX_CLUSTER = 8;
constexpr size_t GR_SMEM =
    size_t(kStages) * (GR_STAGE + GR_A_STAGE) + 64 + 128;
// Tiled TMA writes shared memory at 128-byte aligned addresses only.
static_assert(GR_STAGE % 128 == 0 && GR_A_STAGE % 128 == 0,
              "row-kernel stage slots must keep 128-byte alignment");

__global__ void __launch_bounds__(kThreads)
k_gemv_row_tma(const __grid_constant__ CUtensorMap tmB,
               const __grid_constant__ CUtensorMap tma_, float* __restrict__ c,
               int N, int K, int k_per_block, int cluster, Scale sc,
               int* status) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ float red[GR_GROUPS][GR_COLS];
  __shared__ float part[GR_MAX_CLUSTER][GR_COLS];  // used in rank 0
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* sB = smem_raw + (((raw + 127u) & ~127u) - raw);
  uint8_t* sa = sB + kStages * GR_STAGE;
  const uint32_t bar0 = smem_u32(sa + kStages * GR_A_STAGE);
  const int tid = threadIdx.x;
  const int rank = cluster > 1 ? int(cluster_rank()) : 0;
  const int n0 = blockIdx.x * GR_COLS;
  const int k_lo = rank * k_per_block;
  const int k_hi = min(K, k_lo + k_per_block);
  const int T = k_hi > k_lo ? (k_hi - k_lo + GR_ROWS - 1) / GR_ROWS : 0;

  auto issue = [&](int t, int slot) {
    const uint32_t bar = bar0 + 8 * slot;
    mbar_arrive_expect_tx(bar, GR_STAGE + GR_A_STAGE);
    tma_load_2d(smem_u32(sB + slot * GR_STAGE), &tmB, n0, k_lo + t * GR_ROWS,
                bar);
    tma_load_1d(smem_u32(sa + slot * GR_A_STAGE), &tma_, k_lo + t * GR_ROWS,
                bar);
  };
  if (tid == 0) {
    tma_prefetch_desc(&tmB);
    tma_prefetch_desc(&tma_);
    for (int s = 0; s < kStages; ++s) mbar_init(bar0 + 8 * s, 1);
    mbar_fence_init();
    for (int s = 0; s < kStages && s < T; ++s) issue(s, s);
  }
  __syncthreads();

  const int col = tid % GR_COLS, g = tid / GR_COLS;
  float acc = 0.f;
  bool aborted = false;
  int slot = 0;
  uint32_t phase = 0;
  for (int t = 0; t < T; ++t) {
    const bool ok = mbar_wait_bounded(bar0 + 8 * slot, phase, status,
                                      kSiteGemvRow, kWaitLimitNs);
    if (__syncthreads_or(!ok)) {  // uniform abort; no early return, the
      aborted = true;             // cluster barriers below must be reached
      if (tid == 0)
        for (int v = t; v < T && v < t + kStages; ++v)
          mbar_wait_bounded(bar0 + 8 * ((slot + v - t) % kStages),
                            phase ^ uint32_t(((slot + v - t) / kStages) & 1),
                            nullptr, kSiteGemvRow, kWaitLimitNs / 100);
      break;
    }
    // The barrier above means every thread finished step t - 1: its stage
    // takes step t - 1 + kStages.
    if (tid == 0 && t >= 1 && t - 1 + kStages < T)
      issue(t - 1 + kStages, slot == 0 ? kStages - 1 : slot - 1);
    const float* rows = reinterpret_cast<const float*>(sB + slot * GR_STAGE);
    const float* av = reinterpret_cast<const float*>(sa + slot * GR_A_STAGE);
    // Rows past k_hi belong to the next block's range (or are past K and
    // zero-filled): masked so that a row is never counted twice.
    const int valid = k_hi - (k_lo + t * GR_ROWS);
#pragma unroll
    for (int r = 0; r < GR_ROWS / GR_GROUPS; ++r) {
      const int kr = g + GR_GROUPS * r;
      if (kr < valid) acc = fmaf(av[kr], rows[kr * GR_COLS + col], acc);
    }
    if (++slot == kStages) {
      slot = 0;
      phase ^= 1u;
    }
  }
  red[g][col] = acc;
  __syncthreads();
  float s = 0.f;
  if (tid < GR_COLS) {
#pragma unroll
    for (int q = 0; q < GR_GROUPS; ++q) s += red[q][tid];
  }
  if (cluster == 1) {
    if (tid < GR_COLS && !aborted && n0 + tid < N)
      c[n0 + tid] = epi1(s, c + n0 + tid, sc);
    return;
  }
  // Rank r's 64 partials go to slot r of rank 0's buffer; rank 0 adds the
  // slots in rank order (k order).
  cluster_sync_all();  // every block of the cluster is running
  if (tid < GR_COLS)
    st_cluster_f32(cluster_map(smem_u32(&part[rank][tid]), 0), s);
  cluster_sync_all();  // all partials visible in rank 0
  if (rank == 0 && tid < GR_COLS && !aborted && n0 + tid < N) {
    float total = 0.f;
    for (int q = 0; q < cluster; ++q) total += part[q][tid];
    c[n0 + tid] = epi1(total, c + n0 + tid, sc);
  }
}

// ---------------------------------------------------------------- N == 1

constexpr int GC_ROWS = 16;                       // rows of A per block
constexpr int GC_K = 256;                         // k per stage
constexpr int GC_LANES = kThreads / GC_ROWS;      // 16 lanes per row
constexpr int GC_A_STAGE = GC_ROWS * GC_K * 4;    // 16 KiB
constexpr int GC_B_STAGE = GC_K * 4;              // 1 KiB
// Shared memory of a block with ST stages. Four stages by default; three
// when that lets every block of the grid be resident at once (a grid a
// little larger than one wave of four-stage blocks would otherwise run a
// short second wave).
constexpr size_t gc_smem(int st) {
  return size_t(st) * (GC_A_STAGE + GC_B_STAGE) + 64 + 128;
}
static_assert(GC_A_STAGE % 128 == 0 && GC_B_STAGE % 128 == 0,
              "col-kernel stage slots must keep 128-byte alignment");
static_assert(GC_K / 4 == 4 * GC_LANES, "4 float4 per lane per stage");

template <int ST>
__global__ void __launch_bounds__(kThreads)
k_gemv_col_tma(const __grid_constant__ CUtensorMap tmA,
               const __grid_constant__ CUtensorMap tmb, float* __restrict__ c,
               long long ldc, int M, int K, Scale sc, int* status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* sA = smem_raw + (((raw + 127u) & ~127u) - raw);
  uint8_t* sb = sA + ST * GC_A_STAGE;
  const uint32_t bar0 = smem_u32(sb + ST * GC_B_STAGE);
  const int tid = threadIdx.x;
  const int m0 = blockIdx.x * GC_ROWS;
  const int T = (K + GC_K - 1) / GC_K;

  auto issue = [&](int t, int slot) {
    const uint32_t bar = bar0 + 8 * slot;
    mbar_arrive_expect_tx(bar, GC_A_STAGE + GC_B_STAGE);
    tma_load_2d(smem_u32(sA + slot * GC_A_STAGE), &tmA, t * GC_K, m0, bar);
    tma_load_1d(smem_u32(sb + slot * GC_B_STAGE), &tmb, t * GC_K, bar);
  };
  if (tid == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmb);
    for (int s = 0; s < ST; ++s) mbar_init(bar0 + 8 * s, 1);
    mbar_fence_init();
    for (int s = 0; s < ST && s < T; ++s) issue(s, s);
  }
  __syncthreads();

  const int r = tid / GC_LANES, s = tid % GC_LANES;
  float acc = 0.f;
  int slot = 0;
  uint32_t phase = 0;
  for (int t = 0; t < T; ++t) {
    const bool ok = mbar_wait_bounded(bar0 + 8 * slot, phase, status,
                                      kSiteGemvCol, kWaitLimitNs);
    if (__syncthreads_or(!ok)) {
      if (tid == 0)
        for (int v = t; v < T && v < t + ST; ++v)
          mbar_wait_bounded(bar0 + 8 * ((slot + v - t) % ST),
                            phase ^ uint32_t(((slot + v - t) / ST) & 1),
                            nullptr, kSiteGemvCol, kWaitLimitNs / 100);
      return;
    }
    if (tid == 0 && t >= 1 && t - 1 + ST < T)
      issue(t - 1 + ST, slot == 0 ? ST - 1 : slot - 1);
    const float4* row =
        reinterpret_cast<const float4*>(sA + slot * GC_A_STAGE + r * GC_K * 4);
    const float4* bv = reinterpret_cast<const float4*>(sb + slot * GC_B_STAGE);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 x = row[s + GC_LANES * j], y = bv[s + GC_LANES * j];
      acc = fmaf(x.x, y.x, acc);
      acc = fmaf(x.y, y.y, acc);
      acc = fmaf(x.z, y.z, acc);
      acc = fmaf(x.w, y.w, acc);
    }
    if (++slot == ST) {
      slot = 0;
      phase ^= 1u;
    }
  }
  // 16 lanes per row: fixed butterfly inside each half-warp.
#pragma unroll
  for (int off = GC_LANES / 2; off > 0; off >>= 1)
    acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (s == 0 && m0 + r < M)
    c[(long long)(m0 + r) * ldc] = epi1(acc, c + (long long)(m0 + r) * ldc, sc);
}

}  // namespace

// Resident blocks per SM of the N = 1 kernel with 4 and with 3 stages.
int g_col_per_sm[2] = {0, 0};

cudaError_t gemv_tma_init() {
  cudaError_t e = cudaFuncSetAttribute(
      k_gemv_row_tma, cudaFuncAttributeMaxDynamicSharedMemorySize,
      int(GR_SMEM));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_gemv_col_tma<4>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(gc_smem(4)));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_gemv_col_tma<3>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(gc_smem(3)));
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &g_col_per_sm[0], k_gemv_col_tma<4>, kThreads, gc_smem(4));
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      &g_col_per_sm[1], k_gemv_col_tma<3>, kThreads, gc_smem(3));
}

GemvRowPlan plan_gemv_row(int64_t N, int64_t K, int num_sms) {
  GemvRowPlan pl;
  pl.col_blocks = (N + GR_COLS - 1) / GR_COLS;
  const int64_t stages = (K + GR_ROWS - 1) / GR_ROWS;
  // At most two blocks per SM (more would leave some SMs a third block and
  // the others idle at the end), at most 8 per cluster, at least one stage
  // of k rows per block.
  int64_t S = 2 * int64_t(num_sms) / pl.col_blocks;
  if (S > GR_MAX_CLUSTER) S = GR_MAX_CLUSTER;
  if (S > stages) S = stages;
  if (S < 1) S = 1;
  pl.cluster = int(S);
  pl.k_per_block = ((stages + S - 1) / S) * GR_ROWS;
  return pl;
}

cudaError_t launch_gemv_row_tma(const GemmArgs& g, const CUtensorMap& tmB,
                                const CUtensorMap& tma_, const GemvRowPlan& pl,
                                int* status, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(pl.col_blocks), unsigned(pl.cluster), 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = GR_SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = unsigned(pl.cluster);
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return counted(cudaLaunchKernelEx(&cfg, k_gemv_row_tma, tmB, tma_, g.C, int(g.N),
                            int(g.K), int(pl.k_per_block), pl.cluster, g.sc,
                            status));
}

cudaError_t launch_gemv_col_tma(const GemmArgs& g, const CUtensorMap& tmA,
                                const CUtensorMap& tmb, int num_sms,
                                int* status, cudaStream_t s) {
  const int64_t blocks = (g.M + GC_ROWS - 1) / GC_ROWS;
  const bool three = blocks > int64_t(g_col_per_sm[0]) * num_sms &&
                     blocks <= int64_t(g_col_per_sm[1]) * num_sms;
  if (three)
    k_gemv_col_tma<3><<<unsigned(blocks), kThreads, gc_smem(3), s>>>(
        tmA, tmb, g.C, (long long)g.ldc, int(g.M), int(g.K), g.sc, status);
  else
    k_gemv_col_tma<4><<<unsigned(blocks), kThreads, gc_smem(4), s>>>(
        tmA, tmb, g.C, (long long)g.ldc, int(g.M), int(g.K), g.sc, status);
  return counted(cudaGetLastError());
}

}  // namespace dfm
