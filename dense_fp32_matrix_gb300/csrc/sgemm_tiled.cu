// Block-tiled FP32 matrix product for sm_103a on the CUDA-core FMA pipe.
//
// Structure (prior art: "GEMM from naive to tiled", sections 五-七, and
// "SGEMM 纯 CUDA 优化总结", ex8/ex9 and Q3-Q8; redesigned for GB300):
//   * output-stationary: one block owns a 128 x 128 tile of C and walks all
//     of K ("如何让计算受限问题真正达到计算受限", section 1.2);
//   * BK = 32 k-slices staged through a 3-deep shared-memory ring, so BK is
//     decoupled from BM/BN (ex8) and each k-slice costs one block barrier
//     (ex9 / section 六);
//   * 8 warps in a 2 x 4 grid, each owning a 64 x 32 warp tile; lanes in an
//     8 x 4 grid (Q8: a square-ish lane shape shares both operands), each
//     lane an 8 x 8 register tile updated by rank-1 (outer-product) steps
//     acc[i][j] += a[i] * b[j] (section 五.1; hotelren.com section 2.2);
//   * the FMA is the Blackwell packed form fma.rn.f32x2, two independent
//     IEEE fp32 fused multiply-adds per instruction, which halves the issue
//     slots the 64 FMAs of one k-step need and leaves room for the shared
//     loads; every output element still receives exactly one fp32 FMA per k,
//     k ascending;
//   * A stays K-major in shared memory (a TMA box cannot transpose, section
//     六.3): the lane reads 4 consecutive k of each of its 8 rows with one
//     128-bit load; rows of a lane are 8 apart so the 8 lanes of a load hit 8
//     consecutive rows, and the TMA 128-byte swizzle (16-byte chunk c of row
//     r stored at chunk c ^ (r mod 8), the XOR swizzle of Q7) makes those
//     8 x 16 bytes land in 32 distinct banks;
//   * B is N-major; a lane's 8 columns are two 4-column chunks 16 apart, so
//     the 4 distinct lane columns of a load cover 64 contiguous bytes
//     (section 五.4's split-column fix of the 4-wavefront conflict);
//   * zero-filled out-of-range loads plus predicated stores handle shapes
//     that are not tile multiples (section 七).
//
// Two loaders feed the same core: TMA (cp.async.bulk.tensor, completion on
// an mbarrier with transaction bytes) when A and B allow 16-byte strides and
// bases, else 4-byte cp.async with zero-fill for any layout.
#include "kernels.h"
#include "ptx.cuh"

namespace dfm {
namespace {

constexpr int BM = kTileM, BN = kTileN, BK = kTileK, STAGES = kTileStages;
constexpr int NT = kTileThreads;
constexpr int WM = 64, WN = 32;       // warp tile
constexpr int WARPS_N = BN / WN;      // 4 (2 along M)
constexpr int TM = 8;                 // rows per lane, 8 apart
constexpr int A_ROW = BK * 4;         // bytes per A row in shared memory
constexpr int B_ROW = BN * 4;         // bytes per B row in shared memory
constexpr int A_STAGE = BM * A_ROW;   // 16 KiB
constexpr int B_STAGE = BK * B_ROW;   // 16 KiB
constexpr int STAGE_TX = A_STAGE + B_STAGE;
constexpr int GROUP_M = 8;            // grouped raster of the tile order
constexpr size_t SMEM_BYTES = size_t(STAGES) * STAGE_TX + 64 + 1024;

static_assert(A_ROW == 128, "A rows are one 128-byte swizzle span");
static_assert((BM / WM) * (BN / WN) * 32 == NT, "warp grid");
static_assert(WM == 8 * TM && WN == 4 * 8, "lane grid 8 x 4, lane tile 8 x 8");

// Tile id -> (tile row, tile col) in groups of GROUP_M tile rows, column by
// column inside a group, so blocks running together share A and B slices in
// L2 (the rasterisation argument of "如何让计算受限问题真正达到计算受限",
// section 5.2.3).
__device__ __forceinline__ void tile_coords(int tile, int tiles_m, int tiles_n,
                                            int& pm, int& pn) {
  const int per_group = GROUP_M * tiles_n;
  const int group = tile / per_group;
  const int first_m = group * GROUP_M;
  const int rows = min(tiles_m - first_m, GROUP_M);
  const int in_group = tile - group * per_group;
  pm = first_m + in_group % rows;
  pn = in_group / rows;
}

// One BK-deep k-slice of rank-1 updates from shared memory.
// a_rows: this lane's first A row in the stage; b_cols: this lane's first B
// column in row 0 of the stage; lane_m == (row mod 8) for all of the lane's
// rows.
__device__ __forceinline__ void compute_slice(f2 (&acc)[TM][4],
                                              const uint8_t* a_rows,
                                              const uint8_t* b_cols,
                                              int lane_m) {
#pragma unroll
  for (int kq = 0; kq < BK / 4; ++kq) {
    float4 a[TM];
    const int chunk = (kq ^ lane_m) << 4;
#pragma unroll
    for (int i = 0; i < TM; ++i)
      a[i] = *reinterpret_cast<const float4*>(a_rows + i * 8 * A_ROW + chunk);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint8_t* brow = b_cols + (kq * 4 + kk) * B_ROW;
      const ulonglong2 b0 = *reinterpret_cast<const ulonglong2*>(brow);
      const ulonglong2 b1 = *reinterpret_cast<const ulonglong2*>(brow + 64);
      const f2 bp0{b0.x}, bp1{b0.y}, bp2{b1.x}, bp3{b1.y};
#pragma unroll
      for (int i = 0; i < TM; ++i) {
        const float av = kk == 0 ? a[i].x : kk == 1 ? a[i].y
                       : kk == 2 ? a[i].z : a[i].w;
        const f2 ap = f2_pack(av, av);
        f2_fma(acc[i][0], ap, bp0);
        f2_fma(acc[i][1], ap, bp1);
        f2_fma(acc[i][2], ap, bp2);
        f2_fma(acc[i][3], ap, bp3);
      }
    }
  }
}

// Write the lane's 8 x 8 results. Row i of the lane is m0 + r0 + 8 i; its
// columns are n0 + c0 + {0..3} and n0 + c0 + 16 + {0..3}.
__device__ __forceinline__ void store_tile(const f2 (&acc)[TM][4], float* C,
                                           int M, int N, long long ldc, int m0,
                                           int n0, int r0, int c0, bool vec) {
#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int r = m0 + r0 + 8 * i;
    if (r >= M) continue;
    float* crow = C + (long long)r * ldc;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int c = n0 + c0 + 16 * h;
      if (vec && c + 3 < N) {
        ulonglong2 v;
        v.x = acc[i][2 * h].v;
        v.y = acc[i][2 * h + 1].v;
        *reinterpret_cast<ulonglong2*>(crow + c) = v;
      } else {
        float x[4];
        f2_unpack(acc[i][2 * h], x[0], x[1]);
        f2_unpack(acc[i][2 * h + 1], x[2], x[3]);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (c + e < N) crow[c + e] = x[e];
      }
    }
  }
}

struct Geometry {
  int m0, n0, r0, c0, lane_m, T;
};

__device__ __forceinline__ Geometry block_geometry(int M, int N, int K) {
  Geometry g;
  const int tiles_m = (M + BM - 1) / BM, tiles_n = (N + BN - 1) / BN;
  int pm, pn;
  tile_coords(blockIdx.x, tiles_m, tiles_n, pm, pn);
  g.m0 = pm * BM;
  g.n0 = pn * BN;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  g.lane_m = lane >> 2;
  g.r0 = (warp / WARPS_N) * WM + g.lane_m;
  g.c0 = (warp % WARPS_N) * WN + (lane & 3) * 4;
  g.T = (K + BK - 1) / BK;
  return g;
}

__device__ __forceinline__ uint8_t* aligned_smem(uint8_t* raw) {
  const uint32_t a = smem_u32(raw);
  return raw + (((a + 1023u) & ~1023u) - a);
}

// ------------------------------------------------------------ TMA kernel

__global__ void __launch_bounds__(NT, 2)
k_tiled_tma(const __grid_constant__ CUtensorMap tmA,
            const __grid_constant__ CUtensorMap tmB, float* __restrict__ C,
            int M, int N, int K, long long ldc, int vec_store, int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_STAGE;
  const uint32_t bar0 = smem_u32(sB + STAGES * B_STAGE);
  const Geometry g = block_geometry(M, N, K);
  const int tid = threadIdx.x;

  auto issue = [&](int tile, int slot) {
    const uint32_t bar = bar0 + 8 * slot;
    mbar_arrive_expect_tx(bar, STAGE_TX);
    tma_load_2d(smem_u32(sA + slot * A_STAGE), &tmA, tile * BK, g.m0, bar);
    tma_load_2d(smem_u32(sB + slot * B_STAGE), &tmB, g.n0, tile * BK, bar);
  };

  if (tid == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    for (int s = 0; s < STAGES; ++s) mbar_init(bar0 + 8 * s, 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (tid == 0)
    for (int s = 0; s < STAGES - 1 && s < g.T; ++s) issue(s, s);

  f2 acc[TM][4];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j].v = 0ull;

  const uint8_t* a_rows = sA + g.r0 * A_ROW;
  const uint8_t* b_cols = sB + g.c0 * 4;
  int slot = 0;
  uint32_t phase = 0;
  for (int t = 0; t < g.T; ++t) {
    const bool ok = mbar_wait_bounded(bar0 + 8 * slot, phase, status,
                                      kSiteTiledFull, kWaitLimitNs);
    // Uniform abort decision; also the barrier after which the slot read in
    // step t-1 is free for the refill below.
    if (__syncthreads_or(!ok)) {
      if (tid == 0) {
        // Let this block's own copies still in flight settle (bounded).
        for (int u = t; u < g.T && u < t + STAGES - 1; ++u) {
          const int su = u % STAGES;
          mbar_wait_bounded(bar0 + 8 * su, (u / STAGES) & 1, nullptr,
                            kSiteTiledDrain, kWaitLimitNs / 100);
        }
      }
      return;
    }
    const int nt = t + STAGES - 1;
    if (tid == 0 && nt < g.T) issue(nt, nt % STAGES);
    compute_slice(acc, a_rows + slot * A_STAGE, b_cols + slot * B_STAGE,
                  g.lane_m);
    if (++slot == STAGES) {
      slot = 0;
      phase ^= 1u;
    }
  }
  store_tile(acc, C, M, N, ldc, g.m0, g.n0, g.r0, g.c0, vec_store != 0);
}

// ------------------------------------------------------- cp.async kernel

__global__ void __launch_bounds__(NT, 2)
k_tiled_ldg(const float* __restrict__ A, long long lda,
            const float* __restrict__ B, long long ldb, float* __restrict__ C,
            int M, int N, int K, long long ldc, int vec_store) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * A_STAGE;
  const Geometry g = block_geometry(M, N, K);
  const int tid = threadIdx.x;

  // A: element e = tid + 256 q of the 128 x 32 slice is row (tid >> 5) + 8 q,
  // column k = tid & 31, stored at the swizzled chunk (k / 4) ^ (row mod 8).
  const int a_k = tid & 31, a_r = tid >> 5;
  const uint32_t a_dst = smem_u32(sA) + a_r * A_ROW +
                         ((((a_k >> 2) ^ a_r) << 4) | ((a_k & 3) << 2));
  // B: element e = tid + 256 q is k-row (tid >> 7) + 2 q, column tid & 127.
  const int b_n = tid & 127, b_k = tid >> 7;
  const uint32_t b_dst = smem_u32(sB) + b_k * B_ROW + b_n * 4;
  const bool b_col_ok = g.n0 + b_n < N;

  auto issue = [&](int tile, int slot) {
    const int k0 = tile * BK;
    const bool ak_ok = k0 + a_k < K;
#pragma unroll
    for (int q = 0; q < BM / 8; ++q) {
      const int r = g.m0 + a_r + 8 * q;
      const bool ok = ak_ok && r < M;
      const float* src = ok ? A + (long long)r * lda + k0 + a_k : A;
      cp_async_4(a_dst + slot * A_STAGE + q * 8 * A_ROW, src, ok ? 4u : 0u);
    }
#pragma unroll
    for (int q = 0; q < BK / 2; ++q) {
      const int kr = k0 + b_k + 2 * q;
      const bool ok = b_col_ok && kr < K;
      const float* src = ok ? B + (long long)kr * ldb + g.n0 + b_n : B;
      cp_async_4(b_dst + slot * B_STAGE + q * 2 * B_ROW, src, ok ? 4u : 0u);
    }
  };

  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < g.T) issue(s, s);
    cp_async_commit();
  }

  f2 acc[TM][4];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j].v = 0ull;

  const uint8_t* a_rows = sA + g.r0 * A_ROW;
  const uint8_t* b_cols = sB + g.c0 * 4;
  int slot = 0;
  for (int t = 0; t < g.T; ++t) {
    cp_async_wait<STAGES - 2>();  // this thread's copies of slice t landed
    __syncthreads();              // everyone's did; slice t-1 fully read
    const int nt = t + STAGES - 1;
    if (nt < g.T) issue(nt, nt % STAGES);
    cp_async_commit();
    compute_slice(acc, a_rows + slot * A_STAGE, b_cols + slot * B_STAGE,
                  g.lane_m);
    if (++slot == STAGES) slot = 0;
  }
  cp_async_wait<0>();
  store_tile(acc, C, M, N, ldc, g.m0, g.n0, g.r0, g.c0, vec_store != 0);
}

int grid_tiles(const GemmArgs& g) {
  return int(((g.M + BM - 1) / BM) * ((g.N + BN - 1) / BN));
}

bool vec_ok(const GemmArgs& g) {
  return (g.ldc % 4 == 0) && (reinterpret_cast<uintptr_t>(g.C) % 16 == 0);
}

}  // namespace

size_t tiled_smem_bytes() { return SMEM_BYTES; }

cudaError_t tiled_init() {
  cudaError_t e = cudaFuncSetAttribute(
      k_tiled_tma, cudaFuncAttributeMaxDynamicSharedMemorySize,
      int(SMEM_BYTES));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k_tiled_ldg,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              int(SMEM_BYTES));
}

cudaError_t launch_tiled_tma(const GemmArgs& g, const CUtensorMap& tmA,
                             const CUtensorMap& tmB, int* status,
                             cudaStream_t s) {
  k_tiled_tma<<<grid_tiles(g), NT, SMEM_BYTES, s>>>(
      tmA, tmB, g.C, int(g.M), int(g.N), int(g.K), (long long)g.ldc,
      vec_ok(g) ? 1 : 0, status);
  return cudaGetLastError();
}

cudaError_t launch_tiled_ldg(const GemmArgs& g, int* status, cudaStream_t s) {
  (void)status;
  k_tiled_ldg<<<grid_tiles(g), NT, SMEM_BYTES, s>>>(
      g.A, (long long)g.lda, g.B, (long long)g.ldb, g.C, int(g.M), int(g.N),
      int(g.K), (long long)g.ldc, vec_ok(g) ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace dfm
