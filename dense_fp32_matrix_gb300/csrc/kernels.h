// Host-side launch interface between the C-ABI layer (sgemm_abi.cu) and the
// translation units that hold the kernels. No torch types, plain pointers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dfm {

// Kernel launches this library has issued in this process (all devices and
// streams). Every launcher passes the result of its launch through
// counted(), which adds one when the launch was accepted.
void count_launch();
inline cudaError_t counted(cudaError_t e) {
  if (e == cudaSuccess) count_launch();
  return e;
}

// The BLAS epilogue of every kernel: C = alpha * acc + beta * C_old, with
// C_old not read when beta == 0 (alpha = 1, beta = 0 stores acc exactly).
struct Scale {
  float alpha = 1.f;
  float beta = 0.f;
};

#ifdef __CUDACC__
__device__ __forceinline__ float epi1(float acc, const float* c,
                                      const Scale& sc) {
  return sc.beta == 0.f ? sc.alpha * acc : fmaf(sc.alpha, acc, sc.beta * *c);
}
__device__ __forceinline__ float4 epi4(float4 v, const float* c,
                                       const Scale& sc) {
  if (sc.beta == 0.f)
    return make_float4(sc.alpha * v.x, sc.alpha * v.y, sc.alpha * v.z,
                       sc.alpha * v.w);
  const float4 o = *reinterpret_cast<const float4*>(c);
  return make_float4(fmaf(sc.alpha, v.x, sc.beta * o.x),
                     fmaf(sc.alpha, v.y, sc.beta * o.y),
                     fmaf(sc.alpha, v.z, sc.beta * o.z),
                     fmaf(sc.alpha, v.w, sc.beta * o.w));
}
#endif

// One product as the kernels see it: op(A) is M x K, op(B) is K x N.
// op_a == 0: A stored M x K (lda >= K); 1: A stored K x M (lda >= M).
// op_b == 0: B stored K x N (ldb >= N); 1: B stored N x K (ldb >= K).
// Only the tensor-core kernels take op == 1; the dispatcher gives every
// other kernel row-major copies.
struct GemmArgs {
  int64_t M, N, K;
  const float* A;
  int64_t lda;
  const float* B;
  int64_t ldb;
  float* C;
  int64_t ldc;
  Scale sc = Scale();
  int op_a = 0;
  int op_b = 0;
  // Strided batch (tensor-core kernels only): item b reads A + b * stride_a
  // and B + b * stride_b (stride 0: one operand shared by every item) and
  // writes C + b * stride_c.
  int64_t batch = 1;
  int64_t stride_a = 0, stride_b = 0, stride_c = 0;
};

// Tile geometry of the persistent TMA kernel (also used by the host
// dispatcher). Block tile kTileM x kTileN, k-slices of kTileK, a
// kTileStages-deep ring; kTileThreads consumer threads (plus one producer
// warpgroup that issues the copies), one block per SM; each lane owns
// kLaneRows rows x (4 * kLaneChunks) columns of the block tile, with
// kLanesN lanes of a warp along N.
constexpr int kTileM = 256;
constexpr int kTileN = 128;
constexpr int kTileK = 32;
constexpr int kTileStages = 4;
constexpr int kTileThreads = 256;
constexpr int kLaneRows = 16;
constexpr int kLaneChunks = 2;
constexpr int kLanesN = 8;

// One-time per-device kernel attribute set-up. Returns a cudaError_t;
// tiled_init also reports how many TMA tile blocks fit on one SM.
cudaError_t tiled_init(int* tma_blocks_per_sm);
cudaError_t small_init();

// Schedule of the TMA tile kernel: G = min(resident blocks, T) persistent
// blocks over T = tiles x iters_per_tile k-slices: whole tiles in full
// waves, the k-slices of the other tiles split evenly (stream-K).
struct SkPlan {
  int64_t tiles = 0;
  int64_t iters_per_tile = 0;
  int64_t total_iters = 0;
  int grid = 0;
  int64_t dp_tiles = 0;   // tiles dealt whole in full waves
  int64_t sk_iters = 0;   // k-slices of the other tiles, split evenly
  size_t ws_floats = 0;   // workspace: 2 partial tiles per block
  size_t counters = 0;    // kWarpsPerTile per split tile
};
// Smallest share of split k-slices per block worth a fix-up.
constexpr int64_t kMinSkShare = 8;
// The stream-K fix-up counts pieces per (tile, consumer warp).
constexpr int kWarpsPerTile = kTileThreads / 32;
SkPlan plan_stream_k(int64_t M, int64_t N, int64_t K, int resident_blocks);

// Main kernel with TMA loads. tmA / tmB must describe A (dims {K, M}, box
// {kTileK, kTileM}, 128-byte swizzle) and B (dims {N, K}, box {kTileN,
// kTileK}, no swizzle). ws holds pl.ws_floats floats; counters holds
// pl.counters ints, all zero (the kernel leaves them zero when it completes).
cudaError_t launch_tiled_tma(const GemmArgs& g, const CUtensorMap& tmA,
                             const CUtensorMap& tmB, const SkPlan& pl,
                             float* ws, int* counters, int* status,
                             cudaStream_t s);

// Same tile core, operands fetched with predicated 4-byte cp.async (any
// alignment, any leading dimension).
cudaError_t launch_tiled_ldg(const GemmArgs& g, int* status, cudaStream_t s);

// TMA-staged vector kernels (sgemm_gemv.cu). M == 1: B as dims {N, K}, box
// {64, 64}, and a as a rank-1 map of K elements, box {64}; N == 1: A as dims {K, M}, box {256, 16}, and b as a rank-1 map
// of K elements, box {256}. Need 16-byte aligned bases and row strides.
struct GemvRowPlan {
  int64_t col_blocks = 0;   // 64-column strips
  int cluster = 1;          // blocks per strip (k-split), one cluster
  int64_t k_per_block = 0;  // multiple of 64
};
cudaError_t gemv_tma_init();
GemvRowPlan plan_gemv_row(int64_t N, int64_t K, int num_sms);
cudaError_t launch_gemv_row_tma(const GemmArgs& g, const CUtensorMap& tmB,
                                const CUtensorMap& tma_, const GemvRowPlan& pl,
                                int* status, cudaStream_t s);
cudaError_t launch_gemv_col_tma(const GemmArgs& g, const CUtensorMap& tmA,
                                const CUtensorMap& tmb, int num_sms,
                                int* status, cudaStream_t s);

// 3xTF32 tensor-core kernel (sgemm_tf32x3.cu). tmA: A as dims {K, M}, box
// {32, 128}, 128-byte swizzle; tmB: B as dims {N, K}, box {32, 32}, 128-byte
// swizzle. Needs 16-byte aligned bases and row strides.
// tf32x3_init also reports how many 2-block clusters of the pair kernel fit
// on the device at once.
cudaError_t tf32x3_init(int* pair_clusters);
// Split-k for products whose tiles fill under half of the SMs: splits > 1
// multiplies k ranges into `part` (tf32x3_split_floats floats) and adds them
// in order in a second kernel; splits == 1 (or part == nullptr) stores C
// directly.
int plan_tf32x3_splits(int64_t M, int64_t N, int64_t K, int64_t batch,
                       int sms);
size_t tf32x3_split_floats(int64_t M, int64_t N, int64_t batch, int splits);
cudaError_t launch_tf32x3(const GemmArgs& g, const CUtensorMap& tmA,
                          const CUtensorMap& tmB, int* status, cudaStream_t s,
                          int splits = 1, float* part = nullptr);

// 2-SM variant: 256 x 256 tiles, persistent clusters of 2 blocks with a
// stream-K tail (same maps: each block loads A boxes {32, 128} and B boxes
// {32, 32}).
struct PairPlan {
  int tiles_m, tiles_n, tiles;
  int T;              // k-slices of 32 per tile
  int G;              // clusters launched
  int dp_tiles;       // tiles computed whole
  int sk_tiles;       // tiles split by k-slices over all clusters
  int64_t sk_iters;   // sk_tiles * T
  size_t ws_floats;   // partial-tile workspace (0 without stream-K)
  size_t counters;    // tile counters (zero before the launch)
};
// Stream-K shares shorter than this many k-slices are not worth their
// fix-up; the schedule widens the split part by a wave instead.
constexpr int kPairMinSkIters = 8;
PairPlan plan_pair(int64_t M, int64_t N, int64_t K, int clusters,
                   bool stream_k, int64_t batch = 1);
// tmC (may be null): C as dims {N, M, batch items}, box {32, 32, 1},
// 128-byte swizzle; used for whole tiles when beta == 0.
cudaError_t launch_tf32x3_pair(const GemmArgs& g, const CUtensorMap& tmA,
                               const CUtensorMap& tmB, const CUtensorMap* tmC,
                               const PairPlan& pl, float* ws, int* counters,
                               int* status, cudaStream_t s);

// M == 1 and N == 1 bandwidth kernels for any layout; one-thread-per-output
// kernel.
cudaError_t launch_gemv_row(const GemmArgs& g, int num_sms, cudaStream_t s);
cudaError_t launch_gemv_col(const GemmArgs& g, int num_sms, cudaStream_t s);
cudaError_t launch_naive(const GemmArgs& g, cudaStream_t s);
// 32 x 32 tiles with plain loads for products too small to fill the GPU
// (any layout); grid rows: ceil(M / 32) <= 65535.
cudaError_t launch_small(const GemmArgs& g, cudaStream_t s);
constexpr int64_t kSmallMaxRows = 65535 * 32;
// out (cols x rows, dense, ld = rows) = in (rows x cols, ld) transposed.
cudaError_t launch_transpose(const float* in, int64_t ld, int64_t rows,
                             int64_t cols, float* out, cudaStream_t s);
// dst (rows x cols, ld dld) = src (rows x cols, ld sld).
cudaError_t launch_repack(const float* src, int64_t sld, int64_t rows,
                          int64_t cols, float* dst, int64_t dld,
                          cudaStream_t s);
// C = beta * C over M x N (beta == 0: zeros, C not read).
cudaError_t launch_scale_c(float* C, int64_t ldc, int64_t M, int64_t N,
                           float beta, cudaStream_t s);

// One block waiting on an mbarrier that never completes (bounded).
cudaError_t launch_watchdog_selftest(int* status, uint64_t limit_ns,
                                     cudaStream_t s);

}  // namespace dfm

namespace dfm {

// C = A * B like sgemm, but the stream-K TMA path takes its partial tiles
// and tile counters from caller-provided device scratch (ws: ws_floats
// floats, counters: counters_len ints) with at most grid_cap blocks, and no
// device memory is allocated. That path refuses products of more than
// counters_len / kWarpsPerTile tiles (SGEMM_ERR_TOO_LARGE, nothing
// enqueued). The counters used are cleared on the stream
// before the launch. Returns an SGEMM_* status.
int run_with_scratch(int64_t M, int64_t N, int64_t K, const float* A,
                     int64_t lda, const float* B, int64_t ldb, float* C,
                     int64_t ldc, void* stream, float* ws, size_t ws_floats,
                     int* counters, size_t counters_len, int grid_cap);

}  // namespace dfm
