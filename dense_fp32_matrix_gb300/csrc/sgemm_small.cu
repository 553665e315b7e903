// Bandwidth-bound and debug kernels of the FP32 matrix product.
//
//   * gemv_row (M == 1): c = a * B. Every element of B is used once, so the
//     product is a stream over B ("GEMM from naive to tiled", section 十.2:
//     arithmetic intensity 2 flops per 4 bytes of B). A block owns 16 output
//     columns and all of K: 64 row groups of 4 lanes walk K with stride 64,
//     each lane holding 4 columns (one 16-byte load per row when the layout
//     allows), and a shared-memory reduction adds the 64 partial sums in a
//     fixed order. No cross-block reduction, no workspace.
//   * gemv_col (N == 1): c = A * b. One warp per row of A: coalesced
//     (16-byte when aligned) reads along the row, a fixed shuffle tree at
//     the end ("如何让计算受限问题真正达到计算受限", section 7, the GEMV case).
//   * naive: one thread per output, K-loop from global memory, bounds
//     checked ("GEMM from naive to tiled", section 三: thread x along N so a
//     warp reads one contiguous row segment of B). A debug baseline only.
//   * watchdog self-test: one block waits on an mbarrier nothing arrives at,
//     through the same bounded wait the tiled kernel uses.
#include "kernels.h"
#include "ptx.cuh"

namespace dfm {
namespace {

constexpr int ROW_COLS = 16;    // output columns per gemv_row block
constexpr int ROW_GROUPS = 64;  // k-strided row groups per gemv_row block
constexpr int ROW_THREADS = ROW_GROUPS * 4;
constexpr int ROW_UNROLL = 8;

template <bool VEC>
__global__ void __launch_bounds__(ROW_THREADS)
k_gemv_row(const float* __restrict__ a, const float* __restrict__ B,
           long long ldb, float* __restrict__ c, int N, int K, Scale sc) {
  __shared__ float part[ROW_GROUPS][ROW_COLS + 1];
  const int tid = threadIdx.x;
  const int grp = tid >> 2, q = tid & 3;
  const int n = blockIdx.x * ROW_COLS + q * 4;  // first of this lane's 4 cols
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  if (VEC) {
    // Caller guarantees ldb % 4 == 0, N % 4 == 0 and B 16-byte aligned, so
    // a 4-column chunk is either fully inside [0, N) or fully outside.
    if (n < N) {
      const float* col = B + n;
      int k = grp;
      for (; k + (ROW_UNROLL - 1) * ROW_GROUPS < K; k += ROW_UNROLL * ROW_GROUPS) {
        float4 v[ROW_UNROLL];
        float s[ROW_UNROLL];
#pragma unroll
        for (int u = 0; u < ROW_UNROLL; ++u) {
          v[u] = __ldg(reinterpret_cast<const float4*>(
              col + (long long)(k + u * ROW_GROUPS) * ldb));
          s[u] = __ldg(a + k + u * ROW_GROUPS);
        }
#pragma unroll
        for (int u = 0; u < ROW_UNROLL; ++u) {
          acc[0] = fmaf(s[u], v[u].x, acc[0]);
          acc[1] = fmaf(s[u], v[u].y, acc[1]);
          acc[2] = fmaf(s[u], v[u].z, acc[2]);
          acc[3] = fmaf(s[u], v[u].w, acc[3]);
        }
      }
      for (; k < K; k += ROW_GROUPS) {
        const float4 v =
            __ldg(reinterpret_cast<const float4*>(col + (long long)k * ldb));
        const float s = __ldg(a + k);
        acc[0] = fmaf(s, v.x, acc[0]);
        acc[1] = fmaf(s, v.y, acc[1]);
        acc[2] = fmaf(s, v.z, acc[2]);
        acc[3] = fmaf(s, v.w, acc[3]);
      }
    }
  } else {
    // Any layout: the 4 lanes of a group read 16 consecutive columns, lane
    // q columns n0 + q + 4 e, one float each, predicated on N. ROW_UNROLL
    // rows are loaded before any is used, so that their loads are in
    // flight together; each column still sums its rows in k order.
    const int n0 = blockIdx.x * ROW_COLS;
    int k = grp;
    for (; k + (ROW_UNROLL - 1) * ROW_GROUPS < K; k += ROW_UNROLL * ROW_GROUPS) {
      float s[ROW_UNROLL], v[ROW_UNROLL][4];
#pragma unroll
      for (int u = 0; u < ROW_UNROLL; ++u) {
        s[u] = __ldg(a + k + u * ROW_GROUPS);
        const float* row = B + (long long)(k + u * ROW_GROUPS) * ldb + n0;
#pragma unroll
        for (int e = 0; e < 4; ++e)
          v[u][e] = n0 + q + 4 * e < N ? __ldg(row + q + 4 * e) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < ROW_UNROLL; ++u)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[e] = fmaf(s[u], v[u][e], acc[e]);
    }
    for (; k < K; k += ROW_GROUPS) {
      const float s = __ldg(a + k);
      const float* row = B + (long long)k * ldb + n0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = q + 4 * e;
        if (n0 + j < N) acc[e] = fmaf(s, __ldg(row + j), acc[e]);
      }
    }
  }
#pragma unroll
  for (int e = 0; e < 4; ++e) part[grp][VEC ? q * 4 + e : q + 4 * e] = acc[e];
  __syncthreads();
  if (tid < ROW_COLS) {
    const int j = blockIdx.x * ROW_COLS + tid;
    float s = 0.f;
    for (int g = 0; g < ROW_GROUPS; ++g) s += part[g][tid];
    if (j < N) c[j] = epi1(s, c + j, sc);
  }
}

constexpr int COL_WARPS = 8;
constexpr int COL_UNROLL = 16;

template <bool VEC>
__global__ void __launch_bounds__(COL_WARPS * 32)
k_gemv_col(const float* __restrict__ A, long long lda,
           const float* __restrict__ b, long long ldb, float* __restrict__ c,
           long long ldc, int M, int K, Scale sc) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = blockIdx.x * COL_WARPS + warp; i < M;
       i += gridDim.x * COL_WARPS) {
    const float* row = A + (long long)i * lda;
    float acc = 0.f;
    if (VEC) {
      // Caller guarantees lda % 4 == 0, ldb == 1, A and b 16-byte aligned.
      const int K4 = K >> 2;
      const float4* r4 = reinterpret_cast<const float4*>(row);
      const float4* b4 = reinterpret_cast<const float4*>(b);
      int k = lane;
      for (; k + 96 < K4; k += 128) {
        float4 x[4], y[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          x[u] = __ldg(r4 + k + 32 * u);
          y[u] = __ldg(b4 + k + 32 * u);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          acc = fmaf(x[u].x, y[u].x, acc);
          acc = fmaf(x[u].y, y[u].y, acc);
          acc = fmaf(x[u].z, y[u].z, acc);
          acc = fmaf(x[u].w, y[u].w, acc);
        }
      }
      for (; k < K4; k += 32) {
        const float4 x = __ldg(r4 + k), y = __ldg(b4 + k);
        acc = fmaf(x.x, y.x, acc);
        acc = fmaf(x.y, y.y, acc);
        acc = fmaf(x.z, y.z, acc);
        acc = fmaf(x.w, y.w, acc);
      }
      for (int kk = 4 * K4 + lane; kk < K; kk += 32)
        acc = fmaf(__ldg(row + kk), __ldg(b + kk), acc);
    } else {
      // Any layout: COL_UNROLL k per lane loaded before use (in flight
      // together), summed in k order.
      int k = lane;
      for (; k + 32 * (COL_UNROLL - 1) < K; k += 32 * COL_UNROLL) {
        float x[COL_UNROLL], y[COL_UNROLL];
#pragma unroll
        for (int u = 0; u < COL_UNROLL; ++u) {
          x[u] = __ldg(row + k + 32 * u);
          y[u] = __ldg(b + (long long)(k + 32 * u) * ldb);
        }
#pragma unroll
        for (int u = 0; u < COL_UNROLL; ++u) acc = fmaf(x[u], y[u], acc);
      }
      for (; k < K; k += 32)
        acc = fmaf(__ldg(row + k), __ldg(b + (long long)k * ldb), acc);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
      acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (lane == 0) c[(long long)i * ldc] = epi1(acc, c + (long long)i * ldc, sc);
  }
}

// Products too small to fill the GPU: 32 x 32 tiles over 128 threads,
// each a 2 x 4 patch (rows ty and ty + 16, four adjacent columns); k in
// chunks of 32 through shared memory, the next chunk held in registers
// while the current one computes (the register prefetch of "GEMM from
// naive to tiled", section 六). Plain predicated loads, coalesced along k
// for A and along n for B, so any alignment and leading dimension; only
// k < K is summed. A is stored transposed in shared memory with one float
// of padding per row, so the transposing stores hit distinct banks.
constexpr int SM_T = 32;
constexpr int SM_THREADS = 128;
constexpr int SM_KC = 32;

__global__ void __launch_bounds__(SM_THREADS)
k_small(const float* __restrict__ A, long long lda,
        const float* __restrict__ B, long long ldb, float* __restrict__ C,
        long long ldc, int M, int N, int K, Scale sc) {
  __shared__ float As[SM_KC][SM_T + 1];             // As[k][row]
  __shared__ __align__(16) float Bs[SM_KC][SM_T];   // Bs[k][col]
  const int tid = threadIdx.x;
  const int m0 = blockIdx.y * SM_T, n0 = blockIdx.x * SM_T;
  const int lk = tid & 31, lr = tid >> 5;  // loader lane: k (A) / n (B)
  float ra[SM_KC * SM_T / SM_THREADS], rb[SM_KC * SM_T / SM_THREADS];
  auto load = [&](int k0) {
#pragma unroll
    for (int q = 0; q < SM_KC * SM_T / SM_THREADS; ++q) {
      const int r = m0 + lr + 4 * q, ka = k0 + lk;
      ra[q] = (r < M && ka < K) ? A[(long long)r * lda + ka] : 0.f;
      const int kb = k0 + lr + 4 * q, n = n0 + lk;
      rb[q] = (kb < K && n < N) ? B[(long long)kb * ldb + n] : 0.f;
    }
  };
  const int ty = tid >> 3, tx = tid & 7;   // 16 x 8 threads
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  load(0);
  for (int k0 = 0; k0 < K; k0 += SM_KC) {
    __syncthreads();  // the previous chunk has been read
#pragma unroll
    for (int q = 0; q < SM_KC * SM_T / SM_THREADS; ++q) {
      As[lk][lr + 4 * q] = ra[q];
      Bs[lr + 4 * q][lk] = rb[q];
    }
    __syncthreads();
    if (k0 + SM_KC < K) load(k0 + SM_KC);
    const int kn = min(SM_KC, K - k0);
#pragma unroll 8
    for (int k = 0; k < kn; ++k) {
      const float a0 = As[k][ty], a1 = As[k][ty + 16];
      const float4 b = *reinterpret_cast<const float4*>(&Bs[k][4 * tx]);
      acc[0][0] = fmaf(a0, b.x, acc[0][0]);
      acc[0][1] = fmaf(a0, b.y, acc[0][1]);
      acc[0][2] = fmaf(a0, b.z, acc[0][2]);
      acc[0][3] = fmaf(a0, b.w, acc[0][3]);
      acc[1][0] = fmaf(a1, b.x, acc[1][0]);
      acc[1][1] = fmaf(a1, b.y, acc[1][1]);
      acc[1][2] = fmaf(a1, b.z, acc[1][2]);
      acc[1][3] = fmaf(a1, b.w, acc[1][3]);
    }
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = m0 + ty + 16 * i;
    if (r >= M) continue;
    float* crow = C + (long long)r * ldc;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int c = n0 + 4 * tx + e;
      if (c < N) crow[c] = epi1(acc[i][e], crow + c, sc);
    }
  }
}

__global__ void k_naive(const float* __restrict__ A, long long lda,
                        const float* __restrict__ B, long long ldb,
                        float* __restrict__ C, long long ldc, int M, int N,
                        int K, Scale sc) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  for (int i = blockIdx.y * blockDim.y + threadIdx.y; i < M;
       i += gridDim.y * blockDim.y) {
    if (j >= N) continue;
    float acc = 0.f;
    for (int k = 0; k < K; ++k)
      acc = fmaf(A[(long long)i * lda + k], B[(long long)k * ldb + j], acc);
    C[(long long)i * ldc + j] = epi1(acc, C + (long long)i * ldc + j, sc);
  }
}

// out (cols x rows, dense) = in (rows x cols, ld) transposed. 32 x 32
// tiles through shared memory (one padding column: conflict-free), so both
// the reads and the writes are coalesced rows.
constexpr int TR_TILE = 32, TR_ROWS = 8;

__global__ void __launch_bounds__(TR_TILE * TR_ROWS)
k_transpose(const float* __restrict__ in, long long ld, int rows, int cols,
            float* __restrict__ out) {
  __shared__ float t[TR_TILE][TR_TILE + 1];
  const int c0 = blockIdx.x * TR_TILE;
  const int tx = threadIdx.x, ty = threadIdx.y;
  for (long long r0 = (long long)blockIdx.y * TR_TILE; r0 < rows;
       r0 += (long long)gridDim.y * TR_TILE) {
#pragma unroll
    for (int k = 0; k < TR_TILE; k += TR_ROWS) {
      const long long r = r0 + ty + k;
      const int c = c0 + tx;
      if (r < rows && c < cols) t[ty + k][tx] = in[r * ld + c];
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < TR_TILE; k += TR_ROWS) {
      const int c = c0 + ty + k;
      const long long r = r0 + tx;
      if (r < rows && c < cols) out[(long long)c * rows + r] = t[tx][ty + k];
    }
    __syncthreads();  // t is refilled by the next row tile
  }
}

// dst (rows x cols, ld dld) = src (rows x cols, ld sld): a repack with
// another leading dimension, coalesced on both sides; the padding of dst is
// not written. A block owns 256 columns (one per thread) of a run of 8-row
// groups; each thread issues its 8 loads before its stores so that they are
// in flight together. The grid spans columns as well as rows, so a matrix
// with few rows still fills every SM.
constexpr int RP_ROWS = 8;
constexpr int RP_COLS = 256;  // threads per block, one column each
__global__ void __launch_bounds__(RP_COLS)
k_repack(const float* __restrict__ src, long long sld, int rows, int cols,
         float* __restrict__ dst, long long dld) {
  const int c = blockIdx.x * RP_COLS + threadIdx.x;
  if (c >= cols) return;  // no block barrier below
  for (long long r0 = (long long)blockIdx.y * RP_ROWS; r0 < rows;
       r0 += (long long)gridDim.y * RP_ROWS) {
    const int n = rows - r0 < RP_ROWS ? int(rows - r0) : RP_ROWS;
    const float* p = src + r0 * sld + c;
    float* q = dst + r0 * dld + c;
    float v[RP_ROWS];
#pragma unroll
    for (int i = 0; i < RP_ROWS; ++i) v[i] = i < n ? __ldcs(p + i * sld) : 0.f;
#pragma unroll
    for (int i = 0; i < RP_ROWS; ++i)
      if (i < n) q[i * dld] = v[i];
  }
}

__global__ void k_scale_c(float* __restrict__ C, long long ldc, int M, int N,
                          float beta) {
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= N) return;
  for (int i = blockIdx.y; i < M; i += gridDim.y) {
    float* c = C + (long long)i * ldc + j;
    *c = beta == 0.f ? 0.f : beta * *c;
  }
}

__global__ void k_watchdog_selftest(int* status, unsigned long long limit_ns) {
  __shared__ __align__(8) unsigned long long bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 1);
    mbar_fence_init();
  }
  __syncthreads();
  // Nothing arrives on this barrier: the wait must end by its limit.
  const bool ok = mbar_wait_bounded(b, 0, threadIdx.x == 0 ? status : nullptr,
                                    kSiteSelftest, limit_ns);
  __syncthreads_or(!ok);
}

}  // namespace

cudaError_t small_init() { return cudaSuccess; }

cudaError_t launch_gemv_row(const GemmArgs& g, int num_sms, cudaStream_t s) {
  (void)num_sms;
  // 16-byte loads need aligned rows and whole 4-column chunks (N % 4 == 0),
  // so no load reaches past column N - 1.
  const bool vec = (g.ldb % 4 == 0) && (g.N % 4 == 0) &&
                   (reinterpret_cast<uintptr_t>(g.B) % 16 == 0);
  const unsigned blocks = unsigned((g.N + ROW_COLS - 1) / ROW_COLS);
  if (vec)
    k_gemv_row<true><<<blocks, ROW_THREADS, 0, s>>>(g.A, g.B, g.ldb, g.C,
                                                     int(g.N), int(g.K), g.sc);
  else
    k_gemv_row<false><<<blocks, ROW_THREADS, 0, s>>>(g.A, g.B, g.ldb, g.C,
                                                      int(g.N), int(g.K), g.sc);
  return counted(cudaGetLastError());
}

cudaError_t launch_gemv_col(const GemmArgs& g, int num_sms, cudaStream_t s) {
  const bool vec = (g.lda % 4 == 0) && (g.ldb == 1) &&
                   (reinterpret_cast<uintptr_t>(g.A) % 16 == 0) &&
                   (reinterpret_cast<uintptr_t>(g.B) % 16 == 0);
  long long blocks = (g.M + COL_WARPS - 1) / COL_WARPS;
  const long long cap = (long long)num_sms * 16;
  if (blocks > cap) blocks = cap;
  if (vec)
    k_gemv_col<true><<<unsigned(blocks), COL_WARPS * 32, 0, s>>>(
        g.A, g.lda, g.B, g.ldb, g.C, g.ldc, int(g.M), int(g.K), g.sc);
  else
    k_gemv_col<false><<<unsigned(blocks), COL_WARPS * 32, 0, s>>>(
        g.A, g.lda, g.B, g.ldb, g.C, g.ldc, int(g.M), int(g.K), g.sc);
  return counted(cudaGetLastError());
}

cudaError_t launch_small(const GemmArgs& g, cudaStream_t s) {
  const dim3 grid(unsigned((g.N + SM_T - 1) / SM_T),
                  unsigned((g.M + SM_T - 1) / SM_T));
  k_small<<<grid, SM_THREADS, 0, s>>>(g.A, (long long)g.lda, g.B,
                                       (long long)g.ldb, g.C, (long long)g.ldc,
                                       int(g.M), int(g.N), int(g.K), g.sc);
  return counted(cudaGetLastError());
}

cudaError_t launch_naive(const GemmArgs& g, cudaStream_t s) {
  const dim3 block(32, 8);
  long long gy = (g.M + 7) / 8;
  if (gy > 65535) gy = 65535;
  const dim3 grid(unsigned((g.N + 31) / 32), unsigned(gy));
  k_naive<<<grid, block, 0, s>>>(g.A, g.lda, g.B, g.ldb, g.C, g.ldc, int(g.M),
                                 int(g.N), int(g.K), g.sc);
  return counted(cudaGetLastError());
}

cudaError_t launch_transpose(const float* in, int64_t ld, int64_t rows,
                             int64_t cols, float* out, cudaStream_t s) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  const int64_t row_tiles = (rows + TR_TILE - 1) / TR_TILE;
  const dim3 grid(unsigned((cols + TR_TILE - 1) / TR_TILE),
                  unsigned(row_tiles < 65535 ? row_tiles : 65535));
  k_transpose<<<grid, dim3(TR_TILE, TR_ROWS), 0, s>>>(in, (long long)ld,
                                                      int(rows), int(cols), out);
  return counted(cudaGetLastError());
}

cudaError_t launch_repack(const float* src, int64_t sld, int64_t rows,
                          int64_t cols, float* dst, int64_t dld,
                          cudaStream_t s) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  const int64_t groups = (rows + RP_ROWS - 1) / RP_ROWS;
  const dim3 grid(unsigned((cols + RP_COLS - 1) / RP_COLS),
                  unsigned(groups < 65535 ? groups : 65535));
  k_repack<<<grid, RP_COLS, 0, s>>>(src, (long long)sld, int(rows), int(cols),
                                    dst, (long long)dld);
  return counted(cudaGetLastError());
}

cudaError_t launch_scale_c(float* C, int64_t ldc, int64_t M, int64_t N,
                           float beta, cudaStream_t s) {
  if (M == 0 || N == 0) return cudaSuccess;
  long long gy = M < 65535 ? M : 65535;
  k_scale_c<<<dim3(unsigned((N + 255) / 256), unsigned(gy)), 256, 0, s>>>(
      C, (long long)ldc, int(M), int(N), beta);
  return counted(cudaGetLastError());
}

cudaError_t launch_watchdog_selftest(int* status, uint64_t limit_ns,
                                     cudaStream_t s) {
  k_watchdog_selftest<<<1, 32, 0, s>>>(status, limit_ns);
  return counted(cudaGetLastError());
}

}  // namespace dfm
