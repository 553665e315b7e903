// Block-tiled FP32 matrix product for sm_103a on the CUDA-core FMA pipe.
//
// Structure (prior art: "GEMM from naive to tiled", sections 五-七 and 十,
// and "SGEMM 纯 CUDA 优化总结", ex8/ex9 and Q3-Q8; redesigned for GB300):
//   * output-stationary: a block owns a BM x BN tile of C and accumulates
//     over K in registers ("如何让计算受限问题真正达到计算受限", section 1.2);
//   * BK = 32 k-slices staged through a STAGES-deep shared-memory ring, so
//     BK is decoupled from BM/BN (ex8);
//   * warps tile the block; each lane owns TM rows x 4 TNC columns and
//     updates them by rank-1 (outer-product) steps acc[i][j] += a[i] * b[j]
//     (section 五.1; hotelren.com section 2.2);
//   * the FMA is the Blackwell packed form fma.rn.f32x2: two independent
//     IEEE fp32 fused multiply-adds per instruction on adjacent output
//     columns, with the row operand a[i] used for both halves; it halves the
//     issue slots the FMAs need. Every output element still receives exactly
//     one fp32 FMA per k, k ascending within a block's k-range;
//   * the packed FMAs of one k run row by row with the column order
//     reversed on every other row ("snake" order), so each FMA shares one
//     source operand with the one before it and reads fewer fresh register
//     operands. Measured on GB300: in register-only cores the snake order
//     takes the FMA pipe from 81.5% to 85% of cycles, and in this kernel
//     from 77.6% to 78.7% of the FP32 FMA peak at 4096^3; the 16 x 8 lane
//     tile (one block per SM, 254 registers) beats the 8 x 8 one (two
//     blocks per SM, 128 registers) in shared-memory-fed cores (85.5% vs
//     82%);
//   * A stays K-major in shared memory (a TMA box cannot transpose, section
//     六.3): a lane reads 4 consecutive k of each of its TM rows with one
//     128-bit load. A lane's rows are LANES_M apart, so the lanes of one load
//     hit consecutive rows, and the TMA 128-byte swizzle (16-byte chunk c of
//     row r stored at chunk c ^ (r mod 8), the XOR swizzle of Q7) puts them
//     in distinct banks;
//   * B is N-major; a lane's columns are TNC chunks of 4 spaced 4 LANES_N
//     apart, so the distinct lane columns of one load are contiguous
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

// Tile geometry of one kernel: block tile BM x BN, k-slices of 32, a
// STAGES-deep ring, NT threads; lanes own TM x (4 TNC) outputs with LANES_N
// lanes of a warp along N.
template <int BM_, int BN_, int STAGES_, int NT_, int TM_, int TNC_,
          int LANES_N_, bool SNAKE_>
struct Cfg {
  static constexpr bool SNAKE = SNAKE_;     // snake order of the FMAs
  static constexpr int BM = BM_, BN = BN_, BK = 32, STAGES = STAGES_;
  static constexpr int NT = NT_;
  static constexpr int TM = TM_;            // rows per lane
  static constexpr int TNC = TNC_;          // 4-column chunks per lane
  static constexpr int TJ = 2 * TNC;        // column pairs per lane
  static constexpr int LANES_N = LANES_N_;  // lanes of a warp along N
  static constexpr int LANES_M = 32 / LANES_N;  // rows LANES_M apart
  static constexpr int WM = LANES_M * TM;   // warp tile
  static constexpr int WN = LANES_N * 4 * TNC;
  static constexpr int WARPS_N = BN / WN;
  static constexpr int WARPS_M = NT / 32 / WARPS_N;
  static constexpr int COL_SPLIT = 4 * LANES_N;  // lane column-chunk spacing
  static constexpr int A_ROW = BK * 4;      // bytes per A row in shared memory
  static constexpr int B_ROW = BN * 4;      // bytes per B row in shared memory
  static constexpr int A_STAGE = BM * A_ROW;
  static constexpr int B_STAGE = BK * B_ROW;
  static constexpr int STAGE_TX = A_STAGE + B_STAGE;
  static_assert(A_ROW == 128, "A rows are one 128-byte swizzle span");
  static_assert(LANES_M * LANES_N == 32 && LANES_M <= 8 && 8 % LANES_M == 0,
                "lane grid");
  static_assert(WARPS_M * WM == BM && WARPS_N * WN == BN, "warp grid");
  static_assert(A_STAGE % 1024 == 0, "swizzled stages stay 1024-aligned");
  static_assert(BM <= 256 && BN <= 256, "TMA box limit");
};

// The persistent TMA kernel: one block per SM, 256 x 128 tiles, 16 x 8
// lane tiles on a 4 x 8 lane grid (a warp's A loads hit 4 rows, its B
// loads 8 column chunks: 2.5 points faster than 8 x 4 at 4096^3), a
// 4-stage ring of 48 KiB stages.
using TmaCfg = Cfg<kTileM, kTileN, kTileStages, kTileThreads, kLaneRows,
                   kLaneChunks, kLanesN, true>;
// The any-layout kernel: one block per 128 x 128 tile, two per SM, 8 x 8
// lane tiles (128 registers), a 3-stage ring; row-major FMA order (the
// snake order costs this register-bound kernel spills).
using LdgCfg = Cfg<128, 128, 3, 256, 8, 2, 4, false>;

static_assert(TmaCfg::BK == kTileK, "k-slice depth");

constexpr int GROUP_M = 8;  // grouped raster of the tile order

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
// a_rows: this lane's first A row in the stage (row r0; its rows are
// r0 + LANES_M i); b_cols: this lane's first B column in row 0 of the stage;
// lane_m: r0 mod LANES_M (r0 - lane_m is a multiple of 8).
template <class C>
__device__ __forceinline__ void compute_slice(f2 (&acc)[C::TM][C::TJ],
                                              const uint8_t* a_rows,
                                              const uint8_t* b_cols,
                                              int lane_m) {
#pragma unroll
  for (int kq = 0; kq < C::BK / 4; ++kq) {
    float4 a[C::TM];
#pragma unroll
    for (int i = 0; i < C::TM; ++i) {
      const int chunk = (kq ^ ((lane_m + C::LANES_M * i) & 7)) << 4;
      a[i] = *reinterpret_cast<const float4*>(a_rows + i * C::LANES_M *
                                              C::A_ROW + chunk);
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint8_t* brow = b_cols + (kq * 4 + kk) * C::B_ROW;
      f2 bp[C::TJ];
#pragma unroll
      for (int c = 0; c < C::TNC; ++c) {
        const ulonglong2 b =
            *reinterpret_cast<const ulonglong2*>(brow + 4 * C::COL_SPLIT * c);
        bp[2 * c].v = b.x;
        bp[2 * c + 1].v = b.y;
      }
#pragma unroll
      for (int i = 0; i < C::TM; ++i) {
        const float av = kk == 0 ? a[i].x : kk == 1 ? a[i].y
                       : kk == 2 ? a[i].z : a[i].w;
        const f2 ap = f2_pack(av, av);
#pragma unroll
        for (int jj = 0; jj < C::TJ; ++jj) {
          // snake order: odd rows run their columns backwards
          const int j = (C::SNAKE && (i & 1)) ? C::TJ - 1 - jj : jj;
          f2_fma(acc[i][j], ap, bp[j]);
        }
      }
    }
  }
}

template <class C>
__device__ __forceinline__ void zero_acc(f2 (&acc)[C::TM][C::TJ]) {
#pragma unroll
  for (int i = 0; i < C::TM; ++i)
#pragma unroll
    for (int j = 0; j < C::TJ; ++j) acc[i][j].v = 0ull;
}

// Write the lane's results. Row i of the lane is m0 + r0 + LANES_M i; chunk
// h covers columns n0 + c0 + COL_SPLIT h + {0..3}.
template <class C>
__device__ __forceinline__ void store_tile(const f2 (&acc)[C::TM][C::TJ],
                                           float* Cm, int M, int N,
                                           long long ldc, int m0, int n0,
                                           int r0, int c0, bool vec,
                                           const Scale& sc) {
#pragma unroll
  for (int i = 0; i < C::TM; ++i) {
    const int r = m0 + r0 + C::LANES_M * i;
    if (r >= M) continue;
    float* crow = Cm + (long long)r * ldc;
#pragma unroll
    for (int h = 0; h < C::TNC; ++h) {
      const int c = n0 + c0 + C::COL_SPLIT * h;
      if (vec && c + 3 < N) {
        float4 v;
        f2_unpack(acc[i][2 * h], v.x, v.y);
        f2_unpack(acc[i][2 * h + 1], v.z, v.w);
        *reinterpret_cast<float4*>(crow + c) = epi4(v, crow + c, sc);
      } else {
        float x[4];
        f2_unpack(acc[i][2 * h], x[0], x[1]);
        f2_unpack(acc[i][2 * h + 1], x[2], x[3]);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          if (c + e < N) crow[c + e] = epi1(x[e], crow + c + e, sc);
      }
    }
  }
}

// Per-lane offsets inside the block tile.
template <class C>
__device__ __forceinline__ int lane_row0(int tid) {
  return (tid >> 5) / C::WARPS_N * C::WM + (tid & 31) / C::LANES_N;
}
template <class C>
__device__ __forceinline__ int lane_col0(int tid) {
  return (tid >> 5) % C::WARPS_N * C::WN + (tid % C::LANES_N) * 4;
}

__device__ __forceinline__ uint8_t* aligned_smem(uint8_t* raw) {
  const uint32_t a = smem_u32(raw);
  return raw + (((a + 1023u) & ~1023u) - a);
}

// ------------------------------------------------------------ TMA kernel
//
// Persistent stream-K schedule ("GEMM from naive to tiled", section 十.1:
// split the total multiply-add work, tiles x k-slices, evenly over a fixed
// set of resident blocks instead of dealing whole tiles in waves, so no
// partly filled last wave is left; section 八.2 measures that loss). Block c
// of G owns k-slice iterations [c T / G, (c+1) T / G) of the T = tiles x I
// iterations laid out tile by tile (I = k-slices per tile, tiles in grouped
// raster order). Its range is a run of segments, each a k-range of one tile:
// a segment that covers its whole tile is stored directly; a partial one
// writes its fp32 partial tile to the workspace and bumps the tile's
// counter. The block that brings the counter to (pieces - 1) adds all pieces
// in piece order (k order), stores C and resets the counter. Nobody waits on
// another block, so there is no co-residency requirement; the summation order
// is fixed, so results are deterministic for a given shape and grid size.
//
// Stage hand-over: a producer warpgroup issues the TMA copies (one thread
// of it), completion on one "full" mbarrier per stage (the copies'
// transaction bytes); the 256 consumer threads compute. Each consumer warp
// arrives on the stage's "empty" mbarrier when it has read the stage; the
// producer waits for all eight and refills the stage with the k-slice
// STAGES later. No consumer waits for another (the warps drift apart by up
// to the ring's depth) and the refill's work stays off the consumers' path.
// setmaxnreg gives the consumers 232 registers and the producers 40
// (2 x 128 x 232 + 128 x 40 = 384 threads x 168 at launch).
// Measured at 4096^3 (% of the FP32 FMA peak at the sampled clock):
//   * consumer thread 0 issuing the copies after one block barrier per
//     k-slice: 77.2%; with the producer warpgroup and the consumers still
//     passing a barrier per k-slice: 78.2%; without it (this scheme): 79.4%
//     (80.5% at 8192^3);
//   * without a producer warpgroup, letting warps drift was slower than the
//     barrier: per-warp "stage empty" mbarriers that thread 0 waits on by
//     2.7 points, the last warp to finish a stage refilling it by 1.1;
//   * an explicit shared->register double buffer of the fragments (each
//     row's next 4-k fragment loaded into the registers its last use
//     frees, the next B fragment during the current k) was 0.5 points
//     slower than the compiler's own scheduling of the unrolled slice, and
//     an L2 prefetch of the boxes three k-slices beyond each copy changed
//     nothing.

constexpr int TNT = TmaCfg::NT;                  // consumer threads
constexpr int T_PRODUCER = 128;                  // the producer warpgroup
constexpr int T_THREADS = TNT + T_PRODUCER;
constexpr int kConsumerRegs = 232, kProducerRegs = 40;
static_assert(TNT == 256, "two consumer warpgroups");
static_assert(2 * 128 * kConsumerRegs + T_PRODUCER * kProducerRegs <=
                  T_THREADS * 168,
              "register split within the launch's 168 per thread");


constexpr size_t TMA_SMEM_BYTES =
    size_t(TmaCfg::STAGES) * TmaCfg::STAGE_TX + 16 * TmaCfg::STAGES + 1024;
constexpr size_t LDG_SMEM_BYTES =
    size_t(LdgCfg::STAGES) * LdgCfg::STAGE_TX + 1024;

struct SkParams {
  int M, N, K;
  long long ldc;
  int tiles_m, tiles_n;
  int iters_per_tile;      // I
  int grid;                // G
  int dp_tiles;            // tiles dealt whole, tile t to block t mod G
  int sk_iters;            // k-slices of the other tiles, split evenly
  float* ws;               // 2 G partial tiles of BM x BN floats
  int* counters;           // kWarpsPerTile per split tile, zero between calls
  int vec_store;
  Scale sc;
  int* status;
};

// Start of block c's share of the split k-slices (the T = sk_iters
// k-slices of the tiles past dp_tiles, laid out tile by tile).
__device__ __forceinline__ int range_begin(int c, const SkParams& p) {
  return int((long long)c * p.sk_iters / p.grid);
}

// Index of the block whose range holds iteration x: the largest c with
// floor(c T / G) <= x.
__device__ __forceinline__ int block_of(int x, const SkParams& p) {
  return int(((long long)(x + 1) * p.grid + p.sk_iters - 1) / p.sk_iters) - 1;
}

// Partial tiles are stored thread-major: value q of thread t at q * NT + t,
// so the stores and loads of a block are fully coalesced 8-byte accesses.
__device__ __forceinline__ void store_partial(
    const f2 (&acc)[TmaCfg::TM][TmaCfg::TJ], unsigned long long* w) {
#pragma unroll
  for (int i = 0; i < TmaCfg::TM; ++i)
#pragma unroll
    for (int j = 0; j < TmaCfg::TJ; ++j)
      __stcg(w + (i * TmaCfg::TJ + j) * TNT + threadIdx.x, acc[i][j].v);
}

__device__ __forceinline__ void add_partial(
    f2 (&sum)[TmaCfg::TM][TmaCfg::TJ], const unsigned long long* w) {
#pragma unroll
  for (int i = 0; i < TmaCfg::TM; ++i)
#pragma unroll
    for (int j = 0; j < TmaCfg::TJ; ++j) {
      const unsigned long long v =
          __ldcg(w + (i * TmaCfg::TJ + j) * TNT + threadIdx.x);
      asm("add.rn.f32x2 %0, %0, %1;" : "+l"(sum[i][j].v) : "l"(v));
    }
}

// Finish one partial segment of `tile` held in acc, warp by warp: each
// warp's share of a partial tile (its lanes' values) is separate, so each
// warp stores its share of the piece, counts itself in on its own counter
// (tile, warp) and, if it is the last of that warp position over the
// tile's pieces, adds the pieces' shares in piece order (k order) and
// writes its part of C. No warp waits for another, so warps that have
// drifted apart by a few k-slices stay apart. Every piece, the last one
// included, goes through the workspace, so the sum does not depend on
// which block arrives last. my_slot: workspace slot of this piece.
__device__ __forceinline__ void sk_fixup(
    const f2 (&acc)[TmaCfg::TM][TmaCfg::TJ], int tile, int my_slot,
    const SkParams& p, float* C, int m0, int n0, int r0, int c0) {
  unsigned long long* ws = reinterpret_cast<unsigned long long*>(p.ws);
  constexpr int SLOT = TmaCfg::BM * TmaCfg::BN / 2;  // f2 values per tile
  const int lane = threadIdx.x & 31;
  const int sk_tile = tile - p.dp_tiles;
  int* counter = p.counters + sk_tile * kWarpsPerTile + (threadIdx.x >> 5);
  store_partial(acc, ws + (long long)my_slot * SLOT);
  __threadfence();
  __syncwarp();
  int arrived = 0;
  if (lane == 0) arrived = atomicAdd(counter, 1);
  arrived = __shfl_sync(0xffffffffu, arrived, 0);
  const int x0 = sk_tile * p.iters_per_tile;
  const int c_first = block_of(x0, p);
  const int c_last = block_of(x0 + p.iters_per_tile - 1, p);
  const int pieces = c_last - c_first + 1;
  if (arrived != pieces - 1) return;
  __threadfence();
  f2 sum[TmaCfg::TM][TmaCfg::TJ];
  zero_acc<TmaCfg>(sum);
  for (int j = 0; j < pieces; ++j) {
    const int cj = c_first + j;
    // A block's piece of this tile is its first segment when its range
    // starts inside the tile, else the last segment of its range.
    const int slot = 2 * cj + (range_begin(cj, p) >= x0 ? 0 : 1);
    add_partial(sum, ws + (long long)slot * SLOT);
  }
  store_tile<TmaCfg>(sum, C, p.M, p.N, p.ldc, m0, n0, r0, c0,
                     p.vec_store != 0, p.sc);
  __syncwarp();
  if (lane == 0) *counter = 0;
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar)
               : "memory");
}

// Bounded wait that also gives up at once when a thread of the block has
// already recorded a timeout (*abort_flag != 0). After an abort the block
// runs its remaining iterations without waiting or computing, so every
// thread still reaches every block barrier; the status word tells the host
// that the results are void.
__device__ __forceinline__ bool wait_stage(uint32_t bar, uint32_t parity,
                                           volatile int* abort_flag, int* status,
                                           int site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 1; it < (1u << 31); ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0) {
      if (*abort_flag != 0) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) break;
    }
  }
  record_timeout(status, site);
  *abort_flag = 1;
  return false;
}

// A block's work as a run of segments, each a k-range of one tile: first
// its share of the split k-slices (tile by tile, a partial segment at
// either end), then its whole tiles (b, b + G, ... below dp_tiles). The
// producer and the consumers walk the same sequence.
struct Segments {
  int x, x_end;  // next split k-slice, end of the share
  int dp_next;   // next whole tile
};
struct Segment {
  int tile, kt0, len;
  bool whole;
};

__device__ __forceinline__ Segments block_segments(const SkParams& p) {
  Segments sg;
  sg.x = range_begin(blockIdx.x, p);
  sg.x_end = range_begin(blockIdx.x + 1, p);
  sg.dp_next = blockIdx.x;
  return sg;
}

__device__ __forceinline__ bool next_segment(Segments& sg, const SkParams& p,
                                             Segment& g) {
  const int I = p.iters_per_tile;
  if (sg.x < sg.x_end) {
    const int t = sg.x / I;
    const int end = min(sg.x_end, (t + 1) * I);
    g.tile = p.dp_tiles + t;
    g.kt0 = sg.x - t * I;
    g.len = end - sg.x;
    g.whole = g.kt0 == 0 && g.len == I;
    sg.x = end;
    return true;
  }
  if (sg.dp_next < p.dp_tiles) {
    g.tile = sg.dp_next;
    g.kt0 = 0;
    g.len = I;
    g.whole = true;
    sg.dp_next += p.grid;
    return true;
  }
  return false;
}

__global__ void __launch_bounds__(T_THREADS, 1)
k_tiled_tma(const __grid_constant__ CUtensorMap tmA,
            const __grid_constant__ CUtensorMap tmB, float* __restrict__ C,
            const SkParams p) {
  using Cf = TmaCfg;
  constexpr int STAGES = Cf::STAGES;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_abort;
  uint8_t* smem = aligned_smem(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * Cf::A_STAGE;
  const uint32_t full0 = smem_u32(sB + STAGES * Cf::B_STAGE);
  const uint32_t empty0 = full0 + 8 * STAGES;
  volatile int* abort_flag = &s_abort;
  const int tid = threadIdx.x;

  if (tid == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
    for (int sl = 0; sl < STAGES; ++sl) {
      mbar_init(full0 + 8 * sl, 1);
      mbar_init(empty0 + 8 * sl, TNT / 32);  // one arrival per warp
    }
    mbar_fence_init();
    s_abort = 0;
  }
  __syncthreads();  // the last barrier the producer warpgroup joins

  if (tid >= TNT) {
    // ---- producer warpgroup: one thread issues the copies.
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProducerRegs));
    if (tid != TNT) return;
    Segments sg = block_segments(p);
    Segment g;
    int issued = 0;  // local k-slices issued
    bool stop = false;
    while (!stop && next_segment(sg, p, g)) {
      int pm, pn;
      tile_coords(g.tile, p.tiles_m, p.tiles_n, pm, pn);
      for (int s = 0; s < g.len; ++s) {
        const int v = issued, sl = v % STAGES;
        // use v / STAGES - 1 of the slot (local k-slice v - STAGES) read
        if ((v >= STAGES &&
             !wait_stage(empty0 + 8 * sl, uint32_t(v / STAGES - 1) & 1u,
                         abort_flag, p.status, kSiteTiledEmpty)) ||
            *abort_flag != 0) {
          stop = true;
          break;
        }
        const uint32_t bar = full0 + 8 * sl;
        mbar_arrive_expect_tx(bar, Cf::STAGE_TX);
        tma_load_2d(smem_u32(sA + sl * Cf::A_STAGE), &tmA,
                    (g.kt0 + s) * Cf::BK, pm * Cf::BM, bar);
        tma_load_2d(smem_u32(sB + sl * Cf::B_STAGE), &tmB, pn * Cf::BN,
                    (g.kt0 + s) * Cf::BK, bar);
        issued = v + 1;
      }
    }
    // The block's shared memory lives until this thread exits: let the
    // last copy of each slot land (at once unless the block aborted).
    for (int v = issued - STAGES > 0 ? issued - STAGES : 0; v < issued; ++v)
      mbar_wait_bounded(full0 + 8 * (v % STAGES), uint32_t(v / STAGES) & 1u,
                        nullptr, kSiteTiledDrain, kWaitLimitNs / 100);
    return;
  }

  // ---- consumers
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kConsumerRegs));
  f2 acc[Cf::TM][Cf::TJ];
  zero_acc<Cf>(acc);

  const int lane_m = (tid & 31) / Cf::LANES_N;
  const int r0 = lane_row0<Cf>(tid), c0 = lane_col0<Cf>(tid);
  const uint8_t* a_rows = sA + r0 * Cf::A_ROW;
  const uint8_t* b_cols = sB + c0 * 4;
  int slot = 0;
  uint32_t phase = 0;
  Segments sg = block_segments(p);
  Segment g;
  for (int seg = 0; next_segment(sg, p, g); ++seg) {
    for (int s = 0; s < g.len; ++s) {
      const bool landed = wait_stage(full0 + 8 * slot, phase, abort_flag,
                                     p.status, kSiteTiledFull);
      if (__all_sync(0xffffffffu, landed))
        compute_slice<Cf>(acc, a_rows + slot * Cf::A_STAGE,
                          b_cols + slot * Cf::B_STAGE, lane_m);
      // this warp is done with the stage: once all eight are, the
      // producer refills it with the k-slice STAGES later
      __syncwarp();
      if ((tid & 31) == 0) mbar_arrive(empty0 + 8 * slot);
      if (++slot == STAGES) {
        slot = 0;
        phase ^= 1u;
      }
    }
    int pm, pn;
    tile_coords(g.tile, p.tiles_m, p.tiles_n, pm, pn);
    if (g.whole)
      store_tile<Cf>(acc, C, p.M, p.N, p.ldc, pm * Cf::BM, pn * Cf::BN, r0,
                     c0, p.vec_store != 0, p.sc);
    else  // the first segment of a share is piece 0, its last one piece 1
      sk_fixup(acc, g.tile, 2 * blockIdx.x + (seg == 0 ? 0 : 1), p, C,
               pm * Cf::BM, pn * Cf::BN, r0, c0);
    zero_acc<Cf>(acc);
  }
}

// ------------------------------------------------------- cp.async kernel
//
// One block per output tile (no persistence), operands copied 4 bytes at a
// time with zero-fill, into the same shared layouts as the TMA path.

__global__ void __launch_bounds__(LdgCfg::NT, 2)
k_tiled_ldg(const float* __restrict__ A, long long lda,
            const float* __restrict__ B, long long ldb, float* __restrict__ C,
            int M, int N, int K, long long ldc, int vec_store, Scale sc) {
  using Cf = LdgCfg;
  constexpr int NT = Cf::NT, STAGES = Cf::STAGES, BM = Cf::BM, BN = Cf::BN,
                BK = Cf::BK;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = aligned_smem(smem_raw);
  uint8_t* sA = smem;
  uint8_t* sB = smem + STAGES * Cf::A_STAGE;
  const int tid = threadIdx.x;
  const int tiles_m = (M + BM - 1) / BM, tiles_n = (N + BN - 1) / BN;
  int pm, pn;
  tile_coords(blockIdx.x, tiles_m, tiles_n, pm, pn);
  const int m0 = pm * BM, n0 = pn * BN;
  const int T = (K + BK - 1) / BK;

  // A: element e = tid + NT q of the BM x 32 slice is row tid / 32 +
  // (NT / 32) q, column k = tid mod 32, stored at the swizzled chunk
  // (k / 4) ^ (row mod 8).
  constexpr int A_ROWS_PER_PASS = NT / 32;
  static_assert(A_ROWS_PER_PASS % 8 == 0, "row mod 8 fixed per thread");
  const int a_k = tid & 31, a_r = tid >> 5;
  const uint32_t a_dst = smem_u32(sA) + a_r * Cf::A_ROW +
                         ((((a_k >> 2) ^ (a_r & 7)) << 4) | ((a_k & 3) << 2));
  // B: element e = tid + NT q is k-row tid / BN + (NT / BN) q, column
  // tid mod BN.
  constexpr int B_ROWS_PER_PASS = NT / BN;
  static_assert(NT % BN == 0, "B rows per pass");
  const int b_n = tid % BN, b_k = tid / BN;
  const uint32_t b_dst = smem_u32(sB) + b_k * Cf::B_ROW + b_n * 4;
  const bool b_col_ok = n0 + b_n < N;

  auto issue = [&](int tile, int slot) {
    const int k0 = tile * BK;
    const bool ak_ok = k0 + a_k < K;
#pragma unroll
    for (int q = 0; q < BM / A_ROWS_PER_PASS; ++q) {
      const int r = m0 + a_r + A_ROWS_PER_PASS * q;
      const bool ok = ak_ok && r < M;
      const float* src = ok ? A + (long long)r * lda + k0 + a_k : A;
      cp_async_4(a_dst + slot * Cf::A_STAGE + q * A_ROWS_PER_PASS * Cf::A_ROW,
                 src, ok ? 4u : 0u);
    }
#pragma unroll
    for (int q = 0; q < BK / B_ROWS_PER_PASS; ++q) {
      const int kr = k0 + b_k + B_ROWS_PER_PASS * q;
      const bool ok = b_col_ok && kr < K;
      const float* src = ok ? B + (long long)kr * ldb + n0 + b_n : B;
      cp_async_4(b_dst + slot * Cf::B_STAGE + q * B_ROWS_PER_PASS * Cf::B_ROW,
                 src, ok ? 4u : 0u);
    }
  };

  for (int s = 0; s < STAGES - 1; ++s) {
    if (s < T) issue(s, s);
    cp_async_commit();
  }

  f2 acc[Cf::TM][Cf::TJ];
  zero_acc<Cf>(acc);
  const int lane_m = (tid & 31) / Cf::LANES_N;
  const uint8_t* a_rows = sA + lane_row0<Cf>(tid) * Cf::A_ROW;
  const uint8_t* b_cols = sB + lane_col0<Cf>(tid) * 4;
  int slot = 0;
  for (int t = 0; t < T; ++t) {
    cp_async_wait<STAGES - 2>();  // this thread's copies of slice t landed
    __syncthreads();              // everyone's did; slice t-1 fully read
    const int nt = t + STAGES - 1;
    if (nt < T) issue(nt, nt % STAGES);
    cp_async_commit();
    compute_slice<Cf>(acc, a_rows + slot * Cf::A_STAGE,
                      b_cols + slot * Cf::B_STAGE, lane_m);
    if (++slot == STAGES) slot = 0;
  }
  cp_async_wait<0>();
  store_tile<Cf>(acc, C, M, N, ldc, m0, n0, lane_row0<Cf>(tid),
                 lane_col0<Cf>(tid), vec_store != 0, sc);
}

bool vec_ok(const GemmArgs& g) {
  return (g.ldc % 4 == 0) && (reinterpret_cast<uintptr_t>(g.C) % 16 == 0);
}

}  // namespace

cudaError_t tiled_init(int* tma_blocks_per_sm) {
  cudaError_t e = cudaFuncSetAttribute(
      k_tiled_tma, cudaFuncAttributeMaxDynamicSharedMemorySize,
      int(TMA_SMEM_BYTES));
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_tiled_ldg,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           int(LDG_SMEM_BYTES));
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      tma_blocks_per_sm, k_tiled_tma, T_THREADS, TMA_SMEM_BYTES);
}

SkPlan plan_stream_k(int64_t M, int64_t N, int64_t K, int resident_blocks) {
  SkPlan pl;
  pl.tiles = ((M + kTileM - 1) / kTileM) * ((N + kTileN - 1) / kTileN);
  pl.iters_per_tile = (K + kTileK - 1) / kTileK;
  pl.total_iters = pl.tiles * pl.iters_per_tile;
  pl.grid = resident_blocks < pl.total_iters ? resident_blocks
                                             : int(pl.total_iters);
  if (pl.grid < 1) pl.grid = 1;
  // Whole tiles in full waves; the k-slices of the remaining tiles split
  // evenly over all blocks. A share under kMinSkShare k-slices would cut
  // each of those tiles into many small pieces: one more wave is split.
  int64_t waves = pl.tiles / pl.grid;
  const int64_t rest = pl.tiles - waves * pl.grid;
  if (waves > 0 && rest > 0 &&
      rest * pl.iters_per_tile < kMinSkShare * int64_t(pl.grid))
    --waves;
  pl.dp_tiles = waves * pl.grid;
  pl.sk_iters = (pl.tiles - pl.dp_tiles) * pl.iters_per_tile;
  pl.ws_floats = size_t(2) * pl.grid * kTileM * kTileN;
  pl.counters = size_t(pl.tiles - pl.dp_tiles) * kWarpsPerTile;
  return pl;
}

cudaError_t launch_tiled_tma(const GemmArgs& g, const CUtensorMap& tmA,
                             const CUtensorMap& tmB, const SkPlan& pl,
                             float* ws, int* counters, int* status,
                             cudaStream_t s) {
  SkParams p;
  p.M = int(g.M);
  p.N = int(g.N);
  p.K = int(g.K);
  p.ldc = (long long)g.ldc;
  p.tiles_m = int((g.M + kTileM - 1) / kTileM);
  p.tiles_n = int((g.N + kTileN - 1) / kTileN);
  p.iters_per_tile = int(pl.iters_per_tile);
  p.dp_tiles = int(pl.dp_tiles);
  p.sk_iters = int(pl.sk_iters);
  p.grid = pl.grid;
  p.ws = ws;
  p.counters = counters;
  p.vec_store = vec_ok(g) ? 1 : 0;
  p.sc = g.sc;
  p.status = status;
  k_tiled_tma<<<pl.grid, T_THREADS, TMA_SMEM_BYTES, s>>>(tmA, tmB, g.C, p);
  return counted(cudaGetLastError());
}

cudaError_t launch_tiled_ldg(const GemmArgs& g, int* status, cudaStream_t s) {
  (void)status;
  const int grid = int(((g.M + LdgCfg::BM - 1) / LdgCfg::BM) *
                       ((g.N + LdgCfg::BN - 1) / LdgCfg::BN));
  k_tiled_ldg<<<grid, LdgCfg::NT, LDG_SMEM_BYTES, s>>>(
      g.A, (long long)g.lda, g.B, (long long)g.ldb, g.C, int(g.M), int(g.N),
      int(g.K), (long long)g.ldc, vec_ok(g) ? 1 : 0, g.sc);
  return counted(cudaGetLastError());
}

}  // namespace dfm
