// FP32 matrix product on the tcgen05 tensor cores by three TF32 products
// (3xTF32; the surveyed error-compensated split of Ootomo and Yokota, 2022).
//
// Every fp32 operand x is split exactly into x = hi + lo, hi = x with its 13
// low mantissa bits cleared (a TF32 value) and lo = x - hi (at most 13
// significant bits). The product is accumulated in fp32 tensor memory as
//     C = A_lo B_hi + A_hi B_lo + A_hi B_hi
// (the A_lo B_lo term, about 2^-22 of the product, is dropped). TF32 products
// are exact in fp32, so each product carries a relative error of about
// 2^-21 against the exact fp32 product: far inside the 1e-4 sum-of-|products|
// bound the FFMA path is held to, and exact on small-integer data (lo = 0).
// The pages name TF32 only as a hazard (a cuBLAS switch that silently drops
// precision, "GEMM from naive to tiled" 十一.2); the compensated split is what
// makes the tensor cores usable for an fp32 result.
//
// One block per 128 x 128 output tile, k-slices of 32, a 3-stage ring of
// {A, A_lo, B, B_lo} tiles (64 KiB each) in shared memory:
//   warp 0      TMA producer: A box {32 k, 128 rows}, B as 4 boxes
//               {32 n, 32 k}, all with the 128-byte swizzle;
//   warps 2..5  split each landed stage: A elementwise in place (hi) and
//               into the A_lo buffer; B transposed as well (below); then
//               after the last stage read the accumulator from tensor
//               memory and store C;
//   warp 1      allocates 128 tensor-memory columns and issues the MMAs
//               (M = 128, N = 128, K = 8 per instruction) from one thread,
//               releasing each stage with tcgen05.commit.
// The TF32 MMA takes only K-major operands (the MN-major descriptor bit
// gives zeros for kind::tf32 on this part), so both A and B are presented as
// 128-byte rows of 32 k in the canonical 128-byte-swizzled layout. A lands
// that way from TMA. B lands N-major (box rows are 32 n of one k); each split
// warp owns one 32 x 32 box: every lane gathers one column n across the 32 k
// rows, then the warp writes the box back in place as 32 K-major rows (hi)
// and the matching rows of B_lo. Same 4 KiB footprint, no extra buffer.
#include "kernels.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace dfm {
namespace {

constexpr int XM = 128, XN = 128, XK = 32, XSTAGES = 3;
constexpr int X_THREADS = 192;                       // 6 warps
constexpr int X_A_BYTES = XM * XK * 4;               // 16 KiB
constexpr int X_B_BYTES = XK * XN * 4;               // 16 KiB
constexpr int X_B_BOX = XK * 32 * 4;                 // 4 KiB: 32 k x 32 n
constexpr int X_STAGE = 2 * X_A_BYTES + 2 * X_B_BYTES;
constexpr int X_TMEM_COLS = 128;
constexpr int X_CONV_THREADS = 128;                  // warps 2..5
constexpr size_t X_SMEM = size_t(XSTAGES) * X_STAGE + 1024 + 256;
constexpr int X_GROUP_M = 8;

static_assert(X_A_BYTES % 1024 == 0 && X_B_BOX % 1024 == 0, "swizzle atoms");
static_assert(XN / 32 == X_CONV_THREADS / 32, "one B box per split warp");

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void fence_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// hi: x with the low 13 mantissa bits cleared; lo = x - hi (exact). Inf and
// NaN keep their bits in hi and give lo = 0.
__device__ __forceinline__ void split_tf32(float x, float& hi, float& lo) {
  const uint32_t b = __float_as_uint(x);
  const bool special = (b & 0x7F800000u) == 0x7F800000u;
  const uint32_t h = special ? b : (b & 0xFFFFE000u);
  hi = __uint_as_float(h);
  lo = special ? 0.f : x - hi;
}

__device__ __forceinline__ void split4(uint8_t* hi_buf, uint8_t* lo_buf,
                                       int idx) {
  float4* hp = reinterpret_cast<float4*>(hi_buf) + idx;
  float4* lp = reinterpret_cast<float4*>(lo_buf) + idx;
  const float4 x = *hp;
  float4 h, l;
  split_tf32(x.x, h.x, l.x);
  split_tf32(x.y, h.y, l.y);
  split_tf32(x.z, h.z, l.z);
  split_tf32(x.w, h.w, l.w);
  *hp = h;
  *lp = l;
}

// Box j of a B stage (32 k rows x 32 n, N-major, TMA 128-byte swizzle) ->
// K-major rows n = 32 j + lane of B (hi, in place) and B_lo.
__device__ __forceinline__ void split_transpose_box(uint8_t* box, uint8_t* lo_box,
                                                   int lane) {
  float x[32];
  const int cb = (lane * 4) / 16, cw = (lane * 4) % 16;
#pragma unroll
  for (int k = 0; k < 32; ++k)
    x[k] = *reinterpret_cast<const float*>(box + k * 128 +
                                           ((cb ^ (k & 7)) << 4) + cw);
  __syncwarp();  // every lane has read the whole box before any write
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    float4 h, l;
    split_tf32(x[4 * c + 0], h.x, l.x);
    split_tf32(x[4 * c + 1], h.y, l.y);
    split_tf32(x[4 * c + 2], h.z, l.z);
    split_tf32(x[4 * c + 3], h.w, l.w);
    const int off = lane * 128 + ((c ^ (lane & 7)) << 4);
    *reinterpret_cast<float4*>(box + off) = h;
    *reinterpret_cast<float4*>(lo_box + off) = l;
  }
}

__device__ __forceinline__ void tile_of(int tile, int tiles_m, int tiles_n,
                                        int& pm, int& pn) {
  const int per_group = X_GROUP_M * tiles_n;
  const int group = tile / per_group;
  const int first_m = group * X_GROUP_M;
  const int rows = min(tiles_m - first_m, X_GROUP_M);
  const int in_group = tile - group * per_group;
  pm = first_m + in_group % rows;
  pn = in_group / rows;
}

__global__ void __launch_bounds__(X_THREADS, 1)
k_tf32x3(const __grid_constant__ CUtensorMap tmA,
         const __grid_constant__ CUtensorMap tmB, float* __restrict__ C, int M,
         int N, int K, long long ldc, int tiles_m, int tiles_n, int vec_store,
         int* status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t* ctrl = smem + XSTAGES * X_STAGE;
  const uint32_t full0 = smem_u32(ctrl);          // TMA landed
  const uint32_t conv0 = full0 + 8 * XSTAGES;     // split done
  const uint32_t empty0 = conv0 + 8 * XSTAGES;    // MMAs done reading
  const uint32_t accf = empty0 + 8 * XSTAGES;     // accumulator complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 8 * (3 * XSTAGES + 1));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  auto A_of = [&](int s) { return smem + s * X_STAGE; };
  auto Alo_of = [&](int s) { return smem + s * X_STAGE + X_A_BYTES; };
  auto B_of = [&](int s) { return smem + s * X_STAGE + 2 * X_A_BYTES; };
  auto Blo_of = [&](int s) {
    return smem + s * X_STAGE + 2 * X_A_BYTES + X_B_BYTES;
  };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int pm, pn;
  tile_of(blockIdx.x, tiles_m, tiles_n, pm, pn);
  const int m0 = pm * XM, n0 = pn * XN;
  const int T = (K + XK - 1) / XK;

  if (tid == 0) {
    for (int s = 0; s < XSTAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(conv0 + 8 * s, X_CONV_THREADS / 32);
      mbar_init(empty0 + 8 * s, 1);
    }
    mbar_init(accf, 1);
    *abort_flag = 0;
    mbar_fence_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tc::tmem_alloc(smem_u32(tmem_slot), X_TMEM_COLS);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      for (int t = 0; t < T && !*abort_flag; ++t) {
        const int s = t % XSTAGES;
        if (t >= XSTAGES &&
            !mbar_wait_bounded(empty0 + 8 * s, ((t / XSTAGES) - 1) & 1, status,
                               kSiteTf32Empty, kWaitLimitNs)) {
          *abort_flag = 1;
          break;
        }
        const uint32_t bar = full0 + 8 * s;
        mbar_arrive_expect_tx(bar, X_A_BYTES + X_B_BYTES);
        tma_load_2d(smem_u32(A_of(s)), &tmA, t * XK, m0, bar);
        for (int j = 0; j < XN / 32; ++j)
          tma_load_2d(smem_u32(B_of(s) + j * X_B_BOX), &tmB, n0 + 32 * j,
                      t * XK, bar);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_tf32(XM, XN, false, false);
      for (int t = 0; t < T; ++t) {
        const int s = t % XSTAGES;
        if (*abort_flag ||
            !mbar_wait_bounded(conv0 + 8 * s, (t / XSTAGES) & 1, status,
                               kSiteTf32Conv, kWaitLimitNs)) {
          *abort_flag = 1;
          break;
        }
        tc::fence_after_sync();
        const uint32_t a = smem_u32(A_of(s)), al = smem_u32(Alo_of(s));
        const uint32_t b = smem_u32(B_of(s)), bl = smem_u32(Blo_of(s));
#pragma unroll
        for (int ks = 0; ks < XK / 8; ++ks) {
          // K-major, 128-byte rows of 32 k, 8-row groups 1 KiB apart; the
          // k-step of 8 advances 32 bytes inside the swizzled rows.
          const uint64_t da = tc::smem_desc(a + 32 * ks, 16, 1024,
                                            tc::kLayoutSwizzle128);
          const uint64_t dal = tc::smem_desc(al + 32 * ks, 16, 1024,
                                             tc::kLayoutSwizzle128);
          const uint64_t db = tc::smem_desc(b + 32 * ks, 16, 1024,
                                            tc::kLayoutSwizzle128);
          const uint64_t dbl = tc::smem_desc(bl + 32 * ks, 16, 1024,
                                             tc::kLayoutSwizzle128);
          tc::mma_tf32(tmem, dal, db, idesc, (t > 0 || ks > 0) ? 1u : 0u);
          tc::mma_tf32(tmem, da, dbl, idesc, 1u);
          tc::mma_tf32(tmem, da, db, idesc, 1u);
        }
        tc::commit(empty0 + 8 * s);   // stage s may be refilled
      }
      tc::commit(accf);               // accumulator complete
    }
  } else {
    // ---------------------------------------------------------- split
    const int ct = tid - 64;  // 0..127
    for (int t = 0; t < T; ++t) {
      const int s = t % XSTAGES;
      if (*abort_flag ||
          !mbar_wait_bounded(full0 + 8 * s, (t / XSTAGES) & 1, status,
                             kSiteTf32Full, kWaitLimitNs)) {
        *abort_flag = 1;
        break;
      }
#pragma unroll
      for (int q = 0; q < X_A_BYTES / 16 / X_CONV_THREADS; ++q)
        split4(A_of(s), Alo_of(s), ct + X_CONV_THREADS * q);
      // warp w - 2 owns B box w - 2 (columns 32 (w - 2) .. + 31)
      split_transpose_box(B_of(s) + (warp - 2) * X_B_BOX,
                          Blo_of(s) + (warp - 2) * X_B_BOX, lane);
      fence_async_shared();  // generic writes -> visible to the MMA
      __syncwarp();
      if (lane == 0) mbar_arrive(conv0 + 8 * s);
    }
    // ---------------------------------------------------------- epilogue
    const bool ok = mbar_wait_bounded(accf, 0, status, kSiteTf32Acc,
                                      *abort_flag ? kWaitLimitNs / 100
                                                  : kWaitLimitNs);
    tc::fence_after_sync();
    const int quarter = warp & 3;  // this warp's tensor-memory lanes
    const int r = m0 + 32 * quarter + lane;
    float* crow = C + (long long)r * ldc;
#pragma unroll 1
    for (int cb = 0; cb < XN / 32; ++cb) {
      uint32_t v[32];
      tc::tmem_ld_32x32b_x32(tmem + (uint32_t(32 * quarter) << 16) + 32 * cb,
                             v);
      tc::tmem_ld_wait();
      if (!ok || *abort_flag || r >= M) continue;
      const int c0 = n0 + 32 * cb;
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const int c = c0 + e;
        if (vec_store && c + 3 < N) {
          *reinterpret_cast<float4*>(crow + c) =
              make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]),
                          __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
        } else {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (c + u < N) crow[c + u] = __uint_as_float(v[e + u]);
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, X_TMEM_COLS);
  }
}

// ---------------------------------------------------------------- pairs
//
// 2-SM variant: a cluster of two blocks computes a 256 x 256 tile with the
// pair MMA (M = 256, N = 256, K = 8). Block r of the pair holds rows
// 128 r .. 128 r + 127 of A's slice and columns 128 r .. 128 r + 127 of B's,
// in the same 64 KiB stage layout as above; every operand byte is read from
// shared memory once for both tensor cores, which halves the operand reads
// per flop. The split warps of each block arrive on their own block's split
// barrier; in the odd block one thread of warp 1 waits for that barrier and
// forwards a single cluster-scope release arrival to the even block's peer
// barrier (one cluster-scope fence per stage instead of one per split warp).
// The even block's thread 32 waits for both, issues the MMAs and commits
// each stage's release and the final accumulator to both blocks. Each block
// stores its own 128 x 256 rows from its tensor memory.
constexpr int PM = 256, PN = 256;
constexpr int P_TMEM_COLS = 256;

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile(
      "mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(
          cluster_addr)
      : "memory");
}

__global__ void __launch_bounds__(X_THREADS, 1)
k_tf32x3_pair(const __grid_constant__ CUtensorMap tmA,
              const __grid_constant__ CUtensorMap tmB, float* __restrict__ C,
              int M, int N, int K, long long ldc, int tiles_m, int tiles_n,
              int vec_store, int* status) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t* ctrl = smem + XSTAGES * X_STAGE;
  const uint32_t full0 = smem_u32(ctrl);          // own TMA landed
  const uint32_t conv0 = full0 + 8 * XSTAGES;     // own split done
  const uint32_t empty0 = conv0 + 8 * XSTAGES;    // pair MMAs done reading
  const uint32_t peer0 = empty0 + 8 * XSTAGES;    // odd block split (even)
  const uint32_t accf = peer0 + 8 * XSTAGES;      // accumulator complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 8 * (4 * XSTAGES + 1));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  auto A_of = [&](int s) { return smem + s * X_STAGE; };
  auto Alo_of = [&](int s) { return smem + s * X_STAGE + X_A_BYTES; };
  auto B_of = [&](int s) { return smem + s * X_STAGE + 2 * X_A_BYTES; };
  auto Blo_of = [&](int s) {
    return smem + s * X_STAGE + 2 * X_A_BYTES + X_B_BYTES;
  };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  int pm, pn;
  tile_of(blockIdx.x >> 1, tiles_m, tiles_n, pm, pn);
  const int m_own = pm * PM + 128 * int(rank);  // this block's rows
  const int n_pair = pn * PN;                   // the pair's columns
  const int n_own = n_pair + 128 * int(rank);   // this block's B columns
  const int T = (K + XK - 1) / XK;

  if (tid == 0) {
    for (int s = 0; s < XSTAGES; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(conv0 + 8 * s, X_CONV_THREADS / 32);
      mbar_init(empty0 + 8 * s, 1);
      mbar_init(peer0 + 8 * s, 1);
    }
    mbar_init(accf, 1);
    *abort_flag = 0;
    mbar_fence_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tc::tmem_alloc_pair(smem_u32(tmem_slot), P_TMEM_COLS);
    tc::tmem_relinquish_pair();
  }
  tc::fence_before_sync();
  __syncthreads();
  cluster_sync_all();  // both blocks' barriers exist before any remote use
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      for (int t = 0; t < T && !*abort_flag; ++t) {
        const int s = t % XSTAGES;
        if (t >= XSTAGES &&
            !mbar_wait_bounded(empty0 + 8 * s, ((t / XSTAGES) - 1) & 1, status,
                               kSiteTf32Empty, kWaitLimitNs)) {
          *abort_flag = 1;
          break;
        }
        const uint32_t bar = full0 + 8 * s;
        mbar_arrive_expect_tx(bar, X_A_BYTES + X_B_BYTES);
        tma_load_2d(smem_u32(A_of(s)), &tmA, t * XK, m_own, bar);
        for (int j = 0; j < 128 / 32; ++j)
          tma_load_2d(smem_u32(B_of(s) + j * X_B_BOX), &tmB, n_own + 32 * j,
                      t * XK, bar);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issue
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = tc::idesc_tf32(PM, PN, false, false);
      for (int t = 0; t < T; ++t) {
        const int s = t % XSTAGES;
        const uint32_t par = (t / XSTAGES) & 1;
        if (*abort_flag ||
            !mbar_wait_bounded(conv0 + 8 * s, par, status, kSiteTf32Conv,
                               kWaitLimitNs) ||
            !mbar_wait_bounded<true>(peer0 + 8 * s, par, status,
                                     kSiteTf32Peer, kWaitLimitNs)) {
          *abort_flag = 1;
          break;
        }
        tc::fence_after_sync();
        const uint32_t a = smem_u32(A_of(s)), al = smem_u32(Alo_of(s));
        const uint32_t b = smem_u32(B_of(s)), bl = smem_u32(Blo_of(s));
#pragma unroll
        for (int ks = 0; ks < XK / 8; ++ks) {
          const uint64_t da = tc::smem_desc(a + 32 * ks, 16, 1024,
                                            tc::kLayoutSwizzle128);
          const uint64_t dal = tc::smem_desc(al + 32 * ks, 16, 1024,
                                             tc::kLayoutSwizzle128);
          const uint64_t db = tc::smem_desc(b + 32 * ks, 16, 1024,
                                            tc::kLayoutSwizzle128);
          const uint64_t dbl = tc::smem_desc(bl + 32 * ks, 16, 1024,
                                             tc::kLayoutSwizzle128);
          tc::mma_tf32_pair(tmem, dal, db, idesc, (t > 0 || ks > 0) ? 1u : 0u);
          tc::mma_tf32_pair(tmem, da, dbl, idesc, 1u);
          tc::mma_tf32_pair(tmem, da, db, idesc, 1u);
        }
        tc::commit_pair_multicast(empty0 + 8 * s, 0x3);
      }
      tc::commit_pair_multicast(accf, 0x3);
    } else if (lane == 0) {
      // odd block: forward each completed split to the even block. The
      // acquire of the local wait and the cumulative cluster-scope release
      // order all four split warps' writes before the even block's MMAs.
      const uint32_t peer_leader = cluster_map(peer0, 0);
      for (int t = 0; t < T; ++t) {
        const int s = t % XSTAGES;
        if (*abort_flag ||
            !mbar_wait_bounded(conv0 + 8 * s, (t / XSTAGES) & 1, status,
                               kSiteTf32Conv, kWaitLimitNs)) {
          *abort_flag = 1;
          break;
        }
        mbar_arrive_cluster(peer_leader + 8 * s);
      }
    }
  } else {
    // ---------------------------------------------------------- split
    const int ct = tid - 64;  // 0..127
    for (int t = 0; t < T; ++t) {
      const int s = t % XSTAGES;
      if (*abort_flag ||
          !mbar_wait_bounded(full0 + 8 * s, (t / XSTAGES) & 1, status,
                             kSiteTf32Full, kWaitLimitNs)) {
        *abort_flag = 1;
        break;
      }
#pragma unroll
      for (int q = 0; q < X_A_BYTES / 16 / X_CONV_THREADS; ++q)
        split4(A_of(s), Alo_of(s), ct + X_CONV_THREADS * q);
      split_transpose_box(B_of(s) + (warp - 2) * X_B_BOX,
                          Blo_of(s) + (warp - 2) * X_B_BOX, lane);
      fence_async_shared();  // generic writes -> visible to the MMA
      __syncwarp();
      if (lane == 0) mbar_arrive(conv0 + 8 * s);
    }
    // ---------------------------------------------------------- epilogue
    const bool ok = mbar_wait_bounded(accf, 0, status, kSiteTf32Acc,
                                      *abort_flag ? kWaitLimitNs / 100
                                                  : kWaitLimitNs);
    tc::fence_after_sync();
    const int quarter = warp & 3;
    const int r = m_own + 32 * quarter + lane;
    float* crow = C + (long long)r * ldc;
#pragma unroll 1
    for (int cb = 0; cb < PN / 32; ++cb) {
      uint32_t v[32];
      tc::tmem_ld_32x32b_x32(tmem + (uint32_t(32 * quarter) << 16) + 32 * cb,
                             v);
      tc::tmem_ld_wait();
      if (!ok || *abort_flag || r >= M) continue;
      const int c0 = n_pair + 32 * cb;
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const int c = c0 + e;
        if (vec_store && c + 3 < N) {
          *reinterpret_cast<float4*>(crow + c) =
              make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]),
                          __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3]));
        } else {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (c + u < N) crow[c + u] = __uint_as_float(v[e + u]);
        }
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  cluster_sync_all();  // the pair's MMAs and both blocks' reads are done
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc_pair(tmem, P_TMEM_COLS);
  }
}

}  // namespace

cudaError_t tf32x3_init() {
  const cudaError_t e = cudaFuncSetAttribute(
      k_tf32x3, cudaFuncAttributeMaxDynamicSharedMemorySize, int(X_SMEM));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k_tf32x3_pair,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              int(X_SMEM));
}

cudaError_t launch_tf32x3_pair(const GemmArgs& g, const CUtensorMap& tmA,
                               const CUtensorMap& tmB, int* status,
                               cudaStream_t s) {
  const int tiles_m = int((g.M + PM - 1) / PM);
  const int tiles_n = int((g.N + PN - 1) / PN);
  const bool vec = (g.ldc % 4 == 0) &&
                   (reinterpret_cast<uintptr_t>(g.C) % 16 == 0);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2u * unsigned(tiles_m) * unsigned(tiles_n), 1, 1);
  cfg.blockDim = dim3(X_THREADS, 1, 1);
  cfg.dynamicSmemBytes = X_SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_tf32x3_pair, tmA, tmB, g.C, int(g.M),
                            int(g.N), int(g.K), (long long)g.ldc, tiles_m,
                            tiles_n, vec ? 1 : 0, status);
}

cudaError_t launch_tf32x3(const GemmArgs& g, const CUtensorMap& tmA,
                          const CUtensorMap& tmB, int* status,
                          cudaStream_t s) {
  const int tiles_m = int((g.M + XM - 1) / XM);
  const int tiles_n = int((g.N + XN - 1) / XN);
  const bool vec = (g.ldc % 4 == 0) &&
                   (reinterpret_cast<uintptr_t>(g.C) % 16 == 0);
  k_tf32x3<<<unsigned(tiles_m) * unsigned(tiles_n), X_THREADS, X_SMEM, s>>>(
      tmA, tmB, g.C, int(g.M), int(g.N), int(g.K), (long long)g.ldc, tiles_m,
      tiles_n, vec ? 1 : 0, status);
  return cudaGetLastError();
}

}  // namespace dfm
