// FP32 matrix product on the tcgen05 tensor cores by three TF32 products
// (3xTF32; the published error-compensated split of Ootomo and Yokota, 2022).
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
//               memory and store C (or, with split k, the block's piece);
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
// Products with few tiles split k over the idle SMs (k_splitk_reduce adds
// the pieces in order).
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

// As split4, but leaves x in place as the high part: the MMA reads an fp32
// operand as TF32 by ignoring its 13 low mantissa bits, which is the same
// hi as above (Inf and NaN included), so only lo is written.
__device__ __forceinline__ void split4_lo(const uint8_t* x_buf, uint8_t* lo_buf,
                                          int idx) {
  const float4 x = reinterpret_cast<const float4*>(x_buf)[idx];
  float4 h, l;
  split_tf32(x.x, h.x, l.x);
  split_tf32(x.y, h.y, l.y);
  split_tf32(x.z, h.z, l.z);
  split_tf32(x.w, h.w, l.w);
  reinterpret_cast<float4*>(lo_buf)[idx] = l;
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

// Named barrier over `threads` threads (a multiple of 32) with id 1..15.
__device__ __forceinline__ void named_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// All of `threads` threads at named barrier `id` learn whether every one of
// them passed pred != 0.
__device__ __forceinline__ bool named_all(int id, int threads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "r"(id), "r"(threads)
      : "memory");
  return r != 0;
}

// Half of split_transpose_box for two warps sharing a box: this warp reads
// k rows 16 half .. 16 half + 15 (column n = 32 j + lane), waits until the
// other warp has read its half too (the box is rewritten in place), then
// writes the matching 16-k half of K-major row n (hi in place, and B_lo).
__device__ __forceinline__ void split_transpose_half(uint8_t* box,
                                                    uint8_t* lo_box, int lane,
                                                    int half, int bar_id) {
  float x[16];
  const int cb = (lane * 4) / 16, cw = (lane * 4) % 16;
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const int kk = 16 * half + k;
    x[k] = *reinterpret_cast<const float*>(box + kk * 128 +
                                           ((cb ^ (kk & 7)) << 4) + cw);
  }
  named_sync(bar_id, 64);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    float4 h, l;
    split_tf32(x[4 * c + 0], h.x, l.x);
    split_tf32(x[4 * c + 1], h.y, l.y);
    split_tf32(x[4 * c + 2], h.z, l.z);
    split_tf32(x[4 * c + 3], h.w, l.w);
    const int off = lane * 128 + (((4 * half + c) ^ (lane & 7)) << 4);
    *reinterpret_cast<float4*>(box + off) = h;
    *reinterpret_cast<float4*>(lo_box + off) = l;
  }
}

// ------------------------------------------------- operand layouts (op)
//
// Both MMA operands are presented K-major: on this part a kind::tf32 MMA
// with either MN-major descriptor bit set returned zeros. Per operand the
// stored layout decides the work:
//   A, op_a == 0 (stored M x K) and B, op_b == 1 (stored N x K): K-major
//     already; one TMA box {32 k, 128 rows} lands in the canonical
//     128-byte-swizzled layout and only the low part is split off.
//   A, op_a == 1 (stored K x M) and B, op_b == 0 (stored K x N): MN-major;
//     four boxes {32 rows, 32 k} land N-major and are transposed in place
//     into K-major rows (split_transpose_box / _half).
// (128-row halves: the 1-SM kernel's tile and each block's half of a pair.)
// The maps are 3-D: {inner, outer, batch item}; za / zb pick the item of
// A / B (0 for an operand shared by all items).
template <int OA, int OB>
__device__ __forceinline__ void load_stage(uint8_t* a_buf, uint8_t* b_buf,
                                           const CUtensorMap* tmA,
                                           const CUtensorMap* tmB, int k,
                                           int m0, int n0, int za, int zb,
                                           uint32_t bar) {
  if (OA == 0) {
    tma_load_3d(smem_u32(a_buf), tmA, k * XK, m0, za, bar);
  } else {
    for (int j = 0; j < 4; ++j)
      tma_load_3d(smem_u32(a_buf + j * X_B_BOX), tmA, m0 + 32 * j, k * XK, za,
                  bar);
  }
  if (OB == 0) {
    for (int j = 0; j < 4; ++j)
      tma_load_3d(smem_u32(b_buf + j * X_B_BOX), tmB, n0 + 32 * j, k * XK, zb,
                  bar);
  } else {
    tma_load_3d(smem_u32(b_buf), tmB, k * XK, n0, zb, bar);
  }
}

template <int OA, int OB>
__device__ __forceinline__ void prefetch_stage(const CUtensorMap* tmA,
                                               const CUtensorMap* tmB, int k,
                                               int m0, int n0, int za,
                                               int zb) {
  if (OA == 0) {
    tma_prefetch_l2_3d(tmA, k * XK, m0, za);
  } else {
    for (int j = 0; j < 4; ++j)
      tma_prefetch_l2_3d(tmA, m0 + 32 * j, k * XK, za);
  }
  if (OB == 0) {
    for (int j = 0; j < 4; ++j)
      tma_prefetch_l2_3d(tmB, n0 + 32 * j, k * XK, zb);
  } else {
    tma_prefetch_l2_3d(tmB, k * XK, n0, zb);
  }
}

// Batch description shared by the tensor-core kernels: tiles are numbered
// item by item (tiles_m x tiles_n per item, grouped raster order inside an
// item); C of item b starts at C + b * stride_c.
struct Batch {
  int items;            // >= 1
  int a_batched;        // 0: every item reads item 0 of A (shared A)
  int b_batched;
  long long stride_c;   // floats
};

// 1-SM kernel: 4 split warps (w = 0..3, ct = 0..127). K-major operands are
// split elementwise by all of them (hi masked in place, lo beside), an
// MN-major operand box by box, one box per warp.
template <int OA, int OB>
__device__ __forceinline__ void split_stage_1sm(uint8_t* A, uint8_t* Alo,
                                                uint8_t* B, uint8_t* Blo,
                                                int w, int lane, int ct) {
  if (OA == 0) {
#pragma unroll
    for (int q = 0; q < X_A_BYTES / 16 / X_CONV_THREADS; ++q)
      split4(A, Alo, ct + X_CONV_THREADS * q);
  } else {
    split_transpose_box(A + w * X_B_BOX, Alo + w * X_B_BOX, lane);
  }
  if (OB == 0) {
    split_transpose_box(B + w * X_B_BOX, Blo + w * X_B_BOX, lane);
  } else {
#pragma unroll
    for (int q = 0; q < X_B_BYTES / 16 / X_CONV_THREADS; ++q)
      split4(B, Blo, ct + X_CONV_THREADS * q);
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

// Split-k (splits > 1, blockIdx.y = split): the block multiplies k-slices
// [split T / splits, (split + 1) T / splits) of its tile and writes the raw
// accumulator to `part`, block-major (tile x splits, 4096 float4 each,
// warp-major inside: float4 ((q * 4 + cb) * 8 + e) * 32 + lane holds row
// 32 q + lane, columns 32 cb + 4 e .. + 3); k_splitk_reduce adds the splits
// in order and applies the epilogue.
template <int OA, int OB>
__global__ void __launch_bounds__(X_THREADS, 1)
k_tf32x3(const __grid_constant__ CUtensorMap tmA,
         const __grid_constant__ CUtensorMap tmB, float* __restrict__ C, int M,
         int N, int K, long long ldc, int tiles_m, int tiles_n, int vec_store,
         Scale sc, Batch bt, int splits, float4* __restrict__ part,
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
  const int tpb = tiles_m * tiles_n;
  const int item = int(blockIdx.x) / tpb;
  tile_of(int(blockIdx.x) - item * tpb, tiles_m, tiles_n, pm, pn);
  const int m0 = pm * XM, n0 = pn * XN;
  const int za = bt.a_batched ? item : 0, zb = bt.b_batched ? item : 0;
  C += item * bt.stride_c;
  const int T = (K + XK - 1) / XK;
  const int split = int(blockIdx.y);
  const int t0 = split * T / splits, nT = (split + 1) * T / splits - t0;

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
      for (int t = 0; t < nT && !*abort_flag; ++t) {
        const int s = t % XSTAGES;
        if (t >= XSTAGES &&
            !mbar_wait_bounded(empty0 + 8 * s, ((t / XSTAGES) - 1) & 1, status,
                               kSiteTf32Empty, kWaitLimitNs)) {
          *abort_flag = 1;
          break;
        }
        const uint32_t bar = full0 + 8 * s;
        mbar_arrive_expect_tx(bar, X_A_BYTES + X_B_BYTES);
        load_stage<OA, OB>(A_of(s), B_of(s), &tmA, &tmB, t0 + t, m0, n0, za,
                           zb, bar);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc = tc::idesc_tf32(XM, XN, false, false);
      for (int t = 0; t < nT; ++t) {
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
    for (int t = 0; t < nT; ++t) {
      const int s = t % XSTAGES;
      if (*abort_flag ||
          !mbar_wait_bounded(full0 + 8 * s, (t / XSTAGES) & 1, status,
                             kSiteTf32Full, kWaitLimitNs)) {
        *abort_flag = 1;
        break;
      }
      split_stage_1sm<OA, OB>(A_of(s), Alo_of(s), B_of(s), Blo_of(s), warp - 2,
                              lane, ct);
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
    float4* piece = part + ((long long)blockIdx.x * splits + split) *
                               (XM * XN / 4) +
                    quarter * 4 * 8 * 32 + lane;
#pragma unroll 1
    for (int cb = 0; cb < XN / 32; ++cb) {
      uint32_t v[32];
      tc::tmem_ld_32x32b_x32(tmem + (uint32_t(32 * quarter) << 16) + 32 * cb,
                             v);
      tc::tmem_ld_wait();
      if (!ok || *abort_flag) continue;
      if (splits > 1) {  // (an empty k range contributes zeros)
#pragma unroll
        for (int e = 0; e < 8; ++e)
          __stcg(piece + (cb * 8 + e) * 32,
                 nT == 0 ? make_float4(0.f, 0.f, 0.f, 0.f)
                         : make_float4(__uint_as_float(v[4 * e]),
                                       __uint_as_float(v[4 * e + 1]),
                                       __uint_as_float(v[4 * e + 2]),
                                       __uint_as_float(v[4 * e + 3])));
        continue;
      }
      if (r >= M) continue;
      const int c0 = n0 + 32 * cb;
#pragma unroll
      for (int e = 0; e < 32; e += 4) {
        const int c = c0 + e;
        if (vec_store && c + 3 < N) {
          *reinterpret_cast<float4*>(crow + c) = epi4(
              make_float4(__uint_as_float(v[e]), __uint_as_float(v[e + 1]),
                          __uint_as_float(v[e + 2]), __uint_as_float(v[e + 3])),
              crow + c, sc);
        } else {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            if (c + u < N)
              crow[c + u] = epi1(__uint_as_float(v[e + u]), crow + c + u, sc);
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

// Adds the split-k pieces of k_tf32x3 in split order and stores C: one
// thread per float4 of a tile (grid: tiles x 16 blocks of 256), loads
// coalesced over the warp-major pieces.
__global__ void __launch_bounds__(256)
k_splitk_reduce(const float4* __restrict__ part, int splits,
                float* __restrict__ C, int M, int N, long long ldc,
                int tiles_m, int tiles_n, int vec_store, Scale sc,
                long long stride_c) {
  const int idx = int(blockIdx.y) * 256 + int(threadIdx.x);  // 0..4095
  const int lane = idx & 31, e = (idx >> 5) & 7, cb = (idx >> 8) & 3,
            q = idx >> 10;
  const int tpb = tiles_m * tiles_n;
  const int item = int(blockIdx.x) / tpb;
  int pm, pn;
  tile_of(int(blockIdx.x) - item * tpb, tiles_m, tiles_n, pm, pn);
  const int r = pm * XM + 32 * q + lane;
  const int c = pn * XN + 32 * cb + 4 * e;
  if (r >= M || c >= N) return;
  const float4* src = part + (long long)blockIdx.x * splits * (XM * XN / 4) + idx;
  float4 acc = __ldcg(src);
  for (int sp = 1; sp < splits; ++sp) {
    const float4 x = __ldcg(src + (long long)sp * (XM * XN / 4));
    acc.x += x.x;
    acc.y += x.y;
    acc.z += x.z;
    acc.w += x.w;
  }
  float* crow = C + item * stride_c + (long long)r * ldc;
  if (vec_store && c + 3 < N) {
    *reinterpret_cast<float4*>(crow + c) = epi4(acc, crow + c, sc);
  } else {
    const float v[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (c + u < N) crow[c + u] = epi1(v[u], crow + c + u, sc);
  }
}

// ---------------------------------------------------------------- pairs
//
// 2-SM variant: a cluster of two blocks computes 256 x 256 tiles with the
// pair MMA (M = 256, N = 256, K = 8). Block r of the pair holds rows
// 128 r .. 128 r + 127 of A's slice and columns 128 r .. 128 r + 127 of B's,
// in the same 64 KiB stage layout as above; every operand byte is read from
// shared memory once for both tensor cores, which halves the operand reads
// per flop.
//
// Persistent, with a stream-K tail: the grid is the G clusters that fit on
// the GPU at once. Whole tiles are dealt round-robin in full waves (tile
// c + i G to cluster c); the k-slices of the remaining tiles (fewer than one
// wave, or one wave more when that share would be short) are split evenly
// over all G clusters, so no partly filled last wave is left. A cluster's
// share is a run of k-ranges ("units"), taken before its whole tiles; a unit
// that covers its whole tile stores C directly, a partial one writes its
// fp32 piece to the workspace and the last of the tile's pieces to arrive
// adds them all in k order and stores C (no cluster waits on another; the
// sum order is fixed).
//
// Roles in each block (448 threads):
//   warp 0      TMA producer over the cluster's units, one ring of stages;
//   warp 1      even block: allocates 512 tensor-memory columns for both
//               blocks (row-major A: one 256-column accumulator, four
//               32-column A_lo stages and 128 columns for a parked half
//               accumulator; transposed A: two accumulators) and issues the
//               MMAs; odd block: forwards each completed split to the even
//               block with one arrival per stage;
//   warps 2..9  split and transpose each landed stage and arrive on their
//               own block's split barrier; two warps share each B box, one
//               per 16-k half (the split sits on the path from a freed
//               stage to its next MMAs);
//   warps 10..13 epilogue, one tensor-memory lane quarter each: read a
//               finished accumulator, store C or the piece, hand the
//               accumulator back. With two accumulators the MMAs of the
//               next unit run while the previous one is stored; with one,
//               its upper half is parked in tensor memory first and stored
//               after the hand-back. They also sum the split tiles' pieces
//               (under the next whole tile's MMAs when one follows).
constexpr int PM = 256, PN = 256;
constexpr int P_THREADS = 448;
constexpr int P_PREFETCH = 3;                        // k-slices ahead into L2
constexpr int P_CONV_WARPS = 8;
constexpr int P_ACC_COLS = 256;                      // one accumulator
constexpr int P_TMEM_COLS = 2 * P_ACC_COLS;           // all of it
constexpr int P_ALO_COL = P_ACC_COLS;                 // A_lo stages (K-major A)
constexpr int P_PARK_COL = P_ALO_COL + 128;           // parked half accumulator
static_assert(P_ALO_COL + XSTAGES * XK <= P_TMEM_COLS, "A_lo stages fit");
constexpr int P_EPI_WARP0 = 2 + P_CONV_WARPS;
constexpr int P_EPI_ARRIVALS = 2 * 4;                // 4 warps x 2 blocks
constexpr int P_PIECE_FLOATS = 128 * PN;             // one block's half tile
// Epilogue staging for the bulk tensor stores of C: per epilogue warp two
// 4 KiB boxes of 32 rows x 32 columns (128-byte rows, 128-byte swizzle).
constexpr int P_STG_BOX = 32 * 32 * 4;
constexpr int P_STG_BYTES = 4 * 2 * P_STG_BOX;       // 32 KiB
// Stream-K fix-ups reuse the stage ring: per epilogue warp 48 KiB, 11
// slots of 4 KiB and their mbarriers.
constexpr int kFixSlots = 11;
constexpr int kFixRegion = 48 * 1024;
static_assert(kFixSlots * P_STG_BOX + 8 * kFixSlots <= kFixRegion, "slots");
static_assert(4 * kFixRegion <= XSTAGES * X_STAGE, "fix-up regions");
constexpr size_t P_SMEM =
    size_t(XSTAGES) * X_STAGE + P_STG_BYTES + 1024 + 256;
static_assert(P_SMEM <= 232448, "shared memory per block");

struct PairParams {
  float* C;
  int M, N, K;
  long long ldc;
  int tiles_m, tiles_n;
  int T;                // k-slices per tile
  int G;                // clusters
  int dp_tiles;         // tiles dealt whole, a multiple of G (or all tiles)
  int sk_tiles;         // tiles after them, split by k-slices
  long long sk_iters;   // sk_tiles * T
  float* ws;            // 2 pieces per block: G x 2 x 2 x P_PIECE_FLOATS
  int* counters;        // sk_tiles x 2 blocks x 4 quarters, zero between calls
  int vec_store;
  int tma_c;            // C written by bulk tensor stores (beta == 0)
  Scale sc;
  Batch bt;
  int* status;
};

// Tile t of the pair schedule -> batch item and 256 x 256 tile in it.
__device__ __forceinline__ void pair_tile(int t, const PairParams& p, int& item,
                                          int& pm, int& pn) {
  const int tpb = p.tiles_m * p.tiles_n;
  item = t / tpb;
  tile_of(t - item * tpb, p.tiles_m, p.tiles_n, pm, pn);
}

// Pair kernel, K-major A: A_lo goes to tensor memory instead of shared
// memory (the MMA takes its A operand from there), which saves the split's
// A_lo stores and the tensor core's A_lo reads in shared memory. Warp
// 2 + cw may only reach tensor-memory lanes 32 q .. 32 q + 31 with
// q = (2 + cw) & 3: it takes those rows of the block's 128 and the k half
// cw >> 2. Each lane splits its row's 16 values from the 128-byte-swizzled
// stage and stores the low parts to columns col + 16 (cw >> 2) .. + 15.
__device__ __forceinline__ void a_lo_to_tmem(const uint8_t* A, uint32_t col,
                                             int cw, int lane) {
  const int q = (2 + cw) & 3, h = cw >> 2;
  const int r = 32 * q + lane;
  uint32_t lo[16];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int chunk = 4 * h + c;
    const float4 x = *reinterpret_cast<const float4*>(
        A + r * 128 + ((chunk ^ (r & 7)) << 4));
    float hi, l;
    split_tf32(x.x, hi, l);
    lo[4 * c + 0] = __float_as_uint(l);
    split_tf32(x.y, hi, l);
    lo[4 * c + 1] = __float_as_uint(l);
    split_tf32(x.z, hi, l);
    lo[4 * c + 2] = __float_as_uint(l);
    split_tf32(x.w, hi, l);
    lo[4 * c + 3] = __float_as_uint(l);
  }
  tc::tmem_st_32x32b_x16(col + (uint32_t(32 * q) << 16) + 16 * h, lo);
}

// Pair kernel: 8 split warps (cw = 0..7, ct = 0..255). K-major operands:
// the landed tile is the high part, all threads write the low part. One
// MN-major operand: two warps per box, one per 16-k half. Both MN-major:
// one box per warp.
// Copies accumulator columns 128 .. 255 of this warp's lanes to the
// tensor-memory columns park .. park + 127 (not used by the MMAs), so that
// the accumulator can be handed back after only its lower half has gone out
// through the staging boxes; the parked half is stored under the next
// tile's MMAs. Tensor-memory loads take tens of cycles, a bulk store's
// staging box about a thousand.
__device__ __forceinline__ void park_upper_half(uint32_t acc, uint32_t park) {
#pragma unroll 1
  for (int cb = 4; cb < 8; ++cb) {
    uint32_t v[32];
    tc::tmem_ld_32x32b_x32(acc + 32 * cb, v);
    tc::tmem_ld_wait();
    uint32_t lo[16], hi[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      lo[i] = v[i];
      hi[i] = v[16 + i];
    }
    tc::tmem_st_32x32b_x16(park + 32 * (cb - 4), lo);
    tc::tmem_st_32x32b_x16(park + 32 * (cb - 4) + 16, hi);
  }
  tc::tmem_st_wait();
}

template <int OA, int OB>
__device__ __forceinline__ void split_stage_pair(uint8_t* A, uint8_t* Alo,
                                                 uint8_t* B, uint8_t* Blo,
                                                 int cw, int lane, int ct,
                                                 uint32_t alo_col) {
  constexpr int kThreads = 256;
  const int box = cw >> 1, half = cw & 1, bar_id = 1 + box;
  if (OA == 0) a_lo_to_tmem(A, alo_col, cw, lane);
  if (OB == 1) {
#pragma unroll
    for (int q = 0; q < X_B_BYTES / 16 / kThreads; ++q)
      split4_lo(B, Blo, ct + kThreads * q);
  }
  if (OA == 1 && OB == 0) {
    uint8_t* x = cw < 4 ? A : B;
    uint8_t* lo = cw < 4 ? Alo : Blo;
    split_transpose_box(x + (cw & 3) * X_B_BOX, lo + (cw & 3) * X_B_BOX, lane);
  } else if (OA == 1) {
    split_transpose_half(A + box * X_B_BOX, Alo + box * X_B_BOX, lane, half,
                         bar_id);
  } else if (OB == 0) {
    split_transpose_half(B + box * X_B_BOX, Blo + box * X_B_BOX, lane, half,
                         bar_id);
  }
}

__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile(
      "mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(
          cluster_addr)
      : "memory");
}

// Arrive on a barrier of the other block with the default (CTA-scope)
// release. Used for the split hand-over only: the split results and the
// tensor core that reads them are on the same SM (this block's shared
// memory), the writers made their stores visible to the async proxy
// (fence.proxy.async) before arriving on this block's barrier, and the
// CTA-scope release performs them in shared memory before the arrival
// leaves the SM; the arrival only gates when the even block issues the MMA.
// (The cluster-scope release costs about a thousand cycles per stage here,
// on the refill path of every stage.) This is the cluster-barrier arrive of
// the CUDA template library's 2-SM pipelines.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.shared::cluster.b64 _, [%0];" ::"r"(
                   cluster_addr)
               : "memory");
}

__device__ __forceinline__ long long sk_begin(int c, const PairParams& p) {
  return (long long)c * p.sk_iters / p.G;
}

// The cluster whose stream-K share holds iteration x: the largest c with
// sk_begin(c) <= x.
__device__ __forceinline__ int sk_owner(long long x, const PairParams& p) {
  return int(((x + 1) * p.G + p.sk_iters - 1) / p.sk_iters) - 1;
}

struct Unit {
  int tile;    // output tile (grouped raster order)
  int kb, ke;  // k-slices [kb, ke)
  int sk;      // stream-K tile index when the unit is a partial piece, else -1
};

// Unit u of cluster c; false past the cluster's last unit. A cluster first
// works through its stream-K share (at most two partial segments), then its
// whole tiles: the fix-ups of the split tiles then run while the clusters
// multiply their whole tiles, instead of after them at the end of the launch.
__device__ __forceinline__ bool unit_of(int c, int u, const PairParams& p,
                                        Unit& w) {
  const int dp_units = c < p.dp_tiles ? (p.dp_tiles - c + p.G - 1) / p.G : 0;
  int sk_units = 0;
  long long b = 0, e = 0;
  if (p.sk_tiles > 0) {
    b = sk_begin(c, p);
    e = sk_begin(c + 1, p);
    if (b < e) sk_units = int((e - 1) / p.T - b / p.T + 1);
  }
  if (u < sk_units) {
    const long long x = u == 0 ? b : (b / p.T + u) * p.T;
    const int tau = int(x / p.T);
    const long long x0 = (long long)tau * p.T;
    w.tile = p.dp_tiles + tau;
    w.kb = int(x - x0);
    w.ke = int(e - x0 < p.T ? e - x0 : p.T);
    w.sk = (w.kb == 0 && w.ke == p.T) ? -1 : tau;
    return true;
  }
  u -= sk_units;
  if (u >= dp_units) return false;
  w.tile = c + u * p.G;
  w.kb = 0;
  w.ke = p.T;
  w.sk = -1;
  return true;
}

// Stores one lane-quarter's 32 rows x 256 columns of C from accumulator
// columns `acc` (rows m0 + lane, columns n0 ..).
// Direct stores of C (beta != 0, C not 16-byte aligned, stream-K fix-up)
// also go through the warp's staging box, so that they are coalesced rows:
// each lane stages its row (32 values, 128-byte swizzle), then the warp
// writes the box back row by row with lane j on column j (one 128-byte
// row per instruction; the old C is read the same way when beta != 0).
// rows / cols: the box's part inside C.
__device__ __forceinline__ void write_box_rows(const uint8_t* box, float* c0,
                                               long long ldc, int rows,
                                               int cols, int lane,
                                               const Scale& sc) {
  if (lane >= cols) return;
  const int w = lane >> 2, b = (lane & 3) * 4;
  // 8 rows per round: their loads (box, and the old C when beta != 0) are
  // issued before their stores.
#pragma unroll 1
  for (int r0 = 0; r0 < rows; r0 += 8) {
    float x[8], y[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int rr = r0 + u;
      x[u] = 0.f;
      y[u] = 0.f;
      if (rr < rows) {
        x[u] = *reinterpret_cast<const float*>(
            box + rr * 128 + ((w ^ (rr & 7)) << 4) + b);
        if (sc.beta != 0.f) y[u] = c0[rr * ldc + lane];
      }
    }
#pragma unroll
    for (int u = 0; u < 8; ++u)
      if (r0 + u < rows)
        c0[(r0 + u) * ldc + lane] = sc.beta == 0.f
                                        ? sc.alpha * x[u]
                                        : fmaf(sc.alpha, x[u], sc.beta * y[u]);
  }
}

// One lane quarter's 32 rows x 256 columns of C from accumulator columns
// `acc`, written through the staging box; cq = C at the quarter's first row
// and the tile's first column.
__device__ __forceinline__ void store_c_staged(uint32_t acc, uint8_t* box,
                                               float* cq, long long ldc,
                                               int rows, int cols, int lane,
                                               const Scale& sc) {
  if (lane == 0) bulk_wait_group_read<0>();  // box free of bulk stores
#pragma unroll 1
  for (int cb = 0; cb < PN / 32; ++cb) {
    uint32_t v[32];
    tc::tmem_ld_32x32b_x32(acc + 32 * cb, v);
    tc::tmem_ld_wait();
    __syncwarp();  // the previous box's rows have been written out
#pragma unroll
    for (int c = 0; c < 8; ++c)
      *reinterpret_cast<float4*>(box + lane * 128 + ((c ^ (lane & 7)) << 4)) =
          make_float4(__uint_as_float(v[4 * c]), __uint_as_float(v[4 * c + 1]),
                      __uint_as_float(v[4 * c + 2]),
                      __uint_as_float(v[4 * c + 3]));
    __syncwarp();
    write_box_rows(box, cq + 32 * cb, ldc, rows,
                   cols - 32 * cb < 32 ? cols - 32 * cb : 32, lane, sc);
  }
}

// One lane quarter's 32 rows x 256 columns of C from accumulator columns
// `acc` through the warp's two staging boxes and bulk tensor stores (the
// store clips rows >= M and columns >= N). Each lane writes its row of a
// 32 x 32 box with the 128-byte swizzle (16-byte chunk c of row r at
// c ^ (r & 7): conflict-free), then lane 0 stores the box. A box is reused
// once the store issued from it two boxes earlier has read it.
// Column blocks cb0 .. cb1 - 1 of 32 (accumulator column acc + 32 cb).
__device__ __forceinline__ void store_c_tma(uint32_t acc, uint8_t* stg,
                                            const CUtensorMap* tmC, int lane,
                                            int x0, int y0, int z,
                                            float alpha, int cb0, int cb1) {
#pragma unroll 1
  for (int cb = cb0; cb < cb1; ++cb) {
    uint32_t v[32];
    tc::tmem_ld_32x32b_x32(acc + 32 * cb, v);
    tc::tmem_ld_wait();
    uint8_t* box = stg + (cb & 1) * P_STG_BOX;
    if (lane == 0) bulk_wait_group_read<1>();
    __syncwarp();
#pragma unroll
    for (int c = 0; c < 8; ++c)
      *reinterpret_cast<float4*>(box + lane * 128 + ((c ^ (lane & 7)) << 4)) =
          make_float4(alpha * __uint_as_float(v[4 * c]),
                      alpha * __uint_as_float(v[4 * c + 1]),
                      alpha * __uint_as_float(v[4 * c + 2]),
                      alpha * __uint_as_float(v[4 * c + 3]));
    fence_async_shared();  // generic writes -> visible to the bulk store
    __syncwarp();
    if (lane == 0) {
      tma_store_3d(tmC, smem_u32(box), x0 + 32 * cb, y0, z);
      bulk_commit_group();
    }
  }
}

// Piece j of stream-K tile `sk` for one block and lane quarter: the
// contributors are clusters c_first .. c_first + pieces - 1 in k order, and
// only the first one's share can start before the tile, so only its piece
// can sit in its second workspace slot.
__device__ __forceinline__ const float4* sk_piece(const float4* ws4, int sk,
                                                  int j, uint32_t rank,
                                                  int quarter,
                                                  const PairParams& p) {
  const long long x0 = (long long)sk * p.T;
  const int c_first = sk_owner(x0, p);
  const int s_first = sk_begin(c_first, p) >= x0 ? 0 : 1;
  return ws4 + ((long long)((c_first + j) * 2 + (j == 0 ? s_first : 0)) * 2 +
                rank) * (P_PIECE_FLOATS / 4) + quarter * 8 * 256;
}

// Stream-K fix-up of one lane quarter of a tile while the block still has a
// whole tile to multiply: the stage ring is busy, so the pieces are read
// straight from L2 (a piece's column block is 4 KiB, warp-major: element
// (e, lane) at e * 32 + lane, so each load is 512 coalesced bytes) and each
// lane writes its row's sums straight to C (its 32 columns of a block are
// 128 contiguous bytes). The pieces are added in k order, exactly as in the
// end-of-kernel fix-up, so the result does not depend on which of the two
// runs.
__device__ __forceinline__ void fixup_direct(const float4* ws4, int tile,
                                             uint32_t rank, int quarter,
                                             int lane, const PairParams& p) {
  int item, pm, pn;
  pair_tile(tile, p, item, pm, pn);
  const int sk = tile - p.dp_tiles;
  const long long x0 = (long long)sk * p.T;
  const int pieces = sk_owner(x0 + p.T - 1, p) - sk_owner(x0, p) + 1;
  const int n0 = pn * PN;
  const int r0q = pm * PM + 128 * int(rank) + 32 * quarter;
  if (r0q + lane >= p.M) return;
  float* crow = p.C + item * p.bt.stride_c + (long long)(r0q + lane) * p.ldc +
                n0;
  const int cols_in = p.N - n0 < PN ? p.N - n0 : PN;
#pragma unroll 1
  for (int cb = 0; cb < PN / 32; ++cb) {
    float4 acc[8];
#pragma unroll 1
    for (int j = 0; j < pieces; ++j) {
      const float4* src =
          sk_piece(ws4, sk, j, rank, quarter, p) + cb * 256 + lane;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const float4 x = __ldcg(src + e * 32);
        if (j == 0) {
          acc[e] = x;
        } else {
          acc[e].x += x.x;
          acc[e].y += x.y;
          acc[e].z += x.z;
          acc[e].w += x.w;
        }
      }
    }
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int col = 32 * cb + 4 * e;
      float* c = crow + col;
      if (p.vec_store && col + 3 < cols_in) {
        *reinterpret_cast<float4*>(c) = epi4(acc[e], c, p.sc);
      } else {
        const float v[4] = {acc[e].x, acc[e].y, acc[e].z, acc[e].w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (col + i < cols_in) c[i] = epi1(v[i], c + i, p.sc);
      }
    }
  }
}

// kEarlyFix: schedules with whole tiles after the stream-K shares sum a
// split tile's pieces as soon as they are in (under the next MMAs). It is
// a template switch so that schedules without whole tiles (all split, or
// none split) keep the code of the end-of-kernel fix-up alone.
template <int OA, int OB, bool kEarlyFix>
__global__ void __launch_bounds__(P_THREADS, 1)
k_tf32x3_pair(const __grid_constant__ CUtensorMap tmA,
              const __grid_constant__ CUtensorMap tmB,
              const __grid_constant__ CUtensorMap tmC, const PairParams p) {
  // K-major A: A_lo lives in tensor memory after the accumulator, so only
  // one accumulator fits (the epilogue of a tile holds up the next tile's
  // MMAs); otherwise two accumulators let them overlap.
  constexpr bool kLoTmem = OA == 0;
  constexpr int kAccs = kLoTmem ? 1 : 2;
  // Without A_lo in shared memory a stage is 48 KiB and four fit where
  // three of 64 KiB did: a deeper ring for the same bytes.
  constexpr int kStageBytes = kLoTmem ? X_STAGE - X_A_BYTES : X_STAGE;
  constexpr int kStages = kLoTmem ? 4 : 3;
  static_assert(kStages * kStageBytes <= XSTAGES * X_STAGE, "ring fits");
  static_assert(P_ALO_COL + kStages * XK <= P_TMEM_COLS, "A_lo fits");
  static_assert(!kLoTmem || (P_ALO_COL + kStages * XK <= P_PARK_COL &&
                             P_PARK_COL + 128 <= P_TMEM_COLS),
                "the parked half is clear of A_lo");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t* stg0 = smem + kStages * kStageBytes;  // epilogue staging
  uint8_t* ctrl = stg0 + P_STG_BYTES;
  const uint32_t full0 = smem_u32(ctrl);          // own TMA landed
  const uint32_t conv0 = full0 + 8 * kStages;     // own split done
  const uint32_t empty0 = conv0 + 8 * kStages;    // pair MMAs done reading
  const uint32_t peer0 = empty0 + 8 * kStages;    // odd block split (even)
  const uint32_t accf0 = peer0 + 8 * kStages;     // accumulator b complete
  const uint32_t acce0 = accf0 + 16;              // accumulator b read (even)
  const uint32_t drain = acce0 + 16;              // teardown (even)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ctrl + 8 * (4 * kStages + 5));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  // stage s: A | A_lo (transposed A only) | B | B_lo
  auto A_of = [&](int s) { return smem + s * kStageBytes; };
  auto Alo_of = [&](int s) { return smem + s * kStageBytes + X_A_BYTES; };
  auto B_of = [&](int s) { return A_of(s) + kStageBytes - 2 * X_B_BYTES; };
  auto Blo_of = [&](int s) { return A_of(s) + kStageBytes - X_B_BYTES; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = cluster_rank();
  const int cl = int(blockIdx.x >> 1);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(conv0 + 8 * s, P_CONV_WARPS);
      mbar_init(empty0 + 8 * s, 1);
      mbar_init(peer0 + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(accf0 + 8 * b, 1);
      mbar_init(acce0 + 8 * b, P_EPI_ARRIVALS);
    }
    mbar_init(drain, 1);
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
      int g = 0;  // stages issued
      Unit w;
      for (int u = 0; !*abort_flag && unit_of(cl, u, p, w); ++u) {
        int item, pm, pn;
        pair_tile(w.tile, p, item, pm, pn);
        const int m_own = pm * PM + 128 * int(rank);
        const int n_own = pn * PN + 128 * int(rank);
        const int za = p.bt.a_batched ? item : 0;
        const int zb = p.bt.b_batched ? item : 0;
        for (int k = w.kb; k < w.ke; ++k, ++g) {
          const int s = g % kStages;
          if (g >= kStages &&
              !mbar_wait_bounded(empty0 + 8 * s, ((g / kStages) - 1) & 1,
                                 p.status, kSiteTf32Empty, kWaitLimitNs)) {
            *abort_flag = 1;
            break;
          }
          const uint32_t bar = full0 + 8 * s;
          mbar_arrive_expect_tx(bar, X_A_BYTES + X_B_BYTES);
          load_stage<OA, OB>(A_of(s), B_of(s), &tmA, &tmB, k, m_own, n_own, za,
                             zb, bar);
          // warm L2 with the tiles of a later k-slice of this unit, so that
          // its load (issued when a stage frees up) is an L2 hit
          if (k + P_PREFETCH < w.ke)
            prefetch_stage<OA, OB>(&tmA, &tmB, k + P_PREFETCH, m_own, n_own,
                                   za, zb);
        }
      }
      // Let the last loads land before the block can exit (they complete
      // even when nobody consumes them).
      for (int d = g - kStages < 0 ? 0 : g - kStages; d < g; ++d)
        mbar_wait_bounded(full0 + 8 * (d % kStages), (d / kStages) & 1,
                          p.status, kSiteTf32Full, kWaitLimitNs / 100);
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // -------------------------------------------------------- MMA issue
      constexpr uint32_t idesc = tc::idesc_tf32(PM, PN, false, false);
      // completion of the pair's MMAs, signalled on the same barrier of
      // both blocks (two commits; the odd block's barrier by its cluster
      // address)
      auto commit_both = [](uint32_t bar) {
        tc::commit_pair(bar);
        tc::commit_pair(cluster_map(bar, 1));
      };
      int g = 0;
      Unit w;
      for (int u = 0; !*abort_flag && unit_of(cl, u, p, w); ++u) {
        const int b = u % kAccs, n = u / kAccs;
        if (n >= 1 &&
            !mbar_wait_bounded<true>(acce0 + 8 * b, (n - 1) & 1, p.status,
                                     kSiteTf32Acc, kWaitLimitNs)) {
          *abort_flag = 1;
          break;
        }
        tc::fence_after_sync();
        const uint32_t acc = tmem + uint32_t(b * P_ACC_COLS);
        for (int k = w.kb; k < w.ke; ++k, ++g) {
          const int s = g % kStages;
          const uint32_t par = (g / kStages) & 1;
          if (*abort_flag ||
              !mbar_wait_bounded(conv0 + 8 * s, par, p.status, kSiteTf32Conv,
                                 kWaitLimitNs) ||
              !mbar_wait_bounded<true>(peer0 + 8 * s, par, p.status,
                                       kSiteTf32Peer, kWaitLimitNs)) {
            *abort_flag = 1;
            break;
          }
          tc::fence_after_sync();
          const uint32_t a = smem_u32(A_of(s)), al = smem_u32(Alo_of(s));
          const uint32_t bb = smem_u32(B_of(s)), bl = smem_u32(Blo_of(s));
#pragma unroll
          for (int ks = 0; ks < XK / 8; ++ks) {
            const uint64_t da = tc::smem_desc(a + 32 * ks, 16, 1024,
                                              tc::kLayoutSwizzle128);
            const uint64_t dal = tc::smem_desc(al + 32 * ks, 16, 1024,
                                               tc::kLayoutSwizzle128);
            const uint64_t db = tc::smem_desc(bb + 32 * ks, 16, 1024,
                                              tc::kLayoutSwizzle128);
            const uint64_t dbl = tc::smem_desc(bl + 32 * ks, 16, 1024,
                                               tc::kLayoutSwizzle128);
            if (kLoTmem)
              tc::mma_tf32_pair_tmem_a(
                  acc, tmem + uint32_t(P_ALO_COL + XK * s + 8 * ks), db, idesc,
                  (k > w.kb || ks > 0) ? 1u : 0u);
            else
              tc::mma_tf32_pair(acc, dal, db, idesc,
                                (k > w.kb || ks > 0) ? 1u : 0u);
            tc::mma_tf32_pair(acc, da, dbl, idesc, 1u);
            tc::mma_tf32_pair(acc, da, db, idesc, 1u);
          }
          commit_both(empty0 + 8 * s);  // stage s may be refilled
        }
        if (*abort_flag) break;
        commit_both(accf0 + 8 * b);   // accumulator b complete
      }
      // Every MMA issued has finished before the blocks may exit.
      tc::commit_pair(drain);
      mbar_wait_bounded(drain, 0, p.status, kSiteTf32Acc, kWaitLimitNs);
    } else if (lane == 0) {
      // ----------------------------------------- odd block: forward splits
      // One arrival per stage once all split warps of this block are done
      // (see mbar_arrive_remote for the ordering).
      const uint32_t peer_leader = cluster_map(peer0, 0);
      int g = 0;
      Unit w;
      for (int u = 0; !*abort_flag && unit_of(cl, u, p, w); ++u) {
        for (int k = w.kb; k < w.ke; ++k, ++g) {
          const int s = g % kStages;
          if (*abort_flag ||
              !mbar_wait_bounded(conv0 + 8 * s, (g / kStages) & 1, p.status,
                                 kSiteTf32Conv, kWaitLimitNs)) {
            *abort_flag = 1;
            break;
          }
          tc::fence_after_sync();   // the split's tensor-memory stores ...
          tc::fence_before_sync();  // ... ordered before the hand-over
          mbar_arrive_remote(peer_leader + 8 * s);
        }
      }
    }
  } else if (warp < P_EPI_WARP0) {
    // ---------------------------------------------------------- split
    const int ct = tid - 64;  // 0..255
    // named barrier of warps 2c and 2c + 1 (they may share a B box)
    const int bar_id = 1 + ((warp - 2) >> 1);
    int g = 0;
    bool ok = true;
    Unit w;
    // The two warps of a box take every continue/abort decision together
    // (bar.red), so neither can leave the other waiting at a named barrier.
    for (int u = 0; ok && unit_of(cl, u, p, w); ++u) {
      for (int k = w.kb; k < w.ke; ++k, ++g) {
        const int s = g % kStages;
        ok = !*abort_flag &&
             mbar_wait_bounded(full0 + 8 * s, (g / kStages) & 1, p.status,
                               kSiteTf32Full, kWaitLimitNs);
        ok = named_all(bar_id, 64, ok);
        if (!ok) {
          *abort_flag = 1;
          break;
        }
        // the MMAs that read this stage's A_lo columns last time are done
        // (their commit freed the stage before it was reloaded)
        if (kLoTmem) tc::fence_after_sync();
        split_stage_pair<OA, OB>(A_of(s), Alo_of(s), B_of(s), Blo_of(s),
                                 warp - 2, lane, ct,
                                 tmem + uint32_t(P_ALO_COL + XK * s));
        if (kLoTmem) {
          tc::tmem_st_wait();      // A_lo in tensor memory ...
          tc::fence_before_sync();  // ... before the arrival
        }
        fence_async_shared();  // generic writes -> visible to the MMA
        __syncwarp();
        if (lane == 0) mbar_arrive(conv0 + 8 * s);
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int quarter = warp & 3;  // tensor-memory lanes of this warp
    const uint32_t acce_leader = cluster_map(acce0, 0);
    float4* ws4 = reinterpret_cast<float4*>(p.ws);
    // Stream-K tiles whose pieces this warp sums (a cluster's share of
    // split k-slices has at most two partial segments).
    constexpr int kMaxFix = 2;
    int fix_tile[kMaxFix];
    int nfix = 0;
    Unit w;
    for (int u = 0; !*abort_flag && unit_of(cl, u, p, w); ++u) {
      const int b = u % kAccs;
      if (!mbar_wait_bounded(accf0 + 8 * b, (u / kAccs) & 1, p.status,
                             kSiteTf32Acc, kWaitLimitNs)) {
        *abort_flag = 1;
        break;
      }
      tc::fence_after_sync();
      const uint32_t acc = tmem + uint32_t(b * P_ACC_COLS) +
                           (uint32_t(32 * quarter) << 16);
      int item, pm, pn;
      pair_tile(w.tile, p, item, pm, pn);
      const int n0 = pn * PN;
      const int r0q = pm * PM + 128 * int(rank) + 32 * quarter;
      float* cq = p.C + item * p.bt.stride_c + (long long)r0q * p.ldc + n0;
      const int rows_in = p.M - r0q < 32 ? p.M - r0q : 32;
      const int cols_in = p.N - n0 < PN ? p.N - n0 : PN;
      uint8_t* stg = stg0 + (warp - P_EPI_WARP0) * 2 * P_STG_BOX;
      int slot = 0;
      // one accumulator (A_lo holds the rest of tensor memory except the
      // last 128 columns): park its upper half there, hand it back sooner
      const uint32_t park = tmem + uint32_t(P_PARK_COL) +
                            (uint32_t(32 * quarter) << 16);
      const bool parked = kLoTmem && w.sk < 0 && p.tma_c;
      if (parked) {
        park_upper_half(acc, park);
        store_c_tma(acc, stg, &tmC, lane, n0, r0q, item, p.sc.alpha, 0, 4);
      } else if (w.sk < 0 && p.tma_c) {
        store_c_tma(acc, stg, &tmC, lane, n0, r0q, item, p.sc.alpha, 0,
                    PN / 32);
      } else if (w.sk < 0) {
        store_c_staged(acc, stg, cq, p.ldc, rows_in, cols_in, lane, p.sc);
      } else {
        // this block's piece, warp-major: lane quarter q's column block cb
        // is 4 KiB at float4 (q * 8 + cb) * 256, element (e, lane) at
        // e * 32 + lane (stores coalesced per warp; one bulk copy per block
        // for the fix-up)
        const long long x0 = (long long)w.sk * p.T;
        slot = sk_begin(cl, p) >= x0 ? 0 : 1;
        float4* piece = ws4 + ((long long)(cl * 2 + slot) * 2 + rank) *
                                  (P_PIECE_FLOATS / 4) +
                        quarter * 8 * 256 + lane;
#pragma unroll 1
        for (int cb = 0; cb < PN / 32; ++cb) {
          uint32_t v[32];
          tc::tmem_ld_32x32b_x32(acc + 32 * cb, v);
          tc::tmem_ld_wait();
#pragma unroll
          for (int e = 0; e < 8; ++e)
            __stcg(piece + (cb * 8 + e) * 32,
                   make_float4(__uint_as_float(v[4 * e]),
                               __uint_as_float(v[4 * e + 1]),
                               __uint_as_float(v[4 * e + 2]),
                               __uint_as_float(v[4 * e + 3])));
        }
      }
      // accumulator b may be overwritten by the next unit's MMAs
      tc::fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0)
          mbar_arrive(acce0 + 8 * b);
        else
          mbar_arrive_cluster(acce_leader + 8 * b);
      }
      if (parked)  // column block cb of the parked half at park + 32 (cb - 4)
        store_c_tma(park - 128, stg, &tmC, lane, n0, r0q, item, p.sc.alpha, 4,
                    PN / 32);
      if (w.sk < 0) continue;
      // ------------------------------------------------ stream-K fixup
      __threadfence();
      __syncwarp();
      int* counter = p.counters + (w.sk * 2 + int(rank)) * 4 + quarter;
      int arrived = 0;
      if (lane == 0) arrived = atomicAdd(counter, 1);
      arrived = __shfl_sync(0xffffffffu, arrived, 0);
      const long long x0 = (long long)w.sk * p.T;
      const int c_first = sk_owner(x0, p);
      const int pieces = sk_owner(x0 + p.T - 1, p) - c_first + 1;
      if (arrived != pieces - 1) continue;
      __threadfence();
      // The last piece is in. If this cluster's stream-K share ends inside
      // this tile and whole tiles follow (they come after the share), the
      // stage ring stays busy for a whole tile: sum the pieces now, under
      // those MMAs. Otherwise (only partial segments left) defer it until
      // this warp's units are done, when the ring is free for a deep copy
      // pipeline.
      if (kEarlyFix && w.ke < p.T && cl < p.dp_tiles) {
        fixup_direct(ws4, w.tile, rank, quarter, lane, p);
        __syncwarp();
        if (lane == 0) p.counters[(w.sk * 2 + int(rank)) * 4 + quarter] = 0;
        continue;
      }
      if (nfix < kMaxFix) fix_tile[nfix++] = w.tile;

    }
    // ------------------------------------------------ stream-K fix-ups
    // All MMAs of this cluster have completed (its last accumulator is
    // in), so the stage ring is free: each epilogue warp streams the
    // pieces through 12 slots of 4 KiB of it with cp.async (11 chunks in
    // flight), every lane its own row, and adds them into the staging box
    // in piece (k) order; a finished box goes out as coalesced rows.
    if (lane == 0) bulk_wait_group_read<0>();  // boxes free of bulk stores
    __syncwarp();
    for (int f = 0; f < nfix && !*abort_flag; ++f) {
      int item, pm, pn;
      pair_tile(fix_tile[f], p, item, pm, pn);
      const int sk = fix_tile[f] - p.dp_tiles;
      const long long x0 = (long long)sk * p.T;
      const int c_first = sk_owner(x0, p);
      const int pieces = sk_owner(x0 + p.T - 1, p) - c_first + 1;
      const int n0 = pn * PN;
      const int r0q = pm * PM + 128 * int(rank) + 32 * quarter;
      float* cq = p.C + item * p.bt.stride_c + (long long)r0q * p.ldc + n0;
      const int rows_in = p.M - r0q < 32 ? p.M - r0q : 32;
      const int cols_in = p.N - n0 < PN ? p.N - n0 : PN;
      uint8_t* stg = stg0 + (warp - P_EPI_WARP0) * 2 * P_STG_BOX;
      uint8_t* slots = smem + (warp - P_EPI_WARP0) * kFixRegion;
      // Piece of contributor j: only the first contributor's share can
      // start before the tile, so only its piece can be its second slot.
      const int s_first = sk_begin(c_first, p) >= x0 ? 0 : 1;
      auto piece = [&](int j) {
        return ws4 + ((long long)((c_first + j) * 2 + (j == 0 ? s_first : 0)) *
                          2 + rank) * (P_PIECE_FLOATS / 4) + quarter * 8 * 256;
      };
      // Chunk (column block icb, piece ij) = 4 KiB, one bulk copy by lane 0
      // into slot islot, completing on that slot's mbarrier.
      const uint32_t bar0 = smem_u32(slots + kFixSlots * P_STG_BOX);
      if (lane == 0) {
        for (int i = 0; i < kFixSlots; ++i) mbar_init(bar0 + 8 * i, 1);
        mbar_fence_init();
        // the other blocks' piece stores (generic) before the bulk reads
        asm volatile("fence.proxy.async.global;" ::: "memory");
      }
      __syncwarp();
      const int nb = pieces * (PN / 32);
      int icb = 0, ij = 0, issued = 0;
      auto issue_next = [&]() {
        if (issued < nb) {
          if (lane == 0) {
            const int sl = issued % kFixSlots;
            mbar_arrive_expect_tx(bar0 + 8 * sl, P_STG_BOX);
            bulk_load(smem_u32(slots + sl * P_STG_BOX), piece(ij) + icb * 256,
                      P_STG_BOX, bar0 + 8 * sl);
          }
          if (++ij == pieces) {
            ij = 0;
            ++icb;
          }
          ++issued;
        }
      };
      for (int t = 0; t < kFixSlots; ++t) issue_next();
      bool fix_ok = true;
      int t = 0;
#pragma unroll 1
      for (int cb = 0; cb < PN / 32 && fix_ok; ++cb) {
        float4 acc[8];
#pragma unroll 1
        for (int j = 0; j < pieces; ++j, ++t) {
          const int sl = t % kFixSlots;
          fix_ok = mbar_wait_bounded(bar0 + 8 * sl, (t / kFixSlots) & 1,
                                     p.status, kSiteTf32Fix, kWaitLimitNs);
          fix_ok = __all_sync(0xffffffffu, fix_ok);
          if (!fix_ok) break;
          const float4* slot4 =
              reinterpret_cast<const float4*>(slots + sl * P_STG_BOX) + lane;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float4 x = slot4[e * 32];
            if (j == 0) {
              acc[e] = x;
            } else {
              acc[e].x += x.x;
              acc[e].y += x.y;
              acc[e].z += x.z;
              acc[e].w += x.w;
            }
          }
          __syncwarp();   // every lane has read the slot ...
          issue_next();   // ... before it is refilled
        }
        if (!fix_ok) break;
        if (p.tma_c) {
          // bulk tensor store of the block (the two boxes alternate; a box
          // is rewritten once the store issued from it has read it)
          uint8_t* box = stg + (cb & 1) * P_STG_BOX;
          if (lane == 0) bulk_wait_group_read<1>();
          __syncwarp();
#pragma unroll
          for (int e = 0; e < 8; ++e)
            *reinterpret_cast<float4*>(box + lane * 128 +
                                       ((e ^ (lane & 7)) << 4)) =
                make_float4(p.sc.alpha * acc[e].x, p.sc.alpha * acc[e].y,
                            p.sc.alpha * acc[e].z, p.sc.alpha * acc[e].w);
          fence_async_shared();  // generic writes -> visible to the store
          __syncwarp();
          if (lane == 0) {
            tma_store_3d(&tmC, smem_u32(box), n0 + 32 * cb, r0q, item);
            bulk_commit_group();
          }
          continue;
        }
        __syncwarp();  // the previous block's rows have been written out
#pragma unroll
        for (int e = 0; e < 8; ++e)
          *reinterpret_cast<float4*>(stg + lane * 128 + ((e ^ (lane & 7)) << 4)) =
              acc[e];
        __syncwarp();
        write_box_rows(stg, cq + 32 * cb, p.ldc, rows_in,
                       cols_in - 32 * cb < 32 ? cols_in - 32 * cb : 32, lane,
                       p.sc);
      }
      if (!fix_ok) *abort_flag = 1;
      // copies still in flight land before the slots' barriers go away
      if (lane == 0) {
        for (int d = t; d < issued; ++d)
          mbar_wait_bounded(bar0 + 8 * (d % kFixSlots), (d / kFixSlots) & 1,
                            p.status, kSiteTf32Fix, kWaitLimitNs / 100);
        for (int i = 0; i < kFixSlots; ++i) mbar_inval(bar0 + 8 * i);
      }
      __syncwarp();
      if (lane == 0)
        p.counters[(sk * 2 + int(rank)) * 4 + quarter] = 0;
    }
    if (lane == 0) bulk_wait_group_all();  // C stores complete
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

template <int OA, int OB>
cudaError_t set_smem_attrs() {
  const cudaError_t e = cudaFuncSetAttribute(
      k_tf32x3<OA, OB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
      int(X_SMEM));
  if (e != cudaSuccess) return e;
  const cudaError_t e2 = cudaFuncSetAttribute(
      k_tf32x3_pair<OA, OB, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
      int(P_SMEM));
  if (e2 != cudaSuccess) return e2;
  return cudaFuncSetAttribute(k_tf32x3_pair<OA, OB, true>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              int(P_SMEM));
}

cudaError_t tf32x3_init(int* pair_clusters) {
  cudaError_t e = set_smem_attrs<0, 0>();
  if (e == cudaSuccess) e = set_smem_attrs<0, 1>();
  if (e == cudaSuccess) e = set_smem_attrs<1, 0>();
  if (e == cudaSuccess) e = set_smem_attrs<1, 1>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(P_THREADS, 1, 1);
  cfg.dynamicSmemBytes = P_SMEM;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, k_tf32x3_pair<0, 0, false>, &cfg);
  if (e != cudaSuccess) return e;
  *pair_clusters = n;
  return n > 0 ? cudaSuccess : cudaErrorInvalidConfiguration;
}

PairPlan plan_pair(int64_t M, int64_t N, int64_t K, int clusters,
                   bool stream_k, int64_t batch) {
  PairPlan pl;
  pl.tiles_m = int((M + PM - 1) / PM);
  pl.tiles_n = int((N + PN - 1) / PN);
  pl.tiles = int(batch) * pl.tiles_m * pl.tiles_n;  // checked by the host
  pl.T = int((K + XK - 1) / XK);
  if (clusters < 1) clusters = 1;
  pl.G = pl.tiles < clusters ? pl.tiles : clusters;
  pl.dp_tiles = pl.tiles;
  pl.sk_tiles = 0;
  const int64_t rem = pl.tiles % clusters;
  if (stream_k && rem != 0) {
    if (pl.tiles < clusters) {
      // One partial wave: spread all k-slices over more clusters, when whole
      // tiles would leave over a quarter of them idle (above that, the
      // fix-up costs more than the idle clusters).
      const int64_t by_work = 4 * pl.tiles <= 3 * int64_t(clusters)
                                  ? int64_t(pl.tiles) * pl.T / kPairMinSkIters
                                  : 0;
      const int64_t G = by_work < clusters ? by_work : clusters;
      if (G > pl.tiles) {
        pl.G = int(G);
        pl.sk_tiles = pl.tiles;
        pl.dp_tiles = 0;
      }
    } else {
      int64_t sk = rem;
      if (sk * pl.T / clusters < kPairMinSkIters) sk += clusters;
      if (sk * pl.T / clusters >= kPairMinSkIters) {  // else: short K
        pl.G = clusters;
        pl.sk_tiles = int(sk);
        pl.dp_tiles = pl.tiles - pl.sk_tiles;
      }
    }
  }
  pl.sk_iters = int64_t(pl.sk_tiles) * pl.T;
  pl.ws_floats =
      pl.sk_tiles ? size_t(pl.G) * 2 * 2 * size_t(P_PIECE_FLOATS) : 0;
  pl.counters = size_t(pl.sk_tiles) * 2 * 4;
  return pl;
}

cudaError_t launch_tf32x3_pair(const GemmArgs& g, const CUtensorMap& tmA,
                               const CUtensorMap& tmB, const CUtensorMap* tmC,
                               const PairPlan& pl, float* ws, int* counters,
                               int* status, cudaStream_t s) {
  PairParams p;
  p.C = g.C;
  p.M = int(g.M);
  p.N = int(g.N);
  p.K = int(g.K);
  p.ldc = (long long)g.ldc;
  p.tiles_m = pl.tiles_m;
  p.tiles_n = pl.tiles_n;
  p.T = pl.T;
  p.G = pl.G;
  p.dp_tiles = pl.dp_tiles;
  p.sk_tiles = pl.sk_tiles;
  p.sk_iters = (long long)pl.sk_iters;
  p.ws = ws;
  p.counters = counters;
  // 16-byte stores need every item's rows on 16 bytes: the base, the row
  // pitch and, for a batch, the item stride.
  p.vec_store = (g.ldc % 4 == 0) &&
                (reinterpret_cast<uintptr_t>(g.C) % 16 == 0) &&
                (g.batch <= 1 || g.stride_c % 4 == 0);
  p.sc = g.sc;
  p.tma_c = tmC != nullptr && g.sc.beta == 0.f;
  const CUtensorMap& mapC = p.tma_c ? *tmC : tmA;  // unused without tma_c
  p.bt.items = int(g.batch);
  p.bt.a_batched = g.batch > 1 && g.stride_a != 0;
  p.bt.b_batched = g.batch > 1 && g.stride_b != 0;
  p.bt.stride_c = (long long)g.stride_c;
  p.status = status;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2u * unsigned(pl.G), 1, 1);
  cfg.blockDim = dim3(P_THREADS, 1, 1);
  cfg.dynamicSmemBytes = P_SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const bool early = pl.dp_tiles > 0 && pl.sk_tiles > 0;
  switch (g.op_a * 4 + g.op_b * 2 + (early ? 1 : 0)) {
    case 0: return counted(cudaLaunchKernelEx(&cfg, k_tf32x3_pair<0, 0, false>, tmA,
                                       tmB, mapC, p));
    case 1: return counted(cudaLaunchKernelEx(&cfg, k_tf32x3_pair<0, 0, true>, tmA,
                                       tmB, mapC, p));
    case 2: return counted(cudaLaunchKernelEx(&cfg, k_tf32x3_pair<0, 1, false>, tmA,
                                       tmB, mapC, p));
    case 3: return counted(cudaLaunchKernelEx(&cfg, k_tf32x3_pair<0, 1, true>, tmA,
                                       tmB, mapC, p));
    case 4: return counted(cudaLaunchKernelEx(&cfg, k_tf32x3_pair<1, 0, false>, tmA,
                                       tmB, mapC, p));
    case 5: return counted(cudaLaunchKernelEx(&cfg, k_tf32x3_pair<1, 0, true>, tmA,
                                       tmB, mapC, p));
    case 6: return counted(cudaLaunchKernelEx(&cfg, k_tf32x3_pair<1, 1, false>, tmA,
                                       tmB, mapC, p));
    default: return counted(cudaLaunchKernelEx(&cfg, k_tf32x3_pair<1, 1, true>, tmA,
                                        tmB, mapC, p));
  }
}

int plan_tf32x3_splits(int64_t M, int64_t N, int64_t K, int64_t batch,
                       int sms) {
  // Split k when the tiles fill under half of the SMs: up to the SMs the
  // tiles leave idle, at least 2 k-slices a split, at most 16 splits.
  const int64_t tiles = batch * ((M + XM - 1) / XM) * ((N + XN - 1) / XN);
  const int64_t T = (K + XK - 1) / XK;
  if (tiles <= 0 || 2 * tiles > sms) return 1;
  int64_t sp = sms / tiles;
  if (sp > T / 2) sp = T / 2;
  if (sp > 16) sp = 16;
  return sp < 2 ? 1 : int(sp);
}

size_t tf32x3_split_floats(int64_t M, int64_t N, int64_t batch, int splits) {
  if (splits <= 1) return 0;
  return size_t(batch) * size_t((M + XM - 1) / XM) * size_t((N + XN - 1) / XN) *
         size_t(splits) * XM * XN;
}

cudaError_t launch_tf32x3(const GemmArgs& g, const CUtensorMap& tmA,
                          const CUtensorMap& tmB, int* status, cudaStream_t s,
                          int splits, float* part) {
  const int tiles_m = int((g.M + XM - 1) / XM);
  const int tiles_n = int((g.N + XN - 1) / XN);
  const bool vec = (g.ldc % 4 == 0) &&
                   (reinterpret_cast<uintptr_t>(g.C) % 16 == 0) &&
                   (g.batch <= 1 || g.stride_c % 4 == 0);
  const unsigned grid = unsigned(g.batch) * unsigned(tiles_m) *
                        unsigned(tiles_n);  // < 2^31, checked by the host
  Batch bt;
  bt.items = int(g.batch);
  bt.a_batched = g.batch > 1 && g.stride_a != 0;
  bt.b_batched = g.batch > 1 && g.stride_b != 0;
  bt.stride_c = (long long)g.stride_c;
  if (splits < 1 || part == nullptr) splits = 1;
  float4* part4 = reinterpret_cast<float4*>(part);
  auto go = [&](auto kernel) {
    kernel<<<dim3(grid, unsigned(splits)), X_THREADS, X_SMEM, s>>>(
        tmA, tmB, g.C, int(g.M), int(g.N), int(g.K), (long long)g.ldc,
        tiles_m, tiles_n, vec ? 1 : 0, g.sc, bt, splits, part4, status);
  };
  switch (g.op_a * 2 + g.op_b) {
    case 0: go(k_tf32x3<0, 0>); break;
    case 1: go(k_tf32x3<0, 1>); break;
    case 2: go(k_tf32x3<1, 0>); break;
    default: go(k_tf32x3<1, 1>); break;
  }
  cudaError_t e = counted(cudaGetLastError());
  if (e != cudaSuccess || splits == 1) return e;
  k_splitk_reduce<<<dim3(grid, XM * XN / 4 / 256), 256, 0, s>>>(
      part4, splits, g.C, int(g.M), int(g.N), (long long)g.ldc, tiles_m,
      tiles_n, vec ? 1 : 0, g.sc, (long long)g.stride_c);
  return counted(cudaGetLastError());
}

}  // namespace dfm
