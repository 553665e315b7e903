// C ABI of the FP32 matrix-product library (declared in include/dfm_sgemm.h):
// argument checks, the host-side path decision, one-time per-device set-up,
// TMA descriptor encoding and the launches. The argument checks follow the
// host wrappers of "GEMM from naive to tiled", section 十一.1 (device,
// dtype, 2-D shape agreement), turned into status codes.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <memory>
#include <mutex>
#include <vector>

#include "dfm_sgemm.h"
#include "kernels.h"
#include "ptx.cuh"

namespace dfm {

std::atomic<uint64_t> g_launches{0};
void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
namespace {

// Per-device status word of the bounded waits (see ptx.cuh).
__device__ int g_status[4];

constexpr int kMaxDevices = 64;
std::atomic<int> g_math_mode{SGEMM_MATH_AUTO};
// Misaligned operands: repacked for the tensor path from this many
// multiply-adds on (below, the CUDA-core kernel that reads them as they are).
constexpr int64_t kTf32RepackMinMacs = int64_t(1) << 24;
// The same for the CUDA-core path: from this size the TMA-fed tile kernel
// (about 80% of the FMA peak) on repacked copies beats the any-layout
// kernel (about 57% on 4095 x 4097 x 1023) by more than the copies cost.
constexpr int64_t kFfmaRepackMinMacs = int64_t(1) << 32;
// From this much work on (256 x 256 tiles x k-slices of 32) the 2-SM pair
// kernel, which splits k-slices over all clusters when tiles are few, beats
// one 1-SM block per 128 x 128 tile (measured: every long-K shape of few
// tiles goes to pairs, 512^3 stays on single blocks), except for the short-k
// few-tile products below.
constexpr int64_t kTf32PairMinWork = 256;
// Below this many 128 x 128 tiles (half of GB300's 152 SMs) single blocks
// split k over the idle SMs; with short k (up to this many k-slices) that
// beats the pairs' stream-K split (1024^3: 29 vs 35 us), with longer k the
// pairs win (1024 x 1024 x 4096: 59 vs 78 us).
constexpr int64_t kSplitMaxTiles = 76;
// Up to this many multiply-adds the small-tile kernel takes the product.
constexpr int64_t kSmallMaxMacs = int64_t(1) << 23;
constexpr int64_t kSplitMaxSlices = 32;

int64_t pair_work(int64_t M, int64_t N, int64_t K, int64_t batch) {
  return batch * ((M + 255) / 256) * ((N + 255) / 256) * ((K + 31) / 32);
}

// The tensor path's kernel: 2-SM pairs, or single blocks (split-k when the
// tiles are few).
bool use_pair(int64_t M, int64_t N, int64_t K, int64_t batch) {
  if (pair_work(M, N, K, batch) < kTf32PairMinWork) return false;
  const int64_t tiles = batch * ((M + 127) / 128) * ((N + 127) / 128);
  return !(tiles <= kSplitMaxTiles && (K + 31) / 32 <= kSplitMaxSlices);
}
// Largest M, N or K the int-indexed kernels accept (tile rounding included).
constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1024;

struct Workspace {
  float* ws = nullptr;
  size_t ws_floats = 0;
  int* counters = nullptr;
  size_t counters_len = 0;
  float* tr = nullptr;   // row-major copies of transposed operands
  size_t tr_floats = 0;
  cudaStream_t stream = nullptr;  // the stream it serves now
  cudaEvent_t done = nullptr;     // recorded after each call's launches
  bool recorded = false;          // `done` holds a record
  bool pinned = false;  // used inside a stream capture: a graph holds its
                        // addresses, so it is never handed to another stream
  uint64_t last_use = 0;

  size_t bytes() const {
    return (ws_floats + tr_floats) * sizeof(float) + counters_len * sizeof(int);
  }
};

// Workspaces cached per device. Up to kMaxWorkspaces are kept; a call on a
// stream that has none takes a new one while there is room, else the least
// recently used one that no captured graph holds, after making its stream
// wait (on the device) for that workspace's last call.
constexpr size_t kMaxWorkspaces = 8;

struct DeviceState {
  std::once_flag once;
  int err = SGEMM_OK;
  int sms = 0;
  int tma_blocks_per_sm = 0;
  int pair_clusters = 0;  // 2-block clusters of the pair kernel at once
  int* status = nullptr;
  // Stream-K workspaces (partial tiles and tile counters) and transposed
  // copies: kernels on unordered streams may run at the same time, so a
  // workspace serves one stream at a time.
  std::mutex ws_mu;
  std::vector<std::unique_ptr<Workspace>> pool;
  uint64_t tick = 0;
};

DeviceState g_dev[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t,
                                   void*, const cuuint64_t*, const cuuint64_t*,
                                   const cuuint32_t*, const cuuint32_t*,
                                   CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);
std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

EncodeTiledFn encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
  });
  return g_encode;
}

void init_device(DeviceState& st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    st.err = SGEMM_ERR_CUDA;
    return;
  }
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev) !=
          cudaSuccess) {
    st.err = SGEMM_ERR_CUDA;
    return;
  }
  if (major != 10 || minor != 3) {  // built for sm_103a only
    st.err = SGEMM_ERR_UNSUPPORTED_DEVICE;
    return;
  }
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&st.status), g_status) !=
          cudaSuccess ||
      cudaMemset(st.status, 0, sizeof(int) * 4) != cudaSuccess ||
      tiled_init(&st.tma_blocks_per_sm) != cudaSuccess ||
      st.tma_blocks_per_sm < 1 || small_init() != cudaSuccess ||
      gemv_tma_init() != cudaSuccess ||
      tf32x3_init(&st.pair_clusters) != cudaSuccess) {
    st.err = SGEMM_ERR_CUDA;
    return;
  }
  st.err = SGEMM_OK;
}

// One-time set-up of the current device; returns its state or an error.
int device_state(DeviceState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SGEMM_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SGEMM_ERR_UNSUPPORTED_DEVICE;
  DeviceState& st = g_dev[dev];
  std::call_once(st.once, [&] { init_device(st); });
  *out = &st;
  return st.err;
}

bool capturing(cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  return cudaStreamIsCapturing(s, &cs) == cudaSuccess &&
         cs != cudaStreamCaptureStatusNone;
}

// One call's hold on the workspace of its stream: holds the device's
// workspace lock from construction to destruction (after the call's
// launches are enqueued) and, if the call used a workspace, records that
// workspace's `done` event on the stream at the end.
class Lease {
 public:
  Lease(DeviceState& st, cudaStream_t s) : st_(st), s_(s), lock_(st.ws_mu) {}
  ~Lease() {
    if (w_ == nullptr) return;
    if (capturing(s_)) {
      w_->pinned = true;
    } else if (cudaEventRecord(w_->done, s_) == cudaSuccess) {
      w_->recorded = true;
    }
  }
  Lease(const Lease&) = delete;
  Lease& operator=(const Lease&) = delete;

  cudaStream_t stream() const { return s_; }

  // The workspace serving this stream (taken on first use).
  int get(Workspace** out) {
    if (w_ == nullptr) {
      const int rc = take();
      if (rc != SGEMM_OK) return rc;
    }
    w_->last_use = ++st_.tick;
    *out = w_;
    return SGEMM_OK;
  }

 private:
  int take() {
    const bool cap = capturing(s_);
    Workspace* w = nullptr;
    for (auto& e : st_.pool)
      if (e->stream == s_) w = e.get();
    if (w == nullptr && st_.pool.size() >= kMaxWorkspaces && !cap) {
      // hand the least recently used unpinned workspace to this stream
      for (auto& e : st_.pool)
        if (!e->pinned && (w == nullptr || e->last_use < w->last_use))
          w = e.get();
    }
    if (w == nullptr) {
      auto e = std::make_unique<Workspace>();
      if (cudaEventCreateWithFlags(&e->done, cudaEventDisableTiming) !=
          cudaSuccess)
        return SGEMM_ERR_CUDA;
      e->stream = s_;
      w = e.get();
      st_.pool.push_back(std::move(e));
    }
    // Order this call after the workspace's previous call: a workspace
    // handed over from another stream, or a stream handle that was
    // destroyed and reissued with work of its old stream still running.
    if (w->recorded && !cap &&
        cudaStreamWaitEvent(s_, w->done, 0) != cudaSuccess)
      return SGEMM_ERR_CUDA;
    w->stream = s_;
    w_ = w;
    return SGEMM_OK;
  }

  DeviceState& st_;
  cudaStream_t s_;
  std::lock_guard<std::mutex> lock_;
  Workspace* w_ = nullptr;
};

// Free `p` once the workspace's previous call is done (the host waits for
// it; cudaFree itself may also wait for the device).
void release(Workspace& w, void* p) {
  if (p == nullptr) return;
  if (w.recorded) cudaEventSynchronize(w.done);
  cudaFree(p);
}

// Make the stream's workspace at least `floats` partial-tile floats and
// `counters` tile counters. Growing replaces the buffer (cudaFree and
// cudaMalloc: these may synchronise the device) and zeroes new counters
// on the stream; the kernels leave the counters at zero when they finish.
int ensure_workspace(Lease& ls, size_t floats, size_t counters,
                     Workspace** out) {
  Workspace* wp = nullptr;
  const int rc = ls.get(&wp);
  if (rc != SGEMM_OK) return rc;
  Workspace& w = *wp;
  if (floats > w.ws_floats) {
    release(w, w.ws);
    w.ws = nullptr;
    w.ws_floats = 0;
    if (cudaMalloc(&w.ws, floats * sizeof(float)) != cudaSuccess)
      return SGEMM_ERR_CUDA;
    w.ws_floats = floats;
  }
  if (counters > w.counters_len) {
    release(w, w.counters);
    w.counters = nullptr;
    w.counters_len = 0;
    if (cudaMalloc(&w.counters, counters * sizeof(int)) != cudaSuccess ||
        cudaMemsetAsync(w.counters, 0, counters * sizeof(int),
                        ls.stream()) != cudaSuccess)
      return SGEMM_ERR_CUDA;
    w.counters_len = counters;
  }
  *out = &w;
  return SGEMM_OK;
}

// Grow the transposed-copy buffer of the stream's workspace.
int ensure_tr(Lease& ls, size_t floats, Workspace** out) {
  Workspace* wp = nullptr;
  const int rc = ls.get(&wp);
  if (rc != SGEMM_OK) return rc;
  Workspace& w = *wp;
  *out = &w;
  if (floats <= w.tr_floats) return SGEMM_OK;
  release(w, w.tr);
  w.tr = nullptr;
  w.tr_floats = 0;
  if (cudaMalloc(&w.tr, floats * sizeof(float)) != cudaSuccess)
    return SGEMM_ERR_CUDA;
  w.tr_floats = floats;
  return SGEMM_OK;
}

int check_args(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
               const void* B, int64_t ldb, const void* C, int64_t ldc) {
  if (M < 0 || N < 0 || K < 0) return SGEMM_ERR_INVALID_VALUE;
  if (lda < (K > 1 ? K : 1) || ldb < (N > 1 ? N : 1) || ldc < (N > 1 ? N : 1))
    return SGEMM_ERR_INVALID_VALUE;
  if (M > kMaxDim || N > kMaxDim || K > kMaxDim) return SGEMM_ERR_TOO_LARGE;
  if (M > 0 && N > 0) {
    if (C == nullptr) return SGEMM_ERR_NULL_POINTER;
    if (K > 0 && (A == nullptr || B == nullptr)) return SGEMM_ERR_NULL_POINTER;
  }
  return SGEMM_OK;
}

// Byte span [lo, hi) touched by a rows x cols matrix with leading dim ld.
void span(uint64_t base, int64_t rows, int64_t cols, int64_t ld, uint64_t& lo,
          uint64_t& hi) {
  lo = base;
  hi = base + uint64_t(((rows - 1) * ld + cols) * 4);
}

bool overlaps(uint64_t a, int64_t ar, int64_t ac, int64_t ald, uint64_t c,
              int64_t cr, int64_t cc, int64_t cld) {
  if (ar <= 0 || ac <= 0 || cr <= 0 || cc <= 0) return false;
  uint64_t alo, ahi, clo, chi;
  span(a, ar, ac, ald, alo, ahi);
  span(c, cr, cc, cld, clo, chi);
  return alo < chi && clo < ahi;
}

bool tma_operand_ok(uint64_t addr, int64_t ld) {
  // TMA: 16-byte aligned base, row stride a multiple of 16 bytes and < 2^40.
  return addr % 16 == 0 && (ld * 4) % 16 == 0 && ld * 4 < (int64_t(1) << 40);
}

int encode_maps(const GemmArgs& g, CUtensorMap* tmA, CUtensorMap* tmB) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return SGEMM_ERR_CUDA;
  // A: dims {K, M} (innermost first), row stride lda * 4 bytes, box
  // {kTileK, kTileM} = 128 bytes x 128 rows, 128-byte swizzle.
  {
    const cuuint64_t dims[2] = {cuuint64_t(g.K), cuuint64_t(g.M)};
    const cuuint64_t strides[1] = {cuuint64_t(g.lda) * 4};
    const cuuint32_t box[2] = {cuuint32_t(kTileK), cuuint32_t(kTileM)};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(tmA, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(g.A),
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return SGEMM_ERR_CUDA;
  }
  // B: dims {N, K}, row stride ldb * 4 bytes, box {kTileN, kTileK} = 512
  // bytes x 32 rows, no swizzle.
  {
    const cuuint64_t dims[2] = {cuuint64_t(g.N), cuuint64_t(g.K)};
    const cuuint64_t strides[1] = {cuuint64_t(g.ldb) * 4};
    const cuuint32_t box[2] = {cuuint32_t(kTileN), cuuint32_t(kTileK)};
    const cuuint32_t estr[2] = {1, 1};
    if (enc(tmB, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(g.B),
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return SGEMM_ERR_CUDA;
  }
  return SGEMM_OK;
}

// Generic 2-D fp32 tensor map: dims {inner, outer}, row stride ld floats.
int encode_2d(CUtensorMap* map, const float* base, int64_t inner,
              int64_t outer, int64_t ld, uint32_t box_inner,
              uint32_t box_outer,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return SGEMM_ERR_CUDA;
  const cuuint64_t dims[2] = {cuuint64_t(inner), cuuint64_t(outer)};
  const cuuint64_t strides[1] = {cuuint64_t(ld) * 4};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float*>(base),
             dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? SGEMM_OK
             : SGEMM_ERR_CUDA;
}

// 3-D fp32 map {inner, outer, items}: rows ld floats apart, items `stride`
// floats apart (one item: stride = the packed ld * outer), box
// {box_inner, box_outer, 1}.
int encode_3d(CUtensorMap* map, const float* base, int64_t inner,
              int64_t outer, int64_t ld, int64_t items, int64_t stride,
              uint32_t box_inner, uint32_t box_outer,
              CUtensorMapSwizzle swizzle) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return SGEMM_ERR_CUDA;
  if (items <= 1) {
    items = 1;
    stride = ld * outer;
  }
  const cuuint64_t dims[3] = {cuuint64_t(inner), cuuint64_t(outer),
                              cuuint64_t(items)};
  const cuuint64_t strides[2] = {cuuint64_t(ld) * 4, cuuint64_t(stride) * 4};
  const cuuint32_t box[3] = {box_inner, box_outer, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(base),
             dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? SGEMM_OK
             : SGEMM_ERR_CUDA;
}

int encode_1d(CUtensorMap* map, const float* base, int64_t n, uint32_t box) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return SGEMM_ERR_CUDA;
  const cuuint64_t dims[1] = {cuuint64_t(n)};
  const cuuint64_t unused_strides[1] = {cuuint64_t((n * 4 + 15) / 16 * 16)};
  const cuuint32_t boxd[1] = {box};
  const cuuint32_t estr[1] = {1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 1, const_cast<float*>(base),
             dims, unused_strides, boxd, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? SGEMM_OK
             : SGEMM_ERR_CUDA;
}

cudaError_t run_gemv_row(const GemmArgs& g, const DeviceState& st,
                         cudaStream_t s, int* rc_out) {
  *rc_out = SGEMM_OK;
  if (tma_operand_ok(reinterpret_cast<uint64_t>(g.B), g.ldb) &&
      reinterpret_cast<uint64_t>(g.A) % 16 == 0) {
    CUtensorMap tmB, tma_;
    int rc = encode_2d(&tmB, g.B, g.N, g.K, g.ldb, 64, 64);
    if (rc == SGEMM_OK) rc = encode_1d(&tma_, g.A, g.K, 64);
    if (rc != SGEMM_OK) {
      *rc_out = rc;
      return cudaSuccess;
    }
    return launch_gemv_row_tma(g, tmB, tma_, plan_gemv_row(g.N, g.K, st.sms),
                               st.status, s);
  }
  return launch_gemv_row(g, st.sms, s);
}

cudaError_t run_gemv_col(const GemmArgs& g, const DeviceState& st,
                         cudaStream_t s, int* rc_out) {
  *rc_out = SGEMM_OK;
  if (tma_operand_ok(reinterpret_cast<uint64_t>(g.A), g.lda) && g.ldb == 1 &&
      reinterpret_cast<uint64_t>(g.B) % 16 == 0) {
    CUtensorMap tmA, tmb;
    int rc = encode_2d(&tmA, g.A, g.K, g.M, g.lda, 256, 16);
    if (rc == SGEMM_OK) rc = encode_1d(&tmb, g.B, g.K, 256);
    if (rc != SGEMM_OK) {
      *rc_out = rc;
      return cudaSuccess;
    }
    return launch_gemv_col_tma(g, tmA, tmb, st.sms, st.status, s);
  }
  return launch_gemv_col(g, st.sms, s);
}

int to_status(cudaError_t e) {
  if (e == cudaSuccess) return SGEMM_OK;
  return (e == cudaErrorLaunchFailure || e == cudaErrorInvalidConfiguration ||
          e == cudaErrorLaunchOutOfResources || e == cudaErrorInvalidValue)
             ? SGEMM_ERR_LAUNCH
             : SGEMM_ERR_CUDA;
}

// Maps of the tensor-core kernels. A K-major operand (A stored M x K, or B
// stored N x K) is one box {32 k, 128 rows}; an MN-major one (A stored
// K x M, or B stored K x N) is read as boxes {32 rows, 32 k}. All with the
// 128-byte swizzle.
// The third dimension is the batch item (extent 1 unless the operand
// differs between items).
int encode_tf32x3(const GemmArgs& g, CUtensorMap* tmA, CUtensorMap* tmB) {
  const int64_t ia = g.batch > 1 && g.stride_a != 0 ? g.batch : 1;
  const int64_t ib = g.batch > 1 && g.stride_b != 0 ? g.batch : 1;
  const auto sw = CU_TENSOR_MAP_SWIZZLE_128B;
  const int rc =
      g.op_a == 0
          ? encode_3d(tmA, g.A, g.K, g.M, g.lda, ia, g.stride_a, 32, 128, sw)
          : encode_3d(tmA, g.A, g.M, g.K, g.lda, ia, g.stride_a, 32, 32, sw);
  if (rc != SGEMM_OK) return rc;
  return g.op_b == 0
             ? encode_3d(tmB, g.B, g.N, g.K, g.ldb, ib, g.stride_b, 32, 32, sw)
             : encode_3d(tmB, g.B, g.K, g.N, g.ldb, ib, g.stride_b, 32, 128,
                         sw);
}

// ls: the call's hold on its stream's workspace; nullptr when the call
// may not allocate (then no split-k and the caller handles pairs).
int run_tf32x3(const GemmArgs& g, DeviceState& st, cudaStream_t s,
               bool pair, Lease* ls) {
  const bool may_alloc = ls != nullptr;
  CUtensorMap tmA, tmB;
  const int rc = encode_tf32x3(g, &tmA, &tmB);
  if (rc != SGEMM_OK) return rc;
  if (!pair) {
    // few tiles: split k over the idle SMs (the pieces need workspace)
    const int splits =
        may_alloc ? plan_tf32x3_splits(g.M, g.N, g.K, g.batch, st.sms) : 1;
    if (splits == 1)
      return to_status(launch_tf32x3(g, tmA, tmB, st.status, s));
    Workspace* w = nullptr;
    const int wrc = ensure_workspace(
        *ls, tf32x3_split_floats(g.M, g.N, g.batch, splits), 0, &w);
    if (wrc != SGEMM_OK) return wrc;
    return to_status(
        launch_tf32x3(g, tmA, tmB, st.status, s, splits, w->ws));
  }
  const PairPlan pl =
      plan_pair(g.M, g.N, g.K, st.pair_clusters, true, g.batch);
  Workspace* w = nullptr;
  if (ls == nullptr) return SGEMM_ERR_PATH;
  const int wrc = ensure_workspace(*ls, pl.ws_floats, pl.counters, &w);
  if (wrc != SGEMM_OK) return wrc;
  // C by bulk tensor stores when it is not read (beta == 0) and aligned.
  // Rows must also end on a 16-byte boundary (N a multiple of 4): a bulk
  // tensor store writes the last 16-byte chunk of a row whole, so with
  // N % 4 != 0 it would write up to 3 floats past column N - 1 (into the
  // pitch padding, or past the end of C on the last row).
  CUtensorMap tmC;
  const bool c_ok =
      g.sc.beta == 0.f && g.N % 4 == 0 &&
      tma_operand_ok(reinterpret_cast<uint64_t>(g.C), g.ldc) &&
      (g.batch <= 1 || g.stride_c % 4 == 0) &&
      encode_3d(&tmC, g.C, g.N, g.M, g.ldc, g.batch, g.stride_c, 32, 32,
                CU_TENSOR_MAP_SWIZZLE_128B) == SGEMM_OK;
  return to_status(launch_tf32x3_pair(g, tmA, tmB, c_ok ? &tmC : nullptr, pl,
                                      w->ws, w->counters, st.status, s));
}

// ---------------------------------------------------------------- calls
//
// Every computing entry point is one call C = alpha * op(A) * op(B) +
// beta * C (sgemm: no transposes, alpha = 1, beta = 0).
struct Call {
  int op_a, op_b;
  int64_t M, N, K;
  float alpha;
  const float* A;
  int64_t lda;
  const float* B;
  int64_t ldb;
  float beta;
  float* C;
  int64_t ldc;
};

// A and B are read only when there are products to form (BLAS: alpha == 0
// leaves them unreferenced).
bool reads_ab(const Call& c) { return c.alpha != 0.f && c.K > 0; }

int check_call(const Call& c) {
  if ((c.op_a != SGEMM_OP_N && c.op_a != SGEMM_OP_T) ||
      (c.op_b != SGEMM_OP_N && c.op_b != SGEMM_OP_T))
    return SGEMM_ERR_INVALID_VALUE;
  if (c.M < 0 || c.N < 0 || c.K < 0) return SGEMM_ERR_INVALID_VALUE;
  const int64_t a_cols = c.op_a ? c.M : c.K, b_cols = c.op_b ? c.K : c.N;
  if (c.lda < (a_cols > 1 ? a_cols : 1) || c.ldb < (b_cols > 1 ? b_cols : 1) ||
      c.ldc < (c.N > 1 ? c.N : 1))
    return SGEMM_ERR_INVALID_VALUE;
  if (c.M > kMaxDim || c.N > kMaxDim || c.K > kMaxDim)
    return SGEMM_ERR_TOO_LARGE;
  if (c.M > 0 && c.N > 0) {
    if (c.C == nullptr) return SGEMM_ERR_NULL_POINTER;
    if (reads_ab(c) && (c.A == nullptr || c.B == nullptr))
      return SGEMM_ERR_NULL_POINTER;
  }
  return SGEMM_OK;
}

bool call_overlaps(const Call& c) {
  if (!reads_ab(c)) return false;
  const uint64_t a = reinterpret_cast<uint64_t>(c.A);
  const uint64_t b = reinterpret_cast<uint64_t>(c.B);
  const uint64_t cc = reinterpret_cast<uint64_t>(c.C);
  return overlaps(a, c.op_a ? c.K : c.M, c.op_a ? c.M : c.K, c.lda, cc, c.M,
                  c.N, c.ldc) ||
         overlaps(b, c.op_b ? c.N : c.K, c.op_b ? c.K : c.N, c.ldb, cc, c.M,
                  c.N, c.ldc);
}

// N == 1 with A stored transposed (K x M): c^T = b^T A_stored is a row
// vector times a row-major matrix, streamed by the M == 1 kernel without a
// transposed copy of A, when c and b are contiguous.
bool gemv_col_as_row(const Call& c) {
  return c.N == 1 && c.op_a && c.ldc == 1 && (c.op_b || c.ldb == 1);
}

// Host-only path choice (no device access): the kernel that computes the
// products. AUTO when no kernel runs (empty C, or nothing to multiply).
int plan_call(const Call& c) {
  if (c.M == 0 || c.N == 0 || !reads_ab(c)) return SGEMM_PATH_AUTO;
  const uint64_t a = reinterpret_cast<uint64_t>(c.A);
  const uint64_t b = reinterpret_cast<uint64_t>(c.B);
  // c = a * B^T is a product of B's rows with a: the N == 1 kernel; and
  // c = A^T b (A stored K x M) is the row b^T A: the M == 1 kernel.
  if (c.M == 1) return c.op_b ? SGEMM_PATH_GEMV_COL : SGEMM_PATH_GEMV_ROW;
  if (c.N == 1)
    return gemv_col_as_row(c) ? SGEMM_PATH_GEMV_ROW : SGEMM_PATH_GEMV_COL;
  // Products too small to fill the GPU: the 32 x 32 tile kernel, in either
  // math mode (measured faster than every other path up to about 2^23
  // multiply-adds: 127 x 129 x 33 in 7.7 us against 16.8, 128^3 10.3 against
  // 15.3; at 256^3 the tensor kernel ties, above it wins).
  if (double(c.M) * double(c.N) * double(c.K) <= double(kSmallMaxMacs) &&
      c.M <= kSmallMaxRows)
    return SGEMM_PATH_SMALL;
  const int64_t tiles = ((c.M + kTileM - 1) / kTileM) *
                        ((c.N + kTileN - 1) / kTileN);
  // Operands the tensor maps cannot take (row stride or base not 16-byte
  // aligned) are repacked first when the product is large enough to pay
  // for the extra pass over them.
  const bool aligned = tma_operand_ok(a, c.lda) && tma_operand_ok(b, c.ldb);
  const bool repack_pays =
      double(c.M) * double(c.N) * double(c.K) >= double(kTf32RepackMinMacs);
  if ((aligned || repack_pays) &&
      g_math_mode.load(std::memory_order_relaxed) == SGEMM_MATH_AUTO) {
    return use_pair(c.M, c.N, c.K, 1) ? SGEMM_PATH_TF32X3_PAIR
                                      : SGEMM_PATH_TF32X3;
  }
  // CUDA-core tile kernels take row-major operands; a transposed one is
  // first copied row-major (dense, ld = its width) into the workspace.
  const bool a_ok = c.op_a ? c.K % 4 == 0 : tma_operand_ok(a, c.lda);
  const bool b_ok = c.op_b ? c.N % 4 == 0 : tma_operand_ok(b, c.ldb);
  // Untransposed operands TMA cannot map are repacked to 16-byte rows
  // first when the product is large enough to pay for it.
  const bool repack = !c.op_a && !c.op_b &&
                      double(c.M) * double(c.N) * double(c.K) >=
                          double(kFfmaRepackMinMacs);
  // The stream-K schedule counts k-slice iterations in 32 bits.
  const int64_t iters = tiles * ((c.K + kTileK - 1) / kTileK);
  return ((a_ok && b_ok) || repack) && iters < (1ll << 31)
             ? SGEMM_PATH_TILED_TMA
             : SGEMM_PATH_TILED_LDG;
}

int plan_path(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
              uint64_t a, uint64_t b) {
  const Call c{SGEMM_OP_N, SGEMM_OP_N, M, N, K, 1.f,
               reinterpret_cast<const float*>(a), lda,
               reinterpret_cast<const float*>(b), ldb, 0.f, nullptr, 1};
  return plan_call(c);
}

// Replace transposed operands of g by row-major copies in the workspace of
// the call's stream: op(A) as M x K (ld K), op(B) as K x N (ld N).
int make_row_major(GemmArgs& g, Lease& ls) {
  const cudaStream_t s = ls.stream();
  if (!g.op_a && !g.op_b) return SGEMM_OK;
  const size_t a_floats = g.op_a ? size_t(g.M) * size_t(g.K) : 0;
  const size_t a_pad = (a_floats + 63) / 64 * 64;  // B copy 256-byte aligned
  const size_t b_floats = g.op_b ? size_t(g.K) * size_t(g.N) : 0;
  Workspace* w = nullptr;
  int rc = ensure_tr(ls, a_pad + b_floats, &w);
  if (rc != SGEMM_OK) return rc;
  if (g.op_a) {  // A stored K x M -> M x K
    rc = to_status(launch_transpose(g.A, g.lda, g.K, g.M, w->tr, s));
    if (rc != SGEMM_OK) return rc;
    g.A = w->tr;
    g.lda = g.K > 1 ? g.K : 1;
    g.op_a = 0;
  }
  if (g.op_b) {  // B stored N x K -> K x N
    rc = to_status(launch_transpose(g.B, g.ldb, g.N, g.K, w->tr + a_pad, s));
    if (rc != SGEMM_OK) return rc;
    g.B = w->tr + a_pad;
    g.ldb = g.N > 1 ? g.N : 1;
    g.op_b = 0;
  }
  return SGEMM_OK;
}

// Give the tensor maps operands they can take: each operand whose base or
// row stride is not 16-byte aligned is copied (as stored, op unchanged)
// into the workspace of the call's stream with its row stride rounded up to
// 4 floats.
int make_tensor_ready(GemmArgs& g, Lease& ls) {
  const cudaStream_t s = ls.stream();
  const bool a_ok = tma_operand_ok(reinterpret_cast<uint64_t>(g.A), g.lda);
  const bool b_ok = tma_operand_ok(reinterpret_cast<uint64_t>(g.B), g.ldb);
  if (a_ok && b_ok) return SGEMM_OK;
  const int64_t ar = g.op_a ? g.K : g.M, ac = g.op_a ? g.M : g.K;
  const int64_t br = g.op_b ? g.N : g.K, bc = g.op_b ? g.K : g.N;
  const int64_t ald = (ac + 3) / 4 * 4, bld = (bc + 3) / 4 * 4;
  const size_t a_floats = a_ok ? 0 : (size_t(ar) * size_t(ald) + 63) / 64 * 64;
  const size_t b_floats = b_ok ? 0 : size_t(br) * size_t(bld);
  Workspace* w = nullptr;
  int rc = ensure_tr(ls, a_floats + b_floats, &w);
  if (rc != SGEMM_OK) return rc;
  if (!a_ok) {
    rc = to_status(launch_repack(g.A, g.lda, ar, ac, w->tr, ald, s));
    if (rc != SGEMM_OK) return rc;
    g.A = w->tr;
    g.lda = ald;
  }
  if (!b_ok) {
    rc = to_status(launch_repack(g.B, g.ldb, br, bc, w->tr + a_floats, bld,
                                 s));
    if (rc != SGEMM_OK) return rc;
    g.B = w->tr + a_floats;
    g.ldb = bld;
  }
  return SGEMM_OK;
}

int run_call(const Call& call, void* stream, int path) {
  int rc = check_call(call);
  if (rc != SGEMM_OK) return rc;
  if (path < 0 || path >= SGEMM_PATH_COUNT) return SGEMM_ERR_INVALID_VALUE;
  if (call.M == 0 || call.N == 0) return SGEMM_OK;
  if (call_overlaps(call)) return SGEMM_ERR_OVERLAP;

  DeviceState* st = nullptr;
  rc = device_state(&st);
  if (rc != SGEMM_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  if (!reads_ab(call)) {  // empty sum or alpha == 0: C = beta * C
    if (call.beta == 1.f) return SGEMM_OK;
    if (call.beta == 0.f)
      return to_status(cudaMemset2DAsync(call.C, size_t(call.ldc) * 4, 0,
                                         size_t(call.N) * 4, size_t(call.M),
                                         s));
    return to_status(
        launch_scale_c(call.C, call.ldc, call.M, call.N, call.beta, s));
  }

  const bool chosen = path == SGEMM_PATH_AUTO;
  if (chosen) path = plan_call(call);
  GemmArgs g{call.M,   call.N, call.K,   call.A, call.lda,
             call.B,   call.ldb, call.C, call.ldc};
  g.sc.alpha = call.alpha;
  g.sc.beta = call.beta;
  g.op_a = call.op_a;
  g.op_b = call.op_b;
  Lease lease(*st, s);  // the workspace of stream s
  switch (path) {
    case SGEMM_PATH_TF32X3:
    case SGEMM_PATH_TF32X3_PAIR:
      rc = make_tensor_ready(g, lease);
      if (rc != SGEMM_OK) return rc;
      return run_tf32x3(g, *st, s, path == SGEMM_PATH_TF32X3_PAIR, &lease);
    case SGEMM_PATH_GEMV_COL: {
      if (call.M == 1 && call.N != 1 && call.op_b) {
        // c = op(a) * B^T: row j of B (stored N x K) times the vector a
        // (A's row, or its column with stride lda when stored K x 1).
        GemmArgs h{call.N, 1, call.K, call.B, call.ldb, call.A,
                   call.op_a ? call.lda : 1, call.C, 1};
        h.sc = g.sc;
        const cudaError_t e = run_gemv_col(h, *st, s, &rc);
        return rc != SGEMM_OK ? rc : to_status(e);
      }
      if (call.N != 1) return SGEMM_ERR_PATH;
      if (g.op_a) {
        g.op_b = 0;  // B's column is read with its own stride below
        g.op_a = 1;
        rc = make_row_major(g, lease);
        if (rc != SGEMM_OK) return rc;
      }
      // the vector b = op(B)'s column: stride ldb (stored K x 1) or 1
      g.ldb = call.op_b ? 1 : call.ldb;
      g.op_b = 0;
      const cudaError_t e = run_gemv_col(g, *st, s, &rc);
      return rc != SGEMM_OK ? rc : to_status(e);
    }
    case SGEMM_PATH_GEMV_ROW: {
      if (call.M != 1 && gemv_col_as_row(call)) {
        // c^T (1 x M) = b^T (1 x K) * A_stored (K x M, row pitch lda)
        GemmArgs h{1, call.M, call.K, call.B, std::max<int64_t>(call.K, 1),
                   call.A, call.lda, call.C, std::max<int64_t>(call.M, 1)};
        h.sc = g.sc;
        const cudaError_t e = run_gemv_row(h, *st, s, &rc);
        return rc != SGEMM_OK ? rc : to_status(e);
      }
      if (call.M != 1) return SGEMM_ERR_PATH;
      rc = make_row_major(g, lease);
      if (rc != SGEMM_OK) return rc;
      const cudaError_t e = run_gemv_row(g, *st, s, &rc);
      return rc != SGEMM_OK ? rc : to_status(e);
    }
    case SGEMM_PATH_TILED_TMA: {
      rc = make_row_major(g, lease);
      if (rc != SGEMM_OK) return rc;
      if (!tma_operand_ok(reinterpret_cast<uint64_t>(g.A), g.lda) ||
          !tma_operand_ok(reinterpret_cast<uint64_t>(g.B), g.ldb)) {
        // Only the library's own choice repacks (plan_call picks this path
        // for misaligned operands only when neither is transposed, so the
        // workspace copy below is the only one); a forced path on layouts
        // TMA cannot map is refused.
        if (!chosen || call.op_a || call.op_b) return SGEMM_ERR_PATH;
        rc = make_tensor_ready(g, lease);
        if (rc != SGEMM_OK) return rc;
      }
      if (plan_stream_k(g.M, g.N, g.K, 1).total_iters >= (1ll << 31))
        return SGEMM_ERR_TOO_LARGE;
      CUtensorMap tmA, tmB;
      rc = encode_maps(g, &tmA, &tmB);
      if (rc != SGEMM_OK) return rc;
      const SkPlan pl =
          plan_stream_k(g.M, g.N, g.K, st->sms * st->tma_blocks_per_sm);
      Workspace* w = nullptr;
      rc = ensure_workspace(lease, pl.ws_floats, pl.counters, &w);
      if (rc != SGEMM_OK) return rc;
      return to_status(launch_tiled_tma(g, tmA, tmB, pl, w->ws, w->counters,
                                        st->status, s));
    }
    case SGEMM_PATH_TILED_LDG:
      rc = make_row_major(g, lease);
      if (rc != SGEMM_OK) return rc;
      return to_status(launch_tiled_ldg(g, st->status, s));
    case SGEMM_PATH_NAIVE:
      rc = make_row_major(g, lease);
      if (rc != SGEMM_OK) return rc;
      return to_status(launch_naive(g, s));
    case SGEMM_PATH_SMALL:
      if (call.M > kSmallMaxRows) return SGEMM_ERR_PATH;
      rc = make_row_major(g, lease);
      if (rc != SGEMM_OK) return rc;
      return to_status(launch_small(g, s));
    default:
      return SGEMM_ERR_PATH;
  }
}

int run(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
        const float* B, int64_t ldb, float* C, int64_t ldc, void* stream,
        int path) {
  const Call c{SGEMM_OP_N, SGEMM_OP_N, M, N, K, 1.f, A, lda, B, ldb, 0.f,
               C, ldc};
  return run_call(c, stream, path);
}

// ---------------------------------------------------------------- batches
//
// Item b: C_b = alpha * op(A_b) * op(B_b) + beta * C_b with X_b = X + b *
// stride_x (stride 0: one operand shared by every item). The tensor-core
// kernels take the whole batch in one launch (3-D tensor maps, tiles of all
// items in one persistent schedule); every other path runs item by item.
int run_batched(const Call& c, int64_t stride_a, int64_t stride_b,
                int64_t stride_c, int64_t batch, void* stream, int path) {
  int rc = check_call(c);
  if (rc != SGEMM_OK) return rc;
  if (path < 0 || path >= SGEMM_PATH_COUNT) return SGEMM_ERR_INVALID_VALUE;
  if (batch < 0 || stride_a < 0 || stride_b < 0 || stride_c < 0)
    return SGEMM_ERR_INVALID_VALUE;
  if (batch == 0 || c.M == 0 || c.N == 0) return SGEMM_OK;
  if (batch == 1) return run_call(c, stream, path);
  // Items of C must not share memory: stacked (each item past the previous
  // one's last element) or side by side inside one row pitch.
  const bool stacked = stride_c >= (c.M - 1) * c.ldc + c.N;
  const bool side_by_side =
      stride_c >= c.N && (batch - 1) * stride_c + c.N <= c.ldc;
  if (!stacked && !side_by_side) return SGEMM_ERR_INVALID_VALUE;
  if (batch > kMaxDim) return SGEMM_ERR_TOO_LARGE;
  if (reads_ab(c)) {  // C (all items) against A and B (all items)
    const uint64_t cc = reinterpret_cast<uint64_t>(c.C);
    const uint64_t c_hi =
        cc + uint64_t(((batch - 1) * stride_c + (c.M - 1) * c.ldc + c.N) * 4);
    auto hits = [&](const float* x, int64_t rows, int64_t cols, int64_t ld,
                    int64_t stride) {
      const uint64_t lo = reinterpret_cast<uint64_t>(x);
      const uint64_t hi =
          lo + uint64_t(((batch - 1) * stride + (rows - 1) * ld + cols) * 4);
      return lo < c_hi && cc < hi;
    };
    if (hits(c.A, c.op_a ? c.K : c.M, c.op_a ? c.M : c.K, c.lda, stride_a) ||
        hits(c.B, c.op_b ? c.N : c.K, c.op_b ? c.K : c.N, c.ldb, stride_b))
      return SGEMM_ERR_OVERLAP;
  }
  const bool strides_ok = stride_a % 4 == 0 && stride_b % 4 == 0;
  const int64_t tiles = ((c.M + kTileM - 1) / kTileM) *
                        ((c.N + kTileN - 1) / kTileN);
  const bool tensor_ok =
      reads_ab(c) && strides_ok &&
      tma_operand_ok(reinterpret_cast<uint64_t>(c.A), c.lda) &&
      tma_operand_ok(reinterpret_cast<uint64_t>(c.B), c.ldb) &&
      batch * tiles < (int64_t(1) << 31);
  if (path == SGEMM_PATH_AUTO && tensor_ok &&
      g_math_mode.load(std::memory_order_relaxed) == SGEMM_MATH_AUTO &&
      c.M > 1 && c.N > 1)
    path = use_pair(c.M, c.N, c.K, batch) ? SGEMM_PATH_TF32X3_PAIR
                                          : SGEMM_PATH_TF32X3;
  // One launch for the batch on the tensor path; a forced tensor path on
  // operands it cannot map whole (misaligned rows or strides) runs item by
  // item below, where each item is repacked like a single call.
  if (reads_ab(c) && tensor_ok &&
      (path == SGEMM_PATH_TF32X3 || path == SGEMM_PATH_TF32X3_PAIR)) {
    DeviceState* st = nullptr;
    rc = device_state(&st);
    if (rc != SGEMM_OK) return rc;
    GemmArgs g{c.M, c.N, c.K, c.A, c.lda, c.B, c.ldb, c.C, c.ldc};
    g.sc.alpha = c.alpha;
    g.sc.beta = c.beta;
    g.op_a = c.op_a;
    g.op_b = c.op_b;
    g.batch = batch;
    g.stride_a = stride_a;
    g.stride_b = stride_b;
    g.stride_c = stride_c;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    {
      Lease lease(*st, s);
      rc = run_tf32x3(g, *st, s, path == SGEMM_PATH_TF32X3_PAIR, &lease);
    }
    // a batch layout the tensor-map encoder refuses runs item by item
    if (rc != SGEMM_ERR_CUDA) return rc;
    path = SGEMM_PATH_AUTO;
  }
  for (int64_t b = 0; b < batch; ++b) {
    Call item = c;
    item.A = c.A + b * stride_a;
    item.B = c.B + b * stride_b;
    item.C = c.C + b * stride_c;
    rc = run_call(item, stream, path);
    if (rc != SGEMM_OK) return rc;
  }
  return SGEMM_OK;
}

}  // namespace

int run_with_scratch(int64_t M, int64_t N, int64_t K, const float* A,
                     int64_t lda, const float* B, int64_t ldb, float* C,
                     int64_t ldc, void* stream, float* ws, size_t ws_floats,
                     int* counters, size_t counters_len, int grid_cap) {
  int rc = check_args(M, N, K, A, lda, B, ldb, C, ldc);
  if (rc != SGEMM_OK) return rc;
  if (M == 0 || N == 0) return SGEMM_OK;
  const uint64_t a = reinterpret_cast<uint64_t>(A);
  const uint64_t b = reinterpret_cast<uint64_t>(B);
  const uint64_t c = reinterpret_cast<uint64_t>(C);
  if (K > 0 && (overlaps(a, M, K, lda, c, M, N, ldc) ||
                overlaps(b, K, N, ldb, c, M, N, ldc)))
    return SGEMM_ERR_OVERLAP;
  DeviceState* st = nullptr;
  rc = device_state(&st);
  if (rc != SGEMM_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (K == 0)
    return to_status(cudaMemset2DAsync(C, size_t(ldc) * 4, 0, size_t(N) * 4,
                                       size_t(M), s));
  int path = plan_path(M, N, K, lda, ldb, a, b);
  // The tensor paths and the TMA tile kernel take misaligned operands
  // through a repacked copy, which needs device memory: here such operands
  // go to the any-layout tile kernel instead.
  if ((path == SGEMM_PATH_TF32X3 || path == SGEMM_PATH_TF32X3_PAIR ||
       path == SGEMM_PATH_TILED_TMA) &&
      !(tma_operand_ok(a, lda) && tma_operand_ok(b, ldb)))
    path = SGEMM_PATH_TILED_LDG;
  const GemmArgs g{M, N, K, A, lda, B, ldb, C, ldc};
  switch (path) {
    case SGEMM_PATH_TILED_TMA: {
      CUtensorMap tmA, tmB;
      rc = encode_maps(g, &tmA, &tmB);
      if (rc != SGEMM_OK) return rc;
      int resident = st->sms * st->tma_blocks_per_sm;
      if (resident > grid_cap) resident = grid_cap;
      const SkPlan pl = plan_stream_k(M, N, K, resident);
      // The documented limit: counters for every tile (whatever part of
      // them this schedule splits), before anything is enqueued.
      if (pl.ws_floats > ws_floats ||
          size_t(pl.tiles) * kWarpsPerTile > counters_len ||
          pl.counters > counters_len)
        return SGEMM_ERR_TOO_LARGE;
      rc = to_status(
          cudaMemsetAsync(counters, 0, pl.counters * sizeof(int), s));
      if (rc != SGEMM_OK) return rc;
      return to_status(
          launch_tiled_tma(g, tmA, tmB, pl, ws, counters, st->status, s));
    }
    case SGEMM_PATH_TILED_LDG:
      return to_status(launch_tiled_ldg(g, st->status, s));
    case SGEMM_PATH_SMALL:
      return to_status(launch_small(g, s));
    case SGEMM_PATH_TF32X3:
      return run_tf32x3(g, *st, s, false, nullptr);
    case SGEMM_PATH_TF32X3_PAIR: {
      CUtensorMap tmA, tmB;
      rc = encode_tf32x3(g, &tmA, &tmB);
      if (rc != SGEMM_OK) return rc;
      // stream-K tail only when its workspace fits in the scratch
      PairPlan pl = plan_pair(M, N, K, st->pair_clusters, true);
      if (pl.ws_floats > ws_floats || pl.counters > counters_len)
        pl = plan_pair(M, N, K, st->pair_clusters, false);
      if (pl.counters > 0) {
        rc = to_status(
            cudaMemsetAsync(counters, 0, pl.counters * sizeof(int), s));
        if (rc != SGEMM_OK) return rc;
      }
      return to_status(launch_tf32x3_pair(g, tmA, tmB, nullptr, pl, ws,
                                          counters, st->status, s));
    }
    case SGEMM_PATH_GEMV_ROW: {
      const cudaError_t e = run_gemv_row(g, *st, s, &rc);
      return rc != SGEMM_OK ? rc : to_status(e);
    }
    case SGEMM_PATH_GEMV_COL: {
      const cudaError_t e = run_gemv_col(g, *st, s, &rc);
      return rc != SGEMM_OK ? rc : to_status(e);
    }
    default:
      return SGEMM_ERR_PATH;
  }
}

// ---------------------------------------------------------------- host I/O
//
// sgemm_host for large products: the copies over the host link take longer
// than the product itself, so they are overlapped with it. B goes first
// (every row block of C needs all of it), then A in row blocks on a copy
// stream; each row block of C is computed on the caller's stream as soon as
// its rows of A have landed and is copied back on a second copy stream while
// the next block computes. The copy streams are ordered after the caller's
// earlier work by an event and the caller's stream waits for the last copy,
// so the call stays asynchronous on `stream` with the same ordering as the
// single-pass version.
constexpr int kHostMaxChunks = 4;
constexpr int64_t kHostChunkRows = 256;          // a pair tile's height

struct HostPipe {
  std::once_flag once;
  int err = SGEMM_OK;
  std::mutex mu;  // one call's enqueue sequence at a time (shared events)
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, b_ready = nullptr, done = nullptr;
  cudaEvent_t a_ready[kHostMaxChunks] = {}, c_ready[kHostMaxChunks] = {};
};
HostPipe g_pipe[kMaxDevices];

// Row blocks for a product: one (no pipelining) below about 2^31
// multiply-adds or 512 rows, else up to 4 blocks of whole 256-row tiles.
int host_chunks(int64_t M, int64_t N, int64_t K) {
  if (K == 0 || M < 2 * kHostChunkRows ||
      double(M) * double(N) * double(K) < double(int64_t(1) << 31))
    return 1;
  const int64_t tiles = M / kHostChunkRows;
  return int(tiles < kHostMaxChunks ? tiles : kHostMaxChunks);
}

int host_pipe(HostPipe** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SGEMM_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SGEMM_ERR_UNSUPPORTED_DEVICE;
  HostPipe& hp = g_pipe[dev];
  std::call_once(hp.once, [&] {
    bool ok =
        cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking) ==
            cudaSuccess &&
        cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking) ==
            cudaSuccess &&
        cudaEventCreateWithFlags(&hp.start, cudaEventDisableTiming) ==
            cudaSuccess &&
        cudaEventCreateWithFlags(&hp.b_ready, cudaEventDisableTiming) ==
            cudaSuccess &&
        cudaEventCreateWithFlags(&hp.done, cudaEventDisableTiming) ==
            cudaSuccess;
    for (int i = 0; ok && i < kHostMaxChunks; ++i)
      ok = cudaEventCreateWithFlags(&hp.a_ready[i], cudaEventDisableTiming) ==
               cudaSuccess &&
           cudaEventCreateWithFlags(&hp.c_ready[i], cudaEventDisableTiming) ==
               cudaSuccess;
    hp.err = ok ? SGEMM_OK : SGEMM_ERR_CUDA;
  });
  *out = &hp;
  return hp.err;
}

int host_pipelined(int64_t M, int64_t N, int64_t K, const float* hA,
                   int64_t lda, const float* hB, int64_t ldb, float* hC,
                   int64_t ldc, float* dA, float* dB, float* dC,
                   cudaStream_t s, int chunks) {
  HostPipe* hp = nullptr;
  int rc = host_pipe(&hp);
  if (rc != SGEMM_OK) return rc;
  std::lock_guard<std::mutex> lock(hp->mu);
  // row blocks on 256-row boundaries
  int64_t r[kHostMaxChunks + 1];
  const int64_t tiles = (M + kHostChunkRows - 1) / kHostChunkRows;
  for (int i = 0; i <= chunks; ++i)
    r[i] = i == chunks ? M : (tiles * i / chunks) * kHostChunkRows;
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  if (!ok(cudaEventRecord(hp->start, s)) ||
      !ok(cudaStreamWaitEvent(hp->h2d, hp->start, 0)) ||
      !ok(cudaStreamWaitEvent(hp->d2h, hp->start, 0)) ||
      !ok(cudaMemcpy2DAsync(dB, size_t(N) * 4, hB, size_t(ldb) * 4,
                            size_t(N) * 4, size_t(K), cudaMemcpyHostToDevice,
                            hp->h2d)) ||
      !ok(cudaEventRecord(hp->b_ready, hp->h2d)))
    return SGEMM_ERR_CUDA;
  for (int i = 0; i < chunks; ++i) {
    const int64_t rows = r[i + 1] - r[i];
    if (!ok(cudaMemcpy2DAsync(dA + r[i] * K, size_t(K) * 4, hA + r[i] * lda,
                              size_t(lda) * 4, size_t(K) * 4, size_t(rows),
                              cudaMemcpyHostToDevice, hp->h2d)) ||
        !ok(cudaEventRecord(hp->a_ready[i], hp->h2d)))
      return SGEMM_ERR_CUDA;
  }
  if (!ok(cudaStreamWaitEvent(s, hp->b_ready, 0))) return SGEMM_ERR_CUDA;
  for (int i = 0; i < chunks; ++i) {
    const int64_t rows = r[i + 1] - r[i];
    if (!ok(cudaStreamWaitEvent(s, hp->a_ready[i], 0))) return SGEMM_ERR_CUDA;
    rc = run(rows, N, K, dA + r[i] * K, K, dB, N, dC + r[i] * N, N, s,
             SGEMM_PATH_AUTO);
    if (rc != SGEMM_OK) return rc;
    if (!ok(cudaEventRecord(hp->c_ready[i], s)) ||
        !ok(cudaStreamWaitEvent(hp->d2h, hp->c_ready[i], 0)) ||
        !ok(cudaMemcpy2DAsync(hC + r[i] * ldc, size_t(ldc) * 4, dC + r[i] * N,
                              size_t(N) * 4, size_t(N) * 4, size_t(rows),
                              cudaMemcpyDeviceToHost, hp->d2h)))
      return SGEMM_ERR_CUDA;
  }
  if (!ok(cudaEventRecord(hp->done, hp->d2h)) ||
      !ok(cudaStreamWaitEvent(s, hp->done, 0)))
    return SGEMM_ERR_CUDA;
  return SGEMM_OK;
}

}  // namespace dfm

extern "C" {

int sgemm(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
          const float* B, int64_t ldb, float* C, int64_t ldc, void* stream) {
  return dfm::run(M, N, K, A, lda, B, ldb, C, ldc, stream, SGEMM_PATH_AUTO);
}

int sgemm_path(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda,
               const float* B, int64_t ldb, float* C, int64_t ldc,
               void* stream, int path) {
  return dfm::run(M, N, K, A, lda, B, ldb, C, ldc, stream, path);
}

int sgemm_ex(int op_a, int op_b, int64_t M, int64_t N, int64_t K,
             float alpha, const float* A, int64_t lda, const float* B,
             int64_t ldb, float beta, float* C, int64_t ldc, void* stream) {
  const dfm::Call c{op_a, op_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc};
  return dfm::run_call(c, stream, SGEMM_PATH_AUTO);
}

int sgemm_ex_path(int op_a, int op_b, int64_t M, int64_t N, int64_t K,
                  float alpha, const float* A, int64_t lda, const float* B,
                  int64_t ldb, float beta, float* C, int64_t ldc, void* stream,
                  int path) {
  const dfm::Call c{op_a, op_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc};
  return dfm::run_call(c, stream, path);
}

int sgemm_plan_ex(int op_a, int op_b, int64_t M, int64_t N, int64_t K,
                  int64_t lda, int64_t ldb, int64_t ldc, uint64_t a_addr,
                  uint64_t b_addr, uint64_t c_addr, int* path) {
  if (path == nullptr) return SGEMM_ERR_NULL_POINTER;
  const dfm::Call c{op_a, op_b, M, N, K, 1.f,
                    reinterpret_cast<const float*>(a_addr), lda,
                    reinterpret_cast<const float*>(b_addr), ldb, 0.f,
                    reinterpret_cast<float*>(c_addr), ldc};
  const int rc = dfm::check_call(c);
  if (rc != SGEMM_OK) return rc;
  *path = dfm::plan_call(c);
  return SGEMM_OK;
}

int sgemm_strided_batched(int op_a, int op_b, int64_t M, int64_t N,
                          int64_t K, float alpha, const float* A, int64_t lda,
                          int64_t stride_a, const float* B, int64_t ldb,
                          int64_t stride_b, float beta, float* C, int64_t ldc,
                          int64_t stride_c, int64_t batch, void* stream) {
  const dfm::Call c{op_a, op_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc};
  return dfm::run_batched(c, stride_a, stride_b, stride_c, batch, stream,
                          SGEMM_PATH_AUTO);
}

int sgemm_strided_batched_path(int op_a, int op_b, int64_t M, int64_t N,
                               int64_t K, float alpha, const float* A,
                               int64_t lda, int64_t stride_a, const float* B,
                               int64_t ldb, int64_t stride_b, float beta,
                               float* C, int64_t ldc, int64_t stride_c,
                               int64_t batch, void* stream, int path) {
  const dfm::Call c{op_a, op_b, M, N, K, alpha, A, lda, B, ldb, beta, C, ldc};
  return dfm::run_batched(c, stride_a, stride_b, stride_c, batch, stream,
                          path);
}

int sgemm_set_math_mode(int mode) {
  if (mode != SGEMM_MATH_AUTO && mode != SGEMM_MATH_FFMA)
    return SGEMM_ERR_INVALID_VALUE;
  return dfm::g_math_mode.exchange(mode);
}

int sgemm_plan(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
               int64_t ldc, uint64_t a_addr, uint64_t b_addr, uint64_t c_addr,
               int* path) {
  if (path == nullptr) return SGEMM_ERR_NULL_POINTER;
  // Pointer values stand in for the matrices: a zero address with elements
  // to touch is a null-pointer error, as in sgemm.
  const int rc = dfm::check_args(M, N, K, reinterpret_cast<const void*>(a_addr),
                                 lda, reinterpret_cast<const void*>(b_addr),
                                 ldb, reinterpret_cast<const void*>(c_addr), ldc);
  if (rc != SGEMM_OK) return rc;
  *path = dfm::plan_path(M, N, K, lda, ldb, a_addr, b_addr);
  return SGEMM_OK;
}

int sgemm_host(int64_t M, int64_t N, int64_t K, const float* hA, int64_t lda,
               const float* hB, int64_t ldb, float* hC, int64_t ldc,
               float* dA, float* dB, float* dC, void* stream) {
  int rc = dfm::check_args(M, N, K, hA, lda, hB, ldb, hC, ldc);
  if (rc != SGEMM_OK) return rc;
  if (M == 0 || N == 0) return SGEMM_OK;
  if (dC == nullptr || (K > 0 && (dA == nullptr || dB == nullptr)))
    return SGEMM_ERR_NULL_POINTER;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int chunks = dfm::host_chunks(M, N, K);
  if (chunks > 1) return dfm::host_pipelined(M, N, K, hA, lda, hB, ldb, hC,
                                             ldc, dA, dB, dC, s, chunks);
  if (K > 0) {
    if (cudaMemcpy2DAsync(dA, size_t(K) * 4, hA, size_t(lda) * 4,
                          size_t(K) * 4, size_t(M), cudaMemcpyHostToDevice,
                          s) != cudaSuccess ||
        cudaMemcpy2DAsync(dB, size_t(N) * 4, hB, size_t(ldb) * 4,
                          size_t(N) * 4, size_t(K), cudaMemcpyHostToDevice,
                          s) != cudaSuccess)
      return SGEMM_ERR_CUDA;
  }
  rc = sgemm(M, N, K, dA, K > 0 ? K : 1, dB, N, dC, N, stream);
  if (rc != SGEMM_OK) return rc;
  if (cudaMemcpy2DAsync(hC, size_t(ldc) * 4, dC, size_t(N) * 4, size_t(N) * 4,
                        size_t(M), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return SGEMM_ERR_CUDA;
  return SGEMM_OK;
}

int sgemm_watchdog_status(int* site) {
  dfm::DeviceState* st = nullptr;
  const int rc = dfm::device_state(&st);
  if (rc != SGEMM_OK) return rc;
  int word[4] = {0, 0, 0, 0};
  if (cudaMemcpy(word, st->status, sizeof(word), cudaMemcpyDeviceToHost) !=
          cudaSuccess ||
      cudaMemset(st->status, 0, sizeof(word)) != cudaSuccess)
    return SGEMM_ERR_CUDA;
  if (word[0] == 0) return SGEMM_OK;
  if (site != nullptr) *site = word[1];
  // A block that abandoned its range may have left stream-K tile counters
  // raised; clear them so later calls start from zero.
  {
    std::lock_guard<std::mutex> lock(st->ws_mu);
    for (auto& w : st->pool)
      if (w->counters != nullptr &&
          cudaMemset(w->counters, 0, w->counters_len * sizeof(int)) !=
              cudaSuccess)
        return SGEMM_ERR_CUDA;
  }
  return SGEMM_ERR_WATCHDOG;
}

int sgemm_workspace_info(int* count, int64_t* bytes) {
  dfm::DeviceState* st = nullptr;
  const int rc = dfm::device_state(&st);
  if (rc != SGEMM_OK) return rc;
  std::lock_guard<std::mutex> lock(st->ws_mu);
  int64_t total = 0;
  for (auto& w : st->pool) total += int64_t(w->bytes());
  if (count != nullptr) *count = int(st->pool.size());
  if (bytes != nullptr) *bytes = total;
  return SGEMM_OK;
}

int sgemm_watchdog_selftest(void* stream, int64_t timeout_ns) {
  dfm::DeviceState* st = nullptr;
  int rc = dfm::device_state(&st);
  if (rc != SGEMM_OK) return rc;
  if (timeout_ns < 1000000) timeout_ns = 1000000;
  if (timeout_ns > 2000000000) timeout_ns = 2000000000;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (dfm::launch_watchdog_selftest(st->status, uint64_t(timeout_ns), s) !=
      cudaSuccess)
    return SGEMM_ERR_LAUNCH;
  if (cudaStreamSynchronize(s) != cudaSuccess) return SGEMM_ERR_CUDA;
  return sgemm_watchdog_status(nullptr);
}

const char* sgemm_status_string(int status) {
  switch (status) {
    case SGEMM_OK: return "ok";
    case SGEMM_ERR_INVALID_VALUE: return "invalid value";
    case SGEMM_ERR_NULL_POINTER: return "null pointer";
    case SGEMM_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs sm_103)";
    case SGEMM_ERR_LAUNCH: return "kernel launch failed";
    case SGEMM_ERR_WATCHDOG: return "device wait timed out";
    case SGEMM_ERR_OVERLAP: return "C overlaps A or B";
    case SGEMM_ERR_CUDA: return "CUDA runtime error";
    case SGEMM_ERR_PATH: return "path cannot take these arguments";
    case SGEMM_ERR_TOO_LARGE: return "size beyond the supported range";
    default: return "unknown status";
  }
}

const char* sgemm_path_name(int path) {
  switch (path) {
    case SGEMM_PATH_AUTO: return "auto";
    case SGEMM_PATH_TILED_TMA: return "tiled_tma";
    case SGEMM_PATH_TILED_LDG: return "tiled_ldg";
    case SGEMM_PATH_GEMV_ROW: return "gemv_row";
    case SGEMM_PATH_GEMV_COL: return "gemv_col";
    case SGEMM_PATH_NAIVE: return "naive";
    case SGEMM_PATH_SMALL: return "small";
    case SGEMM_PATH_TF32X3: return "tf32x3";
    case SGEMM_PATH_TF32X3_PAIR: return "tf32x3_pair";
    default: return "?";
  }
}

int sgemm_version(void) { return 100; }

uint64_t sgemm_launch_count(void) {
  return dfm::g_launches.load(std::memory_order_relaxed);
}

}  // extern "C"
