// sgemm_noalloc: the matrix product without any device allocation.
//
// Who needs it: callers that may not call cudaMalloc at the point of use,
// e.g. code running under an allocator that owns all device memory (a
// framework's caching pool or a fixed memory budget), code that must not
// trigger the implicit device synchronisation of cudaMalloc/cudaFree in a
// latency-critical loop, or plug-ins loaded into a host that forbids
// allocation after start-up. sgemm() may grow its stream's workspace with
// cudaMalloc on a call whose shape needs more; this entry point never does.
//
// How: the stream-K partial tiles and tile counters of the TMA path live in
// one file-scope __device__ array of fixed size, present on every device
// that loads the library until the process exits. Host code cannot use the
// array's name as a device address, so the address is fetched once per
// device with cudaGetSymbolAddress, on the first call made with that device
// current. Every call shares the array: calls whose kernels overlap on the
// GPU (different streams, no ordering) race on it. The counters a call uses
// are cleared on its stream before its kernel runs; the partial tiles need
// no clearing (every slot read in a call was written earlier in that call).
#include <cuda_runtime.h>

#include <mutex>

#include "dfm_sgemm.h"
#include "kernels.h"

namespace dfm {
namespace {

// Largest stream-K grid the scratch serves (GB300 has 152 SMs and the
// kernel runs one block per SM; more resident blocks are capped to this).
constexpr int kNoAllocMaxBlocks = 160;
// Partial tiles: two 256 x 128 fp32 tiles per block (40 MiB).
constexpr size_t kNoAllocPartialFloats =
    size_t(2) * kNoAllocMaxBlocks * kTileM * kTileN;
// Tile counters: stream-K products with at most this many 256 x 128 output
// tiles (for example M = 32768, N = 16384).
constexpr size_t kNoAllocMaxTiles = 16384;
// The fix-up counts pieces per (tile, warp of the block).
constexpr size_t kNoAllocCounters = kNoAllocMaxTiles * kWarpsPerTile;
constexpr size_t kNoAllocBytes =
    kNoAllocPartialFloats * sizeof(float) + kNoAllocCounters * sizeof(int);

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

constexpr int kMaxDevices = 64;
struct ScratchAddr {
  std::once_flag once;
  cudaError_t err = cudaSuccess;
  unsigned char* base = nullptr;
};
ScratchAddr g_addr[kMaxDevices];

}  // namespace
}  // namespace dfm

extern "C" int sgemm_noalloc(int64_t M, int64_t N, int64_t K, const float* A,
                             int64_t lda, const float* B, int64_t ldb,
                             float* C, int64_t ldc, void* stream) {
  using namespace dfm;
  // The tile limit applies where the scratch is used (the stream-K tile
  // kernel): run_with_scratch rejects such a product before it enqueues
  // anything; paths without scratch take any size sgemm takes.
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SGEMM_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SGEMM_ERR_UNSUPPORTED_DEVICE;
  ScratchAddr& sa = g_addr[dev];
  std::call_once(sa.once, [&] {
    void* p = nullptr;
    sa.err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    sa.base = static_cast<unsigned char*>(p);
  });
  if (sa.err != cudaSuccess || sa.base == nullptr) return SGEMM_ERR_CUDA;
  float* partials = reinterpret_cast<float*>(sa.base);
  int* counters = reinterpret_cast<int*>(
      sa.base + kNoAllocPartialFloats * sizeof(float));
  return run_with_scratch(M, N, K, A, lda, B, ldb, C, ldc, stream, partials,
                          kNoAllocPartialFloats, counters, kNoAllocCounters,
                          kNoAllocMaxBlocks);
}
