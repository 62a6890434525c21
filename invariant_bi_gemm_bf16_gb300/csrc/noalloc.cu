// noalloc.cu -- the fused RMSNorm -> GEMM layer for callers that cannot
// allocate device memory.
//
// bi_rmsnorm_gemm_bf16 stages the normalised rows in a workspace that the
// caller allocates.  Some callers cannot allocate: a plugin running inside a
// host runtime that reserved the device's memory up front and gives plugins
// no allocator, or code on a latency-critical path where cudaMalloc/cudaFree
// would synchronise the device.  This variant takes only inputs and outputs
// and stages the normalised rows in the static array below instead.
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library's module holds its BI_NOALLOC_SCRATCH_BYTES until the process
// exits.  Host code cannot use the array's name as a device address, so the
// first call on each device (with that device current) looks the address up
// with cudaGetSymbolAddress and caches it; make that first call before any
// stream capture.  All calls on a device share the array and it keeps the
// last call's contents; nothing in it needs to start at zero, because each
// call overwrites the rows it reads.  Calls whose work overlaps on the GPU
// (different streams, or launches racing on one device) race on the array.
//
// The paper has no counterpart to this entry point.
#include <mutex>

#include <cuda_runtime.h>

#include "internal.h"

#define BI_API extern "C" __attribute__((visibility("default")))

namespace bi {
namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[BI_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// The device address of g_noalloc_scratch on the current device, looked up
// once per device.  Returns nullptr on failure.
void* scratch_for_current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace bi

using namespace bi;

BI_API bi_status bi_rmsnorm_gemm_bf16_noalloc(const void* X, const void* g, const void* W, void* Y,
                                              int64_t M, int64_t N, int64_t K, float eps,
                                              const bi_pins* pins, bi_stream_t stream) {
  // Every argument is checked before anything is launched.
  if (M < 0 || N < 1 || K < 1) return BI_ERR_INVALID_ARG;
  if (!(eps > 0.0f) || !(eps < 3.0e38f)) return BI_ERR_INVALID_ARG;
  if (K % 8 != 0 || K > 65536 || N > 0x7FFFFFFFll || M > 0x7FFFFFFFll) return BI_ERR_UNSUPPORTED_SHAPE;
  bi_pins resolved;
  if (pins) {
    resolved = *pins;
  } else {
    bi_status st = bi_pins_default(N, K, &resolved);
    if (st != BI_OK) return st;
  }
  bi_status st = bi_pins_validate(N, K, &resolved);
  if (st != BI_OK) return st;
  if (M == 0) return BI_OK;
  if (!X || !g || !W || !Y) return BI_ERR_INVALID_ARG;
  if (!aligned16(X) || !aligned16(g) || !aligned16(W) || !aligned16(Y)) return BI_ERR_ALIGNMENT;
  if ((uint64_t)M * (uint64_t)K * 2u > (uint64_t)BI_NOALLOC_SCRATCH_BYTES) return BI_ERR_WORKSPACE;

  void* scratch = scratch_for_current_device();
  if (!scratch) return BI_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (launch_rmsnorm(X, g, scratch, M, K, eps, s) != cudaSuccess) return BI_ERR_CUDA;
  return bi_gemm_bf16(scratch, W, Y, M, N, K, &resolved, stream);
}
