// noalloc.cu -- the fused RMSNorm -> GEMM layer for callers that cannot
// allocate device memory.
//
// bi_rmsnorm_gemm_bf16 keeps each row's RMSNorm scale r (one fp32 value per
// row), and for large batches the normalised rows, in a workspace that the
// caller allocates.  Some callers cannot allocate: a plugin running inside a
// host runtime that reserved the device's memory up front and gives plugins
// no allocator, or code on a latency-critical path where cudaMalloc/cudaFree
// would synchronise the device.  This variant takes only inputs and outputs
// and keeps the same data in the static array below instead; where the
// normalised rows would not fit, it normalises them in shared memory (the
// same bits, never staged).
//
// The array is a file-scope __device__ variable: every GPU that loads this
// library's module holds its BI_NOALLOC_SCRATCH_BYTES until the process
// exits.  Host code cannot use the array's name as a device address, so the
// first call on each device (with that device current) looks the address up
// with cudaGetSymbolAddress and caches it; make that first call before any
// stream capture.  The cached address does not survive cudaDeviceReset (the
// module, and with it the array, may be loaded elsewhere afterwards): do not
// call this entry point again in a process that reset the device.  All calls
// on a device share the array and it keeps the last call's contents; nothing
// in it needs to start at zero, because each call writes the values it reads.
// Calls whose work overlaps on the GPU (different streams, or launches racing
// on one device) race on the array.
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

}  // namespace
}  // namespace bi

using namespace bi;

BI_API size_t bi_noalloc_scratch_bytes(void) { return (size_t)BI_NOALLOC_SCRATCH_BYTES; }

BI_API bi_status bi_rmsnorm_gemm_bf16_noalloc(const void* X, const void* g, const void* W, void* Y,
                                              int64_t M, int64_t N, int64_t K, float eps,
                                              const bi_pins* pins, bi_stream_t stream) {
  // Every argument is checked, and the GEMM planned, before anything is launched.
  GemmLaunch L;
  bi_status st = plan_fused(X, g, W, Y, M, N, K, eps, pins, reinterpret_cast<cudaStream_t>(stream), &L);
  if (st != BI_OK || L.M == 0) return st;
  const size_t cap = (size_t)BI_NOALLOC_SCRATCH_BYTES;
  if (fused_r_bytes(M) > cap) return BI_ERR_WORKSPACE;
  // the staged form needs room for the normalised rows; where they would not
  // fit, normalise in shared memory instead (the same bits)
  const bool in_smem = fused_in_smem(L) || fused_workspace_bytes(M, K) > cap;
  void* scratch = scratch_for_current_device();
  if (!scratch) return BI_ERR_CUDA;
  return launch_fused(L, scratch, in_smem);
}
