// gemm.cu -- host side of the batch-invariant GEMM: ring depths, shared-memory
// sizes, the plain (bf16 and E4M3) kernel instances, and the device status
// word that bounded waits report to.  The kernel itself is in gemm_kernel.cuh;
// the fused RMSNorm instances are compiled in gemm_fused.cu.
#include "gemm_kernel.cuh"

namespace bi {

// [0]: 0, or a bi_status code set by a kernel that gave up; [2..3]: the
// debug-bounds build's detail word (the first failed index check)
__device__ __align__(8) int g_stall_status[4];

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

int max_w_stages(int x_rows, int x_stages, int kps) {
  const int left = kRingBytes - x_stages * kps * x_stage_bytes(x_rows);
  int w = left / (kps * kWStageBytes);
  return w > kMaxStages ? kMaxStages : w;
}

void choose_stages(int x_rows, int x_box_rows, int w_pin, int kps, int* w_stages, int* x_stages) {
  const int xb = kps * x_stage_bytes(x_rows);
  const int wb = kps * kWStageBytes;
  int xs, w;
  if (x_box_rows <= 64) {
    // Decode: X is a few rows from L2, W streams from HBM -- put the shared
    // memory into W bytes in flight, then give X every stage that costs no W
    // depth (an X slot's round trip -- copy from L2, and in the fused form the
    // normalisation -- is longer than the W stream's time per stage).
    xs = 3;
    w = max_w_stages(x_rows, xs, kps);
    while (xs < 8 && max_w_stages(x_rows, xs + 1, kps) >= w) ++xs;
  } else {
    // Both operands matter: as many balanced stages as fit, then extra W.
    int n = kRingBytes / (wb + xb);
    if (n > kMaxStages) n = kMaxStages;
    xs = n;
    w = max_w_stages(x_rows, xs, kps);
  }
  if (w_pin > 0) {
    w = w_pin;
    int xfit = (kRingBytes - w * wb) / xb;
    if (xs > xfit) xs = xfit;
  }
  *w_stages = w;
  *x_stages = xs;
}

int64_t gemm_smem_bytes(int T, int x_rows, int w_stages, int x_stages, int kps, bool cluster) {
  int64_t ring = (int64_t)kps * ((int64_t)w_stages * kWStageBytes + (int64_t)x_stages * x_stage_bytes(x_rows));
  int64_t part = cluster ? (int64_t)T * kTileN * 4 : 0;
  return 1024 + (ring > part ? ring : part) + kCtlBytes;
}

cudaError_t launch_gemm(const GemmLaunch& L) {
  return L.pair ? launch_p<false, true>(L) : launch_p<false, false>(L);
}

int* device_status_word() {
  // Looked up once per device (the module is loaded once per device and
  // process; a cudaDeviceReset would invalidate the cached address).
  static std::atomic<int*> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  if (dev >= 0 && dev < 64) {
    int* c = cached[dev].load(std::memory_order_acquire);
    if (c) return c;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_stall_status) != cudaSuccess) return nullptr;
  if (dev >= 0 && dev < 64) cached[dev].store(static_cast<int*>(p), std::memory_order_release);
  return static_cast<int*>(p);
}

cudaError_t fetch_and_clear_stall(int* host_dst, cudaStream_t stream) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(host_dst, g_stall_status, sizeof(int), 0,
                                            cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  const int zero = 0;
  e = cudaMemcpyToSymbolAsync(g_stall_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(stream);
}

cudaError_t fetch_and_clear_bounds_detail(uint64_t* host_dst, cudaStream_t stream) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(host_dst, g_stall_status, sizeof(uint64_t), 2 * sizeof(int),
                                            cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  const uint64_t zero = 0;
  e = cudaMemcpyToSymbolAsync(g_stall_status, &zero, sizeof(uint64_t), 2 * sizeof(int), cudaMemcpyHostToDevice,
                              stream);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(stream);
}

}  // namespace bi
