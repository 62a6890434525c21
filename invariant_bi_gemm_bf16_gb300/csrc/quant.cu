// quant.cu -- per-row E4M3 quantisation for the FP8 GEMM.
//
// For each row (a token of the activations, or an output channel of the
// weights): amax = max_k |x_k|, scale = amax / 448 and inv = 448 / amax (IEEE
// divisions once per row; both 1 for a zero row; inv clamped to the largest
// finite float when 448 / amax overflows), q_k = E4M3(x_k * inv), the
// fp32 product rounded to nearest even and saturated at +-448
// (cvt.rn.satfinite).  A row holding a NaN or an infinity gets scale NaN
// and NaN codes (0x7F).  The maximum is exact whatever the order it is taken
// in, and every code depends on its own row only.  Detent (Batch-Invariant LLM
// Serving and RL Rollouts at Near-Stock Speed), Limits: dynamic per-tensor FP8
// activation scales span the batch; per-token scales keep each row's bits its
// own.
#include <atomic>

#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "rowmath.cuh"

namespace bi {

constexpr int kQuantWarps = 8;

// X [M,K] bf16 -> Q [M,K] E4M3, scale [M]; one warp per row, vectors of 8.
__global__ void __launch_bounds__(32 * kQuantWarps)
    quantize_e4m3_kernel(const uint4* X, uint2* Q, float* scale, int64_t M, int64_t K) {
  grid_dep_launch_dependents();
  grid_dep_wait();  // X may come from the previous kernel in the stream
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kQuantWarps + (threadIdx.x >> 5);
  if (row >= M) return;
  const int64_t nvec = K / 8;
  const uint4* x = X + row * nvec;
  float amax = 0.0f;
  bool bad = false;
  for (int64_t i = lane; i < nvec; i += 32) {
    const uint4 v = x[i];
    amax2(v.x, amax, bad);
    amax2(v.y, amax, bad);
    amax2(v.z, amax, bad);
    amax2(v.w, amax, bad);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    bad = __shfl_xor_sync(0xffffffffu, (int)bad, off) || bad;
  }
  const float s = e4m3_row_scale(amax, bad);
  const float inv = e4m3_row_inv(amax);
  if (lane == 0) scale[row] = s;
  uint2* q = Q + row * nvec;
  for (int64_t i = lane; i < nvec; i += 32) {
    if (bad) {
      q[i] = make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu);
    } else {
      const uint4 v = x[i];
      q[i] = make_uint2(codes4(v.x, v.y, inv), codes4(v.z, v.w, inv));
    }
  }
}

// X [M,K] bf16 -> Q, scale; one CTA of kQRowThreads per row, the row held in
// registers (VPT vectors of 8 per thread), so HBM is read once.  The same
// arithmetic as quantize_e4m3_kernel: the maximum is exact in any order.
constexpr int kQRowThreads = 256;
constexpr int kQRowMaxVpt = 16;

template <int VPT>
__global__ void __launch_bounds__(kQRowThreads)
    quantize_e4m3_row_kernel(const uint4* X, uint2* Q, float* scale, int64_t K) {
  __shared__ float wmax[kQRowThreads / 32];
  __shared__ int wbad[kQRowThreads / 32];
  grid_dep_launch_dependents();
  grid_dep_wait();  // X may come from the previous kernel in the stream
  const int64_t row = blockIdx.x, nvec = K / 8;
  const uint4* x = X + row * nvec;
  uint4 v[VPT];
  float amax = 0.0f;
  bool bad = false;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int64_t j = threadIdx.x + (int64_t)i * kQRowThreads;
    if (j < nvec) {
      v[i] = x[j];
      amax2(v[i].x, amax, bad);
      amax2(v[i].y, amax, bad);
      amax2(v[i].z, amax, bad);
      amax2(v[i].w, amax, bad);
    }
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    bad = __shfl_xor_sync(0xffffffffu, (int)bad, off) || bad;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    wmax[warp] = amax;
    wbad[warp] = bad;
  }
  __syncthreads();
  amax = wmax[0];
  bad = wbad[0] != 0;
#pragma unroll
  for (int w = 1; w < kQRowThreads / 32; ++w) {
    amax = fmaxf(amax, wmax[w]);
    bad = bad || wbad[w] != 0;
  }
  const float s = e4m3_row_scale(amax, bad);
  const float inv = e4m3_row_inv(amax);
  if (threadIdx.x == 0) scale[row] = s;
  uint2* q = Q + row * nvec;
#pragma unroll
  for (int i = 0; i < VPT; ++i) {
    const int64_t j = threadIdx.x + (int64_t)i * kQRowThreads;
    if (j < nvec)
      q[j] = bad ? make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu)
                 : make_uint2(codes4(v[i].x, v[i].y, inv), codes4(v[i].z, v[i].w, inv));
  }
}

// The same arithmetic with the row staged in shared memory (16-byte
// asynchronous copies; each thread reads back only the vectors it copied), so
// few registers are held and more rows per SM are in flight than with the
// row in registers.  For rows of up to kQSmemMaxVec vectors.
constexpr int kQSmemMaxVec = 6144;  // 96 KB
__global__ void __launch_bounds__(kQRowThreads)
    quantize_e4m3_smem_kernel(const uint4* X, uint2* Q, float* scale, int64_t K) {
  extern __shared__ __align__(16) uint4 qrow[];
  __shared__ float wmax[kQRowThreads / 32];
  __shared__ int wbad[kQRowThreads / 32];
  grid_dep_launch_dependents();
  grid_dep_wait();  // X may come from the previous kernel in the stream
  const int64_t row = blockIdx.x;
  const int nvec = (int)(K / 8);
  const uint4* x = X + row * nvec;
  for (int j = threadIdx.x; j < nvec; j += kQRowThreads)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(qrow + j)), "l"(x + j) : "memory");
  asm volatile("cp.async.commit_group;" ::: "memory");
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  float amax = 0.0f;
  bool bad = false;
  for (int j = threadIdx.x; j < nvec; j += kQRowThreads) {
    const uint4 v = qrow[j];
    amax2(v.x, amax, bad);
    amax2(v.y, amax, bad);
    amax2(v.z, amax, bad);
    amax2(v.w, amax, bad);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    bad = __shfl_xor_sync(0xffffffffu, (int)bad, off) || bad;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    wmax[warp] = amax;
    wbad[warp] = bad;
  }
  __syncthreads();
  amax = wmax[0];
  bad = wbad[0] != 0;
#pragma unroll
  for (int w = 1; w < kQRowThreads / 32; ++w) {
    amax = fmaxf(amax, wmax[w]);
    bad = bad || wbad[w] != 0;
  }
  const float s = e4m3_row_scale(amax, bad);
  const float inv = e4m3_row_inv(amax);
  if (threadIdx.x == 0) scale[row] = s;
  uint2* q = Q + row * nvec;
  for (int j = threadIdx.x; j < nvec; j += kQRowThreads) {
    const uint4 v = qrow[j];
    q[j] = bad ? make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu) : make_uint2(codes4(v.x, v.y, inv), codes4(v.z, v.w, inv));
  }
}

static cudaError_t launch_rows_smem(const void* X, void* Q, float* scale, int64_t M, int64_t K,
                                    cudaStream_t stream) {
  // the shared-memory limit is per device: set it once for each
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t)1 << dev : 0;
  if (!bit || !(configured.load() & bit)) {
    e = cudaFuncSetAttribute(quantize_e4m3_smem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kQSmemMaxVec * 16);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  return launch_overlapped_smem(quantize_e4m3_smem_kernel, dim3((unsigned)M), dim3(kQRowThreads),
                                (size_t)(K / 8) * 16, stream, static_cast<const uint4*>(X), static_cast<uint2*>(Q),
                                scale, K);
}

template <int VPT>
static cudaError_t launch_rows_vpt(const void* X, void* Q, float* scale, int64_t M, int64_t K,
                                   cudaStream_t stream) {
  return launch_overlapped(quantize_e4m3_row_kernel<VPT>, dim3((unsigned)M), dim3(kQRowThreads), stream,
                           static_cast<const uint4*>(X), static_cast<uint2*>(Q), scale, K);
}

// ---------------------------------------------------------------------------
// RMSNorm and quantisation in one pass over X
// ---------------------------------------------------------------------------
// Row m: y = bf16_rne((x * r) * g) with the RMSNorm tree of bi_rmsnorm_bf16
// (lane l of the row's warp sums the squares of vectors l, l + 32, ... in
// order; the xor butterfly combines the lanes), then the E4M3 codes of y with
// the row's scale, as bi_quantize_rows_e4m3 takes them from y.  One warp per
// row; the block stages g once and each warp its row in shared memory by
// 16-byte asynchronous copies, so X is read once and y never leaves the chip.
// Three passes over the staged row: the sum of squares; y (written back over
// x) with its packed NaN-propagating maximum; the codes of y.
constexpr int kRqSmemBudget = 100 * 1024;  // shared memory per block: rows and g

int rq_rows_per_block(int64_t H) {
  const int64_t r = kRqSmemBudget / (2 * H) - 1;
  return r < 1 ? 1 : (r > 8 ? 8 : (int)r);
}

__global__ void __launch_bounds__(256)
    rmsnorm_quantize_kernel(const uint4* X, const uint4* __restrict__ g, uint2* Q, float* scale, int64_t M,
                            int64_t H, float eps) {
  extern __shared__ __align__(16) uint4 rq_smem[];
  grid_dep_launch_dependents();
  grid_dep_wait();  // X may come from the previous kernel in the stream
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, wpb = blockDim.x >> 5;
  const int nvec = (int)(H / 8);
  uint4* gs = rq_smem;  // g, then one row per warp
  for (int i = threadIdx.x; i < nvec; i += blockDim.x)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(gs + i)), "l"(g + i) : "memory");
  const int64_t row = (int64_t)blockIdx.x * wpb + warp;
  const bool live = row < M;
  const uint4* x = X + (live ? row : 0) * nvec;
  uint4* buf = rq_smem + (int64_t)(warp + 1) * nvec;
  if (live)
    for (int i = lane; i < nvec; i += 32)
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(buf + i)), "l"(x + i) : "memory");
  asm volatile("cp.async.commit_group;" ::: "memory");
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  __syncthreads();  // g was copied by the whole block
  if (!live) return;
  float ss = 0.0f;
#pragma unroll 4
  for (int i = lane; i < nvec; i += 32) ss = sumsq8(buf[i], ss);
  ss = butterfly_sum(ss);
  const float r = inv_rms(ss, H, eps);
  uint32_t am = 0u;
#pragma unroll 4
  for (int i = lane; i < nvec; i += 32) {
    const uint4 y = norm8(buf[i], gs[i], r);
    buf[i] = y;  // each lane reads back only its own vectors
    am = absmax8(am, y);
  }
  const float amax = warp_amax(am);
  const bool bad = !isfinite(amax);
  const float s = e4m3_row_scale(amax, bad);
  const float inv = e4m3_row_inv(amax);
  if (lane == 0) scale[row] = s;
  uint2* q = Q + row * nvec;
#pragma unroll 4
  for (int i = lane; i < nvec; i += 32) {
    const uint4 y = buf[i];
    q[i] = bad ? make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu) : make_uint2(codes4(y.x, y.y, inv), codes4(y.z, y.w, inv));
  }
}

// The same with the row in registers (H = 256 * VPL): every vector of a
// lane is loaded at once, normalised in place, and quantised from there.  The
// block stages g in shared memory first, so that the norm pass holds one
// gain vector at a time beside the row (at most 128 registers: two blocks of
// 8 rows per SM).
template <int VPL>
__global__ void __launch_bounds__(256, 2)
    rmsnorm_quantize_regs_kernel(const uint4* X, const uint4* __restrict__ g, uint2* Q, float* scale, int64_t M,
                                 float eps) {
  constexpr int kVecs = VPL * 32;
  __shared__ uint4 gs[kVecs];
  for (int i = threadIdx.x; i < kVecs; i += blockDim.x) gs[i] = __ldg(g + i);  // g is a weight
  grid_dep_launch_dependents();
  grid_dep_wait();
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const bool live = row < M;
  uint4 v[VPL];
  if (live) {
    const uint4* x = X + row * kVecs;
#pragma unroll
    for (int i = 0; i < VPL; ++i) v[i] = __ldcs(x + lane + 32 * i);
  }
  __syncthreads();  // gs is complete
  if (!live) return;
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < VPL; ++i) ss = sumsq8(v[i], ss);
  ss = butterfly_sum(ss);
  const float r = inv_rms(ss, (int64_t)kVecs * 8, eps);
  uint32_t am = 0u;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    v[i] = norm8(v[i], gs[lane + 32 * i], r);
    am = absmax8(am, v[i]);
  }
  const float amax = warp_amax(am);
  const bool bad = !isfinite(amax);
  const float s = e4m3_row_scale(amax, bad);
  const float inv = e4m3_row_inv(amax);
  if (lane == 0) scale[row] = s;
  uint2* q = Q + row * kVecs;
#pragma unroll
  for (int i = 0; i < VPL; ++i)
    q[lane + 32 * i] = bad ? make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu)
                           : make_uint2(codes4(v[i].x, v[i].y, inv), codes4(v[i].z, v[i].w, inv));
}

cudaError_t launch_rmsnorm_quantize_e4m3(const void* X, const void* g, void* Q, float* scale, int64_t M, int64_t H,
                                         float eps, cudaStream_t stream) {
  // the shared-memory limit is per device: set it once for each
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t)1 << dev : 0;
  if (!bit || !(configured.load() & bit)) {
    e = cudaFuncSetAttribute(rmsnorm_quantize_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kRqSmemBudget);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  // the row in registers for H = 2048, 4096 below 4096 rows (measured at
  // H = 4096, M = 2048: 7.5 us with g staged in shared memory and 128
  // registers, 8.8 with g from L2 and 205 registers, 12.4 staged).  At
  // M = 8192 the staged kernel takes 20.7 us (0.72 of HBM; 26.4 before y was
  // written back and the maximum taken packed) against 23.1 for the register
  // kernel; a persistent variant with two rows per warp in flight took 23.1.
  if ((H == 2048 || H == 4096) && M < 4096) {
    // rows (warps) per block: ceil(M / 152) up to 8, as for the RMSNorm
    int64_t wpb = (M + 151) / 152;
    wpb = wpb < 1 ? 1 : (wpb > 8 ? 8 : wpb);
    const int64_t b2 = (M + wpb - 1) / wpb;
    if (b2 > 0x7FFFFFFF) return cudaErrorInvalidValue;
    auto kern = H == 2048 ? rmsnorm_quantize_regs_kernel<8> : rmsnorm_quantize_regs_kernel<16>;
    return launch_overlapped(kern, dim3((unsigned)b2), dim3((unsigned)(32 * wpb)), stream,
                             static_cast<const uint4*>(X), static_cast<const uint4*>(g), static_cast<uint2*>(Q),
                             scale, M, eps);
  }
  const int wpb = rq_rows_per_block(H);
  const int64_t blocks = (M + wpb - 1) / wpb;
  if (blocks > 0x7FFFFFFF || H > kRqMaxH) return cudaErrorInvalidValue;
  return launch_overlapped_smem(rmsnorm_quantize_kernel, dim3((unsigned)blocks), dim3(32 * wpb),
                                (size_t)(wpb + 1) * H * 2, stream, static_cast<const uint4*>(X),
                                static_cast<const uint4*>(g), static_cast<uint2*>(Q), scale, M, H, eps);
}

cudaError_t launch_quantize_e4m3(const void* X, void* Q, float* scale, int64_t M, int64_t K,
                                 cudaStream_t stream) {
  const int64_t vpt = (K / 8 + kQRowThreads - 1) / kQRowThreads;
  if (M <= 0x7FFFFFFF && vpt >= 4 && K / 8 <= kQSmemMaxVec) return launch_rows_smem(X, Q, scale, M, K, stream);
  if (M <= 0x7FFFFFFF && vpt <= kQRowMaxVpt) {
    if (vpt <= 1) return launch_rows_vpt<1>(X, Q, scale, M, K, stream);
    if (vpt <= 2) return launch_rows_vpt<2>(X, Q, scale, M, K, stream);
    if (vpt <= 4) return launch_rows_vpt<4>(X, Q, scale, M, K, stream);
    if (vpt <= 8) return launch_rows_vpt<8>(X, Q, scale, M, K, stream);
    return launch_rows_vpt<16>(X, Q, scale, M, K, stream);
  }
  // rows too long for registers: one warp per row, two reads of the row
  const int64_t blocks = (M + kQuantWarps - 1) / kQuantWarps;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  return launch_overlapped(quantize_e4m3_kernel, dim3((unsigned)blocks), dim3(32 * kQuantWarps), stream,
                           static_cast<const uint4*>(X), static_cast<uint2*>(Q), scale, M, K);
}

}  // namespace bi
