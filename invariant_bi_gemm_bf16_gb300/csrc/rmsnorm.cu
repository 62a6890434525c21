// rmsnorm.cu -- batch-invariant RMSNorm, one warp per row.
//
// y_h = bf16_rne((x_h * r) * g_h),  r = 1 / sqrt(ss / H + eps),  ss = sum_h x_h^2.
//
// The reduction tree of a row depends on H only:
//   * the row is read as 16-byte vectors of 8 bf16; lane l owns vectors
//     l, l + 32, l + 64, ... and adds their squares in ascending vector order,
//     element 0..7 within a vector, into one fp32 partial (x*x of a bf16 x is
//     exact in fp32, so the fused multiply-add rounds only the sum);
//   * the 32 lane partials are combined by an xor butterfly with offsets
//     16, 8, 4, 2, 1.  Both operands of every butterfly add are the same two
//     values in every lane, so all lanes end with the same total;
//   * ss / H, the square root and 1 / sqrt are IEEE-rounded (no fast math).
// LLM-42 (Enabling Determinism in LLM Inference with Verified Speculation),
// Sec. 2.1: normalisation reduces over the hidden dimension of each token; a
// row is never split across warps, so neither M nor the other rows reach it.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace bi {

constexpr int kRmsWarps = 8;

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ float sumsq8(const uint4& v, float ss) {
  ss = __fmaf_rn(bf_lo(v.x), bf_lo(v.x), ss);
  ss = __fmaf_rn(bf_hi(v.x), bf_hi(v.x), ss);
  ss = __fmaf_rn(bf_lo(v.y), bf_lo(v.y), ss);
  ss = __fmaf_rn(bf_hi(v.y), bf_hi(v.y), ss);
  ss = __fmaf_rn(bf_lo(v.z), bf_lo(v.z), ss);
  ss = __fmaf_rn(bf_hi(v.z), bf_hi(v.z), ss);
  ss = __fmaf_rn(bf_lo(v.w), bf_lo(v.w), ss);
  ss = __fmaf_rn(bf_hi(v.w), bf_hi(v.w), ss);
  return ss;
}

__device__ __forceinline__ uint32_t norm2(uint32_t x, uint32_t g, float r) {
  const float a = __fmul_rn(__fmul_rn(bf_lo(x), r), bf_lo(g));
  const float b = __fmul_rn(__fmul_rn(bf_hi(x), r), bf_hi(g));
  __nv_bfloat162 o = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&o);
}

__device__ __forceinline__ uint4 norm8(const uint4& x, const uint4& g, float r) {
  uint4 o;
  o.x = norm2(x.x, g.x, r);
  o.y = norm2(x.y, g.y, r);
  o.z = norm2(x.z, g.z, r);
  o.w = norm2(x.w, g.w, r);
  return o;
}

__device__ __forceinline__ float butterfly_sum(float v) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

__device__ __forceinline__ float inv_rms(float ss, int64_t H, float eps) {
  const float mean = __fdiv_rn(ss, (float)H);
  return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
}

// H = 256 * VPL: each lane holds its VPL vectors in registers.
template <int VPL>
__global__ void __launch_bounds__(32 * kRmsWarps)
    rmsnorm_regs_kernel(const uint4* X, const uint4* __restrict__ g, uint4* Y, int64_t M,
                        float eps) {
  grid_dep_launch_dependents();
  grid_dep_wait();  // X may come from the previous kernel in the stream
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kRmsWarps + (threadIdx.x >> 5);
  if (row >= M) return;
  constexpr int kVecs = VPL * 32;
  const uint4* x = X + row * kVecs;
  uint4 v[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) v[i] = __ldcs(x + lane + 32 * i);  // streamed once
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < VPL; ++i) ss = sumsq8(v[i], ss);
  ss = butterfly_sum(ss);
  const float r = inv_rms(ss, (int64_t)kVecs * 8, eps);
  uint4* y = Y + row * kVecs;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const uint4 gv = __ldg(g + lane + 32 * i);
    __stcs(y + lane + 32 * i, norm8(v[i], gv, r));
  }
}

// H = 256 * VPL, wide rows: each warp streams its rows (row w, w + W, ...,
// W warps in the grid) through a ring of kRmsStages row buffers in shared
// memory, filled by 16-byte asynchronous copies.  Lane l copies exactly the
// vectors it later reads (l, l + 32, ...), so its own wait_group makes them
// visible and no lane waits for another.  The arithmetic is that of
// rmsnorm_regs_kernel, vector for vector; the copies only keep kRmsStages rows
// of every warp in flight without holding them in registers.
constexpr int kRmsStages = 3;

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* gmem_src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <int VPL>
__global__ void __launch_bounds__(256)
    rmsnorm_async_kernel(const uint4* X, const uint4* __restrict__ g, uint4* Y, int64_t M, float eps) {
  extern __shared__ uint4 rms_ring[];
  grid_dep_launch_dependents();
  grid_dep_wait();  // X may come from the previous kernel in the stream
  constexpr int kVecs = VPL * 32;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t first = (int64_t)blockIdx.x * (blockDim.x >> 5) + warp;
  uint4* ring = rms_ring + (size_t)warp * kRmsStages * kVecs;
  // prologue: the warp's first kRmsStages rows (one commit group per row,
  // empty groups past M keep the count uniform)
#pragma unroll
  for (int st = 0; st < kRmsStages; ++st) {
    const int64_t row = first + st * nwarps;
    if (row < M) {
      const uint4* x = X + row * kVecs;
#pragma unroll 8
      for (int i = 0; i < VPL; ++i) cp_async16(ring + st * kVecs + lane + 32 * i, x + lane + 32 * i);
    }
    cp_async_commit();
  }
  // Software pipeline: the serial sum-of-squares chain of the next row runs
  // interleaved with the (independent) normalisation and stores of the
  // current one.  Commit groups go one per row in row order, so before the
  // step for the k-th row k + 3 groups exist and waiting down to one pending
  // group means rows k and k + 1 have landed.
  int st = 0;
  float r = 0.0f;
  if (first < M) {
    cp_async_wait<kRmsStages - 1>();
    const uint4* v = ring;
    float ss = 0.0f;
#pragma unroll 8
    for (int i = 0; i < VPL; ++i) ss = sumsq8(v[lane + 32 * i], ss);
    r = inv_rms(butterfly_sum(ss), (int64_t)kVecs * 8, eps);
  }
  for (int64_t row = first; row < M; row += nwarps) {
    const int64_t nxt = row + nwarps;
    const bool has_next = nxt < M;  // the same in every lane
    const int st_next = st + 1 == kRmsStages ? 0 : st + 1;
    cp_async_wait<1>();
    const uint4* v = ring + st * kVecs;
    const uint4* vn = ring + st_next * kVecs;
    uint4* y = Y + row * kVecs;
    float ss = 0.0f;
    if (has_next) {
#pragma unroll 8
      for (int i = 0; i < VPL; ++i) {
        ss = sumsq8(vn[lane + 32 * i], ss);
        __stcs(y + lane + 32 * i, norm8(v[lane + 32 * i], __ldg(g + lane + 32 * i), r));
      }
    } else {
#pragma unroll 8
      for (int i = 0; i < VPL; ++i) __stcs(y + lane + 32 * i, norm8(v[lane + 32 * i], __ldg(g + lane + 32 * i), r));
    }
    // refill this stage with the row kRmsStages ahead
    const int64_t ahead = row + (int64_t)kRmsStages * nwarps;
    if (ahead < M) {
      const uint4* x = X + ahead * kVecs;
#pragma unroll 8
      for (int i = 0; i < VPL; ++i) cp_async16(ring + st * kVecs + lane + 32 * i, x + lane + 32 * i);
    }
    cp_async_commit();
    if (has_next) r = inv_rms(butterfly_sum(ss), (int64_t)kVecs * 8, eps);
    st = st_next;
  }
  cp_async_wait<0>();
}

// H = 256 * VPL, VPL a multiple of 8, rows too wide to stage per warp at
// high occupancy: two passes over the row, each issuing 8 vector loads per
// lane before using them.  The first pass caches the row in L2 only, and the
// second reads it back from there; the arithmetic is vector for vector that
// of rmsnorm_regs_kernel.  About 40 registers, so many warps per SM hide the
// serial sum-of-squares chain of each row.
template <int VPL>
__global__ void __launch_bounds__(32 * kRmsWarps)
    rmsnorm_wide_kernel(const uint4* X, const uint4* __restrict__ g, uint4* Y, int64_t M, float eps) {
  grid_dep_launch_dependents();
  grid_dep_wait();
  constexpr int kVecs = VPL * 32;
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kRmsWarps + (threadIdx.x >> 5);
  if (row >= M) return;
  const uint4* x = X + row * kVecs;
  float ss = 0.0f;
  for (int i0 = 0; i0 < VPL; i0 += 8) {
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = __ldcg(x + lane + 32 * (i0 + j));
#pragma unroll
    for (int j = 0; j < 8; ++j) ss = sumsq8(v[j], ss);
  }
  ss = butterfly_sum(ss);
  const float r = inv_rms(ss, (int64_t)kVecs * 8, eps);
  uint4* y = Y + row * kVecs;
  for (int i0 = 0; i0 < VPL; i0 += 8) {
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = __ldcs(x + lane + 32 * (i0 + j));
#pragma unroll
    for (int j = 0; j < 8; ++j) __stcs(y + lane + 32 * (i0 + j), norm8(v[j], __ldg(g + lane + 32 * (i0 + j)), r));
  }
}

// Any H with H % 8 == 0: the same lane partition and order, two passes over
// the row (the second pass re-reads it, typically from L1/L2).
__global__ void __launch_bounds__(32 * kRmsWarps)
    rmsnorm_loop_kernel(const uint4* X, const uint4* __restrict__ g, uint4* Y, int64_t M,
                        int64_t H, float eps) {
  grid_dep_launch_dependents();
  grid_dep_wait();
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kRmsWarps + (threadIdx.x >> 5);
  if (row >= M) return;
  const int64_t nvec = H / 8;
  const uint4* x = X + row * nvec;
  float ss = 0.0f;
  for (int64_t i = lane; i < nvec; i += 32) ss = sumsq8(x[i], ss);
  ss = butterfly_sum(ss);
  const float r = inv_rms(ss, H, eps);
  uint4* y = Y + row * nvec;
  for (int64_t i = lane; i < nvec; i += 32) y[i] = norm8(x[i], __ldg(g + i), r);
}

// Wide rows through rmsnorm_async_kernel: warps per block so that the rings
// fill about 192 KB of shared memory, and one block per SM (grid-stride rows).
template <int VPL>
static cudaError_t launch_async(const uint4* x, const uint4* g, uint4* y, int64_t M, float eps,
                                cudaStream_t stream) {
  constexpr int64_t kRowBytes = (int64_t)VPL * 32 * 16;
  int warps = (int)((192 * 1024) / (kRmsStages * kRowBytes));
  if (warps > 8) warps = 8;
  if (warps < 1) warps = 1;
  const int smem = warps * kRmsStages * (int)kRowBytes;
  auto kern = rmsnorm_async_kernel<VPL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  int64_t blocks = (M + warps - 1) / warps;
  if (blocks > sms) blocks = sms;
  if (blocks < 1) blocks = 1;
  return launch_overlapped_smem(kern, dim3((unsigned)blocks), dim3(32 * warps), (size_t)smem, stream, x, g, y,
                                M, eps);
}

cudaError_t launch_rmsnorm(const void* X, const void* g, void* Y, int64_t M, int64_t H, float eps,
                           cudaStream_t stream) {
  const int64_t blocks = (M + kRmsWarps - 1) / kRmsWarps;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)blocks), block(32 * kRmsWarps);
  auto x = static_cast<const uint4*>(X);
  auto gg = static_cast<const uint4*>(g);
  auto y = static_cast<uint4*>(Y);
  switch (H) {
    case 256: return launch_overlapped(rmsnorm_regs_kernel<1>, grid, block, stream, x, gg, y, M, eps);
    case 512: return launch_overlapped(rmsnorm_regs_kernel<2>, grid, block, stream, x, gg, y, M, eps);
    case 1024: return launch_overlapped(rmsnorm_regs_kernel<4>, grid, block, stream, x, gg, y, M, eps);
    case 2048: return launch_async<8>(x, gg, y, M, eps, stream);
    case 4096: return launch_async<16>(x, gg, y, M, eps, stream);
    case 8192: return launch_overlapped(rmsnorm_wide_kernel<32>, grid, block, stream, x, gg, y, M, eps);
    case 16384: return launch_overlapped(rmsnorm_wide_kernel<64>, grid, block, stream, x, gg, y, M, eps);
    default: return launch_overlapped(rmsnorm_loop_kernel, grid, block, stream, x, gg, y, M, H, eps);
  }
}

}  // namespace bi
