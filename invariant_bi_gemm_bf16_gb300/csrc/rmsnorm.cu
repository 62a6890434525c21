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
#include "rowmath.cuh"

namespace bi {

constexpr int kRmsWarps = 8;
constexpr int64_t kRmsSmCount = 152;  // spreads small batches; any value gives the same bits
constexpr int kRmsSmemWarps = 2;                                 // rows per block of the shared-memory kernel
constexpr int64_t kRmsSmemMinRows = kRmsWarps * kRmsSmCount;     // H = 4096, 8192: from full blocks on every SM

// H = 256 * VPL: each lane holds its VPL vectors in registers.
template <int VPL>
__global__ void __launch_bounds__(32 * kRmsWarps)
    rmsnorm_regs_kernel(const uint4* X, const uint4* __restrict__ g, uint4* Y, int64_t M,
                        float eps) {
  grid_dep_launch_dependents();
  grid_dep_wait();  // X may come from the previous kernel in the stream
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
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

// H = 256 * VPL, VPL a multiple of 8: two passes over the row, each issuing 8
// vector loads per lane before using them.  The first pass caches the row in L2 only, and the
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
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
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

// H = 256 * VPL: each warp stages its row in shared memory (VPL * 512 bytes)
// by 16-byte asynchronous copies, then runs the arithmetic of
// rmsnorm_regs_kernel vector for vector from there.  Few registers and small
// blocks, so more rows per SM are in flight than with the row in registers.
template <int VPL>
__global__ void __launch_bounds__(32 * kRmsSmemWarps)
    rmsnorm_smem_kernel(const uint4* X, const uint4* __restrict__ g, uint4* Y, int64_t M, float eps) {
  extern __shared__ __align__(16) uint4 rms_rows[];
  grid_dep_launch_dependents();
  grid_dep_wait();
  constexpr int kVecs = VPL * 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int64_t row = (int64_t)blockIdx.x * kRmsSmemWarps + warp;
  if (row >= M) return;
  const uint4* x = X + row * kVecs;
  uint4* buf = rms_rows + warp * kVecs;
#pragma unroll
  for (int i = 0; i < VPL; ++i)
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(buf + lane + 32 * i)),
                 "l"(x + lane + 32 * i)
                 : "memory");
  asm volatile("cp.async.commit_group;" ::: "memory");
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  // each lane reads back only the vectors it copied
  float ss = 0.0f;
#pragma unroll 8
  for (int i = 0; i < VPL; ++i) ss = sumsq8(buf[lane + 32 * i], ss);
  ss = butterfly_sum(ss);
  const float r = inv_rms(ss, (int64_t)kVecs * 8, eps);
  uint4* y = Y + row * kVecs;
#pragma unroll 8
  for (int i = 0; i < VPL; ++i) __stcs(y + lane + 32 * i, norm8(buf[lane + 32 * i], __ldg(g + lane + 32 * i), r));
}

// Any H with H % 8 == 0: the same lane partition and order, two passes over
// the row (the second pass re-reads it, typically from L1/L2).
__global__ void __launch_bounds__(32 * kRmsWarps)
    rmsnorm_loop_kernel(const uint4* X, const uint4* __restrict__ g, uint4* Y, int64_t M,
                        int64_t H, float eps) {
  grid_dep_launch_dependents();
  grid_dep_wait();
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
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

// r[m] = 1 / sqrt(ss / H + eps) of each row, for the GEMM that applies the
// RMSNorm to X in shared memory.  The lane partition, the order of the
// squares within a lane and the butterfly are those of the kernels above
// (vectors lane, lane + 32, ... in ascending order, each vector's 8 values in
// order), so r has their bits.  Eight vector loads per lane are issued before
// they are summed, in the same order.
__global__ void __launch_bounds__(32 * kRmsWarps)
    row_scale_kernel(const uint4* X, float* R, int64_t M, int64_t H, float eps) {
  grid_dep_launch_dependents();
  grid_dep_wait();  // X may come from the previous kernel in the stream
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (row >= M) return;
  const int64_t nvec = H / 8;
  const uint4* x = X + row * nvec;
  float ss = 0.0f;
  int64_t i = lane;
  for (; i + 32 * 7 < nvec; i += 32 * 8) {
    uint4 v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = x[i + 32 * j];
#pragma unroll
    for (int j = 0; j < 8; ++j) ss = sumsq8(v[j], ss);
  }
  for (; i < nvec; i += 32) ss = sumsq8(x[i], ss);
  ss = butterfly_sum(ss);
  if (lane == 0) R[row] = inv_rms(ss, H, eps);
}

cudaError_t launch_row_scale(const void* X, float* r, int64_t M, int64_t H, float eps, cudaStream_t stream) {
  int64_t wpb = (M + kRmsSmCount - 1) / kRmsSmCount;
  wpb = wpb < 1 ? 1 : (wpb > kRmsWarps ? kRmsWarps : wpb);
  const int64_t blocks = (M + wpb - 1) / wpb;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  return launch_overlapped(row_scale_kernel, dim3((unsigned)blocks), dim3((unsigned)(32 * wpb)), stream,
                           static_cast<const uint4*>(X), r, M, H, eps);
}

// Kernel per width and batch size, measured on GB300 as fractions of the
// copy bandwidth at M = 16384: registers for H <= 2048 (2048: 1.00); for
// H = 4096 and 8192 the row in shared memory from full blocks on every SM
// (0.94 and 0.96; two passes gave 0.89 and 0.79) and registers below (2.3 us
// at M <= 64 for H = 4096, 1.1-1.8x F.rms_norm); two passes for 16384.  All
// run the same lane partition and order, so the choice never changes a bit.
cudaError_t launch_rmsnorm(const void* X, const void* g, void* Y, int64_t M, int64_t H, float eps,
                           cudaStream_t stream) {
  // rows (warps) per block: ceil(M / SMs) up to kRmsWarps, so a small batch
  // puts at most one block, of as few rows as possible, on each SM
  int64_t wpb = (M + kRmsSmCount - 1) / kRmsSmCount;
  wpb = wpb < 1 ? 1 : (wpb > kRmsWarps ? kRmsWarps : wpb);
  const int64_t blocks = (M + wpb - 1) / wpb;
  if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
  const dim3 grid((unsigned)blocks), block((unsigned)(32 * wpb));
  auto x = static_cast<const uint4*>(X);
  auto gg = static_cast<const uint4*>(g);
  auto y = static_cast<uint4*>(Y);
  switch (H) {
    case 256: return launch_overlapped(rmsnorm_regs_kernel<1>, grid, block, stream, x, gg, y, M, eps);
    case 512: return launch_overlapped(rmsnorm_regs_kernel<2>, grid, block, stream, x, gg, y, M, eps);
    case 1024: return launch_overlapped(rmsnorm_regs_kernel<4>, grid, block, stream, x, gg, y, M, eps);
    case 2048: return launch_overlapped(rmsnorm_regs_kernel<8>, grid, block, stream, x, gg, y, M, eps);
    case 4096:
      if (M >= kRmsSmemMinRows) {
        const int64_t b2 = (M + kRmsSmemWarps - 1) / kRmsSmemWarps;
        if (b2 > 0x7FFFFFFF) return cudaErrorInvalidValue;
        return launch_overlapped_smem(rmsnorm_smem_kernel<16>, dim3((unsigned)b2), dim3(32 * kRmsSmemWarps),
                                      (size_t)kRmsSmemWarps * 16 * 512, stream, x, gg, y, M, eps);
      }
      return launch_overlapped(rmsnorm_regs_kernel<16>, grid, block, stream, x, gg, y, M, eps);
    case 8192:
      if (M >= kRmsSmemMinRows) {
        const int64_t b2 = (M + kRmsSmemWarps - 1) / kRmsSmemWarps;
        if (b2 > 0x7FFFFFFF) return cudaErrorInvalidValue;
        return launch_overlapped_smem(rmsnorm_smem_kernel<32>, dim3((unsigned)b2), dim3(32 * kRmsSmemWarps),
                                      (size_t)kRmsSmemWarps * 32 * 512, stream, x, gg, y, M, eps);
      }
      return launch_overlapped(rmsnorm_regs_kernel<32>, grid, block, stream, x, gg, y, M, eps);
    case 16384: return launch_overlapped(rmsnorm_wide_kernel<64>, grid, block, stream, x, gg, y, M, eps);
    default: return launch_overlapped(rmsnorm_loop_kernel, grid, block, stream, x, gg, y, M, H, eps);
  }
}

}  // namespace bi
