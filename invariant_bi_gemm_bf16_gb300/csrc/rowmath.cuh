// rowmath.cuh -- the per-row arithmetic shared by the RMSNorm, the E4M3
// quantiser and their fused form, so that the fused kernel gives the bits of
// the two calls in sequence by construction.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace bi {

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ---- RMSNorm: lane l of the row's warp owns vectors l, l + 32, ...

// sum of squares of a vector's 8 values, in order (x*x is exact for bf16 x)
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

// bf16_rne((x * r) * g) for two packed values
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

// the 32 lane partials by the xor butterfly 16, 8, 4, 2, 1 (every lane ends
// with the same total)
__device__ __forceinline__ float butterfly_sum(float v) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

__device__ __forceinline__ float inv_rms(float ss, int64_t H, float eps) {
  const float mean = __fdiv_rn(ss, (float)H);
  return __fdiv_rn(1.0f, __fsqrt_rn(__fadd_rn(mean, eps)));
}

// ---- E4M3 quantisation of a row (order-free amax, then codes)

__device__ __forceinline__ void amax2(uint32_t w, float& amax, bool& bad) {
  const float a = bf_lo(w), b = bf_hi(w);
  bad = bad || !isfinite(a) || !isfinite(b);
  amax = fmaxf(amax, fmaxf(fabsf(a), fabsf(b)));
}

// The largest |value| of packed bf16 pairs, NaN-propagating (max.NaN): a NaN
// anywhere gives NaN, an infinity gives infinity, so one test of the row's
// final maximum finds a row holding either.  The maximum is exact in any
// order, and the sign is cleared first (so -0 and +0 both count as 0).
__device__ __forceinline__ uint32_t absmax_bf16x2(uint32_t acc, uint32_t w) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(acc), "r"(w & 0x7FFF7FFFu));
  return d;
}

__device__ __forceinline__ uint32_t absmax8(uint32_t acc, const uint4& v) {
  acc = absmax_bf16x2(acc, v.x);
  acc = absmax_bf16x2(acc, v.y);
  acc = absmax_bf16x2(acc, v.z);
  return absmax_bf16x2(acc, v.w);
}

__device__ __forceinline__ float fmax_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}

// The packed maxima of a warp's lanes -> the row's amax (all lanes agree).
__device__ __forceinline__ float warp_amax(uint32_t acc) {
  float m = fmax_nan(bf_lo(acc), bf_hi(acc));
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) m = fmax_nan(m, __shfl_xor_sync(0xffffffffu, m, off));
  return m;
}

// Four E4M3 codes of x[0..3] * inv, x[0] in the lowest byte.
__device__ __forceinline__ uint32_t codes4(uint32_t w0, uint32_t w1, float inv) {
  const uint32_t lo = cvt_e4m3x2(__fmul_rn(bf_lo(w0), inv), __fmul_rn(bf_hi(w0), inv));
  const uint32_t hi = cvt_e4m3x2(__fmul_rn(bf_lo(w1), inv), __fmul_rn(bf_hi(w1), inv));
  return lo | (hi << 16);
}

// scale = amax / 448 (1 for a zero row, NaN for a row holding a NaN or an
// infinity) and inv = 448 / amax (1 for a zero row, clamped to the largest
// finite float when it overflows)
__device__ __forceinline__ float e4m3_row_scale(float amax, bool bad) {
  return bad ? __int_as_float(0x7fc00000) : (amax == 0.0f ? 1.0f : __fdiv_rn(amax, 448.0f));
}
__device__ __forceinline__ float e4m3_row_inv(float amax) {
  return amax == 0.0f ? 1.0f : fminf(__fdiv_rn(448.0f, amax), 3.40282347e38f);
}

// ---- RMSNorm fused with the quantisation (quant.cu)

constexpr int64_t kRqMaxH = 16384;  // widest row the fused kernel stages (32 KB per warp)

cudaError_t launch_rmsnorm_quantize_e4m3(const void* X, const void* g, void* Q, float* scale, int64_t M, int64_t H,
                                         float eps, cudaStream_t stream);

}  // namespace bi
