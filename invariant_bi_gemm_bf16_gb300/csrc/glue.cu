// glue.cu -- the element-wise steps of a Llama-style decode layer that sit
// between its GEMMs.  Each is row-local and has no reduction, so none of them
// can make a row depend on the batch.  16-byte vector loads and stores, a
// grid-stride loop over vectors.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace bi {

constexpr int kGlueThreads = 256;

__device__ __forceinline__ float lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack(float a, float b) {
  __nv_bfloat162 o = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&o);
}

__device__ __forceinline__ uint32_t add2(uint32_t a, uint32_t b) {
  return pack(__fadd_rn(lo(a), lo(b)), __fadd_rn(hi(a), hi(b)));
}

// out = bf16_rne(a + b)
__global__ void residual_add_kernel(const uint4* a, const uint4* b, uint4* out, int64_t nvec) {
  grid_dep_launch_dependents();
  grid_dep_wait();  // inputs may come from the previous kernel in the stream
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec;
       i += (int64_t)gridDim.x * blockDim.x) {
    const uint4 x = a[i], y = b[i];
    uint4 o;
    o.x = add2(x.x, y.x);
    o.y = add2(x.y, y.y);
    o.z = add2(x.z, y.z);
    o.w = add2(x.w, y.w);
    out[i] = o;
  }
}

// silu(v) * u in fp32: v / (1 + exp(-v)) * u, each step rounded.
__device__ __forceinline__ float silu_mul1(float v, float u) {
  const float e = expf(-v);
  const float s = __fdiv_rn(v, __fadd_rn(1.0f, e));
  return __fmul_rn(s, u);
}

__device__ __forceinline__ uint32_t silu_mul2(uint32_t g, uint32_t u) {
  return pack(silu_mul1(lo(g), lo(u)), silu_mul1(hi(g), hi(u)));
}

// gu [M, 2I] -> out [M, I]; vectors of 8 along I.
__global__ void silu_mul_kernel(const uint4* gu, uint4* out, int64_t M, int64_t I) {
  grid_dep_launch_dependents();
  grid_dep_wait();
  const int64_t vpr = I / 8;  // vectors per output row
  const int64_t nvec = M * vpr;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = i / vpr, v = i % vpr;
    const uint4 g = gu[m * 2 * vpr + v];
    const uint4 u = gu[m * 2 * vpr + vpr + v];
    uint4 o;
    o.x = silu_mul2(g.x, u.x);
    o.y = silu_mul2(g.y, u.y);
    o.z = silu_mul2(g.z, u.z);
    o.w = silu_mul2(g.w, u.w);
    out[i] = o;
  }
}

// qkv [M, (nq + 2 nkv) D] -> out [M, nq D]: query head j copies v of group
// j / (nq / nkv) (the softmax over a single key is exactly 1).
__global__ void attention_ctx1_kernel(const uint4* qkv, uint4* out, int64_t M, int64_t nq,
                                      int64_t nkv, int64_t D) {
  grid_dep_launch_dependents();
  grid_dep_wait();
  const int64_t dv = D / 8;                       // vectors per head
  const int64_t in_row = (nq + 2 * nkv) * dv;     // vectors per qkv row
  const int64_t out_row = nq * dv;
  const int64_t group = nq / nkv;
  const int64_t nvec = M * out_row;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nvec;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t m = i / out_row, c = i % out_row;
    const int64_t j = c / dv, d = c % dv;
    out[i] = qkv[m * in_row + (nq + nkv) * dv + (j / group) * dv + d];
  }
}

static dim3 glue_grid(int64_t nvec) {
  int64_t b = (nvec + kGlueThreads - 1) / kGlueThreads;
  if (b < 1) b = 1;
  if (b > 152 * 16) b = 152 * 16;
  return dim3((unsigned)b);
}

cudaError_t launch_residual_add(const void* a, const void* b, void* out, int64_t count,
                                cudaStream_t stream) {
  const int64_t nvec = count / 8;
  return launch_overlapped(residual_add_kernel, glue_grid(nvec), dim3(kGlueThreads), stream,
                           static_cast<const uint4*>(a), static_cast<const uint4*>(b),
                           static_cast<uint4*>(out), nvec);
}

cudaError_t launch_silu_mul(const void* gu, void* out, int64_t M, int64_t I, cudaStream_t stream) {
  return launch_overlapped(silu_mul_kernel, glue_grid(M * I / 8), dim3(kGlueThreads), stream,
                           static_cast<const uint4*>(gu), static_cast<uint4*>(out), M, I);
}

cudaError_t launch_attention_ctx1(const void* qkv, void* out, int64_t M, int64_t nq, int64_t nkv,
                                  int64_t D, cudaStream_t stream) {
  return launch_overlapped(attention_ctx1_kernel, glue_grid(M * nq * D / 8), dim3(kGlueThreads), stream,
                           static_cast<const uint4*>(qkv), static_cast<uint4*>(out), M, nq, nkv, D);
}

}  // namespace bi
