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

// {a.x * b.x, a.y * b.y}: two IEEE fp32 products rounded to nearest even in
// one packed instruction (the same two results as two __fmul_rn)
__device__ __forceinline__ float2 mul2_rn(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 pa, pb, pd;\n\t"
      "mov.b64 pa, {%2, %3};\n\t"
      "mov.b64 pb, {%4, %5};\n\t"
      "mul.rn.f32x2 pd, pa, pb;\n\t"
      "mov.b64 {%0, %1}, pd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

// norm2 with the products taken in pairs (the same bits)
__device__ __forceinline__ uint32_t norm2_packed(uint32_t x, uint32_t g, float r) {
  const float2 t = mul2_rn(make_float2(bf_lo(x), bf_hi(x)), make_float2(r, r));
  const float2 y = mul2_rn(t, make_float2(bf_lo(g), bf_hi(g)));
  __nv_bfloat162 o = __floats2bfloat162_rn(y.x, y.y);
  return *reinterpret_cast<uint32_t*>(&o);
}

__device__ __forceinline__ uint4 norm8_packed(const uint4& x, const uint4& g, float r) {
  uint4 o;
  o.x = norm2_packed(x.x, g.x, r);
  o.y = norm2_packed(x.y, g.y, r);
  o.z = norm2_packed(x.z, g.z, r);
  o.w = norm2_packed(x.w, g.w, r);
  return o;
}

// codes4 with the products taken in pairs (the same bits)
__device__ __forceinline__ uint32_t codes4_packed(uint32_t w0, uint32_t w1, float inv) {
  const float2 a = mul2_rn(make_float2(bf_lo(w0), bf_hi(w0)), make_float2(inv, inv));
  const float2 b = mul2_rn(make_float2(bf_lo(w1), bf_hi(w1)), make_float2(inv, inv));
  return (uint32_t)cvt_e4m3x2(a.x, a.y) | ((uint32_t)cvt_e4m3x2(b.x, b.y) << 16);
}

// The same one pass with the rows streamed: a persistent grid of one block
// per SM, whose warps take rows w, w + G, w + 2G, ... (G warps in all,
// numbered warp-major across the blocks, so that the last, partial round of
// rows is spread over every SM).  Each warp keeps NB of its rows in flight
// through its own ring in shared memory: each lane copies its own vectors of
// a row by 16-byte cp.async, one commit group per row (an empty group past
// the warp's last row, so that every wait leaves NB - 1 newer groups
// pending).  A lane reads back only what it copied, so its own wait (the
// hardware's, no spin) is the only synchronisation.  It reads its vectors of
// the row once, into registers, and normalises, takes the maximum and
// quantises there.  The lane-to-vector split, and so every operation and its
// order, is the register kernel's; the products go in packed pairs (the same
// IEEE products).
constexpr int kRqRingWarps = 12;
constexpr int64_t kRqRingMinRows = 1024;  // from this many rows the ring kernel runs

template <int VPL, int NB>
struct RqRing {
  static constexpr int vecs = VPL * 32;
  static constexpr int smem = (1 + kRqRingWarps * NB) * vecs * 16;  // g, then the warps' rings
  static_assert(smem <= kMaxDynSmem, "ring too large");
};

// The per-row work once a lane holds its vectors v of the row: the sum of
// squares (split out so that the caller can refill the row's slot once every
// vector has been consumed), then the norm, the maximum and the codes.
template <int VPL>
__device__ __forceinline__ float rq_row_sumsq(const uint4 (&v)[VPL]) {
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < VPL; ++i) ss = sumsq8(v[i], ss);
  return butterfly_sum(ss);
}

template <int VPL>
__device__ __forceinline__ void rq_row_finish(uint4 (&v)[VPL], float ss, const uint4* gs, int lane, float eps,
                                              int64_t row, uint2* Q, float* scale) {
  const float r = inv_rms(ss, (int64_t)VPL * 256, eps);
  uint32_t am = 0u;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    v[i] = norm8_packed(v[i], gs[lane + 32 * i], r);
    am = absmax8(am, v[i]);
  }
  const float amax = warp_amax(am);
  const bool bad = !isfinite(amax);
  const float s = e4m3_row_scale(amax, bad);
  const float inv = e4m3_row_inv(amax);
  if (lane == 0) scale[row] = s;
  uint2* q = Q + row * (VPL * 32);
#pragma unroll
  for (int i = 0; i < VPL; ++i)
    q[lane + 32 * i] = bad ? make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu)
                           : make_uint2(codes4_packed(v[i].x, v[i].y, inv), codes4_packed(v[i].z, v[i].w, inv));
}

template <int VPL, int NB>
__global__ void __launch_bounds__(32 * kRqRingWarps, 1)
    rmsnorm_quantize_ring_kernel(const uint4* X, const uint4* __restrict__ g, uint2* Q, float* scale, int64_t M,
                                 float eps) {
  constexpr int kVecs = VPL * 32;
  extern __shared__ __align__(128) uint4 rr_smem[];
  uint4* gs = rr_smem;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint4* ring = rr_smem + (1 + warp * NB) * kVecs;
  for (int i = threadIdx.x; i < kVecs; i += blockDim.x) gs[i] = __ldg(g + i);  // g is a weight
  __syncthreads();
  grid_dep_launch_dependents();
  grid_dep_wait();  // X may come from the previous kernel in the stream
  const int64_t G = (int64_t)gridDim.x * kRqRingWarps;
  const int64_t w0 = (int64_t)warp * gridDim.x + blockIdx.x;
  const int64_t n = w0 < M ? (M - 1 - w0) / G + 1 : 0;  // rows of this warp
  auto issue = [&](int64_t k) {
    if (k < n) {
      const uint4* x = X + (w0 + k * G) * kVecs + lane;
      const uint32_t dst = smem_u32(ring + (int)(k % NB) * kVecs + lane);
#pragma unroll
      for (int i = 0; i < VPL; ++i)
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + 512u * i), "l"(x + 32 * i) : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
#pragma unroll
  for (int b = 0; b < NB; ++b) issue(b);
  for (int64_t k = 0; k < n; ++k) {
    asm volatile("cp.async.wait_group %0;" ::"n"(NB - 1) : "memory");  // row k has landed
    uint4 v[VPL];
    const uint4* buf = ring + (int)(k % NB) * kVecs + lane;
#pragma unroll
    for (int i = 0; i < VPL; ++i) v[i] = buf[32 * i];
    const float ss = rq_row_sumsq(v);
    asm volatile("" ::"f"(ss) : "memory");  // every vector of the slot has been read: refill it
    issue(k + NB);
    rq_row_finish<VPL>(v, ss, gs, lane, eps, w0 + k * G, Q, scale);
  }
}

template <int VPL, int NB>
cudaError_t launch_rq_ring(const void* X, const void* g, void* Q, float* scale, int64_t M, float eps,
                           cudaStream_t stream) {
  using C = RqRing<VPL, NB>;
  static std::atomic<uint64_t> configured{0};  // the shared-memory limit is per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t)1 << dev : 0;
  if (!bit || !(configured.load() & bit)) {
    e = cudaFuncSetAttribute(rmsnorm_quantize_ring_kernel<VPL, NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             C::smem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  int64_t blocks = (M + kRqRingWarps - 1) / kRqRingWarps;
  blocks = blocks < sms ? blocks : sms;
  return launch_overlapped_smem(rmsnorm_quantize_ring_kernel<VPL, NB>, dim3((unsigned)blocks),
                                dim3(32 * kRqRingWarps), (size_t)C::smem, stream, static_cast<const uint4*>(X),
                                static_cast<const uint4*>(g), static_cast<uint2*>(Q), scale, M, eps);
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
  // H = 2048, 4096: the streamed ring from 1024 rows, the row in registers
  // below.  Measured (H = 4096, graph-replayed): ring against registers 4.8
  // against 5.9 us at M = 1024, 9.1 against 10.6 at 3072, 18.0 against 20.7
  // (the staged kernel) at 8192; 4.2 against 3.0 at M = 128.  At H = 2048 the
  // ring wins from 1024 rows too (4.5 against 6.1 at 2560) except around
  // 2048 rows (4.1 against 3.7), where the warps take two rows each.
  if ((H == 2048 || H == 4096) && M >= kRqRingMinRows)
    return H == 2048 ? launch_rq_ring<8, 4>(X, g, Q, scale, M, eps, stream)
                     : launch_rq_ring<16, 2>(X, g, Q, scale, M, eps, stream);
  if (H == 2048 || H == 4096) {
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
