// logsoftmax.cu -- batch-invariant log-probabilities of a row of bf16 logits
// (the lm_head output): out_v = x_v - lse, lse = m + log(sum_v exp(x_v - m)),
// m = max_v x_v, all in fp32.
//
// A cluster of kLsmCtas CTAs of kLsmThreads threads per row; the reduction
// tree depends on V only:
//   * the row is read as 16-byte vectors of 8 bf16; thread g = rank *
//     kLsmThreads + t of the cluster owns vectors g, g + G, g + 2G, ...
//     (G = kLsmCtas * kLsmThreads): it takes the maximum m of their elements,
//     then s = the sum of exp(x - m) over them, in ascending order, giving the
//     thread's pair (m, s); its first vectors stay in registers for the
//     output pass, so a row of up to 131072 logits is read once;
//   * pairs combine as m = max(m1, m2), s = s1 exp(m1 - m) + s2 exp(m2 - m):
//     by an xor butterfly (16, 8, 4, 2, 1) within each warp, then the warp
//     results by the same butterfly in warp 0, then the CTA results (read
//     from the cluster's shared memory) by the same butterfly in warp 0 of
//     rank 0; lanes past the count hold the identity (-inf, 0).  The two
//     operands of every combine are the same two pairs in both lanes and IEEE
//     addition commutes, so every lane ends with the same pair;
//   * exp(x - m) is 2^((x - m) log2 e) by the ex2.approx instruction (the
//     pair combines use CUDA's expf), and logf is CUDA's.
// Rows holding a NaN or a +Inf, or -Inf everywhere, give NaN everywhere.
// Detent (Batch-Invariant LLM Serving and RL Rollouts at Near-Stock Speed),
// Sec. 8, Table 6, and CoRun (Padding is Simple and Efficient for
// Deterministic LLM Inference), Sec. IV: per-token log-probabilities are
// what batch invariance is judged on; a row never leaves its cluster, so
// neither M nor the other rows reach its tree.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace bi {

constexpr int kLsmThreads = 512;
constexpr int kLsmWarps = kLsmThreads / 32;
constexpr int kLsmCtas = 8;                        // cluster size: CTAs per row
constexpr int kLsmStride = kLsmCtas * kLsmThreads;  // vectors between a thread's vectors

__device__ __forceinline__ float lsm_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float lsm_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void ms_combine(float& m, float& s, float m2, float s2) {
  const float mm = fmaxf(m, m2);
  if (mm == -INFINITY) {
    s = 0.0f;
  } else {
    s = __fadd_rn(__fmul_rn(s, expf(m - mm)), __fmul_rn(s2, expf(m2 - mm)));
  }
  m = mm;
}

__device__ __forceinline__ void ms_butterfly(float& m, float& s, bool& bad) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, off);
    const int b2 = __shfl_xor_sync(0xffffffffu, (int)bad, off);
    ms_combine(m, s, m2, s2);
    bad = bad || b2;
  }
}

// Shared state of one CTA: per-warp pairs, then the CTA's pair and the row's lse.
struct LsmShared {
  float m[kLsmWarps], s[kLsmWarps];
  int bad[kLsmWarps];
  float cta_m, cta_s, cta_bad;  // cta_bad: 1.0f if the CTA saw a NaN or +Inf
  float lse;
};

// Vectors a thread keeps in registers between the lse and the output pass
// (V up to kLsmCache * 8 * kLsmStride = 131072 is read once).
constexpr int kLsmCache = 4;

__device__ __forceinline__ float max8(const uint4& v) {
  return fmaxf(fmaxf(fmaxf(lsm_lo(v.x), lsm_hi(v.x)), fmaxf(lsm_lo(v.y), lsm_hi(v.y))),
               fmaxf(fmaxf(lsm_lo(v.z), lsm_hi(v.z)), fmaxf(lsm_lo(v.w), lsm_hi(v.w))));
}

__device__ __forceinline__ bool bad8(const uint4& v) {
  // NaN or +Inf anywhere (-Inf is an ordinary logit)
  return !(lsm_lo(v.x) < INFINITY) || !(lsm_hi(v.x) < INFINITY) || !(lsm_lo(v.y) < INFINITY) ||
         !(lsm_hi(v.y) < INFINITY) || !(lsm_lo(v.z) < INFINITY) || !(lsm_hi(v.z) < INFINITY) ||
         !(lsm_lo(v.w) < INFINITY) || !(lsm_hi(v.w) < INFINITY);
}

// exp(d) for d = x - m <= 0 as 2^(d * log2(e)) by the ex2.approx
// instruction: the product rounds once (relative error |d| 2^-24 in the
// result, and terms with large |d| are tiny), ex2.approx adds about 2^-22.
__device__ __forceinline__ float exp_le0(float d) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(__fmul_rn(d, 1.4426950408889634f)));
  return y;
}

// sum of exp(x - m) over a vector, elements in order (m finite)
__device__ __forceinline__ float sumexp8(const uint4& v, float m, float s) {
  s = __fadd_rn(s, exp_le0(__fsub_rn(lsm_lo(v.x), m)));
  s = __fadd_rn(s, exp_le0(__fsub_rn(lsm_hi(v.x), m)));
  s = __fadd_rn(s, exp_le0(__fsub_rn(lsm_lo(v.y), m)));
  s = __fadd_rn(s, exp_le0(__fsub_rn(lsm_hi(v.y), m)));
  s = __fadd_rn(s, exp_le0(__fsub_rn(lsm_lo(v.z), m)));
  s = __fadd_rn(s, exp_le0(__fsub_rn(lsm_hi(v.z), m)));
  s = __fadd_rn(s, exp_le0(__fsub_rn(lsm_lo(v.w), m)));
  s = __fadd_rn(s, exp_le0(__fsub_rn(lsm_hi(v.w), m)));
  return s;
}

// The row's lse (every thread of the cluster returns it).  Thread g of the
// cluster owns vectors g, g + G, g + 2G, ...: it takes the maximum m of its
// elements, then s = sum of exp(x - m) over them in ascending order; the
// per-thread pairs (m, s) then combine by the fixed butterflies.  The first
// kLsmCache vectors stay in v[] for the output pass.
__device__ float row_lse(const uint4* x, int64_t nvec, LsmShared& sh, uint4 (&v)[kLsmCache]) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  const int64_t g0 = (int64_t)rank * kLsmThreads + tid;
  float m = -INFINITY, s = 0.0f;
  bool bad = false;
#pragma unroll
  for (int i = 0; i < kLsmCache; ++i) {
    const int64_t k = g0 + (int64_t)i * kLsmStride;
    if (k < nvec) {
      v[i] = x[k];
      m = fmaxf(m, max8(v[i]));
      bad = bad || bad8(v[i]);
    }
  }
  for (int64_t k = g0 + (int64_t)kLsmCache * kLsmStride; k < nvec; k += kLsmStride) {
    const uint4 w = x[k];
    m = fmaxf(m, max8(w));
    bad = bad || bad8(w);
  }
  if (m != -INFINITY) {
#pragma unroll
    for (int i = 0; i < kLsmCache; ++i) {
      const int64_t k = g0 + (int64_t)i * kLsmStride;
      if (k < nvec) s = sumexp8(v[i], m, s);
    }
    for (int64_t k = g0 + (int64_t)kLsmCache * kLsmStride; k < nvec; k += kLsmStride) s = sumexp8(x[k], m, s);
  }
  ms_butterfly(m, s, bad);
  if (lane == 0) {
    sh.m[warp] = m;
    sh.s[warp] = s;
    sh.bad[warp] = bad;
  }
  __syncthreads();
  if (warp == 0) {
    m = lane < kLsmWarps ? sh.m[lane] : -INFINITY;
    s = lane < kLsmWarps ? sh.s[lane] : 0.0f;
    bad = lane < kLsmWarps ? sh.bad[lane] != 0 : false;
    ms_butterfly(m, s, bad);
    if (lane == 0) {
      sh.cta_m = m;
      sh.cta_s = s;
      sh.cta_bad = bad ? 1.0f : 0.0f;
    }
  }
  cluster_sync();  // every CTA's pair is in its shared memory
  if (rank == 0 && warp == 0) {
    m = -INFINITY;
    s = 0.0f;
    bad = false;
    if (lane < kLsmCtas) {
      m = ld_dsmem_f32(mapa_shared(smem_u32(&sh.cta_m), (uint32_t)lane));
      s = ld_dsmem_f32(mapa_shared(smem_u32(&sh.cta_s), (uint32_t)lane));
      bad = ld_dsmem_f32(mapa_shared(smem_u32(&sh.cta_bad), (uint32_t)lane)) != 0.0f;
    }
    ms_butterfly(m, s, bad);
    if (lane == 0) sh.lse = (bad || m == -INFINITY) ? __int_as_float(0x7fc00000) : m + logf(s);
  }
  cluster_sync();  // rank 0 has the lse
  const float lse = ld_dsmem_f32(mapa_shared(smem_u32(&sh.lse), 0u));
  cluster_sync();  // nobody leaves while its shared memory may still be read
  return lse;
}

__device__ __forceinline__ void write_out(float4* y, int64_t k, const uint4& v, float lse) {
  y[2 * k] = make_float4(lsm_lo(v.x) - lse, lsm_hi(v.x) - lse, lsm_lo(v.y) - lse, lsm_hi(v.y) - lse);
  y[2 * k + 1] = make_float4(lsm_lo(v.z) - lse, lsm_hi(v.z) - lse, lsm_lo(v.w) - lse, lsm_hi(v.w) - lse);
}

// X [M,V] bf16 -> Y [M,V] fp32 log-probabilities; cluster r of the grid is row r.
__global__ void __launch_bounds__(kLsmThreads)
    log_softmax_kernel(const uint4* X, float4* Y, int64_t nvec) {
  __shared__ LsmShared sh;
  grid_dep_launch_dependents();
  grid_dep_wait();  // the logits may come from the previous kernel in the stream
  const int64_t row = blockIdx.x / kLsmCtas;
  const uint4* x = X + row * nvec;
  uint4 v[kLsmCache];
  const float lse = row_lse(x, nvec, sh, v);
  float4* y = Y + row * nvec * 2;
  const int64_t g0 = (int64_t)cluster_ctarank() * kLsmThreads + threadIdx.x;
#pragma unroll
  for (int i = 0; i < kLsmCache; ++i) {
    const int64_t k = g0 + (int64_t)i * kLsmStride;
    if (k < nvec) write_out(y, k, v[i], lse);
  }
  for (int64_t k = g0 + (int64_t)kLsmCache * kLsmStride; k < nvec; k += kLsmStride) write_out(y, k, x[k], lse);
}

// out[row] = log-probability of ids[row] in row `row`; NaN for an id outside [0, V).
__global__ void __launch_bounds__(kLsmThreads)
    token_logprobs_kernel(const uint4* X, const int32_t* ids, float* out, int64_t nvec) {
  __shared__ LsmShared sh;
  grid_dep_launch_dependents();
  grid_dep_wait();
  const int64_t row = blockIdx.x / kLsmCtas;
  const uint4* x = X + row * nvec;
  uint4 v[kLsmCache];
  const float lse = row_lse(x, nvec, sh, v);
  if (cluster_ctarank() == 0 && threadIdx.x == 0) {
    const int32_t id = ids[row];
    const int64_t V = nvec * 8;
    float r = __int_as_float(0x7fc00000);
    if (id >= 0 && id < V) {
      const uint16_t b = reinterpret_cast<const uint16_t*>(x)[id];
      r = __uint_as_float((uint32_t)b << 16) - lse;
    }
    out[row] = r;
  }
}

// ---------------------------------------------------------------------------
// The same tree on one CTA per row, for many rows
// ---------------------------------------------------------------------------
// A cluster spreads a row over kLsmCtas SMs, which keeps a single row fast;
// with many rows the cluster barriers and the waves of 8-CTA clusters cost
// more than they save.  This variant runs the identical arithmetic on one CTA
// of kLsmCtaThreads threads: thread t plays the cluster's threads t + 1024 j
// (j < kLsmVirt), whose lanes and warps are its own lane and warp (mod 16),
// and every butterfly combines the same pairs in the same order.  Both
// variants give the same bits for every row; which one runs is speed only.
constexpr int kLsmCtaThreads = 1024;
constexpr int kLsmVirt = kLsmCtas * kLsmThreads / kLsmCtaThreads;  // cluster threads per thread
#ifndef BI_LSM_CTA_MIN_ROWS
#define BI_LSM_CTA_MIN_ROWS 64
#endif

struct LsmCtaShared {
  float m[kLsmCtas][kLsmWarps], s[kLsmCtas][kLsmWarps];
  int bad[kLsmCtas][kLsmWarps];
  float cm[kLsmCtas], cs[kLsmCtas];
  int cb[kLsmCtas];
  float lse;
};

__device__ float row_lse_cta(const uint4* x, int64_t nvec, LsmCtaShared& sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
#pragma unroll 1
  for (int j = 0; j < kLsmVirt; ++j) {
    const int g = tid + j * kLsmCtaThreads;   // the cluster thread played
    const int vr = g / kLsmThreads;           // its CTA rank
    const int vw = (g % kLsmThreads) >> 5;    // its warp
    uint4 v[kLsmCache];
    float m = -INFINITY, s = 0.0f;
    bool bad = false;
#pragma unroll
    for (int i = 0; i < kLsmCache; ++i) {
      const int64_t k = g + (int64_t)i * kLsmStride;
      if (k < nvec) {
        v[i] = x[k];
        m = fmaxf(m, max8(v[i]));
        bad = bad || bad8(v[i]);
      }
    }
    for (int64_t k = g + (int64_t)kLsmCache * kLsmStride; k < nvec; k += kLsmStride) {
      const uint4 w = x[k];
      m = fmaxf(m, max8(w));
      bad = bad || bad8(w);
    }
    if (m != -INFINITY) {
#pragma unroll
      for (int i = 0; i < kLsmCache; ++i) {
        const int64_t k = g + (int64_t)i * kLsmStride;
        if (k < nvec) s = sumexp8(v[i], m, s);
      }
      for (int64_t k = g + (int64_t)kLsmCache * kLsmStride; k < nvec; k += kLsmStride) s = sumexp8(x[k], m, s);
    }
    ms_butterfly(m, s, bad);
    if (lane == 0) {
      sh.m[vr][vw] = m;
      sh.s[vr][vw] = s;
      sh.bad[vr][vw] = bad;
    }
  }
  __syncthreads();
  if (warp < kLsmCtas) {  // warp r plays warp 0 of cluster CTA r
    float m = lane < kLsmWarps ? sh.m[warp][lane] : -INFINITY;
    float s = lane < kLsmWarps ? sh.s[warp][lane] : 0.0f;
    bool bad = lane < kLsmWarps ? sh.bad[warp][lane] != 0 : false;
    ms_butterfly(m, s, bad);
    if (lane == 0) {
      sh.cm[warp] = m;
      sh.cs[warp] = s;
      sh.cb[warp] = bad;
    }
  }
  __syncthreads();
  if (warp == 0) {  // warp 0 of cluster CTA 0
    float m = lane < kLsmCtas ? sh.cm[lane] : -INFINITY;
    float s = lane < kLsmCtas ? sh.cs[lane] : 0.0f;
    bool bad = lane < kLsmCtas ? sh.cb[lane] != 0 : false;
    ms_butterfly(m, s, bad);
    if (lane == 0) sh.lse = (bad || m == -INFINITY) ? __int_as_float(0x7fc00000) : m + logf(s);
  }
  __syncthreads();
  return sh.lse;
}

__global__ void __launch_bounds__(kLsmCtaThreads)
    log_softmax_cta_kernel(const uint4* X, float4* Y, int64_t nvec) {
  __shared__ LsmCtaShared sh;
  grid_dep_launch_dependents();
  grid_dep_wait();
  const int64_t row = blockIdx.x;
  const uint4* x = X + row * nvec;
  const float lse = row_lse_cta(x, nvec, sh);
  float4* y = Y + row * nvec * 2;
  for (int64_t k = threadIdx.x; k < nvec; k += kLsmCtaThreads) write_out(y, k, x[k], lse);
}

__global__ void __launch_bounds__(kLsmCtaThreads)
    token_logprobs_cta_kernel(const uint4* X, const int32_t* ids, float* out, int64_t nvec) {
  __shared__ LsmCtaShared sh;
  grid_dep_launch_dependents();
  grid_dep_wait();
  const int64_t row = blockIdx.x;
  const uint4* x = X + row * nvec;
  const float lse = row_lse_cta(x, nvec, sh);
  if (threadIdx.x == 0) {
    const int32_t id = ids[row];
    const int64_t V = nvec * 8;
    float r = __int_as_float(0x7fc00000);
    if (id >= 0 && id < V) {
      const uint16_t b = reinterpret_cast<const uint16_t*>(x)[id];
      r = __uint_as_float((uint32_t)b << 16) - lse;
    }
    out[row] = r;
  }
}

template <typename... KArgs, typename... Args>
static cudaError_t launch_rows(void (*kern)(KArgs...), int64_t M, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(M * kLsmCtas));
  cfg.blockDim = dim3(kLsmThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kLsmCtas;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

cudaError_t launch_log_softmax(const void* X, void* Y, int64_t M, int64_t V, cudaStream_t stream) {
  if (M >= BI_LSM_CTA_MIN_ROWS && M <= 0x7FFFFFFFll)
    return launch_overlapped(log_softmax_cta_kernel, dim3((unsigned)M), dim3(kLsmCtaThreads), stream,
                             static_cast<const uint4*>(X), static_cast<float4*>(Y), V / 8);
  if (M > 0x7FFFFFFFll / kLsmCtas) return cudaErrorInvalidValue;
  return launch_rows(log_softmax_kernel, M, stream, static_cast<const uint4*>(X), static_cast<float4*>(Y),
                     V / 8);
}

cudaError_t launch_token_logprobs(const void* X, const int32_t* ids, float* out, int64_t M, int64_t V,
                                  cudaStream_t stream) {
  if (M >= BI_LSM_CTA_MIN_ROWS && M <= 0x7FFFFFFFll)
    return launch_overlapped(token_logprobs_cta_kernel, dim3((unsigned)M), dim3(kLsmCtaThreads), stream,
                             static_cast<const uint4*>(X), ids, out, V / 8);
  if (M > 0x7FFFFFFFll / kLsmCtas) return cudaErrorInvalidValue;
  return launch_rows(token_logprobs_kernel, M, stream, static_cast<const uint4*>(X), ids, out, V / 8);
}

}  // namespace bi
