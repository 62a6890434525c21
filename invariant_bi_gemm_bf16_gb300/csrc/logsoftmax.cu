// logsoftmax.cu -- batch-invariant log-probabilities of a row of bf16 logits
// (the lm_head output): out_v = x_v - lse, lse = m + log(sum_v exp(x_v - m)),
// m = max_v x_v, all in fp32.
//
// A cluster of kLsmCtas CTAs of kLsmThreads threads per row; the reduction
// tree depends on V only:
//   * the row is read as 16-byte vectors of 8 bf16; thread g = rank *
//     kLsmThreads + t of the cluster owns vectors g, g + G, g + 2G, ...
//     (G = kLsmCtas * kLsmThreads) and folds their elements, in ascending
//     order, into a running pair (m, s): s is the sum of exp(x - m) for the
//     elements seen, rescaled by exp(m_old - m_new) whenever the maximum grows;
//   * pairs combine as m = max(m1, m2), s = s1 exp(m1 - m) + s2 exp(m2 - m):
//     by an xor butterfly (16, 8, 4, 2, 1) within each warp, then the warp
//     results by the same butterfly in warp 0, then the CTA results (read
//     from the cluster's shared memory) by the same butterfly in warp 0 of
//     rank 0; lanes past the count hold the identity (-inf, 0).  The two
//     operands of every combine are the same two pairs in both lanes and IEEE
//     addition commutes, so every lane ends with the same pair;
//   * expf and logf are CUDA's (no fast math).
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

// One logit into the running pair.  With m = -inf (nothing finite seen yet),
// s = 0 and a larger x gives s = 0 * exp(-inf) + 1 = 1.  A -inf logit adds
// exp(-inf) = 0.  A NaN or +Inf logit marks the row undefined.
__device__ __forceinline__ void ms_add(float& m, float& s, bool& bad, float x) {
  if (!(x < INFINITY)) bad = true;  // NaN or +Inf
  if (x > m) {
    s = __fadd_rn(__fmul_rn(s, expf(m - x)), 1.0f);
    m = x;
  } else if (m != -INFINITY) {
    s = __fadd_rn(s, expf(x - m));
  }
}

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

// The row's lse (every thread of the cluster returns it).
__device__ float row_lse(const uint4* x, int64_t nvec, LsmShared& sh) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t rank = cluster_ctarank();
  float m = -INFINITY, s = 0.0f;
  bool bad = false;
  for (int64_t i = (int64_t)rank * kLsmThreads + tid; i < nvec; i += kLsmStride) {
    const uint4 v = x[i];
    ms_add(m, s, bad, lsm_lo(v.x));
    ms_add(m, s, bad, lsm_hi(v.x));
    ms_add(m, s, bad, lsm_lo(v.y));
    ms_add(m, s, bad, lsm_hi(v.y));
    ms_add(m, s, bad, lsm_lo(v.z));
    ms_add(m, s, bad, lsm_hi(v.z));
    ms_add(m, s, bad, lsm_lo(v.w));
    ms_add(m, s, bad, lsm_hi(v.w));
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

// X [M,V] bf16 -> Y [M,V] fp32 log-probabilities; cluster r of the grid is row r.
__global__ void __launch_bounds__(kLsmThreads)
    log_softmax_kernel(const uint4* X, float4* Y, int64_t nvec) {
  __shared__ LsmShared sh;
  grid_dep_launch_dependents();
  grid_dep_wait();  // the logits may come from the previous kernel in the stream
  const int64_t row = blockIdx.x / kLsmCtas;
  const uint4* x = X + row * nvec;
  const float lse = row_lse(x, nvec, sh);
  float4* y = Y + row * nvec * 2;
  for (int64_t i = (int64_t)cluster_ctarank() * kLsmThreads + threadIdx.x; i < nvec; i += kLsmStride) {
    const uint4 v = x[i];
    y[2 * i] = make_float4(lsm_lo(v.x) - lse, lsm_hi(v.x) - lse, lsm_lo(v.y) - lse, lsm_hi(v.y) - lse);
    y[2 * i + 1] = make_float4(lsm_lo(v.z) - lse, lsm_hi(v.z) - lse, lsm_lo(v.w) - lse, lsm_hi(v.w) - lse);
  }
}

// out[row] = log-probability of ids[row] in row `row`; NaN for an id outside [0, V).
__global__ void __launch_bounds__(kLsmThreads)
    token_logprobs_kernel(const uint4* X, const int32_t* ids, float* out, int64_t nvec) {
  __shared__ LsmShared sh;
  grid_dep_launch_dependents();
  grid_dep_wait();
  const int64_t row = blockIdx.x / kLsmCtas;
  const uint4* x = X + row * nvec;
  const float lse = row_lse(x, nvec, sh);
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
  if (M > 0x7FFFFFFFll / kLsmCtas) return cudaErrorInvalidValue;
  return launch_rows(log_softmax_kernel, M, stream, static_cast<const uint4*>(X), static_cast<float4*>(Y),
                     V / 8);
}

cudaError_t launch_token_logprobs(const void* X, const int32_t* ids, float* out, int64_t M, int64_t V,
                                  cudaStream_t stream) {
  if (M > 0x7FFFFFFFll / kLsmCtas) return cudaErrorInvalidValue;
  return launch_rows(token_logprobs_kernel, M, stream, static_cast<const uint4*>(X), ids, out, V / 8);
}

}  // namespace bi
