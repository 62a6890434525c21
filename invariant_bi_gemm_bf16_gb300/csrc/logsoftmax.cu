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
#include <atomic>

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

// m = max(m, m2), s = s exp(m_old - m) + s2 exp(m2 - m).  The side holding
// the maximum is multiplied by exp(0) = 1, which is exact, so only the other
// side's factor is evaluated (the same bits as evaluating both).
__device__ __forceinline__ void ms_combine(float& m, float& s, float m2, float s2) {
  const float mm = fmaxf(m, m2);
  if (mm == -INFINITY) {
    s = 0.0f;
  } else {
    const bool keep = m == mm;                 // this side holds the maximum
    const float e = expf((keep ? m2 : m) - mm);
    s = keep ? __fadd_rn(s, __fmul_rn(s2, e)) : __fadd_rn(__fmul_rn(s, e), s2);
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

// NaN-propagating maxima (exact in any order): a row holding a NaN or a +Inf
// shows it in its maximum, so no separate test of the elements is needed.
__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ float fmax_nan(float a, float b) {
  float d;
  asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
  return d;
}
__device__ __forceinline__ float max8(const uint4& v) {
  const uint32_t w = bmax2_nan(bmax2_nan(v.x, v.y), bmax2_nan(v.z, v.w));
  return fmax_nan(lsm_lo(w), lsm_hi(w));
}
// a maximum from max8 / fmax_nan that marks the row undefined (NaN or +Inf;
// -Inf is an ordinary logit)
__device__ __forceinline__ bool bad_max(float m) { return !(m < INFINITY) && m != -INFINITY; }

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
      m = fmax_nan(m, max8(v[i]));
    }
  }
  for (int64_t k = g0 + (int64_t)kLsmCache * kLsmStride; k < nvec; k += kLsmStride) m = fmax_nan(m, max8(x[k]));
  bad = bad_max(m);
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
// The same tree on a pair of CTAs per row, for many rows
// ---------------------------------------------------------------------------
// A cluster of kLsmCtas CTAs per row keeps a single row fast; with many rows
// its barriers and waves cost more than they save.  This variant runs the
// identical arithmetic on a cluster of two CTAs of kLsmCtaThreads threads:
// thread t of rank r plays the cluster threads g = r * kLsmHalf + t +
// kLsmCtaThreads j (j < kLsmVirt), whose lanes and warps are its own, and
// every butterfly combines the same pairs in the same order (the last one
// reads the other CTA's four results through distributed shared memory).
// Both variants give the same bits for every row; which one runs is speed
// only.
//
// The half row is read from HBM once and kept on chip: cluster thread g's
// vectors g + kLsmStride i for i < 3 in shared memory (96 KB, staged by
// 16-byte asynchronous copies) and its vector i = 3 in a register.  Rows
// longer than kLsmCache * 8 * kLsmStride logits read their further vectors
// from global memory in each pass.
//
// Pair p takes rows p, p + P, p + 2P, ... for a grid of P pairs.  A thread
// stages only its own vectors and reads back only those, so as soon as it
// has written a slot's outputs (or, for the token variant, finished its sums)
// it copies the next row's vector into that slot: the next row's loads
// overlap this row's stores and reductions.  The token variant runs one pair
// per SM from kLsmPersistRows rows (M = 256: 23.2 against 25.6 us with a
// pair per row; M = 1024: 68.1 against 76.9).  Full rows run one pair per
// row, the loop once: persistent pairs move in step, all reducing at once
// while HBM idles, and took longer (M = 256: 56.8 against 55.2 us; M = 1024:
// 171 against 161), where pairs that start wave by wave drift apart and fill
// each other's gaps.
constexpr int kLsmCtaThreads = 512;
constexpr int kLsmHalf = kLsmCtas * kLsmThreads / 2;                 // cluster threads per CTA
constexpr int kLsmVirt = kLsmHalf / kLsmCtaThreads;                   // cluster threads per thread
constexpr int kLsmSmemVec = (kLsmCache - 1) * kLsmHalf;              // vectors i < 3 of the CTA's threads
constexpr int kLsmSmemBytes = kLsmSmemVec * 16;
static_assert(kLsmVirt * 2 == kLsmCtas && kLsmThreads == kLsmCtaThreads, "rank j of the cluster is played as 4r + j");
#ifndef BI_LSM_CTA_MIN_ROWS
#define BI_LSM_CTA_MIN_ROWS 128  // measured: 8-CTA clusters win below (M = 96: 28 against 31 us)
#endif
constexpr int64_t kLsmPersistRows = 256;  // token variant: one pair per SM from this many rows

struct LsmPairShared {
  float m[kLsmVirt][kLsmWarps], s[kLsmVirt][kLsmWarps];
  int bad[kLsmVirt][kLsmWarps];
  float cm[kLsmVirt], cs[kLsmVirt], cb[kLsmVirt];  // cb: 1.0f if that cluster CTA saw a NaN or +Inf
  float lse;
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

// Holds until the thread's load of v has completed (before a copy may
// rewrite the shared-memory slot v came from).
__device__ __forceinline__ void lsm_consumed(const uint4& v) {
  asm volatile("" ::"r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

template <bool FULL>
__global__ void __launch_bounds__(kLsmCtaThreads, 2)
    lsm_rows_kernel(const uint4* __restrict__ X, float4* __restrict__ Y, const int32_t* ids, float* out,
                    int64_t nvec, int64_t M) {
  extern __shared__ __align__(16) uint4 lsm_row[];
  __shared__ LsmPairShared sh;
  grid_dep_launch_dependents();
  grid_dep_wait();  // the logits may come from the previous kernel in the stream
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint32_t rank = cluster_ctarank();
  const int64_t pairs = gridDim.x >> 1;
  const int64_t g0 = (int64_t)rank * kLsmHalf;  // this CTA's first cluster thread
  const int64_t per = (nvec + kLsmStride - 1) / kLsmStride;  // vectors of cluster thread 0
  int nvs[kLsmVirt];  // vectors of each played cluster thread (the same for every row)
#pragma unroll
  for (int j = 0; j < kLsmVirt; ++j) {
    const int64_t g = g0 + t + j * kLsmCtaThreads;
    nvs[j] = (int)(per - (g >= nvec - (per - 1) * kLsmStride ? 1 : 0));
  }
  // the first row: vectors i < 3 into shared memory, i = 3 into registers
  int64_t row = blockIdx.x >> 1;
  uint4 r[kLsmVirt];
  {
    const uint4* x = X + row * nvec;
#pragma unroll
    for (int i = 0; i < kLsmCache - 1; ++i)
#pragma unroll
      for (int j = 0; j < kLsmVirt; ++j) {
        const int h = t + j * kLsmCtaThreads;
        if (i < nvs[j]) cp_async16(smem_u32(lsm_row + i * kLsmHalf + h), x + g0 + h + (int64_t)i * kLsmStride);
      }
    asm volatile("cp.async.commit_group;" ::: "memory");
#pragma unroll
    for (int j = 0; j < kLsmVirt; ++j)
      r[j] = nvs[j] >= kLsmCache ? __ldg(x + g0 + t + j * kLsmCtaThreads + (int64_t)(kLsmCache - 1) * kLsmStride)
                                 : make_uint4(0, 0, 0, 0);
  }
  for (; row < M; row += pairs) {
    const uint4* x = X + row * nvec;
    const int64_t next = row + pairs;
    const uint4* xn = X + (next < M ? next : row) * nvec;
    asm volatile("cp.async.wait_group 0;" ::: "memory");  // this thread's copies of the row have landed
#pragma unroll
    for (int j = 0; j < kLsmVirt; ++j) {
      const int h = t + j * kLsmCtaThreads;
      const int64_t g = g0 + h;
      const int nv = nvs[j];
      // vectors i < 3 (shared memory), i = 3 (register), i >= 4 (global), in order
      float m = -INFINITY, s = 0.0f;
#pragma unroll
      for (int i = 0; i < kLsmCache - 1; ++i)
        if (i < nv) m = fmax_nan(m, max8(lsm_row[i * kLsmHalf + h]));
      if (nv >= kLsmCache) m = fmax_nan(m, max8(r[j]));
      for (int i = kLsmCache; i < nv; ++i) m = fmax_nan(m, max8(__ldg(x + g + (int64_t)i * kLsmStride)));
      bool bad = bad_max(m);
      if (m != -INFINITY) {
#pragma unroll
        for (int i = 0; i < kLsmCache - 1; ++i)
          if (i < nv) s = sumexp8(lsm_row[i * kLsmHalf + h], m, s);
        if (nv >= kLsmCache) s = sumexp8(r[j], m, s);
        for (int i = kLsmCache; i < nv; ++i) s = sumexp8(__ldg(x + g + (int64_t)i * kLsmStride), m, s);
      }
      if (!FULL && next < M) {
        // the token variant is done with the staged row (m holds every
        // staged value's maximum, so every load has completed): stage the next one
        asm volatile("" ::"f"(m) : "memory");
#pragma unroll
        for (int i = 0; i < kLsmCache - 1; ++i)
          if (i < nv) cp_async16(smem_u32(lsm_row + i * kLsmHalf + h), xn + g + (int64_t)i * kLsmStride);
        if (nv >= kLsmCache) r[j] = __ldg(xn + g + (int64_t)(kLsmCache - 1) * kLsmStride);
      }
      ms_butterfly(m, s, bad);
      if (lane == 0) {  // cluster CTA 4 rank + j, warp `warp`
        sh.m[j][warp] = m;
        sh.s[j][warp] = s;
        sh.bad[j][warp] = bad;
      }
    }
    if (!FULL) asm volatile("cp.async.commit_group;" ::: "memory");
    __syncthreads();
    if (warp < kLsmVirt) {  // warp j plays warp 0 of cluster CTA 4 rank + j
      float m = lane < kLsmWarps ? sh.m[warp][lane] : -INFINITY;
      float s = lane < kLsmWarps ? sh.s[warp][lane] : 0.0f;
      bool bad = lane < kLsmWarps ? sh.bad[warp][lane] != 0 : false;
      ms_butterfly(m, s, bad);
      if (lane == 0) {
        sh.cm[warp] = m;
        sh.cs[warp] = s;
        sh.cb[warp] = bad ? 1.0f : 0.0f;
      }
    }
    cluster_sync();  // both CTAs' results are in their shared memory
    if (rank == 0 && warp == 0) {  // warp 0 of cluster CTA 0
      float m = -INFINITY, s = 0.0f;
      bool bad = false;
      if (lane < kLsmCtas) {
        const uint32_t src = (uint32_t)(lane / kLsmVirt), w = (uint32_t)(lane % kLsmVirt);
        m = ld_dsmem_f32(mapa_shared(smem_u32(&sh.cm[w]), src));
        s = ld_dsmem_f32(mapa_shared(smem_u32(&sh.cs[w]), src));
        bad = ld_dsmem_f32(mapa_shared(smem_u32(&sh.cb[w]), src)) != 0.0f;
      }
      ms_butterfly(m, s, bad);
      if (lane == 0) sh.lse = (bad || m == -INFINITY) ? __int_as_float(0x7fc00000) : m + logf(s);
    }
    cluster_sync();  // rank 0 has the lse
    const float lse = ld_dsmem_f32(mapa_shared(smem_u32(&sh.lse), 0u));
    cluster_sync();  // the lse is read everywhere before the next row rewrites the pairs
    if constexpr (FULL) {
      float4* y = Y + row * nvec * 2;
#pragma unroll
      for (int j = 0; j < kLsmVirt; ++j) {
        const int h = t + j * kLsmCtaThreads;
        const int64_t g = g0 + h;
        const int nv = nvs[j];
        auto put = [&](const uint4& v, int i) {
          const int64_t k = g + (int64_t)i * kLsmStride;
          __stcs(y + 2 * k, make_float4(lsm_lo(v.x) - lse, lsm_hi(v.x) - lse, lsm_lo(v.y) - lse, lsm_hi(v.y) - lse));
          __stcs(y + 2 * k + 1,
                 make_float4(lsm_lo(v.z) - lse, lsm_hi(v.z) - lse, lsm_lo(v.w) - lse, lsm_hi(v.w) - lse));
        };
#pragma unroll
        for (int i = 0; i < kLsmCache - 1; ++i)
          if (i < nv) {
            const uint4 v = lsm_row[i * kLsmHalf + h];
            put(v, i);
            if (next < M) {  // the slot is free: stage the next row's vector
              lsm_consumed(v);
              cp_async16(smem_u32(lsm_row + i * kLsmHalf + h), xn + g + (int64_t)i * kLsmStride);
            }
          }
        if (nv >= kLsmCache) {
          put(r[j], kLsmCache - 1);
          if (next < M) r[j] = __ldg(xn + g + (int64_t)(kLsmCache - 1) * kLsmStride);
        }
        for (int i = kLsmCache; i < nv; ++i) put(__ldg(x + g + (int64_t)i * kLsmStride), i);
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    } else if (rank == 0 && t == 0) {
      const int32_t id = ids[row];
      const int64_t V = nvec * 8;
      float res = __int_as_float(0x7fc00000);
      if (id >= 0 && id < V) {
        const uint16_t b = reinterpret_cast<const uint16_t*>(x)[id];
        res = __uint_as_float((uint32_t)b << 16) - lse;
      }
      out[row] = res;
    }
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");  // no copy outlives the block
}

template <bool FULL>
static cudaError_t launch_lsm_rows(const void* X, void* Y, const int32_t* ids, float* out, int64_t M, int64_t V,
                                   cudaStream_t stream) {
  // the shared-memory limit is per device: set it once for each
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t)1 << dev : 0;
  if (!bit || !(configured.load() & bit)) {
    e = cudaFuncSetAttribute(lsm_rows_kernel<FULL>, cudaFuncAttributeMaxDynamicSharedMemorySize, kLsmSmemBytes);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  // pairs: one per row, or for the token variant from kLsmPersistRows rows
  // one per SM (two CTAs of a pair's size fit on an SM)
  int sms = 0;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int64_t pairs = (!FULL && M >= kLsmPersistRows && M > sms) ? sms : M;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * pairs));
  cfg.blockDim = dim3(kLsmCtaThreads);
  cfg.dynamicSmemBytes = kLsmSmemBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, lsm_rows_kernel<FULL>, static_cast<const uint4*>(X), static_cast<float4*>(Y), ids,
                            out, V / 8, M);
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
  if (M >= BI_LSM_CTA_MIN_ROWS && M <= 0x7FFFFFFFll / 2)
    return launch_lsm_rows<true>(X, Y, nullptr, nullptr, M, V, stream);
  if (M > 0x7FFFFFFFll / kLsmCtas) return cudaErrorInvalidValue;
  return launch_rows(log_softmax_kernel, M, stream, static_cast<const uint4*>(X), static_cast<float4*>(Y),
                     V / 8);
}

cudaError_t launch_token_logprobs(const void* X, const int32_t* ids, float* out, int64_t M, int64_t V,
                                  cudaStream_t stream) {
  if (M >= BI_LSM_CTA_MIN_ROWS && M <= 0x7FFFFFFFll / 2)
    return launch_lsm_rows<false>(X, nullptr, ids, out, M, V, stream);
  if (M > 0x7FFFFFFFll / kLsmCtas) return cudaErrorInvalidValue;
  return launch_rows(token_logprobs_kernel, M, stream, static_cast<const uint4*>(X), ids, out, V / 8);
}

}  // namespace bi
