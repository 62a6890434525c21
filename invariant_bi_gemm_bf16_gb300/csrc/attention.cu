// attention.cu -- batch-invariant decode attention over a paged key/value
// cache: one query token per request, grouped-query heads, the request's
// positions split at fixed multiples of a pinned split size.
//
// Detent (Batch-Invariant LLM Serving and RL Rollouts at Near-Stock Speed),
// Sec. 7 (Kernels): split-KV is kept, but a request's split boundaries follow
// a fixed split size, so they never depend on the batch.  LLM-42, Sec. 4.4,
// and CoRun, Sec. IV-B, get the same invariance by disabling the split; a
// fixed split size keeps the parallelism of a long context and still gives
// every request a tree of its own.
//
// The reduction tree of query head h of request b, a function of the
// request's length L, the split size and the head dimension only:
//   * split s covers positions [s*S, min((s+1)*S, L));
//   * within a split, tiles of 64 positions in ascending order; warp w of the
//     CTA owns positions 16w .. 16w+15 of every tile and keeps a running
//     (max m, sum l, unnormalised output o) over them: per tile, the scores
//     t = (q . k) * scale * log2(e) (fp32 MMA accumulation over d in
//     ascending 16-wide steps), m' = max(m, max t), then o and l are scaled
//     by 2^(m - m'), p = 2^(t - m') is rounded to bf16, l gains the sum of
//     the rounded p, and o gains p . v (fp32 MMA accumulation);
//   * per-lane partial sums of l are added by a fixed xor butterfly;
//   * the four warps' states fold in warp order, then the splits' states
//     fold in split order, both with
//       m = max(m1, m2), a_i = 2^(m_i - m), l = l1 a1 + l2 a2, o = o1 a1 + o2 a2;
//   * out = bf16_rne(o / l).
// No other request, and no batch size, reaches any of these steps.
#include <cuda_bf16.h>

#include "attention.h"
#include "internal.h"
#include "ptx.cuh"

namespace bi {

constexpr int kAttnD = 128;                             // head dimension
constexpr int kAttnTile = 64;                           // positions per staged tile
constexpr int kAttnCWarps = 4;                          // compute warps (16 positions of a tile each)
constexpr int kAttnThreads = 32 * (kAttnCWarps + 1);    // + one copy warp
// Ring depth and resident CTAs per SM, for up to 8 query heads per group
// (NT = 1) and for 9 to 16 (NT = 2, more registers per thread).  Speed only.
#ifndef BI_ATTN_STAGES_NT1
#define BI_ATTN_STAGES_NT1 2
#endif
#ifndef BI_ATTN_CTAS_NT1
#define BI_ATTN_CTAS_NT1 3
#endif
#ifndef BI_ATTN_STAGES_NT2
#define BI_ATTN_STAGES_NT2 3
#endif
#ifndef BI_ATTN_CTAS_NT2
#define BI_ATTN_CTAS_NT2 2
#endif
template <int NT> struct AttnCfg;
template <> struct AttnCfg<1> { static constexpr int stages = BI_ATTN_STAGES_NT1, ctas = BI_ATTN_CTAS_NT1; };
template <> struct AttnCfg<2> { static constexpr int stages = BI_ATTN_STAGES_NT2, ctas = BI_ATTN_CTAS_NT2; };
constexpr int kAttnHalfBytes = kAttnTile * 128;         // 64 positions x 64 values
constexpr int kAttnKVBytes = 2 * kAttnHalfBytes;        // 64 positions x 128 values
constexpr int kAttnStageBytes = 2 * kAttnKVBytes;       // K tile, then V tile
template <int NT>
constexpr int attn_smem_bytes() { return AttnCfg<NT>::stages * kAttnStageBytes + 1024; }
constexpr int kAttnMaxSplitPages = BI_ATTN_MAX_SPLIT / 8 + 1;
constexpr uint64_t kAttnWaitNs = 2000000000ull;

__device__ __forceinline__ void attn_flag(int* status, int code) { atomicCAS(status, 0, code); }

// Waits for the phase of `parity` on `bar`; false once the CTA gives up (this
// wait ran 2 s, or another warp gave up).
__device__ __noinline__ bool attn_wait_slow(uint32_t bar, uint32_t parity, volatile int* abort,
                                            int* status) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > kAttnWaitNs) {
      *abort = 1;
      attn_flag(status, (int)BI_ERR_DEVICE_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ bool attn_wait(uint32_t bar, uint32_t parity, volatile int* abort, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  return attn_wait_slow(bar, parity, abort, status);
}

// Bounded wait that ignores the abort flag (for copies still in flight).
__device__ __noinline__ void attn_drain(uint32_t bar, uint32_t parity, int* status) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kAttnWaitNs) {
      attn_flag(status, (int)BI_ERR_DEVICE_TIMEOUT);
      return;
    }
  }
}

__device__ __forceinline__ uint32_t pack_bf16(__nv_bfloat16 lo, __nv_bfloat16 hi) {
  return (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
}

// The fold of two running states (one column of o).
__device__ __forceinline__ void attn_scales(float m1, float m2, float& m, float& a1, float& a2) {
  m = fmaxf(m1, m2);
  a1 = (m1 == m) ? 1.0f : exp2f(__fsub_rn(m1, m));
  a2 = (m2 == m) ? 1.0f : exp2f(__fsub_rn(m2, m));
}

// One CTA per (key/value head, split s, request): the running state of the
// split's positions, written as a partial record.
template <int NT>
__global__ void __launch_bounds__(kAttnThreads, AttnCfg<NT>::ctas)
    decode_attn_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                             const AttnParams p) {
  constexpr int GP = 8 * NT;  // query-head columns of the MMAs (G <= GP)
  constexpr int kAttnStages = AttnCfg<NT>::stages;
  extern __shared__ uint8_t attn_smem_raw[];
  __shared__ __align__(8) uint64_t full[kAttnStages];
  __shared__ __align__(8) uint64_t empty[kAttnStages];
  __shared__ int32_t pages[kAttnMaxSplitPages];
  __shared__ int abort_flag;

  grid_dep_launch_dependents();
  grid_dep_wait();  // q and the cache may come from the previous kernel in the stream

  // The heads of one (request, split) are neighbours in the grid: they run
  // together and read the same cache rows (each its 256 bytes of a row).
  const int kvh = blockIdx.x, s = blockIdx.y;
  const int64_t b = blockIdx.z;
  const int64_t L = p.seq_lens[b];
  if (L < 0 || L > p.max_len) {
    if (threadIdx.x == 0 && s == 0 && kvh == 0) attn_flag(p.status, (int)BI_ERR_INVALID_ARG);
    return;
  }
  const int64_t p0 = (int64_t)s * p.split_size;
  if (p0 >= L) return;  // past the request's end: nothing to do
  const int64_t p1 = min(p0 + (int64_t)p.split_size, L);
  const int n_tiles = (int)((p1 - p0 + kAttnTile - 1) / kAttnTile);
  const uint32_t base = (smem_u32(attn_smem_raw) + 1023u) & ~1023u;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int* abort = &abort_flag;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kAttnStages; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), kAttnCWarps);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp == kAttnCWarps) {
    // ---------------- copy warp: the split's page ids, then the K/V tiles
    const int64_t first_page = p0 / p.page_size;
    const int n_pages = (int)((p1 - 1) / p.page_size - first_page + 1);
    const int64_t rows = p.num_pages * p.page_size;
    for (int i = lane; i < n_pages; i += 32) {
      int32_t pg = p.block_table[b * p.bt_stride + first_page + i];
      if (pg < 0 || (int64_t)pg >= p.num_pages) {
        attn_flag(p.status, (int)BI_ERR_INVALID_ARG);
        pg = -1;  // loaded from past the cache's end: zeros
      }
      pages[i] = pg;
    }
    __syncwarp();
    if (lane == 0) {
      int issued = 0;
      for (int t = 0; t < n_tiles; ++t) {
        const int st = t % kAttnStages;
        if (t >= kAttnStages &&
            !attn_wait(smem_u32(&empty[st]), ((t / kAttnStages) - 1) & 1, abort, p.status))
          break;
        const int64_t tp = p0 + (int64_t)t * kAttnTile;
        int boxes = 0;
        for (int r = 0; r < kAttnTile && tp + r < p1; r += p.box_rows) ++boxes;
        const uint32_t fb = smem_u32(&full[st]);
        mbar_arrive_expect_tx(fb, (uint32_t)(boxes * p.box_rows * 128 * 4));
        const uint32_t kdst = base + (uint32_t)st * kAttnStageBytes;
        for (int r = 0; r < kAttnTile && tp + r < p1; r += p.box_rows) {
          const int64_t pos = tp + r;
          const int32_t pg = pages[pos / p.page_size - first_page];
          const int32_t y = pg < 0 ? (int32_t)rows : (int32_t)((int64_t)pg * p.page_size + pos % p.page_size);
          const int32_t x = kvh * kAttnD;
          const uint32_t off = (uint32_t)r * 128u;
          tma_load_2d(kdst + off, &tmK, fb, x, y);
          tma_load_2d(kdst + kAttnHalfBytes + off, &tmK, fb, x + 64, y);
          tma_load_2d(kdst + kAttnKVBytes + off, &tmV, fb, x, y);
          tma_load_2d(kdst + kAttnKVBytes + kAttnHalfBytes + off, &tmV, fb, x + 64, y);
        }
        ++issued;
      }
      // every copy issued has landed before the CTA may end
      for (int t = issued > kAttnStages ? issued - kAttnStages : 0; t < issued; ++t)
        attn_drain(smem_u32(&full[t % kAttnStages]), (t / kAttnStages) & 1, p.status);
    }
    return;
  }

  // ---------------- compute warps
  const int g = lane >> 2, c = lane & 3;
  // q as the MMA's B operand (k = d, n = query head of the group): lane holds
  // q[head g][d = 16 ks + 2c, +1] and [.. + 8, + 9] for every 16-wide step ks.
  uint32_t qf[NT][8][2];
  const __nv_bfloat16* qg = static_cast<const __nv_bfloat16*>(p.q) + (b * p.Hq + (int64_t)kvh * p.G) * kAttnD;
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    const int h = j * 8 + g;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t lo = 0, hi = 0;
      if (h < p.G) {
        const uint32_t* qr = reinterpret_cast<const uint32_t*>(qg + (int64_t)h * kAttnD + ks * 16 + 2 * c);
        lo = qr[0];
        hi = qr[4];
      }
      qf[j][ks][0] = lo;
      qf[j][ks][1] = hi;
    }
  }

  // Running state.  o is o^T [d][head]: o[i][j] covers d = 16 i + g (+ 8) and
  // heads 8 j + 2c (+ 1); m and l are per head column (2c, 2c + 1).
  float m[NT][2], l[NT][2], o[8][NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    m[j][0] = m[j][1] = -INFINITY;
    l[j][0] = l[j][1] = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) o[i][j][0] = o[i][j][1] = o[i][j][2] = o[i][j][3] = 0.0f;
  }

  const int row0 = warp * 16;
  for (int t = 0; t < n_tiles; ++t) {
    const int st = t % kAttnStages;
    if (!attn_wait(smem_u32(&full[st]), (t / kAttnStages) & 1, abort, p.status)) break;
    const uint32_t kb = base + (uint32_t)st * kAttnStageBytes, vb = kb + kAttnKVBytes;
    const int64_t tp = p0 + (int64_t)t * kAttnTile + row0;  // position of this warp's first row
    if (tp < p1) {
      if (tp + 16 > p1) {
        // The request ends inside these rows: the cache past L is not ours to
        // read (stale values, Inf, NaN), so its V rows become zeros; its
        // scores are masked below.
        const int bad0 = (int)(p1 - tp);
        for (int i = lane; i < (16 - bad0) * 16; i += 32) {
          const int rr = row0 + bad0 + i / 16, ch = i % 16;
          const uint32_t a = vb + (uint32_t)(ch / 8) * kAttnHalfBytes + (uint32_t)rr * 128u + (uint32_t)(ch % 8) * 16u;
          asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u) : "memory");
        }
        fence_proxy_async_smem();
        __syncwarp();
      }

      // scores^T [16 positions][GP heads] = K . q^T
      float acc[NT][4];
#pragma unroll
      for (int j = 0; j < NT; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.0f;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const int row = row0 + (lane & 15);
        const int chunk = ((ks & 3) << 1) + (lane >> 4);
        uint32_t a[4];
        ldmatrix_x4(a, kb + (uint32_t)(ks >> 2) * kAttnHalfBytes + (uint32_t)row * 128u +
                           (uint32_t)((chunk ^ (row & 7)) << 4));
#pragma unroll
        for (int j = 0; j < NT; ++j) mma_m16n8k16_bf16(acc[j], a, qf[j][ks][0], qf[j][ks][1]);
      }

      // online softmax over the 16 positions, then p^T as the B operand of p . v
      const bool ok0 = tp + g < p1, ok1 = tp + g + 8 < p1;
      uint32_t pb[NT][2];
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        __nv_bfloat16 r[2][2];  // [column][row g, g + 8]
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const float t0 = ok0 ? __fmul_rn(acc[j][cc], p.qk_log2) : -INFINITY;
          const float t1 = ok1 ? __fmul_rn(acc[j][2 + cc], p.qk_log2) : -INFINITY;
          float mx = fmaxf(t0, t1);
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float mn = fmaxf(m[j][cc], mx);
          const float alpha = (mn == m[j][cc]) ? 1.0f : exp2f(__fsub_rn(m[j][cc], mn));
          const float e0 = (mn == -INFINITY) ? 0.0f : exp2f(__fsub_rn(t0, mn));
          const float e1 = (mn == -INFINITY) ? 0.0f : exp2f(__fsub_rn(t1, mn));
          r[cc][0] = __float2bfloat16_rn(e0);
          r[cc][1] = __float2bfloat16_rn(e1);
          l[j][cc] = __fadd_rn(__fmul_rn(l[j][cc], alpha),
                               __fadd_rn(__bfloat162float(r[cc][0]), __bfloat162float(r[cc][1])));
          m[j][cc] = mn;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            o[i][j][cc] = __fmul_rn(o[i][j][cc], alpha);
            o[i][j][2 + cc] = __fmul_rn(o[i][j][2 + cc], alpha);
          }
        }
        pb[j][0] = movmatrix_trans(pack_bf16(r[0][0], r[1][0]));
        pb[j][1] = movmatrix_trans(pack_bf16(r[0][1], r[1][1]));
      }

      // o^T [128 d][GP heads] += V^T . p^T
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int row = row0 + (lane & 7) + ((lane >> 4) << 3);
        const int chunk = ((i & 3) << 1) + ((lane >> 3) & 1);
        uint32_t a[4];
        ldmatrix_x4_trans(a, vb + (uint32_t)(i >> 2) * kAttnHalfBytes + (uint32_t)row * 128u +
                                 (uint32_t)((chunk ^ (row & 7)) << 4));
#pragma unroll
        for (int j = 0; j < NT; ++j) mma_m16n8k16_bf16(o[i][j], a, pb[j][0], pb[j][1]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[st]));
  }

  // l: the eight lanes of a column hold partial sums over their rows
#pragma unroll
  for (int j = 0; j < NT; ++j)
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      l[j][cc] = __fadd_rn(l[j][cc], __shfl_xor_sync(0xffffffffu, l[j][cc], 4));
      l[j][cc] = __fadd_rn(l[j][cc], __shfl_xor_sync(0xffffffffu, l[j][cc], 8));
      l[j][cc] = __fadd_rn(l[j][cc], __shfl_xor_sync(0xffffffffu, l[j][cc], 16));
    }

  // Fold the four warps in order through shared memory (the ring is idle now).
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kAttnCWarps) : "memory");
  if (*abort) return;  // the call was abandoned: the output is unspecified
  constexpr int NR = 8 * NT * 4 + 4 * NT;  // floats of state per lane
  float* scratch = reinterpret_cast<float*>(attn_smem_raw + (base - smem_u32(attn_smem_raw)));
  if (warp > 0) {
    float* w = scratch + (warp - 1) * NR * 32 + lane;
    int r = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) w[32 * r++] = o[i][j][e];
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        w[32 * r++] = m[j][cc];
        w[32 * r++] = l[j][cc];
      }
  }
  asm volatile("bar.sync 1, %0;" ::"n"(32 * kAttnCWarps) : "memory");
  if (warp > 0) return;
  for (int src = 0; src < kAttnCWarps - 1; ++src) {
    const float* w = scratch + src * NR * 32 + lane;
    float a1[NT][2], a2[NT][2];
    int r = 8 * NT * 4;
#pragma unroll
    for (int j = 0; j < NT; ++j)
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const float m2 = w[32 * r++], l2 = w[32 * r++];
        float mm;
        attn_scales(m[j][cc], m2, mm, a1[j][cc], a2[j][cc]);
        l[j][cc] = __fadd_rn(__fmul_rn(l[j][cc], a1[j][cc]), __fmul_rn(l2, a2[j][cc]));
        m[j][cc] = mm;
      }
    r = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float o2 = w[32 * r++];
          o[i][j][e] = __fadd_rn(__fmul_rn(o[i][j][e], a1[j][e & 1]), __fmul_rn(o2, a2[j][e & 1]));
        }
  }

  // The split's record: o^T [D][GP], then m [GP], then l [GP].
  float* rec = p.part + ((b * p.Hkv + kvh) * (int64_t)p.n_split + s) * (int64_t)((kAttnD + 2) * GP);
#pragma unroll
  for (int i = 0; i < 8; ++i)
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int d = 16 * i + g, h = 8 * j + 2 * c;
      *reinterpret_cast<float2*>(rec + d * GP + h) = make_float2(o[i][j][0], o[i][j][1]);
      *reinterpret_cast<float2*>(rec + (d + 8) * GP + h) = make_float2(o[i][j][2], o[i][j][3]);
    }
  if (g == 0) {
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int h = 8 * j + 2 * c;
      *reinterpret_cast<float2*>(rec + kAttnD * GP + h) = make_float2(m[j][0], m[j][1]);
      *reinterpret_cast<float2*>(rec + kAttnD * GP + GP + h) = make_float2(l[j][0], l[j][1]);
    }
  }
}

// One CTA per (key/value head, request): folds the request's split records
// in split order and writes out[b][h][d] for the group's heads.  Thread t owns
// head h = t % GP and the values d = t / GP + (256 / GP) i; the records come
// into shared memory kCombChunk at a time by bulk copy, double-buffered, so
// the fold runs at shared-memory speed.
constexpr int kCombThreads = 256;
constexpr int kCombChunk = 8;

template <int NT>
constexpr int comb_smem_bytes() {
  return 2 * kCombChunk * (kAttnD + 2) * 8 * NT * 4 + 16;
}

template <int NT>
__global__ void __launch_bounds__(kCombThreads) decode_attn_combine_kernel(const AttnParams p, __nv_bfloat16* out) {
  constexpr int GP = 8 * NT;
  constexpr int RS = (kAttnD + 2) * GP;            // floats per record
  constexpr int DSTEP = kCombThreads / GP;         // distance between a thread's d values
  constexpr int DPT = kAttnD / DSTEP;              // d values per thread
  extern __shared__ __align__(16) float comb_smem[];
  __shared__ __align__(8) uint64_t bars[2];
  grid_dep_launch_dependents();
  grid_dep_wait();  // the split records come from the previous kernel
  const int kvh = blockIdx.x, t = threadIdx.x, h = t % GP, d0 = t / GP;
  const int64_t b = blockIdx.y;
  const int64_t L = p.seq_lens[b];
  __nv_bfloat16* ob = out + (b * p.Hq + (int64_t)kvh * p.G + h) * kAttnD;
  if (L <= 0 || L > p.max_len) {
    // an empty request gives zeros; an invalid length (flagged by the split
    // kernel) gives NaN
    if (h < p.G) {
      const __nv_bfloat16 v = __float2bfloat16_rn(L == 0 ? 0.0f : __int_as_float(0x7fc00000));
#pragma unroll
      for (int i = 0; i < DPT; ++i) ob[d0 + DSTEP * i] = v;
    }
    return;
  }
  const int ns = (int)((L + p.split_size - 1) / p.split_size);
  const int nchunks = (ns + kCombChunk - 1) / kCombChunk;
  const float* rec0 = p.part + (b * p.Hkv + kvh) * (int64_t)p.n_split * RS;
  if (t == 0) {
    mbar_init(smem_u32(&bars[0]), 1);
    mbar_init(smem_u32(&bars[1]), 1);
    fence_mbar_init();
  }
  __syncthreads();
  auto issue = [&](int c) {
    const int n = min(kCombChunk, ns - c * kCombChunk);
    const uint32_t bar = smem_u32(&bars[c & 1]);
    mbar_arrive_expect_tx(bar, (uint32_t)(n * RS * 4));
    bulk_load(smem_u32(comb_smem + (c & 1) * kCombChunk * RS), rec0 + (int64_t)c * kCombChunk * RS,
              (uint32_t)(n * RS * 4), bar);
  };
  if (t == 0) {
    issue(0);
    if (nchunks > 1) issue(1);
  }
  float m = 0.0f, l = 0.0f, o[DPT];
  bool ok = true;
  for (int c = 0; c < nchunks; ++c) {
    const uint32_t bar = smem_u32(&bars[c & 1]);
    if (!mbar_try_wait(bar, (c >> 1) & 1)) {
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(bar, (c >> 1) & 1)) {
        if (globaltimer_ns() - t0 > kAttnWaitNs) {
          ok = false;
          break;
        }
      }
    }
    if (!__syncthreads_and(ok)) {
      if (t == 0) attn_flag(p.status, (int)BI_ERR_DEVICE_TIMEOUT);
      // the other buffer's copy, if one was issued, must land before the CTA ends
      if (t == 0 && c + 1 < nchunks) attn_drain(smem_u32(&bars[(c + 1) & 1]), ((c + 1) >> 1) & 1, p.status);
      return;
    }
    const float* buf = comb_smem + (c & 1) * kCombChunk * RS;
    const int n = min(kCombChunk, ns - c * kCombChunk);
    for (int r = 0; r < n; ++r) {
      const float* rec = buf + r * RS;
      const float m2 = rec[kAttnD * GP + h], l2 = rec[kAttnD * GP + GP + h];
      if (c == 0 && r == 0) {
        m = m2;
        l = l2;
#pragma unroll
        for (int i = 0; i < DPT; ++i) o[i] = rec[t + kCombThreads * i];
      } else {
        float mm, a1, a2;
        attn_scales(m, m2, mm, a1, a2);
        l = __fadd_rn(__fmul_rn(l, a1), __fmul_rn(l2, a2));
#pragma unroll
        for (int i = 0; i < DPT; ++i) o[i] = __fadd_rn(__fmul_rn(o[i], a1), __fmul_rn(rec[t + kCombThreads * i], a2));
        m = mm;
      }
    }
    __syncthreads();  // the buffer is read by everyone before it is refilled
    if (t == 0 && c + 2 < nchunks) issue(c + 2);
  }
  if (h < p.G) {
#pragma unroll
    for (int i = 0; i < DPT; ++i) ob[d0 + DSTEP * i] = __float2bfloat16_rn(__fdiv_rn(o[i], l));
  }
}

template <int NT>
static cudaError_t launch_attn_t(const AttnLaunch& A) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(decode_attn_split_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         attn_smem_bytes<NT>());
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(decode_attn_combine_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             comb_smem_bytes<NT>());
    if (e != cudaSuccess) return e;
    configured = true;
  }
  if (A.p.n_split > 0) {
    cudaError_t e = launch_overlapped_smem(decode_attn_split_kernel<NT>,
                                           dim3((unsigned)A.p.Hkv, (unsigned)A.p.n_split, (unsigned)A.B),
                                           dim3(kAttnThreads), attn_smem_bytes<NT>(), A.stream, A.tmK, A.tmV, A.p);
    if (e != cudaSuccess) return e;
  }
  return launch_overlapped_smem(decode_attn_combine_kernel<NT>, dim3((unsigned)A.p.Hkv, (unsigned)A.B),
                                dim3(kCombThreads), comb_smem_bytes<NT>(), A.stream, A.p, A.out);
}

cudaError_t launch_decode_attention(const AttnLaunch& A) {
  return A.p.G <= 8 ? launch_attn_t<1>(A) : launch_attn_t<2>(A);
}

}  // namespace bi
