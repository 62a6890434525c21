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
//   * one warp runs a split alone, over steps of 32 positions in ascending
//     order, keeping a running (max m, sum l, unnormalised output o): per
//     step, the scores t = (q . k) * scale * log2(e) (fp32 MMA accumulation
//     over d in ascending 16-wide steps), m' = max(m, max t), then o and l
//     are scaled by 2^(m - m'), p = 2^(t - m') (ex2.approx) is rounded to
//     bf16, l gains the sum of the rounded p (ascending position within a
//     lane: rows g, g + 8, g + 16, g + 24), and o gains p . v (fp32 MMA
//     accumulation, the step's two 16-position chunks in order);
//   * per-lane partial sums of l are added by a fixed xor butterfly;
//   * the splits' states (m_s, l_s, o_s) combine as M = max_s m_s,
//     w_s = 2^(m_s - M), l = sum_s l_s w_s and o = sum_s o_s w_s, each sum
//     an fmaf chain in ascending split order;
//   * out = bf16_rne(o / l).
// No other request, and no batch size, reaches any of these steps: which
// warp runs a split, and when, is scheduling only.
//
// Three kernels per call, chained by programmatic dependent launch:
//   plan     one CTA lists the (request, split) items, full splits first,
//            and resets the ticket counter;
//   stream   persistent, one CTA per SM; every warp is an independent
//            stream: it takes items by ticket, stages their 32-position K/V
//            tiles through its own ring of TMA copies (and q into its own
//            buffer), runs the split and writes its record;
//   combine  combines each request's split records, one CTA per (piece of
//            d, key/value head, request).
#include <atomic>

#include <cuda_bf16.h>

#include "attention.h"
#include "bounds.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace bi {

constexpr int kAttnD = 128;                        // head dimension
constexpr int kAttnTile = 32;                      // positions per staged tile and per softmax step
constexpr int kAttnRowBytes = kAttnD * 2;          // one position of one head's K (or V)
constexpr int kAttnKVBytes = kAttnTile * kAttnRowBytes;  // a tile of K (or of V)
constexpr uint64_t kAttnWaitNs = 2000000000ull;

// Stream warps per CTA and their shared memory, for up to 8 query heads per
// group (NT = 1) and for 9 to 16 (NT = 2): a pool of `pool` stages (a stage
// holds one tile's K then V) shared out among the warps, and a buffer per
// warp for the group's q rows, which arrive with an item's first tile.
// Every warp owns 2 stages when all may have work; when the static schedule
// leaves warps of a CTA without items (one long request), the pool is split
// among the busy ones, up to kAttnMaxRing stages each, so that as much of the
// cache is in flight per SM as when every warp is busy.
//
// A tile lands as the cache's TMA boxes put it: for each position, its two
// 64-value halves as consecutive 128-byte rows (row 2 r + h of the tile),
// under the 128-byte swizzle (16-byte group u of row R sits at group
// u ^ (R % 8)).
constexpr int kAttnMaxRing = 6;
template <int NT>
struct AttnCfg {
  static constexpr int warps = 6;
  static constexpr int pool = 2 * warps;
  static constexpr int q_bytes = 8 * NT * kAttnD * 2;
  static constexpr int stage_bytes = 2 * kAttnKVBytes;
  static constexpr int smem = pool * stage_bytes + warps * q_bytes + 1024;
  static_assert(stage_bytes % 1024 == 0, "stages must keep the 1024-byte alignment of the 128-byte swizzle");
  static_assert(smem <= kMaxDynSmem, "ring too large");
};

__device__ __forceinline__ void attn_flag(int* status, int code) { atomicCAS(status, 0, code); }

// Waits for the phase of `parity` on `bar`, at most 2 s; false if it ran out
// (the status word is set).
__device__ __noinline__ bool attn_wait_slow(uint32_t bar, uint32_t parity, int* status) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kAttnWaitNs) {
      attn_flag(status, (int)BI_ERR_DEVICE_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ bool attn_wait(uint32_t bar, uint32_t parity, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  return attn_wait_slow(bar, parity, status);
}

__device__ __forceinline__ void attn_drain(uint32_t bar, uint32_t parity, int* status) {
  attn_wait(bar, parity, status);
}

// 2^x by the ex2.approx instruction (relative error about 2^-22, far below
// the bf16 rounding the weights get next); 2^-inf = 0.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// plan: the list of (request, split) items and the ticket counter
// ---------------------------------------------------------------------------

constexpr int kPlanThreads = 1024;

// Exclusive prefix sum over the CTA (kPlanThreads threads); *total gets the sum.
__device__ __forceinline__ uint64_t plan_scan(uint64_t v, uint64_t* sh, uint64_t* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint64_t x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint64_t y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) sh[warp] = x;
  __syncthreads();
  if (warp == 0) {
    uint64_t w = sh[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const uint64_t y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    sh[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const uint64_t before = warp > 0 ? sh[warp - 1] : 0;
  *total = sh[31];
  __syncthreads();  // sh is reused by the next call
  return before + x - v;
}

// Items: full splits first (request-major), then the requests' partial last
// splits.  Entry = (b << 16) | s.  An invalid length gives no items (and is
// flagged; the combine writes NaN for it).
__global__ void __launch_bounds__(kPlanThreads) decode_attn_plan_kernel(const AttnParams p, int64_t B) {
  __shared__ uint64_t sh[32];
  grid_dep_launch_dependents();
  grid_dep_wait();  // the lengths may come from the previous kernel in the stream
  auto length = [&](int64_t b) -> int64_t {
    const int64_t L = p.seq_lens[b];
    if (L < 0 || L > p.max_len) {
      attn_flag(p.status, (int)BI_ERR_INVALID_ARG);
      return 0;
    }
    return L;
  };
  uint64_t nfull = 0;
  for (int64_t b = threadIdx.x; b < B; b += kPlanThreads) nfull += (uint64_t)(length(b) / p.split_size);
  uint64_t ftot = 0;
  plan_scan(nfull, sh, &ftot);
  uint64_t carry_f = 0, carry_p = 0;
  for (int64_t b0 = 0; b0 < B; b0 += kPlanThreads) {
    const int64_t b = b0 + threadIdx.x;
    uint64_t f = 0, part = 0;
    if (b < B) {
      const int64_t L = length(b);
      f = (uint64_t)(L / p.split_size);
      part = (L % p.split_size) != 0 ? 1u : 0u;
    }
    uint64_t tot = 0;
    const uint64_t ex = plan_scan((f << 32) | part, sh, &tot);
    if (b < B) {
      uint32_t* dst = p.items + carry_f + (ex >> 32);
      for (uint64_t s = 0; s < f; ++s) dst[s] = ((uint32_t)b << 16) | (uint32_t)s;
      if (part) p.items[ftot + carry_p + (ex & 0xFFFFFFFFu)] = ((uint32_t)b << 16) | (uint32_t)f;
    }
    carry_f += tot >> 32;
    carry_p += tot & 0xFFFFFFFFu;
  }
  if (threadIdx.x == 0) {
    p.ctl[0] = 0;                             // the ticket counter
    p.ctl[1] = (uint32_t)(ftot + carry_p);    // items
  }
}

// ---------------------------------------------------------------------------
// stream: persistent warps, one split at a time
// ---------------------------------------------------------------------------

struct AttnItem {
  const int32_t* bt;  // request b's row of the block table
  int32_t p0, p1;     // positions [p0, p1) of request b
  int32_t b, s, kvh, ntiles;
};

// Two floats rounded to bf16 and packed: lo in the low half, hi in the high
// half (the rounding of __float2bfloat16_rn on each).
__device__ __forceinline__ uint32_t cvt_bf16x2(float lo, float hi) {
  uint32_t d;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}

// One 32-position step of a split (the step of the tree in the header
// comment) on the stage at kb: K tile at kb, V tile at kb + kAttnKVBytes.
// nv = positions of the tile that belong to the split (kAttnTile for every
// step but possibly a split's last); TAIL is false when nv == kAttnTile,
// which drops the masks and the chunk count.  offK / offV are the lane's
// swizzled ldmatrix offsets in the first 16-position chunk of a tile, one
// for each 16-wide block of d.
template <int NT, bool TAIL>
__device__ __forceinline__ void attn_step(uint32_t kb, int nv, float qk_log2, const uint32_t (&offK)[8],
                                          const uint32_t (&offV)[8], const uint32_t (&qf)[NT][8][2],
                                          float (&m)[NT][2], float (&l)[NT][2], float (&o)[8][NT][4]) {
  constexpr int NC = kAttnTile / 16;
  constexpr uint32_t kChunk = 16 * kAttnRowBytes;  // one 16-position chunk of a tile
  const int lane = threadIdx.x & 31, g = lane >> 2;
  const uint32_t vb = kb + kAttnKVBytes;
  if (TAIL) {
    // The request ends inside this tile: the cache past its length is not
    // ours to read (stale values, Inf, NaN), so those V rows become zeros;
    // their scores are masked below.
    for (int i = lane; i < (kAttnTile - nv) * (kAttnRowBytes / 16); i += 32) {
      const uint32_t a = vb + (uint32_t)(nv * kAttnRowBytes + i * 16);
      asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u) : "memory");
    }
    fence_proxy_async_smem();  // before a later copy rewrites this stage
    __syncwarp();
  }
  const int nc = TAIL ? (nv + 15) >> 4 : NC;  // chunks holding positions
  // scores^T [32 positions][GP heads] = K . q^T, as two 16-position chunks
  float acc[NC][NT][4];
#pragma unroll
  for (int k = 0; k < NC; ++k)
#pragma unroll
    for (int j = 0; j < NT; ++j) acc[k][j][0] = acc[k][j][1] = acc[k][j][2] = acc[k][j][3] = 0.0f;
#pragma unroll
  for (int k = 0; k < NC; ++k) {
    if (TAIL && k >= nc) break;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      uint32_t a[4];
      ldmatrix_x4(a, kb + offK[ks] + k * kChunk);
#pragma unroll
      for (int j = 0; j < NT; ++j) mma_m16n8k16_bf16(acc[k][j], a, qf[j][ks][0], qf[j][ks][1]);
    }
  }
  // online softmax over the tile's 32 positions (one step), then p^T as the
  // B operand of p . v.  Lane (g, c) holds the scores of positions 16 k + g
  // and 16 k + g + 8 for heads 8 j + 2 c + cc.
  uint32_t pb[NC][NT][2];
  bool moved = false;
  float alpha[NT][2];
#pragma unroll
  for (int j = 0; j < NT; ++j) {
    float t[2][NC][2], mx[2];
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      mx[cc] = -INFINITY;
#pragma unroll
      for (int k = 0; k < NC; ++k) {
        const int r = k * 16 + g;  // position within the tile
        t[cc][k][0] = (!TAIL || r < nv) ? __fmul_rn(acc[k][j][cc], qk_log2) : -INFINITY;
        t[cc][k][1] = (!TAIL || r + 8 < nv) ? __fmul_rn(acc[k][j][2 + cc], qk_log2) : -INFINITY;
        mx[cc] = fmaxf(mx[cc], fmaxf(t[cc][k][0], t[cc][k][1]));
      }
    }
#pragma unroll
    for (int off = 4; off < 32; off <<= 1)
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) mx[cc] = fmaxf(mx[cc], __shfl_xor_sync(0xffffffffu, mx[cc], off));
    float mn[2], e[2][NC][2];
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      mn[cc] = fmaxf(m[j][cc], mx[cc]);
      alpha[j][cc] = (mn[cc] == m[j][cc]) ? 1.0f : ex2_approx(__fsub_rn(m[j][cc], mn[cc]));
      moved = moved || mn[cc] != m[j][cc];
      const bool none = mn[cc] == -INFINITY;
#pragma unroll
      for (int k = 0; k < NC; ++k) {
        e[cc][k][0] = none ? 0.0f : ex2_approx(__fsub_rn(t[cc][k][0], mn[cc]));
        e[cc][k][1] = none ? 0.0f : ex2_approx(__fsub_rn(t[cc][k][1], mn[cc]));
      }
    }
    // rows g and g + 8 of chunk k, columns 2c and 2c + 1 packed (the
    // accumulator layout), rounded to bf16; l gains the rounded values
    float sum[2] = {0.0f, 0.0f};
#pragma unroll
    for (int k = 0; k < NC; ++k) {
      pb[k][j][0] = cvt_bf16x2(e[0][k][0], e[1][k][0]);
      pb[k][j][1] = cvt_bf16x2(e[0][k][1], e[1][k][1]);
      sum[0] = __fadd_rn(sum[0], __fadd_rn(__uint_as_float(pb[k][j][0] << 16), __uint_as_float(pb[k][j][1] << 16)));
      sum[1] = __fadd_rn(sum[1], __fadd_rn(__uint_as_float(pb[k][j][0] & 0xFFFF0000u),
                                           __uint_as_float(pb[k][j][1] & 0xFFFF0000u)));
    }
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      l[j][cc] = __fadd_rn(__fmul_rn(l[j][cc], alpha[j][cc]), sum[cc]);
      m[j][cc] = mn[cc];
    }
#pragma unroll
    for (int k = 0; k < NC; ++k) {
      pb[k][j][0] = movmatrix_trans(pb[k][j][0]);
      pb[k][j][1] = movmatrix_trans(pb[k][j][1]);
    }
  }
  // o is rescaled only when some column's maximum moved (x * 1 == x)
  if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        o[i][j][0] = __fmul_rn(o[i][j][0], alpha[j][0]);
        o[i][j][1] = __fmul_rn(o[i][j][1], alpha[j][1]);
        o[i][j][2] = __fmul_rn(o[i][j][2], alpha[j][0]);
        o[i][j][3] = __fmul_rn(o[i][j][3], alpha[j][1]);
      }
  }
  // o^T [128 d][GP heads] += V^T . p^T, chunk by chunk
#pragma unroll
  for (int k = 0; k < NC; ++k) {
    if (TAIL && k >= nc) break;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      uint32_t a[4];
      ldmatrix_x4_trans(a, vb + offV[i] + k * kChunk);
#pragma unroll
      for (int j = 0; j < NT; ++j) mma_m16n8k16_bf16(o[i][j], a, pb[k][j][0], pb[k][j][1]);
    }
  }
}

// STATIC: the items come from the lengths of the (at most 32) requests
// themselves, warp w of CTA c taking items w C + c, w C + c + (all warps),
// ... for C CTAs (no plan kernel, no tickets); else by ticket from the plan
// kernel's list.
template <int NT, bool STATIC>
__global__ void __launch_bounds__(32 * AttnCfg<NT>::warps, 1)
    decode_attn_stream_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                              const AttnParams p) {
  constexpr int GP = 8 * NT;  // query-head columns of the MMAs (G <= GP)
  constexpr int W = AttnCfg<NT>::warps;
  constexpr int SB = AttnCfg<NT>::stage_bytes;
  constexpr int NS = AttnCfg<NT>::pool;
  // Items fetched ahead of the one being issued: a fetch starts while fewer
  // than kAhead are ready and adds one, so the items between the one being
  // consumed and the last one fetched number at most kAttnMaxRing + kAhead.
  constexpr int kAhead = 2;
  constexpr int kQ = 16;
  static_assert(kQ >= kAttnMaxRing + kAhead + 1 && (kQ & (kQ - 1)) == 0, "item queue");
  extern __shared__ uint8_t attn_smem_raw[];
  __shared__ __align__(8) uint64_t full[NS];
  __shared__ AttnItem queue[W][kQ];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const uint32_t smem0 = (smem_u32(attn_smem_raw) + 1023u) & ~1023u;
  const uint32_t qbuf = smem0 + (uint32_t)(NS * SB + warp * AttnCfg<NT>::q_bytes);  // the warp's q rows
  if (threadIdx.x == 0) {
    for (int i = 0; i < NS; ++i) mbar_init(smem_u32(&full[i]), 1);
    fence_mbar_init();
  }
  __syncthreads();
  grid_dep_wait();  // the item list, q, the lengths and the cache come from earlier kernels
  // Only now may the combine start: its CTAs read the lengths before their
  // own wait, which is safe once every earlier kernel has completed.
  grid_dep_launch_dependents();
  const uint32_t n_tickets = STATIC ? 0u : p.ctl[1] * (uint32_t)p.Hkv;
  AttnItem* Q = queue[warp];
  // Positions stay below 2^28 (n_split <= 65535 splits of <= 4096) and cache
  // rows below 2^31 (checked by the host), so 32-bit arithmetic holds them;
  // page and box sizes are powers of two.
  const int32_t rows = (int32_t)(p.num_pages * p.page_size);
  const uint32_t npages = (uint32_t)p.num_pages;
  const int pshift = p.page_shift, bshift = p.box_shift;
  const int32_t pmask = (1 << pshift) - 1;
  const int full_nb = kAttnTile >> bshift;  // boxes of a whole tile
  // The lane's ldmatrix addresses in a tile's first 16-position chunk, for
  // d block i (half h = i / 4): the lane gives position r (lane % 16 for K;
  // lane % 8 + 8 (lane / 16) for V^T, whose matrices are transposed on the
  // way) and 16-byte group u = 2 (i % 4) + lane / 16 (K) or
  // 2 (i % 4) + (lane / 8) % 2 (V) of that position's half; it sits in
  // 128-byte row R = 2 r + h at group u ^ (R % 8).
  uint32_t offK[8], offV[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int h = i >> 2;
    const int rk = 2 * (lane & 15) + h, uk = ((i & 3) << 1) + (lane >> 4);
    const int rv = 2 * ((lane & 7) + ((lane >> 4) << 3)) + h, uv = ((i & 3) << 1) + ((lane >> 3) & 1);
    offK[i] = (uint32_t)(rk * 128 + ((uk ^ (rk & 7)) << 4));
    offV[i] = (uint32_t)(rv * 128 + ((uv ^ (rv & 7)) << 4));
  }

  // ---- item fetch, one step per loop turn so that each global load has a
  // whole tile of work to land in: ticket -> list entry -> length -> item.
  // Tickets run over items x key/value heads, heads fastest, so the heads of
  // one split are taken together.
  int fs = 0;            // 0 idle, 1 ticket in flight, 2 entry in flight, 3 length in flight
  bool fetch_done = false;
  uint32_t tk = 0, fe = 0, ft = 0;
  int32_t fL = 0;
  int nready = 0;        // items fetched into Q (sequence numbers 0 .. nready - 1)
  // The static schedule: lane b < nreq holds request b's length sL, split
  // count sn and the inclusive prefix pre of the counts; items run over
  // (request, split, key/value head), heads fastest.
  int32_t sL = 0, sn = 0, pre = 0;
  uint32_t next_i = 0, total_i = 0, wstride = 0;
  if (STATIC) {
    if (lane < p.nreq) {
      const int64_t L = p.seq_lens[lane];
      if (L < 0 || L > p.max_len) {
        attn_flag(p.status, (int)BI_ERR_INVALID_ARG);  // the combine writes NaN for it
      } else {
        sL = (int32_t)L;
        sn = (sL + p.split_size - 1) / p.split_size;
      }
    }
    pre = sn;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int32_t y = __shfl_up_sync(0xffffffffu, pre, off);
      if (lane >= off) pre += y;
    }
    total_i = (uint32_t)__shfl_sync(0xffffffffu, pre, 31) * (uint32_t)p.Hkv;
    next_i = (uint32_t)warp * gridDim.x + blockIdx.x;  // first items spread over the CTAs
    wstride = gridDim.x * (uint32_t)W;
  }
  // The warp's stages: pool stages [sbase, sbase + nst).  Under the static
  // schedule the warps of this CTA with items are its first nbusy (warp w's
  // first item is item w * CTAs + CTA), and they share the pool.
  int nst = 2, sbase = 2 * warp;
  if (STATIC) {
    const int64_t left = ((int64_t)total_i - (int64_t)blockIdx.x + gridDim.x - 1) / gridDim.x;
    const int nbusy = (int)(left < 0 ? 0 : (left > W ? W : left));
    if (warp < nbusy) {
      nst = min(kAttnMaxRing, NS / nbusy);
      sbase = warp * nst;
    }
  }
  const uint32_t ring = smem0 + (uint32_t)(sbase * SB);
  auto fetch_step = [&](int pi) {
    if (STATIC) {
      if (fetch_done || nready - pi >= kAhead) return;
      if (next_i >= total_i) {
        fetch_done = true;
        return;
      }
      const uint32_t si = next_i / (uint32_t)p.Hkv;  // split over all requests
      const int32_t kvh = (int32_t)(next_i % (uint32_t)p.Hkv);
      next_i += wstride;
      const int b = __ffs(__ballot_sync(0xffffffffu, (uint32_t)pre > si)) - 1;
      const int32_t first = __shfl_sync(0xffffffffu, pre - sn, b);
      const int32_t L = __shfl_sync(0xffffffffu, sL, b);
      if (lane == 0) {
        AttnItem x;
        x.b = b;
        x.s = (int32_t)si - first;
        x.kvh = kvh;
        x.bt = p.block_table + (int64_t)b * p.bt_stride;
        x.p0 = x.s * p.split_size;
        x.p1 = min(x.p0 + p.split_size, L);
        x.ntiles = (x.p1 - x.p0 + kAttnTile - 1) / kAttnTile;
        Q[nready & (kQ - 1)] = x;
      }
      __syncwarp();
      ++nready;
      return;
    }
    if (fs == 0) {
      if (fetch_done || nready - pi >= kAhead) return;
      if (lane == 0) tk = atomicAdd(p.ctl, 1u);
      fs = 1;
    } else if (fs == 1) {
      ft = __shfl_sync(0xffffffffu, tk, 0);
      if (ft >= n_tickets) {
        fetch_done = true;
        fs = 0;
        return;
      }
      if (lane == 0) fe = p.items[ft / (uint32_t)p.Hkv];
      fs = 2;
    } else if (fs == 2) {
      if (lane == 0) fL = p.seq_lens[fe >> 16];
      fs = 3;
    } else {
      if (lane == 0) {
        AttnItem x;
        x.b = (int32_t)(fe >> 16);
        x.s = (int32_t)(fe & 0xFFFFu);
        x.kvh = (int32_t)(ft % (uint32_t)p.Hkv);
        x.bt = p.block_table + (int64_t)x.b * p.bt_stride;
        x.p0 = x.s * p.split_size;
        x.p1 = min(x.p0 + p.split_size, fL);
        x.ntiles = (x.p1 - x.p0 + kAttnTile - 1) / kAttnTile;
        Q[nready & (kQ - 1)] = x;
      }
      __syncwarp();
      ++nready;
      fs = 0;
    }
  };

  // ---- page ids.  A window is 32 consecutive pages of an item (from the
  // page holding its first position), lane j holding page 32 w + j of
  // window w (-1 past the item's last page).  The issue side keeps the
  // window in use (wcur) and the next one (wnx: the item's next window, or
  // the next item's first), loaded while the current one is in use, so that
  // no tile waits for the block table.
  auto win_load = [&](const AttnItem& it, int w) -> int32_t {
    const int32_t fp = it.p0 >> pshift;
    const int32_t np = ((it.p1 - 1) >> pshift) - fp + 1;
    const int32_t j = 32 * w + lane;
    return j < np ? it.bt[fp + j] : -1;
  };
  int32_t wcur = -1, wnx = -1;
  int wcur_item = -1, wcur_w = 0, wnx_item = -1, wnx_w = 0;
  int wpf_ready = -1;  // nready when the last prefetch attempt found nothing to load

  // ---- cache rows of tile t of item number ii: lane j < nb holds the row
  // of box j.
  auto tile_rows = [&](const AttnItem& it, int ii, int t, int& nb) -> int32_t {
    const int32_t tp = it.p0 + t * kAttnTile, left = it.p1 - tp;
    nb = left >= kAttnTile ? full_nb : (left + (1 << bshift) - 1) >> bshift;
    const int32_t pos = tp + (lane << bshift);
    const int32_t rel = (pos >> pshift) - (it.p0 >> pshift);  // page of the item
    const int w = ((tp >> pshift) - (it.p0 >> pshift)) >> 5;  // a tile never spans two windows
    if (wcur_item != ii || wcur_w != w) {
      if (wnx_item == ii && wnx_w == w) {
        wcur = wnx;
      } else {
        wcur = win_load(it, w);  // not prefetched (the item was not fetched in time)
      }
      wcur_item = ii;
      wcur_w = w;
      wnx_item = -1;
      wpf_ready = -1;
    }
    const int32_t pg = __shfl_sync(0xffffffffu, wcur, rel & 31);
    int32_t y = 0;
    if (lane < nb) {
      if ((uint32_t)pg >= npages) {
        attn_flag(p.status, (int)BI_ERR_INVALID_ARG);
        y = rows;  // past the cache's end: zeros
      } else {
        y = (pg << pshift) | (pos & pmask);
      }
    }
    return y;
  };
  // Loads the window after the one in use, if it is known and not loaded
  // (tried again only once another item has been fetched).
  auto win_prefetch = [&]() {
    if (wnx_item >= 0 || wcur_item < 0 || wpf_ready == nready) return;
    const AttnItem& it = Q[wcur_item & (kQ - 1)];
    const int32_t np = ((it.p1 - 1) >> pshift) - (it.p0 >> pshift) + 1;
    if (32 * (wcur_w + 1) < np) {
      wnx = win_load(it, wcur_w + 1);
      wnx_item = wcur_item;
      wnx_w = wcur_w + 1;
    } else if (wcur_item + 1 < nready) {
      wnx = win_load(Q[(wcur_item + 1) & (kQ - 1)], 0);
      wnx_item = wcur_item + 1;
      wnx_w = 0;
    } else {
      wpf_ready = nready;
    }
  };

  // Issues tile t of item it into stage st (rows y from tile_rows): the K and
  // V boxes (one per lane, lanes < nb), and q into the q buffer with the
  // item's first tile.
  auto issue = [&](const AttnItem& it, int t, int st, int nb, int32_t y) {
    // debug-bounds build: the stage within the pool, the item within range
    if (!bounds_ok(st >= 0 && st < nst && sbase + nst <= NS, p.status, kChkAttnStage, (uint64_t)(sbase + st)) ||
        !bounds_ok(it.b >= 0 && it.b < p.nreq && it.kvh >= 0 && it.kvh < p.Hkv && it.s >= 0 && it.s < p.n_split,
                   p.status, kChkAttnItem, ((uint64_t)(uint32_t)it.b << 32) | (uint32_t)it.s))
      return;  // the stage's barrier stays short: the wait gives up
    const uint32_t stage = ring + (uint32_t)(st * SB);
    const uint32_t fb = smem_u32(&full[sbase + st]);
    if (lane == 0)
      mbar_arrive_expect_tx(fb, (uint32_t)((nb << bshift) * kAttnRowBytes * 2 + (t == 0 ? p.G * kAttnD * 2 : 0)));
    __syncwarp();
    if (lane < nb) {
      // box {64 values, both halves of head kvh, box_rows positions}
      const uint32_t off = (uint32_t)((lane << bshift) * kAttnRowBytes);
      tma_load_3d(stage + off, &tmK, fb, 0, it.kvh * 2, y);
      tma_load_3d(stage + kAttnKVBytes + off, &tmV, fb, 0, it.kvh * 2, y);
    }
    if (t == 0 && lane == 0) {
      const __nv_bfloat16* qsrc = static_cast<const __nv_bfloat16*>(p.q) +
                                  ((int64_t)it.b * p.Hq + (int64_t)it.kvh * p.G) * kAttnD;
      bulk_load(qbuf, qsrc, (uint32_t)(p.G * kAttnD * 2), fb);
    }
  };

  uint32_t qf[NT][8][2];
  float m[NT][2], l[NT][2], o[8][NT][4];
  int pi = 0, pt = 0, ci = 0, ct = 0, issued = 0, consumed = 0;
  int ist = 0, cst = 0;  // stages of the next issue and of the next tile consumed
  uint32_t cph = 0;      // phase parity of stage cst
  AttnItem iit, cit;     // the items being issued (number iit_n) and consumed
  int iit_n = -1;
  bool ok = true;
  while (ok) {
    fetch_step(pi);
    // keep nst tiles in flight
    while (pi < nready && issued - consumed < nst) {
      // an item's first tile overwrites the q buffer: not before the
      // previous item has read it (its first tile consumed)
      if (pt == 0 && ci < pi && !(ci == pi - 1 && ct > 0)) break;
      if (iit_n != pi) {
        iit = Q[pi & (kQ - 1)];
        iit_n = pi;
      }
      int nb = 0;
      const int32_t y = tile_rows(iit, pi, pt, nb);
      issue(iit, pt, ist, nb, y);
      ++issued;
      if (++ist == nst) ist = 0;
      if (++pt == iit.ntiles) {
        pt = 0;
        ++pi;
      }
    }
    win_prefetch();
    if (consumed == issued) {
      if (fetch_done && pi == nready && fs == 0) break;
      continue;  // waiting for the next item's fetch
    }

    const int st = cst;
    const bool got = attn_wait(smem_u32(&full[sbase + st]), cph, p.status);
    if (!__all_sync(0xffffffffu, got)) {
      ok = false;
      break;
    }
    if (ct == 0) cit = Q[ci & (kQ - 1)];
    const AttnItem& it = cit;
    const uint32_t kb = ring + (uint32_t)(st * SB);
    if (ct == 0) {
      // a new split: fresh state, and q as the MMA's B operand (k = d, n =
      // query head): lane holds q[head g][d = 16 ks + 2c, +1] and [.. + 8, + 9]
      const uint32_t qs = qbuf;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const int h = j * 8 + g;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          uint32_t lo = 0, hi = 0;
          if (h < p.G) {
            const uint32_t a = qs + (uint32_t)(h * kAttnD * 2 + (ks * 16 + 2 * c) * 2);
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(lo) : "r"(a));
            asm volatile("ld.shared.u32 %0, [%1];" : "=r"(hi) : "r"(a + 16u));
          }
          qf[j][ks][0] = lo;
          qf[j][ks][1] = hi;
        }
        m[j][0] = m[j][1] = -INFINITY;
        l[j][0] = l[j][1] = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i][j][0] = o[i][j][1] = o[i][j][2] = o[i][j][3] = 0.0f;
      }
    }
    const int nv = it.p1 - (it.p0 + ct * kAttnTile);
    if (nv >= kAttnTile)
      attn_step<NT, false>(kb, kAttnTile, p.qk_log2, offK, offV, qf, m, l, o);
    else
      attn_step<NT, true>(kb, nv, p.qk_log2, offK, offV, qf, m, l, o);
    __syncwarp();  // every lane is done with the stage before it is refilled
    ++consumed;
    if (++cst == nst) {
      cst = 0;
      cph ^= 1u;
    }
    if (++ct == it.ntiles) {
      // the split's record: o^T [D][GP], then m [GP], then l [GP]
#pragma unroll
      for (int j = 0; j < NT; ++j)
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          l[j][cc] = __fadd_rn(l[j][cc], __shfl_xor_sync(0xffffffffu, l[j][cc], 4));
          l[j][cc] = __fadd_rn(l[j][cc], __shfl_xor_sync(0xffffffffu, l[j][cc], 8));
          l[j][cc] = __fadd_rn(l[j][cc], __shfl_xor_sync(0xffffffffu, l[j][cc], 16));
        }
      const int64_t rec_i = ((int64_t)it.b * p.Hkv + it.kvh) * (int64_t)p.n_split + it.s;
      if (!bounds_ok(rec_i >= 0 && rec_i < (int64_t)p.nreq * p.Hkv * p.n_split, p.status, kChkAttnRecord,
                     (uint64_t)rec_i)) {
        ct = 0;
        ++ci;
        continue;
      }
      float* rec = p.part + rec_i * (int64_t)((kAttnD + 2) * GP);
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
      ct = 0;
      ++ci;
    }
  }
  if (!ok) {
    // abandoned (a copy did not land in 2 s): every copy still in flight must
    // land before the CTA ends
    if (lane == 0)
      for (int k = consumed; k < issued; ++k)
        attn_drain(smem_u32(&full[sbase + k % nst]), (uint32_t)(k / nst) & 1u, p.status);
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------
// combine
// ---------------------------------------------------------------------------

// One CTA per (slice of d, key/value head, request) combines the request's
// split states in two passes:
//   M = max over splits of m_s (per head; max is exact in any order);
//   w_s = 2^(m_s - M) (exp2f), l = sum of l_s w_s and o = sum of o_s w_s,
//   each a chain of fmaf in ascending split order from 0;
//   out = bf16_rne(o / l).
// Thread t owns head h = t % GP and the d values t / GP + (CT / GP) i of the
// slice; a record holds o[d][h], then m[h] and l[h], so the CTA's loads of
// one record's slice are contiguous.  A request of at most A splits takes
// one round of loads (m, l and o together); for longer ones the CTA reads
// every m while the first A records are in flight.  The records are read straight from L2 (the previous kernel just
// wrote them).  CT and SL change no operation: every (h, d) combines the
// same records the same way.  The host takes more, smaller CTAs when there
// are few (request, head) pairs.
template <int NT, int CT, int SL>
__global__ void __launch_bounds__(CT) decode_attn_combine_kernel(const AttnParams p, __nv_bfloat16* out) {
  constexpr int GP = 8 * NT;
  constexpr int RS = (kAttnD + 2) * GP;  // floats per record
  constexpr int SD = kAttnD / SL;        // d values of the slice
  constexpr int DSTEP = CT / GP;         // distance between a thread's d values
  constexpr int DPT = SD / DSTEP;        // d values per thread
  static_assert(DPT >= 1 && SD % DSTEP == 0, "combine layout");
  // records whose loads are in flight together (about 32 values per thread)
  constexpr int A = 32 / DPT < 4 ? 4 : (32 / DPT > 32 ? 32 : 32 / DPT);
  const int kvh = blockIdx.x / SL, slice = blockIdx.x % SL;
  const int t = threadIdx.x, h = t % GP, d0 = slice * SD + t / GP;
  const int64_t b = blockIdx.y;
  // The stream kernel lets this grid start only after its own wait, so the
  // kernels that wrote the lengths have completed: read them before waiting.
  const int64_t L = p.seq_lens[b];
  grid_dep_launch_dependents();
  grid_dep_wait();  // the split records come from the previous kernel
  __nv_bfloat16* ob = out + (b * p.Hq + (int64_t)kvh * p.G + h) * kAttnD + d0;
  if (L <= 0 || L > p.max_len) {
    // an empty request gives zeros; an invalid length (flagged by the plan
    // or stream kernel) gives NaN
    if (h < p.G) {
      const __nv_bfloat16 v = __float2bfloat16_rn(L == 0 ? 0.0f : __int_as_float(0x7fc00000));
#pragma unroll
      for (int i = 0; i < DPT; ++i) ob[DSTEP * i] = v;
    }
    return;
  }
  const int ns = (int)((L + p.split_size - 1) / p.split_size);
  const float* rec0 = p.part + (b * p.Hkv + kvh) * (int64_t)p.n_split * RS;
  const float* pm = rec0 + kAttnD * GP + h;  // m of split 0; l follows at + GP
  const float* po = rec0 + d0 * GP + h;
  float mv[A], lv[A], ov[A][DPT];
  auto load_batch = [&](int s0) {
#pragma unroll
    for (int u = 0; u < A; ++u) {
      if (s0 + u < ns) {
        const int64_t r = (int64_t)(s0 + u) * RS;
        mv[u] = __ldcg(pm + r);
        lv[u] = __ldcg(pm + r + GP);
#pragma unroll
        for (int i = 0; i < DPT; ++i) ov[u][i] = __ldcg(po + r + DSTEP * i * GP);
      }
    }
  };
  load_batch(0);
  float M = -INFINITY;
  if (ns > A) {
    // M over every split, while the first batch is in flight: the DSTEP
    // threads of head h share the splits, then reduce (lanes h + GP k of a
    // warp by shuffles, the warps through shared memory)
    __shared__ float red[CT / 32][GP];
    for (int s0 = t / GP; s0 < ns; s0 += 8 * DSTEP) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = s0 + u * DSTEP < ns ? __ldcg(pm + (int64_t)(s0 + u * DSTEP) * RS) : -INFINITY;
#pragma unroll
      for (int u = 0; u < 8; ++u) M = fmaxf(M, v[u]);
    }
#pragma unroll
    for (int off = GP; off < 32; off <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    if ((t & 31) < GP) red[t >> 5][h] = M;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < CT / 32; ++w) M = fmaxf(M, red[w][h]);
  } else {
#pragma unroll
    for (int u = 0; u < A; ++u)
      if (u < ns) M = fmaxf(M, mv[u]);
  }
  float o[DPT], l = 0.0f;
#pragma unroll
  for (int i = 0; i < DPT; ++i) o[i] = 0.0f;
  for (int s0 = 0; s0 < ns; s0 += A) {
    if (s0 > 0) load_batch(s0);
#pragma unroll
    for (int u = 0; u < A; ++u) {
      if (s0 + u >= ns) break;
      const float w = exp2f(__fsub_rn(mv[u], M));
      l = fmaf(lv[u], w, l);
#pragma unroll
      for (int i = 0; i < DPT; ++i) o[i] = fmaf(ov[u][i], w, o[i]);
    }
  }
  if (h < p.G) {
#pragma unroll
    for (int i = 0; i < DPT; ++i) ob[DSTEP * i] = __float2bfloat16_rn(__fdiv_rn(o[i], l));
  }
}

template <int NT, bool STATIC>
static cudaError_t launch_attn_t(const AttnLaunch& A) {
  auto kern = decode_attn_stream_kernel<NT, STATIC>;
  constexpr int smem = AttnCfg<NT>::smem;
  // the shared-memory limits are per device: set them once for each
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t de = cudaGetDevice(&dev);
  if (de != cudaSuccess) return de;
  const uint64_t bit = dev < 64 ? (uint64_t)1 << dev : 0;
  if (!bit || !(configured.load() & bit)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  cudaError_t e = cudaSuccess;
  if (!STATIC) {
    e = launch_overlapped(decode_attn_plan_kernel, dim3(1), dim3(kPlanThreads), A.stream, A.p, A.B);
    if (e != cudaSuccess) return e;
  }
  e = launch_overlapped_smem(kern, dim3((unsigned)A.grid), dim3(32 * AttnCfg<NT>::warps), smem, A.stream, A.tmK,
                             A.tmV, A.p);
  if (e != cudaSuccess) return e;
  // few (request, head) pairs: CTAs of 128 threads on slices of 16 / 8 d
  if (A.B * A.p.Hkv < A.grid)
    return launch_overlapped(decode_attn_combine_kernel<NT, 128, 8 * NT>, dim3((unsigned)(A.p.Hkv * 8 * NT), (unsigned)A.B),
                             dim3(128), A.stream, A.p, A.out);
  return launch_overlapped(decode_attn_combine_kernel<NT, 256, 1>, dim3((unsigned)A.p.Hkv, (unsigned)A.B), dim3(256),
                           A.stream, A.p, A.out);
}

template <int NT>
static cudaError_t launch_attn_nt(const AttnLaunch& A) {
  return A.B <= kAttnStaticMaxB ? launch_attn_t<NT, true>(A) : launch_attn_t<NT, false>(A);
}

cudaError_t launch_decode_attention(const AttnLaunch& A) {
  return A.p.G <= 8 ? launch_attn_nt<1>(A) : launch_attn_nt<2>(A);
}

}  // namespace bi
