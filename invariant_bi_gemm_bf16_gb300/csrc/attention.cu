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
//   * the splits' states fold in split order with
//       m = max(m1, m2), a_i = 2^(m_i - m), l = l1 a1 + l2 a2, o = o1 a1 + o2 a2;
//   * out = bf16_rne(o / l).
// No other request, and no batch size, reaches any of these steps: which
// warp runs a split, and when, is scheduling only.
//
// Three kernels per call, chained by programmatic dependent launch:
//   plan     one CTA lists the (request, split) items, full splits first,
//            and resets the ticket counter;
//   stream   persistent, one CTA per SM; every warp is an independent
//            stream: it takes items by ticket, stages their 32-position K/V
//            tiles (and q) through its own ring of TMA copies, runs the
//            split and writes its record;
//   combine  folds each request's split records in order, one CTA per
//            (key/value head, request), or per (key/value head, slice of
//            d, request) when there are few requests.
#include <atomic>

#include <cuda_bf16.h>

#include "attention.h"
#include "internal.h"
#include "ptx.cuh"

namespace bi {

constexpr int kAttnD = 128;                        // head dimension
constexpr int kAttnTile = 32;                      // positions per staged tile (two chunks of 16)
constexpr int kAttnStages = 2;                     // tiles in flight per warp
constexpr int kAttnHalfBytes = kAttnTile * 128;    // 32 positions x 64 values
constexpr int kAttnKVBytes = 2 * kAttnHalfBytes;   // 32 positions x 128 values
constexpr uint64_t kAttnWaitNs = 2000000000ull;

// Stream warps per CTA and stage layout, for up to 8 query heads per group
// (NT = 1) and for 9 to 16 (NT = 2).  A stage holds the K tile, the V tile
// and room for the group's q rows (copied with an item's first tile).
template <int NT>
struct AttnCfg {
  static constexpr int warps = NT == 1 ? 6 : 5;
  static constexpr int q_bytes = 8 * NT * kAttnD * 2;
  static constexpr int stage_bytes = 2 * kAttnKVBytes + q_bytes;
  static constexpr int smem = warps * kAttnStages * stage_bytes + 1024;
};
static_assert(AttnCfg<1>::stage_bytes % 1024 == 0 && AttnCfg<2>::stage_bytes % 1024 == 0,
              "stages must keep the 1024-byte alignment of the 128-byte swizzle");
static_assert(AttnCfg<1>::smem <= kMaxDynSmem && AttnCfg<2>::smem <= kMaxDynSmem, "ring too large");

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

__device__ __forceinline__ uint32_t pack_bf16(__nv_bfloat16 lo, __nv_bfloat16 hi) {
  return (uint32_t)__bfloat16_as_ushort(lo) | ((uint32_t)__bfloat16_as_ushort(hi) << 16);
}

// 2^x by the ex2.approx instruction (relative error about 2^-22, far below
// the bf16 rounding the weights get next); 2^-inf = 0.
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The fold of two running states (one column of o).
__device__ __forceinline__ void attn_scales(float m1, float m2, float& m, float& a1, float& a2) {
  m = fmaxf(m1, m2);
  a1 = (m1 == m) ? 1.0f : exp2f(__fsub_rn(m1, m));
  a2 = (m2 == m) ? 1.0f : exp2f(__fsub_rn(m2, m));
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
  int64_t p0, p1;  // positions [p0, p1) of request b
  int32_t b, s, kvh, ntiles;
};

template <int NT>
__global__ void __launch_bounds__(32 * AttnCfg<NT>::warps, 1)
    decode_attn_stream_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                              const AttnParams p) {
  constexpr int GP = 8 * NT;  // query-head columns of the MMAs (G <= GP)
  constexpr int W = AttnCfg<NT>::warps;
  constexpr int SB = AttnCfg<NT>::stage_bytes;
  // Items fetched ahead of the one being issued: a fetch starts while fewer
  // than kAhead are ready and adds one, so the items between the one being
  // consumed and the last one fetched number at most kAttnStages + kAhead.
  constexpr int kAhead = 2;
  constexpr int kQ = kAttnStages + kAhead + 1;
  extern __shared__ uint8_t attn_smem_raw[];
  __shared__ __align__(8) uint64_t full[W][kAttnStages];
  __shared__ AttnItem queue[W][kQ];

  grid_dep_launch_dependents();
  grid_dep_wait();  // the item list, q and the cache come from earlier kernels

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, c = lane & 3;
  const uint32_t ring = ((smem_u32(attn_smem_raw) + 1023u) & ~1023u) + (uint32_t)(warp * kAttnStages * SB);
  if (lane == 0) {
    for (int i = 0; i < kAttnStages; ++i) mbar_init(smem_u32(&full[warp][i]), 1);
    fence_mbar_init();
  }
  __syncwarp();
  const uint32_t n_tickets = p.ctl[1] * (uint32_t)p.Hkv;
  AttnItem* Q = queue[warp];
  const int64_t rows = p.num_pages * p.page_size;

  // ---- item fetch, one step per loop turn so that each global load has a
  // whole tile of work to land in: ticket -> list entry -> length -> item.
  // Tickets run over items x key/value heads, heads fastest, so the heads of
  // one split are taken together.
  int fs = 0;            // 0 idle, 1 ticket in flight, 2 entry in flight, 3 length in flight
  bool fetch_done = false;
  uint32_t tk = 0, fe = 0, ft = 0;
  int32_t fL = 0;
  int nready = 0;        // items fetched into Q (sequence numbers 0 .. nready - 1)
  auto fetch_step = [&](int pi) {
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
        x.p0 = (int64_t)x.s * p.split_size;
        x.p1 = min(x.p0 + (int64_t)p.split_size, (int64_t)fL);
        x.ntiles = (int32_t)((x.p1 - x.p0 + kAttnTile - 1) / kAttnTile);
        Q[nready % kQ] = x;
      }
      __syncwarp();
      ++nready;
      fs = 0;
    }
  };

  // ---- page ids of one tile: lane j < nb holds the row of box j.
  auto tile_rows = [&](const AttnItem& it, int t, int& nb) -> int32_t {
    const int64_t tp = it.p0 + (int64_t)t * kAttnTile;
    nb = (int)min((int64_t)(kAttnTile / p.box_rows), (it.p1 - tp + p.box_rows - 1) / p.box_rows);
    int32_t y = 0;
    if (lane < nb) {
      const int64_t pos = tp + (int64_t)lane * p.box_rows;
      const int32_t pg = p.block_table[(int64_t)it.b * p.bt_stride + pos / p.page_size];
      if (pg < 0 || (int64_t)pg >= p.num_pages) {
        attn_flag(p.status, (int)BI_ERR_INVALID_ARG);
        y = (int32_t)rows;  // past the cache's end: zeros
      } else {
        y = (int32_t)((int64_t)pg * p.page_size + pos % p.page_size);
      }
    }
    return y;
  };

  // Issues tile t of item it into stage st (rows y from tile_rows): the K and
  // V boxes (one per lane, lanes < nb), and q with the item's first tile.
  auto issue = [&](const AttnItem& it, int t, int st, int nb, int32_t y) {
    const uint32_t stage = ring + (uint32_t)(st * SB);
    const uint32_t fb = smem_u32(&full[warp][st]);
    if (lane == 0)
      mbar_arrive_expect_tx(fb, (uint32_t)(nb * p.box_rows * 128 * 4 + (t == 0 ? p.G * kAttnD * 2 : 0)));
    __syncwarp();
    if (lane < nb) {
      const int32_t x = it.kvh * kAttnD;
      const uint32_t off = (uint32_t)(lane * p.box_rows * 128);
      tma_load_2d(stage + off, &tmK, fb, x, y);
      tma_load_2d(stage + kAttnHalfBytes + off, &tmK, fb, x + 64, y);
      tma_load_2d(stage + kAttnKVBytes + off, &tmV, fb, x, y);
      tma_load_2d(stage + kAttnKVBytes + kAttnHalfBytes + off, &tmV, fb, x + 64, y);
    }
    if (t == 0 && lane == 0) {
      const __nv_bfloat16* qsrc = static_cast<const __nv_bfloat16*>(p.q) +
                                  ((int64_t)it.b * p.Hq + (int64_t)it.kvh * p.G) * kAttnD;
      bulk_load(stage + 2 * kAttnKVBytes, qsrc, (uint32_t)(p.G * kAttnD * 2), fb);
    }
  };

  uint32_t qf[NT][8][2];
  float m[NT][2], l[NT][2], o[8][NT][4];
  int pi = 0, pt = 0, ci = 0, ct = 0, issued = 0, consumed = 0;
  int pf_item = -1, pf_tile = 0, pf_nb = 0;  // the tile whose rows pf_y holds
  int32_t pf_y = 0;
  bool ok = true;
  while (ok) {
    fetch_step(pi);
    // keep kAttnStages tiles in flight
    while (pi < nready && issued - consumed < kAttnStages) {
      const AttnItem it = Q[pi % kQ];
      int nb = pf_nb;
      int32_t y = pf_y;
      if (pf_item != pi || pf_tile != pt) y = tile_rows(it, pt, nb);
      issue(it, pt, issued % kAttnStages, nb, y);
      ++issued;
      if (++pt == it.ntiles) {
        pt = 0;
        ++pi;
      }
      // the next tile's rows load while this one is in flight
      pf_item = -1;
      if (pi < nready) {
        pf_y = tile_rows(Q[pi % kQ], pt, pf_nb);
        pf_item = pi;
        pf_tile = pt;
      }
    }
    if (consumed == issued) {
      if (fetch_done && pi == nready && fs == 0) break;
      continue;  // waiting for the next item's fetch
    }

    const int st = consumed % kAttnStages;
    const bool got = attn_wait(smem_u32(&full[warp][st]), (uint32_t)(consumed / kAttnStages) & 1u, p.status);
    if (!__all_sync(0xffffffffu, got)) {
      ok = false;
      break;
    }
    const AttnItem it = Q[ci % kQ];
    const uint32_t kb = ring + (uint32_t)(st * SB), vb = kb + kAttnKVBytes;
    if (ct == 0) {
      // a new split: fresh state, and q as the MMA's B operand (k = d, n =
      // query head): lane holds q[head g][d = 16 ks + 2c, +1] and [.. + 8, + 9]
      const uint32_t qs = kb + 2 * kAttnKVBytes;
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
    const int64_t tp = it.p0 + (int64_t)ct * kAttnTile;
    if (tp + kAttnTile > it.p1) {
      // The request ends inside this tile: the cache past L is not ours to
      // read (stale values, Inf, NaN), so its V rows become zeros; its scores
      // are masked below.
      const int bad0 = (int)(it.p1 - tp);
      for (int i = lane; i < (kAttnTile - bad0) * 16; i += 32) {
        const int rr = bad0 + i / 16, ch = i % 16;
        const uint32_t a = vb + (uint32_t)(ch / 8) * kAttnHalfBytes + (uint32_t)rr * 128u + (uint32_t)(ch % 8) * 16u;
        asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0u) : "memory");
      }
      fence_proxy_async_smem();  // before a later copy rewrites this stage
      __syncwarp();
    }
    // scores^T [32 positions][GP heads] = K . q^T, as two 16-position chunks
    constexpr int NC = kAttnTile / 16;
    const int nc = (int)min((int64_t)NC, (it.p1 - tp + 15) / 16);  // chunks holding positions
    float acc[NC][NT][4];
#pragma unroll
    for (int k = 0; k < NC; ++k)
#pragma unroll
      for (int j = 0; j < NT; ++j) acc[k][j][0] = acc[k][j][1] = acc[k][j][2] = acc[k][j][3] = 0.0f;
#pragma unroll
    for (int k = 0; k < NC; ++k) {
      if (k >= nc) break;
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const int row = k * 16 + (lane & 15);
        const int ch = ((ks & 3) << 1) + (lane >> 4);
        uint32_t a[4];
        ldmatrix_x4(a, kb + (uint32_t)(ks >> 2) * kAttnHalfBytes + (uint32_t)row * 128u +
                           (uint32_t)((ch ^ (row & 7)) << 4));
#pragma unroll
        for (int j = 0; j < NT; ++j) mma_m16n8k16_bf16(acc[k][j], a, qf[j][ks][0], qf[j][ks][1]);
      }
    }
    // online softmax over the tile's 32 positions (one step), then p^T as the
    // B operand of p . v
    uint32_t pb[NC][NT][2];
    bool moved = false;
    float alpha[NT][2];
#pragma unroll
    for (int j = 0; j < NT; ++j) {
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        float t[NC][2];
        float mx = -INFINITY;
#pragma unroll
        for (int k = 0; k < NC; ++k) {
          const int64_t r = tp + k * 16 + g;
          t[k][0] = r < it.p1 ? __fmul_rn(acc[k][j][cc], p.qk_log2) : -INFINITY;
          t[k][1] = r + 8 < it.p1 ? __fmul_rn(acc[k][j][2 + cc], p.qk_log2) : -INFINITY;
          mx = fmaxf(mx, fmaxf(t[k][0], t[k][1]));
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        const float mn = fmaxf(m[j][cc], mx);
        alpha[j][cc] = (mn == m[j][cc]) ? 1.0f : ex2_approx(__fsub_rn(m[j][cc], mn));
        moved = moved || mn != m[j][cc];
        float sum = 0.0f;
        __nv_bfloat16 r[NC][2];
#pragma unroll
        for (int k = 0; k < NC; ++k) {
          r[k][0] = __float2bfloat16_rn(mn == -INFINITY ? 0.0f : ex2_approx(__fsub_rn(t[k][0], mn)));
          r[k][1] = __float2bfloat16_rn(mn == -INFINITY ? 0.0f : ex2_approx(__fsub_rn(t[k][1], mn)));
          sum = __fadd_rn(sum, __fadd_rn(__bfloat162float(r[k][0]), __bfloat162float(r[k][1])));
        }
        l[j][cc] = __fadd_rn(__fmul_rn(l[j][cc], alpha[j][cc]), sum);
        m[j][cc] = mn;
#pragma unroll
        for (int k = 0; k < NC; ++k) {
          // column cc of rows g and g + 8 of chunk k
          if (cc == 0) {
            pb[k][j][0] = (uint32_t)__bfloat16_as_ushort(r[k][0]);
            pb[k][j][1] = (uint32_t)__bfloat16_as_ushort(r[k][1]);
          } else {
            pb[k][j][0] |= (uint32_t)__bfloat16_as_ushort(r[k][0]) << 16;
            pb[k][j][1] |= (uint32_t)__bfloat16_as_ushort(r[k][1]) << 16;
          }
        }
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
      if (k >= nc) break;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int row = k * 16 + (lane & 7) + ((lane >> 4) << 3);
        const int ch = ((i & 3) << 1) + ((lane >> 3) & 1);
        uint32_t a[4];
        ldmatrix_x4_trans(a, vb + (uint32_t)(i >> 2) * kAttnHalfBytes + (uint32_t)row * 128u +
                                 (uint32_t)((ch ^ (row & 7)) << 4));
#pragma unroll
        for (int j = 0; j < NT; ++j) mma_m16n8k16_bf16(o[i][j], a, pb[k][j][0], pb[k][j][1]);
      }
    }
    __syncwarp();  // every lane is done with the stage before it is refilled
    ++consumed;
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
      float* rec = p.part + (((int64_t)it.b * p.Hkv + it.kvh) * (int64_t)p.n_split + it.s) *
                                (int64_t)((kAttnD + 2) * GP);
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
        attn_drain(smem_u32(&full[warp][k % kAttnStages]), (uint32_t)(k / kAttnStages) & 1u, p.status);
    __syncwarp();
  }
}

// ---------------------------------------------------------------------------
// combine
// ---------------------------------------------------------------------------

// One CTA per (key/value head, slice of 128 / SL d, request): folds the
// request's split records in split order and writes out[b][h][d] for the
// group's heads and the slice's d.  Thread t owns head h = t % GP and the
// values d = t / GP + (256 / GP) i of the slice; a record holds o[d][h], then
// m[h] and l[h], so the CTA's loads of one record are contiguous.  The records
// are read straight from L2 (the previous kernel just wrote them), several
// records' loads at a time.  SL changes no operation: every (h, d) folds the
// same records in the same order.  Slicing only pays when there are few
// (request, head) pairs, so the host takes SL = 4 when there are fewer pairs
// than SMs.
constexpr int kCombThreads = 256;

template <int NT, int SL>
__global__ void __launch_bounds__(kCombThreads) decode_attn_combine_kernel(const AttnParams p, __nv_bfloat16* out) {
  constexpr int GP = 8 * NT;
  constexpr int SD = kAttnD / SL;                  // d values of the slice
  constexpr int RS = (kAttnD + 2) * GP;            // floats per record
  constexpr int DSTEP = kCombThreads / GP;         // distance between a thread's d values
  constexpr int DPT = SD / DSTEP;                  // d values per thread
  // records whose loads are in flight together (about 32 values per thread)
  constexpr int kCombAhead = 32 / DPT < 4 ? 4 : (32 / DPT > 16 ? 16 : 32 / DPT);
  grid_dep_launch_dependents();
  grid_dep_wait();  // the split records come from the previous kernel
  const int kvh = blockIdx.x / SL, slice = blockIdx.x % SL;
  const int t = threadIdx.x, h = t % GP, d0 = t / GP;
  const int64_t b = blockIdx.y;
  const int64_t L = p.seq_lens[b];
  __nv_bfloat16* ob = out + (b * p.Hq + (int64_t)kvh * p.G + h) * kAttnD + slice * SD;
  if (L <= 0 || L > p.max_len) {
    // an empty request gives zeros; an invalid length (flagged by the plan
    // kernel) gives NaN
    if (h < p.G) {
      const __nv_bfloat16 v = __float2bfloat16_rn(L == 0 ? 0.0f : __int_as_float(0x7fc00000));
#pragma unroll
      for (int i = 0; i < DPT; ++i) ob[d0 + DSTEP * i] = v;
    }
    return;
  }
  const int ns = (int)((L + p.split_size - 1) / p.split_size);
  const float* rec0 = p.part + (b * p.Hkv + kvh) * (int64_t)p.n_split * RS;
  float m = 0.0f, l = 0.0f, o[DPT];
  for (int r0 = 0; r0 < ns; r0 += kCombAhead) {
    float mv[kCombAhead], lv[kCombAhead], ov[kCombAhead][DPT];
#pragma unroll
    for (int u = 0; u < kCombAhead; ++u) {
      if (r0 + u < ns) {
        const float* rec = rec0 + (int64_t)(r0 + u) * RS;
        mv[u] = __ldcg(rec + kAttnD * GP + h);
        lv[u] = __ldcg(rec + (kAttnD + 1) * GP + h);
#pragma unroll
        for (int i = 0; i < DPT; ++i) ov[u][i] = __ldcg(rec + slice * SD * GP + t + kCombThreads * i);
      }
    }
#pragma unroll
    for (int u = 0; u < kCombAhead; ++u) {
      if (r0 + u >= ns) break;
      if (r0 + u == 0) {
        m = mv[u];
        l = lv[u];
#pragma unroll
        for (int i = 0; i < DPT; ++i) o[i] = ov[u][i];
      } else {
        float mm, a1, a2;
        attn_scales(m, mv[u], mm, a1, a2);
        l = __fadd_rn(__fmul_rn(l, a1), __fmul_rn(lv[u], a2));
#pragma unroll
        for (int i = 0; i < DPT; ++i) o[i] = __fadd_rn(__fmul_rn(o[i], a1), __fmul_rn(ov[u][i], a2));
        m = mm;
      }
    }
  }
  if (h < p.G) {
#pragma unroll
    for (int i = 0; i < DPT; ++i) ob[d0 + DSTEP * i] = __float2bfloat16_rn(__fdiv_rn(o[i], l));
  }
}

template <int NT>
static cudaError_t launch_attn_t(const AttnLaunch& A) {
  // the shared-memory limits are per device: set them once for each
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t de = cudaGetDevice(&dev);
  if (de != cudaSuccess) return de;
  const uint64_t bit = dev < 64 ? (uint64_t)1 << dev : 0;
  if (!bit || !(configured.load() & bit)) {
    cudaError_t e = cudaFuncSetAttribute(decode_attn_stream_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         AttnCfg<NT>::smem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit);
  }
  cudaError_t e = launch_overlapped(decode_attn_plan_kernel, dim3(1), dim3(kPlanThreads), A.stream, A.p, A.B);
  if (e != cudaSuccess) return e;
  e = launch_overlapped_smem(decode_attn_stream_kernel<NT>, dim3((unsigned)A.grid), dim3(32 * AttnCfg<NT>::warps),
                             AttnCfg<NT>::smem, A.stream, A.tmK, A.tmV, A.p);
  if (e != cudaSuccess) return e;
  if ((int64_t)A.B * A.p.Hkv < A.grid)
    return launch_overlapped(decode_attn_combine_kernel<NT, 4>, dim3((unsigned)(A.p.Hkv * 4), (unsigned)A.B),
                             dim3(kCombThreads), A.stream, A.p, A.out);
  return launch_overlapped(decode_attn_combine_kernel<NT, 1>, dim3((unsigned)A.p.Hkv, (unsigned)A.B),
                           dim3(kCombThreads), A.stream, A.p, A.out);
}

cudaError_t launch_decode_attention(const AttnLaunch& A) {
  return A.p.G <= 8 ? launch_attn_t<1>(A) : launch_attn_t<2>(A);
}

}  // namespace bi
