// gemm_kernel.cuh -- the batch-invariant GEMM kernel on the 5th-generation
// tensor cores, and its launch templates (instantiated by gemm.cu and
// gemm_fused.cu).
//
// Y[M,N] = X[M,K] . W[N,K]^T with fp32 accumulation in tensor memory (TMEM).
//
// The reduction tree of every output element y[m,n] is fixed by (N, K, pins):
//   * K is cut into K tiles of 64 elements; split s (0 <= s < S) owns K tiles
//     [floor(s*KT/S), floor((s+1)*KT/S)).
//   * Inside a split, the partial acc_s is one chain of tcgen05.mma
//     instructions of shape (128 * mma_ctas) x T x 16 in ascending k, the first
//     of which overwrites the accumulator.  W rows sit on the MMA's M side
//     (TMEM lanes), tokens on its N side (TMEM columns).  T and mma_ctas
//     (cta_group::1, or cta_group::2 across a CTA pair) are pins.
//   * The partials are added in ascending s in fp32: (((acc_0 + acc_1) + acc_2) ...).
// CoRun (Padding is Simple and Efficient for Deterministic LLM Inference),
// Sec. III-A, Fig. 3(b): a batch-invariant reduction uses one fixed partition
// and one fixed combine order at every batch size.  Detent, Sec. 7, keeps
// split-KV in attention with split boundaries set by a fixed split size; here
// the split count and boundaries are pins in the same spirit.
//
// What may depend on M (and changes no bit): the number of token tiles, the
// grid, which SM runs which tile, how many token rows a copy brings in, the
// ring depths, and whether the S chains of a tile run on one CTA (pair) or on a
// cluster (LOCAL vs CLUSTER):
//   LOCAL   a persistent CTA (pair) walks its tiles; for each tile it runs the S
//           chains one after the other into two ping-pong TMEM accumulators;
//           the epilogue warps fold them into registers as they complete.
//   CLUSTER each CTA (pair) of a cluster runs one chain; the partials go to
//           shared memory and are folded in ascending split order through
//           distributed shared memory.  No atomics and no global workspace.
//
// Warp roles (608 threads): warp 0 = W producer (TMA, one lane), warp 1 = MMA
// issuer (one lane) and TMEM owner, warp 2 = X producer, warps 3..18 =
// epilogue (four warps per TMEM lane quadrant, each owning a quarter of the T
// accumulator columns).  The fused RMSNorm form adds warps 19..22, which
// normalise each X stage in shared memory (736 threads).  W and X have
// separate shared-memory rings so that the W stream (from HBM) can run further
// ahead than the X stream.
//
// In a CTA pair (mma_ctas = 2) both CTAs load their own W rows and their half
// of the token rows; the even CTA waits for both halves on its own mbarriers,
// issues the cta_group::2 MMAs, and its commits free both CTAs' stages
// (multicast).  Both CTAs' epilogues release an accumulator on the even CTA's
// barrier.
//
// Every wait is bounded (2 s of wall clock).  When one runs out, the kernel
// records BI_ERR_DEVICE_TIMEOUT in a device status word, every role abandons
// its work, in-flight copies and MMAs are drained (again with bounded waits),
// tensor memory is freed and the CTA returns normally.
#pragma once

#include <atomic>

#include <cuda_bf16.h>

#include "internal.h"
#include "bounds.cuh"
#include "ptx.cuh"
#include "rowmath.cuh"

namespace bi {

constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct GemmParams {
  __nv_bfloat16* Y;
  int64_t M, N, K;
  int32_t n_tiles, m_tiles, k_tiles, S;
  int32_t w_stages, x_stages, x_box_rows;
  int32_t group_n;  // LOCAL tile order: groups of group_n W tiles (speed only)
  int32_t units;    // CLUSTER: units (CTAs or pairs) per tile; S (one split each) or ceil(S/2)
  const float* sx;  // FP8: per-token scales [M]
  const float* sw;  // FP8: per-channel scales [N]
  const __nv_bfloat16* g;  // FUSED: RMSNorm gain [K]
  const float* rrow;       // FUSED: r = 1 / sqrt(mean(x^2) + eps) of each row [M], or
                           // nullptr: computed in the kernel (M <= kRowScaleInKernelMax)
  const __nv_bfloat16* xraw;  // FUSED with rrow == nullptr: X [M,K], for the sums of squares
  float eps;
  float* fold_part;        // GLOBAL: chain partials [n_tiles * S][T][128] fp32, or nullptr (other schedules)
  uint32_t* fold_count;    // GLOBAL: per-tile arrival counts, zero between calls
  int* status;             // device status word: 0, or the bi_status of a call that gave up
  uint32_t flags;  // BI_FLAG_DEBUG_STALL_PRODUCER | kFlagStreamW | kFlagZeroX
};

struct __align__(8) SmemCtl {
  uint64_t w_full[kMaxStages];
  uint64_t w_empty[kMaxStages];
  uint64_t x_full[kMaxStages];
  uint64_t x_empty[kMaxStages];
  uint64_t x_ready[kMaxStages];  // FUSED: the stage's X rows are normalised in place
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
  float rrow[kRowScaleInKernelMax];  // FUSED, tiny batches: r of the CTA's rows, computed here
  int fold_last;                     // GLOBAL: this chain was its tile's last to finish
};
static_assert(sizeof(SmemCtl) <= kCtlBytes, "control block too large");

__device__ __forceinline__ void record_stall(int* status) {
  atomicCAS(status, 0, (int)BI_ERR_DEVICE_TIMEOUT);
}

// Slow path of wait_or_abort: polls until the phase completes, the CTA starts
// abandoning the call, or kWaitLimitNs pass (then it starts the abandonment).
// CL: acquire at cluster scope (the phase completes on arrivals of another CTA
// of the cluster, whose shared-memory writes must be visible afterwards).
template <bool CL>
__device__ __noinline__ bool wait_or_abort_slow(uint32_t bar, uint32_t parity, volatile int* abort, int* status) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (CL ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      record_stall(status);
      return false;
    }
  }
}

// Waits for the phase of `parity` on `bar`; false if the call is abandoned.
template <bool CL = false>
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort, int* status) {
  if (CL ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
  return wait_or_abort_slow<CL>(bar, parity, abort, status);
}

// Bounded wait that ignores the abort flag (for draining work in flight).
static __device__ __noinline__ bool wait_drain(uint32_t bar, uint32_t parity, int* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      record_stall(status);
      return false;
    }
  }
}

__device__ __forceinline__ int64_t split_begin(int32_t s, int32_t S, int32_t KT) {
  return ((int64_t)s * KT) / S;
}

// LOCAL tile order.  Tiles come in groups of G consecutive W tiles (the last
// group may be narrower); within a group the token tiles run slowest.  Units
// working on consecutive tiles then share G W tiles and about units / G token
// tiles, a working set that stays in L2 even when W does not.  Each tile's
// result is independent of when it is computed.
__device__ __forceinline__ void tile_coords(int64_t t, int32_t n_tiles, int32_t m_tiles, int32_t G,
                                            int32_t* n_tile, int32_t* m_tile) {
  const int64_t full = (int64_t)(n_tiles / G) * G * m_tiles;  // tiles in full-width groups
  if (t < full) {
    const int64_t per = (int64_t)G * m_tiles;
    const int64_t g = t / per, r = t % per;
    *n_tile = (int32_t)(g * G + r % G);
    *m_tile = (int32_t)(r / G);
  } else {
    const int32_t w = n_tiles % G;  // width of the last group
    const int64_t r = t - full;
    *n_tile = (int32_t)((n_tiles / G) * G + r % w);
    *m_tile = (int32_t)(r / w);
  }
}

// Epilogue of the GLOBAL schedule (single-CTA MMAs, one chain per work
// item).  Each chain's partial goes to the workspace as [item][column][W row]
// fp32, columns below M only.  The epilogue warps then publish it (fence,
// barrier) and count the chain in on its tile's arrival counter; the chain
// whose arrival completes the count folds the tile's S partials from the
// workspace in ascending split order, (((P0 + P1) + P2) + ...), the order of
// the register and shared-memory folds, writes Y and sets the counter back to
// zero.  Nobody waits on anybody: the count only decides who folds.  The
// atomic touches the count, never a value.  Every barrier is taken by all
// 16 epilogue warps; a bounded wait that runs out is agreed on by all of
// them (bar.red.and) before anyone leaves.
constexpr int kFoldMaxS = BI_GLOBAL_MAX_SPLIT_K;  // splits the GLOBAL schedule folds (one column group's loads in flight together)

template <int T, bool FP8, typename Work>
__device__ __forceinline__ void global_fold_epilogue(const GemmParams& p, SmemCtl* ctl, uint32_t tmem_base,
                                                     volatile int* abort, int64_t tile_first, int64_t tile_step,
                                                     int64_t tile_end, int32_t S, Work&& work) {
  constexpr int kColGroups = kEpiWarps / 4;
  constexpr int kHalf = T / kColGroups;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ew = warp - kFirstEpiWarp;
  const int quad = warp & 3, half = ew >> 2;
  const int n_local = quad * 32 + lane;
  const uint32_t t_lane = (uint32_t)(quad * 32) << 16;
  const int et = (int)threadIdx.x - 32 * kFirstEpiWarp;  // 0 .. 511
  const int frow = et & (kTileN - 1);                      // fold: this thread's W row
  const int fcol = et >> 7;                                // and first column (then every 4th)
  uint32_t acc_iter = 0;
  for (int64_t t = tile_first; t < tile_end; t += tile_step) {
    int32_t n_tile, m_tile, s_lo, s_hi;
    work(t, n_tile, m_tile, s_lo, s_hi);
    const int64_t tile = t / S;
    const uint32_t buf = acc_iter & 1u;
    const uint32_t acc_phase = (acc_iter >> 1) & 1u;
    const bool got = wait_or_abort(smem_u32(&ctl->acc_full[buf]), acc_phase, abort, p.status);
    if (!named_barrier_and(2, 32 * kEpiWarps, got)) return;
    tc_fence_after();
    const int64_t mt0 = (int64_t)m_tile * T;              // the tile's first token
    const int64_t mrem = p.M - mt0;
    const int mvt = mrem < T ? (int)mrem : T;              // valid tokens of the tile
    const int mv = min(max(mvt - half * kHalf, 0), kHalf);  // ... in this warp's columns
    float* part = p.fold_part + ((int64_t)t * T + half * kHalf) * kTileN + n_local;
    const uint32_t taddr = tmem_base + t_lane + buf * (uint32_t)T + (uint32_t)(half * kHalf);
    // debug-bounds build: the chain's partial within the workspace's tiles * S
    // partials, its columns within the allocation
    const bool part_ok =
        bounds_ok(t >= 0 && t < (int64_t)p.n_tiles * p.m_tiles * S, p.status, kChkFoldPart, (uint64_t)t) &&
        bounds_ok(buf * (uint32_t)T + (uint32_t)(half * kHalf + kHalf) <= 2u * (uint32_t)T, p.status, kChkTmemCol,
                  (uint64_t)(buf * T + half * kHalf));
#pragma unroll
    for (int c = 0; c < kHalf; c += 4) {
      if (c < mv && part_ok) {
        float v[4];
        tmem_ld4(taddr + (uint32_t)c, v);
#pragma unroll
        for (int i = 0; i < 4; ++i)
          if (c + i < mv) __stcg(part + (int64_t)(c + i) * kTileN, v[i]);
      }
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&ctl->acc_empty[buf]));
    ++acc_iter;
    __threadfence();  // the partial is visible before the count
    named_barrier_sync(2, 32 * kEpiWarps);
    if (et == 0) {
      int last = 0;
      if (bounds_ok(tile >= 0 && tile < (int64_t)p.n_tiles * p.m_tiles, p.status, kChkFoldTile, (uint64_t)tile)) {
        const uint32_t before = atomicAdd(p.fold_count + tile, 1u);
        last = before == (uint32_t)(S - 1);
        if (last) p.fold_count[tile] = 0u;  // all S chains counted in: zero for the next call
      }
      ctl->fold_last = last;
    }
    named_barrier_sync(2, 32 * kEpiWarps);
    if (!ctl->fold_last) continue;
    __threadfence();
    const int64_t n = (int64_t)n_tile * kTileN + frow;
    if (n < p.N) {
      const float* P0 = p.fold_part + tile * S * T * kTileN + frow;  // split 0 of this tile, column 0
      const float swn = FP8 ? p.sw[n] : 1.0f;
      // columns fcol, fcol + 4, ...: four of them at a time, all S loads in flight
      for (int c0 = fcol; c0 < mvt; c0 += 16) {
        float v[4][kFoldMaxS];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int q = 0; q < kFoldMaxS; ++q) {
            const int c = c0 + 4 * i;
            v[i][q] = (q < S && c < mvt) ? __ldcg(P0 + ((int64_t)q * T + c) * kTileN) : 0.0f;
          }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int c = c0 + 4 * i;
          if (c >= mvt) break;
          float acc = v[i][0];
#pragma unroll
          for (int q = 1; q < kFoldMaxS; ++q)
            if (q < S) acc = __fadd_rn(acc, v[i][q]);
          if (FP8) acc = __fmul_rn(__fmul_rn(acc, p.sx[mt0 + c]), swn);
          p.Y[(mt0 + c) * p.N + n] = __float2bfloat16_rn(acc);
        }
      }
    }
  }
}

// KP: K tiles per ring stage (1 or 2).  With KP = 2 a stage is one copy of a
// 3-D box (the [K/64][rows][64] view), or, with kFlagCopy2D, two copies of
// 2-D boxes landing one K tile apart (any K, and X boxes shorter than the
// stage's rows).  The MMAs consume the K tiles of a stage one after the
// other, so KP never changes the reduction; it halves the waits and commits
// per MMA of the issuing thread, which at T = 256 runs close to the tensor
// pipe's rate, and a W stage then covers 256 contiguous bytes of each of its
// 128 rows, which HBM serves faster than 128.
// FP8: E4M3 operands (kind::f8f6f4); a K tile is then 128 values (still 128
// bytes), and the epilogue scales the fp32 result by sx[m] and then sw[n]
// before rounding to bf16.
// FUSED: X holds raw activations, and the RMSNorm prologue runs in shared
// memory.  A warpgroup of transform warps waits for each X stage to land,
// replaces every value x of row m and column k by bf16_rne((x * r[m]) * g[k])
// in place -- the arithmetic and rounding of the standalone RMSNorm, with r[m]
// computed beforehand by the same lane partition and butterfly -- and only
// then releases the stage to the MMA.  The normalised rows never leave the SM.
template <int T, bool CLUSTER, bool PAIR, int KP, bool FP8, bool FUSED>
__global__ void __launch_bounds__(gemm_threads(FUSED), 1)
    bi_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const GemmParams p) {
  constexpr int kXRows = PAIR ? T / 2 : T;          // token rows in this CTA's X tiles
  constexpr int kXTile = kXRows * kBK * 2;          // one K tile of X
  constexpr int kXStage = KP * kXTile;
  constexpr int kWStage = KP * kWStageBytes;
  constexpr int kTileElems = FP8 ? 128 : kBK;       // K values per K tile
  constexpr int kMmaM = PAIR ? 2 * kTileN : kTileN;  // W rows per tile
  // two accumulators of T columns; the allocation is a power of two >= 32
  constexpr uint32_t kTmemCols = 2u * (uint32_t)T <= 128u ? 128u : (2u * (uint32_t)T <= 256u ? 256u : 512u);
  static_assert(T % 32 == 0 && T >= 64 && T <= 256, "token tile");
  constexpr int kColGroups = kEpiWarps / 4;   // epilogue warps per TMEM lane quadrant
  constexpr int kHalf = T / kColGroups;      // accumulator columns per epilogue warp

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int ws = p.w_stages;
  const int xs = p.x_stages;
  const int64_t w_ring = (int64_t)ws * kWStage;
  const int64_t ring_bytes = w_ring + (int64_t)xs * kXStage;
  const int64_t part_bytes = CLUSTER ? (int64_t)T * kTileN * 4 : 0;
  SmemCtl* ctl = reinterpret_cast<SmemCtl*>(smem + (ring_bytes > part_bytes ? ring_bytes : part_bytes));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t smem_base = smem_u32(smem);
  const uint32_t w_base = smem_base;                       // W stage i at w_base + i * kWStage
  const uint32_t x_base = smem_base + (uint32_t)w_ring;    // X stage i at x_base + i * kXStage

  const uint32_t crank = (PAIR || CLUSTER) ? cluster_ctarank() : 0u;
  const uint32_t peer = PAIR ? (crank & 1u) : 0u;          // 0 = the pair's MMA-issuing CTA
  const bool leader = peer == 0;
  const uint32_t leader_rank = crank & ~1u;
  const uint16_t pair_mask = (uint16_t)(3u << leader_rank);

  if (threadIdx.x == 0) {
    for (int i = 0; i < ws; ++i) {
      mbar_init(smem_u32(&ctl->w_full[i]), 1);
      mbar_init(smem_u32(&ctl->w_empty[i]), 1);
    }
    for (int i = 0; i < xs; ++i) {
      mbar_init(smem_u32(&ctl->x_full[i]), 1);
      mbar_init(smem_u32(&ctl->x_empty[i]), 1);
      // every transform warp of the pair arrives on the MMA-issuing CTA's barrier
      if constexpr (FUSED) mbar_init(smem_u32(&ctl->x_ready[i]), kXformWarps * (PAIR ? 2 : 1));
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ctl->acc_full[b]), 1);
      mbar_init(smem_u32(&ctl->acc_empty[b]), kEpiWarps * (PAIR ? 2 : 1));
    }
    mbar_init(smem_u32(&ctl->mma_done), 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  // In a pair, the peer's barriers must be initialised before anyone signals them.
  if constexpr (PAIR) cluster_sync();
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmW);
    prefetch_tensormap(&tmX);
  }
  // The next kernel in the stream may be scheduled now; it waits for this
  // grid before touching memory.
  if (threadIdx.x == 0) grid_dep_launch_dependents();
  if (warp == 1) {
    if constexpr (PAIR) {
      tmem_alloc_pair(smem_u32(&ctl->tmem_base), kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(smem_u32(&ctl->tmem_base), kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  volatile int* abort = &ctl->abort;

  const int32_t S = p.S;
  const int32_t KT = p.k_tiles;
  const int64_t num_tiles = (int64_t)p.n_tiles * p.m_tiles;
  // Work list.  CLUSTER: one tile (blockIdx.y, blockIdx.z); cluster unit u
  // (the cluster rank, counted in pairs when PAIR) of U runs splits
  // [floor(u*S/U), floor((u+1)*S/U)): one split each when U = S, one or two
  // when U = ceil(S/2) (chained).  LOCAL: tiles u, u + U, ... for unit u of U
  // (a unit is a CTA, or a CTA pair), all S splits of each.  GLOBAL (a LOCAL
  // kernel of single-CTA MMAs given a fold workspace): the work items are
  // the chains (tile, split), unit u taking items u, u + U, ...; each chain's
  // partial goes to the workspace, and the last of a tile's S chains to
  // finish folds them there in ascending split order.
  const int32_t U = CLUSTER ? p.units : 1;
  const bool chained = CLUSTER && U != S;
  const bool gfold = !CLUSTER && !PAIR && p.fold_part != nullptr;
  const int32_t my_unit = CLUSTER ? (int32_t)(PAIR ? (crank >> 1) : crank) : 0;
  const int64_t unit = PAIR ? (blockIdx.x >> 1) : blockIdx.x;
  const int64_t units = PAIR ? (gridDim.x >> 1) : gridDim.x;
  const int64_t tile_first = CLUSTER ? 0 : unit;
  const int64_t tile_step = CLUSTER ? 1 : units;
  const int64_t tile_end = CLUSTER ? 1 : (gfold ? num_tiles * S : num_tiles);
  const int32_t s_first = CLUSTER ? (int32_t)(((int64_t)my_unit * S) / U) : 0;
  const int32_t s_end = CLUSTER ? (int32_t)(((int64_t)(my_unit + 1) * S) / U) : S;
  // work item t -> its tile and its splits [s_lo, s_hi)
  auto work = [&](int64_t t, int32_t& n_tile, int32_t& m_tile, int32_t& s_lo, int32_t& s_hi) {
    if (CLUSTER) {
      n_tile = (int32_t)blockIdx.y;
      m_tile = (int32_t)blockIdx.z;
      s_lo = s_first;
      s_hi = s_end;
      return;
    }
    tile_coords(gfold ? t / S : t, p.n_tiles, p.m_tiles, p.group_n, &n_tile, &m_tile);
    s_lo = gfold ? (int32_t)(t % S) : 0;
    s_hi = gfold ? s_lo + 1 : S;
  };
  const bool stream_w = (p.flags & kFlagStreamW) != 0;
  bool chain_ok = false;  // epilogue threads of a CLUSTER unit: its chains completed

  if (warp == 0 || warp == 2) {
    // ------------------------------------------------ producers (W: warp 0, X: warp 2)
    const bool is_w = warp == 0;
    if (!is_w && (p.flags & kFlagZeroX)) {
      // The X boxes cover fewer rows than the MMA reads: zero the whole X ring
      // once; the loads then only ever overwrite the leading rows.
      const uint4 z = make_uint4(0, 0, 0, 0);
      for (int64_t off = (int64_t)lane * 16; off < (int64_t)xs * kXStage; off += 32 * 16)
        *reinterpret_cast<uint4*>(smem + w_ring + off) = z;
      fence_proxy_async_smem();
      __syncwarp();
    }
    if (lane == 0) {
      // In a fused pair each CTA's X copies complete on its own barrier: its
      // transform warps must see them land before normalising the rows.
      const bool local_x = FUSED && PAIR && !is_w;
      // Inputs may come from the previous kernel in the stream: wait for it
      // before the first copy (W may start earlier when the caller allows).
      if (!is_w || (p.flags & BI_FLAG_PREFETCH_W) == 0) grid_dep_wait();
      const bool stall = is_w && (p.flags & BI_FLAG_DEBUG_STALL_PRODUCER) != 0;
      const int nst = is_w ? ws : xs;
      uint64_t* full_bar = is_w ? ctl->w_full : ctl->x_full;
      uint64_t* empty_bar = is_w ? ctl->w_empty : ctl->x_empty;
      const uint32_t ring = is_w ? w_base : x_base;
      const uint32_t stage_sz = is_w ? (uint32_t)kWStage : (uint32_t)kXStage;
      // transaction bytes per stage (whole boxes, also where one lies past K),
      // both CTAs of a pair counted on the even CTA
      const uint32_t tx = (uint32_t)KP * (is_w ? (uint32_t)kWStageBytes : (uint32_t)p.x_box_rows * kBK * 2) *
                          ((PAIR && !local_x) ? 2u : 1u);
      const CUtensorMap* map = is_w ? &tmW : &tmX;
      const bool hinted = stream_w;
      const bool copy2d = (p.flags & kFlagCopy2D) != 0;
      const uint64_t policy = is_w ? policy_evict_first() : policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int64_t t = tile_first; ok && t < tile_end; t += tile_step) {
        int32_t n_tile, m_tile, s_lo, s_hi;
        work(t, n_tile, m_tile, s_lo, s_hi);
        const int32_t row = is_w ? n_tile * kMmaM + (int32_t)peer * kTileN
                                 : m_tile * T + (int32_t)peer * kXRows;
        for (int32_t s = s_lo; ok && s < s_hi; ++s) {
          const int64_t k0 = split_begin(s, S, KT), k1 = split_begin(s + 1, S, KT);
          // the last copy of a split may reach one K tile past it (loaded, unused)
          for (int64_t kt = k0; kt < k1; kt += KP) {
            if (!wait_or_abort(smem_u32(&empty_bar[stage]), phase ^ 1u, abort, p.status)) {
              ok = false;
              break;
            }
            // debug-bounds build: the stage, the K tile and the row of the copy
#ifdef BI_DEBUG_BOUNDS
            const int32_t row_c = (is_w && issued == 0 && (p.flags & kFlagDebugPokeWRow)) ? row + (1 << 24) : row;
#else
            const int32_t row_c = row;
#endif
            const bool in_bounds =
                bounds_ok(stage < nst, p.status, is_w ? kChkWStage : kChkXStage, (uint64_t)stage) &&
                bounds_ok(kt >= 0 && kt < KT, p.status, kChkKTile, (uint64_t)kt) &&
                bounds_ok(is_w ? row_c < p.n_tiles * kMmaM : row_c < p.m_tiles * T, p.status,
                          is_w ? kChkWRow : kChkXRow, (uint64_t)row_c);
            if (!(stall && issued == 0) && in_bounds) {
              const uint32_t full = smem_u32(&full_bar[stage]);
              const uint32_t dst = ring + (uint32_t)stage * stage_sz;
              const int32_t kx = (int32_t)(kt * kTileElems);  // 2-D maps: element column
              const int32_t kz = (int32_t)kt;          // 3-D maps: K tile index
              if (PAIR && local_x) {
                mbar_arrive_expect_tx(full, tx);
                if constexpr (KP == 1) {
                  if (hinted)
                    tma_load_2d_hint(dst, map, full, kx, row, policy);
                  else
                    tma_load_2d(dst, map, full, kx, row);
                } else {
                  if (hinted)
                    tma_load_3d_hint(dst, map, full, 0, row, kz, policy);
                  else
                    tma_load_3d(dst, map, full, 0, row, kz);
                }
              } else if constexpr (PAIR) {
                const uint32_t bar = leader ? full : mapa_shared(full, leader_rank);
                if (leader) mbar_arrive_expect_tx(full, tx);
                if constexpr (KP == 1) {
                  if (hinted)
                    tma_load_2d_pair_hint(dst, map, bar, kx, row, policy);
                  else
                    tma_load_2d_pair(dst, map, bar, kx, row);
                } else {
                  if (hinted)
                    tma_load_3d_pair_hint(dst, map, bar, 0, row, kz, policy);
                  else
                    tma_load_3d_pair(dst, map, bar, 0, row, kz);
                }
              } else {
                mbar_arrive_expect_tx(full, tx);
                if constexpr (KP == 1) {
                  if (hinted)
                    tma_load_2d_hint(dst, map, full, kx, row, policy);
                  else
                    tma_load_2d(dst, map, full, kx, row);
                } else if (copy2d) {
                  // K tiles kt and kt + 1, one tile of this operand apart
                  const uint32_t sub = is_w ? (uint32_t)kWStageBytes : (uint32_t)kXTile;
                  for (int j = 0; j < KP; ++j) {
                    if (hinted)
                      tma_load_2d_hint(dst + j * sub, map, full, kx + j * kTileElems, row, policy);
                    else
                      tma_load_2d(dst + j * sub, map, full, kx + j * kTileElems, row);
                  }
                } else {
                  if (hinted)
                    tma_load_3d_hint(dst, map, full, 0, row, kz, policy);
                  else
                    tma_load_3d(dst, map, full, 0, row, kz);
                }
              }
            }
            ++issued;
            if (++stage == nst) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      // Drain: the copies of the last `nst` loads must have landed before the
      // CTA may exit (they write into this CTA's shared memory).  In a pair the
      // odd CTA's copies complete on the even CTA's barriers, which that CTA
      // drains; both CTAs meet at a cluster barrier before either exits.
      // (A fused pair's X copies complete on each CTA's own barriers.)
      if (leader || local_x) {
        const int64_t first = issued > nst ? issued - nst : 0;
        for (int64_t i = first; i < issued; ++i) {
          if (stall && i == 0) continue;
          wait_drain(smem_u32(&full_bar[i % nst]), (uint32_t)((i / nst) & 1), p.status);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0 && leader) {
      constexpr uint32_t idesc = FP8 ? make_idesc_e4m3(kMmaM, T) : make_idesc_bf16(kMmaM, T);
      int wi = 0, xi = 0;
      uint32_t wph = 0, xph = 0;
      uint32_t acc_iter = 0;
      bool ok = true;
      for (int64_t t = tile_first; ok && t < tile_end; t += tile_step) {
        int32_t n_tile, m_tile, s_lo, s_hi;
        work(t, n_tile, m_tile, s_lo, s_hi);
        for (int32_t s = s_lo; ok && s < s_hi; ++s) {
          const uint32_t buf = acc_iter & 1u;
          const uint32_t acc_phase = (acc_iter >> 1) & 1u;
          if (!wait_or_abort(smem_u32(&ctl->acc_empty[buf]), acc_phase ^ 1u, abort, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (!bounds_ok(buf * (uint32_t)T + (uint32_t)T <= kTmemCols && wi < ws && xi < xs, p.status, kChkTmemCol,
                         (uint64_t)buf * T)) {
            ok = false;
            break;
          }
          const uint32_t d_tmem = tmem_base + buf * (uint32_t)T;
          const int64_t k0 = split_begin(s, S, KT), k1 = split_begin(s + 1, S, KT);
          for (int64_t kt = k0; kt < k1; kt += KP) {
            // FUSED: the X stage is ready once the transform warps (of both
            // CTAs of a pair) have normalised it
            bool ready = wait_or_abort(smem_u32(&ctl->w_full[wi]), wph, abort, p.status);
            if (ready)
              ready = FUSED ? wait_or_abort<PAIR>(smem_u32(&ctl->x_ready[xi]), xph, abort, p.status)
                            : wait_or_abort(smem_u32(&ctl->x_full[xi]), xph, abort, p.status);
            if (!ready) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint64_t a_desc = make_sdesc_sw128(w_base + (uint32_t)wi * kWStage);
            const uint64_t b_desc = make_sdesc_sw128(x_base + (uint32_t)xi * kXStage);
#pragma unroll
            for (int sub = 0; sub < KP; ++sub) {
              // sub-tile sub holds K tile kt + sub (absent past the split's end)
              if (sub > 0 && kt + sub >= k1) break;
#pragma unroll
              for (int j = 0; j < kBK / kMmaK; ++j) {
                // +32 bytes per 16 K elements, in the descriptor's 16-byte units
                const uint64_t da = (uint64_t)(sub * (kWStageBytes >> 4) + 2 * j);
                const uint64_t db = (uint64_t)(sub * (kXTile >> 4) + 2 * j);
                const uint32_t acc = (kt > k0 || sub > 0 || j > 0) ? 1u : 0u;
                if constexpr (PAIR && FP8)
                  mma_e4m3_pair(d_tmem, a_desc + da, b_desc + db, idesc, acc);
                else if constexpr (PAIR)
                  mma_bf16_pair(d_tmem, a_desc + da, b_desc + db, idesc, acc);
                else if constexpr (FP8)
                  mma_e4m3(d_tmem, a_desc + da, b_desc + db, idesc, acc);
                else
                  mma_bf16(d_tmem, a_desc + da, b_desc + db, idesc, acc);
              }
            }
            if constexpr (PAIR) {
              mma_commit_pair_mc(smem_u32(&ctl->w_empty[wi]), pair_mask);
              mma_commit_pair_mc(smem_u32(&ctl->x_empty[xi]), pair_mask);
            } else {
              mma_commit(smem_u32(&ctl->w_empty[wi]));
              mma_commit(smem_u32(&ctl->x_empty[xi]));
            }
            if (++wi == ws) {
              wi = 0;
              wph ^= 1u;
            }
            if (++xi == xs) {
              xi = 0;
              xph ^= 1u;
            }
          }
          if (!ok) break;
          if constexpr (PAIR)
            mma_commit_pair_mc(smem_u32(&ctl->acc_full[buf]), pair_mask);
          else
            mma_commit(smem_u32(&ctl->acc_full[buf]));
          ++acc_iter;
        }
      }
      // Every MMA this thread issued must be complete before TMEM is freed.
      if constexpr (PAIR)
        mma_commit_pair(smem_u32(&ctl->mma_done));
      else
        mma_commit(smem_u32(&ctl->mma_done));
      wait_drain(smem_u32(&ctl->mma_done), 0, p.status);
    }
  } else if (FUSED && warp >= kFirstXformWarp) {
    // ------------------------------------------------- RMSNorm prologue (FUSED)
    // Thread t normalises the 16-byte chunk at physical position t % 8 of rows
    // t / 8, t / 8 + 16, ... of each K tile.  The 128-byte swizzle stores
    // logical chunk c of row j at position c ^ (j % 8), and rows 16 apart share
    // j % 8, so a thread always holds the same 8 consecutive k of a K tile and
    // loads one gain vector per K tile.  Rows past M are left as they are
    // (zeros); the K tail past K is zero-filled and stays zero.
    constexpr int kRowsPer = kXRows / 16;
    static_assert(kXRows % 16 == 0, "token rows per CTA");
    const int xt = (int)threadIdx.x - 32 * kFirstXformWarp;
    const int pch = xt & 7;
    const int r0 = xt >> 3;
    const int lch = pch ^ (r0 & 7);
    // gain vectors of the stage at K tile kt of a split ending at k1: sub-tiles
    // past the split or columns past K get zeros (never used)
    auto load_g = [&](int64_t kt, int64_t k1, uint4 (&gv)[KP]) {
#pragma unroll
      for (int sub = 0; sub < KP; ++sub) {
        const int64_t k = (kt + sub) * kBK + lch * 8;
        gv[sub] = ((sub == 0 || kt + sub < k1) && k < p.K) ? __ldg(reinterpret_cast<const uint4*>(p.g + k))
                                                            : make_uint4(0, 0, 0, 0);
      }
    };
    uint4 gcur[KP], gnext[KP];
    // g is a weight: with BI_FLAG_PREFETCH_W the caller allows reading it
    // before the previous kernel in the stream has finished
    const bool g_early = (p.flags & BI_FLAG_PREFETCH_W) != 0;
    // the first split of work item t
    auto first_split = [&](int64_t t) -> int32_t {
      int32_t nt, mt, lo, hi;
      work(t, nt, mt, lo, hi);
      return lo;
    };
    if (g_early && tile_first < tile_end) {
      const int32_t s0 = first_split(tile_first);
      load_g(split_begin(s0, S, KT), split_begin(s0 + 1, S, KT), gcur);
    }
    grid_dep_wait();  // r, X and g may come from the previous kernel in the stream
    if (!g_early && tile_first < tile_end) {
      const int32_t s0 = first_split(tile_first);
      load_g(split_begin(s0, S, KT), split_begin(s0 + 1, S, KT), gcur);
    }
    if (p.rrow == nullptr) {
      // Tiny batch (M <= kRowScaleInKernelMax, one token tile): r of each row
      // here, one transform warp per row with the RMSNorm's lane partition,
      // order and butterfly (rowmath.cuh), so with the standalone kernel's bits.
      const int xw = warp - kFirstXformWarp;
      const int64_t nvec = p.K / 8;
      for (int row = xw; row < kRowScaleInKernelMax; row += kXformWarps) {
        if (row >= p.M) break;
        const uint4* x = reinterpret_cast<const uint4*>(p.xraw) + row * nvec;
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
        if (lane == 0) ctl->rrow[row] = inv_rms(ss, p.K, p.eps);
      }
      named_barrier_sync(1, 32 * kXformWarps);  // the transform warps only
    }
    int xi = 0;
    uint32_t xph = 0;
    bool ok = true;
    int64_t have_m0 = -1;
    int nrows = 0;
    float rr[kRowsPer];
#pragma unroll
    for (int j = 0; j < kRowsPer; ++j) rr[j] = 0.0f;
    // The gain vectors of each stage are loaded one stage ahead (the stages
    // run in the X producer's order: tile, split, K tile), so their latency
    // overlaps the wait for the stage before.
    for (int64_t t = tile_first; ok && t < tile_end; t += tile_step) {
      int32_t n_tile, m_tile, s_lo, s_hi;
      work(t, n_tile, m_tile, s_lo, s_hi);
      const int64_t m0 = (int64_t)m_tile * T + (int64_t)peer * kXRows;  // this CTA's first token row
      if (m0 != have_m0) {
        have_m0 = m0;
        const int64_t left = p.M - m0 - r0;  // rows r0 + 16 j below M
        nrows = left <= 0 ? 0 : (left >= 16 * kRowsPer ? kRowsPer : (int)((left + 15) / 16));
#pragma unroll
        for (int j = 0; j < kRowsPer; ++j)
          rr[j] = j >= nrows ? 0.0f : (p.rrow ? p.rrow[m0 + r0 + 16 * j] : ctl->rrow[m0 + r0 + 16 * j]);
      }
      for (int32_t s = s_lo; ok && s < s_hi; ++s) {
        const int64_t k0 = split_begin(s, S, KT), k1 = split_begin(s + 1, S, KT);
        for (int64_t kt = k0; kt < k1; kt += KP) {
          // the next stage: the next K tiles of this split, else the next
          // split's first, else the first split of this CTA's next work item
          if (kt + KP < k1) {
            load_g(kt + KP, k1, gnext);
          } else if (s + 1 < s_hi) {
            load_g(k1, split_begin(s + 2, S, KT), gnext);
          } else if (t + tile_step < tile_end) {
            const int32_t s0 = first_split(t + tile_step);
            load_g(split_begin(s0, S, KT), split_begin(s0 + 1, S, KT), gnext);
          }
          ok = __all_sync(0xffffffffu, wait_or_abort(smem_u32(&ctl->x_full[xi]), xph, abort, p.status));
          if (!ok) break;
#pragma unroll
          for (int sub = 0; sub < KP; ++sub) {
            if (sub > 0 && kt + sub >= k1) break;                   // loaded past the split, never used
            if ((kt + sub) * kBK + lch * 8 >= p.K) continue;       // zero-filled past K, stays zero
            const uint32_t a0 = x_base + (uint32_t)(xi * kXStage + sub * kXTile + r0 * 128 + pch * 16);
            // four rows at a time, loads before stores (16 rows = 2048 bytes apart)
#pragma unroll
            for (int j0 = 0; j0 < kRowsPer; j0 += 4) {
              uint4 v[4];
#pragma unroll
              for (int j = 0; j < 4; ++j)
                if (j0 + j < kRowsPer && j0 + j < nrows) v[j] = ld_shared_v4(a0 + (uint32_t)((j0 + j) * 2048));
#pragma unroll
              for (int j = 0; j < 4; ++j)
                if (j0 + j < kRowsPer && j0 + j < nrows)
                  st_shared_v4(a0 + (uint32_t)((j0 + j) * 2048), norm8(v[j], gcur[sub], rr[j0 + j]));
            }
          }
          // the MMA reads the stage through the async proxy
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const uint32_t rb = smem_u32(&ctl->x_ready[xi]);
            if constexpr (PAIR)
              mbar_arrive_remote(mapa_shared(rb, leader_rank));
            else
              mbar_arrive(rb);
          }
          if (++xi == xs) {
            xi = 0;
            xph ^= 1u;
          }
#pragma unroll
          for (int sub = 0; sub < KP; ++sub) gcur[sub] = gnext[sub];
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - kFirstEpiWarp;
    const int quad = warp & 3;            // TMEM lanes [32*quad, 32*quad + 32)
    const int half = ew >> 2;             // accumulator columns [half*kHalf, (half+1)*kHalf)
    const int n_local = quad * 32 + lane; // W row within this CTA's 128 rows
    const uint32_t t_lane = (uint32_t)(quad * 32) << 16;
    uint32_t acc_iter = 0;
    bool ok = true;
    if constexpr (!CLUSTER && !PAIR) {
      if (gfold) {
        global_fold_epilogue<T, FP8>(p, ctl, tmem_base, abort, tile_first, tile_step, tile_end, S, work);
        ok = false;  // the loop below is for the other schedules
      }
    }
    if constexpr (!CLUSTER) {
      for (int64_t t = tile_first; ok && t < tile_end; t += tile_step) {
        int32_t n_tile, m_tile;
        tile_coords(t, p.n_tiles, p.m_tiles, p.group_n, &n_tile, &m_tile);
        // Running sum of the splits.  It starts at -0.0, the identity of
        // IEEE addition (-0 + x == x for every x, zeros included), so the
        // first add yields P0 exactly and the sum is ((P0 + P1) + P2) + ...
        float R[kHalf];
#pragma unroll
        for (int i = 0; i < kHalf; ++i) R[i] = -0.0f;
        for (int32_t s = 0; s < S; ++s) {
          const uint32_t buf = acc_iter & 1u;
          const uint32_t acc_phase = (acc_iter >> 1) & 1u;
          bool got = wait_or_abort(smem_u32(&ctl->acc_full[buf]), acc_phase, abort, p.status);
          got = __all_sync(0xffffffffu, got);
          if (!got) {
            ok = false;
            break;
          }
          tc_fence_after();
          if (!bounds_ok(buf * (uint32_t)T + (uint32_t)(half * kHalf + kHalf) <= kTmemCols, p.status, kChkTmemCol,
                         (uint64_t)(buf * T + half * kHalf))) {
            ok = false;
            break;
          }
          const uint32_t taddr = tmem_base + t_lane + buf * (uint32_t)T + (uint32_t)(half * kHalf);
          // four columns per load: with the 64-float sum live, wider loads
          // push the epilogue past its register budget (and into local memory)
#pragma unroll
          for (int c = 0; c < kHalf; c += 4) {
            float v[4];
            tmem_ld4(taddr + (uint32_t)c, v);
#pragma unroll
            for (int i = 0; i < 4; ++i) R[c + i] = __fadd_rn(R[c + i], v[i]);
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            const uint32_t ae = smem_u32(&ctl->acc_empty[buf]);
            if constexpr (PAIR)
              mbar_arrive_remote(mapa_shared(ae, leader_rank));
            else
              mbar_arrive(ae);
          }
          ++acc_iter;
        }
        if (!ok) break;
        const int64_t n = (int64_t)n_tile * kMmaM + (int64_t)peer * kTileN + n_local;
        if (n < p.N) {
          const int64_t m0 = (int64_t)m_tile * T + half * kHalf;
          __nv_bfloat16* y = p.Y + m0 * p.N + n;
          const int64_t mrem = p.M - m0;
          const int mv = mrem < kHalf ? (int)mrem : kHalf;
          const float swn = FP8 ? p.sw[n] : 1.0f;
#pragma unroll
          for (int j = 0; j < kHalf; ++j) {
            if (j < mv) *y = __float2bfloat16_rn(FP8 ? __fmul_rn(__fmul_rn(R[j], p.sx[m0 + j]), swn) : R[j]);
            y += p.N;
          }
        }
      }
    } else {
      // This unit's chains, one per TMEM buffer.  Unchained (one split per
      // unit) and unit 0 of a chain move their partial -- unit 0 the sum of
      // its splits, in order -- into shared memory as [token][n].  Later units
      // of a chain keep theirs in TMEM until the running sum reaches them.
      const int nch = s_end - s_first;
      bool got = true;
      for (int b = 0; b < nch; ++b) got = got && wait_or_abort(smem_u32(&ctl->acc_full[b]), 0, abort, p.status);
      got = __all_sync(0xffffffffu, got);
      chain_ok = got;
      if (got && (!chained || my_unit == 0)) {
        tc_fence_after();
        const int64_t m0 = (int64_t)blockIdx.z * T;
        const int64_t rem = p.M - m0;
        const int mv = rem < T ? (int)rem : T;              // valid tokens in this tile
        int c_end = min(half * kHalf + kHalf, (mv + 7) & ~7);
        // debug-bounds build: the partial's rows within the [T][128] tile, the
        // chains' columns within the allocation
        if (!bounds_ok(c_end <= T && (uint32_t)(nch * T) <= kTmemCols, p.status, kChkClusterPart, (uint64_t)c_end))
          c_end = 0;
        float* P = reinterpret_cast<float*>(smem);
        for (int c = half * kHalf; c < c_end; c += 8) {
          float v[8];
          tmem_ld8(tmem_base + t_lane + (uint32_t)c, v);
          if (nch == 2) {
            float w[8];
            tmem_ld8(tmem_base + t_lane + (uint32_t)T + (uint32_t)c, w);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = __fadd_rn(v[i], w[i]);
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) P[(c + i) * kTileN + n_local] = v[i];
        }
        tc_fence_before();
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  __syncthreads();
  if (chained) {
    // The running sum moves down the chain of units: at step u, unit u adds
    // its splits, in ascending order, to the sum unit u - 1 left in its shared
    // memory, and leaves the result in its own (the last unit writes Y).
    // Every thread of the cluster takes part in every barrier.
    for (int32_t u = 1; u < U; ++u) {
      cluster_sync();
      if (my_unit == u && warp >= kFirstEpiWarp && chain_ok) {
        const int ew = warp - kFirstEpiWarp;
        const int quad = warp & 3;
        const int half = ew >> 2;
        const int n_local = quad * 32 + lane;
        const uint32_t t_lane = (uint32_t)(quad * 32) << 16;
        const int nch = s_end - s_first;
        const int64_t m0 = (int64_t)blockIdx.z * T;
        const int64_t rem = p.M - m0;
        const int mv = rem < T ? (int)rem : T;
        const int c_end = min(half * kHalf + kHalf, (mv + 7) & ~7);
        const uint32_t prev = (uint32_t)(u - 1) * (PAIR ? 2u : 1u) + peer;  // same W rows, unit u - 1
        const bool last = u == U - 1;
        const int64_t n = (int64_t)blockIdx.y * kMmaM + (int64_t)peer * kTileN + n_local;
        float* P = reinterpret_cast<float*>(smem);
        tc_fence_after();
        for (int c = half * kHalf; c < c_end; c += 8) {
          float v[8], a[8];
          tmem_ld8(tmem_base + t_lane + (uint32_t)c, a);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const uint32_t off = smem_base + (uint32_t)(((c + i) * kTileN + n_local) * 4);
            v[i] = __fadd_rn(ld_dsmem_f32(mapa_shared(off, prev)), a[i]);
          }
          if (nch == 2) {
            tmem_ld8(tmem_base + t_lane + (uint32_t)T + (uint32_t)c, a);
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = __fadd_rn(v[i], a[i]);
          }
          if (last) {
            if (n < p.N) {
              __nv_bfloat16* y = p.Y + (m0 + c) * p.N + n;
              const float swn = FP8 ? p.sw[n] : 1.0f;
#pragma unroll
              for (int i = 0; i < 8; ++i)
                if (c + i < mv)
                  y[(int64_t)i * p.N] = __float2bfloat16_rn(
                      FP8 ? __fmul_rn(__fmul_rn(v[i], p.sx[m0 + c + i]), swn) : v[i]);
            }
          } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) P[(c + i) * kTileN + n_local] = v[i];
          }
        }
        tc_fence_before();
      }
    }
    cluster_sync();  // no CTA leaves, or frees its tensor memory, while another reads it
  }
  // In a pair, the even CTA's MMAs write both CTAs' TMEM: nobody frees TMEM
  // (or exits) until that CTA has drained them.
  if constexpr (PAIR) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR)
      tmem_dealloc_pair(tmem_base, kTmemCols);
    else
      tmem_dealloc(tmem_base, kTmemCols);
  }
  if (CLUSTER && !chained) {
    // Fold the S partials of the tile in ascending split order.  The CTA of
    // split r folds tokens r, r + S, r + 2S, ... of its own 128 W rows; element
    // pairs are spread over all threads.
    cluster_sync();
    const int32_t rank = my_unit;
    const int64_t m0 = (int64_t)blockIdx.z * T;
    const int64_t n0 = (int64_t)blockIdx.y * kMmaM + (int64_t)peer * kTileN;
    const int64_t remm = p.M - m0;
    const int mv = remm < T ? (int)remm : T;
    const int64_t remn = p.N - n0;
    const int nv = remn <= 0 ? 0 : (remn < kTileN ? (int)remn : kTileN);
    const int rows_mine = rank < mv ? (mv - rank + S - 1) / S : 0;
    const int items = rows_mine * (kTileN / 2);
    const bool even_n = (p.N & 1) == 0;
    for (int it = threadIdx.x; it < items; it += blockDim.x) {
      const int j = rank + S * (it / (kTileN / 2));
      const int n = 2 * (it % (kTileN / 2));
      if (n >= nv) continue;
      const uint32_t off = smem_base + (uint32_t)((j * kTileN + n) * 4);
      // split c's partial of these W rows sits in cluster CTA c (or 2c + peer)
      float2 r = ld_dsmem_f32x2(mapa_shared(off, PAIR ? peer : 0u));
      for (int c = 1; c < S; ++c) {
        const uint32_t src = PAIR ? (uint32_t)(2 * c) + peer : (uint32_t)c;
        const float2 v = ld_dsmem_f32x2(mapa_shared(off, src));
        r.x = __fadd_rn(r.x, v.x);
        r.y = __fadd_rn(r.y, v.y);
      }
      __nv_bfloat16* y = p.Y + (m0 + j) * p.N + n0 + n;
      if constexpr (FP8) {
        const float sxm = p.sx[m0 + j];
        r.x = __fmul_rn(__fmul_rn(r.x, sxm), p.sw[n0 + n]);
        if (n + 1 < nv) r.y = __fmul_rn(__fmul_rn(r.y, sxm), p.sw[n0 + n + 1]);
      }
      if (even_n && n + 1 < nv) {
        *reinterpret_cast<__nv_bfloat162*>(y) = __floats2bfloat162_rn(r.x, r.y);
      } else {
        y[0] = __float2bfloat16_rn(r.x);
        if (n + 1 < nv) y[1] = __float2bfloat16_rn(r.y);
      }
    }
    cluster_sync();  // no CTA leaves while others may still read its partial
  }
}

// ---------------------------------------------------------------------------
// launch templates (host)
// ---------------------------------------------------------------------------

template <bool FUSED, int T, bool CLUSTER, bool PAIR, int KP, bool FP8 = false>
static cudaError_t launch_t(const GemmLaunch& L) {
  auto kern = bi_gemm_kernel<T, CLUSTER, PAIR, KP, FP8, FUSED>;
  // Kernel attributes are per device: raise this instance's shared-memory
  // limit to the largest ring (and allow clusters above 8) once per device,
  // not on every launch.
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t)1 << dev : 0;
  if (!bit || !(configured.load() & bit)) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxDynSmem);
    if (e != cudaSuccess) return e;
    if (CLUSTER) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
    configured.fetch_or(bit);
  }
  if (L.smem > kMaxDynSmem) return cudaErrorInvalidValue;
  const int cluster = CLUSTER ? L.units * (PAIR ? 2 : 1) : (PAIR ? 2 : 1);
  GemmParams prm;
  prm.Y = static_cast<__nv_bfloat16*>(L.Y);
  prm.M = L.M;
  prm.N = L.N;
  prm.n_tiles = L.n_tiles;
  prm.m_tiles = L.m_tiles;
  prm.k_tiles = L.k_tiles;
  prm.S = L.S;
  prm.w_stages = L.w_stages;
  prm.x_stages = L.x_stages;
  prm.x_box_rows = L.x_box_rows;
  prm.group_n = L.group_n;
  prm.units = L.units;
  prm.sx = L.sx;
  prm.sw = L.sw;
  prm.g = static_cast<const __nv_bfloat16*>(L.g);
  prm.rrow = L.rrow;
  prm.xraw = static_cast<const __nv_bfloat16*>(L.X);
  prm.eps = L.eps;
  prm.fold_part = L.fold_part;
  prm.fold_count = L.fold_count;
  prm.status = L.status;
  prm.K = L.K;
  prm.flags = L.flags;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)L.grid_x, (unsigned)L.grid_y, (unsigned)L.grid_z);
  cfg.blockDim = dim3((unsigned)gemm_threads(FUSED), 1, 1);
  cfg.dynamicSmemBytes = (size_t)L.smem;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = (unsigned)cluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, L.tmW, L.tmX, prm);
}

// E4M3 operands: T = 256, or a decode tile of 64 or 128.
template <bool PAIR>
static cudaError_t launch_fp8(const GemmLaunch& L) {
  {
    if (L.T == 64 || L.T == 128) {
      if constexpr (PAIR) {
        return cudaErrorInvalidValue;
      } else {
        if (L.kps != 2 || !(L.flags & kFlagCopy2D)) return cudaErrorInvalidValue;
        if (L.T == 64)
          return L.cluster ? launch_t<false, 64, true, false, 2, true>(L) : launch_t<false, 64, false, false, 2, true>(L);
        return L.cluster ? launch_t<false, 128, true, false, 2, true>(L) : launch_t<false, 128, false, false, 2, true>(L);
      }
    }
    if (L.T != 256) return cudaErrorInvalidValue;
    if (L.kps == 2)
      return L.cluster ? launch_t<false, 256, true, PAIR, 2, true>(L) : launch_t<false, 256, false, PAIR, 2, true>(L);
    return L.cluster ? launch_t<false, 256, true, PAIR, 1, true>(L) : launch_t<false, 256, false, PAIR, 1, true>(L);
  }
}

template <bool FUSED, bool PAIR>
static cudaError_t launch_p(const GemmLaunch& L) {
  if (FUSED && L.fp8) return cudaErrorInvalidValue;  // the fused prologue is bf16 only
  if constexpr (!FUSED) {
    if (L.fp8) return launch_fp8<PAIR>(L);
  }
  switch (L.T) {
    case 64:
    case 128:
      if (L.kps == 2) {
        // decode tiles: two K tiles per stage by 2-D copies, single-CTA MMAs
        if constexpr (PAIR) {
          return cudaErrorInvalidValue;
        } else {
          if (!(L.flags & kFlagCopy2D)) return cudaErrorInvalidValue;
          if (L.T == 64) return L.cluster ? launch_t<FUSED, 64, true, false, 2>(L) : launch_t<FUSED, 64, false, false, 2>(L);
          return L.cluster ? launch_t<FUSED, 128, true, false, 2>(L) : launch_t<FUSED, 128, false, false, 2>(L);
        }
      }
      if (L.kps != 1) return cudaErrorInvalidValue;
      if (L.T == 64) return L.cluster ? launch_t<FUSED, 64, true, PAIR, 1>(L) : launch_t<FUSED, 64, false, PAIR, 1>(L);
      return L.cluster ? launch_t<FUSED, 128, true, PAIR, 1>(L) : launch_t<FUSED, 128, false, PAIR, 1>(L);
    case 256:
      if (L.kps == 2)
        return L.cluster ? launch_t<FUSED, 256, true, PAIR, 2>(L) : launch_t<FUSED, 256, false, PAIR, 2>(L);
      return L.cluster ? launch_t<FUSED, 256, true, PAIR, 1>(L) : launch_t<FUSED, 256, false, PAIR, 1>(L);
    default:
      break;
  }
  // Narrower token tiles, chosen per launch to fill the last wave of a
  // persistent paired launch (the MMA's N extent never changes a bit):
  // LOCAL, CTA pairs, two K tiles per copy only.
  if constexpr (PAIR) {
    if (L.cluster || L.kps != 2) return cudaErrorInvalidValue;
    switch (L.T) {
      case 224: return launch_t<FUSED, 224, false, true, 2>(L);
      case 192: return launch_t<FUSED, 192, false, true, 2>(L);
      case 160: return launch_t<FUSED, 160, false, true, 2>(L);
      default: return cudaErrorInvalidValue;
    }
  } else {
    return cudaErrorInvalidValue;
  }
}

}  // namespace bi
