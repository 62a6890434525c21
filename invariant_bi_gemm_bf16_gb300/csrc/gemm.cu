// gemm.cu -- the batch-invariant bf16 GEMM on the 5th-generation tensor cores.
//
// Y[M,N] = X[M,K] . W[N,K]^T with fp32 accumulation in tensor memory (TMEM).
//
// The reduction tree of every output element y[m,n] is fixed by (N, K, pins):
//   * K is cut into K tiles of 64 elements; split s (0 <= s < S) owns K tiles
//     [floor(s*KT/S), floor((s+1)*KT/S)).
//   * Inside a split, the partial acc_s is one chain of tcgen05.mma
//     instructions of shape 128 x T x 16 in ascending k, the first of which
//     overwrites the accumulator.  W rows sit on the MMA's M side (TMEM lanes),
//     tokens on its N side (TMEM columns); T is a pin.
//   * The partials are added in ascending s in fp32: (((acc_0 + acc_1) + acc_2) ...).
// CoRun (Padding is Simple and Efficient for Deterministic LLM Inference),
// Sec. III-A, Fig. 3(b): a batch-invariant reduction uses one fixed partition
// and one fixed combine order at every batch size.  Detent, Sec. 7, keeps
// split-KV in attention with split boundaries set by a fixed split size; here
// the split count and boundaries are pins in the same spirit.
//
// What may depend on M (and changes no bit): the number of token tiles, the
// grid, which SM runs which tile, and whether the S chains of a tile run on one
// CTA (LOCAL) or on a cluster of S CTAs (CLUSTER):
//   LOCAL   a persistent CTA walks its tiles; for each tile it runs the S
//           chains one after the other into two ping-pong TMEM accumulators;
//           the epilogue warps fold them into registers as they complete.
//   CLUSTER each CTA of an S-CTA cluster runs one chain; the partials go to
//           shared memory and are folded in ascending rank order through
//           distributed shared memory.  No atomics and no global workspace.
//
// Warp roles (320 threads): warp 0 = TMA producer (one lane), warp 1 = MMA
// issuer (one lane) and TMEM owner, warps 2..9 = epilogue (two warps per TMEM
// lane quadrant, each owning half of the T accumulator columns).
//
// Every wait is bounded (2 s of wall clock).  When one runs out, the kernel
// records BI_ERR_DEVICE_TIMEOUT in a device status word, every role abandons
// its work, in-flight copies and MMAs are drained (again with bounded waits),
// tensor memory is freed and the CTA returns normally.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace bi {

__device__ int g_stall_status;  // 0, or a bi_status code set by a kernel that gave up

constexpr uint64_t kWaitLimitNs = 2000000000ull;

struct GemmParams {
  __nv_bfloat16* Y;
  int64_t M, N;
  int32_t n_tiles, m_tiles, k_tiles, S, stages;
  uint32_t flags;
};

struct __align__(8) SmemCtl {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(SmemCtl) <= kCtlBytes, "control block too large");

__device__ __forceinline__ void record_stall() {
  atomicCAS(&g_stall_status, 0, (int)BI_ERR_DEVICE_TIMEOUT);
}

// Slow path of wait_or_abort: polls until the phase completes, the CTA starts
// abandoning the call, or kWaitLimitNs pass (then it starts the abandonment).
__device__ __noinline__ bool wait_or_abort_slow(uint32_t bar, uint32_t parity, volatile int* abort) {
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *abort = 1;
      record_stall();
      return false;
    }
  }
}

// Waits for the phase of `parity` on `bar`; false if the call is abandoned.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  return wait_or_abort_slow(bar, parity, abort);
}

// Bounded wait that ignores the abort flag (for draining work in flight).
__device__ __noinline__ bool wait_drain(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      record_stall();
      return false;
    }
  }
}

__device__ __forceinline__ int64_t split_begin(int32_t s, int32_t S, int32_t KT) {
  return ((int64_t)s * KT) / S;
}

template <int T, bool CLUSTER>
__global__ void __launch_bounds__(kGemmThreads, 1)
    bi_gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const GemmParams p) {
  constexpr int kStage = stage_bytes(T);
  constexpr int kWBytes = kTileN * kBK * 2;
  constexpr uint32_t kTmemCols = CLUSTER ? (uint32_t)T : 2u * (uint32_t)T;
  constexpr int kHalf = T / 2;  // accumulator columns per epilogue warp

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int stages = p.stages;
  const int64_t ring_bytes = (int64_t)stages * kStage;
  const int64_t part_bytes = CLUSTER ? (int64_t)T * kTileN * 4 : 0;
  SmemCtl* ctl = reinterpret_cast<SmemCtl*>(smem + (ring_bytes > part_bytes ? ring_bytes : part_bytes));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t smem_base = smem_u32(smem);

  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      mbar_init(smem_u32(&ctl->full[s]), 1);
      mbar_init(smem_u32(&ctl->empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&ctl->acc_full[b]), 1);
      mbar_init(smem_u32(&ctl->acc_empty[b]), kEpiWarps);
    }
    mbar_init(smem_u32(&ctl->mma_done), 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmW);
    prefetch_tensormap(&tmX);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&ctl->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = ctl->tmem_base;
  volatile int* abort = &ctl->abort;

  const int32_t S = p.S;
  const int32_t KT = p.k_tiles;
  const int64_t num_tiles = (int64_t)p.n_tiles * p.m_tiles;
  // Work list.  CLUSTER: one tile (blockIdx.y, blockIdx.z), one split (the
  // cluster rank).  LOCAL: tiles blockIdx.x, blockIdx.x + gridDim.x, ... and
  // all S splits of each.
  const int32_t my_split = CLUSTER ? (int32_t)cluster_ctarank() : 0;
  const int64_t tile_first = CLUSTER ? 0 : blockIdx.x;
  const int64_t tile_step = CLUSTER ? 1 : gridDim.x;
  const int64_t tile_end = CLUSTER ? 1 : num_tiles;
  const int32_t s_first = CLUSTER ? my_split : 0;
  const int32_t s_end = CLUSTER ? my_split + 1 : S;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const bool stall = (p.flags & BI_FLAG_DEBUG_STALL_PRODUCER) != 0;
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      for (int64_t t = tile_first; ok && t < tile_end; t += tile_step) {
        const int32_t n_tile = CLUSTER ? (int32_t)blockIdx.y : (int32_t)(t % p.n_tiles);
        const int32_t m_tile = CLUSTER ? (int32_t)blockIdx.z : (int32_t)(t / p.n_tiles);
        for (int32_t s = s_first; ok && s < s_end; ++s) {
          const int64_t k0 = split_begin(s, S, KT), k1 = split_begin(s + 1, S, KT);
          for (int64_t kt = k0; kt < k1; ++kt) {
            const uint32_t empty = smem_u32(&ctl->empty[stage]);
            if (!wait_or_abort(empty, phase ^ 1u, abort)) {
              ok = false;
              break;
            }
            if (!(stall && issued == 0)) {
              const uint32_t full = smem_u32(&ctl->full[stage]);
              const uint32_t sw = smem_base + stage * kStage;
              mbar_arrive_expect_tx(full, (uint32_t)kStage);
              tma_load_2d(sw, &tmW, full, (int32_t)(kt * kBK), n_tile * kTileN);
              tma_load_2d(sw + kWBytes, &tmX, full, (int32_t)(kt * kBK), m_tile * T);
            }
            ++issued;
            if (++stage == stages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
      }
      // Drain: the copies of the last `stages` loads must have landed before
      // the CTA may exit (they write into this CTA's shared memory).
      const int64_t first = issued > stages ? issued - stages : 0;
      for (int64_t i = first; i < issued; ++i) {
        if (stall && i == 0) continue;
        wait_drain(smem_u32(&ctl->full[i % stages]), (uint32_t)((i / stages) & 1));
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc_bf16(kTileN, T);
      int stage = 0;
      uint32_t phase = 0;
      uint32_t acc_iter = 0;
      bool ok = true;
      for (int64_t t = tile_first; ok && t < tile_end; t += tile_step) {
        for (int32_t s = s_first; ok && s < s_end; ++s) {
          const uint32_t buf = CLUSTER ? 0u : (acc_iter & 1u);
          const uint32_t acc_phase = CLUSTER ? 0u : ((acc_iter >> 1) & 1u);
          if (!wait_or_abort(smem_u32(&ctl->acc_empty[buf]), acc_phase ^ 1u, abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + buf * (uint32_t)T;
          const int64_t k0 = split_begin(s, S, KT), k1 = split_begin(s + 1, S, KT);
          for (int64_t kt = k0; kt < k1; ++kt) {
            if (!wait_or_abort(smem_u32(&ctl->full[stage]), phase, abort)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sw = smem_base + stage * kStage;
            const uint64_t a_desc = make_sdesc_sw128(sw);
            const uint64_t b_desc = make_sdesc_sw128(sw + kWBytes);
#pragma unroll
            for (int j = 0; j < kBK / kMmaK; ++j) {
              // +32 bytes per 16 K elements, in the descriptor's 16-byte units
              mma_bf16(d_tmem, a_desc + 2 * j, b_desc + 2 * j, idesc,
                       (kt > k0 || j > 0) ? 1u : 0u);
            }
            mma_commit(smem_u32(&ctl->empty[stage]));
            if (++stage == stages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          mma_commit(smem_u32(&ctl->acc_full[buf]));
          ++acc_iter;
        }
      }
      // Every MMA this thread issued must be complete before TMEM is freed.
      mma_commit(smem_u32(&ctl->mma_done));
      wait_drain(smem_u32(&ctl->mma_done), 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - 2;
    const int quad = warp & 3;            // TMEM lanes [32*quad, 32*quad + 32)
    const int half = ew >> 2;             // accumulator columns [half*T/2, half*T/2 + T/2)
    const int n_local = quad * 32 + lane; // W row within the tile
    const uint32_t t_lane = (uint32_t)(quad * 32) << 16;
    uint32_t acc_iter = 0;
    bool ok = true;
    if constexpr (!CLUSTER) {
      for (int64_t t = tile_first; ok && t < tile_end; t += tile_step) {
        const int32_t n_tile = (int32_t)(t % p.n_tiles);
        const int32_t m_tile = (int32_t)(t / p.n_tiles);
        float R[kHalf];
        for (int32_t s = 0; s < S; ++s) {
          const uint32_t buf = acc_iter & 1u;
          const uint32_t acc_phase = (acc_iter >> 1) & 1u;
          bool got = wait_or_abort(smem_u32(&ctl->acc_full[buf]), acc_phase, abort);
          got = __all_sync(0xffffffffu, got);
          if (!got) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t taddr = tmem_base + t_lane + buf * (uint32_t)T + (uint32_t)(half * kHalf);
#pragma unroll
          for (int c = 0; c < kHalf; c += 32) {
            float v[32];
            tmem_ld32(taddr + (uint32_t)c, v);
            if (s == 0) {
#pragma unroll
              for (int i = 0; i < 32; ++i) R[c + i] = v[i];
            } else {
#pragma unroll
              for (int i = 0; i < 32; ++i) R[c + i] = __fadd_rn(R[c + i], v[i]);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&ctl->acc_empty[buf]));
          ++acc_iter;
        }
        if (!ok) break;
        const int64_t n = (int64_t)n_tile * kTileN + n_local;
        if (n < p.N) {
          const int64_t m0 = (int64_t)m_tile * T + half * kHalf;
          __nv_bfloat16* y = p.Y + m0 * p.N + n;
          const int64_t mrem = p.M - m0;
#pragma unroll
          for (int c = 0; c < kHalf; c += 32) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              if (c + i < mrem) y[(int64_t)(c + i) * p.N] = __float2bfloat16_rn(R[c + i]);
            }
          }
        }
      }
    } else {
      // One chain: move this CTA's partial into shared memory as [token][n].
      bool got = wait_or_abort(smem_u32(&ctl->acc_full[0]), 0, abort);
      got = __all_sync(0xffffffffu, got);
      if (got) {
        tc_fence_after();
        const int64_t m0 = (int64_t)blockIdx.z * T;
        const int64_t rem = p.M - m0;
        const int mv = rem < T ? (int)rem : T;              // valid tokens in this tile
        const int c_end = min(half * kHalf + kHalf, (mv + 7) & ~7);
        float* P = reinterpret_cast<float*>(smem);
        for (int c = half * kHalf; c < c_end; c += 8) {
          float v[8];
          tmem_ld8(tmem_base + t_lane + (uint32_t)c, v);
#pragma unroll
          for (int i = 0; i < 8; ++i) P[(c + i) * kTileN + n_local] = v[i];
        }
        tc_fence_before();
      }
    }
  }

  // ---------------------------------------------------------------- teardown
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
  if constexpr (CLUSTER) {
    // Fold the S partials of the tile in ascending rank order.  CTA r folds
    // tokens r, r + S, r + 2S, ...; element pairs are spread over all threads.
    cluster_sync();
    const int32_t rank = my_split;
    const int64_t m0 = (int64_t)blockIdx.z * T;
    const int64_t n0 = (int64_t)blockIdx.y * kTileN;
    const int64_t remm = p.M - m0;
    const int mv = remm < T ? (int)remm : T;
    const int64_t remn = p.N - n0;
    const int nv = remn < kTileN ? (int)remn : kTileN;
    const int rows_mine = rank < mv ? (mv - rank + S - 1) / S : 0;
    const int items = rows_mine * (kTileN / 2);
    const bool even_n = (p.N & 1) == 0;
    for (int it = threadIdx.x; it < items; it += blockDim.x) {
      const int j = rank + S * (it / (kTileN / 2));
      const int n = 2 * (it % (kTileN / 2));
      if (n >= nv) continue;
      const uint32_t off = smem_base + (uint32_t)((j * kTileN + n) * 4);
      float2 r = ld_dsmem_f32x2(mapa_shared(off, 0));
      for (int c = 1; c < S; ++c) {
        const float2 v = ld_dsmem_f32x2(mapa_shared(off, (uint32_t)c));
        r.x = __fadd_rn(r.x, v.x);
        r.y = __fadd_rn(r.y, v.y);
      }
      __nv_bfloat16* y = p.Y + (m0 + j) * p.N + n0 + n;
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
// host side
// ---------------------------------------------------------------------------

int max_stages(int T) {
  const int avail = kMaxDynSmem - 1024 - kCtlBytes;
  int s = avail / stage_bytes(T);
  return s > kMaxStages ? kMaxStages : s;
}

int default_stages(int T) {
  const int m = max_stages(T);
  return m > 6 ? 6 : m;
}

int64_t gemm_smem_bytes(int T, int stages, bool cluster) {
  int64_t ring = (int64_t)stages * stage_bytes(T);
  int64_t part = cluster ? (int64_t)T * kTileN * 4 : 0;
  return 1024 + (ring > part ? ring : part) + kCtlBytes;
}

template <int T, bool CLUSTER>
static cudaError_t launch_t(const GemmLaunch& L) {
  auto kern = bi_gemm_kernel<T, CLUSTER>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L.smem);
  if (e != cudaSuccess) return e;
  if (CLUSTER && L.S > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  GemmParams prm;
  prm.Y = static_cast<__nv_bfloat16*>(L.Y);
  prm.M = L.M;
  prm.N = L.N;
  prm.n_tiles = L.n_tiles;
  prm.m_tiles = L.m_tiles;
  prm.k_tiles = L.k_tiles;
  prm.S = L.S;
  prm.stages = L.stages;
  prm.flags = L.flags;

  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)L.grid_x, (unsigned)L.grid_y, (unsigned)L.grid_z);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)L.smem;
  cfg.stream = L.stream;
  cudaLaunchAttribute attr[1];
  cfg.numAttrs = 0;
  if (CLUSTER) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)L.S;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kern, L.tmW, L.tmX, prm);
}

cudaError_t launch_gemm(const GemmLaunch& L) {
  switch (L.T) {
    case 64:
      return L.cluster ? launch_t<64, true>(L) : launch_t<64, false>(L);
    case 128:
      return L.cluster ? launch_t<128, true>(L) : launch_t<128, false>(L);
    case 256:
      return L.cluster ? launch_t<256, true>(L) : launch_t<256, false>(L);
    default:
      return cudaErrorInvalidValue;
  }
}

cudaError_t fetch_and_clear_stall(int* host_dst, cudaStream_t stream) {
  cudaError_t e = cudaMemcpyFromSymbolAsync(host_dst, g_stall_status, sizeof(int), 0,
                                            cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  const int zero = 0;
  e = cudaMemcpyToSymbolAsync(g_stall_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(stream);
}

}  // namespace bi
