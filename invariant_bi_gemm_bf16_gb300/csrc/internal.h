// internal.h -- declarations shared by the host entry points (api.cu) and the
// kernel files.  Not part of the public ABI.
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_runtime.h>

#include "bi_gemm.h"

namespace bi {

constexpr int kTileN = BI_TILE_N;  // W rows per tile: the MMA's M extent
constexpr int kBK = BI_BK;         // K elements per K tile (one 128-byte swizzle row)
constexpr int kMmaK = 16;          // K per tcgen05.mma.kind::f16 instruction
constexpr int kEpiWarps = 8;       // epilogue warps (two per TMEM lane quadrant)
constexpr int kGemmThreads = 64 + 32 * kEpiWarps;  // producer warp, MMA warp, epilogue
constexpr int kMaxStages = 16;
constexpr int kMaxDynSmem = 232448;  // 227 KB opt-in per block on sm_100-class parts

// Shared-memory bytes of one ring stage: a W tile [128 x 64] and an X tile [T x 64].
constexpr int stage_bytes(int T) { return (kTileN + T) * kBK * 2; }
// Bytes after the ring for mbarriers and bookkeeping.
constexpr int kCtlBytes = 512;
int max_stages(int T);
int default_stages(int T);
// Dynamic shared memory of one GEMM CTA (includes 1 KB of alignment slack).
int64_t gemm_smem_bytes(int T, int stages, bool cluster);

struct GemmLaunch {
  CUtensorMap tmW;   // W [N,K], box 64 x 128, 128-byte swizzle
  CUtensorMap tmX;   // X [M,K], box 64 x T, 128-byte swizzle, zero fill past M / K
  void* Y;
  int64_t M, N, K;
  int32_t n_tiles, m_tiles, k_tiles, S, T, stages;
  bool cluster;
  int32_t grid_x, grid_y, grid_z;
  int64_t smem;
  uint32_t flags;
  cudaStream_t stream;
};

cudaError_t launch_gemm(const GemmLaunch& L);
cudaError_t launch_rmsnorm(const void* X, const void* g, void* Y, int64_t M, int64_t H, float eps,
                           cudaStream_t stream);
cudaError_t launch_residual_add(const void* a, const void* b, void* out, int64_t count,
                                cudaStream_t stream);
cudaError_t launch_silu_mul(const void* gu, void* out, int64_t M, int64_t I, cudaStream_t stream);
cudaError_t launch_attention_ctx1(const void* qkv, void* out, int64_t M, int64_t nq, int64_t nkv,
                                  int64_t D, cudaStream_t stream);
// Reads and clears the current device's stall word (asynchronously on
// `stream`; the caller synchronises).
cudaError_t fetch_and_clear_stall(int* host_dst, cudaStream_t stream);

}  // namespace bi
