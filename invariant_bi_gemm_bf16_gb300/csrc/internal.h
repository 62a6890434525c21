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
constexpr int kEpiWarps = 16;      // epilogue warps (four per TMEM lane quadrant)
constexpr int kFirstEpiWarp = 3;   // warps 0..2: W producer, MMA issuer, X producer
constexpr int kGemmThreads = 32 * (kFirstEpiWarp + kEpiWarps);
constexpr int kXformWarps = 4;     // fused RMSNorm prologue: warps that normalise X stages
constexpr int kFirstXformWarp = kFirstEpiWarp + kEpiWarps;
constexpr int gemm_threads(bool fused) { return kGemmThreads + (fused ? 32 * kXformWarps : 0); }
// Fused layer, in shared memory: up to this many rows, the GEMM computes the
// rows' RMSNorm scales itself instead of a separate row-scale kernel.
constexpr int kRowScaleInKernelMax = 4;
constexpr int kMaxStages = 16;
constexpr int kMaxDynSmem = 232448;  // 227 KB opt-in per block on sm_100-class parts

// Internal GEMM flags (above the public BI_FLAG_* bits).
constexpr uint32_t kFlagStreamW = 1u << 16;  // W read once: evict-first, X evict-last in L2
constexpr uint32_t kFlagZeroX = 1u << 17;    // X boxes hold fewer rows than T: zero the ring once
constexpr uint32_t kFlagCopy2D = 1u << 18;   // KP = 2 by two 2-D copies per stage (single-CTA MMAs only)
// Debug-bounds build only: the first W copy of each CTA is aimed past the
// tile grid, for the negative test of the index checks (set from the
// BI_DEBUG_POKE=wrow environment variable; never in the ordinary build).
constexpr uint32_t kFlagDebugPokeWRow = 1u << 19;

// Shared-memory bytes of one W stage [128 x 64] and one X stage [rows x 64]
// (rows = T, or T/2 per CTA of a pair).
constexpr int kWStageBytes = kTileN * kBK * 2;
constexpr int x_stage_bytes(int x_rows) { return x_rows * kBK * 2; }
// Bytes after the rings for mbarriers and bookkeeping.
constexpr int kCtlBytes = 1024;
// Bytes available to the two rings (the rest is alignment slack and control).
constexpr int kRingBytes = kMaxDynSmem - 1024 - kCtlBytes;
// Deepest W ring that still leaves `x_stages` X stages of `x_rows` rows, with
// stages of `kps` K tiles.
int max_w_stages(int x_rows, int x_stages, int kps);
// Ring depths for a launch: deep W and shallow X when the X box is small
// (decode), balanced otherwise.  `w_pin` (the pins' stages field) overrides the
// W depth when non-zero.  Speed only.
void choose_stages(int x_rows, int x_box_rows, int w_pin, int kps, int* w_stages, int* x_stages);
// Dynamic shared memory of one GEMM CTA (includes 1 KB of alignment slack).
int64_t gemm_smem_bytes(int T, int x_rows, int w_stages, int x_stages, int kps, bool cluster);

struct GemmLaunch {
  CUtensorMap tmW;   // W [N,K], box 64 x 128 (x kps), 128-byte swizzle
  CUtensorMap tmX;   // X [M,K], box 64 x x_box_rows (x kps), 128-byte swizzle, zero fill past M / K
  void* Y;
  int64_t M, N, K;
  int32_t n_tiles, m_tiles, k_tiles, S, T, w_stages, x_stages, x_box_rows;
  int32_t kps;       // K tiles per copy: 1 (2-D maps) or 2 (3-D maps, T = 256 only)
  int32_t group_n;   // LOCAL tile order: W tiles per group (1 .. n_tiles)
  int32_t units;     // CLUSTER: units (CTAs or pairs) per tile: S, or ceil(S/2) when chained
  bool fp8;          // E4M3 operands (kind::f8f6f4), K tiles of 128 values; Y scaled by sx, sw
  const float* sx;   // fp8: per-token scales [M]
  const float* sw;   // fp8: per-channel scales [N]
  const void* X;     // operands, for the tensor maps
  const void* W;
  const void* g;     // fused: RMSNorm gain [K] (bf16)
  float eps;         // fused: RMSNorm epsilon
  const float* rrow; // fused: per-row r = 1 / sqrt(mean(x^2) + eps) [M], or nullptr (computed in the GEMM)
  int* status;       // device status word (bounded waits report there)
  float* fold_part;        // GLOBAL schedule: chain partials in the fold workspace (else nullptr)
  uint32_t* fold_count;    // GLOBAL schedule: per-tile arrival counters
  bool cluster;      // one chain per CTA (pair), folded through DSMEM
  bool pair;         // cta_group::2 MMA across a CTA pair
  int32_t grid_x, grid_y, grid_z;
  int64_t smem;
  uint32_t flags;
  cudaStream_t stream;
};

// Launches `kern` with programmatic stream serialization allowed (the kernel
// must call griddepcontrol.wait before touching memory).
template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kern)(KArgs...), dim3 grid, dim3 block, cudaStream_t stream,
                              Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped_smem(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                   cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}


// Device address of the status word that bi_last_device_status() reads
// (looked up once per device).
int* device_status_word();

cudaError_t launch_gemm(const GemmLaunch& L);
// The GEMM with the RMSNorm prologue applied to X in shared memory (L.g and
// L.rrow set; bf16 only).
cudaError_t launch_gemm_fused(const GemmLaunch& L);
// r[m] = 1 / sqrt(mean_h(x[m,h]^2) + eps) of each row of X [M,H], by the
// lane partition and butterfly of the RMSNorm kernels (the same bits).
cudaError_t launch_row_scale(const void* X, float* r, int64_t M, int64_t H, float eps, cudaStream_t stream);
cudaError_t launch_rmsnorm(const void* X, const void* g, void* Y, int64_t M, int64_t H, float eps,
                           cudaStream_t stream);
cudaError_t launch_residual_add(const void* a, const void* b, void* out, int64_t count,
                                cudaStream_t stream);
cudaError_t launch_silu_mul(const void* gu, void* out, int64_t M, int64_t I, cudaStream_t stream);
cudaError_t launch_quantize_e4m3(const void* X, void* Q, float* scale, int64_t M, int64_t K,
                                 cudaStream_t stream);
cudaError_t launch_log_softmax(const void* X, void* Y, int64_t M, int64_t V, cudaStream_t stream);
cudaError_t launch_token_logprobs(const void* X, const int32_t* ids, float* out, int64_t M, int64_t V,
                                  cudaStream_t stream);
cudaError_t launch_attention_ctx1(const void* qkv, void* out, int64_t M, int64_t nq, int64_t nkv,
                                  int64_t D, cudaStream_t stream);
// The fused RMSNorm -> GEMM layer in two steps, so that a caller can check
// and plan everything before it launches anything.  plan_fused checks the
// arguments (as bi_rmsnorm_gemm_bf16, less the workspace), resolves the pins
// and plans the GEMM (with the GLOBAL schedule where `fold_avail` bytes of
// fold workspace at `fold_ws` allow it), with no CUDA call; L->M == 0 means
// nothing to do.
// launch_fused encodes the tensor maps (returning BI_ERR_CUDA before any
// launch if that fails) and launches the layer in one of its two forms:
// in shared memory (r in the first fused_r_bytes(M) bytes of `ws`) or staged
// (r's part unused, the normalised rows in the fused_staged_bytes(M, K) bytes
// after it).
bi_status plan_fused(const void* X, const void* g, const void* W, void* Y, int64_t M, int64_t N, int64_t K,
                     float eps, const bi_pins* pins, cudaStream_t stream, GemmLaunch* L, void* fold_ws = nullptr,
                     size_t fold_avail = 0);
bi_status launch_fused(GemmLaunch& L, void* ws, bool in_smem);
// The form the pins choose: in shared memory with BI_FLAG_NORM_SMEM, else staged.
bool fused_in_smem(const GemmLaunch& L);
// Workspace bytes: r (4 bytes a row), the staged rows (M * K * 2), and both,
// each part rounded up to 256.
size_t fused_r_bytes(int64_t M);
size_t fused_staged_bytes(int64_t M, int64_t K);
size_t fused_workspace_bytes(int64_t M, int64_t K);

// Reads and clears the current device's stall word (asynchronously on
// `stream`; the caller synchronises).
cudaError_t fetch_and_clear_stall(int* host_dst, cudaStream_t stream);
// the debug-bounds build's detail word (bounds.cuh), then cleared
cudaError_t fetch_and_clear_bounds_detail(uint64_t* host_dst, cudaStream_t stream);

}  // namespace bi
