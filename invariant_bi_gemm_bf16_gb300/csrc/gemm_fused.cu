// gemm_fused.cu -- the GEMM kernel instances with the RMSNorm prologue in
// shared memory (bi_rmsnorm_gemm_bf16): the kernel of gemm_kernel.cuh with
// FUSED = true, compiled in its own translation unit so that the two sets of
// instances build in parallel.
#include "gemm_kernel.cuh"

namespace bi {

cudaError_t launch_gemm_fused(const GemmLaunch& L) {
  if (!L.g || (!L.rrow && (L.M > kRowScaleInKernelMax || L.m_tiles != 1 || !L.X))) return cudaErrorInvalidValue;
  return L.pair ? launch_p<true, true>(L) : launch_p<true, false>(L);
}

}  // namespace bi
