// Instantiations of the deferred-scale grouped GEMM with the model-variant
// epilogues (biases, clamped SwiGLU).
#include "gemm_defer_launch.cuh"

namespace wna16 {

cudaError_t launch_gemm_defer_var(int bits, int act, int scl, int gemm, dim3 grid, size_t smem,
                                  cudaStream_t stream, const CUtensorMap& q, const CUtensorMap& s,
                                  const CUtensorMap& z, const CUtensorMap& b, const CUtensorMap& x,
                                  const GemmArgs& a) {
  return defer_detail::launch<1>(bits, act, scl, gemm, grid, smem, stream, q, s, z, b, x, a);
}

}  // namespace wna16
