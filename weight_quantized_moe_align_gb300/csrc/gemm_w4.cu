// Instantiations of the general grouped dequant GEMM for 4-bit weights,
// two CTAs per SM (token tiles up to 64); the one-CTA-per-SM layout is in
// gemm_w4_wide.cu.
#include "gemm_general_launch.cuh"

namespace wna16 {

cudaError_t launch_gemm_w4(int act, int scl, int gemm, int wide, dim3 grid, size_t smem, cudaStream_t stream,
                           const CUtensorMap& q, const CUtensorMap& s, const CUtensorMap& z, const CUtensorMap& b,
                           const GemmArgs& a) {
  if (wide) return launch_gemm_w4_wide(act, scl, gemm, grid, smem, stream, q, s, z, b, a);
  return general_detail::launch<4, 0>(act, scl, gemm, grid, smem, stream, q, s, z, b, a);
}

}  // namespace wna16
