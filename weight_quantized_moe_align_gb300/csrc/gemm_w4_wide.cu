// Instantiations of the general grouped dequant GEMM for 4-bit weights, one
// CTA per SM with three dequant warpgroups (token tiles of 128 and 256).
#include "gemm_general_launch.cuh"

namespace wna16 {

cudaError_t launch_gemm_w4_wide(int act, int scl, int gemm, dim3 grid, size_t smem, cudaStream_t stream,
                                 const CUtensorMap& q, const CUtensorMap& s, const CUtensorMap& z,
                                 const CUtensorMap& b, const GemmArgs& a) {
  return general_detail::launch<4, 1>(act, scl, gemm, grid, smem, stream, q, s, z, b, a);
}

}  // namespace wna16
