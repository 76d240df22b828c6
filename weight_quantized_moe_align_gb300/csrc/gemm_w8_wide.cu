// Instantiations of the general grouped dequant GEMM for 8-bit weights, one
// CTA per SM with three dequant warpgroups (token tiles of 128 and 256).
#include "gemm_general_launch.cuh"

namespace wna16 {

cudaError_t launch_gemm_w8_wide(int act, int scl, int gemm, dim3 grid, size_t smem, cudaStream_t stream,
                                 const CUtensorMap& q, const CUtensorMap& s, const CUtensorMap& z,
                                 const CUtensorMap& b, const GemmArgs& a) {
  return general_detail::launch<8, 1>(act, scl, gemm, grid, smem, stream, q, s, z, b, a);
}

}  // namespace wna16
