// Instantiations of the deferred-scale grouped GEMM, default epilogues.
#include "gemm_defer_launch.cuh"

namespace wna16 {

bool defer_supported(int bits, int act) { return bits == 4 || (bits == 8 && act == 0); }

cudaError_t launch_gemm_defer(int bits, int act, int scl, int gemm, dim3 grid, size_t smem, cudaStream_t stream,
                              const CUtensorMap& q, const CUtensorMap& s, const CUtensorMap& z,
                              const CUtensorMap& b, const CUtensorMap& x, const GemmArgs& a) {
  if (a.wpack || a.bias || a.glu || a.atomic_out) return launch_gemm_defer_var(bits, act, scl, gemm, grid, smem, stream, q, s, z, b, x, a);
  return defer_detail::launch<0>(bits, act, scl, gemm, grid, smem, stream, q, s, z, b, x, a);
}

}  // namespace wna16
