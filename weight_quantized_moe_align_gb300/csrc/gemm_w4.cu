// Instantiations of the grouped dequant GEMM for 4-bit weights.
#include "gemm_kernel.cuh"
#include "gemm_launch.cuh"

namespace wna16 {

namespace {

template <int ACT, int SCL, int GEMM, int LEAN, int EXT>
cudaError_t launch_one(dim3 grid, size_t smem, cudaStream_t stream, const CUtensorMap& q,
                       const CUtensorMap& s, const CUtensorMap& z, const CUtensorMap& b, const GemmArgs& a) {
  auto* fn = moe_gemm_kernel<4, ACT, SCL, GEMM, LEAN, EXT>;
  // The opt-in shared-memory limit is per function and context; set it at most
  // once per device.
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (err != cudaSuccess) return err;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  return launch_kernel(fn, grid, dim3(gemm_threads(LEAN)), smem, stream, a.pdl != 0, q, s, z, b, a);
}

template <int GEMM, int LEAN, int EXT>
cudaError_t by_dtype(int act, int scl, dim3 grid, size_t smem, cudaStream_t stream,
                     const CUtensorMap& q, const CUtensorMap& s, const CUtensorMap& z,
                     const CUtensorMap& b, const GemmArgs& a) {
  if (act == 0 && scl == 0) return launch_one<0, 0, GEMM, LEAN, EXT>(grid, smem, stream, q, s, z, b, a);
  if (act == 0 && scl == 1) return launch_one<0, 1, GEMM, LEAN, EXT>(grid, smem, stream, q, s, z, b, a);
  if (act == 1 && scl == 0) return launch_one<1, 0, GEMM, LEAN, EXT>(grid, smem, stream, q, s, z, b, a);
  return launch_one<1, 1, GEMM, LEAN, EXT>(grid, smem, stream, q, s, z, b, a);
}

}  // namespace

cudaError_t launch_gemm_w4(int act, int scl, int gemm, int lean, dim3 grid, size_t smem,
                            cudaStream_t stream, const CUtensorMap& q, const CUtensorMap& s,
                            const CUtensorMap& z, const CUtensorMap& b, const GemmArgs& a) {
  // EXT: prepacked weights, biases, clamped SwiGLU or act-order (not built for the lean layout)
  const bool ext = a.wpack || a.bias || a.glu || a.act_pos || a.atomic_out;
  if (lean) {
    if (ext) return cudaErrorInvalidValue;
    if (gemm == 1) return by_dtype<1, 1, 0>(act, scl, grid, smem, stream, q, s, z, b, a);
    return by_dtype<2, 1, 0>(act, scl, grid, smem, stream, q, s, z, b, a);
  }
  if (ext)
    return gemm == 1 ? by_dtype<1, 0, 1>(act, scl, grid, smem, stream, q, s, z, b, a)
                     : by_dtype<2, 0, 1>(act, scl, grid, smem, stream, q, s, z, b, a);
  if (gemm == 1) return by_dtype<1, 0, 0>(act, scl, grid, smem, stream, q, s, z, b, a);
  return by_dtype<2, 0, 0>(act, scl, grid, smem, stream, q, s, z, b, a);
}

}  // namespace wna16
