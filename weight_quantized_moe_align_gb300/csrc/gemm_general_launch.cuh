// Launchers of the general grouped dequant GEMM, templated on the code width
// and the layout; gemm_w4.cu / gemm_w8.cu instantiate the two-CTA-per-SM
// layout, gemm_w4_wide.cu / gemm_w8_wide.cu the one-CTA-per-SM one (four
// translation units, compiled in parallel).
#pragma once
#include "gemm_kernel.cuh"
#include "gemm_launch.cuh"

namespace wna16 {

namespace general_detail {

template <int BITS, int ACT, int SCL, int GEMM, int WIDE, int EXT>
cudaError_t launch_one(dim3 grid, size_t smem, cudaStream_t stream, const CUtensorMap& q, const CUtensorMap& s,
                       const CUtensorMap& z, const CUtensorMap& b, const GemmArgs& a) {
  auto* fn = moe_gemm_kernel<BITS, ACT, SCL, GEMM, WIDE, EXT>;
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
  return launch_kernel(fn, grid, dim3(gemm_threads(WIDE)), smem, stream, a.pdl != 0, q, s, z, b, a);
}

template <int BITS, int GEMM, int WIDE, int EXT>
cudaError_t by_dtype(int act, int scl, dim3 grid, size_t smem, cudaStream_t stream, const CUtensorMap& q,
                     const CUtensorMap& s, const CUtensorMap& z, const CUtensorMap& b, const GemmArgs& a) {
  if (act == 0 && scl == 0) return launch_one<BITS, 0, 0, GEMM, WIDE, EXT>(grid, smem, stream, q, s, z, b, a);
  if (act == 0 && scl == 1) return launch_one<BITS, 0, 1, GEMM, WIDE, EXT>(grid, smem, stream, q, s, z, b, a);
  if (act == 1 && scl == 0) return launch_one<BITS, 1, 0, GEMM, WIDE, EXT>(grid, smem, stream, q, s, z, b, a);
  return launch_one<BITS, 1, 1, GEMM, WIDE, EXT>(grid, smem, stream, q, s, z, b, a);
}

// EXT: prepacked weights, biases, clamped SwiGLU, act-order or the atomic down reduction
template <int BITS, int WIDE>
cudaError_t launch(int act, int scl, int gemm, dim3 grid, size_t smem, cudaStream_t stream, const CUtensorMap& q,
                   const CUtensorMap& s, const CUtensorMap& z, const CUtensorMap& b, const GemmArgs& a) {
  const bool ext = a.wpack || a.bias || a.glu || a.act_pos || a.atomic_out;
  if (ext)
    return gemm == 1 ? by_dtype<BITS, 1, WIDE, 1>(act, scl, grid, smem, stream, q, s, z, b, a)
                     : by_dtype<BITS, 2, WIDE, 1>(act, scl, grid, smem, stream, q, s, z, b, a);
  return gemm == 1 ? by_dtype<BITS, 1, WIDE, 0>(act, scl, grid, smem, stream, q, s, z, b, a)
                   : by_dtype<BITS, 2, WIDE, 0>(act, scl, grid, smem, stream, q, s, z, b, a);
}

}  // namespace general_detail

}  // namespace wna16
