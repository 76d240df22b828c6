// Launchers of the deferred-scale grouped GEMM (16- and 32-token tiles),
// templated on the model-variant flag VAR; gemm_defer.cu instantiates VAR = 0,
// gemm_defer_var.cu VAR = 1 (two translation units, compiled in parallel).
#pragma once
#include "gemm_defer.cuh"
#include "gemm_launch.cuh"

namespace wna16 {

namespace defer_detail {

template <int BITS, int ACT, int SCL, int GEMM, int NT, int VAR>
cudaError_t launch_one(dim3 grid, size_t smem, cudaStream_t stream, const CUtensorMap& q, const CUtensorMap& s,
                       const CUtensorMap& z, const CUtensorMap& b, const CUtensorMap& x, const GemmArgs& a) {
  auto* fn = moe_gemm_defer_kernel<BITS, ACT, SCL, GEMM, NT, VAR>;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64 || !configured[dev]) {
    err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (err != cudaSuccess) return err;
    if (dev >= 0 && dev < 64) configured[dev] = true;
  }
  return launch_kernel(fn, grid, dim3(kDeferThreads), smem, stream, a.pdl != 0, q, s, z, b, x, a);
}

template <int BITS, int GEMM, int NT, int VAR>
cudaError_t by_dtype(int act, int scl, dim3 grid, size_t smem, cudaStream_t stream, const CUtensorMap& q,
                     const CUtensorMap& s, const CUtensorMap& z, const CUtensorMap& b, const CUtensorMap& x,
                     const GemmArgs& a) {
  if constexpr (BITS == 8) {
    if (act != 0) return cudaErrorInvalidValue;  // 8-bit codes: fp16 activations only
    if (scl == 0) return launch_one<8, 0, 0, GEMM, NT, VAR>(grid, smem, stream, q, s, z, b, x, a);
    return launch_one<8, 0, 1, GEMM, NT, VAR>(grid, smem, stream, q, s, z, b, x, a);
  } else {
    if (act == 0 && scl == 0) return launch_one<4, 0, 0, GEMM, NT, VAR>(grid, smem, stream, q, s, z, b, x, a);
    if (act == 0 && scl == 1) return launch_one<4, 0, 1, GEMM, NT, VAR>(grid, smem, stream, q, s, z, b, x, a);
    if (act == 1 && scl == 0) return launch_one<4, 1, 0, GEMM, NT, VAR>(grid, smem, stream, q, s, z, b, x, a);
    return launch_one<4, 1, 1, GEMM, NT, VAR>(grid, smem, stream, q, s, z, b, x, a);
  }
}

template <int BITS, int GEMM, int VAR>
cudaError_t by_tile(int nt, int act, int scl, dim3 grid, size_t smem, cudaStream_t stream, const CUtensorMap& q,
                    const CUtensorMap& s, const CUtensorMap& z, const CUtensorMap& b, const CUtensorMap& x,
                    const GemmArgs& a) {
  if (nt == 16) return by_dtype<BITS, GEMM, 16, VAR>(act, scl, grid, smem, stream, q, s, z, b, x, a);
  if (nt == 32) return by_dtype<BITS, GEMM, 32, VAR>(act, scl, grid, smem, stream, q, s, z, b, x, a);
  return cudaErrorInvalidValue;
}

template <int VAR>
cudaError_t launch(int bits, int act, int scl, int gemm, dim3 grid, size_t smem, cudaStream_t stream,
                   const CUtensorMap& q, const CUtensorMap& s, const CUtensorMap& z, const CUtensorMap& b,
                   const CUtensorMap& x, const GemmArgs& a) {
  const int nt = a.block;
  if (bits == 4)
    return gemm == 1 ? by_tile<4, 1, VAR>(nt, act, scl, grid, smem, stream, q, s, z, b, x, a)
                     : by_tile<4, 2, VAR>(nt, act, scl, grid, smem, stream, q, s, z, b, x, a);
  return gemm == 1 ? by_tile<8, 1, VAR>(nt, act, scl, grid, smem, stream, q, s, z, b, x, a)
                   : by_tile<8, 2, VAR>(nt, act, scl, grid, smem, stream, q, s, z, b, x, a);
}

}  // namespace defer_detail

}  // namespace wna16
