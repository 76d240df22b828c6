// wna16_topk_routing: router logits [M, E] -> top-k expert ids and weights.
//
// The layer's first stage (top-k routing ids and weights, vLLM PR #12185 and
// PR #6502, whose Mixtral, Qwen2-MoE and DeepSeek-V3 models route this way).
// The pages give no formulas; the rules are the header's readings.
//
// One warp per token row (routing_row.cuh), four rows per CTA.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>

#include "routing_row.cuh"
#include "wna16_moe.h"

namespace wna16 {

namespace {

using namespace routing;
constexpr int kRouteWarps = 4;  // rows per CTA

template <typename T, int VPL>
__global__ void __launch_bounds__(kRouteWarps * 32) topk_routing_kernel(const T* __restrict__ logits, const RouteArgs a) {
  for (int row = blockIdx.x * kRouteWarps + (threadIdx.x >> 5); row < a.M; row += gridDim.x * kRouteWarps)
    route_row<T, VPL>(logits, a, row);
}

template <typename T>
void launch_routing(const void* logits, const RouteArgs& a, cudaStream_t s) {
  const int vpl = (a.E + 31) / 32;
  const int rows_ctas = (a.M + kRouteWarps - 1) / kRouteWarps;
  const unsigned grid = static_cast<unsigned>(rows_ctas < 152 * 16 ? rows_ctas : 152 * 16);
  const T* p = static_cast<const T*>(logits);
  if (vpl <= 1) topk_routing_kernel<T, 1><<<grid, kRouteWarps * 32, 0, s>>>(p, a);
  else if (vpl <= 2) topk_routing_kernel<T, 2><<<grid, kRouteWarps * 32, 0, s>>>(p, a);
  else if (vpl <= 4) topk_routing_kernel<T, 4><<<grid, kRouteWarps * 32, 0, s>>>(p, a);
  else topk_routing_kernel<T, 8><<<grid, kRouteWarps * 32, 0, s>>>(p, a);
}

}  // namespace

}  // namespace wna16

using namespace wna16;

namespace wna16 {

// Host-side argument checks of the routing call (no CUDA call).
wna16_status routing_check(const void* logits, wna16_dtype logits_dtype, int64_t M, int E, int topk,
                           wna16_scoring scoring, int n_groups, int topk_groups, const int32_t* topk_ids,
                           const float* topk_weights) {
  if (M < 0 || M >= (int64_t(1) << 31) || E < 1 || E > 256 || topk < 1 || topk > 32 || topk > E)
    return WNA16_ERR_INVALID_ARG;
  if (scoring != WNA16_SCORE_SOFTMAX && scoring != WNA16_SCORE_SIGMOID) return WNA16_ERR_INVALID_ARG;
  if (logits_dtype != WNA16_F16 && logits_dtype != WNA16_BF16 && logits_dtype != WNA16_F32)
    return WNA16_ERR_INVALID_ARG;
  if (n_groups < 1 || n_groups > 32 || E % n_groups) return WNA16_ERR_INVALID_ARG;
  if (n_groups > 1) {
    const int gs = E / n_groups;
    if (gs < 2 || topk_groups < 1 || topk_groups > n_groups || topk > topk_groups * gs)
      return WNA16_ERR_INVALID_ARG;
  }
  if (M == 0) return WNA16_OK;
  if (!logits || !topk_ids || !topk_weights) return WNA16_ERR_INVALID_ARG;
  const size_t esz = logits_dtype == WNA16_F32 ? 4 : 2;
  if ((reinterpret_cast<uintptr_t>(logits) % esz) || (reinterpret_cast<uintptr_t>(topk_ids) & 3u) ||
      (reinterpret_cast<uintptr_t>(topk_weights) & 3u))
    return WNA16_ERR_INVALID_ARG;
  return WNA16_OK;
}

}  // namespace wna16

extern "C" wna16_status wna16_topk_routing(const void* logits, wna16_dtype logits_dtype, int64_t M, int E,
                                           int topk, wna16_scoring scoring, int renormalize, int n_groups,
                                           int topk_groups, int32_t* topk_ids, float* topk_weights, void* stream) {
  const wna16_status st =
      routing_check(logits, logits_dtype, M, E, topk, scoring, n_groups, topk_groups, topk_ids, topk_weights);
  if (st != WNA16_OK || M == 0) return st;
  RouteArgs a{static_cast<int>(M), E, topk, scoring == WNA16_SCORE_SIGMOID ? 1 : 0, renormalize ? 1 : 0,
              n_groups, n_groups > 1 ? topk_groups : 1, topk_ids, topk_weights};
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (logits_dtype == WNA16_F32) launch_routing<float>(logits, a, s);
  else if (logits_dtype == WNA16_F16) launch_routing<__half>(logits, a, s);
  else launch_routing<__nv_bfloat16>(logits, a, s);
  return cudaGetLastError() == cudaSuccess ? WNA16_OK : WNA16_ERR_CUDA;
}
