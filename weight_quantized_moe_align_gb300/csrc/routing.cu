// wna16_topk_routing: router logits [M, E] -> top-k expert ids and weights.
//
// The layer's first stage (top-k routing ids and weights, vLLM PR #12185 and
// PR #6502, whose Mixtral, Qwen2-MoE and DeepSeek-V3 models route this way).
// The pages give no formulas; the rules are the header's readings.
//
// One warp per token row; lane l holds experts l, l + 32, ... (coalesced
// loads, at most 8 per lane for E <= 256). Every choice is a warp arg-max
// over (key, index), key = the logit with NaN as -inf, larger key first and
// ties to the lower index, so the ids depend only on the input bits; the one
// floating-point decision is the group score (a sum of two fp32 scores).
// The work per row is a few dozen shuffle rounds: the kernel is bound by
// its launch and by the logits read, never near the GEMMs' time.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>

#include "wna16_moe.h"

namespace wna16 {

namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kRouteWarps = 4;  // rows per CTA

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// a candidate: ranking key, expert index, logit
struct Cand {
  float key;
  int idx;
  float v;
};

__device__ __forceinline__ bool better(float ka, int ia, float kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

// Best of the lane's candidates (bit j of `mask` = slot j), then the best over
// the warp; every lane returns the same winner. A lane without candidates
// offers (-inf, INT_MAX), which any real candidate beats.
template <int VPL>
__device__ __forceinline__ Cand warp_best(const float (&key)[VPL], const float (&v)[VPL], uint32_t mask, int lane) {
  Cand c{-INFINITY, 0x7FFFFFFF, 0.f};
#pragma unroll
  for (int j = 0; j < VPL; ++j) {
    const int e = lane + 32 * j;
    if (((mask >> j) & 1u) && better(key[j], e, c.key, c.idx)) c = Cand{key[j], e, v[j]};
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float k2 = __shfl_xor_sync(kFull, c.key, o);
    const int i2 = __shfl_xor_sync(kFull, c.idx, o);
    const float v2 = __shfl_xor_sync(kFull, c.v, o);
    if (better(k2, i2, c.key, c.idx)) c = Cand{k2, i2, v2};
  }
  return c;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
  return x;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(kFull, x, o));
  return x;
}

__device__ __forceinline__ float sigmoid(float v) { return 1.0f / (1.0f + expf(-v)); }

struct RouteArgs {
  int M, E, topk, sigmoid, renorm, n_groups, topk_groups;
  int32_t* ids;
  float* weights;
};

template <typename T, int VPL>
__global__ void __launch_bounds__(kRouteWarps * 32) topk_routing_kernel(const T* __restrict__ logits, const RouteArgs a) {
  const int lane = threadIdx.x & 31;
  const int gs = a.E / a.n_groups;
  for (int row = blockIdx.x * kRouteWarps + (threadIdx.x >> 5); row < a.M; row += gridDim.x * kRouteWarps) {
    const T* src = logits + static_cast<size_t>(row) * a.E;
    float v[VPL], key[VPL];
    uint32_t valid = 0;
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int e = lane + 32 * j;
      v[j] = 0.f;
      key[j] = -INFINITY;
      if (e < a.E) {
        v[j] = to_f32(src[e]);
        key[j] = isnan(v[j]) ? -INFINITY : v[j];
        valid |= 1u << j;
      }
    }
    // softmax over the whole row: max and sum of exp(v - max)
    float m = 0.f, denom = 1.f;
    if (!a.sigmoid && (!a.renorm || a.n_groups > 1)) {
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < VPL; ++j)
        if ((valid >> j) & 1u) mx = fmaxf(mx, v[j]);
      m = warp_max(mx);
      float s = 0.f;
#pragma unroll
      for (int j = 0; j < VPL; ++j)
        if ((valid >> j) & 1u) s += expf(v[j] - m);
      denom = warp_sum(s);
    }
    auto score = [&](float x) { return a.sigmoid ? sigmoid(x) : expf(x - m) / denom; };

    uint32_t cand = valid;
    if (a.n_groups > 1) {
      // group score = score of its best expert + score of its second best;
      // lane g keeps group g's score
      float my_gscore = -INFINITY;
      for (int g = 0; g < a.n_groups; ++g) {
        const int lo = g * gs, hi = lo + gs;
        uint32_t gm = 0;
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
          const int e = lane + 32 * j;
          if (e >= lo && e < hi) gm |= 1u << j;
        }
        gm &= valid;
        const Cand b1 = warp_best<VPL>(key, v, gm, lane);
        if ((b1.idx & 31) == lane) gm &= ~(1u << (b1.idx >> 5));
        const Cand b2 = warp_best<VPL>(key, v, gm, lane);
        const float gsc = score(b1.v) + score(b2.v);
        if (lane == g) my_gscore = isnan(gsc) ? -INFINITY : gsc;
      }
      // keep the topk_groups best groups (ties to the lower group)
      uint32_t kept = 0;
      for (int r = 0; r < a.topk_groups; ++r) {
        float bk = (lane < a.n_groups && !((kept >> lane) & 1u)) ? my_gscore : -INFINITY;
        int bi = (lane < a.n_groups && !((kept >> lane) & 1u)) ? lane : 0x7FFFFFFF;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float k2 = __shfl_xor_sync(kFull, bk, o);
          const int i2 = __shfl_xor_sync(kFull, bi, o);
          if (better(k2, i2, bk, bi)) {
            bk = k2;
            bi = i2;
          }
        }
        kept |= 1u << bi;
      }
      uint32_t km = 0;
#pragma unroll
      for (int j = 0; j < VPL; ++j) {
        const int e = lane + 32 * j;
        if (e < a.E && ((kept >> (e / gs)) & 1u)) km |= 1u << j;
      }
      cand &= km;
    }

    // the top-k experts among the candidates, best first; lane r keeps pick r
    int my_id = 0;
    float my_v = 0.f;
    for (int r = 0; r < a.topk; ++r) {
      const Cand b = warp_best<VPL>(key, v, cand, lane);
      if ((b.idx & 31) == lane) cand &= ~(1u << (b.idx >> 5));
      if (lane == r) {
        my_id = b.idx;
        my_v = b.v;
      }
    }
    const bool mine = lane < a.topk;
    float w;
    if (a.sigmoid) {
      w = sigmoid(my_v);
      if (a.renorm) w = w / warp_sum(mine ? w : 0.f);
    } else if (a.renorm) {
      // softmax over the selected logits, relative to the best one
      const float v0 = __shfl_sync(kFull, my_v, 0);
      const float ex = expf(my_v - v0);
      w = ex / warp_sum(mine ? ex : 0.f);
    } else {
      w = expf(my_v - m) / denom;
    }
    if (mine) {
      a.ids[static_cast<size_t>(row) * a.topk + lane] = my_id;
      a.weights[static_cast<size_t>(row) * a.topk + lane] = w;
    }
  }
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
