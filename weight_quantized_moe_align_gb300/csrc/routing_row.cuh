// Top-k routing of one token row by one warp, shared by the routing kernel
// (routing.cu) and the align kernel that routes small batches first
// (align_combine.cu). The rules are those of wna16_topk_routing in the header.
//
// Lane l holds the consecutive experts l*V .. l*V+V-1 (V = the power of two
// >= E/32, at most 8). Experts are ranked by (key, index): key = the logit
// with NaN as -inf, larger key first, ties to the lower index, so the ids
// depend only on the input bits; the one floating-point decision is the group
// score (a sum of two fp32 scores). Each lane sorts its V experts once in
// registers; a top-k pick is then a warp maximum over the lanes' heads (two
// redux.sync: the key, then the lowest index at that key), and the winning
// lane drops its head. When every group is a power-of-two run of whole lanes,
// a group's best two come from a segmented butterfly over its lanes and the
// groups are ranked in one pass of broadcasts; other group shapes take the
// groups one at a time.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>

namespace wna16 {
namespace routing {

constexpr unsigned kFull = 0xFFFFFFFFu;
constexpr int kNone = 0x7FFFFFFF;  // index of an empty list entry (key 0)

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__half x) { return __half2float(x); }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// Order-preserving map of a ranking key (never NaN) to an unsigned integer:
// larger key -> larger integer, -0 and +0 alike (they tie), -inf -> 0x7FFFFF,
// so 0 (an empty entry) ranks below every expert.
__device__ __forceinline__ uint32_t order_key(float k) {
  uint32_t b = __float_as_uint(k);
  if ((b << 1) == 0u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ bool ahead(uint32_t ka, int ia, uint32_t kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

// compare-exchange: the entry ranked ahead goes to position a
template <int N>
__device__ __forceinline__ void cex(uint32_t (&k)[N], int (&x)[N], int a, int b) {
  const bool s = ahead(k[b], x[b], k[a], x[a]);
  const uint32_t ka = s ? k[b] : k[a], kb = s ? k[a] : k[b];
  const int xa = s ? x[b] : x[a], xb = s ? x[a] : x[b];
  k[a] = ka;
  k[b] = kb;
  x[a] = xa;
  x[b] = xb;
}

// bitonic sort of the lane's entries, best first (N a power of two)
template <int N>
__device__ __forceinline__ void sort_ranked(uint32_t (&k)[N], int (&x)[N]) {
#pragma unroll
  for (int size = 2; size <= N; size <<= 1)
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1)
#pragma unroll
      for (int i = 0; i < N; ++i) {
        const int j = i ^ stride;
        if (j > i) {
          if ((i & size) == 0) cex(k, x, i, j);
          else cex(k, x, j, i);
        }
      }
}

// the best of one entry per lane: its key and index, the same on every lane
__device__ __forceinline__ void warp_top(uint32_t k, int x, uint32_t& mk, int& mx) {
  mk = __reduce_max_sync(kFull, k);
  mx = static_cast<int>(__reduce_min_sync(kFull, k == mk ? static_cast<uint32_t>(x) : 0xFFFFFFFFu));
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

// Routes token row `row` with one whole warp (lane = threadIdx.x % 32): writes
// its top-k ids and weights to a.ids / a.weights. Every lane of the warp must
// call it with the same row.
template <typename T, int VPL>
__device__ __forceinline__ void route_row(const T* __restrict__ logits, const RouteArgs& a, int row) {
  const int lane = threadIdx.x & 31;
  const int ng = a.n_groups;
  const int gs = a.E / ng;
  const int lpg = gs / VPL;  // lanes per group when groups are runs of whole lanes
  const bool whole_lanes = ng > 1 && gs % VPL == 0 && (lpg & (lpg - 1)) == 0;
  {
    const T* src = logits + static_cast<size_t>(row) * a.E;
    uint32_t k[VPL];
    int x[VPL];
    float v[VPL];
#pragma unroll
    for (int j = 0; j < VPL; ++j) {
      const int e = lane * VPL + j;
      v[j] = 0.f;
      k[j] = 0u;
      x[j] = kNone;
      if (e < a.E) {
        v[j] = to_f32(src[e]);
        k[j] = order_key(isnan(v[j]) ? -INFINITY : v[j]);
        x[j] = e;
      }
    }
    // softmax over the whole row: max and sum of exp(v - max)
    float m = 0.f, denom = 1.f;
    if (!a.sigmoid && (!a.renorm || ng > 1)) {
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < VPL; ++j)
        if (x[j] != kNone) mx = fmaxf(mx, v[j]);
      m = warp_max(mx);
      float s = 0.f;
#pragma unroll
      for (int j = 0; j < VPL; ++j)
        if (x[j] != kNone) s += expf(v[j] - m);
      denom = warp_sum(s);
    }
    auto score = [&](float y) { return a.sigmoid ? sigmoid(y) : expf(y - m) / denom; };
    // group score = score of its best expert + score of its second best (NaN -> -inf)
    auto group_score = [&](int e1, int e2) {
      const float s = score(to_f32(src[e1])) + score(to_f32(src[e2]));
      return isnan(s) ? -INFINITY : s;
    };
    // rank of the group scored `gsc` (group g) among the groups, whose scores
    // sit on lanes 0, stride, 2*stride ...; ties to the lower group
    auto group_rank = [&](float gsc, int g, int stride) {
      int rank = 0;
      for (int h = 0; h < ng; ++h) {
        const float o = __shfl_sync(kFull, gsc, h * stride);
        rank += (o > gsc || (o == gsc && h < g)) ? 1 : 0;
      }
      return rank;
    };

    sort_ranked<VPL>(k, x);
    if (whole_lanes) {
      // group g = lanes g*lpg .. g*lpg+lpg-1: merge the lanes' best two
      uint32_t k1 = k[0], k2 = VPL > 1 ? k[VPL > 1 ? 1 : 0] : 0u;
      int x1 = x[0], x2 = VPL > 1 ? x[VPL > 1 ? 1 : 0] : kNone;
      for (int o = lpg >> 1; o > 0; o >>= 1) {
        const uint32_t p1 = __shfl_xor_sync(kFull, k1, o), p2 = __shfl_xor_sync(kFull, k2, o);
        const int q1 = __shfl_xor_sync(kFull, x1, o), q2 = __shfl_xor_sync(kFull, x2, o);
        if (ahead(p1, q1, k1, x1)) {
          if (!ahead(k1, x1, p2, q2)) {
            k1 = p2;
            x1 = q2;
          }
          k2 = k1;
          x2 = x1;
          k1 = p1;
          x1 = q1;
        } else if (ahead(p1, q1, k2, x2)) {
          k2 = p1;
          x2 = q1;
        }
      }
      const int g = lane / lpg;
      // a group holds >= 2 experts, so x1 and x2 are experts on the lanes of a group
      const float gsc = g < ng ? group_score(x1, x2) : -INFINITY;
      const int rank = group_rank(gsc, g, lpg);
      if (g >= ng || rank >= a.topk_groups) {
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
          k[j] = 0u;
          x[j] = kNone;
        }
      }
    } else if (ng > 1) {
      // any other group shape: the groups one at a time; lane g keeps group g's score
      float my_gscore = -INFINITY;
      for (int g = 0; g < ng; ++g) {
        const int lo = g * gs, hi = lo + gs;
        // this lane's first two entries of group g (the list is sorted)
        uint32_t f1 = 0u, f2 = 0u;
        int y1 = kNone, y2 = kNone;
        bool h1 = false, h2 = false;
#pragma unroll
        for (int j = 0; j < VPL; ++j) {
          const bool in = x[j] >= lo && x[j] < hi;
          if (in && h1 && !h2) {
            f2 = k[j];
            y2 = x[j];
            h2 = true;
          }
          if (in && !h1) {
            f1 = k[j];
            y1 = x[j];
            h1 = true;
          }
        }
        uint32_t mk;
        int b1, b2;
        warp_top(f1, y1, mk, b1);
        const bool won = y1 == b1;
        warp_top(won ? f2 : f1, won ? y2 : y1, mk, b2);
        if (lane == g) my_gscore = group_score(b1, b2);
      }
      const int rank = group_rank(my_gscore, lane, 1);
      const uint32_t kept = __ballot_sync(kFull, lane < ng && rank < a.topk_groups);
#pragma unroll
      for (int j = 0; j < VPL; ++j)
        if (x[j] != kNone && !((kept >> (x[j] / gs)) & 1u)) {
          k[j] = 0u;
          x[j] = kNone;
        }
      sort_ranked<VPL>(k, x);
    }

    // the top-k experts, best first: each pick takes the best head and its lane
    // drops it; lane r keeps pick r
    int my_id = 0;
    for (int r = 0; r < a.topk; ++r) {
      uint32_t mk;
      int mx;
      warp_top(k[0], x[0], mk, mx);
      if (x[0] == mx) {
#pragma unroll
        for (int j = 0; j + 1 < VPL; ++j) {
          k[j] = k[j + 1];
          x[j] = x[j + 1];
        }
        k[VPL - 1] = 0u;
        x[VPL - 1] = kNone;
      }
      if (lane == r) my_id = mx;
    }
    const bool mine = lane < a.topk;
    const float my_v = mine ? to_f32(src[my_id]) : 0.f;
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

}  // namespace routing
}  // namespace wna16
