// wna16_act_order_prepare: act-order (GPTQ desc_act) weights -> the plain
// grouped layout plus the K permutation the layer applies to its operands.
//
// With act-order, column k of an expert's matrix belongs to group g_idx[k]
// (vLLM PR #14138 passes g_idx and sort_indices to the marlin GEMM, empty in its
// benchmark). Listing the columns by ascending group, ascending k inside a
// group (perm), puts every group's G columns side by side, so that
// W'[:, i] = W[:, perm[i]] is a plain grouped matrix with group i / G and
// W x = W' x' for x'[i] = x[perm[i]]. The scales and zero points, stored per
// group, are already in that order.
#include <cuda_runtime.h>

#include <algorithm>

#include "common.cuh"
#include "wna16_moe.h"

namespace wna16 {

namespace {

// One CTA per expert. perm and inv start as the identity; thread g then lists
// the columns of group g. Every output stays in [0, K) whatever g_idx holds; a
// group that does not have exactly G columns sets WNA16_DEV_BAD_GROUPS.
__global__ void __launch_bounds__(256) act_order_perm_kernel(const int32_t* __restrict__ g_idx, int K, int G,
                                                             int32_t* __restrict__ perm, int32_t* __restrict__ inv,
                                                             int32_t* __restrict__ status) {
  const int e = blockIdx.x;
  const int32_t* gi = g_idx + static_cast<size_t>(e) * K;
  int32_t* pe = perm + static_cast<size_t>(e) * K;
  int32_t* ie = inv ? inv + static_cast<size_t>(e) * K : nullptr;
  for (int k = threadIdx.x; k < K; k += blockDim.x) {
    pe[k] = k;
    if (ie) ie[k] = k;
  }
  __syncthreads();
  const int groups = K / G;
  bool bad = false;
  for (int g = threadIdx.x; g < groups; g += blockDim.x) {
    int c = 0;
    for (int k = 0; k < K; ++k) {
      if (gi[k] != g) continue;
      if (c < G) {
        pe[g * G + c] = k;
        if (ie) ie[k] = g * G + c;
      }
      ++c;
    }
    bad |= c != G;
  }
  if (bad) atomicOr(status, WNA16_DEV_BAD_GROUPS);
}

// One thread per packed output word: codes of columns perm[i] gathered into
// position i (out-of-range entries give code 0).
template <int BITS>
__global__ void __launch_bounds__(256) act_order_repack_kernel(const uint32_t* __restrict__ q,
                                                               const int32_t* __restrict__ perm, int N, int K,
                                                               long long total, uint32_t* __restrict__ q_out) {
  constexpr int PF = 32 / BITS;
  constexpr uint32_t MASK = (1u << BITS) - 1;
  const int kw = K / PF;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total; idx += stride) {
    const int w = static_cast<int>(idx % kw);
    const long long rn = idx / kw;  // e * N + n
    const int e = static_cast<int>(rn / N);
    const uint32_t* row = q + rn * kw;
    const int32_t* pe = perm + static_cast<size_t>(e) * K + w * PF;
    uint32_t out = 0;
#pragma unroll
    for (int j = 0; j < PF; ++j) {
      const int k = pe[j];
      if (static_cast<unsigned>(k) < static_cast<unsigned>(K))
        out |= ((row[k / PF] >> (BITS * (k % PF))) & MASK) << (BITS * j);
    }
    q_out[idx] = out;
  }
}

}  // namespace

}  // namespace wna16

using namespace wna16;

extern "C" wna16_status wna16_act_order_prepare(const int32_t* q, const int32_t* g_idx, int E, int64_t N,
                                                int64_t K, int bits, int group_size, int32_t* q_out,
                                                int32_t* perm, int32_t* inv_perm, int32_t* device_status,
                                                void* stream) {
  if (E < 1 || E > 256 || N <= 0 || K <= 0 || (bits != 4 && bits != 8) || group_size <= 0)
    return WNA16_ERR_INVALID_ARG;
  const int pf = 32 / bits;
  if (K % group_size || K % pf || N >= (int64_t(1) << 24) || K >= (int64_t(1) << 24)) return WNA16_ERR_UNSUPPORTED;
  if (!g_idx || !perm || !device_status || (q == nullptr) != (q_out == nullptr)) return WNA16_ERR_INVALID_ARG;
  const void* ptrs[] = {q, g_idx, q_out, perm, inv_perm, device_status};
  for (const void* p : ptrs)
    if (reinterpret_cast<uintptr_t>(p) & 3u) return WNA16_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  act_order_perm_kernel<<<E, 256, 0, s>>>(g_idx, static_cast<int>(K), group_size, perm, inv_perm, device_status);
  if (cudaGetLastError() != cudaSuccess) return WNA16_ERR_CUDA;
  if (q) {
    const long long total = static_cast<long long>(E) * N * (K / pf);
    const long long want = (total + 255) / 256;
    const unsigned blocks = static_cast<unsigned>(std::min<long long>(want, 152ll * 16));
    if (bits == 4)
      act_order_repack_kernel<4><<<blocks, 256, 0, s>>>(reinterpret_cast<const uint32_t*>(q), perm,
                                                        static_cast<int>(N), static_cast<int>(K), total,
                                                        reinterpret_cast<uint32_t*>(q_out));
    else
      act_order_repack_kernel<8><<<blocks, 256, 0, s>>>(reinterpret_cast<const uint32_t*>(q), perm,
                                                        static_cast<int>(N), static_cast<int>(K), total,
                                                        reinterpret_cast<uint32_t*>(q_out));
    if (cudaGetLastError() != cudaSuccess) return WNA16_ERR_CUDA;
  }
  return WNA16_OK;
}
