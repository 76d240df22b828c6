// Host-side entry points of the kernel translation units.
#pragma once

#include "common.cuh"
#include "wna16_moe.h"

namespace wna16 {

// gemm: 1 = gate/up + silu*up epilogue, 2 = down + top-k weight epilogue.
cudaError_t launch_gemm_w4(int act, int scl, int gemm, int lean, dim3 grid, size_t smem, cudaStream_t stream,
                           const CUtensorMap& q, const CUtensorMap& s, const CUtensorMap& z,
                           const CUtensorMap& b, const GemmArgs& a);
cudaError_t launch_gemm_w8(int act, int scl, int gemm, int lean, dim3 grid, size_t smem, cudaStream_t stream,
                           const CUtensorMap& q, const CUtensorMap& s, const CUtensorMap& z,
                           const CUtensorMap& b, const GemmArgs& a);

// Deferred-scale GEMM for 16-token tiles; `x` maps the per-stage token sums.
bool defer_supported(int bits, int act);
cudaError_t launch_gemm_defer(int bits, int act, int scl, int gemm, dim3 grid, size_t smem, cudaStream_t stream,
                              const CUtensorMap& q, const CUtensorMap& s, const CUtensorMap& z,
                              const CUtensorMap& b, const CUtensorMap& x, const GemmArgs& a);
// the same for prepacked weights or the model-variant epilogues (a.wpack, a.bias or a.glu set)
cudaError_t launch_gemm_defer_var(int bits, int act, int scl, int gemm, dim3 grid, size_t smem, cudaStream_t stream,
                              const CUtensorMap& q, const CUtensorMap& s, const CUtensorMap& z,
                              const CUtensorMap& b, const CUtensorMap& x, const GemmArgs& a);

cudaError_t launch_align(const int32_t* ids, int P, int E, int block, int cap, int32_t* sorted_ids,
                         int32_t* expert_ids, int32_t* num_post_pad, int32_t* counts,
                         int32_t* status, int32_t* slot_of_pair, int32_t* block_rows, cudaStream_t stream);
// Routing of a small batch (M <= kRouteAlignRows rows) and its align in one
// launch of one CTA; logits_dtype: 0 fp16, 1 bf16, 2 fp32.
constexpr int kRouteAlignRows = 128;
cudaError_t launch_route_align(const void* logits, int logits_dtype, int M, int E, int topk, int sigmoid, int renorm,
                               int n_groups, int topk_groups, int32_t* routed_ids, float* routed_weights, int block,
                               int cap, int32_t* sorted_ids, int32_t* expert_ids, int32_t* num_post_pad,
                               int32_t* counts, int32_t* status, int32_t* slot_of_pair, int32_t* block_rows,
                               cudaStream_t stream);
// Expert-sorted copy of the hidden rows; with `xs` also the deferred-scale
// token sums [H/128 stages][4 parts][cap]. It also zeroes the `zero_n` 32-bit
// words at each `zero_ptr` (token-sum parts of a stage half with no K
// elements, the gate/up GEMM's split arrival counters, the down GEMM's atomic
// accumulator).
cudaError_t launch_gather(const void* hidden, const int32_t* ids, const int32_t* slot_of_pair, int P,
                          int topk, int E, int H, int permute, int act_dtype, int max_ctas, void* x_sorted,
                          float* xs, int cap, float* zero_ptr0, int zero_n0, float* zero_ptr1, int zero_n1,
                          float* zero_ptr2, int zero_n2, float* zero_ptr3, int zero_n3, cudaStream_t stream,
                          bool pdl);
// the gather for act-order gate/up weights: x_sorted rows in each expert's K order kperm [E, H]
cudaError_t launch_gather_perm(const void* hidden, const int32_t* ids, const int32_t* slot_of_pair,
                               const int32_t* kperm, int P, int topk, int E, int H, int permute, int max_ctas,
                               void* x_sorted, cudaStream_t stream, bool pdl);
// argument checks of wna16_topk_routing, without any CUDA call
wna16_status routing_check(const void* logits, wna16_dtype logits_dtype, int64_t M, int E, int topk,
                           wna16_scoring scoring, int n_groups, int topk_groups, const int32_t* topk_ids,
                           const float* topk_weights);
// summed != 0: `slab` is the down GEMM's [M, H] fp32 atomic accumulator (round only)
cudaError_t launch_combine(const float* slab, const int32_t* ids, int M, int H, int topk, int E,
                           int split, int summed, int act_dtype, void* out, cudaStream_t stream, bool pdl);

}  // namespace wna16
