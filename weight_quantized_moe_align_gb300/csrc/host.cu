// C ABI of the fused weight-quantized MoE layer: argument checks, workspace
// layout, block/split heuristics, TMA descriptors and the launch sequence
// align -> gate/up GEMM -> down GEMM -> combine (all on the caller's stream,
// no host synchronization, no allocation).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>

#include "wna16_moe.h"
#include "common.cuh"
#include "gemm_launch.cuh"
#include "layer_plan.h"

using namespace wna16;

namespace {

bool is_pow2(long long v) { return v > 0 && (v & (v - 1)) == 0; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  static int cache[64] = {};
  if (dev >= 0 && dev < 64 && cache[dev]) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Encodes a described tiled map (see layer_plan.h).
bool encode_map(CUtensorMap* m, const MapDesc& d) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3], st[2];
  cuuint32_t box[3], es[3] = {1, 1, 1};
  for (int i = 0; i < d.rank; ++i) {
    dims[i] = d.dims[i];
    box[i] = d.box[i];
  }
  for (int i = 0; i + 1 < d.rank; ++i) st[i] = d.strides[i];
  return fn(m, d.dt, d.rank, const_cast<void*>(d.base), dims, st, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, d.swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct EncodedMaps {
  CUtensorMap q, s, z, b, x;
};

bool encode_maps(EncodedMaps* e, const GemmMaps& g, bool weights) {
  std::memset(e, 0, sizeof(*e));
  if (weights && (!encode_map(&e->q, g.q) || !encode_map(&e->s, g.s) || (g.has_z && !encode_map(&e->z, g.z))))
    return false;
  if (!encode_map(&e->b, g.b)) return false;
  return !g.has_x || encode_map(&e->x, g.x);
}

cudaError_t launch_gemm(int bits, int act, int scl, int gemm, int lean, dim3 grid, size_t smem, cudaStream_t st,
                        const EncodedMaps& m, const GemmArgs& a) {
  return bits == 4 ? launch_gemm_w4(act, scl, gemm, lean, grid, smem, st, m.q, m.s, m.z, m.b, a)
                   : launch_gemm_w8(act, scl, gemm, lean, grid, smem, st, m.q, m.s, m.z, m.b, a);
}

}  // namespace

extern "C" {

int64_t wna16_align_capacity(int64_t num_pairs, int E, int block) {
  if (num_pairs < 0 || E < 1 || block < 1) return -1;
  return capacity(num_pairs, E, block);
}

int wna16_choose_block(int64_t M, int topk, int E) { return choose_block_impl(M, topk, E); }

wna16_status wna16_moe_align_block_size(const int32_t* topk_ids, int64_t M, int topk, int E, int block,
                                        int32_t* sorted_ids, int32_t* expert_ids,
                                        int32_t* num_tokens_post_padded, int32_t* expert_counts,
                                        int32_t* device_status, void* stream) {
  if (M < 0 || topk < 1 || E < 1) return WNA16_ERR_INVALID_ARG;
  if (E > 256) return WNA16_ERR_UNSUPPORTED;
  if (!is_pow2(block) || block < 16 || block > 256) return WNA16_ERR_INVALID_ARG;
  const int64_t P = M * topk;
  if (P >= (int64_t(1) << 31)) return WNA16_ERR_UNSUPPORTED;
  if ((P > 0 && !topk_ids) || !sorted_ids || !expert_ids || !num_tokens_post_padded)
    return WNA16_ERR_INVALID_ARG;
  const int64_t cap = capacity(P, E, block);
  if (launch_align(topk_ids, static_cast<int>(P), E, block, static_cast<int>(cap), sorted_ids, expert_ids,
                   num_tokens_post_padded, expert_counts, device_status, nullptr, nullptr,
                   static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return WNA16_ERR_CUDA;
  return WNA16_OK;
}

size_t wna16_fused_moe_workspace_bytes(int64_t M, int64_t H, int64_t I, int E, int topk, int bits,
                                       int group_size, int block, int split_k) {
  Resolved r;
  if (resolve(M, H, I, E, topk, bits, group_size, block, split_k, sm_count(), &r) != WNA16_OK) return 0;
  return ws_layout(M, H, I, E, topk, r.block, r.split, r.split1).total;
}

}  // extern "C"

namespace {

// The fused layer on either weight form: the plain layout (w13_q, ...,
// w2_zeros, read by TMA boxes) or prepacked stage images (w13_pack, w2_pack,
// one bulk copy per stage; the plain pointers are then unused).
wna16_status run_layer(const void* hidden, wna16_dtype act_dtype, int64_t M, int64_t H, int64_t I, int E,
                       int topk, const int32_t* w13_q, const void* w13_scales, const int32_t* w13_zeros,
                       const int32_t* w2_q, const void* w2_scales, const int32_t* w2_zeros,
                       const void* w13_pack, const void* w2_pack, int pack_zeros, wna16_dtype scale_dtype,
                       int bits, int group_size, const int32_t* topk_ids, const float* topk_weights, void* out,
                       void* workspace, size_t workspace_bytes, int block, int split_k, void* stream,
                       void* const* events, const wna16_moe_options* opt,
                       const EncodedMaps* weight_maps = nullptr) {
  if (act_dtype != WNA16_F16 && act_dtype != WNA16_BF16) return WNA16_ERR_INVALID_ARG;
  if (opt) {
    if (opt->activation != WNA16_ACT_SILU && opt->activation != WNA16_ACT_SWIGLU_CLAMP) return WNA16_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(opt->w13_bias) & 1u) || (reinterpret_cast<uintptr_t>(opt->w2_bias) & 1u))
      return WNA16_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(opt->w13_perm) & 3u) || (reinterpret_cast<uintptr_t>(opt->w2_inv_perm) & 3u))
      return WNA16_ERR_INVALID_ARG;
    if (opt->activation == WNA16_ACT_SWIGLU_CLAMP &&
        (!std::isfinite(opt->swiglu_alpha) || !std::isfinite(opt->swiglu_beta) || std::isnan(opt->swiglu_limit)))
      return WNA16_ERR_INVALID_ARG;
  }
  if (scale_dtype != WNA16_F16 && scale_dtype != WNA16_BF16) return WNA16_ERR_INVALID_ARG;
  if (opt && opt->atomic_reduce && (opt->w13_perm || opt->w2_inv_perm)) return WNA16_ERR_INVALID_ARG;
  if (M * H >= (int64_t(1) << 31)) return WNA16_ERR_UNSUPPORTED;
  Resolved r;
  const int sms = sm_count();
  const wna16_status st = resolve(M, H, I, E, topk, bits, group_size, block, split_k, sms, &r);
  if (st != WNA16_OK) return st;
  if (M == 0) return WNA16_OK;
  // routing on the device first: the layer runs on the ids and weights it writes
  const bool routed = opt && opt->router_logits;
  if (routed) {
    const wna16_status rs = routing_check(opt->router_logits, opt->logits_dtype, M, E, topk, opt->scoring,
                                          opt->n_groups, opt->topk_groups, opt->routed_ids, opt->routed_weights);
    if (rs != WNA16_OK) return rs;
    topk_ids = opt->routed_ids;
    topk_weights = opt->routed_weights;
  }
  const bool packed = w13_pack != nullptr || w2_pack != nullptr;
  if (!hidden || !topk_ids || !topk_weights || !out || !workspace) return WNA16_ERR_INVALID_ARG;
  if (packed) {
    if (!w13_pack || !w2_pack || !aligned16(w13_pack) || !aligned16(w2_pack)) return WNA16_ERR_INVALID_ARG;
  } else {
    if (!w13_q || !w13_scales || !w2_q || !w2_scales) return WNA16_ERR_INVALID_ARG;
    if ((w13_zeros == nullptr) != (w2_zeros == nullptr)) return WNA16_ERR_INVALID_ARG;
  }
  const void* ptrs[] = {hidden, w13_q, w13_scales, w13_zeros, w2_q, w2_scales, w2_zeros, out, workspace};
  for (const void* p : ptrs)
    if (p && !aligned16(p)) return WNA16_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(topk_ids) & 3u) || (reinterpret_cast<uintptr_t>(topk_weights) & 3u))
    return WNA16_ERR_INVALID_ARG;
  LayerPlan plan;
  const wna16_status ps =
      plan_layer(act_dtype, M, H, I, E, topk, w13_q, w13_scales, w13_zeros, w2_q, w2_scales, w2_zeros, w13_pack,
                 w2_pack, pack_zeros, scale_dtype, bits, group_size, topk_weights, workspace, workspace_bytes, block,
                 split_k, events != nullptr, opt, sms, &plan);
  if (ps != WNA16_OK) return ps;
  const LayerPlan& p = plan;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* status = reinterpret_cast<int32_t*>(ws + p.L.status);
  int32_t* sorted = reinterpret_cast<int32_t*>(ws + p.L.sorted);
  int32_t* experts = reinterpret_cast<int32_t*>(ws + p.L.experts);
  int32_t* npp = reinterpret_cast<int32_t*>(ws + p.L.npp);
  int32_t* counts = reinterpret_cast<int32_t*>(ws + p.L.counts);
  int32_t* slot_of_pair = reinterpret_cast<int32_t*>(ws + p.L.slot_of_pair);
  void* x_sorted = ws + p.L.x_sorted;
  float* ws_words = reinterpret_cast<float*>(ws);
  auto mark = [&](int i) {
    if (events && events[i]) return cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s) == cudaSuccess;
    return true;
  };
  // weight maps: encoded once by a plan (wna16_plan_create), else here
  EncodedMaps m1, m2;
  const bool fresh = weight_maps == nullptr;
  if (!encode_maps(&m1, p.m1, !packed && fresh) || !encode_maps(&m2, p.m2, !packed && fresh)) return WNA16_ERR_CUDA;
  if (!fresh) {
    m1.q = weight_maps[0].q, m1.s = weight_maps[0].s, m1.z = weight_maps[0].z;
    m2.q = weight_maps[1].q, m2.s = weight_maps[1].s, m2.z = weight_maps[1].z;
  }

  int32_t* block_rows = reinterpret_cast<int32_t*>(ws + p.L.block_rows);
  if (routed && M <= kRouteAlignRows) {
    // a small batch is routed and aligned by one launch
    if (!mark(0) || launch_route_align(opt->router_logits, opt->logits_dtype, static_cast<int>(M), E, topk,
                                       opt->scoring == WNA16_SCORE_SIGMOID ? 1 : 0, opt->renormalize ? 1 : 0,
                                       opt->n_groups, opt->topk_groups, opt->routed_ids, opt->routed_weights, p.B,
                                       static_cast<int>(p.cap), sorted, experts, npp, counts, status, slot_of_pair,
                                       block_rows, s) != cudaSuccess)
      return WNA16_ERR_CUDA;
  } else {
    if (routed) {
      // its own argument checks ran above; its launch is the first of this call
      const wna16_status rs = wna16_topk_routing(opt->router_logits, opt->logits_dtype, M, E, topk, opt->scoring,
                                                 opt->renormalize, opt->n_groups, opt->topk_groups, opt->routed_ids,
                                                 opt->routed_weights, stream);
      if (rs != WNA16_OK) return rs;
    }
    if (!mark(0) || launch_align(topk_ids, p.P, E, p.B, static_cast<int>(p.cap), sorted, experts, npp, counts,
                                 status, slot_of_pair, block_rows, s) != cudaSuccess)
      return WNA16_ERR_CUDA;
  }
  float* zero1 = p.zero1_n ? ws_words + p.zero1_off : nullptr;
  float* zero2 = p.zero2_n ? ws_words + p.zero2_off : nullptr;
  float* cnt1 = p.cnt1_n ? ws_words + p.cnt1_off : nullptr;
  if (opt && opt->w13_perm) {
    if (!mark(1) || launch_gather_perm(hidden, topk_ids, slot_of_pair, opt->w13_perm, p.P, topk, E,
                                       static_cast<int>(H), bits == 4 ? 1 : 0, p.gather_ctas, x_sorted, s,
                                       p.pdl) != cudaSuccess)
      return WNA16_ERR_CUDA;
  } else if (!mark(1) || launch_gather(hidden, topk_ids, slot_of_pair, p.P, topk, E, static_cast<int>(H),
                                       bits == 4 ? 1 : 0, act_dtype, p.gather_ctas, x_sorted,
                                       p.defer ? ws_words + p.L.xs1 / 4 : nullptr, static_cast<int>(p.cap), zero1,
                                       p.zero1_n, zero2, p.zero2_n, cnt1, p.cnt1_n,
                                       p.acc_n ? ws_words + p.acc_off : nullptr, p.acc_n, s, p.pdl) != cudaSuccess) {
    return WNA16_ERR_CUDA;
  }

  if (!mark(2)) return WNA16_ERR_CUDA;
  const cudaError_t e1 =
      p.defer ? launch_gemm_defer(bits, act_dtype, scale_dtype, 1, dim3(p.grid1), p.smem1, s, m1.q, m1.s, m1.z, m1.b,
                                  m1.x, p.a1)
              : launch_gemm(bits, act_dtype, scale_dtype, 1, p.pipe.lean, dim3(p.grid1), p.smem1, s, m1, p.a1);
  if (e1 != cudaSuccess) return WNA16_ERR_CUDA;
  if (!mark(3)) return WNA16_ERR_CUDA;
  const cudaError_t e2 =
      p.defer ? launch_gemm_defer(bits, act_dtype, scale_dtype, 2, dim3(p.grid2), p.smem2, s, m2.q, m2.s, m2.z, m2.b,
                                  m2.x, p.a2)
              : launch_gemm(bits, act_dtype, scale_dtype, 2, p.pipe.lean, dim3(p.grid2), p.smem2, s, m2, p.a2);
  if (e2 != cudaSuccess) return WNA16_ERR_CUDA;

  if (!mark(4) || launch_combine(reinterpret_cast<const float*>(ws + p.L.slab), topk_ids, static_cast<int>(M),
                                 static_cast<int>(H), topk, E, p.r.split, p.atomic ? 1 : 0, act_dtype, out, s,
                                 p.pdl) != cudaSuccess)
    return WNA16_ERR_CUDA;
  if (!mark(5)) return WNA16_ERR_CUDA;
  return WNA16_OK;
}

}  // namespace

extern "C" {

wna16_status wna16_fused_moe_timed(const void* hidden, wna16_dtype act_dtype, int64_t M, int64_t H,
                                   int64_t I, int E, int topk, const int32_t* w13_q,
                                   const void* w13_scales, const int32_t* w13_zeros, const int32_t* w2_q,
                                   const void* w2_scales, const int32_t* w2_zeros,
                                   wna16_dtype scale_dtype, int bits, int group_size,
                                   const int32_t* topk_ids, const float* topk_weights, void* out,
                                   void* workspace, size_t workspace_bytes, int block, int split_k,
                                   void* stream, void* const* events) {
  return run_layer(hidden, act_dtype, M, H, I, E, topk, w13_q, w13_scales, w13_zeros, w2_q, w2_scales, w2_zeros,
                   nullptr, nullptr, 0, scale_dtype, bits, group_size, topk_ids, topk_weights, out, workspace,
                   workspace_bytes, block, split_k, stream, events, nullptr);
}

wna16_status wna16_fused_moe_prepacked(const void* hidden, wna16_dtype act_dtype, int64_t M, int64_t H,
                                       int64_t I, int E, int topk, const void* w13_packed, const void* w2_packed,
                                       int has_zeros, wna16_dtype scale_dtype, int bits, int group_size,
                                       const int32_t* topk_ids, const float* topk_weights, void* out,
                                       void* workspace, size_t workspace_bytes, int block, int split_k,
                                       void* stream, void* const* events) {
  if (!w13_packed || !w2_packed) return WNA16_ERR_INVALID_ARG;
  return run_layer(hidden, act_dtype, M, H, I, E, topk, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                   w13_packed, w2_packed, has_zeros, scale_dtype, bits, group_size, topk_ids, topk_weights, out,
                   workspace, workspace_bytes, block, split_k, stream, events, nullptr);
}

wna16_status wna16_fused_moe_ex(const void* hidden, wna16_dtype act_dtype, int64_t M, int64_t H, int64_t I,
                                int E, int topk, const int32_t* w13_q, const void* w13_scales,
                                const int32_t* w13_zeros, const int32_t* w2_q, const void* w2_scales,
                                const int32_t* w2_zeros, wna16_dtype scale_dtype, int bits, int group_size,
                                const int32_t* topk_ids, const float* topk_weights, void* out, void* workspace,
                                size_t workspace_bytes, int block, int split_k, void* stream,
                                void* const* events, const wna16_moe_options* options) {
  return run_layer(hidden, act_dtype, M, H, I, E, topk, w13_q, w13_scales, w13_zeros, w2_q, w2_scales, w2_zeros,
                   nullptr, nullptr, 0, scale_dtype, bits, group_size, topk_ids, topk_weights, out, workspace,
                   workspace_bytes, block, split_k, stream, events, options);
}

wna16_status wna16_fused_moe_prepacked_ex(const void* hidden, wna16_dtype act_dtype, int64_t M, int64_t H,
                                          int64_t I, int E, int topk, const void* w13_packed,
                                          const void* w2_packed, int has_zeros, wna16_dtype scale_dtype, int bits,
                                          int group_size, const int32_t* topk_ids, const float* topk_weights,
                                          void* out, void* workspace, size_t workspace_bytes, int block,
                                          int split_k, void* stream, void* const* events,
                                          const wna16_moe_options* options) {
  if (!w13_packed || !w2_packed) return WNA16_ERR_INVALID_ARG;
  return run_layer(hidden, act_dtype, M, H, I, E, topk, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                   w13_packed, w2_packed, has_zeros, scale_dtype, bits, group_size, topk_ids, topk_weights, out,
                   workspace, workspace_bytes, block, split_k, stream, events, options);
}

wna16_status wna16_fused_moe(const void* hidden, wna16_dtype act_dtype, int64_t M, int64_t H, int64_t I,
                             int E, int topk, const int32_t* w13_q, const void* w13_scales,
                             const int32_t* w13_zeros, const int32_t* w2_q, const void* w2_scales,
                             const int32_t* w2_zeros, wna16_dtype scale_dtype, int bits, int group_size,
                             const int32_t* topk_ids, const float* topk_weights, void* out,
                             void* workspace, size_t workspace_bytes, int block, int split_k,
                             void* stream) {
  return wna16_fused_moe_timed(hidden, act_dtype, M, H, I, E, topk, w13_q, w13_scales, w13_zeros, w2_q,
                               w2_scales, w2_zeros, scale_dtype, bits, group_size, topk_ids, topk_weights,
                               out, workspace, workspace_bytes, block, split_k, stream, nullptr);
}

}  // extern "C"

struct wna16_plan_t {
  wna16_dtype act_dtype, scale_dtype;
  int64_t H, I;
  int E, topk, bits, group_size;
  const int32_t *w13_q, *w13_zeros, *w2_q, *w2_zeros;
  const void *w13_scales, *w2_scales;
  EncodedMaps maps[2];  // weight maps of the gate/up and down projections
};

extern "C" {

wna16_status wna16_plan_create(wna16_dtype act_dtype, int64_t H, int64_t I, int E, int topk, const int32_t* w13_q,
                               const void* w13_scales, const int32_t* w13_zeros, const int32_t* w2_q,
                               const void* w2_scales, const int32_t* w2_zeros, wna16_dtype scale_dtype, int bits,
                               int group_size, wna16_plan_t** plan) {
  if (!plan) return WNA16_ERR_INVALID_ARG;
  *plan = nullptr;
  if (act_dtype != WNA16_F16 && act_dtype != WNA16_BF16) return WNA16_ERR_INVALID_ARG;
  if (scale_dtype != WNA16_F16 && scale_dtype != WNA16_BF16) return WNA16_ERR_INVALID_ARG;
  if (!w13_q || !w13_scales || !w2_q || !w2_scales) return WNA16_ERR_INVALID_ARG;
  if ((w13_zeros == nullptr) != (w2_zeros == nullptr)) return WNA16_ERR_INVALID_ARG;
  const void* ptrs[] = {w13_q, w13_scales, w13_zeros, w2_q, w2_scales, w2_zeros};
  for (const void* q : ptrs)
    if (q && !aligned16(q)) return WNA16_ERR_INVALID_ARG;
  // the weight maps do not depend on the batch: plan a one-token call with a
  // stand-in workspace to describe them
  LayerPlan lp;
  uint8_t* const stand_in = reinterpret_cast<uint8_t*>(uintptr_t(1) << 40);
  const wna16_status st = plan_layer(act_dtype, 1, H, I, E, topk, w13_q, w13_scales, w13_zeros, w2_q, w2_scales,
                                     w2_zeros, nullptr, nullptr, 0, scale_dtype, bits, group_size, nullptr, stand_in,
                                     ~size_t(0) >> 2, 0, 0, false, nullptr, sm_count(), &lp);
  if (st != WNA16_OK) return st;
  wna16_plan_t* p = new (std::nothrow) wna16_plan_t();
  if (!p) return WNA16_ERR_UNSUPPORTED;
  p->act_dtype = act_dtype;
  p->scale_dtype = scale_dtype;
  p->H = H;
  p->I = I;
  p->E = E;
  p->topk = topk;
  p->bits = bits;
  p->group_size = group_size;
  p->w13_q = w13_q;
  p->w13_scales = w13_scales;
  p->w13_zeros = w13_zeros;
  p->w2_q = w2_q;
  p->w2_scales = w2_scales;
  p->w2_zeros = w2_zeros;
  std::memset(p->maps, 0, sizeof(p->maps));
  if (!encode_map(&p->maps[0].q, lp.m1.q) || !encode_map(&p->maps[0].s, lp.m1.s) ||
      (lp.m1.has_z && !encode_map(&p->maps[0].z, lp.m1.z)) || !encode_map(&p->maps[1].q, lp.m2.q) ||
      !encode_map(&p->maps[1].s, lp.m2.s) || (lp.m2.has_z && !encode_map(&p->maps[1].z, lp.m2.z))) {
    delete p;
    return WNA16_ERR_CUDA;
  }
  *plan = p;
  return WNA16_OK;
}

void wna16_plan_destroy(wna16_plan_t* plan) { delete plan; }

wna16_status wna16_fused_moe_plan(const wna16_plan_t* plan, const void* hidden, int64_t M, const int32_t* topk_ids,
                                  const float* topk_weights, void* out, void* workspace, size_t workspace_bytes,
                                  int block, int split_k, void* stream) {
  if (!plan) return WNA16_ERR_INVALID_ARG;
  const wna16_plan_t& p = *plan;
  return run_layer(hidden, p.act_dtype, M, p.H, p.I, p.E, p.topk, p.w13_q, p.w13_scales, p.w13_zeros, p.w2_q,
                   p.w2_scales, p.w2_zeros, nullptr, nullptr, 0, p.scale_dtype, p.bits, p.group_size, topk_ids,
                   topk_weights, out, workspace, workspace_bytes, block, split_k, stream, nullptr, nullptr, p.maps);
}

wna16_status wna16_read_device_status(const void* status_word, int32_t* bits_out, void* stream) {
  if (!status_word) return WNA16_ERR_INVALID_ARG;
  int32_t v = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&v, status_word, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess) return WNA16_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return WNA16_ERR_CUDA;
  if (bits_out) *bits_out = v;
  if (v & WNA16_DEV_TIMEOUT) return WNA16_ERR_DEVICE_TIMEOUT;
  if (v & WNA16_DEV_BAD_EXPERT_ID) return WNA16_ERR_DEVICE_BAD_EXPERT_ID;
  if (v & WNA16_DEV_BAD_GROUPS) return WNA16_ERR_DEVICE_BAD_GROUPS;
  return WNA16_OK;
}

const char* wna16_status_string(wna16_status status) {
  switch (status) {
    case WNA16_OK: return "ok";
    case WNA16_ERR_INVALID_ARG: return "invalid argument";
    case WNA16_ERR_UNSUPPORTED: return "unsupported shape or format";
    case WNA16_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case WNA16_ERR_CUDA: return "CUDA call failed";
    case WNA16_ERR_DEVICE_BAD_EXPERT_ID: return "device: expert id out of range (pair dropped)";
    case WNA16_ERR_DEVICE_TIMEOUT: return "device: pipeline wait timed out";
    case WNA16_ERR_DEVICE_BAD_GROUPS: return "device: act-order g_idx is not a split into groups of G";
  }
  return "unknown status";
}

}  // extern "C"
