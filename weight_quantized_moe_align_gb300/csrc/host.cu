// C ABI of the fused weight-quantized MoE layer: argument checks, workspace
// layout, block/split heuristics, TMA descriptors and the launch sequence
// align -> gate/up GEMM -> down GEMM -> combine (all on the caller's stream,
// no host synchronization, no allocation).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "wna16_moe.h"
#include "common.cuh"
#include "gemm_launch.cuh"

using namespace wna16;

namespace {

constexpr int kMaxSmem = 232448;   // opt-in dynamic shared memory per CTA on sm_103a
constexpr int kHalfSmem = 112 * 1024;  // two CTAs per SM
constexpr int kQuarterSmem = 55 * 1024;  // four CTAs per SM
constexpr int kMinSmem = 120 * 1024;   // a whole-SM CTA (512 TMEM columns) runs alone on its SM

bool is_pow2(long long v) { return v > 0 && (v & (v - 1)) == 0; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

int64_t capacity(int64_t P, int E, int block) {
  const int64_t raw = P + std::min<int64_t>(P, E) * (block - 1);
  return (raw + block - 1) / block * block;
}

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

int choose_block_impl(int64_t M, int topk, int E) {
  const int64_t P = M * topk;
  if (P <= 0) return 16;
  const int64_t active = std::min<int64_t>(P, E);
  const double avg = static_cast<double>(P) / static_cast<double>(active);  // pairs per active expert
  if (avg <= 64.0) {
    // Weight streaming dominates: every token block of an expert streams the
    // expert's whole weights once. Pick the tile with the fewest streaming
    // passes times the cost of one pass, measured on GB300 (Mixtral-8x7B
    // gate/up): 16-token tiles 1.0, 32-token 1.28 (both the deferred-scale
    // kernel), 64-token 1.34. Expert loads are uneven, so a block count of
    // ceil(1.3 * avg / tile) is assumed.
    const int tiles[3] = {16, 32, 64};
    const double cost[3] = {1.0, 1.28, 1.34};
    int best = 16;
    double best_cost = 1e30;
    for (int i = 0; i < 3; ++i) {
      const double passes = std::ceil(1.3 * avg / tiles[i]);
      if (passes * cost[i] < best_cost - 1e-9) {
        best_cost = passes * cost[i];
        best = tiles[i];
      }
    }
    return best;
  }
  // Larger batches are tensor-bound: the smallest power of two covering the
  // average, up to 128.
  int b = 64;
  while (b < 128 && b < avg) b <<= 1;
  return b;
}

// Pipeline shape of one GEMM launch for a token tile of `block`.
//  * lean layout (when selected): four CTAs per SM (128 TMEM columns: one
//    accumulator and one A slot; <= 55 KB of shared memory each), four
//    MMA-issuing threads sharing the tensor core.
//  * tiles up to 64: two CTAs per SM of the full layout (256 TMEM columns,
//    <= 112 KB of shared memory).
//  * larger tiles: one CTA per SM.
struct Pipe {
  int stages, aslots, acc, ctas_per_sm, lean;
  uint32_t tmem_cols;
  size_t smem;
};

Pipe pipe_for(int bits, int block) {
  Pipe p;
  // The lean layout (LEAN = 1) is built and selectable here; measured on
  // Mixtral-8x7B decode it was slower than two full-layout CTAs per SM (its
  // single A slot serialises dequant and MMA inside each CTA), so it is off.
  p.lean = 0;
  const bool half_sm = !p.lean && block <= 64;
  p.ctas_per_sm = p.lean ? 4 : (half_sm ? 2 : 1);
  p.tmem_cols = p.lean ? 128 : (half_sm ? 256 : 512);
  const int smem_cap = p.lean ? kQuarterSmem : (half_sm ? kHalfSmem : kMaxSmem);
  p.acc = p.lean ? 1 : ((2 * block + 2 * kASlotCols <= static_cast<int>(p.tmem_cols)) ? 2 : 1);
  p.stages = kMaxStages;
  while (p.stages > 2 && gemm_smem_bytes(bits, block, p.stages) > smem_cap) --p.stages;
  p.aslots = std::min({kMaxASlots, (static_cast<int>(p.tmem_cols) - p.acc * block) / kASlotCols, p.stages - 1});
  p.smem = gemm_smem_bytes(bits, block, p.stages);
  if (p.ctas_per_sm == 1) p.smem = std::max<size_t>(p.smem, kMinSmem);
  return p;
}

// Stages of the deferred-scale kernel (two CTAs per SM).
int defer_stages(int bits, int gemm, int nt) {
  int st = kMaxStages;
  while (st > 2 && defer_smem_bytes(bits, gemm, nt, st) > kHalfSmem) --st;
  return st;
}

// Token blocks per panel of the GEMM work-unit order: as many as keep their
// token rows (block x K x 2 bytes) within about a third of the L2.
int panel_blocks(int block, int64_t K, int max_blocks) {
  const int64_t budget = 48ll << 20;
  const int64_t per_block = static_cast<int64_t>(block) * K * 2;
  const int64_t p = std::max<int64_t>(1, budget / std::max<int64_t>(per_block, 1));
  return static_cast<int>(std::min<int64_t>(p, std::max(max_blocks, 1)));
}

// Expected token blocks of a batch (the host does not see the routing): the
// active experts times the blocks an expert of average load needs. The
// capacity bound would overcount the padding.
int64_t expected_blocks(int64_t M, int topk, int E, int block) {
  const int64_t P = M * topk;
  if (P <= 0) return 0;
  const int64_t active = std::min<int64_t>(P, E);
  const int64_t avg = (P + active - 1) / active;
  return active * ((avg + block - 1) / block);
}

// K split of a GEMM launch: only when the units do not fill the persistent CTA
// slots, then as many splits as fit (at most 8, keeping >= 8 K stages per
// split). Finer splits that merely even out the rounds were measured slower:
// every unit boundary stalls the dequant chain (accumulator handoff, epilogue,
// and for the gate/up GEMM the partial-sum exchange).
int choose_split(int64_t units, int kt_total, int ctas_per_sm) {
  const int64_t slots = static_cast<int64_t>(sm_count()) * ctas_per_sm;
  if (units >= slots) return 1;
  int s = static_cast<int>(slots / std::max<int64_t>(units, 1));
  s = std::min(s, 8);
  s = std::min(s, std::max(1, kt_total / 8));
  return std::max(s, 1);
}

struct WsLayout {
  size_t status, sorted, experts, npp, counts, slot_of_pair, x_sorted, act, slab, xs1, xs2, part1, cnt1, total;
};

WsLayout ws_layout(int64_t M, int64_t H, int64_t I, int E, int topk, int block, int split, int split1) {
  const int64_t P = M * topk;
  const int64_t cap = capacity(P, E, block);
  WsLayout w;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t r = o;
    o = align_up(o + bytes, 256);
    return r;
  };
  w.status = take(4);
  w.sorted = take(static_cast<size_t>(cap) * 4);
  w.experts = take(static_cast<size_t>(cap / block) * 4);
  w.npp = take(4);
  w.counts = take(static_cast<size_t>(E) * 4);
  w.slot_of_pair = take(static_cast<size_t>(P) * 4);
  w.x_sorted = take(static_cast<size_t>(cap) * H * 2);
  w.act = take(static_cast<size_t>(cap) * I * 2);
  w.slab = take(static_cast<size_t>(split) * P * H * 4);
  // token sums of the deferred-scale GEMMs (16-token tiles only):
  // [H/128 stages][4][cap] and [I/128 stages][16][cap] floats
  const size_t kt1 = static_cast<size_t>((H + kTileK - 1) / kTileK);
  const size_t kt2 = static_cast<size_t>((I + kTileK - 1) / kTileK);
  const bool defer = defer_tile(block);
  w.xs1 = take(defer ? kt1 * defer_xs_parts(1) * cap * 4 : 0);
  w.xs2 = take(defer ? kt2 * defer_xs_parts(2) * cap * 4 : 0);
  // K-split partial sums of the deferred-scale gate/up GEMM and their arrival
  // counters: [I/64 tiles][cap/block][split1][128][block] floats, [I/64][cap/block][4] ints
  const size_t tiles1 = static_cast<size_t>(I / kGateUpRows), blocks = static_cast<size_t>(cap / block);
  w.part1 = take(split1 > 1 ? tiles1 * blocks * split1 * kTileRows * block * 4 : 0);
  w.cnt1 = take(split1 > 1 ? tiles1 * blocks * 4 * 4 : 0);
  w.total = o;
  return w;
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

// Tiled map of rank 2 or 3: dims[0] innermost (elements), strides in bytes of
// dims 1.. (dims[0] is contiguous).
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, int rank, const uint64_t* dims,
              const uint64_t* strides, const uint32_t* box,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_NONE) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[3], st[2];
  cuuint32_t b[3], es[3] = {1, 1, 1};
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
  }
  for (int i = 0; i + 1 < rank; ++i) st[i] = strides[i];
  return fn(m, dt, rank, const_cast<void*>(base), d, st, b, es, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct GemmMaps {
  CUtensorMap q, s, z, b;
};

// Maps of one projection, one box per stage each:
//   gate/up (rows = 2I): codes [E*2 halves, I, K/pf] box {128/pf, 64, 2} (gate rows
//   then the matching up rows), scales [E*K/G, 2, I] box {64, 2, SG}, zeros
//   [E*K/G, 2, I/pf] box {64/pf, 2, SG};
//   down (rows = H): codes [E*H, K/pf] box {128/pf, 128}, scales [E*K/G, H] box
//   {128, SG}, zeros [E*K/G, H/pf] box {128/pf, SG}.
bool make_gemm_maps(GemmMaps* g, const int32_t* q, const void* s, const int32_t* z, int E, int64_t N,
                    int64_t K, int G, int bits, bool gate_up) {
  const int pf = 32 / bits;
  const uint64_t groups = K / G;
  const uint32_t sg = G < kTileK ? kTileK / G : 1;
  const uint32_t kw = kTileK / pf;
  // Code rows of a stage are 64 B (int4) or 128 B (int8): swizzled so that the
  // dequant warps' 16-byte reads of 8 consecutive rows hit distinct banks.
  const CUtensorMapSwizzle qswz = bits == 4 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  std::memset(g, 0, sizeof(*g));
  if (gate_up) {
    const uint64_t I = N / 2;
    const uint64_t qd[3] = {static_cast<uint64_t>(K / pf), I, 2ull * E};
    const uint64_t qs[2] = {static_cast<uint64_t>(K / pf) * 4, I * (K / pf) * 4};
    const uint32_t qb[3] = {kw, kGateUpRows, 2};
    if (!make_map(&g->q, CU_TENSOR_MAP_DATA_TYPE_INT32, q, 3, qd, qs, qb, qswz)) return false;
    const uint64_t sd[3] = {I, 2, E * groups};
    const uint64_t ss[2] = {I * 2, 2 * I * 2};
    const uint32_t sb[3] = {kGateUpRows, 2, sg};
    if (!make_map(&g->s, CU_TENSOR_MAP_DATA_TYPE_UINT16, s, 3, sd, ss, sb)) return false;
    if (z) {
      const uint64_t zd[3] = {I / pf, 2, E * groups};
      const uint64_t zs[2] = {(I / pf) * 4, 2 * (I / pf) * 4};
      const uint32_t zb[3] = {static_cast<uint32_t>(kGateUpRows / pf), 2, sg};
      if (!make_map(&g->z, CU_TENSOR_MAP_DATA_TYPE_INT32, z, 3, zd, zs, zb)) return false;
    }
  } else {
    const uint64_t qd[2] = {static_cast<uint64_t>(K / pf), static_cast<uint64_t>(E) * N};
    const uint64_t qs[1] = {static_cast<uint64_t>(K / pf) * 4};
    const uint32_t qb[2] = {kw, kTileRows};
    if (!make_map(&g->q, CU_TENSOR_MAP_DATA_TYPE_INT32, q, 2, qd, qs, qb, qswz)) return false;
    const uint64_t sd[2] = {static_cast<uint64_t>(N), E * groups};
    const uint64_t ss[1] = {static_cast<uint64_t>(N) * 2};
    const uint32_t sb[2] = {kTileRows, sg};
    if (!make_map(&g->s, CU_TENSOR_MAP_DATA_TYPE_UINT16, s, 2, sd, ss, sb)) return false;
    if (z) {
      const uint64_t zd[2] = {static_cast<uint64_t>(N / pf), E * groups};
      const uint64_t zs[1] = {static_cast<uint64_t>(N / pf) * 4};
      const uint32_t zb[2] = {static_cast<uint32_t>(kTileRows / pf), sg};
      if (!make_map(&g->z, CU_TENSOR_MAP_DATA_TYPE_INT32, z, 2, zd, zs, zb)) return false;
    }
  }
  return true;
}

// Token tile map: rows of a [rows, K] 16-bit matrix, box {64, block} in the
// 128-byte swizzled layout (two boxes per 128-wide stage).
bool make_token_map(CUtensorMap* m, const void* base, int64_t K, int64_t rows, int block) {
  const uint64_t d[2] = {static_cast<uint64_t>(K), static_cast<uint64_t>(rows)};
  const uint64_t st[1] = {static_cast<uint64_t>(K) * 2};
  const uint32_t b[2] = {kChunkK, static_cast<uint32_t>(block)};
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, base, 2, d, st, b, CU_TENSOR_MAP_SWIZZLE_128B);
}

// Token sums of a deferred-scale GEMM: fp32 [stages][parts][rows], box
// {block rows, parts, 1 stage}.
bool make_xs_map(CUtensorMap* m, const float* base, int64_t rows, int parts, int stages, int block) {
  const uint64_t d[3] = {static_cast<uint64_t>(rows), static_cast<uint64_t>(parts), static_cast<uint64_t>(stages)};
  const uint64_t st[2] = {static_cast<uint64_t>(rows) * 4, static_cast<uint64_t>(rows) * parts * 4};
  const uint32_t b[3] = {static_cast<uint32_t>(block), static_cast<uint32_t>(parts), 1};
  return make_map(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, base, 3, d, st, b);
}

cudaError_t launch_gemm(int bits, int act, int scl, int gemm, int lean, dim3 grid, size_t smem, cudaStream_t st,
                        const GemmMaps& m, const GemmArgs& a) {
  return bits == 4 ? launch_gemm_w4(act, scl, gemm, lean, grid, smem, st, m.q, m.s, m.z, m.b, a)
                   : launch_gemm_w8(act, scl, gemm, lean, grid, smem, st, m.q, m.s, m.z, m.b, a);
}

struct Resolved {
  int block, split, split1, G1, G2;
};

wna16_status resolve(int64_t M, int64_t H, int64_t I, int E, int topk, int bits, int group_size,
                     int block, int split_k, Resolved* r) {
  if (M < 0 || H <= 0 || I <= 0 || E < 1 || topk < 1) return WNA16_ERR_INVALID_ARG;
  if (E > 256 || topk > E) return WNA16_ERR_UNSUPPORTED;
  if (bits != 4 && bits != 8) return WNA16_ERR_UNSUPPORTED;
  if (M * topk >= (int64_t(1) << 31)) return WNA16_ERR_UNSUPPORTED;
  if (H % 64 || I % 64) return WNA16_ERR_UNSUPPORTED;
  if (H >= (int64_t(1) << 24) || I >= (int64_t(1) << 24)) return WNA16_ERR_UNSUPPORTED;
  if (group_size == -1) {
    r->G1 = static_cast<int>(H);
    r->G2 = static_cast<int>(I);
  } else {
    // A 128-wide K stage must not straddle two groups: G = 64 (two groups per
    // stage) or a multiple of 128.
    if (group_size <= 0) return WNA16_ERR_INVALID_ARG;
    if ((group_size != 64 && group_size % kTileK) || H % group_size || I % group_size)
      return WNA16_ERR_UNSUPPORTED;
    r->G1 = r->G2 = group_size;
  }
  if (block == 0) block = choose_block_impl(M, topk, E);
  if (!is_pow2(block) || block < 16 || block > 256) return WNA16_ERR_INVALID_ARG;
  r->block = block;
  if (split_k < 0 || split_k > 8) return WNA16_ERR_INVALID_ARG;
  const int kt2 = static_cast<int>((I + kTileK - 1) / kTileK);
  if (split_k == 0) {
    const int64_t units = expected_blocks(M, topk, E, block) * ((H + kTileRows - 1) / kTileRows);
    split_k = choose_split(units, kt2, pipe_for(bits, block).ctas_per_sm);
  }
  r->split = std::min(split_k, kt2);
  // gate/up GEMM: K split only on the deferred-scale path (token tiles of 16 or
  // 32 with groups of >= 128); automatic
  r->split1 = 1;
  const int G1 = r->G1;
  if (defer_tile(block) && G1 >= kTileK && r->G2 >= kTileK) {
    const int kt1 = static_cast<int>((H + kTileK - 1) / kTileK);
    const int64_t units1 = expected_blocks(M, topk, E, block) * (I / kGateUpRows);
    r->split1 = choose_split(units1, kt1, 2);
  }
  return WNA16_OK;
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
                   num_tokens_post_padded, expert_counts, device_status, nullptr,
                   static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return WNA16_ERR_CUDA;
  return WNA16_OK;
}

size_t wna16_fused_moe_workspace_bytes(int64_t M, int64_t H, int64_t I, int E, int topk, int bits,
                                       int group_size, int block, int split_k) {
  Resolved r;
  if (resolve(M, H, I, E, topk, bits, group_size, block, split_k, &r) != WNA16_OK) return 0;
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
                       void* const* events, const wna16_moe_options* opt) {
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
  Resolved r;
  const wna16_status st = resolve(M, H, I, E, topk, bits, group_size, block, split_k, &r);
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
  const WsLayout L = ws_layout(M, H, I, E, topk, r.block, r.split, r.split1);
  if (workspace_bytes < L.total) return WNA16_ERR_WORKSPACE_TOO_SMALL;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* status = reinterpret_cast<int32_t*>(ws + L.status);
  int32_t* sorted = reinterpret_cast<int32_t*>(ws + L.sorted);
  int32_t* experts = reinterpret_cast<int32_t*>(ws + L.experts);
  int32_t* npp = reinterpret_cast<int32_t*>(ws + L.npp);
  int32_t* counts = reinterpret_cast<int32_t*>(ws + L.counts);
  int32_t* slot_of_pair = reinterpret_cast<int32_t*>(ws + L.slot_of_pair);
  void* x_sorted = ws + L.x_sorted;
  void* act = ws + L.act;
  float* slab = reinterpret_cast<float*>(ws + L.slab);

  const int P = static_cast<int>(M * topk);
  const int B = r.block;
  const int64_t cap = capacity(P, E, B);
  const int max_blocks = static_cast<int>(cap / B);
  const bool zeros = packed ? pack_zeros != 0 : w13_zeros != nullptr;
  // 16- and 32-token tiles run the deferred-scale kernel when every stage lies
  // in one group (G >= 128) and the code/activation formats have a
  // magic-number form.
  // Act-order weights run the general kernel: the deferred-scale kernel's
  // token sums assume contiguous feature runs.
  const bool act_order = opt && (opt->w13_perm || opt->w2_inv_perm);
  const bool defer =
      !act_order && defer_tile(B) && r.G1 >= kTileK && r.G2 >= kTileK && defer_supported(bits, act_dtype);
  const int kt1 = static_cast<int>((H + kTileK - 1) / kTileK);
  const int kt2 = static_cast<int>((I + kTileK - 1) / kTileK);
  float* xs1 = defer ? reinterpret_cast<float*>(ws + L.xs1) : nullptr;
  float* xs2 = defer ? reinterpret_cast<float*>(ws + L.xs2) : nullptr;

  // Launches after the first run as programmatic dependents of the previous one
  // (their setup overlaps its tail), except when events are recorded between
  // them for per-kernel timing, and for batches past 8192 routed pairs: on one
  // GB300 the overlap saved 24% of the layer at 2 pairs and 0.6% at 8192, and
  // cost 2% at 16384 (int8 Mixtral-8x22B shapes).
  const bool pdl = events == nullptr && P <= 8192;
  auto mark = [&](int i) {
    if (events && events[i]) return cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s) == cudaSuccess;
    return true;
  };
  GemmMaps m1, m2;
  std::memset(&m1, 0, sizeof(m1));
  std::memset(&m2, 0, sizeof(m2));
  if (!packed &&
      (!make_gemm_maps(&m1, w13_q, w13_scales, zeros ? w13_zeros : nullptr, E, 2 * I, H, r.G1, bits, true) ||
       !make_gemm_maps(&m2, w2_q, w2_scales, zeros ? w2_zeros : nullptr, E, H, I, r.G2, bits, false)))
    return WNA16_ERR_CUDA;
  // Token tiles: `block` expert-sorted rows of 64 elements per stage, in the
  // 128-byte swizzled K-major layout (gathered hidden rows; the act cache).
  if (!make_token_map(&m1.b, x_sorted, H, cap, B) || !make_token_map(&m2.b, act, I, cap, B))
    return WNA16_ERR_CUDA;
  CUtensorMap x1{}, x2{};
  if (defer && (!make_xs_map(&x1, xs1, cap, defer_xs_parts(1), kt1, B) ||
                !make_xs_map(&x2, xs2, cap, defer_xs_parts(2), kt2, B)))
    return WNA16_ERR_CUDA;

  if (routed) {
    // its own argument checks run before its launch, the first of this call
    const wna16_status rs = wna16_topk_routing(opt->router_logits, opt->logits_dtype, M, E, topk, opt->scoring,
                                               opt->renormalize, opt->n_groups, opt->topk_groups, opt->routed_ids,
                                               opt->routed_weights, stream);
    if (rs != WNA16_OK) return rs;
  }
  if (!mark(0) || launch_align(topk_ids, P, E, B, static_cast<int>(cap), sorted, experts, npp, counts, status,
                               slot_of_pair, s) != cudaSuccess)
    return WNA16_ERR_CUDA;
  // Token-sum parts of a stage half that holds no K elements stay zero.
  float* zero1 = nullptr;
  float* zero2 = nullptr;
  int zero1_n = 0, zero2_n = 0;
  if (defer && H % kTileK) {
    zero1 = xs1 + (static_cast<size_t>(kt1 - 1) * 4 + 2) * cap;
    zero1_n = static_cast<int>(2 * cap);
  }
  if (defer && I % kTileK) {
    zero2 = xs2 + (static_cast<size_t>(kt2 - 1) * 16 + 8) * cap;
    zero2_n = static_cast<int>(8 * cap);
  }
  // K split of the deferred-scale gate/up GEMM: its arrival counters start at zero
  const int split1 = defer ? r.split1 : 1;
  float* part1 = split1 > 1 ? reinterpret_cast<float*>(ws + L.part1) : nullptr;
  int* cnt1 = split1 > 1 ? reinterpret_cast<int*>(ws + L.cnt1) : nullptr;
  const int cnt1_n = split1 > 1 ? static_cast<int>((I / kGateUpRows) * max_blocks * 4) : 0;
  if (opt && opt->w13_perm) {
    if (!mark(1) || launch_gather_perm(hidden, topk_ids, slot_of_pair, opt->w13_perm, P, topk, E,
                                       static_cast<int>(H), bits == 4 ? 1 : 0, sm_count() * 8, x_sorted,
                                       s, pdl) != cudaSuccess)
      return WNA16_ERR_CUDA;
  } else if (!mark(1) || launch_gather(hidden, topk_ids, slot_of_pair, P, topk, E, static_cast<int>(H), bits == 4 ? 1 : 0,
                                act_dtype, sm_count() * 8, x_sorted, xs1, static_cast<int>(cap), zero1, zero1_n,
                                zero2, zero2_n, reinterpret_cast<float*>(cnt1), cnt1_n, s, pdl) != cudaSuccess)
    return WNA16_ERR_CUDA;

  const Pipe pipe = pipe_for(bits, B);
  const int sms = sm_count();

  GemmArgs a1{};
  a1.sorted_ids = sorted;
  a1.expert_ids = experts;
  a1.num_post_pad = npp;
  a1.topk_w = topk_weights;
  a1.out = act;
  a1.status = status;
  a1.K = static_cast<int>(H);
  a1.N = static_cast<int>(2 * I);
  a1.I = static_cast<int>(I);
  a1.E = E;
  a1.n_tiles = static_cast<int>(I / kGateUpRows);
  a1.topk = topk;
  a1.P = P;
  a1.block = B;
  a1.groups = static_cast<int>(H / r.G1);
  a1.G = r.G1;
  a1.kt_total = static_cast<int>((H + kTileK - 1) / kTileK);
  a1.split = split1;
  a1.has_zeros = zeros ? 1 : 0;
  a1.max_blocks = max_blocks;
  a1.panel = panel_blocks(B, H, max_blocks);
  a1.num_stages = pipe.stages;
  a1.num_aslots = pipe.aslots;
  a1.num_acc = pipe.acc;
  a1.tmem_cols = pipe.tmem_cols;
  a1.xs_out = xs2;
  a1.cap = static_cast<int>(cap);
  a1.part = part1;
  a1.counters = cnt1;
  a1.bias = opt ? opt->w13_bias : nullptr;
  a1.glu = opt && opt->activation == WNA16_ACT_SWIGLU_CLAMP ? 1 : 0;
  a1.glu_alpha = opt ? opt->swiglu_alpha : 1.f;
  a1.glu_beta = opt ? opt->swiglu_beta : 0.f;
  a1.glu_limit = opt ? opt->swiglu_limit : 0.f;
  a1.act_pos = opt ? opt->w2_inv_perm : nullptr;
  a1.pdl = pdl ? 1 : 0;
  a1.wpack = packed ? static_cast<const uint8_t*>(w13_pack) : nullptr;
  a1.wimg = prepack_image_bytes(bits, prepack_sg(r.G1), zeros ? 1 : 0);
  const int64_t units1 = static_cast<int64_t>(max_blocks) * a1.n_tiles * split1;
  const int64_t slots = static_cast<int64_t>(sms) * pipe.ctas_per_sm;
  const dim3 grid1(static_cast<unsigned>(std::min<int64_t>(units1, slots)));
  if (!mark(2)) return WNA16_ERR_CUDA;
  cudaError_t e1;
  if (defer) {
    a1.num_stages = defer_stages(bits, 1, B);
    e1 = launch_gemm_defer(bits, act_dtype, scale_dtype, 1, grid1, defer_smem_bytes(bits, 1, B, a1.num_stages), s,
                           m1.q, m1.s, m1.z, m1.b, x1, a1);
  } else {
    e1 = launch_gemm(bits, act_dtype, scale_dtype, 1, pipe.lean, grid1, pipe.smem, s, m1, a1);
  }
  if (e1 != cudaSuccess) return WNA16_ERR_CUDA;

  GemmArgs a2 = a1;
  a2.out = slab;
  a2.bias = opt ? opt->w2_bias : nullptr;
  a2.K = static_cast<int>(I);
  a2.N = static_cast<int>(H);
  a2.I = 0;
  a2.n_tiles = static_cast<int>((H + kTileRows - 1) / kTileRows);
  a2.groups = static_cast<int>(I / r.G2);
  a2.panel = panel_blocks(B, I, max_blocks);
  a2.wpack = packed ? static_cast<const uint8_t*>(w2_pack) : nullptr;
  a2.wimg = prepack_image_bytes(bits, prepack_sg(r.G2), zeros ? 1 : 0);
  a2.G = r.G2;
  a2.kt_total = static_cast<int>((I + kTileK - 1) / kTileK);
  a2.split = r.split;
  const int64_t units2 = static_cast<int64_t>(max_blocks) * a2.n_tiles * a2.split;
  const dim3 grid2(static_cast<unsigned>(std::min<int64_t>(units2, slots)));
  if (!mark(3)) return WNA16_ERR_CUDA;
  cudaError_t e2;
  if (defer) {
    a2.num_stages = defer_stages(bits, 2, B);
    e2 = launch_gemm_defer(bits, act_dtype, scale_dtype, 2, grid2, defer_smem_bytes(bits, 2, B, a2.num_stages), s,
                           m2.q, m2.s, m2.z, m2.b, x2, a2);
  } else {
    e2 = launch_gemm(bits, act_dtype, scale_dtype, 2, pipe.lean, grid2, pipe.smem, s, m2, a2);
  }
  if (e2 != cudaSuccess) return WNA16_ERR_CUDA;

  if (!mark(4) || launch_combine(slab, topk_ids, static_cast<int>(M), static_cast<int>(H), topk, E, r.split,
                                 act_dtype, out, s, pdl) != cudaSuccess)
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
