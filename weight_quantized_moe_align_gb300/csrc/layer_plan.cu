// Host-side planning of a fused-layer call (no CUDA calls): block-size and
// K-split choices, workspace layout, pipeline shapes, kernel arguments, grids
// and tensor-map descriptions.
#include "layer_plan.h"

#include <algorithm>
#include <cmath>
#include <cstring>

#include "gemm_launch.cuh"
#include "plan.cuh"

namespace wna16 {

namespace {

constexpr int kMaxSmem = 232448;         // opt-in dynamic shared memory per CTA on sm_103a
constexpr int kHalfSmem = 112 * 1024;    // two CTAs per SM
constexpr int kQuarterSmem = 55 * 1024;  // four CTAs per SM
constexpr int kMinSmem = 120 * 1024;     // a whole-SM CTA (512 TMEM columns) runs alone on its SM
constexpr int kManyExperts = 16;         // layers with more experts take token tiles of at most
constexpr int kMaxBlockManyExperts = 64; // this many tokens

bool is_pow2(long long v) { return v > 0 && (v & (v - 1)) == 0; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

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
// and for the gate/up GEMM the partial-sum exchange). On one GB300, splitting
// the gate/up GEMM of an 8-expert layer at one token (448 units on 304 slots)
// in two raised it from 38 to 49 us.
int choose_split(int64_t units, int kt_total, int ctas_per_sm, int sms) {
  const int64_t slots = static_cast<int64_t>(sms) * ctas_per_sm;
  if (units >= slots) return 1;
  int s = static_cast<int>(slots / std::max<int64_t>(units, 1));
  s = std::min(s, 8);
  s = std::min(s, std::max(1, kt_total / 8));
  return std::max(s, 1);
}

// Gate/up (rows = 2I): codes [E*2 halves, I, K/pf] box {128/pf, 64, 2} (gate
// rows then the matching up rows), scales [E*K/G, 2, I] box {64, 2, SG}, zeros
// [E*K/G, 2, I/pf] box {64/pf, 2, SG}. Down (rows = H): codes [E*H, K/pf] box
// {128/pf, 128}, scales [E*K/G, H] box {128, SG}, zeros [E*K/G, H/pf] box
// {128/pf, SG}.
void describe_weight_maps(GemmMaps* g, const int32_t* q, const void* s, const int32_t* z, int E, int64_t N, int64_t K,
                          int G, int bits, bool gate_up) {
  const int pf = 32 / bits;
  const uint64_t groups = K / G;
  const uint32_t sg = G < kTileK ? kTileK / G : 1;
  const uint32_t kw = kTileK / pf;
  // Code rows of a stage are 64 B (int4) or 128 B (int8): swizzled so that the
  // dequant warps' 16-byte reads of 8 consecutive rows hit distinct banks.
  const CUtensorMapSwizzle qswz = bits == 4 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B;
  auto set = [](MapDesc& m, int rank, int eb, CUtensorMapDataType dt, CUtensorMapSwizzle swz, const void* base,
                std::initializer_list<uint64_t> dims, std::initializer_list<uint64_t> strides,
                std::initializer_list<uint32_t> box) {
    std::memset(&m, 0, sizeof(m));
    m.rank = rank;
    m.elem_bytes = eb;
    m.dt = dt;
    m.swizzle = swz;
    m.base = base;
    std::copy(dims.begin(), dims.end(), m.dims);
    std::copy(strides.begin(), strides.end(), m.strides);
    std::copy(box.begin(), box.end(), m.box);
  };
  g->has_z = z != nullptr;
  if (gate_up) {
    const uint64_t I = N / 2;
    const uint64_t kp = static_cast<uint64_t>(K / pf);
    set(g->q, 3, 4, CU_TENSOR_MAP_DATA_TYPE_INT32, qswz, q, {kp, I, 2ull * E}, {kp * 4, I * kp * 4},
        {kw, kGateUpRows, 2});
    set(g->s, 3, 2, CU_TENSOR_MAP_DATA_TYPE_UINT16, CU_TENSOR_MAP_SWIZZLE_NONE, s, {I, 2, E * groups},
        {I * 2, 2 * I * 2}, {kGateUpRows, 2, sg});
    if (z)
      set(g->z, 3, 4, CU_TENSOR_MAP_DATA_TYPE_INT32, CU_TENSOR_MAP_SWIZZLE_NONE, z, {I / pf, 2, E * groups},
          {(I / pf) * 4, 2 * (I / pf) * 4}, {static_cast<uint32_t>(kGateUpRows / pf), 2, sg});
  } else {
    const uint64_t kp = static_cast<uint64_t>(K / pf);
    set(g->q, 2, 4, CU_TENSOR_MAP_DATA_TYPE_INT32, qswz, q, {kp, static_cast<uint64_t>(E) * N}, {kp * 4},
        {kw, kTileRows});
    set(g->s, 2, 2, CU_TENSOR_MAP_DATA_TYPE_UINT16, CU_TENSOR_MAP_SWIZZLE_NONE, s,
        {static_cast<uint64_t>(N), E * groups}, {static_cast<uint64_t>(N) * 2}, {kTileRows, sg});
    if (z)
      set(g->z, 2, 4, CU_TENSOR_MAP_DATA_TYPE_INT32, CU_TENSOR_MAP_SWIZZLE_NONE, z,
          {static_cast<uint64_t>(N / pf), E * groups}, {static_cast<uint64_t>(N / pf) * 4},
          {static_cast<uint32_t>(kTileRows / pf), sg});
  }
}

// Token tile map: rows of a [rows, K] 16-bit matrix, box {64, block} in the
// 128-byte swizzled layout (two boxes per 128-wide stage).
void describe_token_map(MapDesc* m, const void* base, int64_t K, int64_t rows, int block) {
  std::memset(m, 0, sizeof(*m));
  m->rank = 2;
  m->elem_bytes = 2;
  m->dt = CU_TENSOR_MAP_DATA_TYPE_UINT16;
  m->swizzle = CU_TENSOR_MAP_SWIZZLE_128B;
  m->base = base;
  m->dims[0] = static_cast<uint64_t>(K);
  m->dims[1] = static_cast<uint64_t>(rows);
  m->strides[0] = static_cast<uint64_t>(K) * 2;
  m->box[0] = kChunkK;
  m->box[1] = static_cast<uint32_t>(block);
}

// Token sums of a deferred-scale GEMM: fp32 [stages][parts][rows], box
// {block rows, parts, 1 stage}.
void describe_xs_map(MapDesc* m, const float* base, int64_t rows, int parts, int stages, int block) {
  std::memset(m, 0, sizeof(*m));
  m->rank = 3;
  m->elem_bytes = 4;
  m->dt = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  m->swizzle = CU_TENSOR_MAP_SWIZZLE_NONE;
  m->base = base;
  m->dims[0] = static_cast<uint64_t>(rows);
  m->dims[1] = static_cast<uint64_t>(parts);
  m->dims[2] = static_cast<uint64_t>(stages);
  m->strides[0] = static_cast<uint64_t>(rows) * 4;
  m->strides[1] = static_cast<uint64_t>(rows) * parts * 4;
  m->box[0] = static_cast<uint32_t>(block);
  m->box[1] = static_cast<uint32_t>(parts);
  m->box[2] = 1;
}

}  // namespace

uint64_t box_bytes(const MapDesc& m) {
  uint64_t b = static_cast<uint64_t>(m.elem_bytes);
  for (int i = 0; i < m.rank; ++i) b *= m.box[i];
  return b;
}

int64_t capacity(int64_t P, int E, int block) {
  const int64_t raw = P + std::min<int64_t>(P, E) * (block - 1);
  return (raw + block - 1) / block * block;
}

int choose_block_impl(int64_t M, int topk, int E) {
  const int64_t P = M * topk;
  if (P <= 0) return 16;
  const int64_t active = std::min<int64_t>(P, E);
  const double avg = static_cast<double>(P) / static_cast<double>(active);  // pairs per active expert
  // Few experts with more than 48 pairs each: one 128-token block per expert.
  // The general kernel trims its MMA width to the block's pairs, so the
  // padding costs no tensor work, and each expert's weights are dequantized
  // once instead of twice (8-expert layer at 64 pairs per expert: 283 against
  // 315 us with 64-token blocks). Layers with more experts keep the choices
  // below: larger blocks on them are unverified (see the header).
  if (E <= 16 && avg > 48.0) return 128;
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

wna16_status resolve(int64_t M, int64_t H, int64_t I, int E, int topk, int bits, int group_size, int block,
                     int split_k, int sms, Resolved* r) {
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
  // 128- and 256-token tiles on layers with more than 16 experts ended in an
  // unexplained launch failure on the GPU; the automatic choice never takes
  // them there, and forced ones are refused.
  if (block > kMaxBlockManyExperts && E > kManyExperts) return WNA16_ERR_UNSUPPORTED;
  r->block = block;
  if (split_k < 0 || split_k > 8) return WNA16_ERR_INVALID_ARG;
  const int kt2 = static_cast<int>((I + kTileK - 1) / kTileK);
  if (split_k == 0) {
    const int64_t units = expected_blocks(M, topk, E, block) * ((H + kTileRows - 1) / kTileRows);
    split_k = choose_split(units, kt2, pipe_for(bits, block).ctas_per_sm, sms);
  }
  r->split = std::min(split_k, kt2);
  // gate/up GEMM: K split only on the deferred-scale path (token tiles of 16 or
  // 32 with groups of >= 128); automatic
  r->split1 = 1;
  const int G1 = r->G1;
  if (defer_tile(block) && G1 >= kTileK && r->G2 >= kTileK) {
    const int kt1 = static_cast<int>((H + kTileK - 1) / kTileK);
    const int64_t units1 = expected_blocks(M, topk, E, block) * (I / kGateUpRows);
    r->split1 = choose_split(units1, kt1, 2, sms);
  }
  return WNA16_OK;
}

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
  w.block_rows = take(static_cast<size_t>(cap / block) * 4);
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

wna16_status plan_layer(wna16_dtype act_dtype, int64_t M, int64_t H, int64_t I, int E, int topk,
                        const int32_t* w13_q, const void* w13_scales, const int32_t* w13_zeros, const int32_t* w2_q,
                        const void* w2_scales, const int32_t* w2_zeros, const void* w13_pack, const void* w2_pack,
                        int pack_zeros, wna16_dtype scale_dtype, int bits, int group_size,
                        const float* topk_weights, void* workspace, size_t workspace_bytes, int block, int split_k,
                        bool timed, const wna16_moe_options* opt, int sms, LayerPlan* plan) {
  LayerPlan& p = *plan;
  std::memset(&p, 0, sizeof(p));
  if (act_dtype != WNA16_F16 && act_dtype != WNA16_BF16) return WNA16_ERR_INVALID_ARG;
  if (scale_dtype != WNA16_F16 && scale_dtype != WNA16_BF16) return WNA16_ERR_INVALID_ARG;
  const wna16_status st = resolve(M, H, I, E, topk, bits, group_size, block, split_k, sms, &p.r);
  if (st != WNA16_OK) return st;
  p.sms = sms;
  p.packed = w13_pack != nullptr || w2_pack != nullptr;
  p.zeros = p.packed ? pack_zeros != 0 : w13_zeros != nullptr;
  p.routed = opt && opt->router_logits;
  p.L = ws_layout(M, H, I, E, topk, p.r.block, p.r.split, p.r.split1);
  if (workspace_bytes < p.L.total) return WNA16_ERR_WORKSPACE_TOO_SMALL;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.P = static_cast<int>(M * topk);
  p.B = p.r.block;
  p.cap = capacity(p.P, E, p.B);
  p.max_blocks = static_cast<int>(p.cap / p.B);
  p.kt1 = static_cast<int>((H + kTileK - 1) / kTileK);
  p.kt2 = static_cast<int>((I + kTileK - 1) / kTileK);
  // 16- and 32-token tiles run the deferred-scale kernel when every stage lies
  // in one group (G >= 128) and the code/activation formats have a
  // magic-number form. Act-order weights run the general kernel: the
  // deferred-scale kernel's token sums assume contiguous feature runs.
  p.act_order = opt && (opt->w13_perm || opt->w2_inv_perm);
  p.defer = !p.act_order && defer_tile(p.B) && p.r.G1 >= kTileK && p.r.G2 >= kTileK &&
            defer_supported(bits, act_dtype);
  // Launches after the first run as programmatic dependents of the previous one
  // (their setup overlaps its tail), except when events are recorded between
  // them for per-kernel timing, and for batches past 8192 routed pairs: on one
  // GB300 the overlap saved 24% of the layer at 2 pairs and 0.6% at 8192, and
  // cost 2% at 16384 (int8 Mixtral-8x22B shapes).
  p.pdl = !timed && p.P <= 8192;
  float* xs1 = p.defer ? reinterpret_cast<float*>(ws + p.L.xs1) : nullptr;
  float* xs2 = p.defer ? reinterpret_cast<float*>(ws + p.L.xs2) : nullptr;

  // Token-sum parts of a stage half that holds no K elements stay zero.
  if (p.defer && H % kTileK) {
    p.zero1_off = p.L.xs1 / 4 + (static_cast<size_t>(p.kt1 - 1) * 4 + 2) * p.cap;
    p.zero1_n = static_cast<int>(2 * p.cap);
  }
  if (p.defer && I % kTileK) {
    p.zero2_off = p.L.xs2 / 4 + (static_cast<size_t>(p.kt2 - 1) * 16 + 8) * p.cap;
    p.zero2_n = static_cast<int>(8 * p.cap);
  }
  // K split of the deferred-scale gate/up GEMM: its arrival counters start at zero
  p.split1 = p.defer ? p.r.split1 : 1;
  if (p.split1 > 1) {
    p.cnt1_off = p.L.cnt1 / 4;
    p.cnt1_n = static_cast<int>((I / kGateUpRows) * p.max_blocks * 4);
  }
  // down GEMM reduced with fp32 atomics into an [M, H] accumulator at the
  // slab's start (split * P * H >= M * H floats), zeroed by the gather
  p.atomic = opt && opt->atomic_reduce;
  if (p.atomic) {
    p.acc_off = p.L.slab / 4;
    p.acc_n = static_cast<int>(M * H);
  }
  p.gather_ctas = sms * 8;
  p.pipe = pipe_for(bits, p.B);

  if (!p.packed) {
    describe_weight_maps(&p.m1, w13_q, w13_scales, p.zeros ? w13_zeros : nullptr, E, 2 * I, H, p.r.G1, bits, true);
    describe_weight_maps(&p.m2, w2_q, w2_scales, p.zeros ? w2_zeros : nullptr, E, H, I, p.r.G2, bits, false);
  }
  // Token tiles: `block` expert-sorted rows of 64 elements per stage, in the
  // 128-byte swizzled K-major layout (gathered hidden rows; the act cache).
  describe_token_map(&p.m1.b, ws + p.L.x_sorted, H, p.cap, p.B);
  describe_token_map(&p.m2.b, ws + p.L.act, I, p.cap, p.B);
  if (p.defer) {
    describe_xs_map(&p.m1.x, xs1, p.cap, defer_xs_parts(1), p.kt1, p.B);
    describe_xs_map(&p.m2.x, xs2, p.cap, defer_xs_parts(2), p.kt2, p.B);
    p.m1.has_x = p.m2.has_x = true;
  }

  GemmArgs& a1 = p.a1;
  a1.sorted_ids = reinterpret_cast<int32_t*>(ws + p.L.sorted);
  a1.expert_ids = reinterpret_cast<int32_t*>(ws + p.L.experts);
  a1.block_rows = reinterpret_cast<int32_t*>(ws + p.L.block_rows);
  a1.num_post_pad = reinterpret_cast<int32_t*>(ws + p.L.npp);
  a1.topk_w = topk_weights;
  a1.out = ws + p.L.act;
  a1.status = reinterpret_cast<int32_t*>(ws + p.L.status);
  a1.K = static_cast<int>(H);
  a1.N = static_cast<int>(2 * I);
  a1.I = static_cast<int>(I);
  a1.E = E;
  a1.n_tiles = static_cast<int>(I / kGateUpRows);
  a1.topk = topk;
  a1.P = p.P;
  a1.block = p.B;
  a1.groups = static_cast<int>(H / p.r.G1);
  a1.G = p.r.G1;
  a1.kt_total = p.kt1;
  a1.split = p.split1;
  a1.has_zeros = p.zeros ? 1 : 0;
  a1.max_blocks = p.max_blocks;
  a1.panel = panel_blocks(p.B, H, p.max_blocks);
  a1.num_stages = p.pipe.stages;
  a1.num_aslots = p.pipe.aslots;
  a1.num_acc = p.pipe.acc;
  a1.tmem_cols = p.pipe.tmem_cols;
  a1.xs_out = xs2;
  a1.cap = static_cast<int>(p.cap);
  a1.part = p.split1 > 1 ? reinterpret_cast<float*>(ws + p.L.part1) : nullptr;
  a1.counters = p.split1 > 1 ? reinterpret_cast<int*>(ws + p.L.cnt1) : nullptr;
  a1.bias = opt ? opt->w13_bias : nullptr;
  a1.glu = opt && opt->activation == WNA16_ACT_SWIGLU_CLAMP ? 1 : 0;
  a1.glu_alpha = opt ? opt->swiglu_alpha : 1.f;
  a1.glu_beta = opt ? opt->swiglu_beta : 0.f;
  a1.glu_limit = opt ? opt->swiglu_limit : 0.f;
  a1.act_pos = opt ? opt->w2_inv_perm : nullptr;
  a1.pdl = p.pdl ? 1 : 0;
  a1.wpack = p.packed ? static_cast<const uint8_t*>(w13_pack) : nullptr;
  a1.wimg = prepack_image_bytes(bits, prepack_sg(p.r.G1), p.zeros ? 1 : 0);

  GemmArgs& a2 = p.a2;
  a2 = a1;
  a2.out = ws + p.L.slab;
  a2.bias = opt ? opt->w2_bias : nullptr;
  a2.K = static_cast<int>(I);
  a2.N = static_cast<int>(H);
  a2.I = 0;
  a2.n_tiles = static_cast<int>((H + kTileRows - 1) / kTileRows);
  a2.groups = static_cast<int>(I / p.r.G2);
  a2.panel = panel_blocks(p.B, I, p.max_blocks);
  a2.wpack = p.packed ? static_cast<const uint8_t*>(w2_pack) : nullptr;
  a2.wimg = prepack_image_bytes(bits, prepack_sg(p.r.G2), p.zeros ? 1 : 0);
  a2.G = p.r.G2;
  a2.kt_total = p.kt2;
  a2.split = p.r.split;
  a2.atomic_out = p.atomic ? reinterpret_cast<float*>(ws + p.L.slab) : nullptr;

  const int64_t slots = static_cast<int64_t>(sms) * p.pipe.ctas_per_sm;
  const int64_t units1 = static_cast<int64_t>(p.max_blocks) * a1.n_tiles * a1.split;
  const int64_t units2 = static_cast<int64_t>(p.max_blocks) * a2.n_tiles * a2.split;
  p.grid1 = static_cast<unsigned>(std::min<int64_t>(units1, slots));
  p.grid2 = static_cast<unsigned>(std::min<int64_t>(units2, slots));
  const int bst = token_stage_bytes(p.B);
  if (p.defer) {
    a1.num_stages = defer_stages(bits, 1, p.B);
    a2.num_stages = defer_stages(bits, 2, p.B);
    p.smem1 = defer_smem_bytes(bits, 1, p.B, a1.num_stages);
    p.smem2 = defer_smem_bytes(bits, 2, p.B, a2.num_stages);
    p.stage_tx1 = weight_stage_tx(bits, 1, a1.has_zeros, a1.wpack ? a1.wimg : 0) + bst +
                  defer_xs_parts(1) * p.B * 4;
    p.stage_tx2 = weight_stage_tx(bits, 1, a2.has_zeros, a2.wpack ? a2.wimg : 0) + bst +
                  defer_xs_parts(2) * p.B * 4;
  } else {
    p.smem1 = p.smem2 = p.pipe.smem;
    p.stage_tx1 = weight_stage_tx(bits, a1.G < kTileK ? kTileK / a1.G : 1, a1.has_zeros, a1.wpack ? a1.wimg : 0) + bst;
    p.stage_tx2 = weight_stage_tx(bits, a2.G < kTileK ? kTileK / a2.G : 1, a2.has_zeros, a2.wpack ? a2.wimg : 0) + bst;
  }
  (void)aligned16;
  return WNA16_OK;
}

}  // namespace wna16
