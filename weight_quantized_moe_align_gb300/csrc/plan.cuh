// Index arithmetic of the grouped GEMM kernels: work-unit decoding, the TMA box
// coordinates of each pipeline stage, tensor-memory column ranges and the
// global-memory positions the epilogues write. Everything here is
// __host__ __device__ so that the kernels and the host-side launch-plan check
// (wna16_check_launch_plan) evaluate the same expressions.
#pragma once

#include "common.cuh"

#define WNA16_HD __host__ __device__ __forceinline__

namespace wna16 {

struct Unit {
  int blk, tile, sp, kt0, kt1;
};

// Work-unit order (the same in every role): panels of a.panel consecutive
// token blocks (the align output is expert-sorted, so a panel spans one or a
// few experts); inside a panel the weight tile is the slowest index and the K
// split the fastest. Concurrent CTAs then share a panel's token rows and each
// weight tile across the panel's blocks. The host sizes panels so that their
// token rows stay well inside L2; small batches get one panel.
WNA16_HD Unit decode_unit(int u, int nb, const GemmArgs& a) {
  Unit r;
  const int panel_units = a.panel * a.n_tiles * a.split;
  const int p = u / panel_units;
  const int b0 = p * a.panel;
  const int pbs = nb - b0 < a.panel ? nb - b0 : a.panel;  // blocks in this panel
  int rest = u - p * panel_units;
  r.sp = rest % a.split;
  rest /= a.split;
  r.blk = b0 + rest % pbs;
  r.tile = rest / pbs;
  r.kt0 = static_cast<int>(static_cast<long long>(a.kt_total) * r.sp / a.split);
  r.kt1 = static_cast<int>(static_cast<long long>(a.kt_total) * (r.sp + 1) / a.split);
  return r;
}

// Token blocks the GEMMs run: the align kernel's padded total over the tile,
// clamped to the capacity the launch was sized for.
WNA16_HD int active_blocks(int num_post_pad, int nt, int max_blocks) {
  const int nb = num_post_pad / nt;
  return nb < 0 ? 0 : (nb > max_blocks ? max_blocks : nb);
}

// Routed pairs in the block starting at slot `start` of an expert whose cnt
// pairs begin at slot seg (its padded segment holds them first, then padding).
WNA16_HD int rows_in_block(int cnt, int seg, int start, int block) {
  const int rows = cnt - (start - seg);
  return rows < 0 ? 0 : (rows > block ? block : rows);
}

// MMA width (tokens) of a block holding `rows` routed pairs in a tile of nt:
// the rows rounded up to the MMA's N granule of 16; the padding past it is
// neither multiplied nor written back.
WNA16_HD int trimmed_n(int rows, int nt) {
  const int n = (rows + 15) & ~15;
  return n < 16 ? 16 : (n > nt ? nt : n);
}

// Blocks below the padded total always hold a valid expert id; anything else
// is mapped to expert 0 so that no address is formed from it.
WNA16_HD int clamp_expert(int e, int E) { return (e >= 0 && e < E) ? e : 0; }

// Scale / zero-point row (group row of the [E * K/G, ...] tensors) of stage kt
// of expert e.
WNA16_HD int stage_group_row(const GemmArgs& a, int e, int kt) { return e * a.groups + (kt * kTileK) / a.G; }

// Tensor-map coordinates of one weight stage (innermost first):
//   gate/up (GEMM 1): codes (kt*KW, f0, 2e) in [E*2 halves, I, K/pf], scales
//     (f0, 0, ys) in [E*K/G, 2, I], zero words (f0/pf, 0, ys) in [E*K/G, 2, I/pf]
//     with f0 = tile * 64 (the tile's 64 gate rows and the matching up rows);
//   down (GEMM 2): codes (kt*KW, e*N + r0) in [E*N, K/pf], scales (r0, ys) in
//     [E*K/G, N], zero words (r0/pf, ys) in [E*K/G, N/pf] with r0 = tile * 128.
struct StageCoords {
  int q[3], s[3], z[3];
};

WNA16_HD StageCoords weight_stage_coords(int gemm, int bits, const GemmArgs& a, int tile, int e, int kt, int ys) {
  const int pf = 32 / bits;
  const int kw = kTileK * bits / 32;
  StageCoords c;
  if (gemm == 1) {
    const int f0 = tile * kGateUpRows;
    c.q[0] = kt * kw; c.q[1] = f0; c.q[2] = 2 * e;
    c.s[0] = f0; c.s[1] = 0; c.s[2] = ys;
    c.z[0] = f0 / pf; c.z[1] = 0; c.z[2] = ys;
  } else {
    const int r0 = tile * kTileRows;
    c.q[0] = kt * kw; c.q[1] = e * a.N + r0; c.q[2] = 0;
    c.s[0] = r0; c.s[1] = ys; c.s[2] = 0;
    c.z[0] = r0 / pf; c.z[1] = ys; c.z[2] = 0;
  }
  return c;
}

// Token tile of a stage: 64-wide K chunk c of rows [blk*nt, blk*nt + nt) of
// the expert-sorted [cap, K] matrix; and the stage's token sums (deferred-scale
// kernel): rows [blk*nt, +nt) of parts [0, parts) of stage kt.
WNA16_HD int token_x(int kt, int c) { return kt * kTileK + c * kChunkK; }
WNA16_HD int token_y(int blk, int nt) { return blk * nt; }

// Bytes the producer expects on a stage's barrier: the weight part (plain
// boxes: codes, sg group rows of scales and of zero-point words; or one
// prepacked image of `wimg` bytes), the token tile (`bst`) and, in the
// deferred-scale kernel, the stage's token sums (`xst`).
WNA16_HD uint32_t weight_stage_tx(int bits, int sg, int has_zeros, int wimg) {
  if (wimg) return static_cast<uint32_t>(wimg);
  return static_cast<uint32_t>(weight_code_bytes(bits) + sg * kTileRows * 2 +
                               (has_zeros ? sg * (kTileRows * bits / 32) * 4 : 0));
}

// Prepacked stage image of (expert, tile, stage).
WNA16_HD size_t image_offset(const GemmArgs& a, int e, int tile, int kt) {
  return ((static_cast<size_t>(e) * a.n_tiles + tile) * a.kt_total + kt) * a.wimg;
}

// ---------------------------------------------------------------- epilogues
// Act cache element of token column `col` of block blk, feature column fp.
WNA16_HD size_t act_index(int blk, int nt, int col, int I, int fp) {
  return (static_cast<size_t>(blk) * nt + col) * I + fp;
}
// fp32 slab element of K split sp, pair pid, output row `row`.
WNA16_HD size_t slab_index(int sp, int P, int pid, int N, int row) {
  return (static_cast<size_t>(sp) * P + pid) * N + row;
}
// Deferred-scale gate/up epilogue: token sum of part `part` (0..15) of down
// stage tile/2 for act-cache row `row`.
WNA16_HD size_t xs_out_index(int tile, int part, int cap, size_t row) {
  return (static_cast<size_t>(tile >> 1) * 16 + part) * cap + row;
}
// K-split partial sums of the deferred-scale gate/up GEMM: [tile][block][split][128][nt].
WNA16_HD size_t part_index(const GemmArgs& a, int tile, int blk, int sp, int row, int nt) {
  return (((static_cast<size_t>(tile) * a.max_blocks + blk) * a.split + sp) * kTileRows + row) * nt;
}
WNA16_HD size_t counter_index(const GemmArgs& a, int tile, int blk, int q) {
  return (static_cast<size_t>(tile) * a.max_blocks + blk) * 4 + q;
}

// ---------------------------------------------------------------- shared memory
// Byte offsets of a CTA's dynamic shared memory, from its 1024-aligned base:
// the weight ring, the token ring, (deferred-scale kernel) the two correction
// tiles and the token-sum ring, then the mbarriers, the TMEM address word and
// the abort flag; `end` is the bytes used past the aligned base.
struct SmemLayout {
  int wring, bring, bcorr, xring, bars, n_bars, holder, abort_flag, end;
};

WNA16_HD SmemLayout gemm_smem_layout(int bits, int nt, int stages, int aslots, int accs) {
  SmemLayout l;
  l.wring = 0;
  l.bring = weight_ring_bytes(bits, stages);
  l.bcorr = l.xring = l.bring + stages * token_stage_bytes(nt);
  l.bars = l.xring;
  l.n_bars = 2 * stages + aslots + 2 * accs + 1;  // full, empty, afull, accfull, accempty, drain
  l.holder = l.bars + 8 * l.n_bars;
  l.abort_flag = l.holder + 4;
  l.end = l.abort_flag + 4;
  return l;
}

WNA16_HD SmemLayout defer_smem_layout(int bits, int gemm, int nt, int stages) {
  SmemLayout l;
  l.wring = 0;
  l.bring = weight_ring_bytes(bits, stages);
  l.bcorr = l.bring + stages * token_stage_bytes(nt);  // 2 tiles of nt rows x 128 B
  l.xring = l.bcorr + 2 * nt * 128;                    // stages x [parts][nt] floats
  l.bars = l.xring + stages * defer_xs_parts(gemm) * nt * 4;
  l.n_bars = 2 * stages + 2 + 2 + 3;  // full, empty, afull[2], pfull[2], cfull, cempty, drain
  l.holder = l.bars + 8 * l.n_bars;
  l.abort_flag = l.holder + 4;
  l.end = l.abort_flag + 4;
  return l;
}

// ---------------------------------------------------------------- tensor memory
// Deferred-scale kernel, 256 columns: partial sum P_g at [g*nt, +nt); combine
// buffer C at [32, 48) for 16-token tiles and P_1 itself for 32-token tiles;
// A slot g at 64 + 96 g: 64 columns of codes (128 K) and 8 correction columns.
constexpr int kDeferA0 = 64;
constexpr int kDeferAStride = 96;
constexpr int kDeferACols = 72;
constexpr int kDeferTmemCols = 256;
WNA16_HD int defer_p_col(int g, int nt) { return g * nt; }
WNA16_HD int defer_c_col(int nt) { return nt == 16 ? 32 : nt; }
WNA16_HD int defer_a_col(int g) { return kDeferA0 + g * kDeferAStride; }

// Token columns of a block that the deferred-scale epilogue writes (the
// routed pairs lead a block): the gate/up epilogue finishes columns j and
// j + nt/2 together and stops at the first j past the routed pairs; the down
// epilogue stops at the routed pairs.
WNA16_HD bool defer_writes_col(int gemm, int col, int rows, int nt) {
  if (gemm == 2) return col < rows;
  return (col < nt / 2 ? col : col - nt / 2) < rows;
}

// General kernel: accumulator i at [i*nt, +nt), A slot s at nacc*nt + s*64.
WNA16_HD int gemm_acc_col(int acc, int nt) { return acc * nt; }
WNA16_HD int gemm_a_col(int nacc, int nt, int slot) { return nacc * nt + slot * kASlotCols; }

}  // namespace wna16
