// wna16_check_launch_plan: a host-only replay of one fused-layer call.
//
// Given the shapes, the call's block / split arguments and the align step's
// output (computed by any means, e.g. a reference implementation), it builds
// the same plan the launcher builds (layer_plan.cu) and walks every role of
// every CTA of the two GEMM launches through the same index expressions the
// kernels evaluate (plan.cuh). It checks, without a GPU:
//   * every TMA box of every stage lies inside its tensor map, its innermost
//     coordinate is 16-byte aligned, and the boxes of a stage add up to the
//     bytes the producer expects on the stage barrier;
//   * the deferred-scale producer's running scale row equals the closed form;
//   * the work units decode to every (block, tile, split) exactly once;
//   * tensor-memory columns of accumulators, partial sums and A slots lie in
//     the allocation and do not overlap (except the 32-token tile's combine
//     buffer, which is P_1 by design);
//   * shared-memory carve-ups fit the launch's dynamic shared memory, with the
//     alignment TMA destinations and 128-byte-swizzled operands need;
//   * every global write of the gather, both epilogues and the combine lands
//     in its workspace region, every routed pair's slab row is written once
//     per K split and output row, and every read of the align output stays in
//     its array.
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <vector>

#include "layer_plan.h"
#include "plan.cuh"
#include "wna16_moe.h"

namespace wna16 {
namespace {

struct Checker {
  int64_t violations = 0;
  char* report;
  size_t cap_bytes, used = 0;
  void fail(const char* fmt, ...) {
    ++violations;
    if (!report || used + 1 >= cap_bytes || violations > 20) return;
    va_list ap;
    va_start(ap, fmt);
    const int n = vsnprintf(report + used, cap_bytes - used, fmt, ap);
    va_end(ap);
    if (n > 0) used = std::min(cap_bytes - 1, used + static_cast<size_t>(n));
    if (used + 1 < cap_bytes) report[used++] = '\n';
    report[used] = 0;
  }
};

// A box at `coord` (rank entries) of map m: inside on every dimension.
void check_box(Checker& c, const MapDesc& m, const int* coord, const char* what, int gemm, int unit, int kt) {
  if ((static_cast<int64_t>(coord[0]) * m.elem_bytes) % 16)
    c.fail("GEMM %d unit %d stage %d: %s x=%d not 16-byte aligned", gemm, unit, kt, what, coord[0]);
  for (int d = 0; d < m.rank; ++d) {
    if (coord[d] < 0 || static_cast<uint64_t>(coord[d]) + m.box[d] > m.dims[d]) {
      c.fail("GEMM %d unit %d stage %d: %s box dim %d at %d (+%u) outside [0, %llu)", gemm, unit, kt, what, d,
             coord[d], m.box[d], static_cast<unsigned long long>(m.dims[d]));
      return;
    }
  }
}

struct Range {
  int lo, hi;  // [lo, hi)
};

void check_tmem(Checker& c, int gemm, const std::vector<Range>& r, int cols, int allowed_alias_a, int allowed_alias_b) {
  for (size_t i = 0; i < r.size(); ++i) {
    if (r[i].lo < 0 || r[i].hi > cols) c.fail("GEMM %d: TMEM range %zu [%d, %d) outside %d columns", gemm, i, r[i].lo, r[i].hi, cols);
    for (size_t j = i + 1; j < r.size(); ++j) {
      const bool alias = (static_cast<int>(i) == allowed_alias_a && static_cast<int>(j) == allowed_alias_b);
      if (!alias && r[i].lo < r[j].hi && r[j].lo < r[i].hi)
        c.fail("GEMM %d: TMEM ranges %zu [%d, %d) and %zu [%d, %d) overlap", gemm, i, r[i].lo, r[i].hi, j, r[j].lo,
               r[j].hi);
    }
  }
}

void check_smem(Checker& c, int gemm, const SmemLayout& l, int stages, int wst, int bst, size_t smem, bool defer,
                int xst) {
  // the kernels round their dynamic shared memory base up to 1024 bytes
  if (static_cast<size_t>(l.end) + 1023 > smem)
    c.fail("GEMM %d: shared memory layout needs %d + 1023 bytes, launch gives %zu", gemm, l.end, smem);
  for (int s = 0; s < stages; ++s) {
    if ((l.wring + s * wst) % 1024) c.fail("GEMM %d: weight stage %d not 1024-byte aligned", gemm, s);
    if ((l.bring + s * bst) % 1024) c.fail("GEMM %d: token stage %d not 1024-byte aligned", gemm, s);
    if (defer && (l.xring + s * xst) % 128) c.fail("GEMM %d: token-sum stage %d not 128-byte aligned", gemm, s);
  }
  if (l.bring < stages * wst) c.fail("GEMM %d: weight ring overlaps the token ring", gemm);
  if (defer && (l.bcorr % 1024)) c.fail("GEMM %d: correction tiles not 1024-byte aligned", gemm);
  if (l.bars % 8) c.fail("GEMM %d: barriers not 8-byte aligned", gemm);
}

}  // namespace
}  // namespace wna16

using namespace wna16;

extern "C" int64_t wna16_check_launch_plan(int64_t M, int64_t H, int64_t I, int E, int topk, int bits, int group_size,
                                           int has_zeros, wna16_dtype act_dtype, wna16_dtype scale_dtype, int block,
                                           int split_k, int sms, const int32_t* topk_ids, const int32_t* sorted_ids,
                                           const int32_t* expert_ids, int32_t num_tokens_post_padded, char* report,
                                           size_t report_bytes) {
  Checker c;
  c.report = report;
  c.cap_bytes = report_bytes;
  if (report && report_bytes) report[0] = 0;
  if (sms < 1 || M < 1 || !topk_ids || !sorted_ids || !expert_ids) return -static_cast<int64_t>(WNA16_ERR_INVALID_ARG);
  // Stand-in addresses: the plan only forms pointers from them; nothing is
  // dereferenced except the host arrays given here.
  uint8_t* const ws = reinterpret_cast<uint8_t*>(uintptr_t(1) << 40);
  const int32_t* const wq = reinterpret_cast<const int32_t*>(uintptr_t(1) << 41);
  const void* const wsc = reinterpret_cast<const void*>(uintptr_t(1) << 42);
  const int32_t* const wz = has_zeros ? reinterpret_cast<const int32_t*>(uintptr_t(1) << 43) : nullptr;
  LayerPlan p;
  const wna16_status st = plan_layer(act_dtype, M, H, I, E, topk, wq, wsc, wz, wq, wsc, wz, nullptr, nullptr, 0,
                                     scale_dtype, bits, group_size, nullptr, ws, ~size_t(0) >> 2, block, split_k,
                                     false, nullptr, sms, &p);
  if (st != WNA16_OK) return -static_cast<int64_t>(st);
  const int P = p.P, B = p.B;
  const int64_t cap = p.cap;
  const int npp = num_tokens_post_padded;
  if (npp < 0 || npp > cap || npp % B) c.fail("num_tokens_post_padded %d: not a multiple of %d within %lld", npp, B, (long long)cap);
  const int nb = active_blocks(npp, B, p.max_blocks);
  for (int b = 0; b < nb; ++b)
    if (expert_ids[b] < 0 || expert_ids[b] >= E) c.fail("expert_ids[%d] = %d below the padded total", b, expert_ids[b]);

  // rows per block as the align kernel computes them (from each expert's count
  // and segment start), checked against the align output: the routed pairs
  // lead each block and the padding follows
  std::vector<int> cnt(E, 0), seg(E, -1), block_rows(p.max_blocks, 0);
  for (int pr = 0; pr < P; ++pr)
    if (topk_ids[pr] >= 0 && topk_ids[pr] < E) ++cnt[topk_ids[pr]];
  for (int b = 0; b < nb; ++b) {
    const int e = expert_ids[b];
    if (e >= 0 && e < E && seg[e] < 0) seg[e] = b * B;
  }
  for (int b = 0; b < nb; ++b) {
    const int e = expert_ids[b];
    if (e < 0 || e >= E) continue;
    block_rows[b] = rows_in_block(cnt[e], seg[e], b * B, B);
    for (int col = 0; col < B; ++col) {
      const int pid = sorted_ids[static_cast<int64_t>(b) * B + col];
      const bool routed = pid >= 0 && pid < P;
      if (routed != (col < block_rows[b])) {
        c.fail("block %d: column %d %s, but the block holds %d routed pairs first", b, col,
               routed ? "routed" : "padding", block_rows[b]);
        break;
      }
    }
  }

  // ------------------------------------------------------------ gather
  std::vector<int> slot_of_pair(P, -1);
  for (int64_t i = 0; i < cap; ++i) {
    const int pid = sorted_ids[i];
    if (pid >= 0 && pid < P) {
      if (slot_of_pair[pid] >= 0) c.fail("pair %d appears twice in sorted_ids", pid);
      slot_of_pair[pid] = static_cast<int>(i);
    }
  }
  const size_t h8 = static_cast<size_t>(H) / 8;
  const size_t xs1_words = p.defer ? static_cast<size_t>(p.kt1) * defer_xs_parts(1) * cap : 0;
  for (int pr = 0; pr < P; ++pr) {
    const int e = topk_ids[pr];
    if (e < 0 || e >= E) continue;
    const int slot = slot_of_pair[pr];
    if (slot < 0 || slot >= cap) {
      c.fail("routed pair %d has no slot below the capacity", pr);
      continue;
    }
    if ((static_cast<size_t>(slot) + 1) * h8 * 16 > p.L.act - p.L.x_sorted)
      c.fail("gather: row of slot %d past the gathered-rows region", slot);
    if (p.defer) {
      const size_t chunks = h8 / 8;
      const size_t last = ((chunks - 1) / 2 * 4 + ((chunks - 1) & 1) * 2) * cap + slot + cap;
      if (last >= xs1_words) c.fail("gather: token sum of slot %d past the gate/up token sums", slot);
    }
  }
  if (p.zero1_n && (p.zero1_off + p.zero1_n) * 4 > p.L.xs1 + xs1_words * 4)
    c.fail("gather: zero fill of the gate/up token sums past its region");
  if (p.zero2_n && (p.zero2_off + p.zero2_n) * 4 > p.L.xs2 + static_cast<size_t>(p.kt2) * 16 * cap * 4)
    c.fail("gather: zero fill of the down token sums past its region");
  if (p.cnt1_n && (p.cnt1_off + p.cnt1_n) * 4 > p.L.total) c.fail("gather: counter fill past the workspace");

  // ------------------------------------------------------------ GEMMs
  for (int gemm = 1; gemm <= 2; ++gemm) {
    GemmArgs a = gemm == 1 ? p.a1 : p.a2;
    a.sorted_ids = sorted_ids;
    a.expert_ids = expert_ids;
    a.block_rows = block_rows.data();
    const GemmMaps& maps = gemm == 1 ? p.m1 : p.m2;
    const unsigned grid = gemm == 1 ? p.grid1 : p.grid2;
    const size_t smem = gemm == 1 ? p.smem1 : p.smem2;
    const uint32_t stage_tx = gemm == 1 ? p.stage_tx1 : p.stage_tx2;
    const int NS = a.num_stages;
    const int wst = weight_stage_bytes(bits);
    const int bst = token_stage_bytes(B);
    const int xparts = defer_xs_parts(gemm);
    const int xst = xparts * B * 4;

    // shared memory
    const SmemLayout sl = p.defer ? defer_smem_layout(bits, gemm, B, NS)
                                  : gemm_smem_layout(bits, B, NS, a.num_aslots, a.num_acc);
    check_smem(c, gemm, sl, NS, wst, bst, smem, p.defer, xst);
    // the stage's boxes against the bytes the producer expects
    const int sg = a.G < kTileK ? kTileK / a.G : 1;
    uint64_t boxes = box_bytes(maps.q) + box_bytes(maps.s) + (maps.has_z ? box_bytes(maps.z) : 0) +
                     2 * box_bytes(maps.b) + (p.defer ? box_bytes(maps.x) : 0);
    if (boxes != stage_tx)
      c.fail("GEMM %d: stage boxes hold %llu bytes, producer expects %u", gemm, (unsigned long long)boxes, stage_tx);
    if (box_bytes(maps.q) != static_cast<uint64_t>(weight_code_bytes(bits)) ||
        box_bytes(maps.s) > 512 || (maps.has_z && box_bytes(maps.z) > 512) ||
        2 * box_bytes(maps.b) != static_cast<uint64_t>(bst) || (p.defer && box_bytes(maps.x) != static_cast<uint64_t>(xst)))
      c.fail("GEMM %d: a box does not match its shared-memory slot", gemm);
    (void)sg;

    // tensor memory
    std::vector<Range> cols;
    if (p.defer) {
      cols = {{defer_p_col(0, B), defer_p_col(0, B) + B}, {defer_p_col(1, B), defer_p_col(1, B) + B},
              {defer_c_col(B), defer_c_col(B) + B}, {defer_a_col(0), defer_a_col(0) + kDeferACols},
              {defer_a_col(1), defer_a_col(1) + kDeferACols}};
      // 32-token tiles: C is P_1 (ranges 1 and 2)
      check_tmem(c, gemm, cols, kDeferTmemCols, B == 32 ? 1 : -1, B == 32 ? 2 : -1);
      if (B == 16 && defer_c_col(B) == defer_p_col(1, B)) c.fail("GEMM %d: 16-token C aliases P_1", gemm);
    } else {
      for (int i = 0; i < a.num_acc; ++i) cols.push_back({gemm_acc_col(i, B), gemm_acc_col(i, B) + B});
      for (int i = 0; i < a.num_aslots; ++i)
        cols.push_back({gemm_a_col(a.num_acc, B, i), gemm_a_col(a.num_acc, B, i) + kASlotCols});
      check_tmem(c, gemm, cols, static_cast<int>(a.tmem_cols), -1, -1);
    }

    // work units: a bijection onto (block < nb, tile, split)
    const int64_t units = static_cast<int64_t>(nb) * a.n_tiles * a.split;
    std::vector<uint8_t> seen(static_cast<size_t>(units), 0);
    const size_t act_elems = static_cast<size_t>(cap) * a.I;
    const size_t slab_elems = static_cast<size_t>(p.r.split) * P * H;
    const size_t xs2_elems = static_cast<size_t>(p.kt2) * 16 * cap;
    const size_t part_elems = p.split1 > 1 ? (p.L.cnt1 - p.L.part1) / 4 : 0;
    const size_t cnt_elems = p.split1 > 1 ? static_cast<size_t>(I / kGateUpRows) * p.max_blocks * 4 : 0;
    std::vector<uint16_t> slab_hits(gemm == 2 ? static_cast<size_t>(p.r.split) * P * a.n_tiles : 0, 0);
    const int spg = (a.G + kTileK - 1) / kTileK;
    for (unsigned cta = 0; cta < grid; ++cta) {
      for (int64_t u = cta; u < units; u += grid) {
        const Unit w = decode_unit(static_cast<int>(u), nb, a);
        if (w.blk < 0 || w.blk >= nb || w.tile < 0 || w.tile >= a.n_tiles || w.sp < 0 || w.sp >= a.split ||
            w.kt0 < 0 || w.kt1 > a.kt_total || w.kt0 >= w.kt1) {
          c.fail("GEMM %d: unit %lld decodes to block %d tile %d split %d stages [%d, %d)", gemm, (long long)u, w.blk,
                 w.tile, w.sp, w.kt0, w.kt1);
          continue;
        }
        const size_t key = (static_cast<size_t>(w.tile) * nb + w.blk) * a.split + w.sp;
        if (seen[key]++) c.fail("GEMM %d: unit %lld repeats block %d tile %d split %d", gemm, (long long)u, w.blk, w.tile, w.sp);
        const int e = clamp_expert(expert_ids[w.blk], E);
        // producer: the deferred kernel advances the scale row once per group
        int ys_run = e * a.groups + w.kt0 / spg, gk = w.kt0 % spg;
        for (int kt = w.kt0; kt < w.kt1; ++kt) {
          const int ys = stage_group_row(a, e, kt);
          if (p.defer && ys_run != ys) c.fail("GEMM %d unit %lld stage %d: running scale row %d != %d", gemm, (long long)u, kt, ys_run, ys);
          if (++gk == spg) {
            gk = 0;
            ++ys_run;
          }
          const StageCoords sc = weight_stage_coords(gemm, bits, a, w.tile, e, kt, ys);
          check_box(c, maps.q, sc.q, "codes", gemm, static_cast<int>(u), kt);
          check_box(c, maps.s, sc.s, "scales", gemm, static_cast<int>(u), kt);
          if (maps.has_z) check_box(c, maps.z, sc.z, "zero points", gemm, static_cast<int>(u), kt);
          for (int ch = 0; ch < kTileK / kChunkK; ++ch) {
            const int tc[2] = {token_x(kt, ch), token_y(w.blk, B)};
            check_box(c, maps.b, tc, "token tile", gemm, static_cast<int>(u), kt);
          }
          if (p.defer) {
            const int xc[3] = {token_y(w.blk, B), 0, kt};
            check_box(c, maps.x, xc, "token sums", gemm, static_cast<int>(u), kt);
          }
        }
        // epilogue: the general kernel writes the block's routed columns
        // rounded up to 16, the deferred-scale kernel its routed columns (the
        // gate/up one in pairs j, j + B/2)
        const int rows = a.block_rows[w.blk];
        auto writes = [&](int col) {
          return p.defer ? defer_writes_col(gemm, col, rows, B) : col < trimmed_n(rows, B);
        };
        for (int col = 0; col < block_rows[w.blk]; ++col)
          if (!writes(col)) c.fail("GEMM %d: block %d leaves routed column %d unwritten", gemm, w.blk, col);
        if (gemm == 1) {
          for (int q = 0; q < 4; ++q)
            for (int lane = 0; lane < 32; ++lane) {
              const int f = w.tile * kGateUpRows + 16 * q + (lane & 15);
              const int fp = bits == 4 ? permute_k8(f) : f;
              if (f >= a.I) c.fail("GEMM 1: feature %d of tile %d past I", f, w.tile);
              for (int col = 0; col < B; ++col) {
                if (!writes(col)) continue;
                if (act_index(w.blk, B, col, a.I, fp) >= act_elems)
                  c.fail("GEMM 1: act cache element of block %d column %d feature %d past the act cache", w.blk, col, fp);
              }
              if (p.defer) {
                for (int col = 0; col < B; ++col) {
                  if (!writes(col)) continue;
                  const size_t row = static_cast<size_t>(w.blk) * B + col;
                  const int part = (w.tile & 1) * 8 + q * 2 + (lane & 1);
                  if (xs_out_index(w.tile, part, a.cap, row) >= xs2_elems)
                    c.fail("GEMM 1: down token sum (tile %d, part %d, row %zu) past its region", w.tile, part, row);
                }
                if (a.split > 1) {
                  const int row = q * 32 + lane;
                  if (part_index(a, w.tile, w.blk, w.sp, row, B) + B > part_elems)
                    c.fail("GEMM 1: K-split partial of tile %d block %d split %d past its region", w.tile, w.blk, w.sp);
                  if (counter_index(a, w.tile, w.blk, q) >= cnt_elems)
                    c.fail("GEMM 1: arrival counter of tile %d block %d past its region", w.tile, w.blk);
                }
              }
            }
        } else {
          for (int col = 0; col < B; ++col) {
            if (!writes(col)) continue;
            const int64_t si = static_cast<int64_t>(w.blk) * B + col;
            if (si >= cap) {
              c.fail("GEMM 2: sorted_ids read %lld past the capacity", (long long)si);
              continue;
            }
            const int pid = sorted_ids[si];
            if (pid < 0 || pid >= P) continue;  // padding: not written
            if (topk_ids[pid] != expert_ids[w.blk]) c.fail("GEMM 2: pair %d of block %d routed elsewhere", pid, w.blk);
            for (int r = 0; r < kTileRows; ++r) {
              const int hr = w.tile * kTileRows + r;
              if (hr >= a.N) continue;
              if (slab_index(w.sp, P, pid, a.N, hr) >= slab_elems)
                c.fail("GEMM 2: slab element (split %d, pair %d, row %d) past the slab", w.sp, pid, hr);
            }
            ++slab_hits[(static_cast<size_t>(w.sp) * P + pid) * a.n_tiles + w.tile];
          }
        }
      }
    }
    for (size_t i = 0; i < seen.size(); ++i)
      if (!seen[i]) {
        c.fail("GEMM %d: a (block, tile, split) unit is never run", gemm);
        break;
      }
    if (gemm == 2) {
      // every routed pair's slab row: once per split and row tile
      for (int sp = 0; sp < p.r.split; ++sp)
        for (int pr = 0; pr < P; ++pr) {
          const bool routed = topk_ids[pr] >= 0 && topk_ids[pr] < E;
          for (int t = 0; t < a.n_tiles; ++t) {
            const int hits = slab_hits[(static_cast<size_t>(sp) * P + pr) * a.n_tiles + t];
            if (hits != (routed ? 1 : 0)) {
              c.fail("GEMM 2: slab rows of pair %d split %d tile %d written %d times", pr, sp, t, hits);
              sp = p.r.split;
              pr = P;
              break;
            }
          }
        }
    }
  }
  // ------------------------------------------------------------ combine
  const size_t slab_elems = static_cast<size_t>(p.r.split) * P * H;
  if (static_cast<size_t>(p.r.split - 1) * P * H + (static_cast<size_t>(P) - 1) * H + H > slab_elems)
    c.fail("combine: slab read past the slab");
  if (p.L.slab + slab_elems * 4 > p.L.xs1 && p.L.xs1 > p.L.slab) c.fail("slab overlaps the token sums");
  return c.violations;
}
