// Host-side plan of one fused-layer call: resolved block size and K splits,
// workspace layout, pipeline shapes, the kernels' arguments, grids and the
// tensor-map descriptions. Computing a plan makes no CUDA call, so the same
// plan drives the launches (host.cu) and the host-only replay that checks
// every index a launch forms (plan_check.cu).
#pragma once

#include <cuda.h>

#include <cstddef>
#include <cstdint>

#include "common.cuh"
#include "wna16_moe.h"

namespace wna16 {

int64_t capacity(int64_t P, int E, int block);
int choose_block_impl(int64_t M, int topk, int E);

// Pipeline shape of one general-kernel launch for a token tile of `block`.
struct Pipe {
  int stages, aslots, acc, ctas_per_sm, lean;
  uint32_t tmem_cols;
  size_t smem;
};
Pipe pipe_for(int bits, int block);
int defer_stages(int bits, int gemm, int nt);

struct Resolved {
  int block, split, split1, G1, G2;
};
// Argument checks and the automatic choices; `sms` = SMs of the device.
wna16_status resolve(int64_t M, int64_t H, int64_t I, int E, int topk, int bits, int group_size, int block,
                     int split_k, int sms, Resolved* r);

struct WsLayout {
  size_t status, sorted, experts, block_rows, npp, counts, slot_of_pair, x_sorted, act, slab, xs1, xs2, part1, cnt1,
      total;
};
WsLayout ws_layout(int64_t M, int64_t H, int64_t I, int E, int topk, int block, int split, int split1);

// A tiled tensor map before encoding: dims[0] innermost (elements), byte
// strides of dims 1.., box in elements.
struct MapDesc {
  int rank;
  int elem_bytes;
  CUtensorMapDataType dt;
  CUtensorMapSwizzle swizzle;
  const void* base;
  uint64_t dims[3];
  uint64_t strides[2];
  uint32_t box[3];
};
uint64_t box_bytes(const MapDesc& m);

// Maps of one GEMM: codes, scales, zero points (has_z), token tile, and with
// the deferred-scale kernel the per-stage token sums.
struct GemmMaps {
  MapDesc q, s, z, b, x;
  bool has_z, has_x;
};

struct LayerPlan {
  Resolved r;
  WsLayout L;
  Pipe pipe;
  int P, B, max_blocks, kt1, kt2, split1, sms;
  int64_t cap;
  bool defer, packed, zeros, act_order, pdl, routed, atomic;
  GemmArgs a1, a2;
  unsigned grid1, grid2;
  size_t smem1, smem2;
  uint32_t stage_tx1, stage_tx2;  // bytes the producer expects per stage
  GemmMaps m1, m2;                // unused (zeroed) for prepacked weights, except the token maps
  // zero fills done by the gather launch (token sums of empty stage halves,
  // split arrival counters), as offsets into the workspace in 4-byte words
  size_t zero1_off, zero2_off, cnt1_off, acc_off;
  int zero1_n, zero2_n, cnt1_n, acc_n;
  int gather_ctas;
};

// Everything a call computes before its first launch. Pointers into the
// workspace are formed from `workspace` (may be a stand-in base for a plan
// that is only checked). Returns the call's argument error, if any.
wna16_status plan_layer(wna16_dtype act_dtype, int64_t M, int64_t H, int64_t I, int E, int topk,
                        const int32_t* w13_q, const void* w13_scales, const int32_t* w13_zeros, const int32_t* w2_q,
                        const void* w2_scales, const int32_t* w2_zeros, const void* w13_pack, const void* w2_pack,
                        int pack_zeros, wna16_dtype scale_dtype, int bits, int group_size,
                        const float* topk_weights, void* workspace, size_t workspace_bytes, int block, int split_k,
                        bool timed, const wna16_moe_options* opt, int sms, LayerPlan* plan);

}  // namespace wna16
