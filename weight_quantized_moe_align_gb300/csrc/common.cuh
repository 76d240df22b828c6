// Shared definitions of the host layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace wna16 {

// Threads of the grouped-GEMM kernel and their roles (warp index):
//   0      TMA producer (packed weights, scales, zero points, token tile)
//   1      tcgen05 MMA issuer, owner of the TMEM allocation
//   2..5   epilogue (TMEM -> registers -> global); lane quarter = warp % 4
//   6..13  dequantizers, two stage-parallel warpgroups (shared -> registers -> TMEM)
// A lean layout (producer, MMA issuer, 4 dequant warps that also run the
// epilogue) fits four CTAs per SM for int4 token tiles up to 32 (128 TMEM
// columns, <= 56 KB of shared memory each): four MMA-issuing threads share the
// tensor core. Other tiles up to 64 run two CTAs per SM of the full layout
// (256 TMEM columns, <= 112 KB each); larger tiles take the whole SM.
constexpr int kDequantWarps = 8;   // two warpgroups (LEAN = 0); LEAN = 1 uses one
constexpr int kEpilogueWarps = 4;
__host__ __device__ constexpr int gemm_threads(int lean) { return lean ? 6 * 32 : 14 * 32; }

constexpr int kTileK = 128;      // K elements per pipeline stage
constexpr int kChunkK = 64;      // K elements per 128-byte swizzle atom of the token tile
constexpr int kTileRows = 128;   // weight rows per tile (MMA M)
constexpr int kGateUpRows = 64;  // gate/up GEMM: 64 gate + 64 up rows per tile
constexpr int kMaxStages = 16;
constexpr int kMaxASlots = 8;
constexpr int kASlotCols = kTileK / 2;  // TMEM columns of one stage's A operand (2 halves per column)

// int4 operands run with K permuted inside every group of 8 elements: stored
// position of element k is 2k for k < 4 and 2(k - 4) + 1 for k >= 4 (order
// 0,4,1,5,2,6,3,7), which lets one lop3 extract a pair of codes. The token
// operands (gathered hidden rows, act cache) are written in that order; the
// product does not change since both operands share it.
template <int BITS>
constexpr bool kPermuteK = BITS == 4;
__host__ __device__ constexpr int permute_k8(int k) {
  return (k & ~7) | ((k & 7) < 4 ? 2 * (k & 7) : 2 * ((k & 7) - 4) + 1);
}

// Programmatic dependent launch: a kernel launched with pdl = true may start
// while the previous kernel of the stream still runs. It must call
// grid_dep_wait() before it touches memory the previous kernels write (the
// wait returns once they have completed and their writes are visible; without
// the launch attribute it returns at once). grid_dep_launch() lets the next
// kernel start once every CTA of this one has issued it or exited, so a
// waiting dependent never holds resources an unscheduled CTA of its
// predecessor needs.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
                          Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct GemmArgs {
  const int32_t* sorted_ids;   // [cap]
  const int32_t* expert_ids;   // [cap / block]
  const int32_t* block_rows;   // [cap / block] routed pairs in each block (the rest is padding)
  const int32_t* num_post_pad; // [1]
  const float* topk_w;         // [P] (down GEMM)
  void* out;                   // act cache [cap, I] (gate/up) or slab [split, P, H] fp32 (down)
  int* status;                 // device status word
  int K;                       // reduction length (H or I)
  int N;                       // rows of one expert's matrix (2I or H)
  int I;                       // gate/up GEMM: first up row; down GEMM: unused
  int E;
  int n_tiles;                 // weight-row tiles per expert
  int topk;
  int P;                       // M * topk
  int block;                   // align block = token tile (MMA N)
  int groups;                  // K / G
  int G;                       // quantization group size along K (a multiple of 64)
  int kt_total;                // ceil(K / 128) stages
  int split;                   // K splits (down GEMM), 1 otherwise
  int has_zeros;
  int max_blocks;              // cap / block
  int panel;                   // token blocks per panel of the work-unit order
  const uint8_t* wpack;        // prepacked weights (stage images), or null: TMA boxes from the plain layout
  int wimg;                    // bytes of one stage image
  int num_stages;
  int num_aslots;
  int num_acc;
  uint32_t tmem_cols;
  float* xs_out;               // deferred-scale gate/up GEMM: token sums of the act cache per down stage
  float* part;                 // deferred-scale gate/up GEMM with split > 1: [tile][block][split][128][nt] fp32
  int* counters;               //   arrivals per (tile, block, lane quarter), zero between calls
  int cap;                     // rows of the expert-sorted token matrices
  const void* bias;            // gate/up: [E, 2I], down: [E, H], activation dtype; null: none
  int glu;                     // gate/up activation: 0 silu(g) * u, 1 clamped SwiGLU
  float glu_alpha, glu_beta, glu_limit;
  const int32_t* act_pos;      // gate/up GEMM, act-order down weights: [E, I] column of feature f in the act cache
  int pdl;                     // launched as a programmatic dependent of the previous kernel
  float* atomic_out;           // down GEMM: [M, N] fp32 sum over slots and K splits by atomicAdd
                               // (null: the ordered slab)
};

// One weight stage in shared memory: packed codes of 128 rows x 128 K, then up
// to two group rows of 128 scales (512 B), then up to two group rows of zero
// points (<= 256 B), each part 128-byte aligned (TMA destinations). The token
// ring after the weight ring is 1 KB aligned (128-byte-swizzle atoms).
__host__ __device__ constexpr int weight_code_bytes(int bits) { return kTileRows * kTileK * bits / 8; }
__host__ __device__ constexpr int weight_stage_bytes(int bits) { return weight_code_bytes(bits) + 512 + 512; }
__host__ __device__ constexpr int weight_ring_bytes(int bits, int stages) {
  return (stages * weight_stage_bytes(bits) + 1023) / 1024 * 1024;
}
__host__ __device__ constexpr int token_stage_bytes(int block) { return (kTileK / kChunkK) * block * 128; }

// Prepacked weights (wna16_prepack): for every (expert, 128-row tile, 128-wide
// K stage) one contiguous image, byte-identical to the shared-memory stage the
// TMA boxes of the plain layout produce (same swizzle, zero fill outside the
// matrix): codes, then the stage's group rows of scales (sg x 256 B), then
// their zero points (sg x 128/pf x 4 B) if the weights have them. sg = 2 for
// G = 64, else 1 (a group of G > 128 repeats its scales in each of its stages).
__host__ __device__ constexpr int prepack_sg(int group_size_or_k) { return group_size_or_k == 64 ? 2 : 1; }
__host__ __device__ constexpr int prepack_image_bytes(int bits, int sg, int has_zeros) {
  return weight_code_bytes(bits) + sg * 256 + (has_zeros ? sg * (kTileRows * bits / 32) * 4 : 0);
}


// Fixed extras after the two rings: barriers and flags.
__host__ __device__ constexpr int gemm_extra_bytes() { return 8 * (2 * kMaxStages + kMaxASlots + 4 + 1) + 64; }
__host__ __device__ constexpr int gemm_smem_bytes(int bits, int block, int stages) {
  return 1024 /* base alignment slack */ + weight_ring_bytes(bits, stages) + stages * token_stage_bytes(block) +
         gemm_extra_bytes();
}

// Deferred-scale kernel (16- or 32-token tiles): ring stages of weights, tokens
// and per-stage token sums (4 parts x nt floats for the gate/up GEMM, 16 parts
// for the down GEMM), two correction-operand tiles (nt rows of 128 B) and
// barriers.
__host__ __device__ constexpr bool defer_tile(int block) { return block == 16 || block == 32; }
__host__ __device__ constexpr int defer_xs_parts(int gemm) { return gemm == 1 ? 4 : 16; }
__host__ __device__ constexpr int defer_smem_bytes(int bits, int gemm, int nt, int stages) {
  return 1024 + weight_ring_bytes(bits, stages) + stages * token_stage_bytes(nt) + 2 * nt * 128 +
         stages * defer_xs_parts(gemm) * nt * 4 + 8 * (2 * stages + 8) + 64;
}

}  // namespace wna16
