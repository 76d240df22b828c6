// Grouped expert GEMM with in-kernel dequantization of packed int4/int8 weights,
// on the sm_103a tensor cores (tcgen05, A operand in tensor memory).
//
// One launch covers every expert (vLLM PR #12185: one fused launch instead of
// one GEMM per expert). Work unit = (token block of the align output, tile of
// weight rows, K split). The token block holds `block` expert-sorted (token,
// slot) pairs, all routed to the same expert, so one unit is a dense
//     D[128 rows, block tokens] = Wdeq[128 rows, K] * X[block tokens, K]^T
// with the dequantized weights as the MMA A operand (M = 128) and the tokens as
// the B operand (N = block). Swapping the operands this way keeps M = 128 even
// for a single decode token.
//
// Pipeline per CTA (persistent over units; every wait is time-bounded):
//   TMA producer:  per 128-wide K stage, the packed codes of 128 weight rows,
//                  their scales and zero points, and the stage's token tile
//                  (two 64-wide K chunks of the block's rows) -> ring slot s
//                  (full[s])
//   dequant warps: two warpgroups taking alternate stages: smem codes ->
//                  round((u - z) * s) in fp16/bf16 -> tcgen05.st into a TMEM
//                  A slot (afull)
//   MMA warp:      8 x tcgen05.mma K=16 per stage, N = the block's routed
//                  pairs rounded up to 16; commits empty[s] (frees the ring
//                  slot and the stage's A slot) and, per unit, accfull
//   epilogue:      four warps: TMEM accumulator -> silu(gate)*up -> act cache
//                  (gate/up GEMM), or * top-k weight -> fp32 slab row (down)
// A K stage spans 128 elements inside one quantization group, or two groups
// of 64 (group size 64 or a multiple of 128): the per-stage scale rows are
// those of the groups the stage covers (the BLOCK_SIZE_K vs group-size hazard
// reported on vLLM PR #6502 cannot occur).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "plan.cuh"
#include "ptx.cuh"

namespace wna16 {

template <int ACT>
struct Act;
template <>
struct Act<0> {
  using T = __half;
  using T2 = __half2;
};
template <>
struct Act<1> {
  using T = __nv_bfloat16;
  using T2 = __nv_bfloat162;
};

// Bias of row `row` of expert e's matrix (activation dtype, as fp32).
template <int ACT>
__device__ __forceinline__ float bias_of(const GemmArgs& a, int e, int row) {
  const auto* b = static_cast<const typename Act<ACT>::T*>(a.bias);
  if constexpr (ACT == 0) return __half2float(b[static_cast<size_t>(e) * a.N + row]);
  else return __bfloat162float(b[static_cast<size_t>(e) * a.N + row]);
}

// The gate/up activation: silu(g) * u, or (a.glu) the clamped SwiGLU
// g' sigmoid(alpha g') (u' + beta) with g' = min(g, L), u' = clamp(u, -L, L)
// for L = a.glu_limit > 0 (no clamp otherwise).
__device__ __forceinline__ float gate_up_act(const GemmArgs& a, float g, float u) {
  if (!a.glu) return g / (1.0f + __expf(-g)) * u;
  if (a.glu_limit > 0.f) {
    g = fminf(g, a.glu_limit);
    u = fminf(fmaxf(u, -a.glu_limit), a.glu_limit);
  }
  return g / (1.0f + __expf(-a.glu_alpha * g)) * (u + a.glu_beta);
}

__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(b), "r"(c));  // (a & b) | c
  return d;
}

template <int ACT>
__device__ __forceinline__ uint32_t pack2_rn(float lo, float hi) {
  if constexpr (ACT == 0) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

template <int ACT>
__device__ __forceinline__ uint32_t hsub_hmul(uint32_t v, uint32_t zc, uint32_t sc) {
  using T2 = typename Act<ACT>::T2;
  T2 r = __hmul2(__hsub2(*reinterpret_cast<T2*>(&v), *reinterpret_cast<T2*>(&zc)),
                 *reinterpret_cast<T2*>(&sc));
  return *reinterpret_cast<uint32_t*>(&r);
}

// Exact (code - zero) as fp32: 2^23 + code has the code in its low mantissa bits.
__device__ __forceinline__ float code_minus_zero(uint32_t code, float magic_plus_zero) {
  return __uint_as_float(0x4B000000u | code) - magic_plus_zero;
}

// Dequantizes 32 consecutive K elements of one weight row into 16 packed
// pairs. int8: natural order, out[c] = (element 2c, element 2c+1). int4: each
// word of 8 codes k0..k7 yields the pairs (k0,k4), (k1,k5), (k2,k6), (k3,k7),
// so the operand's K order inside every group of 8 is 0,4,1,5,2,6,3,7 (the
// token operand is stored in the same order; see kPermuteK). Every value is
// round((u - z) * s) to the activation dtype, rounded once: the subtraction of
// the magic-number forms is exact and the multiply rounds once, and in the fp32
// path the product of a <= 8-bit integer and a 16-bit scale is exact.
template <int BITS, int ACT, int SCL>
struct Dequant {
  static __device__ __forceinline__ void run(const uint32_t* w, uint32_t zero, uint32_t scale_bits,
                                             uint32_t (&out)[16]) {
    if constexpr (BITS == 4 && ACT == 0 && SCL == 0) {
      // A nibble OR-ed into bits 0-3 of 1024.0 is exactly 1024 + u; one OR-ed
      // into bits 4-7 of 64.0 is exactly 64 + u. One lop3 per pair extracts
      // (k_j, k_j+4) from bits 4j.. of the word and of the word >> 8.
      const uint32_t z_lo = pack2_rn<0>(1024.f + float(zero), 1024.f + float(zero));
      const uint32_t z_hi = pack2_rn<0>(64.f + float(zero), 64.f + float(zero));
      const uint32_t sc = (scale_bits & 0xFFFFu) | (scale_bits << 16);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t x = w[i];
        const uint32_t x8 = x >> 8;
        out[i * 4 + 0] = hsub_hmul<0>(lop3_and_or(x, 0x000F000Fu, 0x64006400u), z_lo, sc);   // k0, k4
        out[i * 4 + 1] = hsub_hmul<0>(lop3_and_or(x, 0x00F000F0u, 0x54005400u), z_hi, sc);   // k1, k5
        out[i * 4 + 2] = hsub_hmul<0>(lop3_and_or(x8, 0x000F000Fu, 0x64006400u), z_lo, sc);  // k2, k6
        out[i * 4 + 3] = hsub_hmul<0>(lop3_and_or(x8, 0x00F000F0u, 0x54005400u), z_hi, sc);  // k3, k7
      }
    } else if constexpr (BITS == 4 && ACT == 1 && SCL == 1) {
      // bf16: a nibble in bits 0-3 of 128.0 is exactly 128 + u (bits 4-7 would
      // reach the exponent), so each pair is shifted down first.
      const uint32_t zc = pack2_rn<1>(128.f + float(zero), 128.f + float(zero));
      const uint32_t sc = (scale_bits & 0xFFFFu) | (scale_bits << 16);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint32_t x = w[i];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          out[i * 4 + j] = hsub_hmul<1>(lop3_and_or(x >> (4 * j), 0x000F000Fu, 0x43004300u), zc, sc);
      }
    } else if constexpr (BITS == 8 && ACT == 0 && SCL == 0) {
      const uint32_t zc = pack2_rn<0>(1024.f + float(zero), 1024.f + float(zero));
      const uint32_t sc = (scale_bits & 0xFFFFu) | (scale_bits << 16);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const uint32_t x = w[i];
        out[i * 2 + 0] = hsub_hmul<0>(__byte_perm(x, 0x64646464u, 0x4140), zc, sc);
        out[i * 2 + 1] = hsub_hmul<0>(__byte_perm(x, 0x64646464u, 0x4342), zc, sc);
      }
    } else {
      // General path (int8 with bf16, or scale dtype != activation dtype):
      // exact (u - z) in fp32, exact product, one rounding to the act dtype.
      const float s = SCL == 0 ? __half2float(__ushort_as_half((unsigned short)scale_bits))
                               : __bfloat162float(__ushort_as_bfloat16((unsigned short)scale_bits));
      const float mz = 8388608.f + float(zero);
      constexpr uint32_t MASK = (1u << BITS) - 1;
#pragma unroll
      for (int i = 0; i < BITS; ++i) {  // 4 words of int4 or 8 words of int8
        const uint32_t x = w[i];
        if constexpr (BITS == 4) {
#pragma unroll
          for (int j = 0; j < 4; ++j) {  // pairs (k_j, k_j+4)
            const float f0 = code_minus_zero((x >> (4 * j)) & MASK, mz) * s;
            const float f1 = code_minus_zero((x >> (4 * (j + 4))) & MASK, mz) * s;
            out[i * 4 + j] = pack2_rn<ACT>(f0, f1);
          }
        } else {
          // one prmt puts byte c into the low mantissa bits of 2^23 (0x4B0000uu)
#pragma unroll
          for (int c = 0; c < 4; c += 2) {
            const float f0 = (__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7440 + c)) - mz) * s;
            const float f1 = (__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7440 + c + 1)) - mz) * s;
            out[(i * 4 + c) / 2] = pack2_rn<ACT>(f0, f1);
          }
        }
      }
    }
  }
};

__device__ __forceinline__ int unit_expert(const GemmArgs& a, int blk) {
  return clamp_expert(a.expert_ids[blk], a.E);  // blocks below num_post_pad always hold a valid id
}

// The same read from L2 (the align kernel's output, read by a kernel that may
// have started before its predecessor finished).
__device__ __forceinline__ int unit_expert_l2(const GemmArgs& a, int blk) {
  return clamp_expert(__ldcg(a.expert_ids + blk), a.E);
}

// Epilogue of one work unit, run by four warps covering the four TMEM lane
// quarters: waits for the unit's accumulator, reads it 16 token columns at a
// time and writes silu(gate) * up to the act cache (gate/up GEMM) or the
// top-k-weighted fp32 row of each (token, slot) pair (down GEMM), then frees
// the accumulator. Returns false if the wait gave up.
template <int BITS, int ACT, int GEMM, int EXT>
__device__ __forceinline__ bool epilogue_unit(const GemmArgs& a, const Unit& w, uint32_t tmem, int acc,
                                              uint32_t acc_phase, uint64_t* accfull, uint64_t* accempty,
                                              volatile int* abort_flag, int q, int lane) {
  const int NT = a.block;
  // token columns the unit's MMAs wrote: the block's routed pairs, rounded up to 16
  const int ncols = trimmed_n(a.block_rows[w.blk], NT);
  if (!warp_wait_all(&accfull[acc], acc_phase, abort_flag, a.status)) return false;
  tc_fence_after();
  const uint32_t t_base = tmem + ((q * 32) << 16) + gemm_acc_col(acc, NT);
  // bias of this lane's row: gate/up GEMM, gate row f (lanes 0-15) or up row
  // I + f (16-31); down GEMM, row h, added by the first K split only
  float bias = 0.f;
  bool has_bias = false;
  // gate/up GEMM: the act-cache column of this lane's feature in the down
  // GEMM's K order (act-order position, then the int4 pair order)
  int fp = 0;
  bool fp_ok = true;
  if (GEMM == 1) {
    const int f = w.tile * kGateUpRows + 16 * q + (lane & 15);
    int pos = f;
    if (EXT && a.act_pos) {
      pos = a.act_pos[static_cast<size_t>(unit_expert(a, w.blk)) * a.I + f];
      fp_ok = static_cast<unsigned>(pos) < static_cast<unsigned>(a.I);
    }
    fp = kPermuteK<BITS> ? permute_k8(pos) : pos;
  }
  if (EXT && a.bias) {
    const int e = unit_expert(a, w.blk);
    if (GEMM == 1) {
      const int f = w.tile * kGateUpRows + 16 * q + (lane & 15);
      bias = bias_of<ACT>(a, e, lane < 16 ? f : a.I + f);
      has_bias = true;
    } else {
      const int h = w.tile * kTileRows + q * 32 + lane;
      has_bias = w.sp == 0 && h < a.N;
      if (has_bias) bias = bias_of<ACT>(a, e, h);
    }
  }
  for (int c0 = 0; c0 < ncols; c0 += 16) {
    uint32_t v[16];
    tmem_ld16(t_base + c0, v);
    tmem_ld_wait(v);
    if (has_bias) {
#pragma unroll
      for (int j = 0; j < 16; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) + bias);
    }
    if (GEMM == 1) {
      // Lanes 0-15 of this quarter hold gate rows, lanes 16-31 the up rows of
      // the same 16 features; swap halves so each lane owns 8 (feature, token)
      // pairs with both values.
      using T = typename Act<ACT>::T;
      T* act = reinterpret_cast<T*>(a.out);
      const bool lo = lane < 16;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t mine = lo ? v[j] : v[j + 8];
        const uint32_t other = __shfl_xor_sync(0xFFFFFFFFu, lo ? v[j + 8] : v[j], 16);
        const float g = __uint_as_float(lo ? mine : other);
        const float up = __uint_as_float(lo ? other : mine);
        const float val = EXT ? gate_up_act(a, g, up) : g / (1.0f + __expf(-g)) * up;
        const int col = c0 + (lo ? j : j + 8);
        if (!fp_ok) continue;
        const size_t idx = act_index(w.blk, NT, col, a.I, fp);
        if constexpr (ACT == 0)
          act[idx] = __float2half_rn(val);
        else
          act[idx] = __float2bfloat16_rn(val);
      }
    } else {
      float* slab = reinterpret_cast<float*>(a.out);
      const int h = w.tile * kTileRows + q * 32 + lane;
      const int my_pid = a.sorted_ids[w.blk * NT + c0 + (lane & 15)];
      const float my_w = (my_pid >= 0 && my_pid < a.P) ? a.topk_w[my_pid] : 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int pid = __shfl_sync(0xFFFFFFFFu, my_pid, j);
        const float tw = __shfl_sync(0xFFFFFFFFu, my_w, j);
        if (pid >= 0 && pid < a.P && h < a.N) {
          if (EXT && a.atomic_out)  // unordered fp32 sum over the token's slots and the K splits
            atomicAdd(a.atomic_out + static_cast<size_t>(pid / a.topk) * a.N + h, __uint_as_float(v[j]) * tw);
          else
            slab[slab_index(w.sp, a.P, pid, a.N, h)] = __uint_as_float(v[j]) * tw;
        }
      }
    }
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(&accempty[acc]);
  return true;
}

// LEAN = 0: 14 warps (producer, MMA issuer, 4 epilogue warps, two dequant
// warpgroups), two CTAs per SM. LEAN = 1: 6 warps (producer, MMA issuer, one
// dequant warpgroup that also runs the epilogue), four CTAs per SM, so four
// MMA-issuing threads share the SM's tensor core (decode-sized token tiles).
//
// EXT = 1: the instantiations that also serve prepacked weights, biases, the
// clamped SwiGLU and act-order; EXT = 0 carries none of that code (the
// register-bound dequant loop was measurably slower with it).
template <int BITS, int ACT, int SCL, int GEMM, int LEAN, int EXT>
__global__ void __launch_bounds__(gemm_threads(LEAN), LEAN ? 4 : 2)
    moe_gemm_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_s,
                    const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_b,
                    const GemmArgs a) {
  constexpr int PF = 32 / BITS;
  constexpr int KW = kTileK * BITS / 32;  // int32 words per row per stage
  constexpr int W_BYTES = weight_code_bytes(BITS);
  constexpr int S_OFF = W_BYTES;          // [SG][128] scales (gate/up: [SG][2 halves][64])
  constexpr int Z_OFF = W_BYTES + 512;    // [SG][128 / PF] zero words (gate/up: [SG][2][64 / PF])
  constexpr int WST = weight_stage_bytes(BITS);
  constexpr uint32_t ZMASK = (1u << BITS) - 1;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int NS = a.num_stages, NA = a.num_aslots, NACC = a.num_acc, NT = a.block;
  const int BST = token_stage_bytes(NT);
  const int SG = a.G < kTileK ? kTileK / a.G : 1;  // group rows per stage (G = 64 -> 2)

  const SmemLayout sl = gemm_smem_layout(BITS, NT, NS, NA, NACC);
  uint8_t* wring = smem + sl.wring;
  uint8_t* bring = smem + sl.bring;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + sl.bars);  // stage landed: codes, scales, zeros, token tile
  uint64_t* empty = full + NS;       // stage consumed: its MMAs completed (also frees its A slot)
  uint64_t* afull = empty + NS;      // A slot written by a dequant warpgroup
  uint64_t* accfull = afull + NA;    // accumulator ready for the epilogue
  uint64_t* accempty = accfull + NACC;
  uint64_t* drain = accempty + NACC;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + sl.holder);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + sl.abort_flag);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int i = 0; i < NA; ++i) mbar_init(&afull[i], kDequantWarps / 2);  // one warpgroup per stage
    for (int i = 0; i < NACC; ++i) {
      mbar_init(&accfull[i], 1);
      mbar_init(&accempty[i], kEpilogueWarps);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    if (!(EXT && a.wpack)) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_s);
      if (a.has_zeros) prefetch_tmap(&tm_z);
    }
    prefetch_tmap(&tm_b);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, a.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // the setup above overlaps the previous kernel; its outputs are read below
  grid_dep_wait();
  grid_dep_launch();

  const int nb = active_blocks(*a.num_post_pad, NT, a.max_blocks);
  const int units = nb * a.n_tiles * a.split;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // Per stage: codes of 128 rows (gate/up: one 3D box holding the 64 gate and
    // the 64 up rows), their scales and zero points (one box each), and the two
    // 64-wide K chunks of the token tile: five copies for 8-16 KB of codes.
    // The whole warp runs the loop (waits are warp-wide polls); one elected
    // lane issues the copies.
    const uint32_t stage_tx = weight_stage_tx(BITS, SG, a.has_zeros, (EXT && a.wpack) ? a.wimg : 0) + BST;
    const uint64_t pol_w = l2_policy_evict_first();  // weights: streamed once
    const uint64_t pol_b = l2_policy_evict_last();   // token rows: re-read by every row tile
    int it = 0, s = 0;
    uint32_t e_phase = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const Unit w = decode_unit(u, nb, a);
      const int e = unit_expert(a, w.blk);
      bool ok = true;
      for (int kt = w.kt0; kt < w.kt1; ++kt, ++it) {
        if (!warp_wait_all(&empty[s], e_phase ^ 1u, abort_flag, a.status)) { ok = false; break; }
        if (elect_one()) {
          mbar_arrive_expect_tx(&full[s], stage_tx);
          uint8_t* dst = wring + s * WST;
          const int ys = stage_group_row(a, e, kt);
          if (EXT && a.wpack) {
            // prepacked: the stage's codes, scales and zero points as one image
            bulk_load(dst, a.wpack + image_offset(a, e, w.tile, kt), a.wimg, &full[s], pol_w);
          } else {
            const StageCoords c = weight_stage_coords(GEMM, BITS, a, w.tile, e, kt, ys);
            if (GEMM == 1) {
              tma_load_3d(dst, &tm_q, &full[s], c.q[0], c.q[1], c.q[2], pol_w);
              tma_load_3d(dst + S_OFF, &tm_s, &full[s], c.s[0], c.s[1], c.s[2], pol_w);
              if (a.has_zeros) tma_load_3d(dst + Z_OFF, &tm_z, &full[s], c.z[0], c.z[1], c.z[2], pol_w);
            } else {
              tma_load_2d(dst, &tm_q, &full[s], c.q[0], c.q[1], pol_w);
              tma_load_2d(dst + S_OFF, &tm_s, &full[s], c.s[0], c.s[1], pol_w);
              if (a.has_zeros) tma_load_2d(dst + Z_OFF, &tm_z, &full[s], c.z[0], c.z[1], pol_w);
            }
          }
          // token tile: the block's rows of the expert-sorted token matrix
#pragma unroll
          for (int c = 0; c < kTileK / kChunkK; ++c)
            tma_load_2d(bring + s * BST + c * NT * 128, &tm_b, &full[s], token_x(kt, c), token_y(w.blk, NT), pol_b);
        }
        __syncwarp();
        if (++s == NS) {
          s = 0;
          e_phase ^= 1u;
        }
      }
      if (!ok) break;
    }
    // Let every issued copy land before the CTA can exit.
    for (int j = (it > NS ? it - NS : 0); j < it; ++j) wait_bar_drain(&full[j % NS], (j / NS) & 1);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop and one elected lane issues: with the loop
    // values warp-uniform, an 8-MMA stage issues several times faster than from
    // a lone lane. Wrapping counters, precomputed descriptors, unrolled MMAs.
    const uint32_t a_base = tmem + gemm_a_col(NACC, NT, 0);
    const uint64_t chunk_step = static_cast<uint64_t>((NT * 128) >> 4);  // next 64-wide K chunk
    int s = 0, slot = 0, uc = 0;
    uint32_t a_phase = 0;
    bool issued = false;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++uc) {
      const Unit w = decode_unit(u, nb, a);
      const int acc = uc % NACC;
      if (!warp_wait_all(&accempty[acc], ((uc / NACC) & 1) ^ 1, abort_flag, a.status)) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem + gemm_acc_col(acc, NT);
      // MMA width: the block's routed pairs rounded up to 16 (padding skipped)
      const uint32_t idesc = idesc_f16(ACT, trimmed_n(a.block_rows[w.blk], NT));
      bool ok = true;
      for (int kt = w.kt0; kt < w.kt1; ++kt) {
        // afull implies the stage landed (the dequant warps waited on full[s])
        if (!warp_wait_all(&afull[slot], a_phase, abort_flag, a.status)) { ok = false; break; }
        tc_fence_after();
        if (elect_one()) {
          const uint32_t at = a_base + slot * kASlotCols;
          const uint64_t b0 = smem_desc_sw128(smem_u32(bring + s * BST));
          const uint64_t b1 = b0 + chunk_step;
          mma_ts(d_tmem, at, b0, idesc, kt > w.kt0 ? 1u : 0u);
          mma_ts_acc(d_tmem, at + 8, b0 + 2, idesc);  // +32 B per K=16 step
          mma_ts_acc(d_tmem, at + 16, b0 + 4, idesc);
          mma_ts_acc(d_tmem, at + 24, b0 + 6, idesc);
          mma_ts_acc(d_tmem, at + 32, b1, idesc);
          mma_ts_acc(d_tmem, at + 40, b1 + 2, idesc);
          mma_ts_acc(d_tmem, at + 48, b1 + 4, idesc);
          mma_ts_acc(d_tmem, at + 56, b1 + 6, idesc);
          mma_commit(&empty[s]);
        }
        __syncwarp();
        issued = true;
        if (++s == NS) s = 0;
        if (++slot == NA) {
          slot = 0;
          a_phase ^= 1u;
        }
      }
      if (!ok) break;
      if (elect_one()) mma_commit(&accfull[acc]);
      __syncwarp();
    }
    if (issued) {
      if (elect_one()) mma_commit(drain);
      __syncwarp();
      wait_bar_drain(drain, 0);
    }
  } else if (!LEAN && warp < 2 + kEpilogueWarps) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int uc = 0;
    for (int u = blockIdx.x; u < units; u += gridDim.x, ++uc) {
      const Unit w = decode_unit(u, nb, a);
      if (!epilogue_unit<BITS, ACT, GEMM, EXT>(a, w, tmem, uc % NACC, (uc / NACC) & 1, accfull, accempty, abort_flag, q, lane))
        break;
    }
  } else {
    // ------------------------------------------------------------ dequantizers
    // LEAN = 0: two warpgroups, stage-parallel: warpgroup g dequantizes the
    // stages whose running index is congruent to g mod 2, so two stages are in
    // flight. LEAN = 1: one warpgroup takes every stage. One full 128-element K
    // row per thread (thread = TMEM lane = weight row).
    // A slot it % NA is free once the MMAs of stage it - NA completed, which is
    // the completion of that stage's `empty` phase.
    const int q = warp & 3;
    const int grp = LEAN ? 0 : (warp - 2 - kEpilogueWarps) >> 2;
    // Weight row (in the stage's smem tile) of this thread's TMEM lane. Gate/up:
    // lanes 0-15 of quarter q take gate rows 16q.., lanes 16-31 the up rows of
    // the same features, so the epilogue finds gate and up in one warp.
    int srow, half = 0, hrow;
    if (GEMM == 1) {
      half = lane < 16 ? 0 : 1;
      hrow = 16 * q + (lane & 15);
      srow = half * kGateUpRows + hrow;
    } else {
      srow = q * 32 + lane;
      hrow = srow;
    }
    const uint32_t t_lane = (q * 32) << 16;
    const int z_off = (EXT && a.wpack) ? W_BYTES + SG * 256 : Z_OFF;  // zero points: right after the scales in an image
    // This group's stages are the running stage indices gi = grp, grp + step,
    // ... across units (step 2, or 1 for LEAN). Tracked incrementally: the ring
    // slot cs and phase cf of stage gi, its A slot cslot, and the ring slot cps
    // and phase cp of stage gi - NA, whose completed MMAs free that A slot
    // (floor division, so the tracking stays consistent through gi < NA).
    constexpr int step = LEAN ? 1 : 2;  // the ring has NS >= 2 stages, so one wrap suffices for cs, cps
    const int pfirst = grp - NA;
    int cs = grp % NS, cslot = grp % NA, gi = grp;
    int cps = ((pfirst % NS) + NS) % NS;
    uint32_t cf = (grp / NS) & 1u;
    uint32_t cp = static_cast<uint32_t>((pfirst >= 0 ? pfirst / NS : (pfirst - NS + 1) / NS) & 1);
    int it = 0;  // running index of the current unit's first stage
    int uc = 0;  // units finished (epilogue count, LEAN)
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const Unit w = decode_unit(u, nb, a);
      const int n = w.kt1 - w.kt0;
      bool ok = true;
      for (; gi < it + n; gi += step) {
        if (!warp_wait_all(&full[cs], cf, abort_flag, a.status)) { ok = false; break; }
        if (gi >= NA) {
          if (!warp_wait_all(&empty[cps], cp, abort_flag, a.status)) { ok = false; break; }
        }
        const uint8_t* st = wring + cs * WST;
        // scale and zero point of each 64-wide chunk of the stage (group rows 0/1 when G = 64)
        uint32_t sbits[2], zero[2];
#pragma unroll
        for (int c = 0; c < 2; ++c) {
          const int gr = SG == 2 ? c : 0;
          const int si = GEMM == 1 ? (gr * 2 + half) * kGateUpRows + hrow : gr * kTileRows + hrow;
          sbits[c] = reinterpret_cast<const uint16_t*>(st + S_OFF)[si];
          zero[c] = 1u << (BITS - 1);
          if (a.has_zeros) {
            const int zi = GEMM == 1 ? (gr * 2 + half) * (kGateUpRows / PF) + hrow / PF
                                     : gr * (kTileRows / PF) + hrow / PF;
            zero[c] = (reinterpret_cast<const uint32_t*>(st + z_off)[zi] >> (BITS * (hrow % PF))) & ZMASK;
          }
        }
        // Code rows are TMA-swizzled (64-byte rows: 16-byte chunk c of row r sits at
        // chunk c ^ ((r >> 1) & 3); 128-byte rows: at c ^ (r & 7)), so the 8 lanes
        // of a load phase, 8 consecutive rows, hit distinct banks.
        const uint4* src = reinterpret_cast<const uint4*>(st + srow * KW * 4);
        const int swz = BITS == 4 ? ((srow >> 1) & 3) : (srow & 7);
#pragma unroll
        for (int h = 0; h < 4; ++h) {  // four 32-element quarters of the row
          uint32_t wv[BITS];
#pragma unroll
          for (int i = 0; i < BITS / 4; ++i) {
            const uint4 x = src[(h * (BITS / 4) + i) ^ swz];
            wv[4 * i + 0] = x.x;
            wv[4 * i + 1] = x.y;
            wv[4 * i + 2] = x.z;
            wv[4 * i + 3] = x.w;
          }
          uint32_t outv[16];
          Dequant<BITS, ACT, SCL>::run(wv, zero[h >> 1], sbits[h >> 1], outv);
          tmem_st16(tmem + t_lane + gemm_a_col(NACC, NT, cslot) + h * 16, outv);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&afull[cslot]);
        cs += step;
        if (cs >= NS) {
          cs -= NS;
          cf ^= 1u;
        }
        cps += step;
        if (cps >= NS) {
          cps -= NS;
          cp ^= 1u;
        }
        cslot += step;
        while (cslot >= NA) cslot -= NA;  // NA may be 1 (two 256-token stages): then always slot 0
      }
      it += n;
      if (!ok) break;
      if (LEAN) {
        // this warpgroup also runs the epilogue, right after the unit's last stage
        if (!epilogue_unit<BITS, ACT, GEMM, EXT>(a, w, tmem, uc % NACC, (uc / NACC) & 1, accfull, accempty, abort_flag, q,
                                      lane))
          break;
        ++uc;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();  // the drain wait above is per lane: converge before the .aligned dealloc
    tc_fence_after();
    tmem_dealloc(tmem, a.tmem_cols);
  }
}

}  // namespace wna16
