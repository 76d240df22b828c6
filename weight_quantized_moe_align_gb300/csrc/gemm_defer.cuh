// Grouped expert GEMM for decode-sized token tiles (16 or 32 tokens) with the
// quantization scale and zero point taken out of the per-element work.
//
// For one 128-wide K stage of weight row n (one quantization group, or part of
// one) and token j the layer needs
//     s[n] * sum_k (u[n,k] - z[n]) * x[j,k].
// The A operand is loaded with the exact "magic number" forms of the codes
// (a 4-bit code OR-ed into the mantissa of 1024.0 or 64.0 is exactly 1024 + u
// or 64 + u; bf16: 128 + u; 8-bit codes: 1024 + u), which costs one lop3 or
// prmt per pair of codes and nothing else. The offsets and the zero point
// form a rank-one term, c[n] * X[j] with X[j] the sum of the stage's token
// values (kept apart for even and odd k, which carry the two int4 offsets), and
// one extra K = 16 MMA per stage subtracts it inside the tensor core: A gets
// -c split over a few columns, B the token sums split into fp16/bf16 parts
// that add up to the fp32 sum. Each stage's MMAs write a fresh fp32 partial
// sum to tensor memory; the dequant warps read it back and accumulate
// s[n] * partial in fp32 registers. Compared with dequantizing to
// round((u - z) * s) this is at least as accurate (no rounding of the
// weights) and leaves the dequant warps about a third of the instructions.
//
// Warp roles (10 warps, two CTAs per SM, 256 TMEM columns each):
//   0     TMA producer: codes, scales, zero points, token tile, token sums
//   1     MMA issuer (9 MMAs per stage) and TMEM owner
//   2..5  warpgroup 0: even stages; also the epilogue of every unit
//   6..9  warpgroup 1: odd stages
// Warpgroup g owns A slot g and partial-sum buffer P_g: it dequantizes its
// stage into the slot, builds the stage's correction B rows and signals the
// MMA warp; once its next stage's data has landed it waits for those MMAs and
// folds P_g into its accumulators, then dequantizes that next stage. At a
// unit's end warpgroup 1 hands its accumulators over in TMEM (buffer C) and
// warpgroup 0 runs the epilogue; the gate/up epilogue also writes the token
// sums of its act-cache columns that the down GEMM's correction needs.
//
// Token sums in global memory, fp32, [stage][parts][cap rows]:
//   gate/up GEMM (written by the gather kernel): 4 parts = 64-wide half h of
//     the stage x parity p of k, part 2h + p;
//   down GEMM (written by the gate/up epilogue, one value per warp): 16 parts =
//     half h x lane quarter q x parity p, part 8h + 2q + p.
#pragma once

#include "gemm_kernel.cuh"

namespace wna16 {

constexpr int kDeferThreads = 10 * 32;
// TMEM columns (plan.cuh): P_0 [0,16), P_1 [16,32), C [32,48); A slot g at 64 + 96 g:
// 64 columns for the 128 K of the stage, then 8 columns for the correction.
// Combine buffer C: its own 16 columns at [32, 48) for 16-token tiles; for
// 32-token tiles it is P_1 itself (the TMEM budget has no room for a third
// 32-column buffer), which warpgroup 1 may reuse only after warpgroup 0 took C.

// Codes of 32 consecutive K elements (one 16-column TMEM chunk) in magic-number
// form, same pair order as Dequant (int4: pairs (k_j, k_j+4) of every word).
template <int BITS, int ACT>
__device__ __forceinline__ void codes_to_magic(const uint32_t* w, uint32_t (&out)[16]) {
  if constexpr (BITS == 4 && ACT == 0) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t x = w[i], x8 = x >> 8;
      out[i * 4 + 0] = lop3_and_or(x, 0x000F000Fu, 0x64006400u);   // 1024 + u: k0, k4
      out[i * 4 + 1] = lop3_and_or(x, 0x00F000F0u, 0x54005400u);   // 64 + u:   k1, k5
      out[i * 4 + 2] = lop3_and_or(x8, 0x000F000Fu, 0x64006400u);  // 1024 + u: k2, k6
      out[i * 4 + 3] = lop3_and_or(x8, 0x00F000F0u, 0x54005400u);  // 64 + u:   k3, k7
    }
  } else if constexpr (BITS == 4 && ACT == 1) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t x = w[i];
#pragma unroll
      for (int j = 0; j < 4; ++j) out[i * 4 + j] = lop3_and_or(x >> (4 * j), 0x000F000Fu, 0x43004300u);  // 128 + u
    }
  } else {
    static_assert(BITS == 8 && ACT == 0, "8-bit codes: fp16 activations only");
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      out[i * 2 + 0] = __byte_perm(w[i], 0x64646464u, 0x4140);  // 1024 + u
      out[i * 2 + 1] = __byte_perm(w[i], 0x64646464u, 0x4342);
    }
  }
}

__device__ __forceinline__ uint32_t pack_h2(__half lo, __half hi) {
  return static_cast<uint32_t>(__half_as_ushort(lo)) | (static_cast<uint32_t>(__half_as_ushort(hi)) << 16);
}
__device__ __forceinline__ uint32_t pack_b2(__nv_bfloat16 lo, __nv_bfloat16 hi) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(lo)) | (static_cast<uint32_t>(__bfloat16_as_ushort(hi)) << 16);
}

// The correction term c[n] * X[j] enters the MMA as K positions 0..7:
// A holds -c, B the token sum X, each split so that the products add up to
// c * X to about fp32 precision.
//   fp16: v = X / 32 is split into three parts p1 = fp16(v),
//     p2 = fp16((v - p1) * 2^11), p3 = fp16(((v - p1) * 2^11 - p2) * 2^11),
//     with A = -32c, -c / 64, -c * 2^-17 (all exact in fp16 for the offsets
//     and zero points here). The 1/32 keeps sums of large activations in
//     range; the 2^11 steps keep the lower parts out of the fp16 subnormals
//     for small ones (a plain high/low split underflows there).
//   bf16: X = p1 + p2 + p3 (bf16 has the fp32 exponent range), A = -c.
// int4 fp16 needs the even-k and odd-k sums apart (offsets 1024 and 64):
// positions 0..2 carry the even sum, 3..5 the odd one; every other case uses
// one sum with the single offset in positions 0..2.
template <int BITS, int ACT>
__device__ __forceinline__ void corr_a(uint32_t zero, uint32_t (&c)[8]) {
  // The values are built from their bit patterns: for c = 2^e (1 + m) the
  // scaled copies differ only in the exponent field (z < 2^10 for offset 1024,
  // z < 2^6 for offset 64, z < 2^7 for the bf16 offset 128).
  if constexpr (ACT == 0) {
    // even k: -32 (1024 + z) = 0xF800 | z, -(1024 + z) / 64 = 0xCC00 | z,
    //         -(1024 + z) 2^-17 = 0xA000 | z
    c[0] = 0xCC00F800u | (zero * 0x10001u);
    if constexpr (BITS == 4) {
      // odd k: -32 (64 + z) = 0xE800 | z << 4, -(64 + z) / 64 = 0xBC00 | z << 4,
      //        -(64 + z) 2^-17 = 0x9000 | z << 4
      c[1] = 0xE800A000u | (zero << 20) | zero;
      c[2] = 0x9000BC00u | ((zero << 4) * 0x10001u);
    } else {
      c[1] = 0x0000A000u | zero;
    }
  } else {
    const uint32_t v = 0xC300u | zero;  // -(128 + z) in bf16
    c[0] = v * 0x10001u;
    c[1] = v;
  }
}

__device__ __forceinline__ void split3_f16(float x, __half& p1, __half& p2, __half& p3) {
  const float v = x * (1.f / 32.f);
  p1 = __float2half_rn(v);
  const float r1 = (v - __half2float(p1)) * 2048.f;
  p2 = __float2half_rn(r1);
  p3 = __float2half_rn((r1 - __half2float(p2)) * 2048.f);
}

// B-side correction of one token: K positions 0..7 as four packed pairs.
template <int BITS, int ACT>
__device__ __forceinline__ void corr_b(float xe, float xo, uint32_t (&b)[4]) {
  if constexpr (ACT == 0) {
    if constexpr (BITS == 4) {
      __half e1, e2, e3, o1, o2, o3;
      split3_f16(xe, e1, e2, e3);
      split3_f16(xo, o1, o2, o3);
      b[0] = pack_h2(e1, e2);
      b[1] = pack_h2(e3, o1);
      b[2] = pack_h2(o2, o3);
      b[3] = 0u;
    } else {
      __half p1, p2, p3;
      split3_f16(xe + xo, p1, p2, p3);
      b[0] = pack_h2(p1, p2);
      b[1] = pack_h2(p3, __float2half_rn(0.f));
      b[2] = b[3] = 0u;
    }
  } else {
    const float v = xe + xo;
    const __nv_bfloat16 p1 = __float2bfloat16_rn(v);
    const float r1 = v - __bfloat162float(p1);
    const __nv_bfloat16 p2 = __float2bfloat16_rn(r1);
    const __nv_bfloat16 p3 = __float2bfloat16_rn(r1 - __bfloat162float(p2));
    b[0] = pack_b2(p1, p2);
    b[1] = pack_b2(p3, __float2bfloat16_rn(0.f));
    b[2] = b[3] = 0u;
  }
}

template <int SCL>
__device__ __forceinline__ float scale_to_f32(uint32_t bits) {
  if constexpr (SCL == 0) return __half2float(__ushort_as_half(static_cast<unsigned short>(bits)));
  else return __bfloat162float(__ushort_as_bfloat16(static_cast<unsigned short>(bits)));
}

// VAR = 1: prepacked weights and the model-variant epilogues (biases, clamped
// SwiGLU), a separate instantiation so that the default one keeps its
// register allocation.
template <int BITS, int ACT, int SCL, int GEMM, int NT, int VAR>
__global__ void __launch_bounds__(kDeferThreads, 2)
    moe_gemm_defer_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_s,
                          const __grid_constant__ CUtensorMap tm_z, const __grid_constant__ CUtensorMap tm_b,
                          const __grid_constant__ CUtensorMap tm_x, const GemmArgs a) {
  static_assert(NT == 16 || NT == 32, "deferred-scale token tiles: 16 or 32");
  constexpr int PF = 32 / BITS;
  constexpr int KW = kTileK * BITS / 32;
  constexpr int W_BYTES = weight_code_bytes(BITS);
  constexpr int S_OFF = W_BYTES;
  constexpr int Z_OFF = W_BYTES + 512;
  constexpr int WST = weight_stage_bytes(BITS);
  constexpr int BST = token_stage_bytes(NT);
  constexpr int XPARTS = defer_xs_parts(GEMM);
  constexpr int XST = XPARTS * NT * 4;
  constexpr uint32_t ZMASK = (1u << BITS) - 1;

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int NS = a.num_stages;

  const SmemLayout sl = defer_smem_layout(BITS, GEMM, NT, NS);
  uint8_t* wring = smem + sl.wring;
  uint8_t* bring = smem + sl.bring;
  uint8_t* bcorr = smem + sl.bcorr;                          // 2 tiles of NT rows x 128 B
  float* xring = reinterpret_cast<float*>(smem + sl.xring);  // NS x [XPARTS][NT]
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + sl.bars);
  uint64_t* empty = full + NS;
  uint64_t* afull = empty + NS;  // [2]
  uint64_t* pfull = afull + 2;   // [2]
  uint64_t* cfull = pfull + 2;
  uint64_t* cempty = cfull + 1;
  uint64_t* drain = cempty + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(smem + sl.holder);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + sl.abort_flag);

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int g = 0; g < 2; ++g) {
      mbar_init(&afull[g], 4);
      mbar_init(&pfull[g], 1);
    }
    mbar_init(cfull, 4);
    mbar_init(cempty, 4);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    if (!(VAR && a.wpack)) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_s);
      if (a.has_zeros) prefetch_tmap(&tm_z);
    }
    prefetch_tmap(&tm_b);
    prefetch_tmap(&tm_x);
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, kDeferTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  // The setup above overlaps the previous kernel. The align kernel's outputs
  // (block count, expert of each block) were complete before the previous
  // kernel started: read from L2 without waiting. Everything the previous
  // kernel writes is read after grid_dep_wait().
  const int nb = active_blocks(__ldcg(a.num_post_pad), NT, a.max_blocks);
  const int units = nb * a.n_tiles * a.split;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    const uint32_t stage_tx = weight_stage_tx(BITS, 1, a.has_zeros, (VAR && a.wpack) ? a.wimg : 0) + BST + XST;
    const uint64_t pol_w = l2_policy_evict_first();
    const uint64_t pol_b = l2_policy_evict_last();
    int it = 0, s = 0;
    uint32_t e_phase = 0;
    // stages per quantization group: G is a multiple of 128, or the whole K
    // (per-channel scales, one group), where rounding up keeps every stage in it
    const int spg = (a.G + kTileK - 1) / kTileK;
    // weight part of a stage: codes, scales, zero points (no dependence on the
    // previous kernel) / token part: the token tile and its sums (written by it)
    auto load_weights = [&](int s, const Unit& w, int e, int kt, int ys) {
      uint8_t* dst = wring + s * WST;
      if (VAR && a.wpack) {
        // prepacked: the stage's codes, scales and zero points as one image
        bulk_load(dst, a.wpack + image_offset(a, e, w.tile, kt), a.wimg, &full[s], pol_w);
        return;
      }
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
    };
    auto load_tokens = [&](int s, const Unit& w, int kt) {
#pragma unroll
      for (int c = 0; c < kTileK / kChunkK; ++c)
        tma_load_2d(bring + s * BST + c * NT * 128, &tm_b, &full[s], token_x(kt, c), token_y(w.blk, NT), pol_b);
      tma_load_3d(xring + s * (XST / 4), &tm_x, &full[s], token_y(w.blk, NT), 0, kt, pol_b);
    };
    // The first ring's worth of weight stages is requested before waiting for
    // the previous kernel (its slots are fresh); their token parts follow the
    // wait, in the main loop.
    int pre = 0;
    for (int u = blockIdx.x; u < units && pre < NS; u += gridDim.x) {
      const Unit w = decode_unit(u, nb, a);
      const int e = unit_expert_l2(a, w.blk);
      int ys = e * a.groups + w.kt0 / spg, gk = w.kt0 % spg;
      for (int kt = w.kt0; kt < w.kt1 && pre < NS; ++kt, ++pre) {
        if (elect_one()) {
          mbar_arrive_expect_tx(&full[pre], stage_tx);
          load_weights(pre, w, e, kt, ys);
        }
        __syncwarp();
        if (++gk == spg) {
          gk = 0;
          ++ys;
        }
      }
    }
    grid_dep_wait();
    grid_dep_launch();
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const Unit w = decode_unit(u, nb, a);
      const int e = unit_expert_l2(a, w.blk);
      // scale / zero-point row of the current stage, advanced per group
      int ys = e * a.groups + w.kt0 / spg, gk = w.kt0 % spg;
      bool ok = true;
      for (int kt = w.kt0; kt < w.kt1; ++kt, ++it) {
        if (it >= pre && !warp_wait_all(&empty[s], e_phase ^ 1u, abort_flag, a.status)) { ok = false; break; }
        if (elect_one()) {
          if (it >= pre) {
            mbar_arrive_expect_tx(&full[s], stage_tx);
            load_weights(s, w, e, kt, ys);
          }
          load_tokens(s, w, kt);
        }
        __syncwarp();
        if (++s == NS) {
          s = 0;
          e_phase ^= 1u;
        }
        if (++gk == spg) {
          gk = 0;
          ++ys;
        }
      }
      if (!ok) break;
    }
    for (int j = (it > NS ? it - NS : 0); j < it; ++j) wait_bar_drain(&full[j % NS], (j / NS) & 1);
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    grid_dep_wait();
    grid_dep_launch();
    const uint32_t idesc = idesc_f16(ACT, NT);
    const uint64_t chunk_step = static_cast<uint64_t>((NT * 128) >> 4);
    const uint64_t bc0 = smem_desc_sw128(smem_u32(bcorr));
    const uint64_t bc1 = smem_desc_sw128(smem_u32(bcorr + NT * 128));
    int it = 0, s = 0;
    bool issued = false;
    for (int u = blockIdx.x; u < units; u += gridDim.x) {
      const Unit w = decode_unit(u, nb, a);
      bool ok = true;
      for (int kt = w.kt0; kt < w.kt1; ++kt, ++it) {
        const int g = it & 1;
        if (!warp_wait_all(&afull[g], (it >> 1) & 1, abort_flag, a.status)) { ok = false; break; }
        tc_fence_after();
        if (elect_one()) {
          const uint32_t d = tmem + defer_p_col(g, NT);
          const uint32_t at = tmem + defer_a_col(g);
          const uint64_t b0 = smem_desc_sw128(smem_u32(bring + s * BST));
          const uint64_t b1 = b0 + chunk_step;
          mma_ts_first(d, at, b0, idesc);
          mma_ts_acc(d, at + 8, b0 + 2, idesc);
          mma_ts_acc(d, at + 16, b0 + 4, idesc);
          mma_ts_acc(d, at + 24, b0 + 6, idesc);
          mma_ts_acc(d, at + 32, b1, idesc);
          mma_ts_acc(d, at + 40, b1 + 2, idesc);
          mma_ts_acc(d, at + 48, b1 + 4, idesc);
          mma_ts_acc(d, at + 56, b1 + 6, idesc);
          mma_ts_acc(d, at + 64, g ? bc1 : bc0, idesc);  // offsets and zero point
          mma_commit(&empty[s]);
          mma_commit(&pfull[g]);
        }
        __syncwarp();
        issued = true;
        if (++s == NS) s = 0;
      }
      if (!ok) break;
    }
    if (issued) {
      if (elect_one()) mma_commit(drain);
      __syncwarp();
      wait_bar_drain(drain, 0);
    }
  } else {
    // ------------------------------------------------------------ dequant warpgroups
    grid_dep_wait();
    grid_dep_launch();
    const int g = (warp - 2) >> 2;
    const int q = warp & 3;  // TMEM lane quarter
    int srow, half = 0, hrow;
    if (GEMM == 1) {
      half = lane < 16 ? 0 : 1;
      hrow = 16 * q + (lane & 15);
      srow = half * kGateUpRows + hrow;
    } else {
      srow = q * 32 + lane;
      hrow = srow;
    }
    const int si = GEMM == 1 ? half * kGateUpRows + hrow : hrow;
    const int zi = GEMM == 1 ? half * (kGateUpRows / PF) + hrow / PF : hrow / PF;
    const int zshift = BITS * (hrow % PF);
    const int z_off = (VAR && a.wpack) ? W_BYTES + 256 : Z_OFF;  // zero points: right after the scales in an image
    const uint32_t t_lane = static_cast<uint32_t>(q * 32) << 16;
    const uint32_t a_slot = tmem + t_lane + defer_a_col(g);
    const uint32_t p_addr = tmem + t_lane + defer_p_col(g, NT);
    const uint32_t c_addr = tmem + t_lane + defer_c_col(NT);
    const bool builder = ((warp - 2) & 3) == 0 && lane < NT;  // first warp of the group writes the B rows
    uint8_t* my_bcorr = bcorr + g * NT * 128;
    const uint4* row_base = reinterpret_cast<const uint4*>(wring + srow * KW * 4);
    const int swz = BITS == 4 ? ((srow >> 1) & 3) : (srow & 7);

    // This group's stages are the running stage indices g, g + 2, g + 4, ...
    // across units: ring slot cs and phase cf of the next one advance by two
    // slots, the afull / pfull phase pph flips each time.
    int it = 0, uc = 0, cs = g;
    uint32_t cf = 0, pph = 0;
    bool ok = true;
    for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++uc) {
      const Unit w = decode_unit(u, nb, a);
      const int n = w.kt1 - w.kt0;
      // the epilogue's routed-pair count, fetched into L1 now (no register held)
      if (NT == 16 && g == 0) prefetch_l1(a.block_rows + w.blk);
      float acc[NT];
#pragma unroll
      for (int j = 0; j < NT; ++j) acc[j] = 0.f;
      // The previous stage's partial sum is folded in one stage late: its MMA
      // completion is awaited only once this stage's data has landed.
      float pscale = 0.f;
      bool pending = false;
      for (int i = (g - it) & 1; i < n; i += 2) {
        if (!warp_wait_all(&full[cs], cf, abort_flag, a.status)) { ok = false; break; }
        // the previous stage's MMAs done: A slot, correction rows and P_g free;
        // its partial sum, scaled into the accumulators
        if (pending) {
          if (!warp_wait_all(&pfull[g], pph, abort_flag, a.status)) { ok = false; break; }
          tc_fence_after();
          pph ^= 1u;
#pragma unroll
          for (int c0 = 0; c0 < NT; c0 += 16) {
            uint32_t v[16];
            tmem_ld16(p_addr + c0, v);
            tmem_ld_wait(v);
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[c0 + j] = fmaf(pscale, __uint_as_float(v[j]), acc[c0 + j]);
          }
        }
        const uint8_t* st = wring + cs * WST;
        const float scale = scale_to_f32<SCL>(reinterpret_cast<const uint16_t*>(st + S_OFF)[si]);
        uint32_t zero = 1u << (BITS - 1);
        if (a.has_zeros) zero = (reinterpret_cast<const uint32_t*>(st + z_off)[zi] >> zshift) & ZMASK;
        const uint4* src = row_base + cs * (WST / 16);
        // codes of this row -> A slot g (magic-number form)
#pragma unroll
        for (int h = 0; h < 4; ++h) {
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
          codes_to_magic<BITS, ACT>(wv, outv);
          tmem_st16(a_slot + h * 16, outv);
        }
        {
          uint32_t cv[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
          corr_a<BITS, ACT>(zero, cv);
          tmem_st8(a_slot + 64, cv);
        }
        if (builder) {
          // token `lane`: sums of the stage's token values over even and odd k
          const float* xs = xring + cs * (XST / 4);
          float xe = 0.f, xo = 0.f;
#pragma unroll
          for (int pp = 0; pp < XPARTS; pp += 2) {
            xe += xs[pp * NT + lane];
            xo += xs[(pp + 1) * NT + lane];
          }
          uint32_t bv[4];
          corr_b<BITS, ACT>(xe, xo, bv);
          uint4* row = reinterpret_cast<uint4*>(my_bcorr + lane * 128);
          row[0 ^ (lane & 7)] = make_uint4(bv[0], bv[1], bv[2], bv[3]);  // K 0..7 (128-byte swizzle)
          row[1 ^ (lane & 7)] = make_uint4(0u, 0u, 0u, 0u);  // K 8..15
          fence_proxy_async_smem();
        }
        __syncwarp();  // reconverge before the warp-wide tcgen05 wait
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&afull[g]);
        pscale = scale;
        pending = true;
        cs += 2;
        if (cs >= NS) {
          cs -= NS;
          cf ^= 1u;
        }
      }
      // the unit's last stage
      if (ok && pending) {
        if (!warp_wait_all(&pfull[g], pph, abort_flag, a.status)) {
          ok = false;
        } else {
          tc_fence_after();
          pph ^= 1u;
#pragma unroll
          for (int c0 = 0; c0 < NT; c0 += 16) {
            uint32_t v[16];
            tmem_ld16(p_addr + c0, v);
            tmem_ld_wait(v);
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[c0 + j] = fmaf(pscale, __uint_as_float(v[j]), acc[c0 + j]);
          }
        }
      }
      it += n;
      if (!ok) break;
      // combine the two warpgroups' sums (buffer C), epilogue in warpgroup 0
      if (g == 1) {
        if (!warp_wait_all(cempty, (uc & 1) ^ 1, abort_flag, a.status)) break;
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < NT; c0 += 16) {
          uint32_t v[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) v[j] = __float_as_uint(acc[c0 + j]);
          tmem_st16(c_addr + c0, v);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(cfull);
        // C aliases P_1: the next MMA into it must wait until warpgroup 0 took C
        if (defer_c_col(NT) == NT && !warp_wait_all(cempty, uc & 1, abort_flag, a.status)) break;
        continue;
      }
      // routed pairs of the block (they lead it): 16-token epilogues skip the
      // padding (measured: 32-token ones ran slower with the check)
      const int rows = NT == 16 ? a.block_rows[w.blk] : NT;
      if (!warp_wait_all(cfull, uc & 1, abort_flag, a.status)) break;
      tc_fence_after();
#pragma unroll
      for (int c0 = 0; c0 < NT; c0 += 16) {
        uint32_t v[16];
        tmem_ld16(c_addr + c0, v);
        tmem_ld_wait(v);
#pragma unroll
        for (int j = 0; j < 16; ++j) acc[c0 + j] += __uint_as_float(v[j]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(cempty);
      if (GEMM == 1 && a.split > 1) {
        // K split: each split unit publishes its fp32 partial sums; per lane
        // quarter, the last of the split units to arrive adds them up in split
        // order (deterministic) and runs the epilogue. The others stop here.
        const int row = q * 32 + lane;  // TMEM lane = row of the 128-row tile
        float4* mine = reinterpret_cast<float4*>(a.part + part_index(a, w.tile, w.blk, w.sp, row, NT));
#pragma unroll
        for (int j = 0; j < NT; j += 4) mine[j / 4] = make_float4(acc[j], acc[j + 1], acc[j + 2], acc[j + 3]);
        __threadfence();
        __syncwarp();
        int* counter = a.counters + counter_index(a, w.tile, w.blk, q);
        int arrived = 0;
        if (lane == 0) arrived = atomicAdd(counter, 1);
        arrived = __shfl_sync(0xFFFFFFFFu, arrived, 0);
        if (arrived != a.split - 1) continue;
        __threadfence();
#pragma unroll
        for (int j = 0; j < NT; ++j) acc[j] = 0.f;
        for (int sp = 0; sp < a.split; ++sp) {
          const float4* src = reinterpret_cast<const float4*>(a.part + part_index(a, w.tile, w.blk, sp, row, NT));
#pragma unroll
          for (int j = 0; j < NT; j += 4) {
            const float4 v4 = __ldcg(src + j / 4);
            acc[j] += v4.x;
            acc[j + 1] += v4.y;
            acc[j + 2] += v4.z;
            acc[j + 3] += v4.w;
          }
        }
        if (lane == 0) *counter = 0;  // ready for the next call
      }
      if (GEMM == 1) {
        // silu(gate) * up -> act cache; lanes 0-15 hold gate rows, 16-31 the up
        // rows of the same features: each lane finishes half of the NT tokens.
        using T = typename Act<ACT>::T;
        T* act = reinterpret_cast<T*>(a.out);
        const bool lo = lane < 16;
        const int f = w.tile * kGateUpRows + 16 * q + (lane & 15);
        const int fp = kPermuteK<BITS> ? permute_k8(f) : f;
        if (VAR && a.bias) {
          const float b = bias_of<ACT>(a, unit_expert(a, w.blk), lo ? f : a.I + f);
#pragma unroll
          for (int j = 0; j < NT; ++j) acc[j] += b;
        }
#pragma unroll
        for (int j = 0; j < NT / 2; ++j) {
          if (!defer_writes_col(1, j, rows, NT)) break;  // columns j and j + NT/2: padding, as are the rest
          const float mine = lo ? acc[j] : acc[j + NT / 2];
          const float other = __shfl_xor_sync(0xFFFFFFFFu, lo ? acc[j + NT / 2] : acc[j], 16);
          const float gt = lo ? mine : other;
          const float up = lo ? other : mine;
          const float val = VAR ? gate_up_act(a, gt, up) : gt / (1.0f + __expf(-gt)) * up;
          const int col = lo ? j : j + NT / 2;
          const size_t row = static_cast<size_t>(w.blk) * NT + col;
          const size_t idx = act_index(w.blk, NT, col, a.I, fp);
          float stored;
          if constexpr (ACT == 0) {
            const __half hv = __float2half_rn(val);
            act[idx] = hv;
            stored = __half2float(hv);
          } else {
            const __nv_bfloat16 hv = __float2bfloat16_rn(val);
            act[idx] = hv;
            stored = __bfloat162float(hv);
          }
          // token sums of the stored values over this warp's 16 features, by
          // feature parity (= lane parity): lanes 0/1 (16/17) end with them.
          // The tile's 64 features are half (tile & 1) of down stage tile / 2.
          stored += __shfl_xor_sync(0xFFFFFFFFu, stored, 2);
          stored += __shfl_xor_sync(0xFFFFFFFFu, stored, 4);
          stored += __shfl_xor_sync(0xFFFFFFFFu, stored, 8);
          if ((lane & 14) == 0) {
            const int part = (w.tile & 1) * 8 + q * 2 + (lane & 1);
            a.xs_out[xs_out_index(w.tile, part, a.cap, row)] = stored;
          }
        }
      } else {
        float* slab = reinterpret_cast<float*>(a.out);
        const int hr = w.tile * kTileRows + q * 32 + lane;
        const int my_pid = a.sorted_ids[w.blk * NT + (lane & (NT - 1))];
        const float my_w = (my_pid >= 0 && my_pid < a.P) ? a.topk_w[my_pid] : 0.f;
        if (VAR && a.bias && w.sp == 0 && hr < a.N) {
          // the expert's bias, added once (by the first K split)
          const float b = bias_of<ACT>(a, unit_expert(a, w.blk), hr);
#pragma unroll
          for (int j = 0; j < NT; ++j) acc[j] += b;
        }
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          if (!defer_writes_col(2, j, rows, NT)) break;  // padding from here on
          const int pid = __shfl_sync(0xFFFFFFFFu, my_pid, j);
          const float tw = __shfl_sync(0xFFFFFFFFu, my_w, j);
          if (pid >= 0 && pid < a.P && hr < a.N) {
            if (VAR && a.atomic_out)  // unordered fp32 sum over the token's slots and the K splits
              atomicAdd(a.atomic_out + static_cast<size_t>(pid / a.topk) * a.N + hr, acc[j] * tw);
            else
              slab[slab_index(w.sp, a.P, pid, a.N, hr)] = acc[j] * tw;
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();  // the drain wait above is per lane: converge before the .aligned dealloc
    tc_fence_after();
    tmem_dealloc(tmem, kDeferTmemCols);
  }
}

}  // namespace wna16
