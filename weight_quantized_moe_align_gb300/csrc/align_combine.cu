// moe_align_block_size and the ordered top-k combine.
//
// Align (vLLM PR #12185, note 1: a shared-memory align kernel that supports
// DeepSeek-V3's 256 experts and CUDA graphs): one CTA of 1024 threads.
//   1. histogram of expert ids in shared memory;
//   2. exclusive scan of the block-padded counts (one warp, 8 experts/lane);
//   3. sentinel fill of sorted_ids, expert id of every block by binary search;
//   4. stable scatter, 1024 pairs per round: __match_any_sync gives each pair
//      its rank among same-expert lanes of its warp, a per-expert scan over the
//      32 warps gives the warp's base, so the order within an expert is the
//      pair order (deterministic, no atomics on the output).
// All sizes are fixed by the capacity bound, so the launch never depends on
// data read back to the host.
//
// Combine: out[t, h] = sum over slots j (in slot order) of the down GEMM's fp32
// rows (already scaled by the top-k weight; one row per K split), rounded once
// to the activation dtype. Each output element is written by one thread; no
// atomics.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "common.cuh"
#include "plan.cuh"
#include "routing_row.cuh"

namespace wna16 {

constexpr int kAlignThreads = 1024;
constexpr int kAlignWarps = kAlignThreads / 32;
constexpr int kMaxExperts = 256;

__device__ __forceinline__ void align_body(const int32_t* __restrict__ ids, int P, int E, int block, int cap,
                                           int32_t* __restrict__ sorted_ids, int32_t* __restrict__ expert_ids,
                                           int32_t* __restrict__ num_post_pad, int32_t* __restrict__ counts_out,
                                           int32_t* __restrict__ status, int32_t* __restrict__ slot_of_pair,
                                           int32_t* __restrict__ block_rows) {
  __shared__ int cnt[kMaxExperts];
  __shared__ int off_end[kMaxExperts];      // exclusive end of each expert's padded segment
  __shared__ int run[kMaxExperts];          // next free slot of each expert
  __shared__ int wbase[kAlignWarps][kMaxExperts];
  __shared__ int total;
  __shared__ int bad;

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  if (tid < kMaxExperts) cnt[tid] = 0;
  for (int i = tid; i < kAlignWarps * kMaxExperts; i += kAlignThreads) (&wbase[0][0])[i] = 0;
  if (tid == 0) bad = 0;
  if (tid == 0 && status) *status = 0;
  __syncthreads();

  // 1. histogram
  for (int p = tid; p < P; p += kAlignThreads) {
    const int e = ids[p];
    if (e >= 0 && e < E)
      atomicAdd(&cnt[e], 1);
    else
      bad = 1;
  }
  __syncthreads();

  // 2. scan of padded counts (warp 0; lane l owns experts 8l .. 8l+7)
  if (warp == 0) {
    int pad[8];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      const int c = e < E ? cnt[e] : 0;
      pad[i] = (c + block - 1) / block * block;
      sum += pad[i];
    }
    int incl = sum;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int v = __shfl_up_sync(0xFFFFFFFFu, incl, d);
      if (lane >= d) incl += v;
    }
    int start = incl - sum;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane * 8 + i;
      if (e < kMaxExperts) {
        run[e] = start;
        start += pad[i];
        off_end[e] = start;
      }
    }
    if (lane == 31) total = incl;
  }
  __syncthreads();
  const int npp = total;
  if (tid == 0) {
    *num_post_pad = npp;
    if (status && bad) atomicOr(status, 0x1 /* WNA16_DEV_BAD_EXPERT_ID */);
  }
  if (counts_out)
    for (int e = tid; e < E; e += kAlignThreads) counts_out[e] = cnt[e];

  // 3. sentinel fill and per-block expert ids
  for (int i = tid; i < cap; i += kAlignThreads) sorted_ids[i] = P;
  const int nblk = cap / block;
  for (int b = tid; b < nblk; b += kAlignThreads) {
    const int start = b * block;
    int e = -1;
    if (start < npp) {  // first expert whose padded segment ends after `start`
      int lo = 0, hi = E - 1;
      while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (off_end[mid] > start)
          hi = mid;
        else
          lo = mid + 1;
      }
      e = lo;
    }
    expert_ids[b] = e;
    // routed pairs in the block (the rest is padding): the GEMMs size their
    // MMAs and epilogues to it
    if (block_rows) {
      const int seg = e >= 0 ? off_end[e] - (cnt[e] + block - 1) / block * block : 0;  // e's first slot
      block_rows[b] = e >= 0 ? rows_in_block(cnt[e], seg, start, block) : 0;
    }
  }
  __syncthreads();  // orders the sentinel fill before the scatter below

  // 4. stable scatter
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int base = 0; base < P; base += kAlignThreads) {
    const int p = base + tid;
    int e = p < P ? ids[p] : -1;
    const bool valid = e >= 0 && e < E;
    if (!valid) e = -1;
    const unsigned peers = __match_any_sync(0xFFFFFFFFu, e);
    const int rank = __popc(peers & lt_mask);
    const bool leader = (__ffs(peers) - 1) == lane;
    if (valid && leader) wbase[warp][e] = __popc(peers);
    __syncthreads();
    // per-expert exclusive scan across warps (in warp order = pair order)
    for (int x = tid; x < E; x += kAlignThreads) {
      int r = run[x];
#pragma unroll 4
      for (int w = 0; w < kAlignWarps; ++w) {
        const int c = wbase[w][x];
        wbase[w][x] = r;
        r += c;
      }
      run[x] = r;
    }
    __syncthreads();
    if (valid) {
      const int pos = wbase[warp][e] + rank;
      sorted_ids[pos] = p;
      if (slot_of_pair) slot_of_pair[p] = pos;
    }
    __syncthreads();
    for (int x = tid; x < E; x += kAlignThreads)
      for (int w = 0; w < kAlignWarps; ++w) wbase[w][x] = 0;
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kAlignThreads, 1)
    moe_align_kernel(const int32_t* __restrict__ ids, int P, int E, int block, int cap,
                     int32_t* __restrict__ sorted_ids, int32_t* __restrict__ expert_ids,
                     int32_t* __restrict__ num_post_pad, int32_t* __restrict__ counts_out,
                     int32_t* __restrict__ status, int32_t* __restrict__ slot_of_pair,
                     int32_t* __restrict__ block_rows) {
  grid_dep_launch();  // the gather may start its launch; it waits for this kernel's writes
  align_body(ids, P, E, block, cap, sorted_ids, expert_ids, num_post_pad, counts_out, status, slot_of_pair,
             block_rows);
}

// Small batches routed on the device: the 32 warps first route the batch's
// token rows (one warp per row, routing_row.cuh), writing the top-k ids and
// weights, then the CTA aligns those ids; one launch instead of two.
template <typename T, int VPL>
__global__ void __launch_bounds__(kAlignThreads, 1)
    moe_route_align_kernel(const T* __restrict__ logits, const routing::RouteArgs ra, int block, int cap,
                           int32_t* __restrict__ sorted_ids, int32_t* __restrict__ expert_ids,
                           int32_t* __restrict__ num_post_pad, int32_t* __restrict__ counts_out,
                           int32_t* __restrict__ status, int32_t* __restrict__ slot_of_pair,
                           int32_t* __restrict__ block_rows) {
  grid_dep_launch();
  for (int row = threadIdx.x >> 5; row < ra.M; row += kAlignWarps) routing::route_row<T, VPL>(logits, ra, row);
  __syncthreads();  // the routed ids (global memory) are visible to the whole CTA
  align_body(ra.ids, ra.M * ra.topk, ra.E, block, cap, sorted_ids, expert_ids, num_post_pad, counts_out, status,
             slot_of_pair, block_rows);
}

// Copies the hidden row of every routed pair to its expert-sorted slot:
// x_sorted[slot_of_pair[p]] = hidden[p / topk], one thread per 16-byte vector,
// consecutive threads on consecutive vectors of a row (coalesced loads and
// stores). With `permute` (int4 weights) each vector is stored in the GEMM's K
// order 0,4,1,5,2,6,3,7. With `xs` the 8 lanes holding a 64-element chunk also
// add up the fp32 sums of its even-k and odd-k values (the token sums of the
// deferred-scale gate/up GEMM) and the chunk's first lane writes them:
// xs[(stage * 4 + 2 * half + parity) * cap + slot], stage = chunk / 2, half =
// chunk % 2. Padded slots are not written: they only feed MMA columns whose
// results are discarded.
template <int ACT>
__device__ __forceinline__ void add_even_odd(uint32_t w, float& se, float& so) {
  if constexpr (ACT == 0) {
    se += __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu)));
    so += __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
  } else {
    se += __uint_as_float(w << 16);
    so += __uint_as_float(w & 0xFFFF0000u);
  }
}

template <int ACT>
__global__ void __launch_bounds__(256)
    moe_gather_kernel(const uint4* __restrict__ hidden, const int32_t* __restrict__ ids,
                      const int32_t* __restrict__ slot_of_pair, int P, int topk, int E, int h8, int permute,
                      uint4* __restrict__ x_sorted, float* __restrict__ xs, int cap, float* __restrict__ zero0,
                      int zero_n0, float* __restrict__ zero1, int zero_n1, float* __restrict__ zero2, int zero_n2,
                      float* __restrict__ zero3, int zero_n3) {
  grid_dep_wait();
  grid_dep_launch();
  // A CTA takes tiles of kVec x 256 consecutive vectors: thread t the vectors
  // t, t + 256, ... of the tile, loaded together; each warp instruction covers
  // 32 consecutive vectors. h8 (vectors per row) is a multiple of 8, so the 8
  // lanes of a chunk always share one pair. The CTA count matters beyond this
  // kernel: one of its CTAs on an SM keeps the next GEMM's second CTA off it
  // until it exits. Measured on decode batches, 2 vectors per thread did best
  // (Qwen2-57B M=8 layer 105.5 us against 114.0 with 1 and 108.5 with 8).
  constexpr int kVec = 2;
  const long long n = static_cast<long long>(P) * h8;
  const long long tile = static_cast<long long>(kVec) * blockDim.x;
  const unsigned chunk_lanes = 0xFFu << (threadIdx.x & 24);
  for (long long base = static_cast<long long>(blockIdx.x) * tile; base < n; base += tile * gridDim.x) {
    uint4 x[kVec];
    int pp[kVec], vv[kVec];
    int p = static_cast<int>((base + threadIdx.x) / h8), v = static_cast<int>((base + threadIdx.x) % h8);
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      pp[k] = p;
      vv[k] = v;
      if (base + threadIdx.x + static_cast<long long>(k) * blockDim.x < n)
        x[k] = hidden[static_cast<long long>(p / topk) * h8 + v];
      v += blockDim.x;
      while (v >= h8) {
        v -= h8;
        ++p;
      }
    }
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      if (base + threadIdx.x + static_cast<long long>(k) * blockDim.x >= n) continue;
      const int e = ids[pp[k]];
      if (e < 0 || e >= E) continue;
      const int slot = slot_of_pair[pp[k]];
      uint4 y = x[k];
      if (xs) {
        float se = 0.f, so = 0.f;
        add_even_odd<ACT>(y.x, se, so);
        add_even_odd<ACT>(y.y, se, so);
        add_even_odd<ACT>(y.z, se, so);
        add_even_odd<ACT>(y.w, se, so);
#pragma unroll
        for (int m = 1; m < 8; m <<= 1) {
          se += __shfl_xor_sync(chunk_lanes, se, m);
          so += __shfl_xor_sync(chunk_lanes, so, m);
        }
        if ((vv[k] & 7) == 0) {
          const int c = vv[k] >> 3;
          const long long xb = (static_cast<long long>(c >> 1) * 4 + (c & 1) * 2) * cap + slot;
          xs[xb] = se;
          xs[xb + cap] = so;
        }
      }
      if (permute) {  // (x0 x1)(x2 x3)(x4 x5)(x6 x7) -> (x0 x4)(x1 x5)(x2 x6)(x3 x7)
        const uint4 u = y;
        y.x = __byte_perm(u.x, u.z, 0x5410);
        y.y = __byte_perm(u.x, u.z, 0x7632);
        y.z = __byte_perm(u.y, u.w, 0x5410);
        y.w = __byte_perm(u.y, u.w, 0x7632);
      }
      x_sorted[static_cast<long long>(slot) * h8 + vv[k]] = y;
    }
  }
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const long long first = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (long long i = first; i < zero_n0; i += stride) zero0[i] = 0.f;
  for (long long i = first; i < zero_n1; i += stride) zero1[i] = 0.f;
  for (long long i = first; i < zero_n2; i += stride) zero2[i] = 0.f;
  for (long long i = first; i < zero_n3; i += stride) zero3[i] = 0.f;
}

// Act-order gate/up weights: routed row p's expert e reads its hidden row in
// that expert's K order, x_sorted[slot][i] = hidden[t][kperm[e][i]]. One thread
// per 8 consecutive outputs; the int4 pair order of the GEMM (`permute`) is
// applied to the permuted values.
__global__ void __launch_bounds__(256)
    moe_gather_perm_kernel(const uint16_t* __restrict__ hidden, const int32_t* __restrict__ ids,
                           const int32_t* __restrict__ slot_of_pair, const int32_t* __restrict__ kperm, int P,
                           int topk, int E, int H, int permute, uint4* __restrict__ x_sorted) {
  grid_dep_wait();
  grid_dep_launch();
  const int h8 = H / 8;
  const long long n = static_cast<long long>(P) * h8;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < n; idx += stride) {
    const int p = static_cast<int>(idx / h8);
    const int c = static_cast<int>(idx % h8);
    const int e = ids[p];
    if (e < 0 || e >= E) continue;
    const uint16_t* src = hidden + static_cast<long long>(p / topk) * H;
    const int32_t* kp = kperm + static_cast<long long>(e) * H + c * 8;
    uint32_t v[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int k = kp[j];
      v[j] = static_cast<unsigned>(k) < static_cast<unsigned>(H) ? src[k] : 0u;  // caller's table: never trusted
    }
    uint4 o;
    if (permute) {  // (x0 x4)(x1 x5)(x2 x6)(x3 x7)
      o = make_uint4(v[0] | (v[4] << 16), v[1] | (v[5] << 16), v[2] | (v[6] << 16), v[3] | (v[7] << 16));
    } else {
      o = make_uint4(v[0] | (v[1] << 16), v[2] | (v[3] << 16), v[4] | (v[5] << 16), v[6] | (v[7] << 16));
    }
    x_sorted[static_cast<long long>(slot_of_pair[p]) * h8 + c] = o;
  }
}

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// One thread per 4 consecutive output columns, for the tokens blockIdx.y,
// blockIdx.y + gridDim.y, ...: out[t] = sum over the slots (and K splits) of
// the fp32 rows, in slot order, rounded once.
template <typename T>
__global__ void __launch_bounds__(256)
    moe_combine_kernel(const float* __restrict__ slab, const int32_t* __restrict__ ids, int M, int H,
                       int topk, int E, int split, int summed, T* __restrict__ out) {
  grid_dep_wait();
  // x: 4-column vectors of a row, y: tokens (strided when M exceeds the grid)
  const int h = (blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (h >= H) return;
  const long long P = static_cast<long long>(M) * topk;
  for (int t = blockIdx.y; t < M; t += gridDim.y) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    // summed: the down GEMM already added the slots and splits into [M, H]
    if (summed) acc = *reinterpret_cast<const float4*>(slab + static_cast<long long>(t) * H + h);
    for (int j = 0; j < (summed ? 0 : topk); ++j) {
      const int e = ids[t * topk + j];
      if (e < 0 || e >= E) continue;  // dropped pair
      for (int s = 0; s < split; ++s) {
        const float4 v = *reinterpret_cast<const float4*>(slab + ((s * P) + static_cast<long long>(t) * topk + j) * H + h);
        acc.x += v.x;
        acc.y += v.y;
        acc.z += v.z;
        acc.w += v.w;
      }
    }
    T o[4] = {from_f32<T>(acc.x), from_f32<T>(acc.y), from_f32<T>(acc.z), from_f32<T>(acc.w)};
    *reinterpret_cast<uint2*>(out + static_cast<long long>(t) * H + h) = *reinterpret_cast<uint2*>(o);
  }
}

cudaError_t launch_align(const int32_t* ids, int P, int E, int block, int cap, int32_t* sorted_ids,
                         int32_t* expert_ids, int32_t* num_post_pad, int32_t* counts,
                         int32_t* status, int32_t* slot_of_pair, int32_t* block_rows, cudaStream_t stream) {
  moe_align_kernel<<<1, kAlignThreads, 0, stream>>>(ids, P, E, block, cap, sorted_ids, expert_ids,
                                                    num_post_pad, counts, status, slot_of_pair, block_rows);
  return cudaGetLastError();
}

cudaError_t launch_route_align(const void* logits, int logits_dtype, int M, int E, int topk, int sigmoid, int renorm,
                               int n_groups, int topk_groups, int32_t* routed_ids, float* routed_weights, int block,
                               int cap, int32_t* sorted_ids, int32_t* expert_ids, int32_t* num_post_pad,
                               int32_t* counts, int32_t* status, int32_t* slot_of_pair, int32_t* block_rows,
                               cudaStream_t stream) {
  const routing::RouteArgs ra{M, E, topk, sigmoid, renorm, n_groups, n_groups > 1 ? topk_groups : 1, routed_ids,
                              routed_weights};
  const int vpl = (E + 31) / 32;
#define WNA16_ROUTE_ALIGN(T, V)                                                                               \
  moe_route_align_kernel<T, V><<<1, kAlignThreads, 0, stream>>>(static_cast<const T*>(logits), ra, block, cap, \
                                                                sorted_ids, expert_ids, num_post_pad, counts,  \
                                                                status, slot_of_pair, block_rows)
#define WNA16_ROUTE_ALIGN_T(T)            \
  if (vpl <= 1) WNA16_ROUTE_ALIGN(T, 1);  \
  else if (vpl <= 2) WNA16_ROUTE_ALIGN(T, 2); \
  else if (vpl <= 4) WNA16_ROUTE_ALIGN(T, 4); \
  else WNA16_ROUTE_ALIGN(T, 8)
  if (logits_dtype == 2) {
    WNA16_ROUTE_ALIGN_T(float);
  } else if (logits_dtype == 0) {
    WNA16_ROUTE_ALIGN_T(__half);
  } else {
    WNA16_ROUTE_ALIGN_T(__nv_bfloat16);
  }
#undef WNA16_ROUTE_ALIGN_T
#undef WNA16_ROUTE_ALIGN
  return cudaGetLastError();
}

cudaError_t launch_gather(const void* hidden, const int32_t* ids, const int32_t* slot_of_pair, int P,
                          int topk, int E, int H, int permute, int act_dtype, int max_ctas, void* x_sorted,
                          float* xs, int cap, float* zero_ptr0, int zero_n0, float* zero_ptr1, int zero_n1,
                          float* zero_ptr2, int zero_n2, float* zero_ptr3, int zero_n3, cudaStream_t stream,
                          bool pdl) {
  const int h8 = H / 8;  // a multiple of 8 (H % 64 == 0): the kernel's chunk lanes rely on it
  if (h8 % 8) return cudaErrorInvalidValue;
  // threads: one per 2 vectors of the rows, or per zero-filled word
  long long n = static_cast<long long>(P) * h8 / 2;
  n = std::max<long long>(n, std::max({zero_n0, zero_n1, zero_n2, zero_n3}));
  const int threads = 256;
  const long long want = (n + threads - 1) / threads;
  const unsigned blocks = static_cast<unsigned>(want < max_ctas ? want : max_ctas);
  if (blocks == 0) return cudaSuccess;
  auto* fn = act_dtype == 0 ? moe_gather_kernel<0> : moe_gather_kernel<1>;
  return launch_kernel(fn, dim3(blocks), dim3(threads), 0, stream, pdl, static_cast<const uint4*>(hidden), ids,
                       slot_of_pair, P, topk, E, h8, permute, static_cast<uint4*>(x_sorted), xs, cap, zero_ptr0,
                       zero_n0, zero_ptr1, zero_n1, zero_ptr2, zero_n2, zero_ptr3, zero_n3);
}

cudaError_t launch_gather_perm(const void* hidden, const int32_t* ids, const int32_t* slot_of_pair,
                               const int32_t* kperm, int P, int topk, int E, int H, int permute, int max_ctas,
                               void* x_sorted, cudaStream_t stream, bool pdl) {
  const long long n = static_cast<long long>(P) * (H / 8);
  const int threads = 256;
  const long long want = (n + threads - 1) / threads;
  const unsigned blocks = static_cast<unsigned>(want < max_ctas ? want : max_ctas);
  if (blocks == 0) return cudaSuccess;
  return launch_kernel(moe_gather_perm_kernel, dim3(blocks), dim3(threads), 0, stream, pdl,
                       static_cast<const uint16_t*>(hidden), ids, slot_of_pair, kperm, P, topk, E, H, permute,
                       static_cast<uint4*>(x_sorted));
}

cudaError_t launch_combine(const float* slab, const int32_t* ids, int M, int H, int topk, int E,
                           int split, int summed, int act_dtype, void* out, cudaStream_t stream, bool pdl) {
  const int threads = 256;
  const dim3 blocks((H / 4 + threads - 1) / threads, static_cast<unsigned>(std::min(M, 65535)));
  if (M <= 0) return cudaSuccess;
  if (act_dtype == 0)
    return launch_kernel(moe_combine_kernel<__half>, blocks, dim3(threads), 0, stream, pdl, slab, ids, M, H,
                         topk, E, split, summed, static_cast<__half*>(out));
  return launch_kernel(moe_combine_kernel<__nv_bfloat16>, blocks, dim3(threads), 0, stream, pdl, slab, ids, M,
                       H, topk, E, split, summed, static_cast<__nv_bfloat16*>(out));
}

}  // namespace wna16
