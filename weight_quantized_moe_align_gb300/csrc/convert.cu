// wna16_convert_checkpoint: GPTQ / AWQ checkpoint tensors -> the library's
// weight layout (codes [E, N, K/pf] packed along K, zero points
// [E, K/G, N/pf] packed along N, both LSB first).
//
// The fused MoE kernel of vLLM PR #12185 takes its own weight format, one that
// "is just compatible with gptq/awq": checkpoints are converted once at load.
// The checkpoint layouts are those of the public packers:
//   GPTQ qweight [K/pf, N]: the codes of column n packed along K, the same
//     words as the library's [N, K/pf] transposed; qzeros [K/G, N/pf] packed
//     along N, storing z - 1 in the original format (v1), z in the later one.
//   AWQ (4-bit) qweight [K, N/8] and qzeros [K/G, N/8] packed along N with
//     field i of a word holding column 8c + (0 2 4 6 1 3 5 7)[i]; zero points
//     stored as they are.
// Scales are [K/G, N] in both, as in the library.
#include <cuda_runtime.h>

#include <algorithm>

#include "wna16_moe.h"

namespace wna16 {

namespace {

// out[e][c][r] = in[e][r][c] for [R][C] word matrices, 32 x 32 tiles.
__global__ void __launch_bounds__(256) transpose_words_kernel(const uint32_t* __restrict__ in, int R, int C,
                                                              uint32_t* __restrict__ out) {
  __shared__ uint32_t tile[32][33];
  const size_t plane = static_cast<size_t>(R) * C;
  const uint32_t* src = in + blockIdx.z * plane;
  uint32_t* dst = out + blockIdx.z * plane;
  const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int r = r0 + i, c = c0 + threadIdx.x;
    if (r < R && c < C) tile[i][threadIdx.x] = src[static_cast<size_t>(r) * C + c];
  }
  __syncthreads();
  for (int i = threadIdx.y; i < 32; i += blockDim.y) {
    const int c = c0 + i, r = r0 + threadIdx.x;
    if (r < R && c < C) dst[static_cast<size_t>(c) * R + r] = tile[threadIdx.x][i];
  }
}

// field of column j in an AWQ word: the inverse of the pack order 0 2 4 6 1 3 5 7
__device__ __forceinline__ int awq_field(int j) { return (j >> 1) + 4 * (j & 1); }

// AWQ codes [E][K][N/8] -> [E][N][K/8]: one thread per output word (8 K values).
__global__ void __launch_bounds__(256) awq_codes_kernel(const uint32_t* __restrict__ in, int N, int K, long long total,
                                                        uint32_t* __restrict__ out) {
  const int n8 = N / 8, kw = K / 8;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < total; idx += stride) {
    const int w = static_cast<int>(idx % kw);
    const long long rn = idx / kw;
    const int n = static_cast<int>(rn % N);
    const long long e = rn / N;
    const uint32_t* src = in + (e * K + static_cast<long long>(w) * 8) * n8 + n / 8;
    const int sh = 4 * awq_field(n & 7);
    uint32_t v = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) v |= ((src[static_cast<long long>(j) * n8] >> sh) & 0xFu) << (4 * j);
    out[idx] = v;
  }
}

// Zero-point words (packed along N): mode 0 copy, 1 add one to every field
// (GPTQ v1, modulo 2^bits), 2 AWQ field order -> plain.
__global__ void __launch_bounds__(256) zeros_kernel(const uint32_t* __restrict__ in, long long words, int bits,
                                                    int mode, uint32_t* __restrict__ out) {
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  const int pf = 32 / bits;
  const uint32_t mask = (1u << bits) - 1;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < words; i += stride) {
    const uint32_t x = in[i];
    uint32_t v = 0;
    for (int j = 0; j < pf; ++j) {
      const int from = mode == 2 ? awq_field(j) : j;
      uint32_t f = (x >> (bits * from)) & mask;
      if (mode == 1) f = (f + 1) & mask;
      v |= f << (bits * j);
    }
    out[i] = v;
  }
}

unsigned grid_for(long long n) {
  return static_cast<unsigned>(std::max<long long>(1, std::min<long long>((n + 255) / 256, 152ll * 16)));
}

}  // namespace

}  // namespace wna16

using namespace wna16;

extern "C" wna16_status wna16_convert_checkpoint(wna16_checkpoint format, const int32_t* qweight,
                                                 const int32_t* qzeros, int E, int64_t N, int64_t K, int bits,
                                                 int group_size, int32_t* q_out, int32_t* zeros_out, void* stream) {
  if (format != WNA16_CKPT_GPTQ && format != WNA16_CKPT_GPTQ_V2 && format != WNA16_CKPT_AWQ)
    return WNA16_ERR_INVALID_ARG;
  if (E < 1 || E > 256 || N <= 0 || K <= 0 || (bits != 4 && bits != 8)) return WNA16_ERR_INVALID_ARG;
  if (format == WNA16_CKPT_AWQ && bits != 4) return WNA16_ERR_UNSUPPORTED;
  const int pf = 32 / bits;
  const int64_t G = group_size == -1 ? K : group_size;
  if (G <= 0) return WNA16_ERR_INVALID_ARG;
  if (K % pf || N % pf || K % G || N >= (int64_t(1) << 24) || K >= (int64_t(1) << 24)) return WNA16_ERR_UNSUPPORTED;
  if (!qweight || !q_out || (qzeros != nullptr) != (zeros_out != nullptr)) return WNA16_ERR_INVALID_ARG;
  const void* ptrs[] = {qweight, qzeros, q_out, zeros_out};
  for (const void* p : ptrs)
    if (reinterpret_cast<uintptr_t>(p) & 3u) return WNA16_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const uint32_t* qw = reinterpret_cast<const uint32_t*>(qweight);
  uint32_t* qo = reinterpret_cast<uint32_t*>(q_out);
  if (format == WNA16_CKPT_AWQ) {
    const long long total = static_cast<long long>(E) * N * (K / 8);
    awq_codes_kernel<<<grid_for(total), 256, 0, s>>>(qw, static_cast<int>(N), static_cast<int>(K), total, qo);
  } else {
    const int R = static_cast<int>(K / pf), C = static_cast<int>(N);
    const dim3 grid(static_cast<unsigned>((C + 31) / 32), static_cast<unsigned>((R + 31) / 32),
                    static_cast<unsigned>(E));
    transpose_words_kernel<<<grid, dim3(32, 8), 0, s>>>(qw, R, C, qo);
  }
  if (cudaGetLastError() != cudaSuccess) return WNA16_ERR_CUDA;
  if (qzeros) {
    const long long words = static_cast<long long>(E) * (K / G) * (N / pf);
    const int mode = format == WNA16_CKPT_GPTQ ? 1 : (format == WNA16_CKPT_AWQ ? 2 : 0);
    zeros_kernel<<<grid_for(words), 256, 0, s>>>(reinterpret_cast<const uint32_t*>(qzeros), words, bits, mode,
                                                 reinterpret_cast<uint32_t*>(zeros_out));
    if (cudaGetLastError() != cudaSuccess) return WNA16_ERR_CUDA;
  }
  return WNA16_OK;
}
