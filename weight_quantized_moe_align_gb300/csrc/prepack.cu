// wna16_prepack: plain weight layout -> stage images (layout in common.cuh).
//
// One CTA writes one image: the codes of a 128-row tile over one 128-wide K
// stage, swizzled exactly as the GEMM kernels' TMA boxes place them in shared
// memory, then the stage's scales and zero points. Rows and K beyond the
// matrix, and groups beyond the expert, are written as zeros (they only ever
// meet zero token values).
#include <cuda_fp16.h>

#include "common.cuh"
#include "wna16_moe.h"

namespace wna16 {

namespace {

// Shapes of one projection: N rows (w13: 2I, gate rows then up rows), K.
struct PackShape {
  int E, N, K, G, groups, n_tiles, kt_total, sg, img, has_zeros, gate_up;
};

// Row of the expert matrix held by row r (0..127) of a tile's image, or -1.
// Gate/up tiles hold 64 gate rows then the 64 matching up rows.
__device__ __forceinline__ int image_row(const PackShape& p, int tile, int r) {
  if (p.gate_up) {
    const int I = p.N / 2;
    const int f = tile * kGateUpRows + (r & (kGateUpRows - 1));
    return f < I ? (r / kGateUpRows) * I + f : -1;
  }
  const int n = tile * kTileRows + r;
  return n < p.N ? n : -1;
}

template <int BITS>
__global__ void __launch_bounds__(256) prepack_kernel(const int32_t* __restrict__ q,
                                                      const uint16_t* __restrict__ scales,
                                                      const int32_t* __restrict__ zeros, const PackShape p,
                                                      uint8_t* __restrict__ dst) {
  constexpr int PF = 32 / BITS;
  constexpr int KW = kTileK / PF;   // code words per row per stage
  constexpr int CH = KW / 4;        // 16-byte chunks per row (4 or 8)
  const int stage = blockIdx.x;
  const int kt = stage % p.kt_total;
  const int rest = stage / p.kt_total;
  const int tile = rest % p.n_tiles;
  const int e = rest / p.n_tiles;
  uint8_t* out = dst + static_cast<size_t>(stage) * p.img;
  const int kwords = p.K / PF;
  for (int idx = threadIdx.x; idx < kTileRows * CH; idx += blockDim.x) {
    const int r = idx / CH, c = idx % CH;
    const int row = image_row(p, tile, r);
    uint32_t v[4] = {0u, 0u, 0u, 0u};
    if (row >= 0) {
      const int32_t* src = q + (static_cast<size_t>(e) * p.N + row) * kwords;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int wi = kt * KW + c * 4 + j;
        if (wi < kwords) v[j] = static_cast<uint32_t>(src[wi]);
      }
    }
    // 64-byte rows: chunk c of row r at c ^ ((r >> 1) & 3); 128-byte rows: c ^ (r & 7)
    const int pc = BITS == 4 ? (c ^ ((r >> 1) & 3)) : (c ^ (r & 7));
    reinterpret_cast<uint4*>(out + r * KW * 4)[pc] = make_uint4(v[0], v[1], v[2], v[3]);
  }
  // scales [sg][128] (gate/up: [sg][2 halves][64], the same order)
  const int g0 = (kt * kTileK) / p.G;
  uint16_t* so = reinterpret_cast<uint16_t*>(out + weight_code_bytes(BITS));
  for (int idx = threadIdx.x; idx < p.sg * kTileRows; idx += blockDim.x) {
    const int g = g0 + idx / kTileRows;
    const int row = image_row(p, tile, idx % kTileRows);
    so[idx] = (row >= 0 && g < p.groups) ? scales[(static_cast<size_t>(e) * p.groups + g) * p.N + row] : 0;
  }
  // zero points [sg][128 / PF] words (gate/up: [sg][2 halves][64 / PF]), packed along N
  if (p.has_zeros) {
    constexpr int ZW = kTileRows / PF;
    int32_t* zo = reinterpret_cast<int32_t*>(out + weight_code_bytes(BITS) + p.sg * 256);
    for (int idx = threadIdx.x; idx < p.sg * ZW; idx += blockDim.x) {
      const int g = g0 + idx / ZW;
      const int row = image_row(p, tile, (idx % ZW) * PF);  // first row of the word
      zo[idx] = (row >= 0 && g < p.groups)
                    ? zeros[(static_cast<size_t>(e) * p.groups + g) * (p.N / PF) + row / PF]
                    : 0;
    }
  }
}

bool pack_shape(int E, int64_t N, int64_t K, int bits, int group_size, int has_zeros, int gate_up, PackShape* p) {
  if (E < 1 || E > 256 || N <= 0 || K <= 0 || (bits != 4 && bits != 8)) return false;
  if (K % 64 || N % 64 || N >= (int64_t(1) << 24) || K >= (int64_t(1) << 24)) return false;
  if (gate_up && (N % 128)) return false;  // 2I with I a multiple of 64
  const int64_t G = group_size == -1 ? K : group_size;
  if (G <= 0 || K % G || (G != 64 && G % kTileK && group_size != -1)) return false;
  p->E = E;
  p->N = static_cast<int>(N);
  p->K = static_cast<int>(K);
  p->G = static_cast<int>(G);
  p->groups = static_cast<int>(K / G);
  p->n_tiles = gate_up ? static_cast<int>(N / 2 / kGateUpRows) : static_cast<int>((N + kTileRows - 1) / kTileRows);
  p->kt_total = static_cast<int>((K + kTileK - 1) / kTileK);
  p->sg = prepack_sg(static_cast<int>(G));
  p->has_zeros = has_zeros ? 1 : 0;
  p->gate_up = gate_up ? 1 : 0;
  p->img = prepack_image_bytes(bits, p->sg, p->has_zeros);
  return true;
}

}  // namespace

}  // namespace wna16

using namespace wna16;

extern "C" size_t wna16_prepack_bytes(int E, int64_t N, int64_t K, int bits, int group_size, int has_zeros,
                                      int gate_up) {
  PackShape p;
  if (!pack_shape(E, N, K, bits, group_size, has_zeros, gate_up, &p)) return 0;
  return static_cast<size_t>(p.E) * p.n_tiles * p.kt_total * p.img;
}

extern "C" wna16_status wna16_prepack(const int32_t* q, const void* scales, const int32_t* zeros, int E,
                                      int64_t N, int64_t K, int bits, int group_size, int gate_up, void* dst,
                                      void* stream) {
  PackShape p;
  if (!pack_shape(E, N, K, bits, group_size, zeros != nullptr, gate_up, &p)) return WNA16_ERR_UNSUPPORTED;
  if (!q || !scales || !dst) return WNA16_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(dst) & 15u) || (reinterpret_cast<uintptr_t>(q) & 3u) ||
      (reinterpret_cast<uintptr_t>(scales) & 1u) || (reinterpret_cast<uintptr_t>(zeros) & 3u))
    return WNA16_ERR_INVALID_ARG;
  const unsigned images = static_cast<unsigned>(static_cast<int64_t>(p.E) * p.n_tiles * p.kt_total);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (bits == 4)
    prepack_kernel<4><<<images, 256, 0, s>>>(q, static_cast<const uint16_t*>(scales), zeros, p,
                                             static_cast<uint8_t*>(dst));
  else
    prepack_kernel<8><<<images, 256, 0, s>>>(q, static_cast<const uint16_t*>(scales), zeros, p,
                                             static_cast<uint8_t*>(dst));
  return cudaGetLastError() == cudaSuccess ? WNA16_OK : WNA16_ERR_CUDA;
}
