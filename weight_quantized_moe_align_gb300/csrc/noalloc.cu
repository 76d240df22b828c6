// wna16_fused_moe_noalloc: the fused layer with a library-owned workspace,
// for callers that have no allocator to hand the library scratch memory from.
//
// The workspace is a fixed device array in this file. Host code cannot use
// the array's name as a device address (on the host it names a stand-in
// object), so the address is looked up once per device with
// cudaGetSymbolAddress, with that device current, and then passed down like
// any caller-provided workspace. Nothing here allocates.
#include <mutex>

#include "wna16_moe.h"

namespace {

// Every GPU that loads the library reserves this area until the library is
// unloaded.
static __device__ __align__(256) unsigned char g_noalloc_scratch[WNA16_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch area on the current device (set up on the
// first call per device).
wna16_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return WNA16_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return WNA16_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return WNA16_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return WNA16_OK;
}

}  // namespace

extern "C" wna16_status wna16_fused_moe_noalloc(
    const void* hidden, wna16_dtype act_dtype, int64_t M, int64_t H, int64_t I, int E, int topk,
    const int32_t* w13_q, const void* w13_scales, const int32_t* w13_zeros, const int32_t* w2_q,
    const void* w2_scales, const int32_t* w2_zeros, wna16_dtype scale_dtype, int bits, int group_size,
    const int32_t* topk_ids, const float* topk_weights, void* out, int block, int split_k, void* stream) {
  if (M == 0) {
    // Same answer as wna16_fused_moe for an empty batch (it validates and
    // launches nothing), without touching the scratch area.
    return wna16_fused_moe(hidden, act_dtype, M, H, I, E, topk, w13_q, w13_scales, w13_zeros, w2_q, w2_scales,
                           w2_zeros, scale_dtype, bits, group_size, topk_ids, topk_weights, out, nullptr, 0,
                           block, split_k, stream);
  }
  const size_t need = wna16_fused_moe_workspace_bytes(M, H, I, E, topk, bits, group_size, block, split_k);
  if (need == 0) {
    // Invalid sizes: report exactly what wna16_fused_moe reports; it returns
    // from its argument checks before launching anything.
    return wna16_fused_moe(hidden, act_dtype, M, H, I, E, topk, w13_q, w13_scales, w13_zeros, w2_q, w2_scales,
                           w2_zeros, scale_dtype, bits, group_size, topk_ids, topk_weights, out, nullptr, 0,
                           block, split_k, stream);
  }
  if (need > WNA16_NOALLOC_SCRATCH_BYTES) return WNA16_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const wna16_status st = scratch_address(&scratch);
  if (st != WNA16_OK) return st;
  return wna16_fused_moe(hidden, act_dtype, M, H, I, E, topk, w13_q, w13_scales, w13_zeros, w2_q, w2_scales,
                         w2_zeros, scale_dtype, bits, group_size, topk_ids, topk_weights, out, scratch,
                         WNA16_NOALLOC_SCRATCH_BYTES, block, split_k, stream);
}
