// wna16_fused_moe_noalloc: the fused layer with a library-owned workspace,
// for callers that have no allocator to hand the library scratch memory from.
//
// The workspace is a fixed device array in this file. Host code cannot use
// the array's name as a device address (on the host it names a stand-in
// object), so the address is looked up with cudaGetSymbolAddress, with the
// device current, once per device and CUDA context, and then passed down like
// any caller-provided workspace. Nothing here allocates.
#include <cudaTypedefs.h>

#include <mutex>

#include "wna16_moe.h"

namespace {

// Every GPU that loads the library reserves this area until the library is
// unloaded.
static __device__ __align__(256) unsigned char g_noalloc_scratch[WNA16_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

// Cached device address of the area, per device, with the identity of the
// context it was looked up in: after cudaDeviceReset the runtime makes a new
// primary context in which the array lives at a new address, so an address
// from the old context is never reused.
struct ScratchEntry {
  void* ptr;
  unsigned long long ctx_id;
};
std::mutex g_mu;
ScratchEntry g_scratch[kMaxDevices] = {};

// Unique id of the context current on this thread (driver entry points looked
// up through the runtime, so no driver library is linked). False if there is
// no current context or the driver lacks the calls.
bool current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (!get_current || !get_id) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch area on the current device. The first call on
// a device (and the first after its context was replaced) looks it up; later
// calls reuse it.
wna16_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return WNA16_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return WNA16_ERR_UNSUPPORTED;
  unsigned long long id = 0;
  const bool have_id = current_context_id(&id);
  std::lock_guard<std::mutex> lock(g_mu);
  ScratchEntry& entry = g_scratch[dev];
  if (entry.ptr && have_id && entry.ctx_id == id) {
    *out = entry.ptr;
    return WNA16_OK;
  }
  // the lookup also makes the device's primary context current if none was
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return WNA16_ERR_CUDA;
  unsigned long long now = 0;
  if (current_context_id(&now)) {
    entry.ptr = p;
    entry.ctx_id = now;
  } else {
    entry.ptr = nullptr;  // no context identity: look the address up on every call
  }
  *out = p;
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

// The status word of a fused call sits at offset 0 of its workspace; here that
// is the start of the scratch area.
extern "C" wna16_status wna16_noalloc_read_status(int32_t* bits_out, void* stream) {
  void* scratch = nullptr;
  const wna16_status st = scratch_address(&scratch);
  if (st != WNA16_OK) return st;
  return wna16_read_device_status(scratch, bits_out, stream);
}
