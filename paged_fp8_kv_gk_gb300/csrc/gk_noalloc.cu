// gk_noalloc.cu -- decode attention for callers that cannot allocate device
// memory themselves.
//
// Some callers of this library have no way to obtain a workspace buffer:
// a host framework that accounts for every device byte up front (a serving
// engine that sizes its KV pool as total memory x utilisation minus what is
// already resident, so a later allocation by an extension breaks that budget),
// a plugin boundary or foreign-language binding that exposes no device
// allocator, or a latency-critical step where a cudaMalloc, which may
// synchronise the device and may fail, cannot be allowed.  For them the
// library carries its own scratch: a file-scope device array of fixed size,
// created with the module, held by every GPU that loads the library until the
// process exits.  The entry point below allocates nothing and calls no
// allocating routine; it hands that array to gk_decode_attn_stack as the
// workspace.
#include <cuda_runtime.h>

#include "gk_internal.h"

namespace {

static __device__ __align__(256) uint8_t g_gk_static_scratch[GK_STATIC_SCRATCH_BYTES];

// Device address of the scratch array in the current context.  In host code
// g_gk_static_scratch names a host-side stand-in, not device memory, so the
// address is looked up on every call, with the caller's device current: the
// lookup is cheap, enqueues no work, and stays right when the module is loaded
// again at another address (after cudaDeviceReset, or in another context on
// the same device).
gk_status static_scratch_address(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_gk_static_scratch) != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    return GK_ERR_CUDA;
  }
  *out = p;
  return GK_OK;
}

}  // namespace

extern "C" gk_status gk_decode_attn_stack_static(
    const gk_shape* shape, const void* q, const gk_kv_cache* kv, const float* k_scale, const float* v_scale, const float* cos, const float* sin,
    const int32_t* bt_full, const int32_t* bt_swa, const int32_t* pos, const int32_t* pos_w,
    const uint8_t* active, const float* sinks, void* out, float* out_f32, void* stream) {
  const size_t need = gk_attn_workspace_min_bytes(shape);
  if (need == 0)  // invalid or unsupported shape: the regular entry point says which
    return gk_decode_attn_stack(shape, q, kv, k_scale, v_scale, cos, sin, bt_full,
                                bt_swa, pos, pos_w, active, sinks, out, out_f32, nullptr, 0, stream);
  if (need > GK_STATIC_SCRATCH_BYTES) return GK_ERR_WORKSPACE;
  void* scratch = nullptr;
  const gk_status st = static_scratch_address(&scratch);
  if (st != GK_OK) return st;
  // The planner rewrites the work-queue header and the split-row list
  // at the start of every call, so the previous call's contents need no
  // clearing here.
  return gk_decode_attn_stack(shape, q, kv, k_scale, v_scale, cos, sin, bt_full,
                              bt_swa, pos, pos_w, active, sinks, out, out_f32, scratch,
                              GK_STATIC_SCRATCH_BYTES, stream);
}
