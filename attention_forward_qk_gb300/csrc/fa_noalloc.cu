// fa_decode_noalloc: the decode entry point for callers that cannot
// allocate device memory. Its scratch is one library-owned array in device
// global memory instead of a caller-provided workspace.
#include <cuda_runtime.h>

#include "fa_internal.h"

namespace {

// Scratch of every fa_decode_noalloc call on a device: created when the
// library is loaded onto that device and held until the process exits. Its
// first word is the calls' device status word.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

// Device address of the array on the current device. In host code
// `g_noalloc_scratch` names a host-side shadow, not device memory, so only
// this address may be handed to kernels. It is looked up on every call (a
// host-side query, no stream work): an address cached across calls would go
// stale if the device's primary context were reset and the module reloaded.
fa_status scratch_address(void** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
    return FA_ERR_RUNTIME;
  *out = p;
  return FA_OK;
}

}  // namespace

extern "C" fa_status fa_decode_noalloc(const void* q, const void* k, const void* v,
                                       const uint8_t* key_mask, const int64_t* actual_seq_lengths,
                                       int64_t B, int64_t S_kv_max, int64_t num_heads,
                                       int64_t num_kv_heads, int64_t D, float scale, int layout,
                                       int num_splits, void* out, float* lse, void* stream) {
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr ||
      actual_seq_lengths == nullptr)
    return FA_ERR_NULLPTR;
  // every argument is checked before the array's address is looked up; the
  // plan made from these lengths and this device's SM count decides how much
  // of the array the call uses, and a call whose plan does not fit returns
  // FA_ERR_WORKSPACE_TOO_SMALL before anything is enqueued
  return fa::decode_on_scratch(q, k, v, key_mask, actual_seq_lengths, B, S_kv_max, num_heads,
                               num_kv_heads, D, scale, layout, num_splits, out, lse,
                               scratch_address, FA_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" fa_status fa_decode_noalloc_status(void* stream) {
  void* scratch = nullptr;
  const fa_status st = scratch_address(&scratch);
  if (st != FA_OK) return st;
  return fa_workspace_status(scratch, stream);
}
