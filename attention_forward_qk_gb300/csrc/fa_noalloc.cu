// fa_decode_noalloc: the decode entry point for callers that cannot
// allocate device memory. Its scratch is one library-owned array in device
// global memory instead of a caller-provided workspace.
#include <cuda_runtime.h>

#include <mutex>

#include "fa_internal.h"

namespace {

// Scratch of every fa_decode_noalloc call on a device: created when the
// library is loaded onto that device and held until the process exits.
static __device__ __align__(256) unsigned char g_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per
// device with that device current. In host code `g_noalloc_scratch` names a
// host-side shadow, not device memory, so only this address may be handed to
// kernels.
fa_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return FA_ERR_RUNTIME;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
      return FA_ERR_RUNTIME;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
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
  if (B > fa::kDecodeParamBatches) return FA_ERR_PARAM_INVALID;  // lengths must fit the launch
  const size_t need =
      fa_decode_workspace_size(B, S_kv_max, num_heads, num_kv_heads, D, num_splits);
  if (need == 0) return FA_ERR_PARAM_INVALID;
  if (need > FA_NOALLOC_SCRATCH_BYTES) return FA_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  const fa_status st = scratch_address(&scratch);
  if (st != FA_OK) return st;
  return fa_decode(q, k, v, key_mask, actual_seq_lengths, B, S_kv_max, num_heads, num_kv_heads,
                   D, scale, layout, num_splits, out, lse, scratch, FA_NOALLOC_SCRATCH_BYTES,
                   stream);
}
