// dspark_verify_noalloc: dspark_verify for callers that cannot provide a
// workspace.  Its scratch is one fixed array in this library's device image.
//
// Who needs it: code that is handed only its input and output buffers by a
// host framework that owns every other device allocation (a serving engine's
// custom-operator interface, for instance), and code that must not call
// cudaMalloc while it runs, because cudaMalloc may synchronise the device or
// because the process works to a fixed memory budget.
#include <cuda_runtime.h>

#include "internal.h"

namespace {

constexpr size_t kScratchBytes = DSPARK_VERIFY_NOALLOC_MAX_BYTES;

// Zero-initialised at module load; every GPU that loads the library holds it
// until the process exits.  Host code must not pass this name to a kernel: in
// host code it is only a stand-in for the device symbol.
static __device__ __align__(256) unsigned char g_verify_scratch[kScratchBytes];

// Device address of the scratch array on the current device.  Looked up on every
// call (a host-side query): an address cached across calls could outlive the
// context it belongs to (after cudaDeviceReset the module is loaded afresh).
dspark_status_t scratch_for_current_device(void **out) {
  void *p = nullptr;
  if (cudaGetSymbolAddress(&p, g_verify_scratch) != cudaSuccess || p == nullptr) {
    cudaGetLastError();
    return DSPARK_ERR_CUDA;
  }
  *out = p;
  return DSPARK_OK;
}

}  // namespace

extern "C" dspark_status_t dspark_verify_noalloc(int mode, const float *target_logits,
                                                 const int32_t *draft_tokens,
                                                 const int32_t *draft_len,
                                                 const float *draft_logits, const float *q_stats,
                                                 uint64_t seed, const uint32_t *request_id,
                                                 uint32_t step, int32_t *accepted_len,
                                                 int32_t *next_token, int B, int k, int V,
                                                 void *stream) {
  // Every check dspark_verify makes, before anything is enqueued: a rejected call
  // leaves the shared array and the stream untouched.
  dspark_status_t st = dspark::verify_check_args(mode, target_logits, draft_tokens, draft_len,
                                                 draft_logits, q_stats, request_id, accepted_len,
                                                 next_token, B, k, V);
  if (st != DSPARK_OK) return st;
  const size_t need = dspark_verify_workspace_size(B, k, V);
  if (need == 0) return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (need > kScratchBytes) return DSPARK_ERR_WORKSPACE;  // beyond the fixed scratch
  if (!dspark::device_is_blackwell()) return DSPARK_ERR_NO_DEVICE;
  void *ws = nullptr;
  if ((st = scratch_for_current_device(&ws)) != DSPARK_OK) return st;
  // The array keeps the previous call's contents: clear the part this call uses
  // (status word, tickets, partials) before the kernels run, on the same stream.
  if (cudaMemsetAsync(ws, 0, need, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  return dspark_verify(mode, target_logits, draft_tokens, draft_len, draft_logits, q_stats, seed,
                       request_id, step, accepted_len, next_token, B, k, V, ws, kScratchBytes,
                       stream);
}
