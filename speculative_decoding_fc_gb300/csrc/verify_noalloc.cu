// dspark_verify_noalloc: dspark_verify for callers that cannot provide a
// workspace.  Its scratch is one fixed array in this library's device image.
//
// Who needs it: code that is handed only its input and output buffers by a
// host framework that owns every other device allocation (a serving engine's
// custom-operator interface, for instance), and code that must not call
// cudaMalloc while it runs, because cudaMalloc may synchronise the device or
// because the process works to a fixed memory budget.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kScratchBytes = DSPARK_VERIFY_NOALLOC_MAX_BYTES;

// Zero-initialised at module load; every GPU that loads the library holds it
// until the process exits.  Host code must not pass this name to a kernel: in
// host code it is only a stand-in for the device symbol.
static __device__ __align__(256) unsigned char g_verify_scratch[kScratchBytes];

std::mutex g_mutex;
void *g_scratch_ptr[64] = {};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current).
dspark_status_t scratch_for_current_device(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSPARK_ERR_CUDA;
  if (dev < 0 || dev >= 64) return DSPARK_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_verify_scratch) != cudaSuccess || p == nullptr)
      return DSPARK_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
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
  if (B < 1 || k < 1 || V < 1) return DSPARK_ERR_INVALID_ARG;
  const size_t need = dspark_verify_workspace_size(B, k, V);
  if (need == 0) return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (need > kScratchBytes) return DSPARK_ERR_WORKSPACE;  // beyond the fixed scratch
  void *ws = nullptr;
  dspark_status_t st = scratch_for_current_device(&ws);
  if (st != DSPARK_OK) return st;
  // The array keeps the previous call's contents: clear the part this call uses
  // (status word, tickets, partials) before the kernels run, on the same stream.
  if (cudaMemsetAsync(ws, 0, need, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  return dspark_verify(mode, target_logits, draft_tokens, draft_len, draft_logits, q_stats, seed,
                       request_id, step, accepted_len, next_token, B, k, V, ws, kScratchBytes,
                       stream);
}
