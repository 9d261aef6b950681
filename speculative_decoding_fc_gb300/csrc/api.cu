// extern "C" entry points of libdspark: argument checks on the host, then the
// kernels of the other translation units.  Nothing here allocates device
// memory or synchronises the host (except dspark_workspace_status, which is a
// diagnostic read).
#include <cuda_runtime.h>
#include <stdlib.h>
#include <string.h>

#include <cmath>

#include "internal.h"

#include <algorithm>
#include <atomic>
#include <mutex>
#include <unordered_map>

namespace dspark {

namespace {
std::atomic<long long> g_launches{0};
}

void count_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

bool pdl_enabled() {
  static const bool on = [] {
    const char *e = getenv("DSPARK_NO_PDL");
    return !(e && e[0] == '1');
  }();
  return on;
}

int device_sm_count() {
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

bool device_is_blackwell() {
  static int cache[64] = {};  // 0 unknown, 1 yes, 2 no
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (dev >= 0 && dev < 64 && cache[dev] != 0) return cache[dev] == 1;
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return false;
  const bool ok = (major == 10 && minor == 3);  // the library is built for sm_103a only
  if (dev >= 0 && dev < 64) cache[dev] = ok ? 1 : 2;
  return ok;
}

}  // namespace dspark

using namespace dspark;

namespace {

constexpr int kMaxM = 1 << 20;

constexpr size_t kHeader = kWsAlign;  // status word + padding at the start of every workspace

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool aligned2(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 1u) == 0; }
bool aligned8(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 7u) == 0; }

int *status_word(void *ws) { return reinterpret_cast<int *>(ws); }

cudaStream_t as_stream(void *s) { return reinterpret_cast<cudaStream_t>(s); }

dspark_status_t check_ws(const void *ws, size_t have, size_t need) {
  if (!ws) return DSPARK_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(ws) & (kWsAlign - 1)) != 0) return DSPARK_ERR_MISALIGNED;
  if (have < need) return DSPARK_ERR_WORKSPACE;
  return DSPARK_OK;
}

dspark_status_t check_device() { return device_is_blackwell() ? DSPARK_OK : DSPARK_ERR_NO_DEVICE; }

dspark_status_t check_lm_args(const void *h, const void *lm_w, const void *logits, int M, int H,
                              int V) {
  if (!h || !lm_w || !logits) return DSPARK_ERR_INVALID_ARG;
  if (M < 1 || H < 1 || V < 1) return DSPARK_ERR_INVALID_ARG;
  if (M > kMaxM || V > kMaxV || H % 64 != 0 || H > (1 << 20)) return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(h) || !aligned16(lm_w) || !aligned4(logits)) return DSPARK_ERR_MISALIGNED;
  return DSPARK_OK;
}

dspark_status_t check_chain_args(const void *logits, const void *w1, const void *w2, int r,
                                 const void *prev, const void *drafts, const void *q_stats, int B,
                                 int k, int V) {
  if (!logits || !prev || !drafts) return DSPARK_ERR_INVALID_ARG;
  if (B < 1 || k < 1 || V < 1) return DSPARK_ERR_INVALID_ARG;
  if (k > kMaxK || V > kMaxV || B > (1 << 16)) return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (w1) {
    if (!w2) return DSPARK_ERR_INVALID_ARG;
    if (r < 8 || r > kMaxRank || r % 8 != 0) return DSPARK_ERR_UNSUPPORTED_SHAPE;
    if (!aligned2(w1) || !aligned16(w2)) return DSPARK_ERR_MISALIGNED;
  }
  if (!aligned4(logits) || !aligned4(prev) || !aligned4(drafts)) return DSPARK_ERR_MISALIGNED;
  if (q_stats && !aligned4(q_stats)) return DSPARK_ERR_MISALIGNED;
  return DSPARK_OK;
}

}  // namespace

namespace dspark {

dspark_status_t verify_check_args(int mode, const float *target_logits,
                                  const int32_t *draft_tokens, const int32_t *draft_len,
                                  const float *draft_logits, const float *q_stats,
                                  const uint32_t *request_id, const int32_t *accepted_len,
                                  const int32_t *next_token, int B, int k, int V) {
  if (mode != 0 && mode != 1) return DSPARK_ERR_INVALID_ARG;
  if (!target_logits || !draft_tokens || !accepted_len || !next_token) return DSPARK_ERR_INVALID_ARG;
  if (B < 1 || k < 1 || V < 1) return DSPARK_ERR_INVALID_ARG;
  if (k > kMaxK || V > kMaxV || B > (1 << 20)) return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (mode == 1 && draft_logits && q_stats && !aligned8(q_stats)) return DSPARK_ERR_MISALIGNED;
  if (!aligned4(target_logits) || !aligned4(draft_tokens) || !aligned4(accepted_len) ||
      !aligned4(next_token))
    return DSPARK_ERR_MISALIGNED;
  if ((draft_len && !aligned4(draft_len)) || (draft_logits && !aligned4(draft_logits)) ||
      (request_id && !aligned4(request_id)))
    return DSPARK_ERR_MISALIGNED;
  return DSPARK_OK;
}

}  // namespace dspark

namespace {

size_t chain_ws_bytes(int B, int k, int V) { return kHeader + chain_workspace_size(B, k, V); }

// Every kernel leaves its counters at zero, but where the counters sit depends on
// the call's shape: a workspace reused for another shape can hold old partial sums
// where the new shape keeps counters.  The layout each workspace was last used with
// is remembered here; on a change, the new layout's counter regions are cleared on
// the stream first.
std::mutex g_layout_mutex;
std::unordered_map<const void *, uint64_t> g_layout;

uint64_t layout_signature(std::initializer_list<long long> v) {
  uint64_t h = 1469598103934665603ull;  // FNV-1a over the values' bytes
  for (long long x : v)
    for (int i = 0; i < 8; ++i) {
      h ^= static_cast<uint64_t>((x >> (8 * i)) & 0xff);
      h *= 1099511628211ull;
    }
  return h;
}

struct ZeroRange {
  size_t offset, bytes;
};

dspark_status_t prepare_workspace(void *ws, uint64_t sig, std::initializer_list<ZeroRange> ranges,
                                  cudaStream_t s) {
  std::lock_guard<std::mutex> lock(g_layout_mutex);
  auto it = g_layout.find(ws);
  if (it != g_layout.end() && it->second == sig) return DSPARK_OK;
  for (const ZeroRange &z : ranges)
    if (z.bytes && cudaMemsetAsync(static_cast<char *>(ws) + z.offset, 0, z.bytes, s) != cudaSuccess)
      return DSPARK_ERR_CUDA;
  g_layout[ws] = sig;
  return DSPARK_OK;
}

}  // namespace

extern "C" {

const char *dspark_status_string(dspark_status_t s) {
  switch (s) {
    case DSPARK_OK: return "DSPARK_OK";
    case DSPARK_ERR_INVALID_ARG: return "DSPARK_ERR_INVALID_ARG";
    case DSPARK_ERR_UNSUPPORTED_SHAPE: return "DSPARK_ERR_UNSUPPORTED_SHAPE";
    case DSPARK_ERR_MISALIGNED: return "DSPARK_ERR_MISALIGNED";
    case DSPARK_ERR_WORKSPACE: return "DSPARK_ERR_WORKSPACE";
    case DSPARK_ERR_CUDA: return "DSPARK_ERR_CUDA";
    case DSPARK_ERR_DEVICE_TIMEOUT: return "DSPARK_ERR_DEVICE_TIMEOUT";
    case DSPARK_ERR_BAD_TOKEN: return "DSPARK_ERR_BAD_TOKEN";
    case DSPARK_ERR_NO_DEVICE: return "DSPARK_ERR_NO_DEVICE";
    default: return "DSPARK_ERR_UNKNOWN";
  }
}

int dspark_version(void) { return 100; }

long long dspark_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

dspark_status_t dspark_workspace_status(void *ws, void *stream, int32_t *status_out) {
  if (!ws || !status_out) return DSPARK_ERR_INVALID_ARG;
  int32_t v = 0;
  cudaStream_t s = as_stream(stream);
  if (cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return DSPARK_ERR_CUDA;
  if (cudaMemsetAsync(ws, 0, sizeof(v), s) != cudaSuccess) return DSPARK_ERR_CUDA;
  *status_out = v;
  return DSPARK_OK;
}

// ---------------------------------------------------------------- fc projection
size_t dspark_fc_project_workspace_size(int M, int H, int T) {
  if (M < 1 || H < 64 || T < 1 || T > kMaxTaps) return 0;
  return kHeader + gemm_workspace_size(M, H, T * H);
}

dspark_status_t dspark_fc_project(const dspark_bf16_t *const *taps, int T, int64_t tap_ld,
                                  const dspark_bf16_t *fc_w, dspark_bf16_t *h_out, int M, int H,
                                  void *ws, size_t ws_bytes, void *stream) {
  if (!taps || !fc_w || !h_out) return DSPARK_ERR_INVALID_ARG;
  if (T < 1 || M < 1 || H < 1 || tap_ld < H) return DSPARK_ERR_INVALID_ARG;
  if (T > kMaxTaps || H % 64 != 0 || M > kMaxM || H > (1 << 16)) return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (tap_ld % 8 != 0 || !aligned16(fc_w) || !aligned2(h_out)) return DSPARK_ERR_MISALIGNED;
  for (int j = 0; j < T; ++j) {
    if (!taps[j]) return DSPARK_ERR_INVALID_ARG;
    if (!aligned16(taps[j])) return DSPARK_ERR_MISALIGNED;
  }
  dspark_status_t st = check_ws(ws, ws_bytes, dspark_fc_project_workspace_size(M, H, T));
  if (st != DSPARK_OK) return st;
  if ((st = check_device()) != DSPARK_OK) return st;
  st = prepare_workspace(ws, layout_signature({1, M, H, T}),
                         {{0, kHeader + gemm_counter_bytes(M, H, T * H)}}, as_stream(stream));
  if (st != DSPARK_OK) return st;
  GemmProblem p;
  memset(&p, 0, sizeof(p));
  p.w = fc_w;
  for (int j = 0; j < T; ++j) {
    p.x[j] = taps[j];
    p.x_ld[j] = tap_ld;
  }
  p.n_seg = T;
  p.seg_k = H;
  p.N = H;
  p.M = M;
  p.out = h_out;
  p.ldo = H;
  p.out_bf16 = true;
  return gemm_launch(p, static_cast<char *>(ws) + kHeader, ws_bytes - kHeader, status_word(ws),
                     as_stream(stream));
}

// ---------------------------------------------------------------- fc + LM head, one launch
size_t dspark_fc_lm_head_workspace_size(int M, int H, int T, int V) {
  if (M < 1 || H < 64 || T < 1 || T > kMaxTaps || V < 1) return 0;
  const size_t g = gemm2_workspace_size(M, H, T * H, V, H);
  return g ? kHeader + g : 0;
}

dspark_status_t dspark_fc_lm_head(const dspark_bf16_t *const *taps, int T, int64_t tap_ld,
                                  const dspark_bf16_t *fc_w, const dspark_bf16_t *lm_w,
                                  dspark_bf16_t *h_out, float *logits, int M, int H, int V,
                                  void *ws, size_t ws_bytes, void *stream) {
  if (!taps || !fc_w || !lm_w || !h_out || !logits) return DSPARK_ERR_INVALID_ARG;
  if (T < 1 || M < 1 || H < 1 || V < 1 || tap_ld < H) return DSPARK_ERR_INVALID_ARG;
  if (T > kMaxTaps || H % 64 != 0 || M > kMaxM || H > (1 << 16) || V > kMaxV)
    return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (tap_ld % 8 != 0 || !aligned16(fc_w) || !aligned16(lm_w) || !aligned16(h_out) ||
      !aligned4(logits))
    return DSPARK_ERR_MISALIGNED;
  for (int j = 0; j < T; ++j) {
    if (!taps[j]) return DSPARK_ERR_INVALID_ARG;
    if (!aligned16(taps[j])) return DSPARK_ERR_MISALIGNED;
  }
  dspark_status_t st = check_ws(ws, ws_bytes, dspark_fc_lm_head_workspace_size(M, H, T, V));
  if (st != DSPARK_OK) return st;
  if ((st = check_device()) != DSPARK_OK) return st;
  cudaStream_t s = as_stream(stream);
  const size_t p1 = gemm2_phase1_offset(M, H, T * H);
  st = prepare_workspace(ws, layout_signature({8, M, H, T, V}),
                         {{0, kHeader + kWsAlign + gemm_counter_bytes(M, H, T * H)},
                          {kHeader + p1, gemm_counter_bytes(M, V, H)}},
                         s);
  if (st != DSPARK_OK) return st;
  GemmProblem fc, lm;
  memset(&fc, 0, sizeof(fc));
  memset(&lm, 0, sizeof(lm));
  fc.w = fc_w;
  for (int j = 0; j < T; ++j) {
    fc.x[j] = taps[j];
    fc.x_ld[j] = tap_ld;
  }
  fc.n_seg = T;
  fc.seg_k = H;
  fc.N = H;
  fc.M = M;
  fc.out = h_out;
  fc.ldo = H;
  fc.out_bf16 = true;
  lm.w = lm_w;
  lm.x[0] = h_out;
  lm.x_ld[0] = H;
  lm.n_seg = 1;
  lm.seg_k = H;
  lm.N = V;
  lm.M = M;
  lm.out = logits;
  lm.ldo = V;
  lm.out_bf16 = false;
  return gemm_launch2(fc, lm, static_cast<char *>(ws) + kHeader, ws_bytes - kHeader,
                      status_word(ws), s);
}

// ---------------------------------------------------------------- LM head
size_t dspark_lm_head_workspace_size(int M, int H, int V) {
  if (M < 1 || H < 64 || V < 1) return 0;
  return kHeader + gemm_workspace_size(M, V, H);
}

static dspark_status_t lm_head_enqueue(const dspark_bf16_t *h, const dspark_bf16_t *lm_w,
                                       float *logits, int M, int H, int V, void *gemm_ws,
                                       size_t gemm_ws_bytes, int *status, cudaStream_t s) {
  GemmProblem p;
  memset(&p, 0, sizeof(p));
  p.w = lm_w;
  p.x[0] = h;
  p.x_ld[0] = H;
  p.n_seg = 1;
  p.seg_k = H;
  p.N = V;
  p.M = M;
  p.out = logits;
  p.ldo = V;
  p.out_bf16 = false;
  return gemm_launch(p, gemm_ws, gemm_ws_bytes, status, s);
}

dspark_status_t dspark_lm_head(const dspark_bf16_t *h, const dspark_bf16_t *lm_w, float *logits,
                               int M, int H, int V, void *ws, size_t ws_bytes, void *stream) {
  dspark_status_t st = check_lm_args(h, lm_w, logits, M, H, V);
  if (st != DSPARK_OK) return st;
  if ((st = check_ws(ws, ws_bytes, dspark_lm_head_workspace_size(M, H, V))) != DSPARK_OK) return st;
  if ((st = check_device()) != DSPARK_OK) return st;
  st = prepare_workspace(ws, layout_signature({2, M, H, V}),
                         {{0, kHeader + gemm_counter_bytes(M, V, H)}}, as_stream(stream));
  if (st != DSPARK_OK) return st;
  return lm_head_enqueue(h, lm_w, logits, M, H, V, static_cast<char *>(ws) + kHeader,
                         ws_bytes - kHeader, status_word(ws), as_stream(stream));
}

// ---------------------------------------------------------------- Markov greedy drafting
size_t dspark_greedy_sample_workspace_size(int B, int k, int V, int r) {
  (void)r;
  if (B < 1 || k < 1 || V < 1) return 0;
  return chain_ws_bytes(B, k, V);
}

dspark_status_t dspark_greedy_sample(float *logits, const dspark_bf16_t *w1,
                                     const dspark_bf16_t *w2, int r, const int32_t *prev_token,
                                     int32_t *draft_tokens, float *q_stats, int B, int k, int V,
                                     void *ws, size_t ws_bytes, void *stream) {
  dspark_status_t st = check_chain_args(logits, w1, w2, r, prev_token, draft_tokens, q_stats, B, k, V);
  if (st != DSPARK_OK) return st;
  if ((st = check_ws(ws, ws_bytes, chain_ws_bytes(B, k, V))) != DSPARK_OK) return st;
  if ((st = check_device()) != DSPARK_OK) return st;
  st = prepare_workspace(ws, layout_signature({3, B, k, V}), {{0, kHeader + chain_counter_bytes(B, k)}},
                         as_stream(stream));
  if (st != DSPARK_OK) return st;
  return chain_launch(logits, w1, w2, w1 ? r : 0, prev_token, draft_tokens, q_stats, nullptr, B,
                      k, V, static_cast<char *>(ws) + kHeader, status_word(ws), as_stream(stream));
}

// ---------------------------------------------------------------- confidence truncation
dspark_status_t dspark_confidence_truncate(const dspark_bf16_t *h, const dspark_bf16_t *conf_w,
                                           float conf_b, float conf_tau, int32_t *draft_tokens,
                                           int32_t *draft_len, float *conf_out, int B, int k,
                                           int H, void *stream) {
  if (!h || !conf_w || !draft_tokens || !draft_len) return DSPARK_ERR_INVALID_ARG;
  if (B < 1 || k < 1 || H < 1) return DSPARK_ERR_INVALID_ARG;
  if (k > kMaxK || B > (1 << 20) || H % 64 != 0) return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (std::isnan(conf_tau) || std::isnan(conf_b)) return DSPARK_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(conf_w) || !aligned4(draft_tokens) || !aligned4(draft_len) ||
      (conf_out && !aligned4(conf_out)))
    return DSPARK_ERR_MISALIGNED;
  dspark_status_t st = check_device();
  if (st != DSPARK_OK) return st;
  return confidence_launch(h, conf_w, conf_b, conf_tau, 0, nullptr, 0, 0, nullptr, draft_tokens,
                           draft_len, conf_out, B, k, H, nullptr, as_stream(stream));
}

// ---------------------------------------------------------------- confidence with the Markov context
dspark_status_t dspark_confidence_truncate_markov(const dspark_bf16_t *h, const dspark_bf16_t *conf_w,
                                                  float conf_b, float conf_tau, int cumulative,
                                                  const dspark_bf16_t *w1, int r, int V,
                                                  const int32_t *prev_token, int32_t *draft_tokens,
                                                  int32_t *draft_len, float *conf_out, int B, int k,
                                                  int H, int32_t *status, void *stream) {
  if (!h || !conf_w || !draft_tokens || !draft_len) return DSPARK_ERR_INVALID_ARG;
  if (B < 1 || k < 1 || H < 1) return DSPARK_ERR_INVALID_ARG;
  if (w1 && (!prev_token || V < 1)) return DSPARK_ERR_INVALID_ARG;
  if (k > kMaxK || B > (1 << 20) || H % 64 != 0 || V > kMaxV) return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (w1 && (r < 1 || r > kMaxRank)) return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (std::isnan(conf_tau) || std::isnan(conf_b)) return DSPARK_ERR_INVALID_ARG;
  if (!aligned16(h) || !aligned16(conf_w) || !aligned4(draft_tokens) || !aligned4(draft_len) ||
      (conf_out && !aligned4(conf_out)) || (w1 && !aligned2(w1)) ||
      (prev_token && !aligned4(prev_token)) || (status && !aligned4(status)))
    return DSPARK_ERR_MISALIGNED;
  dspark_status_t st = check_device();
  if (st != DSPARK_OK) return st;
  return confidence_launch(h, conf_w, conf_b, conf_tau, cumulative, w1, w1 ? r : 0, V,
                           prev_token, draft_tokens, draft_len, conf_out, B, k, H, status,
                           as_stream(stream));
}

// ---------------------------------------------------------------- whole readout
size_t dspark_draft_readout_workspace_size(int B, int k, int H, int V, int r) {
  (void)r;
  if (B < 1 || k < 1 || H < 64 || V < 1) return 0;
  return kHeader + align_up(gemm_workspace_size(B * k, V, H), kWsAlign) +
         chain_workspace_size(B, k, V);
}

dspark_status_t dspark_draft_readout(const dspark_bf16_t *h, const dspark_bf16_t *lm_w,
                                     const dspark_bf16_t *w1, const dspark_bf16_t *w2, int r,
                                     const int32_t *prev_token, const dspark_bf16_t *conf_w,
                                     float conf_b, float conf_tau, float *logits, float *q_stats,
                                     int32_t *draft_tokens, int32_t *draft_len, float *conf_out,
                                     int B, int k, int H, int V, void *ws, size_t ws_bytes,
                                     void *stream) {
  if (B < 1 || k < 1) return DSPARK_ERR_INVALID_ARG;
  if (B > (1 << 16) || k > kMaxK || static_cast<long long>(B) * k > kMaxM)
    return DSPARK_ERR_UNSUPPORTED_SHAPE;
  const int M = B * k;
  dspark_status_t st = check_lm_args(h, lm_w, logits, M, H, V);
  if (st != DSPARK_OK) return st;
  st = check_chain_args(logits, w1, w2, r, prev_token, draft_tokens, q_stats, B, k, V);
  if (st != DSPARK_OK) return st;
  if (conf_w && !aligned16(conf_w)) return DSPARK_ERR_MISALIGNED;
  if ((draft_len && !aligned4(draft_len)) || (conf_out && !aligned4(conf_out)))
    return DSPARK_ERR_MISALIGNED;
  if (conf_w && !draft_len) return DSPARK_ERR_INVALID_ARG;
  if (std::isnan(conf_tau) || std::isnan(conf_b)) return DSPARK_ERR_INVALID_ARG;
  const size_t need = dspark_draft_readout_workspace_size(B, k, H, V, r);
  if ((st = check_ws(ws, ws_bytes, need)) != DSPARK_OK) return st;
  if ((st = check_device()) != DSPARK_OK) return st;

  cudaStream_t s = as_stream(stream);
  char *base = static_cast<char *>(ws);
  const size_t gemm_bytes = align_up(gemm_workspace_size(M, V, H), kWsAlign);
  st = prepare_workspace(ws, layout_signature({4, B, k, H, V}),
                         {{0, kHeader + gemm_counter_bytes(M, V, H)},
                          {kHeader + gemm_bytes, chain_counter_bytes(B, k)}},
                         s);
  if (st != DSPARK_OK) return st;
  st = lm_head_enqueue(h, lm_w, logits, M, H, V, base + kHeader, gemm_bytes, status_word(ws), s);
  if (st != DSPARK_OK) return st;
  st = chain_launch(logits, w1, w2, w1 ? r : 0, prev_token, draft_tokens, q_stats,
                    conf_w ? nullptr : draft_len, B, k, V, base + kHeader + gemm_bytes,
                    status_word(ws), s);
  if (st != DSPARK_OK) return st;
  if (conf_w)
    st = confidence_launch(h, conf_w, conf_b, conf_tau, 0, nullptr, 0, 0, nullptr, draft_tokens,
                           draft_len, conf_out, B, k, H, status_word(ws), s);
  return st;
}

// ---------------------------------------------------------------- verify
size_t dspark_verify_workspace_size(int B, int k, int V) {
  if (B < 1 || k < 1 || k > kMaxK || V < 1) return 0;
  return verify_workspace_size(B, k, V);
}

dspark_status_t dspark_verify(int mode, const float *target_logits, const int32_t *draft_tokens,
                              const int32_t *draft_len, const float *draft_logits,
                              const float *q_stats, uint64_t seed, const uint32_t *request_id,
                              uint32_t step, int32_t *accepted_len, int32_t *next_token, int B,
                              int k, int V, void *ws, size_t ws_bytes, void *stream) {
  dspark_status_t st = verify_check_args(mode, target_logits, draft_tokens, draft_len,
                                         draft_logits, q_stats, request_id, accepted_len,
                                         next_token, B, k, V);
  if (st != DSPARK_OK) return st;
  if ((st = check_ws(ws, ws_bytes, dspark_verify_workspace_size(B, k, V))) != DSPARK_OK) return st;
  if ((st = check_device()) != DSPARK_OK) return st;
  st = prepare_workspace(ws, layout_signature({5, B, k, V}), {{0, verify_counter_bytes(B, k, V)}},
                         as_stream(stream));
  if (st != DSPARK_OK) return st;
  return verify_launch(mode, target_logits, draft_tokens, draft_len, draft_logits, q_stats, seed,
                       request_id, step, accepted_len, next_token, B, k, V, ws, status_word(ws),
                       as_stream(stream));
}

// ---------------------------------------------------------------- row statistics
size_t dspark_row_stats_workspace_size(int64_t nrows, int V) {
  if (nrows < 1 || nrows > (1LL << 24) || V < 1 || V > kMaxV) return 0;
  return row_stats_workspace_size(nrows, V);
}

dspark_status_t dspark_row_stats(const float *rows, int64_t nrows, int V, float *ms_out,
                                 int32_t *argmax_out, void *ws, size_t ws_bytes, void *stream) {
  if (!rows || (!ms_out && !argmax_out)) return DSPARK_ERR_INVALID_ARG;
  if (nrows < 1 || V < 1) return DSPARK_ERR_INVALID_ARG;
  if (nrows > (1LL << 24) || V > kMaxV) return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (!aligned4(rows) || (ms_out && !aligned8(ms_out)) || (argmax_out && !aligned4(argmax_out)))
    return DSPARK_ERR_MISALIGNED;
  dspark_status_t st = check_ws(ws, ws_bytes, dspark_row_stats_workspace_size(nrows, V));
  if (st != DSPARK_OK) return st;
  if ((st = check_device()) != DSPARK_OK) return st;
  st = prepare_workspace(ws, layout_signature({9, nrows, V}), {{0, row_stats_counter_bytes(nrows, V)}},
                         as_stream(stream));
  if (st != DSPARK_OK) return st;
  return row_stats_launch(rows, nrows, V, ms_out, argmax_out, ws, status_word(ws), as_stream(stream));
}

// ---------------------------------------------------------------- verify from row statistics
size_t dspark_verify_from_stats_workspace_size(int B, int k, int V) {
  if (B < 1 || k < 1 || k > kMaxK || V < 1) return 0;
  return verify_from_stats_workspace_size(B, V);
}

dspark_status_t dspark_verify_from_stats(int mode, const float *target_logits,
                                         const float *target_ms, const int32_t *target_argmax,
                                         const int32_t *draft_tokens, const int32_t *draft_len,
                                         const float *draft_logits, const float *q_stats,
                                         uint64_t seed, const uint32_t *request_id, uint32_t step,
                                         int32_t *accepted_len, int32_t *next_token, int B, int k,
                                         int V, void *ws, size_t ws_bytes, void *stream) {
  dspark_status_t st = verify_check_args(mode, target_logits, draft_tokens, draft_len,
                                         draft_logits, q_stats, request_id, accepted_len,
                                         next_token, B, k, V);
  if (st != DSPARK_OK) return st;
  if (mode == 0 && !target_argmax) return DSPARK_ERR_INVALID_ARG;
  if (mode == 1 && (!target_ms || (draft_logits && !q_stats))) return DSPARK_ERR_INVALID_ARG;
  if ((target_ms && !aligned8(target_ms)) || (target_argmax && !aligned4(target_argmax)) ||
      (mode == 1 && q_stats && !aligned8(q_stats)))
    return DSPARK_ERR_MISALIGNED;
  if ((st = check_ws(ws, ws_bytes, dspark_verify_from_stats_workspace_size(B, k, V))) != DSPARK_OK)
    return st;
  if ((st = check_device()) != DSPARK_OK) return st;
  st = prepare_workspace(ws, layout_signature({10, B, k, V}),
                         {{0, verify_from_stats_counter_bytes(B, V)}}, as_stream(stream));
  if (st != DSPARK_OK) return st;
  return verify_from_stats_launch(mode, target_logits, target_ms, target_argmax, draft_tokens,
                                  draft_len, draft_logits, q_stats, seed, request_id, step,
                                  accepted_len, next_token, B, k, V, ws, status_word(ws),
                                  as_stream(stream));
}

// ---------------------------------------------------------------- FP8 (E4M3) drafter weights
dspark_status_t dspark_quantize_fp8(const dspark_bf16_t *const *segs, int nseg, int64_t seg_ld,
                                    int rows, int seg_cols, uint8_t *codes, float *scales,
                                    void *stream) {
  if (!segs || !codes || !scales) return DSPARK_ERR_INVALID_ARG;
  if (nseg < 1 || rows < 1 || seg_cols < 1 || seg_ld < seg_cols) return DSPARK_ERR_INVALID_ARG;
  if (nseg > kMaxTaps || seg_cols % 16 != 0 || rows > (1 << 24) ||
      static_cast<long long>(nseg) * seg_cols > (1 << 24))
    return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (seg_ld % 8 != 0 || !aligned16(codes) || !aligned4(scales)) return DSPARK_ERR_MISALIGNED;
  const uint16_t *p[kMaxTaps];
  for (int j = 0; j < nseg; ++j) {
    if (!segs[j]) return DSPARK_ERR_INVALID_ARG;
    if (!aligned16(segs[j])) return DSPARK_ERR_MISALIGNED;
    p[j] = reinterpret_cast<const uint16_t *>(segs[j]);
  }
  dspark_status_t st = check_device();
  if (st != DSPARK_OK) return st;
  return quantize_fp8_launch(p, nseg, seg_ld, rows, seg_cols, codes, scales, as_stream(stream));
}

// Workspace of the FP8 GEMMs: [header][GEMM][activation codes M x K][activation scales M].
static size_t fp8_ws_bytes(int M, int N, int K) {
  return kHeader + align_up(gemm_workspace_size_fp8(M, N, K), kWsAlign) +
         align_up(static_cast<size_t>(M) * K, kWsAlign) + align_up(static_cast<size_t>(M) * 4, kWsAlign);
}

static dspark_status_t fp8_gemm(const uint16_t *const *segs, int nseg, int64_t seg_ld, int seg_k,
                                const uint8_t *w8, const float *w_scale, int M, int N, void *out,
                                int64_t ldo, bool out_bf16, long long kind, void *ws,
                                cudaStream_t s) {
  const int K = nseg * seg_k;
  char *base = static_cast<char *>(ws);
  const size_t gemm_bytes = align_up(gemm_workspace_size_fp8(M, N, K), kWsAlign);
  uint8_t *a8 = reinterpret_cast<uint8_t *>(base + kHeader + gemm_bytes);
  float *a_scale =
      reinterpret_cast<float *>(base + kHeader + gemm_bytes + align_up(static_cast<size_t>(M) * K, kWsAlign));
  dspark_status_t st = prepare_workspace(ws, layout_signature({kind, M, N, K}),
                                         {{0, kHeader + gemm_counter_bytes(M, N, K)}}, s);
  if (st != DSPARK_OK) return st;
  if ((st = quantize_fp8_launch(segs, nseg, seg_ld, M, seg_k, a8, a_scale, s)) != DSPARK_OK) return st;
  GemmProblem p;
  memset(&p, 0, sizeof(p));
  p.w = w8;
  p.x[0] = a8;
  p.x_ld[0] = K;
  p.n_seg = 1;
  p.seg_k = K;
  p.N = N;
  p.M = M;
  p.out = out;
  p.ldo = ldo;
  p.out_bf16 = out_bf16;
  p.fp8 = true;
  p.a_scale = a_scale;
  p.w_scale = w_scale;
  return gemm_launch(p, base + kHeader, gemm_bytes, status_word(ws), s);
}

size_t dspark_fc_project_fp8_workspace_size(int M, int H, int T) {
  if (M < 1 || H < 128 || T < 1 || T > kMaxTaps) return 0;
  return fp8_ws_bytes(M, H, T * H);
}

dspark_status_t dspark_fc_project_fp8(const dspark_bf16_t *const *taps, int T, int64_t tap_ld,
                                      const uint8_t *fc_w8, const float *fc_scale,
                                      dspark_bf16_t *h_out, int M, int H, void *ws,
                                      size_t ws_bytes, void *stream) {
  if (!taps || !fc_w8 || !fc_scale || !h_out) return DSPARK_ERR_INVALID_ARG;
  if (T < 1 || M < 1 || H < 1 || tap_ld < H) return DSPARK_ERR_INVALID_ARG;
  if (T > kMaxTaps || H % 128 != 0 || M > kMaxM || H > (1 << 16)) return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (tap_ld % 8 != 0 || !aligned16(fc_w8) || !aligned4(fc_scale) || !aligned2(h_out))
    return DSPARK_ERR_MISALIGNED;
  const uint16_t *p[kMaxTaps];
  for (int j = 0; j < T; ++j) {
    if (!taps[j]) return DSPARK_ERR_INVALID_ARG;
    if (!aligned16(taps[j])) return DSPARK_ERR_MISALIGNED;
    p[j] = reinterpret_cast<const uint16_t *>(taps[j]);
  }
  dspark_status_t st = check_ws(ws, ws_bytes, dspark_fc_project_fp8_workspace_size(M, H, T));
  if (st != DSPARK_OK) return st;
  if ((st = check_device()) != DSPARK_OK) return st;
  return fp8_gemm(p, T, tap_ld, H, fc_w8, fc_scale, M, H, h_out, H, true, 6, ws, as_stream(stream));
}

size_t dspark_lm_head_fp8_workspace_size(int M, int H, int V) {
  if (M < 1 || H < 128 || V < 1) return 0;
  return fp8_ws_bytes(M, V, H);
}

dspark_status_t dspark_lm_head_fp8(const dspark_bf16_t *h, const uint8_t *lm_w8,
                                   const float *lm_scale, float *logits, int M, int H, int V,
                                   void *ws, size_t ws_bytes, void *stream) {
  if (!h || !lm_w8 || !lm_scale || !logits) return DSPARK_ERR_INVALID_ARG;
  if (M < 1 || H < 1 || V < 1) return DSPARK_ERR_INVALID_ARG;
  if (M > kMaxM || V > kMaxV || H % 128 != 0 || H > (1 << 20)) return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(h) || !aligned16(lm_w8) || !aligned4(lm_scale) || !aligned4(logits))
    return DSPARK_ERR_MISALIGNED;
  dspark_status_t st = check_ws(ws, ws_bytes, dspark_lm_head_fp8_workspace_size(M, H, V));
  if (st != DSPARK_OK) return st;
  if ((st = check_device()) != DSPARK_OK) return st;
  const uint16_t *p[1] = {reinterpret_cast<const uint16_t *>(h)};
  return fp8_gemm(p, 1, H, H, lm_w8, lm_scale, M, V, logits, V, false, 7, ws, as_stream(stream));
}


// ---------------------------------------------------------------- drafter backbone
namespace {
constexpr int kMaxNormH = 8192;   // 8 bf16 per 16-byte chunk x 256 threads x 4 chunks
constexpr int kMaxAttnQueries = 48;
bool ld_ok(int64_t ld, int width) { return ld >= width && ld % 8 == 0; }
}  // namespace

size_t dspark_linear_workspace_size(int M, int N, int K) {
  if (M < 1 || N < 1 || K < 64) return 0;
  return kHeader + gemm_workspace_size(M, N, K);
}

dspark_status_t dspark_linear(const dspark_bf16_t *x, int64_t x_ld, const dspark_bf16_t *w, void *out,
                              int64_t out_ld, int out_bf16, int M, int N, int K, void *ws, size_t ws_bytes,
                              void *stream) {
  if (!x || !w || !out) return DSPARK_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1 || !ld_ok(x_ld, K) || out_ld < N) return DSPARK_ERR_INVALID_ARG;
  if (K % 64 != 0 || M > kMaxM || N > kMaxV || K > (1 << 20)) return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || !aligned16(w) || !(out_bf16 ? aligned2(out) : aligned4(out)))
    return DSPARK_ERR_MISALIGNED;
  dspark_status_t st = check_ws(ws, ws_bytes, dspark_linear_workspace_size(M, N, K));
  if (st != DSPARK_OK) return st;
  if ((st = check_device()) != DSPARK_OK) return st;
  st = prepare_workspace(ws, layout_signature({11, M, N, K}), {{0, kHeader + gemm_counter_bytes(M, N, K)}},
                         as_stream(stream));
  if (st != DSPARK_OK) return st;
  GemmProblem p;
  memset(&p, 0, sizeof(p));
  p.w = w;
  p.x[0] = x;
  p.x_ld[0] = x_ld;
  p.n_seg = 1;
  p.seg_k = K;
  p.N = N;
  p.M = M;
  p.out = out;
  p.ldo = out_ld;
  p.out_bf16 = out_bf16 != 0;
  return gemm_launch(p, static_cast<char *>(ws) + kHeader, ws_bytes - kHeader, status_word(ws),
                     as_stream(stream));
}

dspark_status_t dspark_embed_rmsnorm(const dspark_bf16_t *table, int V, const int32_t *tokens,
                                     const dspark_bf16_t *w, float *x_out, dspark_bf16_t *n_out, int rows,
                                     int H, int32_t *status, void *stream) {
  if (!table || !tokens || !w || !x_out || !n_out || rows < 1 || H < 8 || V < 1) return DSPARK_ERR_INVALID_ARG;
  if (H % 8 != 0 || H > kMaxNormH || rows > kMaxM) return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(table) || !aligned4(tokens) || !aligned16(w) || !aligned16(x_out) || !aligned16(n_out) ||
      (status && !aligned4(status)))
    return DSPARK_ERR_MISALIGNED;
  dspark_status_t st = check_device();
  if (st != DSPARK_OK) return st;
  return norm_rows_launch(x_out, nullptr, 0, table, tokens, V, nullptr, 0, w, n_out, H, 0, rows, H, status,
                          as_stream(stream));
}

dspark_status_t dspark_add_rmsnorm(float *x, const dspark_bf16_t *delta, int64_t delta_ld,
                                   const dspark_bf16_t *w, dspark_bf16_t *out, int64_t out_ld, int group,
                                   int rows, int H, void *stream) {
  if (!x || !w || !out || rows < 1 || H < 8 || group < 0 || group == 1) return DSPARK_ERR_INVALID_ARG;
  if (delta && !ld_ok(delta_ld, H)) return DSPARK_ERR_INVALID_ARG;
  if (!ld_ok(out_ld, H) || (group > 0 && rows % group != 0)) return DSPARK_ERR_INVALID_ARG;
  if (H % 8 != 0 || H > kMaxNormH || rows > kMaxM) return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || (delta && !aligned16(delta)) || !aligned16(w) || !aligned16(out))
    return DSPARK_ERR_MISALIGNED;
  dspark_status_t st = check_device();
  if (st != DSPARK_OK) return st;
  return norm_rows_launch(x, delta, delta_ld, nullptr, nullptr, 0, nullptr, 0, w, out, out_ld, group, rows, H,
                          nullptr, as_stream(stream));
}

dspark_status_t dspark_rmsnorm_bf16(const dspark_bf16_t *in, int64_t in_ld, const dspark_bf16_t *w,
                                    dspark_bf16_t *out, int64_t out_ld, int rows, int H, void *stream) {
  if (!in || !w || !out || rows < 1 || H < 8 || !ld_ok(in_ld, H) || !ld_ok(out_ld, H))
    return DSPARK_ERR_INVALID_ARG;
  if (H % 8 != 0 || H > kMaxNormH || rows > kMaxM) return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(in) || !aligned16(w) || !aligned16(out)) return DSPARK_ERR_MISALIGNED;
  dspark_status_t st = check_device();
  if (st != DSPARK_OK) return st;
  return norm_rows_launch(nullptr, nullptr, 0, nullptr, nullptr, 0, in, in_ld, w, out, out_ld, 0, rows, H,
                          nullptr, as_stream(stream));
}

dspark_status_t dspark_qk_norm_rope(const dspark_bf16_t *qkv, int64_t ld, int nq, int nkv,
                                    const dspark_bf16_t *q_norm_w, const dspark_bf16_t *k_norm_w, float theta,
                                    dspark_bf16_t *q_out, dspark_bf16_t *k_cache, dspark_bf16_t *v_cache, int B,
                                    int cache_len, int rows_per_req, int pos0, void *stream) {
  if (!qkv || !k_norm_w || !k_cache || !v_cache || (nq > 0 && (!q_out || !q_norm_w)))
    return DSPARK_ERR_INVALID_ARG;
  if (nq < 0 || nkv < 1 || B < 1 || rows_per_req < 1 || pos0 < 0 || !(theta > 1.0f))
    return DSPARK_ERR_INVALID_ARG;
  if (!ld_ok(ld, (nq + 2 * nkv) * 128) || static_cast<long long>(pos0) + rows_per_req > cache_len)
    return DSPARK_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * rows_per_req > kMaxM || nq + 2 * nkv > 4096) return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(qkv) || !aligned16(k_norm_w) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (nq > 0 && (!aligned16(q_out) || !aligned16(q_norm_w))))
    return DSPARK_ERR_MISALIGNED;
  dspark_status_t st = check_device();
  if (st != DSPARK_OK) return st;
  return qk_norm_rope_launch(qkv, ld, nq, nkv, q_norm_w, k_norm_w, theta, q_out, k_cache, v_cache, cache_len,
                             rows_per_req, pos0, B * rows_per_req, as_stream(stream));
}

dspark_status_t dspark_block_context_rmsnorm(float *x, const dspark_bf16_t *delta, int64_t delta_ld,
                                             const dspark_bf16_t *table, int V, const int32_t *tokens,
                                             const dspark_bf16_t *ctx, int64_t ctx_ld, int ctx_rows,
                                             const dspark_bf16_t *w, dspark_bf16_t *out, int64_t out_ld, int rows,
                                             int H, int32_t *status, void *stream) {
  if (!x || !w || !out || rows < 1 || ctx_rows < 0 || H < 8 || !ld_ok(out_ld, H)) return DSPARK_ERR_INVALID_ARG;
  if (table && (!tokens || V < 1)) return DSPARK_ERR_INVALID_ARG;
  if (!table && delta && !ld_ok(delta_ld, H)) return DSPARK_ERR_INVALID_ARG;
  if (ctx_rows > 0 && (!ctx || !ld_ok(ctx_ld, H))) return DSPARK_ERR_INVALID_ARG;
  if (H % 8 != 0 || H > kMaxNormH || rows + static_cast<long long>(ctx_rows) > kMaxM)
    return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || !aligned16(w) || !aligned16(out) || (table && (!aligned16(table) || !aligned4(tokens))) ||
      (!table && delta && !aligned16(delta)) || (ctx_rows > 0 && !aligned16(ctx)) || (status && !aligned4(status)))
    return DSPARK_ERR_MISALIGNED;
  dspark_status_t st = check_device();
  if (st != DSPARK_OK) return st;
  return norm_rows_launch(x, table ? nullptr : delta, delta_ld, table, tokens, V, nullptr, 0, w, out, out_ld, 0, rows,
                          H, status, as_stream(stream), ctx_rows > 0 ? ctx : nullptr, ctx_ld, ctx_rows);
}

dspark_status_t dspark_qk_norm_rope_block_context(const dspark_bf16_t *qkv, int64_t ld, int nq, int nkv,
                                                  const dspark_bf16_t *q_norm_w, const dspark_bf16_t *k_norm_w,
                                                  float theta, dspark_bf16_t *q_out, dspark_bf16_t *k_cache,
                                                  dspark_bf16_t *v_cache, int B, int cache_len, int rows_per_req,
                                                  int pos0, const dspark_bf16_t *ctx_kv, int64_t ctx_ld,
                                                  int ctx_rows_per_req, int ctx_pos0, void *stream) {
  if (!qkv || !k_norm_w || !k_cache || !v_cache || (nq > 0 && (!q_out || !q_norm_w)))
    return DSPARK_ERR_INVALID_ARG;
  if (nq < 0 || nkv < 1 || B < 1 || rows_per_req < 1 || pos0 < 0 || !(theta > 1.0f) || ctx_rows_per_req < 0 ||
      ctx_pos0 < 0)
    return DSPARK_ERR_INVALID_ARG;
  if (!ld_ok(ld, (nq + 2 * nkv) * 128) || static_cast<long long>(pos0) + rows_per_req > cache_len)
    return DSPARK_ERR_INVALID_ARG;
  if (ctx_rows_per_req > 0 && (!ctx_kv || !ld_ok(ctx_ld, 2 * nkv * 128) ||
                               static_cast<long long>(ctx_pos0) + ctx_rows_per_req > cache_len))
    return DSPARK_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * (rows_per_req + ctx_rows_per_req) > kMaxM || nq + 2 * nkv > 4096)
    return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(qkv) || !aligned16(k_norm_w) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (nq > 0 && (!aligned16(q_out) || !aligned16(q_norm_w))) || (ctx_rows_per_req > 0 && !aligned16(ctx_kv)))
    return DSPARK_ERR_MISALIGNED;
  dspark_status_t st = check_device();
  if (st != DSPARK_OK) return st;
  return qk_norm_rope_launch(qkv, ld, nq, nkv, q_norm_w, k_norm_w, theta, q_out, k_cache, v_cache, cache_len,
                             rows_per_req, pos0, B * rows_per_req, as_stream(stream),
                             ctx_rows_per_req > 0 ? ctx_kv : nullptr, ctx_ld, ctx_rows_per_req, ctx_pos0,
                             B * ctx_rows_per_req);
}

size_t dspark_attention_workspace_size(int B, int nr, int nq, int nkv, int nkeys) {
  if (B < 1 || nr < 1 || nq < 1 || nkv < 1 || nq % nkv != 0 || nkeys < 1) return 0;
  return attention_workspace_bytes(B, nr, nq, nkv, nkeys);
}

dspark_status_t dspark_attention(const dspark_bf16_t *q, const dspark_bf16_t *k_cache,
                                 const dspark_bf16_t *v_cache, dspark_bf16_t *out, int B, int nr, int nq,
                                 int nkv, int cache_len, int nkeys, void *ws, size_t ws_bytes, void *stream) {
  if (!q || !k_cache || !v_cache || !out) return DSPARK_ERR_INVALID_ARG;
  if (B < 1 || nr < 1 || nq < 1 || nkv < 1 || nq % nkv != 0 || nkeys < 1 || nkeys > cache_len)
    return DSPARK_ERR_INVALID_ARG;
  if (nr * (nq / nkv) > kMaxAttnQueries || B > (1 << 16) || nkv > 1024) return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
    return DSPARK_ERR_MISALIGNED;
  dspark_status_t st = check_ws(ws, ws_bytes, dspark_attention_workspace_size(B, nr, nq, nkv, nkeys));
  if (st != DSPARK_OK) return st;
  if ((st = check_device()) != DSPARK_OK) return st;
  return attention_launch(q, k_cache, v_cache, out, B, nr, nq, nkv, cache_len, nkeys, ws, as_stream(stream));
}

namespace {

// Workspace of dspark_backbone_block: [header][GEMM pieces][x][xin][qkv][q][o][d][n2][gu][act][attention].
struct BbLayout {
  size_t gemm, x, xin, qkv, q, o, d, n2, gu, act, attn, total, gemm_bytes, attn_bytes;
};

bool bb_layout(int B, int nr, int H, int L, const dspark_backbone_layer_t *layers, int ctx_rows_per_req, int C,
               BbLayout *lo) {
  const size_t Bb = static_cast<size_t>(B) * nr, M1 = Bb + static_cast<size_t>(B) * ctx_rows_per_req;
  size_t nqkv = 0, nq128 = 0, I = 0, gemm = 0, attn = 0;
  for (int l = 0; l < L; ++l) {
    const dspark_backbone_layer_t &ly = layers[l];
    const size_t nk = static_cast<size_t>(ly.nq + 2 * ly.nkv) * 128;
    nqkv = std::max(nqkv, nk);
    nq128 = std::max(nq128, static_cast<size_t>(ly.nq) * 128);
    I = std::max(I, static_cast<size_t>(ly.I));
    const size_t g[4] = {gemm_workspace_size(static_cast<int>(M1), static_cast<int>(nk), H),
                         gemm_workspace_size(static_cast<int>(Bb), H, ly.nq * 128),
                         gemm_workspace_size(static_cast<int>(Bb), 2 * ly.I, H),
                         gemm_workspace_size(static_cast<int>(Bb), H, ly.I)};
    for (size_t v : g) {
      if (v == 0) return false;
      gemm = std::max(gemm, v);
    }
    attn = std::max(attn, attention_workspace_bytes(B, nr, ly.nq, ly.nkv, C + nr));
  }
  size_t off = kHeader;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align_up(off + bytes, kWsAlign);
    return at;
  };
  lo->gemm = take(gemm);
  lo->x = take(Bb * H * 4);
  lo->xin = take(M1 * H * 2);
  lo->qkv = take(M1 * nqkv * 2);
  lo->q = take(Bb * nq128 * 2);
  lo->o = take(Bb * nq128 * 2);
  lo->d = take(Bb * H * 2);
  lo->n2 = take(Bb * H * 2);
  lo->gu = take(Bb * 2 * I * 2);
  lo->act = take(Bb * I * 2);
  lo->attn = take(attn);
  lo->total = off;
  lo->gemm_bytes = gemm;
  lo->attn_bytes = attn;
  return true;
}

dspark_status_t bb_check_layers(int B, int nr, int H, int L, const dspark_backbone_layer_t *layers, int cache_len,
                                int C) {
  if (!layers || L < 1 || L > 256) return DSPARK_ERR_INVALID_ARG;
  for (int l = 0; l < L; ++l) {
    const dspark_backbone_layer_t &ly = layers[l];
    if (!ly.w_in || !ly.w_post || !ly.w_qn || !ly.w_kn || !ly.w_qkv || !ly.w_o || !ly.w_gu || !ly.w_d ||
        !ly.k_cache || !ly.v_cache)
      return DSPARK_ERR_INVALID_ARG;
    if (ly.nq < 1 || ly.nkv < 1 || ly.nq % ly.nkv != 0 || ly.I < 64 || !(ly.theta > 1.0f))
      return DSPARK_ERR_INVALID_ARG;
    if (ly.I % 64 != 0 || nr * (ly.nq / ly.nkv) > kMaxAttnQueries || ly.nq + 2 * ly.nkv > 4096 ||
        2LL * ly.I > kMaxV)
      return DSPARK_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(ly.w_in) || !aligned16(ly.w_post) || !aligned16(ly.w_qn) || !aligned16(ly.w_kn) ||
        !aligned16(ly.w_qkv) || !aligned16(ly.w_o) || !aligned16(ly.w_gu) || !aligned16(ly.w_d) ||
        !aligned16(ly.k_cache) || !aligned16(ly.v_cache))
      return DSPARK_ERR_MISALIGNED;
  }
  (void)B;
  (void)H;
  (void)cache_len;
  (void)C;
  return DSPARK_OK;
}

}  // namespace

size_t dspark_backbone_block_workspace_size(int B, int nr, int H, int L, const dspark_backbone_layer_t *layers,
                                            int ctx_rows_per_req, int C) {
  if (B < 1 || nr < 2 || H < 64 || H % 64 != 0 || ctx_rows_per_req < 0 || C < 0) return 0;
  if (bb_check_layers(B, nr, H, L, layers, C + nr, C) != DSPARK_OK) return 0;
  BbLayout lo;
  return bb_layout(B, nr, H, L, layers, ctx_rows_per_req, C, &lo) ? lo.total : 0;
}

dspark_status_t dspark_backbone_block(const int32_t *tokens, int B, int nr, const dspark_bf16_t *embed, int V,
                                      int H, int L, const dspark_backbone_layer_t *layers,
                                      const dspark_bf16_t *w_final, int cache_len, int C, const dspark_bf16_t *ctx,
                                      int ctx_rows_per_req, int ctx_pos0, dspark_bf16_t *h_out, void *ws,
                                      size_t ws_bytes, void *stream) {
  if (!tokens || !embed || !w_final || !h_out || V < 1 || B < 1 || nr < 2 || C < 0 || ctx_rows_per_req < 0 ||
      ctx_pos0 < 0)
    return DSPARK_ERR_INVALID_ARG;
  if (ctx_rows_per_req > 0 && (!ctx || static_cast<long long>(ctx_pos0) + ctx_rows_per_req > cache_len))
    return DSPARK_ERR_INVALID_ARG;
  if (static_cast<long long>(C) + nr > cache_len) return DSPARK_ERR_INVALID_ARG;
  if (H < 64 || H % 64 != 0 || H > kMaxNormH || static_cast<long long>(B) * (nr + ctx_rows_per_req) > kMaxM ||
      V > kMaxV)
    return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (!aligned4(tokens) || !aligned16(embed) || !aligned16(w_final) || !aligned16(h_out) ||
      (ctx_rows_per_req > 0 && !aligned16(ctx)))
    return DSPARK_ERR_MISALIGNED;
  dspark_status_t st = bb_check_layers(B, nr, H, L, layers, cache_len, C);
  if (st != DSPARK_OK) return st;
  BbLayout lo;
  if (!bb_layout(B, nr, H, L, layers, ctx_rows_per_req, C, &lo)) return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if ((st = check_ws(ws, ws_bytes, lo.total)) != DSPARK_OK) return st;
  if ((st = check_device()) != DSPARK_OK) return st;
  cudaStream_t s = as_stream(stream);
  char *base = static_cast<char *>(ws);
  int *status = status_word(ws);
  void *gws = base + lo.gemm;
  float *x = reinterpret_cast<float *>(base + lo.x);
  uint16_t *xin = reinterpret_cast<uint16_t *>(base + lo.xin);
  uint16_t *qkv = reinterpret_cast<uint16_t *>(base + lo.qkv);
  uint16_t *q = reinterpret_cast<uint16_t *>(base + lo.q);
  uint16_t *o = reinterpret_cast<uint16_t *>(base + lo.o);
  uint16_t *d = reinterpret_cast<uint16_t *>(base + lo.d);
  uint16_t *n2 = reinterpret_cast<uint16_t *>(base + lo.n2);
  uint16_t *gu = reinterpret_cast<uint16_t *>(base + lo.gu);
  uint16_t *act = reinterpret_cast<uint16_t *>(base + lo.act);
  void *aws = base + lo.attn;
  const int Bb = B * nr, nc = B * ctx_rows_per_req, M1 = Bb + nc;
  const uint16_t *ctx16 = nc > 0 ? reinterpret_cast<const uint16_t *>(ctx) : nullptr;
  auto linear = [&](const void *xa, int M, int N, int K, const void *w, uint16_t *out, PieceView *view) {
    GemmProblem g;
    memset(&g, 0, sizeof(g));
    g.w = w;
    g.x[0] = xa;
    g.x_ld[0] = K;
    g.n_seg = 1;
    g.seg_k = K;
    g.N = N;
    g.M = M;
    g.out = out;
    g.ldo = N;
    g.out_bf16 = true;
    g.pieces_only = true;
    return gemm_launch(g, gws, lo.gemm_bytes, status, s, view);
  };
  PieceView vd;  // the last down projection (the next norm's residual delta)
  for (int l = 0; l < L; ++l) {
    const dspark_backbone_layer_t &ly = layers[l];
    const int nqkv = (ly.nq + 2 * ly.nkv) * 128;
    // block rows' input norm (the embedding gather for the first layer) and the
    // context rows', one launch
    st = norm_rows_launch(x, nullptr, 0, l == 0 ? reinterpret_cast<const uint16_t *>(embed) : nullptr,
                          l == 0 ? tokens : nullptr, V, nullptr, 0, reinterpret_cast<const uint16_t *>(ly.w_in), xin,
                          H, 0, Bb, H, status, s, ctx16, H, nc, l == 0 ? nullptr : &vd);
    if (st != DSPARK_OK) return st;
    PieceView vq, vo, vg;
    if ((st = linear(xin, M1, nqkv, H, ly.w_qkv, qkv, &vq)) != DSPARK_OK) return st;
    st = qk_norm_rope_launch(qkv, nqkv, ly.nq, ly.nkv, reinterpret_cast<const uint16_t *>(ly.w_qn),
                             reinterpret_cast<const uint16_t *>(ly.w_kn), ly.theta, q,
                             reinterpret_cast<uint16_t *>(ly.k_cache), reinterpret_cast<uint16_t *>(ly.v_cache),
                             cache_len, nr, C, Bb, s, nullptr, nqkv, ctx_rows_per_req, ctx_pos0, nc, &vq);
    if (st != DSPARK_OK) return st;
    st = attention_launch(q, reinterpret_cast<const uint16_t *>(ly.k_cache),
                          reinterpret_cast<const uint16_t *>(ly.v_cache), o, B, nr, ly.nq, ly.nkv, cache_len, C + nr,
                          aws, s);
    if (st != DSPARK_OK) return st;
    if ((st = linear(o, Bb, H, ly.nq * 128, ly.w_o, d, &vo)) != DSPARK_OK) return st;
    st = norm_rows_launch(x, nullptr, 0, nullptr, nullptr, 0, nullptr, 0, reinterpret_cast<const uint16_t *>(ly.w_post),
                          n2, H, 0, Bb, H, nullptr, s, nullptr, 0, 0, &vo);
    if (st != DSPARK_OK) return st;
    if ((st = linear(n2, Bb, 2 * ly.I, H, ly.w_gu, gu, &vg)) != DSPARK_OK) return st;
    if ((st = silu_mul_view_launch(vg, act, Bb, ly.I, s)) != DSPARK_OK) return st;
    if ((st = linear(act, Bb, H, ly.I, ly.w_d, d, &vd)) != DSPARK_OK) return st;
  }
  // final norm of the mask rows (the anchor rows left out, the rest compacted)
  return norm_rows_launch(x, nullptr, 0, nullptr, nullptr, 0, nullptr, 0, reinterpret_cast<const uint16_t *>(w_final),
                          reinterpret_cast<uint16_t *>(h_out), H, nr, Bb, H, nullptr, s, nullptr, 0, 0, &vd);
}

dspark_status_t dspark_silu_mul(const dspark_bf16_t *gu, dspark_bf16_t *act, int M, int I, void *stream) {
  if (!gu || !act || M < 1 || I < 8) return DSPARK_ERR_INVALID_ARG;
  if (I % 8 != 0 || M > kMaxM) return DSPARK_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(gu) || !aligned16(act)) return DSPARK_ERR_MISALIGNED;
  dspark_status_t st = check_device();
  if (st != DSPARK_OK) return st;
  return silu_mul_launch(gu, act, M, I, as_stream(stream));
}

}  // extern "C"
