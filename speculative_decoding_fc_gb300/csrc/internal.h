// Host-side declarations shared by the DSpark translation units.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "dspark.h"

namespace dspark {

constexpr size_t kWsAlign = 256;
constexpr int kMaxTaps = 8;
constexpr int kMaxK = 16;
constexpr int kMaxRank = 256;
constexpr int kMaxGemmCtas = 160;  // upper bound of the persistent GEMM grid
constexpr int kMaxV = 1 << 26;     // vocabulary cap (argmax words keep 26 index bits)

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// ------------------------------------------------------------------ GEMM
// out[m, n] = sum_k X[m, k] * W[n, k]   (bf16 in, fp32 accumulate)
// X is the concatenation along k of n_seg segments, each [M, seg_k] with row
// stride x_ld[s] elements.  out is fp32 or bf16 with row stride ldo.
struct GemmProblem {
  const void *w;          // [N, K] bf16
  const void *x[kMaxTaps];
  int64_t x_ld[kMaxTaps];
  int n_seg;
  int seg_k;              // K of one segment (multiple of 64)
  int N;                  // weight rows
  int M;                  // activation rows
  void *out;
  int64_t ldo;
  bool out_bf16;
  bool fp8;                 // E4M3 operands (w, x as uint8 codes); K multiple of 128
  const float *a_scale;     // FP8: per activation row
  const float *w_scale;     // FP8: per weight row
  bool pieces_only;         // bf16 out: split tiles are left as pieces for the reader
};

// Where a GEMM launched with pieces_only left its output: tiles held whole by one CTA
// are stored in `out` (bf16); every other tile is held as fp32 pieces, one per CTA
// that holds part of its k range, which the kernel reading the output adds in CTA
// order from 0 and rounds to bf16: the value the GEMM's own fix-up would have stored.
// Output (m, n) is in tile (n / 128) * tiles_m + m / BN; the CTA holding units
// [units * c / grid, units * (c + 1) / grid) of the tile-major unit order (kb_total
// units per tile) keeps its piece of tile t at partials[((c * 2 + s) * BN + m % BN) *
// 128 + n % 128], s = 0 for the tile its range starts in, else 1.
struct PieceView {
  const float *partials;
  const uint16_t *out;
  long long ldo, units;
  int kb_total, grid, BN, tiles_m, M;
};

size_t gemm_workspace_size(int M, int N, int K);
size_t gemm_workspace_size_fp8(int M, int N, int K);
// Bytes at the start of a GEMM workspace holding counters that must start at zero.
size_t gemm_counter_bytes(int M, int N, int K);
// Enqueues the GEMM.  ws must hold gemm_workspace_size bytes (zeroed once).
dspark_status_t gemm_launch(const GemmProblem &p, void *ws, size_t ws_bytes, int *status,
                            cudaStream_t stream, PieceView *view = nullptr);
// Two GEMMs in one cooperative launch, the second reading the first's output (same
// M and element type): the second's activation loads wait until every output tile of
// the first is stored.  Workspace: [256 B counters][first GEMM][second GEMM at
// gemm2_phase1_offset]; the counters and both GEMMs' tickets must start at zero.
size_t gemm2_workspace_size(int M, int N0, int K0, int N1, int K1);
size_t gemm2_phase1_offset(int M, int N0, int K0);
dspark_status_t gemm_launch2(const GemmProblem &p0, const GemmProblem &p1, void *ws,
                             size_t ws_bytes, int *status, cudaStream_t stream);

// ------------------------------------------------------------------ Markov chain
size_t chain_workspace_size(int B, int k, int V);
size_t chain_counter_bytes(int B, int k);
dspark_status_t chain_launch(float *logits, const uint16_t *w1, const uint16_t *w2, int r,
                             const int32_t *prev_token, int32_t *draft_tokens, float *q_stats,
                             int32_t *draft_len_fill, int B, int k, int V, void *ws,
                             int *status, cudaStream_t stream);
// Confidence head + truncation: over h alone (w1 == null) or over [h ; markov_w1[ctx]]
// (conf_w then has H + r entries); per-position or cumulative rule.
dspark_status_t confidence_launch(const uint16_t *h, const uint16_t *conf_w, float conf_b,
                                  float conf_tau, int cumulative, const uint16_t *w1, int r, int V,
                                  const int32_t *prev_token, int32_t *draft_tokens,
                                  int32_t *draft_len, float *conf_out, int B, int k, int H,
                                  int *status, cudaStream_t stream);

// ------------------------------------------------------------------ drafter backbone
dspark_status_t norm_rows_launch(float *x, const uint16_t *delta, int64_t ld_delta, const uint16_t *table,
                                 const int32_t *tok, int V, const uint16_t *in, int64_t ld_in,
                                 const uint16_t *w, uint16_t *out, int64_t ld_out, int group, int rows,
                                 int H, int *status, cudaStream_t stream, const uint16_t *in2 = nullptr,
                                 int64_t ld_in2 = 0, int rows2 = 0, const PieceView *dv = nullptr);
dspark_status_t qk_norm_rope_launch(const uint16_t *qkv, int64_t ld, int nq, int nkv, const uint16_t *wq,
                                    const uint16_t *wk, float theta, uint16_t *q_out, uint16_t *k_cache,
                                    uint16_t *v_cache, int cache_len, int rows_per_req, int pos0, int rows,
                                    cudaStream_t stream, const uint16_t *kv2 = nullptr, int64_t ld2 = 0,
                                    int rows_per_req2 = 1, int pos02 = 0, int rows2 = 0,
                                    const PieceView *qv = nullptr);
dspark_status_t silu_mul_view_launch(const PieceView &gv, uint16_t *act, int M, int I, cudaStream_t stream);
size_t attention_workspace_bytes(int B, int nr, int nq, int nkv, int nkeys);
dspark_status_t attention_launch(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                                 uint16_t *out, int B, int nr, int nq, int nkv, int cache_len, int nkeys,
                                 void *ws, cudaStream_t stream);
dspark_status_t silu_mul_launch(const uint16_t *gu, uint16_t *act, int M, int I, cudaStream_t stream);

// ------------------------------------------------------------------ FP8 quantisation
// codes[r, :] = E4M3(x[r, :] / scale[r]), scale = amax(row) / 448 (1 if zero); the
// row is the concatenation of nseg segments, each [rows, seg_cols] with row
// stride seg_ld elements.
dspark_status_t quantize_fp8_launch(const uint16_t *const *segs, int nseg, int64_t seg_ld,
                                    int rows, int seg_cols, uint8_t *codes, float *scales,
                                    cudaStream_t stream);

// ------------------------------------------------------------------ verify
// Row statistics of nrows fp32 rows of V entries: ms[r] = (max, sum exp(x - max)),
// argmax[r] = lowest index of the max (either output may be null; without ms only
// the argmax is reduced).
size_t row_stats_workspace_size(long long nrows, int V);
size_t row_stats_counter_bytes(long long nrows, int V);
dspark_status_t row_stats_launch(const float *rows, long long nrows, int V, float *ms,
                                 int32_t *argmax, void *ws, int *status, cudaStream_t stream);
// Decisions (and the draw) of verify from precomputed target-row statistics.
size_t verify_from_stats_workspace_size(int B, int V);
size_t verify_from_stats_counter_bytes(int B, int V);
dspark_status_t verify_from_stats_launch(int mode, const float *target, const float *t_ms,
                                         const int32_t *t_arg, const int32_t *drafts,
                                         const int32_t *draft_len, const float *zlog,
                                         const float *q_ms, uint64_t seed,
                                         const uint32_t *request_id, uint32_t step,
                                         int32_t *accepted_len, int32_t *next_token, int B, int k,
                                         int V, void *ws, int *status, cudaStream_t stream);
// Host-side argument checks shared by every verify entry point (nothing enqueued).
dspark_status_t verify_check_args(int mode, const float *target_logits,
                                  const int32_t *draft_tokens, const int32_t *draft_len,
                                  const float *draft_logits, const float *q_stats,
                                  const uint32_t *request_id, const int32_t *accepted_len,
                                  const int32_t *next_token, int B, int k, int V);
// The whole verify (row statistics, then decisions) in one workspace.
size_t verify_workspace_size(int B, int k, int V);
size_t verify_counter_bytes(int B, int k, int V);
dspark_status_t verify_launch(int mode, const float *target, const int32_t *drafts,
                              const int32_t *draft_len, const float *zlog, const float *q_stats,
                              uint64_t seed, const uint32_t *request_id, uint32_t step,
                              int32_t *accepted_len, int32_t *next_token, int B, int k, int V,
                              void *ws, int *status, cudaStream_t stream);

// ------------------------------------------------------------------ launches
// Whether kernels are launched with programmatic dependent launch (default on;
// DSPARK_NO_PDL=1 turns it off).
bool pdl_enabled();

// cudaLaunchKernelEx with programmatic stream serialization allowed (when enabled):
// the kernel may start before the previous kernel on the stream completes and
// orders itself with griddepcontrol.wait.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// ------------------------------------------------------------------ launch accounting
// Counts every kernel this library enqueues (reported by dspark_launch_count).
void count_launches(int n);

// ------------------------------------------------------------------ device info
int device_sm_count();  // cached per current device; 0 when no device
bool device_is_blackwell();

}  // namespace dspark
