/*
 * dspark.h - C ABI of the GB300 (sm_103a) DSpark / DFlash speculative-decoding
 * readout + verify hot path.
 *
 * The method (web pages this library follows):
 *   [PR620]  "Qwen3.8-27B DFlash drafter recipe - 72.2 tok/s on Arc Pro B70",
 *            the embedded DSpark port description: VanillaMarkov (markov_w1
 *            embedding, markov_w2 projection), AcceptRatePredictor
 *            (confidence head), propose() capturing the accepted bonus token,
 *            _greedy_sample applying the full-vocab bigram bias
 *            semi-autoregressively, _truncate_by_confidence.
 *   [CARD]   "Qwen3.8-27B-DSpark-vLLM" model card: draft config fields,
 *            "num_speculative_tokens": 7, "draft_sample_method":
 *            "probabilistic", taps at layers 4/16/28/40/52, fc 5 x 5120.
 *   [PR128]  "Qwen4Exp DFlash2 hidden-state capture": fc.weight
 *            [2560, 12800] = 5 concatenated layer outputs; acceptance length
 *            = accepted tokens per verification step; "verified by rejection
 *            sampling".
 *
 * Conventions shared by every entry point
 *   - All tensor pointers are DEVICE pointers owned by the caller (allocated
 *     e.g. by PyTorch).  The library allocates no device memory per call and
 *     keeps no pointer after a call returns.
 *   - Tensors are dense row-major; the innermost dimension is contiguous.
 *     bf16 operands read by the tensor-memory engine or with 128-bit loads
 *     (taps, fc_w, h, lm_w, markov_w2, conf_w) must start on a 16-byte
 *     boundary; every other pointer on a multiple of its element size
 *     (else DSPARK_ERR_MISALIGNED).
 *   - bf16 = IEEE bfloat16 bit pattern (dspark_bf16_t); fp32 = IEEE binary32.
 *   - stream is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Every call only enqueues work on it and returns; nothing
 *     synchronises the host.
 *   - ws / ws_bytes: a caller-owned DEVICE workspace of at least
 *     dspark_<call>_workspace_size(...) bytes, 256-byte aligned, ZERO-FILLED
 *     ONCE before its first use.  Every call leaves its counters at zero
 *     again.  The library remembers (on the host, per workspace address) the
 *     layout a workspace was last used with; a call with another call kind or
 *     other sizes first clears its own counter regions with cudaMemsetAsync on
 *     the call's stream, so one workspace may serve calls of any shape that
 *     fits.  Calls that share a workspace must not overlap in time (same
 *     stream, or ordered by events).  After a device-side error, zero the
 *     workspace again before reusing it.
 *   - Kernels are launched with programmatic dependent launch: a kernel may
 *     start while the previous kernel on the stream is finishing and waits for
 *     it (griddepcontrol.wait) before its first access to global memory, so
 *     results are as with plain stream order.  DSPARK_NO_PDL=1 in the
 *     environment launches them plainly.
 *   - Argument errors are detected on the host before anything is enqueued
 *     and returned as a negative dspark_status_t.  Errors the device finds
 *     (a token id outside [0, V), a bounded internal wait running out) are
 *     recorded in the first 4 bytes of ws and read with
 *     dspark_workspace_status(); the kernels then skip the offending access
 *     instead of faulting.
 *   - Sizes: B requests, k draft positions per block (1 <= k <= 16), H hidden
 *     size (multiple of 64), V vocabulary size (>= 1), r Markov rank
 *     (multiple of 8, <= 256), T taps (1..8).
 */
#ifndef DSPARK_H
#define DSPARK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int dspark_status_t;
typedef uint16_t dspark_bf16_t;

#define DSPARK_OK 0
#define DSPARK_ERR_INVALID_ARG (-1)       /* null pointer, negative size, bad mode */
#define DSPARK_ERR_UNSUPPORTED_SHAPE (-2) /* size outside the caps listed above */
#define DSPARK_ERR_MISALIGNED (-3)        /* pointer or row stride not 16-byte aligned */
#define DSPARK_ERR_WORKSPACE (-4)         /* workspace missing or smaller than required */
#define DSPARK_ERR_CUDA (-5)              /* a CUDA runtime or driver call failed */
#define DSPARK_ERR_DEVICE_TIMEOUT (-6)    /* (device) a bounded wait ran out; work skipped */
#define DSPARK_ERR_BAD_TOKEN (-7)         /* (device) token id outside [0, V) */
#define DSPARK_ERR_NO_DEVICE (-8)         /* the current GPU is not an sm_103 device */

/* Human-readable name of a status code.  Never returns NULL. */
const char *dspark_status_string(dspark_status_t status);

/* Library version, major * 10000 + minor * 100 + patch. */
int dspark_version(void);

/* Number of kernels this library has enqueued in this process so far (all
 * devices, all calls); a diagnostic for launch accounting. */
long long dspark_launch_count(void);

/* Reads the device-side status word at the start of ws (enqueued on stream,
 * then the host waits for the stream), stores it in *status_out and resets
 * it to 0.  DSPARK_OK means no device-side error since the last read. */
dspark_status_t dspark_workspace_status(void *ws, void *stream, int32_t *status_out);

/* ------------------------------------------------------------------------
 * fc projection  ([PR128] "fc.weight is [2560, 12800], i.e. 5 features of
 * width 2560", captured features are the layers' completed outputs; [CARD]
 * "the drafter's fc expects 5 x 5120", target hidden states read at layers
 * 4/16/28/40/52.)
 *
 *   h[m, n] = bf16_rne( sum_{j<T} sum_{c<H} taps[j][m, c] * fc_w[n, j*H + c] )
 *
 * accumulated in fp32 on the tensor cores; no bias, no normalisation.  The
 * concatenation of the taps is never materialised: taps is a HOST array of T
 * device pointers, tap j being the output of target layer target_layer_ids[j]
 * in list order, each [M, H] bf16 with row stride tap_ld elements
 * (tap_ld >= H, tap_ld % 8 == 0).  fc_w is [H, T*H] bf16 (PyTorch Linear
 * [out, in]); h_out is [M, H] bf16.  M >= 1 (decode: M = B*k block
 * positions; prefill: M = context tokens).
 * ---------------------------------------------------------------------- */
size_t dspark_fc_project_workspace_size(int M, int H, int T);
dspark_status_t dspark_fc_project(const dspark_bf16_t *const *taps, int T, int64_t tap_ld,
                                  const dspark_bf16_t *fc_w, dspark_bf16_t *h_out, int M,
                                  int H, void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * LM head over every block position of every request in one pass over the
 * [V, H] weight ([PR620] drafter readout; one pass serves all B*k rows).
 *
 *   logits[m, v] = sum_{c<H} h[m, c] * lm_w[v, c]      (fp32 accumulate)
 *
 * h [M, H] bf16, lm_w [V, H] bf16, logits [M, V] fp32.
 * ---------------------------------------------------------------------- */
size_t dspark_lm_head_workspace_size(int M, int H, int V);
dspark_status_t dspark_lm_head(const dspark_bf16_t *h, const dspark_bf16_t *lm_w,
                               float *logits, int M, int H, int V, void *ws,
                               size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * fc projection and LM head in ONE launch (as dspark_fc_project followed by
 * dspark_lm_head on its output):
 *   h[m, n]      = bf16_rne( sum_j sum_c taps[j][m, c] * fc_w[n, j*H + c] )
 *   logits[m, v] = sum_c h[m, c] * lm_w[v, c]                (fp32)
 * Same layouts as the two calls; h_out [M, H] bf16 (16-byte aligned) receives h.
 * One persistent cooperative kernel: a CTA that has finished its share of the
 * fc streams LM-head weight tiles while the other CTAs finish theirs; the LM
 * head's reads of h wait until every fc output tile is stored.  Results are
 * those of the two calls up to the fp32 summation order, and identical to them
 * when both launches use the same number of CTAs (one per SM once each GEMM
 * has at least 4 k-blocks of 128 bytes per SM, e.g. the 27B shapes).
 * ---------------------------------------------------------------------- */
size_t dspark_fc_lm_head_workspace_size(int M, int H, int T, int V);
dspark_status_t dspark_fc_lm_head(const dspark_bf16_t *const *taps, int T, int64_t tap_ld,
                                  const dspark_bf16_t *fc_w, const dspark_bf16_t *lm_w,
                                  dspark_bf16_t *h_out, float *logits, int M, int H, int V,
                                  void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Markov-biased semi-autoregressive greedy drafting ([PR620] VanillaMarkov;
 * _greedy_sample "applies the full-vocab bigram bias semi-autoregressively
 * across block positions (position i conditioned on position i-1's biased
 * prediction)"; propose() "captures the accepted bonus token as the Markov
 * previous-token context").
 *
 * For each request b and position i = 0..k-1, with prev_0 = prev_token[b]:
 *   e[t]    = w1[prev_i, t]                                   (bf16 -> fp32)
 *   bias[v] = fmaf chain over t = 0..r-1 of w2[v, t] * e[t], from +0.0f
 *   z[v]    = logits[b, i, v] + bias[v]                       (fp32 add)
 *   d_i     = smallest v with z[v] == max z   (-0 == +0; NaN never wins)
 *   prev_{i+1} = d_i
 * logits [B, k, V] fp32 is overwritten with z (the biased draft logits).
 * draft_tokens [B, k] int32 receives d; q_stats [B, k, 2] fp32 receives
 * (max z, sum_v exp(z[v] - max z)), the softmax statistics of the draft
 * distribution q used by probabilistic verify (may be NULL).
 * w1 [V, r] and w2 [V, r] bf16 (w2 is the Linear(r -> V) weight); w1 == NULL
 * means no bias (plain argmax), then w2 and r are ignored.
 * prev_token [B] int32 in [0, V) (else DSPARK_ERR_BAD_TOKEN is recorded and
 * that request is drafted without bias).  One cooperative launch covers all k
 * positions (one launch per position when a cooperative launch is refused, r is
 * not 16, 32, 64 or 128, V exceeds 1024 rows per SM, or the batch's contexts do
 * not fit in shared memory: B above 266 at V = 151936, r = 64 on 152 SMs).
 * q_stats == NULL selects a variant that reduces only the argmax (probabilistic
 * verify then reduces q's statistics itself).
 * ---------------------------------------------------------------------- */
size_t dspark_greedy_sample_workspace_size(int B, int k, int V, int r);
dspark_status_t dspark_greedy_sample(float *logits, const dspark_bf16_t *w1,
                                     const dspark_bf16_t *w2, int r,
                                     const int32_t *prev_token, int32_t *draft_tokens,
                                     float *q_stats, int B, int k, int V, void *ws,
                                     size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Confidence head and adaptive truncation alone ([PR620] AcceptRatePredictor,
 * _truncate_by_confidence, DSPARK_ADAPTIVE_BLOCK).  The pages give no
 * formula; the head is read as c[b, i] = sigmoid(conf_w . h[b*k+i] + conf_b),
 * tested per position: draft_len[b] = first i with c[b, i] < conf_tau (k if
 * none) and draft_tokens[b, i >= draft_len[b]] = -1 (in place).
 * conf_tau <= 0 keeps every position; conf_tau >= 1 keeps none.
 *   h [B*k, H] bf16 (the fc output), conf_w [H] bf16, draft_tokens [B, k]
 *   int32 (in/out), draft_len [B] int32 (out), conf_out [B, k] fp32 or NULL.
 * One kernel; needs no workspace.
 * ---------------------------------------------------------------------- */
dspark_status_t dspark_confidence_truncate(const dspark_bf16_t *h, const dspark_bf16_t *conf_w,
                                           float conf_b, float conf_tau, int32_t *draft_tokens,
                                           int32_t *draft_len, float *conf_out, int B, int k,
                                           int H, void *stream);

/* ------------------------------------------------------------------------
 * Confidence head that also sees the Markov context, and cumulative
 * truncation ([PR620] draft config fields enable_confidence_head,
 * confidence_head_with_markov, markov_rank; AcceptRatePredictor,
 * _truncate_by_confidence, DSPARK_ADAPTIVE_BLOCK).  The pages name
 * confidence_head_with_markov without a formula; the reading implemented:
 * one linear layer over the concatenation [h_i ; e_i], where e_i =
 * w1[ctx_i, :] is the Markov embedding of the token position i is
 * conditioned on (ctx_0 = prev_token[b], the bonus token; ctx_i = the draft
 * of position i-1):
 *   zc[b, i] = sum_c conf_w[c] h[b*k+i, c] + sum_t conf_w[H + t] w1[ctx_i, t]
 *              + conf_b,            c[b, i] = sigmoid(zc[b, i])
 * conf_w is [H + r] bf16 (16-byte aligned); w1 == NULL gives the plain head
 * (conf_w [H], prev_token and V unused).  Truncation rule:
 *   cumulative == 0: draft_len[b] = first i with c[b, i] < conf_tau (as
 *     dspark_confidence_truncate);
 *   cumulative != 0: draft_len[b] = first i with
 *     prod_{j <= i} c[b, j] < conf_tau  (evaluated as the running sum of
 *     log sigmoid(zc) against log conf_tau): the predicted probability that
 *     the whole prefix up to i is accepted.
 * conf_tau <= 0 keeps every position, conf_tau >= 1 keeps none.
 * draft_tokens [B, k] int32 (in: the chain's drafts, which give the
 * contexts; out: -1 from draft_len on), draft_len [B] int32, conf_out [B, k]
 * fp32 or NULL.  status: a device int32 (or NULL) where a context token
 * outside [0, V) is recorded as DSPARK_ERR_BAD_TOKEN (its Markov term is
 * then left out).  One kernel; needs no workspace.
 * ---------------------------------------------------------------------- */
dspark_status_t dspark_confidence_truncate_markov(const dspark_bf16_t *h,
                                                  const dspark_bf16_t *conf_w, float conf_b,
                                                  float conf_tau, int cumulative,
                                                  const dspark_bf16_t *w1, int r, int V,
                                                  const int32_t *prev_token,
                                                  int32_t *draft_tokens, int32_t *draft_len,
                                                  float *conf_out, int B, int k, int H,
                                                  int32_t *status, void *stream);

/* ------------------------------------------------------------------------
 * Whole drafter readout: LM head (as dspark_lm_head) + Markov greedy
 * drafting (as dspark_greedy_sample) + optional confidence truncation
 * ([PR620] AcceptRatePredictor "optional per-position acceptance-confidence
 * head", _truncate_by_confidence "adaptive draft block length").
 *
 * Confidence (when conf_w != NULL): c[b, i] = sigmoid(conf_w . h[b*k+i] +
 * conf_b), evaluated per position; draft_len[b] = first i with
 * c[b, i] < conf_tau (k if none); draft_tokens[b, i >= draft_len[b]] = -1.
 * conf_tau <= 0 keeps every position, conf_tau >= 1 keeps none.  Without a
 * confidence head draft_len[b] = k.
 *   h [B*k, H] bf16 (the fc output), lm_w [V, H] bf16,
 *   logits [B, k, V] fp32 (out: biased draft logits z),
 *   q_stats [B, k, 2] fp32 or NULL, draft_tokens [B, k] int32,
 *   draft_len [B] int32 or NULL, conf_out [B, k] fp32 or NULL.
 * ---------------------------------------------------------------------- */
size_t dspark_draft_readout_workspace_size(int B, int k, int H, int V, int r);
dspark_status_t dspark_draft_readout(const dspark_bf16_t *h, const dspark_bf16_t *lm_w,
                                     const dspark_bf16_t *w1, const dspark_bf16_t *w2, int r,
                                     const int32_t *prev_token, const dspark_bf16_t *conf_w,
                                     float conf_b, float conf_tau, float *logits,
                                     float *q_stats, int32_t *draft_tokens,
                                     int32_t *draft_len, float *conf_out, int B, int k, int H,
                                     int V, void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Verification of one draft block per request.
 *
 * mode 0, greedy exact match ([PR620] "greedy spec decode is lossless by
 * construction"): t_j = argmax target[b, j] (lowest index on ties);
 * accepted_len[b] = longest prefix (<= draft_len[b]) with
 * draft_tokens[b, j] == t_j; next_token[b] = t_{accepted_len}.
 *
 * mode 1, probabilistic ([CARD] "draft_sample_method": "probabilistic";
 * [PR128] "verified by rejection sampling"): p_j = softmax(target[b, j]),
 * q_j = softmax(draft_logits[b, j]) (one-hot at the draft when draft_logits
 * is NULL).  Positions are tested in order; draft d_j is accepted iff
 * u_j < p_j(d_j) / q_j(d_j).  At the first rejection j, next_token is drawn
 * from max(0, p_j - q_j) normalised (p_j if that is all zero); if every one
 * of the draft_len drafts is accepted, the bonus token is drawn from
 * p_{draft_len}.  The pages fix only these distributions; every draw here is
 * the Gumbel-max rule: the smallest v maximising log w_v + G_v, where w is
 * the (unnormalised) weight vector and G_v = -log(-log U_v), which samples
 * exactly from w normalised.
 * Uniforms: Philox4x32-10 (Salmon et al., SC'11) with key = (seed low 32
 * bits, seed high 32 bits).  Accept test of position j: counter
 * (request_id[b], j, step, 0), u_j = (word0 >> 8) * 2^-24.  Draw at block row
 * j: counter (request_id[b], j, step, 1 + v/4), word v mod 4, U_v =
 * (2 * (word >> 9) + 1) * 2^-24.
 *
 *   target_logits [B, k+1, V] fp32 (row k+1 of a block is the bonus row),
 *   draft_tokens [B, k] int32, draft_len [B] int32 or NULL (= k),
 *   draft_logits [B, k, V] fp32 (biased draft logits) or NULL,
 *   q_stats [B, k, 2] fp32 from dspark_greedy_sample, or NULL: then the
 *     statistics are recomputed from draft_logits (one more read of it),
 *   request_id [B] uint32 or NULL (= b),
 *   accepted_len [B] int32, next_token [B] int32 (outputs).
 * Mode 0 ignores draft_logits, q_stats, seed, request_id and step.
 * Enqueues dspark_row_stats over the target rows 0..draft_len[b] (and over the
 * draft-logit rows 0..draft_len[b]-1 when q_stats is NULL), then the decision
 * kernel of dspark_verify_from_stats: two or three kernels.
 * q_stats, when given, must be 8-byte aligned.
 * ---------------------------------------------------------------------- */
size_t dspark_verify_workspace_size(int B, int k, int V);
dspark_status_t dspark_verify(int mode, const float *target_logits,
                              const int32_t *draft_tokens, const int32_t *draft_len,
                              const float *draft_logits, const float *q_stats, uint64_t seed,
                              const uint32_t *request_id, uint32_t step,
                              int32_t *accepted_len, int32_t *next_token, int B, int k, int V,
                              void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Softmax statistics and argmax of fp32 rows: the part of verify that needs
 * only the logits of one distribution (p from the target rows, or q from the
 * draft-logit rows).  For each row r of rows [nrows, V] (row-major):
 *   ms_out[r]     = (max_v x[r, v], sum_v exp(x[r, v] - max))   fp32 pair
 *   argmax_out[r] = smallest v with x[r, v] == max               int32
 * (-0 == +0; NaN entries never win and add nothing; an all -inf row gives
 * (-inf, 0) and argmax 0).  Either output may be NULL (not both); with
 * ms_out == NULL only the argmax is reduced.  ms_out must be 8-byte aligned.
 * 1 <= nrows <= 2^24, 1 <= V <= 2^26.  One kernel: every CTA reduces a
 * 16384-entry slice of one row, the last CTA of a row merges the slices
 * (sum in fp64, rounded once to fp32).
 * Applied to the target logits [B, k+1, V] (nrows = B*(k+1)) this depends
 * on nothing the drafter computes, so it may run as soon as the target
 * logits exist, concurrently with drafting work on another stream.
 * ---------------------------------------------------------------------- */
size_t dspark_row_stats_workspace_size(int64_t nrows, int V);
dspark_status_t dspark_row_stats(const float *rows, int64_t nrows, int V, float *ms_out,
                                 int32_t *argmax_out, void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Verify with the row statistics already computed: the same decisions and
 * draws as dspark_verify, in ONE kernel.
 *   target_ms [B, k+1, 2] fp32 and target_argmax [B, k+1] int32: the
 *     dspark_row_stats outputs of target_logits (mode 0 needs target_argmax,
 *     mode 1 target_ms; rows past draft_len[b] are never read);
 *   q_stats [B, k, 2] fp32: required in mode 1 when draft_logits is given
 *     (from dspark_greedy_sample, or dspark_row_stats of the draft logits);
 * every other argument as for dspark_verify.  Mode 0: one warp per request
 * compares the drafts with the target argmaxes.  Mode 1: every CTA of a
 * request takes the request's accept/reject decisions (its drafted tokens,
 * the target and draft logits at them, the row statistics), then reduces one
 * 1024-entry slice of the Gumbel-max draw; the request's last CTA merges the
 * draw.
 * ---------------------------------------------------------------------- */
size_t dspark_verify_from_stats_workspace_size(int B, int k, int V);
dspark_status_t dspark_verify_from_stats(int mode, const float *target_logits,
                                         const float *target_ms, const int32_t *target_argmax,
                                         const int32_t *draft_tokens, const int32_t *draft_len,
                                         const float *draft_logits, const float *q_stats,
                                         uint64_t seed, const uint32_t *request_id, uint32_t step,
                                         int32_t *accepted_len, int32_t *next_token, int B, int k,
                                         int V, void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Allocation-free verify.  No counterpart in the pages: a library
 * convenience with the semantics, arguments and outputs of dspark_verify,
 * minus the workspace.
 *
 * For callers that cannot supply a workspace: code that a host framework
 * hands only its input and output buffers while it owns every other device
 * allocation (a serving engine's custom-operator interface, for instance),
 * and code that must not call cudaMalloc while it runs, because cudaMalloc
 * may synchronise the device or the process keeps to a fixed memory budget.
 *
 * Scratch: one fixed array of DSPARK_VERIFY_NOALLOC_MAX_BYTES inside the
 * library's device image, held by every GPU that loads the library until the
 * process exits.  Every call looks up the array's device address
 * (cudaGetSymbolAddress) with the current device; the first lookup on a
 * device may load the library's device code there, so make the first call on
 * each device before any stream capture.  Each call first clears the part of the
 * array it uses (cudaMemsetAsync on `stream`), then enqueues the same kernels
 * as dspark_verify.  Nothing is allocated: no cudaMalloc, no cudaFree.
 * All calls share the one array, so calls whose GPU work overlaps (streams
 * not ordered with respect to each other, or several host threads) race and
 * corrupt each other's results: order them.
 * Limit: dspark_verify_workspace_size(B, k, V) must not exceed
 * DSPARK_VERIFY_NOALLOC_MAX_BYTES (4 MiB; e.g. B = 64, k = 16, V = 262144
 * fits), otherwise DSPARK_ERR_WORKSPACE is returned and nothing is enqueued.
 * Arguments are checked as for dspark_verify before anything is enqueued: a
 * rejected call queues no GPU work and leaves the array untouched.
 * Device-side errors are recorded in the array's status word, which the next
 * call clears; this variant does not report them.
 * ---------------------------------------------------------------------- */
#define DSPARK_VERIFY_NOALLOC_MAX_BYTES ((size_t)4 << 20)
dspark_status_t dspark_verify_noalloc(int mode, const float *target_logits,
                                      const int32_t *draft_tokens, const int32_t *draft_len,
                                      const float *draft_logits, const float *q_stats,
                                      uint64_t seed, const uint32_t *request_id, uint32_t step,
                                      int32_t *accepted_len, int32_t *next_token, int B, int k,
                                      int V, void *stream);

/* ------------------------------------------------------------------------
 * FP8 (E4M3) drafter weights.  [PR620] ships the drafters as FP8 checkpoints
 * ("drafter-fp8-v5", "qwen3.8-27b-dflash-drafter-fp8-b70") but does not give
 * the scheme; the reading implemented here is per-row W8A8:
 *   E4M3 = OCP FP8 (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
 *   infinity, largest finite 448, code 0x7F/0xFF = NaN);
 *   scale[r] = amax_c |x[r, c]| / 448 in fp32 (IEEE division), 1 for an
 *   all-zero row; code[r, c] = E4M3(x[r, c] / scale[r]) (IEEE division),
 *   rounded to nearest even and saturated to +-448 (NaN -> 0x7F).
 * Weights are quantised once with dspark_quantize_fp8; the fc and LM-head
 * calls below quantise their activation rows the same way on every call
 * (into the workspace) and multiply the fp32 tensor-core sum by
 * scale_x[m] * scale_w[n] in fp32.
 * ---------------------------------------------------------------------- */

/* Quantises rows of a bf16 matrix given as nseg column segments (HOST array of
 * nseg device pointers, each [rows, seg_cols] with row stride seg_ld elements,
 * 16-byte aligned; seg_ld % 8 == 0) whose concatenation is the row.
 *   codes [rows, nseg*seg_cols] uint8 (16-byte aligned), scales [rows] fp32.
 * 1 <= nseg <= 8, seg_cols % 16 == 0, nseg*seg_cols <= 2^24, rows <= 2^24.
 * One kernel, no workspace; the result is bit-exact (no rounding choice is
 * left to the implementation). */
dspark_status_t dspark_quantize_fp8(const dspark_bf16_t *const *segs, int nseg, int64_t seg_ld,
                                    int rows, int seg_cols, uint8_t *codes, float *scales,
                                    void *stream);

/* FP8 fc projection: as dspark_fc_project with fc_w8 [H, T*H] E4M3 codes and
 * fc_scale [H] fp32 (from dspark_quantize_fp8 of the bf16 fc weight):
 *   x = concat_j taps[j][m, :]  quantised per row m -> (x8, sx[m])
 *   h[m, n] = bf16_rne( sx[m] * fc_scale[n] * sum_c E4M3(x8[m,c]) * E4M3(fc_w8[n,c]) )
 * H % 128 == 0.  Two kernels (activation quantisation, FP8 tensor-core GEMM). */
size_t dspark_fc_project_fp8_workspace_size(int M, int H, int T);
dspark_status_t dspark_fc_project_fp8(const dspark_bf16_t *const *taps, int T, int64_t tap_ld,
                                      const uint8_t *fc_w8, const float *fc_scale,
                                      dspark_bf16_t *h_out, int M, int H, void *ws,
                                      size_t ws_bytes, void *stream);

/* FP8 LM head: as dspark_lm_head with lm_w8 [V, H] E4M3 codes and lm_scale [V]
 * fp32; h [M, H] bf16 is quantised per row -> (h8, sh[m]) and
 *   logits[m, v] = sh[m] * lm_scale[v] * sum_c E4M3(h8[m,c]) * E4M3(lm_w8[v,c])
 * in fp32.  H % 128 == 0.  Two kernels. */
size_t dspark_lm_head_fp8_workspace_size(int M, int H, int V);
dspark_status_t dspark_lm_head_fp8(const dspark_bf16_t *h, const uint8_t *lm_w8,
                                   const float *lm_scale, float *logits, int M, int H, int V,
                                   void *ws, size_t ws_bytes, void *stream);

/* ========================================================================
 * Drafter backbone (N1).  The pages name the drafter class ([PR620]
 * "DSparkDraftModel(DFlashQwen3ForCausalLM)", "the DFlash backbone"; [CARD]
 * "Qwen3DSparkModel selects the Qwen3 implementation") and its config fields
 * (layer_types, head_dim, mask_token_id, projector_type) without a forward
 * pass.  The reading built here: L pre-norm decoder layers of the Qwen3 form run
 * the draft block (the anchor token, then k mask tokens) over the fc'd context:
 *   n = rmsnorm(x); q,k,v = n.[Wq;Wk;Wv]^T; per-head rmsnorm of q, k; rotary
 *   (NeoX, theta); o = attention over [context keys; block keys]; x += o.Wo^T;
 *   n2 = rmsnorm(x); x += (silu(n2.Wg^T) * n2.Wu^T).Wd^T
 * and the final rmsnorm of the mask positions is the LM head's input.  The
 * projections are dspark_linear; the calls below are the pieces between them.
 * head_dim is 128.  rmsnorm(x) = x / sqrt(mean(x^2) + 1e-6) * w; all arithmetic
 * fp32, bf16 outputs rounded to nearest even.  Rows are 16-byte aligned with row
 * strides (ld) a multiple of 8 elements.  Device-side errors: only a token
 * outside [0, V) in dspark_embed_rmsnorm (recorded in the optional status word,
 * the token clamped).  None of these calls allocates; all enqueue on `stream`.
 * ======================================================================== */

/* out[m, n] = sum_k x[m, k] * w[n, k]: the tcgen05 GEMM of the fc and LM head
 * with one activation segment.  x [M, K] bf16 (row stride x_ld), w [N, K] bf16,
 * out [M, N] (row stride out_ld) bf16 when out_bf16, else fp32.  K % 64 == 0.
 * Workspace: dspark_linear_workspace_size bytes, 256-byte aligned, zeroed before
 * its first use; calls sharing one workspace must be ordered on the GPU. */
size_t dspark_linear_workspace_size(int M, int N, int K);
dspark_status_t dspark_linear(const dspark_bf16_t *x, int64_t x_ld, const dspark_bf16_t *w, void *out,
                              int64_t out_ld, int out_bf16, int M, int N, int K, void *ws, size_t ws_bytes,
                              void *stream);

/* The block's inputs: x_out[r, :] = table[tokens[r], :] (fp32 residual, [rows, H])
 * and n_out[r, :] = bf16(rmsnorm(x_out[r, :]) * w) ([rows, H]).  table [V, H] bf16
 * (the LM head's weight: tied embeddings).  H % 8 == 0, H <= 8192. */
dspark_status_t dspark_embed_rmsnorm(const dspark_bf16_t *table, int V, const int32_t *tokens,
                                     const dspark_bf16_t *w, float *x_out, dspark_bf16_t *n_out, int rows,
                                     int H, int32_t *status, void *stream);

/* Residual add and norm: x[r, :] += delta[r, :] (fp32 add of the bf16 delta;
 * delta may be NULL), then out = bf16(rmsnorm(x[r, :]) * w).  group > 0: rows come
 * in groups of `group` (a request's block); the first row of each group (the
 * anchor) is not written and the others are stored compacted, row
 * (r / group) * (group - 1) + r % group - 1 (the final norm feeding the LM head). */
dspark_status_t dspark_add_rmsnorm(float *x, const dspark_bf16_t *delta, int64_t delta_ld,
                                   const dspark_bf16_t *w, dspark_bf16_t *out, int64_t out_ld, int group,
                                   int rows, int H, void *stream);

/* out = bf16(rmsnorm(in) * w) of bf16 rows (the context features' input norm). */
dspark_status_t dspark_rmsnorm_bf16(const dspark_bf16_t *in, int64_t in_ld, const dspark_bf16_t *w,
                                    dspark_bf16_t *out, int64_t out_ld, int rows, int H, void *stream);

/* Per-head q/k norm and rotary embedding, into the attention buffers.  Row r of
 * qkv (B * rows_per_req rows, stride ld) holds [q heads (nq x 128, absent when
 * nq == 0) | k heads (nkv x 128) | v heads (nkv x 128)]; it belongs to request
 * r / rows_per_req at position p = pos0 + r % rows_per_req.  Each q and k head:
 * y = rmsnorm(head) * norm_w, then (y1, y2) -> (y1 cos - y2 sin, y2 cos + y1 sin)
 * with y1 = dims 0..63, y2 = dims 64..127 and angle p * theta^(-2d/128).  q goes to
 * q_out [B * rows_per_req, nq, 128]; k and v go to slot p of the caches
 * k_cache, v_cache [B, cache_len, nkv, 128] (bf16).  pos0 + rows_per_req <= cache_len. */
dspark_status_t dspark_qk_norm_rope(const dspark_bf16_t *qkv, int64_t ld, int nq, int nkv,
                                    const dspark_bf16_t *q_norm_w, const dspark_bf16_t *k_norm_w, float theta,
                                    dspark_bf16_t *q_out, dspark_bf16_t *k_cache, dspark_bf16_t *v_cache, int B,
                                    int cache_len, int rows_per_req, int pos0, void *stream);

/* The block's input norm and the new context rows' input norm in one launch (the
 * two are independent; each row's result is the one dspark_embed_rmsnorm,
 * dspark_add_rmsnorm or dspark_rmsnorm_bf16 gives).  Block rows r < rows: when
 * table != NULL, x[r, :] = table[tokens[r], :] (the embedding gather, as
 * dspark_embed_rmsnorm), else x[r, :] += delta[r, :] (delta may be NULL, as
 * dspark_add_rmsnorm with group 0); out[r, :] = bf16(rmsnorm(x[r, :]) * w).  Context
 * rows j < ctx_rows: out[rows + j, :] = bf16(rmsnorm(ctx[j, :]) * w).  x [rows, H]
 * fp32, out rows with stride out_ld, ctx rows with stride ctx_ld (bf16); a token
 * outside [0, V) is recorded in *status (DSPARK_ERR_BAD_TOKEN) and clamped. */
dspark_status_t dspark_block_context_rmsnorm(float *x, const dspark_bf16_t *delta, int64_t delta_ld,
                                             const dspark_bf16_t *table, int V, const int32_t *tokens,
                                             const dspark_bf16_t *ctx, int64_t ctx_ld, int ctx_rows,
                                             const dspark_bf16_t *w, dspark_bf16_t *out, int64_t out_ld, int rows,
                                             int H, int32_t *status, void *stream);

/* dspark_qk_norm_rope of the block rows and of the new context rows in one launch:
 * the block part exactly as dspark_qk_norm_rope (qkv, ld, nq, nkv, ..., B,
 * rows_per_req, pos0); context row j (B * ctx_rows_per_req rows, stride ctx_ld)
 * holds [k heads | v heads] x 128, belongs to request j / ctx_rows_per_req at
 * position ctx_pos0 + j % ctx_rows_per_req, and goes to the caches like a block
 * row's k and v.  ctx_rows_per_req = 0: the block rows alone. */
dspark_status_t dspark_qk_norm_rope_block_context(const dspark_bf16_t *qkv, int64_t ld, int nq, int nkv,
                                                  const dspark_bf16_t *q_norm_w, const dspark_bf16_t *k_norm_w,
                                                  float theta, dspark_bf16_t *q_out, dspark_bf16_t *k_cache,
                                                  dspark_bf16_t *v_cache, int B, int cache_len, int rows_per_req,
                                                  int pos0, const dspark_bf16_t *ctx_kv, int64_t ctx_ld,
                                                  int ctx_rows_per_req, int ctx_pos0, void *stream);

/* Grouped-query attention of the block rows over the cache:
 *   out[b, i, j, :] = sum_t softmax_t(q[b, i, j, :] . K[b, t, j / (nq/nkv), :] / sqrt(128))
 *                     * V[b, t, j / (nq/nkv), :],   t = 0 .. nkeys - 1
 * q, out [B, nr, nq, 128] bf16; caches [B, cache_len, nkv, 128] bf16.  No mask:
 * every block row sees every key below nkeys.  nr * nq / nkv <= 48.  Two kernels
 * (64-key slices, then the merge); workspace dspark_attention_workspace_size bytes
 * (no zeroing needed). */
size_t dspark_attention_workspace_size(int B, int nr, int nq, int nkv, int nkeys);
dspark_status_t dspark_attention(const dspark_bf16_t *q, const dspark_bf16_t *k_cache,
                                 const dspark_bf16_t *v_cache, dspark_bf16_t *out, int B, int nr, int nq,
                                 int nkv, int cache_len, int nkeys, void *ws, size_t ws_bytes, void *stream);

/* act[m, c] = bf16(silu(gu[m, c]) * gu[m, I + c]), silu(g) = g / (1 + e^-g);
 * gu [M, 2I] bf16 (the gate|up GEMM output), act [M, I].  I % 8 == 0. */
dspark_status_t dspark_silu_mul(const dspark_bf16_t *gu, dspark_bf16_t *act, int M, int I, void *stream);

/* ------------------------------------------------------------------------
 * The drafter backbone's block pass, all layers in one call ([PR620]
 * DSparkDraftModel, "the DFlash backbone"; the layer form is a reading: the
 * Qwen3 pre-norm decoder layer, see the calls above).  Per layer, with the
 * block rows x (fp32 residual) and the new context rows ctx:
 *   n      = rmsnorm(x) * w_in (first layer: x = embed[tokens])   and the
 *            context rows' rmsnorm(ctx) * w_in, one launch
 *   qkv    = [n ; ctx rows' norm] . w_qkv^T (one GEMM)
 *   q      = qk norm + rotary of the block rows (positions C .. C + nr - 1); k, v
 *            of the block rows and of the context rows (positions ctx_pos0 ..)
 *            into the layer's caches, one launch
 *   o      = attention over cache slots 0 .. C + nr - 1
 *   x     += o . w_o^T;  n2 = rmsnorm(x) * w_post
 *   act    = silu(n2 . w_g^T) * (n2 . w_u^T)
 *   x     += act . w_d^T
 * then h_out = rmsnorm(x) * w_final of the mask rows (rows 1 .. nr - 1 of each
 * request), the LM head's input.  Every value equals the one the separate calls
 * above give (dspark_block_context_rmsnorm, dspark_linear,
 * dspark_qk_norm_rope_block_context, dspark_attention, dspark_add_rmsnorm,
 * dspark_silu_mul): the projections' split tiles are added by the kernel that
 * reads them, in the same order, instead of by the GEMM.
 *   tokens [B, nr] int32 (the anchor, then nr - 1 mask tokens); embed [V, H] bf16
 *   (the LM head's weight: tied embeddings); layers: a HOST array of L structs
 *   (device pointers inside); the caches hold the context keys and values at
 *   slots 0 .. C - 1 (ctx_rows_per_req of them, from ctx_pos0, written here);
 *   ctx [B * ctx_rows_per_req, H] bf16 or NULL with ctx_rows_per_req = 0;
 *   h_out [B * (nr - 1), H] bf16.  H % 64 == 0, H <= 8192, I % 64 == 0,
 *   nr * nq / nkv <= 48, C + nr <= cache_len.  The workspace
 *   (dspark_backbone_block_workspace_size bytes, 256-byte aligned) needs no
 *   zeroing; device errors (a token outside [0, V), a GEMM wait running out) go
 *   to its status word.
 * ---------------------------------------------------------------------- */
typedef struct {
  const dspark_bf16_t *w_in, *w_post;  /* input and post-attention norm weights [H] */
  const dspark_bf16_t *w_qn, *w_kn;    /* per-head q and k norm weights [128] */
  const dspark_bf16_t *w_qkv;          /* [(nq + 2 nkv) * 128, H]: Wq; Wk; Wv */
  const dspark_bf16_t *w_o;            /* [H, nq * 128] */
  const dspark_bf16_t *w_gu;           /* [2 I, H]: Wg; Wu */
  const dspark_bf16_t *w_d;            /* [H, I] */
  dspark_bf16_t *k_cache, *v_cache;    /* [B, cache_len, nkv, 128] */
  int nq, nkv, I;
  float theta;                         /* rotary base */
} dspark_backbone_layer_t;

size_t dspark_backbone_block_workspace_size(int B, int nr, int H, int L, const dspark_backbone_layer_t *layers,
                                            int ctx_rows_per_req, int C);
dspark_status_t dspark_backbone_block(const int32_t *tokens, int B, int nr, const dspark_bf16_t *embed, int V,
                                      int H, int L, const dspark_backbone_layer_t *layers,
                                      const dspark_bf16_t *w_final, int cache_len, int C, const dspark_bf16_t *ctx,
                                      int ctx_rows_per_req, int ctx_pos0, dspark_bf16_t *h_out, void *ws,
                                      size_t ws_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_H */
