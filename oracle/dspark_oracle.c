/*
 * DSpark readout + verify oracle: plain, slow, obviously-correct CPU code.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this file's library.  The CUDA product
 * path never calls it and shares no code with it.
 *
 * Everything floating-point is accumulated in IEEE binary64, in the plain
 * ascending order of the definitions, except where the method fixes a
 * narrower contract:
 *   - the fc output h is a bf16 tensor (round-to-nearest-even of the fp32
 *     value of the fp64 sum);
 *   - the draft logits the LM head returns are fp32;
 *   - the Markov bias of one vocabulary entry is a sequential chain of
 *     single-precision fused multiply-adds over the rank index, starting from
 *     +0.0f, and the biased logit is the fp32 sum of logit and bias.
 * Build with -ffp-contract=off so that no compiler turns a*b+c into an fma
 * behind our back (gcc on aarch64 contracts by default).
 *
 * Sources (web pages on DFlash/DSpark speculative decoding):
 *   [PR620]  "Qwen3.8-27B DFlash drafter recipe - 72.2 tok/s on Arc Pro B70",
 *            embedded DSpark port description: VanillaMarkov (markov_w1
 *            embedding + markov_w2 projection), AcceptRatePredictor,
 *            propose() bonus-token capture, _greedy_sample
 *            (semi-autoregressive full-vocab bias), _truncate_by_confidence.
 *   [CARD]   "Qwen3.8-27B-DSpark-vLLM" model card: config fields
 *            (target_layer_ids, markov_rank, enable_confidence_head),
 *            "draft_sample_method": "probabilistic", taps 4/16/28/40/52,
 *            fc expects 5 x 5120.
 *   [PR128]  "Qwen4Exp DFlash2 hidden-state capture": fc.weight [2560,12800]
 *            = 5 concatenated features; captured tensor is the layer output;
 *            "verified by rejection sampling"; acceptance length definition.
 * Where the pages give only words, the reading taken is stated beside the
 * function.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_NONFINITE 2
#define ORACLE_ERR_TOKEN 3

/* ------------------------------------------------------------------ */
/* bfloat16 <-> float                                                  */
/* ------------------------------------------------------------------ */

/* A bf16 value is the upper half of an IEEE binary32 word. */
static float bf16_bits_to_float(uint16_t b) {
    uint32_t x = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &x, sizeof f);
    return f;
}

/* Round a binary32 value to the nearest bf16, ties to even.  NaN stays NaN
 * (quiet bit forced so the truncated mantissa cannot become zero). */
uint16_t oracle_f32_to_bf16(float f) {
    uint32_t x;
    memcpy(&x, &f, sizeof x);
    if ((x & 0x7f800000u) == 0x7f800000u && (x & 0x007fffffu) != 0u)
        return (uint16_t)((x >> 16) | 0x0040u);
    uint32_t keep_lsb = (x >> 16) & 1u;
    x += 0x7fffu + keep_lsb;
    return (uint16_t)(x >> 16);
}

float oracle_bf16_to_f32(uint16_t b) { return bf16_bits_to_float(b); }

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------ */
/* Philox4x32-10 counter-based generator                               */
/* ------------------------------------------------------------------ */
/*
 * Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3"
 * (SC'11), Philox-4x32 with 10 rounds.  One round multiplies counter words
 * 0 and 2 by the two round multipliers, takes the 64-bit products apart into
 * high and low halves, and rebuilds the four words as
 *   (hi(M1*c2) ^ c1 ^ k0,  lo(M1*c2),  hi(M0*c0) ^ c3 ^ k1,  lo(M0*c0)).
 * Between rounds the two key words advance by the Weyl constants (golden
 * ratio and sqrt(3)-1, scaled to 32 bits).
 */
static const uint32_t PHILOX_MUL0 = 0xD2511F53u;
static const uint32_t PHILOX_MUL1 = 0xCD9E8D57u;
static const uint32_t PHILOX_WEYL0 = 0x9E3779B9u;
static const uint32_t PHILOX_WEYL1 = 0xBB67AE85u;

void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2],
                          uint32_t out[4]) {
    uint32_t c[4] = {ctr_in[0], ctr_in[1], ctr_in[2], ctr_in[3]};
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += PHILOX_WEYL0;
            k1 += PHILOX_WEYL1;
        }
        uint64_t p0 = (uint64_t)PHILOX_MUL0 * (uint64_t)c[0];
        uint64_t p1 = (uint64_t)PHILOX_MUL1 * (uint64_t)c[2];
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c[1] ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c[3] ^ k1;
        uint32_t n3 = lo0;
        c[0] = n0; c[1] = n1; c[2] = n2; c[3] = n3;
    }
    out[0] = c[0]; out[1] = c[1]; out[2] = c[2]; out[3] = c[3];
}

/* The uniforms of one verify position.  Counter = (request id, position in
 * the block, decode step, 0); key = the 64-bit seed split low/high.  Word 0
 * feeds the accept test (word 1 is reported too but unused: draws take their
 * noise from counters with a non-zero last word).  A uniform is the top 24
 * bits of the word times 2^-24: exact in binary32 and binary64, in [0, 1). */
static void verify_uniforms(uint64_t seed, uint32_t request, uint32_t pos,
                            uint32_t step, double *u_accept, double *u_sample) {
    uint32_t ctr[4] = {request, pos, step, 0u};
    uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
    uint32_t w[4];
    oracle_philox4x32_10(ctr, key, w);
    *u_accept = (double)(w[0] >> 8) * (1.0 / 16777216.0);
    *u_sample = (double)(w[1] >> 8) * (1.0 / 16777216.0);
}

void oracle_verify_uniforms(uint64_t seed, uint32_t request, uint32_t pos,
                            uint32_t step, double out[2]) {
    verify_uniforms(seed, request, pos, step, &out[0], &out[1]);
}

/* ------------------------------------------------------------------ */
/* fc projection: h = bf16( concat(tap_0..tap_{T-1}) . W_fc^T )        */
/* ------------------------------------------------------------------ */
/*
 * [PR128] fc.weight [2560, 12800]: five features of width 2560,
 * concatenated in target_layer_ids order; [CARD] "fc expects 5 x 5120".
 * W_fc is stored [out = H, in = T*H] (PyTorch Linear layout).  No bias and
 * no normalisation are mentioned on the pages, so none is applied.
 *   taps[j]    : M x H bf16, row stride tap_ld elements
 *   fc_w       : N x (T*H) bf16, row-major (N = H for the method; a smaller N
 *                computes the first N output features only)
 *   h_out      : M x N bf16 (row stride N)
 *   h_f32      : optional M x N fp32 copy of the value before bf16 rounding
 */
int oracle_fc_project(const uint16_t *const *taps, int T, int64_t tap_ld,
                      const uint16_t *fc_w, int N, int M, int H, uint16_t *h_out,
                      float *h_f32) {
    if (T < 1 || M < 0 || H < 1 || N < 1 || tap_ld < H || !taps || !fc_w || !h_out)
        return ORACLE_ERR_ARG;
    const int64_t K = (int64_t)T * H;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        const uint16_t *wrow = fc_w + n * K;
        for (int m = 0; m < M; ++m) {
            double acc = 0.0;
            for (int j = 0; j < T; ++j) {
                const uint16_t *arow = taps[j] + (int64_t)m * tap_ld;
                const uint16_t *wseg = wrow + (int64_t)j * H;
                for (int c = 0; c < H; ++c)
                    acc += (double)bf16_bits_to_float(arow[c]) *
                           (double)bf16_bits_to_float(wseg[c]);
            }
            float a32 = (float)acc;
            h_out[(int64_t)m * N + n] = oracle_f32_to_bf16(a32);
            if (h_f32) h_f32[(int64_t)m * N + n] = a32;
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* LM head: logits = h . W_lm^T  (fp32 out)                            */
/* ------------------------------------------------------------------ */
/*
 * Every draft-block position of every request goes through the same LM
 * head; the draft logits are fp32.  W_lm is [V, H].
 */
int oracle_lm_head(const uint16_t *h, int M, int H, const uint16_t *lm_w,
                   int64_t V, float *logits) {
    if (M < 0 || H < 1 || V < 1 || !h || !lm_w || !logits) return ORACLE_ERR_ARG;
    double *hd = (double *)malloc(sizeof(double) * (size_t)M * (size_t)H + 8);
    if (!hd) return ORACLE_ERR_ARG;
    for (int64_t i = 0; i < (int64_t)M * H; ++i) hd[i] = (double)bf16_bits_to_float(h[i]);
#pragma omp parallel for schedule(static)
    for (int64_t v = 0; v < V; ++v) {
        const uint16_t *wrow = lm_w + v * H;
        for (int m = 0; m < M; ++m) {
            const double *hrow = hd + (int64_t)m * H;
            double acc = 0.0;
            for (int c = 0; c < H; ++c)
                acc += hrow[c] * (double)bf16_bits_to_float(wrow[c]);
            logits[(int64_t)m * V + v] = (float)acc;
        }
    }
    free(hd);
    return ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* Semi-autoregressive Markov-biased greedy drafting                   */
/* ------------------------------------------------------------------ */
/*
 * [PR620] VanillaMarkov: markov_w1 is an embedding [V, r], markov_w2 a
 * projection r -> V (stored [V, r]); _greedy_sample applies the full-vocab
 * bigram bias across block positions, position i conditioned on position
 * i-1's biased prediction, and propose() supplies the accepted bonus token
 * as the context of position 0.  Reading taken: bias(prev) = W2 . W1[prev]
 * with no nonlinearity, scale or bias term.
 *
 * For request b and block position i (0 <= i < k):
 *   e[t]     = W1[prev_i, t]                              (bf16 -> fp32)
 *   bias[v]  = fma chain over t = 0..r-1 of W2[v, t] * e[t], from +0.0f
 *   z[v]     = logits[b, i, v] + bias[v]                  (fp32 add)
 *   d_i      = smallest v attaining max_v z[v]            (-0 == +0)
 *   prev_{i+1} = d_i
 * Also the softmax row statistics of z (the draft distribution q):
 *   q_max[b,i] = max_v z[v],  q_sumexp[b,i] = sum_v exp(z[v] - q_max)  (fp64)
 * and, for near-tie accounting, top2_gap[b,i] = z[d_i] - (largest z[v] over
 * v != d_i) in fp64.
 * logits is overwritten with z.  w1 == NULL means no bias (plain argmax).
 * Returns ORACLE_ERR_NONFINITE on a non-finite z, ORACLE_ERR_TOKEN on a
 * prev token outside [0, V).
 */
int oracle_greedy_sample(float *logits, int B, int k, int64_t V,
                         const uint16_t *w1, const uint16_t *w2, int r,
                         const int32_t *prev, int32_t *draft_tokens,
                         double *q_max, double *q_sumexp, double *top2_gap) {
    if (B < 0 || k < 1 || V < 1 || !logits || !prev || !draft_tokens) return ORACLE_ERR_ARG;
    if (w1 && (!w2 || r < 1)) return ORACLE_ERR_ARG;
    int status = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        float *e = (float *)malloc(sizeof(float) * (size_t)(r > 0 ? r : 1));
        int32_t p = prev[b];
        for (int i = 0; i < k; ++i) {
            float *row = logits + ((int64_t)b * k + i) * V;
            if (w1) {
                if (p < 0 || (int64_t)p >= V) {
#pragma omp atomic write
                    status = ORACLE_ERR_TOKEN;
                    break;
                }
                for (int t = 0; t < r; ++t)
                    e[t] = bf16_bits_to_float(w1[(int64_t)p * r + t]);
                for (int64_t v = 0; v < V; ++v) {
                    float acc = 0.0f;
                    for (int t = 0; t < r; ++t)
                        acc = fmaf(bf16_bits_to_float(w2[v * r + t]), e[t], acc);
                    row[v] = row[v] + acc;
                }
            }
            int64_t best = 0;
            for (int64_t v = 0; v < V; ++v) {
                if (!isfinite(row[v])) {
#pragma omp atomic write
                    status = ORACLE_ERR_NONFINITE;
                }
                if (row[v] > row[best]) best = v;
            }
            double mx = (double)row[best];
            double s = 0.0, second = -INFINITY;
            for (int64_t v = 0; v < V; ++v) {
                s += exp((double)row[v] - mx);
                if (v != best && (double)row[v] > second) second = (double)row[v];
            }
            draft_tokens[(int64_t)b * k + i] = (int32_t)best;
            if (q_max) q_max[(int64_t)b * k + i] = mx;
            if (q_sumexp) q_sumexp[(int64_t)b * k + i] = s;
            if (top2_gap) top2_gap[(int64_t)b * k + i] = mx - second;
            p = (int32_t)best;
        }
        free(e);
    }
    return status;
}

/* ------------------------------------------------------------------ */
/* Softmax statistics and argmax of rows                               */
/* ------------------------------------------------------------------ */
/*
 * The per-row quantities verify needs from one distribution's logits (p from
 * the target rows, q from the draft-logit rows; [PR128] "verified by
 * rejection sampling", [CARD] "draft_sample_method": "probabilistic"):
 *   mx[r]  = max_v x[r, v]                    (-inf when every entry is -inf)
 *   se[r]  = sum_v exp(x[r, v] - mx[r])       (fp64; 0 when mx is -inf)
 *   arg[r] = smallest v with x[r, v] == mx[r] (0 when every entry is -inf)
 * NaN entries are skipped (they neither win nor add).  -0 == +0.
 */
int oracle_row_stats(const float *x, int64_t nrows, int64_t V, double *mx, double *se,
                     int32_t *arg) {
    if (nrows < 0 || V < 1 || !x) return ORACLE_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < nrows; ++r) {
        const float *row = x + r * V;
        double m = -INFINITY;
        int64_t best = 0;
        int found = 0;
        for (int64_t v = 0; v < V; ++v) {
            const double xv = (double)row[v];
            if (xv != xv) continue;
            if (!found || xv > m) {
                m = xv;
                best = v;
                found = 1;
            }
        }
        double s = 0.0;
        if (m != -INFINITY)
            for (int64_t v = 0; v < V; ++v) {
                const double xv = (double)row[v];
                if (xv == xv) s += exp(xv - m);
            }
        if (mx) mx[r] = m;
        if (se) se[r] = s;
        if (arg) arg[r] = (int32_t)best;
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* Confidence head and adaptive truncation                             */
/* ------------------------------------------------------------------ */
/*
 * [PR620] AcceptRatePredictor gives a per-position acceptance confidence;
 * _truncate_by_confidence shortens the block at a threshold.  The pages
 * give no formula; the reading taken is c_i = sigmoid(w . h_i + b), where
 * h_i is the fc output of block position i, tested per position (not as a
 * running product): the block keeps positions 0..L-1 where L is the first
 * position with c_i < tau (k if none).  c >= tau  <=>  w.h+b >= logit(tau),
 * so the decision needs no exponential.  Positions >= L become -1.
 *   zc[b,i]   = w . h_{b,i} + b    (fp64)
 *   conf[b,i] = 1 / (1 + exp(-zc)) (fp64)
 * tau <= 0 keeps every position; tau >= 1 keeps none.
 */
int oracle_confidence(const uint16_t *h, int B, int k, int H,
                      const uint16_t *conf_w, float conf_b, float tau,
                      double *zc, double *conf, int32_t *draft_len,
                      int32_t *draft_tokens) {
    if (B < 0 || k < 1 || H < 1 || !h || !conf_w || !draft_len) return ORACLE_ERR_ARG;
    double thr;
    if (tau <= 0.0f) thr = -INFINITY;
    else if (tau >= 1.0f) thr = INFINITY;
    else thr = log((double)tau) - log1p(-(double)tau);
    for (int b = 0; b < B; ++b) {
        int32_t L = k;
        for (int i = 0; i < k; ++i) {
            const uint16_t *hrow = h + ((int64_t)b * k + i) * H;
            double acc = 0.0;
            for (int c = 0; c < H; ++c)
                acc += (double)bf16_bits_to_float(conf_w[c]) *
                       (double)bf16_bits_to_float(hrow[c]);
            acc += (double)conf_b;
            if (zc) zc[(int64_t)b * k + i] = acc;
            if (conf) conf[(int64_t)b * k + i] = 1.0 / (1.0 + exp(-acc));
            if (L == k && !(acc >= thr)) L = i;
        }
        draft_len[b] = L;
        if (draft_tokens)
            for (int i = L; i < k; ++i) draft_tokens[(int64_t)b * k + i] = -1;
    }
    return ORACLE_OK;
}

/* log(sigmoid(z)) without overflow: -log1p(exp(-z)) for z >= 0, z - log1p(exp(z))
 * below. */
static double log_sigmoid(double z) {
    return z >= 0.0 ? -log1p(exp(-z)) : z - log1p(exp(z));
}

/*
 * Confidence head with the Markov context, and the cumulative truncation rule.
 * [PR620] / [CARD] name the draft config field confidence_head_with_markov
 * next to enable_confidence_head and markov_rank, and the AcceptRatePredictor
 * head; the pages give no formula.  Reading taken: with the field set, the
 * head sees the Markov context of the position besides its hidden state, as
 * one linear layer over the concatenation [h_i ; e_i]:
 *   e_i      = markov_w1[c_i, :]   (r values; c_0 = the bonus token prev[b],
 *                                   c_i = the draft token of position i-1)
 *   zc[b,i]  = sum_c w[c] h_i[c] + sum_t w[H + t] e_i[t] + b        (fp64)
 *   conf     = sigmoid(zc)
 * (w1 == NULL: the plain head, w has H entries.)  Truncation:
 *   per position (cumulative == 0): L = first i with zc < logit(tau);
 *   cumulative   (cumulative != 0): L = first i with
 *       sum_{j <= i} log sigmoid(zc_j) < log(tau),
 *     i.e. the product of the acceptance confidences of the prefix falls
 *     below tau (the head predicts per-position acceptance, and the whole
 *     prefix must be accepted for position i to count).
 * tau <= 0 keeps every position, tau >= 1 keeps none.  draft_tokens (in/out,
 * [B, k], the chain's drafts) supply the contexts and get -1 from L on.
 * Also returns cum[b,i] = sum_{j<=i} log sigmoid(zc_j) (may be NULL).
 */
int oracle_confidence_markov(const uint16_t *h, int B, int k, int H, const uint16_t *conf_w,
                             float conf_b, float tau, int cumulative, const uint16_t *w1, int r,
                             int64_t V, const int32_t *prev, int32_t *draft_tokens, double *zc,
                             double *conf, double *cum, int32_t *draft_len) {
    if (B < 0 || k < 1 || H < 1 || !h || !conf_w || !draft_len || !draft_tokens) return ORACLE_ERR_ARG;
    if (w1 && (r < 1 || V < 1 || !prev)) return ORACLE_ERR_ARG;
    int status = ORACLE_OK;
    for (int b = 0; b < B; ++b) {
        double s = 0.0;
        int32_t L = k;
        for (int i = 0; i < k; ++i) {
            const uint16_t *hrow = h + ((int64_t)b * k + i) * H;
            double acc = 0.0;
            for (int c = 0; c < H; ++c)
                acc += (double)bf16_bits_to_float(conf_w[c]) * (double)bf16_bits_to_float(hrow[c]);
            if (w1) {
                const int32_t ctx = i == 0 ? prev[b] : draft_tokens[(int64_t)b * k + i - 1];
                if (ctx < 0 || (int64_t)ctx >= V) {
                    status = ORACLE_ERR_TOKEN;
                } else {
                    for (int t = 0; t < r; ++t)
                        acc += (double)bf16_bits_to_float(conf_w[H + t]) *
                               (double)bf16_bits_to_float(w1[(int64_t)ctx * r + t]);
                }
            }
            acc += (double)conf_b;
            s += log_sigmoid(acc);
            if (zc) zc[(int64_t)b * k + i] = acc;
            if (conf) conf[(int64_t)b * k + i] = 1.0 / (1.0 + exp(-acc));
            if (cum) cum[(int64_t)b * k + i] = s;
            int keep;
            if (tau <= 0.0f) keep = 1;
            else if (tau >= 1.0f) keep = 0;
            else if (cumulative) keep = s >= log((double)tau);
            else keep = acc >= log((double)tau) - log1p(-(double)tau);
            if (L == k && !keep) L = i;
        }
        draft_len[b] = L;
        for (int i = L; i < k; ++i) draft_tokens[(int64_t)b * k + i] = -1;
    }
    return status;
}

/* ------------------------------------------------------------------ */
/* Verification                                                        */
/* ------------------------------------------------------------------ */

/* Softmax of one fp32 row, in fp64: out[v] = exp(x[v] - max) / sum. */
static void softmax_row(const float *x, int64_t V, double *out) {
    double mx = -INFINITY;
    for (int64_t v = 0; v < V; ++v)
        if ((double)x[v] > mx) mx = (double)x[v];
    double s = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        out[v] = exp((double)x[v] - mx);
        s += out[v];
    }
    for (int64_t v = 0; v < V; ++v) out[v] /= s;
}

static int64_t argmax_row(const float *x, int64_t V) {
    int64_t best = 0;
    for (int64_t v = 1; v < V; ++v)
        if (x[v] > x[best]) best = v;
    return best;
}

/* Gumbel noise of vocabulary entry v for the draw made at block row `row`:
 * Philox4x32-10 with counter (request, row, step, 1 + v/4), word w = word
 * v mod 4, U = (2 * (w >> 9) + 1) * 2^-24 (an odd multiple of 2^-24, so U is
 * exact in binary32 and lies strictly inside (0, 1)), G = -log(-log U). */
static double gumbel_noise(uint64_t seed, uint32_t req, uint32_t row, uint32_t step, int64_t v) {
    uint32_t ctr[4] = {req, row, step, 1u + (uint32_t)(v / 4)};
    uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
    uint32_t w[4];
    oracle_philox4x32_10(ctr, key, w);
    double u = (double)(2u * (w[v % 4] >> 9) + 1u) * (1.0 / 16777216.0);
    return -log(-log(u));
}

/* One draw from the distribution proportional to exp(logw[v]) (logw = -inf
 * for zero weight) by the Gumbel-max rule: the smallest v maximising
 * logw[v] + G_v.  Returns -1 when every weight is zero.
 *
 * Diagnostics for parity accounting (not part of the method): err[v] is a
 * bound on how far a binary32 evaluation of logw[v] may stray; *margin =
 * (best - second best) - (bound of both, noise error included).  A negative
 * margin means a faithful fp32 implementation may pick the runner-up. */
static int64_t gumbel_draw(const double *logw, const double *err, int64_t V, uint64_t seed,
                           uint32_t req, uint32_t row, uint32_t step, double *margin) {
    const double eps = 1.0 / 524288.0; /* 2^-19: a few binary32 ulps of headroom */
    int64_t best = -1, second = -1;
    double kb = -INFINITY, ks = -INFINITY, eb = 0.0, es = 0.0;
    for (int64_t v = 0; v < V; ++v) {
        if (logw[v] == -INFINITY) continue;
        double g = gumbel_noise(seed, req, row, step, v);
        double key = logw[v] + g;
        double e = err[v] + eps * (fabs(g) + 1.0);
        if (best < 0 || key > kb) {
            second = best; ks = kb; es = eb;
            best = v; kb = key; eb = e;
        } else if (second < 0 || key > ks) {
            second = v; ks = key; es = e;
        }
    }
    *margin = (second < 0) ? INFINITY : (kb - ks) - (eb + es);
    return best;
}

/*
 * Verify one block per request.
 *
 * Greedy ([PR620] "greedy spec decode is lossless by construction"):
 *   t_j = argmax target_j (lowest index on ties);
 *   a   = length of the longest prefix (at most L) with d_j == t_j;
 *   next = t_a   (the target's own token after the accepted prefix: the
 *                 correction at the first mismatch, or the bonus).
 *
 * Probabilistic ([CARD] draft_sample_method "probabilistic", [PR128]
 * "verified by rejection sampling"): with p_j = softmax(target_j) and
 * q_j = softmax(z_j) (z = biased draft logits; one-hot at d_j when
 * z == NULL), positions are tested in order: d_j is accepted iff
 * u_j < p_j(d_j) / q_j(d_j).  At the first rejection j the next token is
 * drawn from max(0, p_j - q_j) normalised (one-hot q: p_j with d_j removed);
 * if its total is zero it is drawn from p_j.  If all L drafts are accepted,
 * the bonus token is drawn from p_L.  accepted_len = number of accepted
 * drafts.  The pages fix only these distributions; every draw here is the
 * Gumbel-max rule of gumbel_draw (exact in distribution), so that the drawn
 * index is an argmax and not a running-sum threshold.
 *
 * Layouts: target [B, k+1, V]; drafts [B, k]; draft_len [B] (NULL = k);
 * z [B, k, V].  Diagnostics (each may be NULL):
 *   accept_margin [B, k] : |u - p/q| of each decided position, NaN elsewhere
 *   sample_margin [B]    : Gumbel-max gap minus its rounding bound (NaN when
 *                          no draw happened, i.e. greedy)
 *   sample_row    [B]    : block row the draw used (-1 greedy)
 */
int oracle_verify(int mode, const float *target, const int32_t *drafts,
                  const int32_t *draft_len, const float *z, int B, int k,
                  int64_t V, uint64_t seed, const uint32_t *request_id,
                  uint32_t step, int32_t *accepted_len, int32_t *next_token,
                  double *accept_margin, double *sample_margin,
                  int32_t *sample_row) {
    if (B < 0 || k < 1 || V < 1 || !target || !drafts || !accepted_len || !next_token)
        return ORACLE_ERR_ARG;
    if (mode != 0 && mode != 1) return ORACLE_ERR_ARG;
    int status = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        const int32_t L = draft_len ? draft_len[b] : k;
        const uint32_t req = request_id ? request_id[b] : (uint32_t)b;
        if (accept_margin)
            for (int j = 0; j < k; ++j) accept_margin[(int64_t)b * k + j] = NAN;
        if (sample_margin) sample_margin[b] = NAN;
        if (sample_row) sample_row[b] = -1;
        if (L < 0 || L > k) {
#pragma omp atomic write
            status = ORACLE_ERR_ARG;
            continue;
        }
        const float *trow0 = target + (int64_t)b * (k + 1) * V;
        if (mode == 0) {
            int a = 0;
            while (a < L) {
                int64_t t = argmax_row(trow0 + (int64_t)a * V, V);
                if (drafts[(int64_t)b * k + a] != (int32_t)t) break;
                ++a;
            }
            accepted_len[b] = a;
            next_token[b] = (int32_t)argmax_row(trow0 + (int64_t)a * V, V);
            continue;
        }
        double *p = (double *)malloc(sizeof(double) * (size_t)V);
        double *q = (double *)malloc(sizeof(double) * (size_t)V);
        double *lw = (double *)malloc(sizeof(double) * (size_t)V);
        double *er = (double *)malloc(sizeof(double) * (size_t)V);
        const double eps = 1.0 / 524288.0;
        int a = 0;
        int rejected = 0;
        for (; a < L; ++a) {
            int32_t d = drafts[(int64_t)b * k + a];
            if (d < 0 || (int64_t)d >= V) {
#pragma omp atomic write
                status = ORACLE_ERR_TOKEN;
                rejected = 1;
                break;
            }
            const float *trow = trow0 + (int64_t)a * V;
            softmax_row(trow, V, p);
            double qd = 1.0;
            if (z) {
                softmax_row(z + ((int64_t)b * k + a) * V, V, q);
                qd = q[d];
            }
            double ua, us;
            verify_uniforms(seed, req, (uint32_t)a, step, &ua, &us);
            double ratio = p[d] / qd;
            if (accept_margin) accept_margin[(int64_t)b * k + a] = fabs(ua - ratio);
            if (ua < ratio) continue;
            /* rejected at position a: log of the residual weights */
            double R = 0.0;
            for (int64_t v = 0; v < V; ++v) {
                double qv = z ? q[v] : (v == d ? 1.0 : 0.0);
                double rv = p[v] - qv;
                if (rv > 0.0) {
                    R += rv;
                    lw[v] = log(rv);
                    /* binary32 evaluation: log p and log q each to ~eps*(1+|log|); the
                     * difference amplifies that by 1/(1 - q/p) */
                    double lp = log(p[v]), lq = qv > 0.0 ? log(qv) : 0.0;
                    double amp = qv > 0.0 ? 1.0 + qv / rv : 1.0;
                    er[v] = eps * (2.0 + fabs(lp) + fabs(lq) + fabs(lw[v])) * amp;
                } else {
                    lw[v] = -INFINITY;
                    er[v] = 0.0;
                }
            }
            if (!(R > 0.0))
                for (int64_t v = 0; v < V; ++v) {
                    lw[v] = log(p[v]);
                    er[v] = eps * (2.0 + fabs(lw[v]));
                }
            double mg;
            next_token[b] = (int32_t)gumbel_draw(lw, er, V, seed, req, (uint32_t)a, step, &mg);
            if (sample_margin) sample_margin[b] = mg;
            if (sample_row) sample_row[b] = a;
            rejected = 1;
            break;
        }
        if (!rejected) {
            /* every draft accepted: bonus token from p_L */
            softmax_row(trow0 + (int64_t)L * V, V, p);
            for (int64_t v = 0; v < V; ++v) {
                lw[v] = log(p[v]);
                er[v] = eps * (2.0 + fabs(lw[v]));
            }
            double mg;
            next_token[b] = (int32_t)gumbel_draw(lw, er, V, seed, req, (uint32_t)L, step, &mg);
            if (sample_margin) sample_margin[b] = mg;
            if (sample_row) sample_row[b] = L;
        }
        accepted_len[b] = a;
        free(p); free(q); free(lw); free(er);
    }
    return status;
}

/* ------------------------------------------------------------------ */
/* FP8 drafter weights (E4M3, per-row scales)                          */
/* ------------------------------------------------------------------ */
/*
 * [PR620] / [CARD]: the drafters are FP8 checkpoints ("drafter-fp8-v5",
 * "qwen3.8-27b-dflash-drafter-fp8-b70").  The pages do not give the scheme;
 * the reading taken is the common W8A8 one: E4M3 codes (OCP FP8: 1 sign, 4
 * exponent bits with bias 7, 3 mantissa bits, no infinity, largest finite
 * 448), one fp32 scale per weight output row and one per activation row,
 * scale = amax / 448 (1 for an all-zero row), code = E4M3(x / scale) rounded
 * to nearest even and saturated to +-448.
 */

/* E4M3 value of a code. */
float oracle_e4m3_to_f32(uint8_t c) {
    const int s = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
    if (e == 0xF && m == 7) return NAN;
    double v = (e == 0) ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
    return (float)(s ? -v : v);
}

/* Nearest E4M3 code (ties to even), saturating beyond +-448. */
uint8_t oracle_f32_to_e4m3(float x) {
    if (isnan(x)) return 0x7F;
    const uint8_t s = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a > 448.0) return s | 0x7E;
    if (a < ldexp(1.0, -6)) {
        /* subnormals: multiples of 2^-9 */
        double q = nearbyint(a * 512.0);     /* exact scaling; default rounding: to even */
        if (q >= 8.0) return s | 0x08;       /* rounds up to the smallest normal */
        return s | (uint8_t)q;
    }
    int e;
    double f = frexp(a, &e);                 /* a = f * 2^e, f in [0.5, 1) */
    e -= 1;                                  /* a = (2f) * 2^e, 2f in [1, 2) */
    double q = nearbyint((2.0 * f - 1.0) * 8.0);
    if (q >= 8.0) { q = 0.0; e += 1; }
    int E = e + 7;
    if (E > 15 || (E == 15 && q > 6.0)) return s | 0x7E;
    return s | (uint8_t)((E << 3) | (int)q);
}

/* Per-row quantisation of a bf16 matrix [R, C] (row stride ld). */
int oracle_quantize_fp8_rows(const uint16_t *x, int R, int C, int64_t ld, uint8_t *codes,
                             float *scales) {
    if (R < 0 || C < 1 || ld < C || !x || !codes || !scales) return ORACLE_ERR_ARG;
#pragma omp parallel for schedule(static)
    for (int r = 0; r < R; ++r) {
        const uint16_t *row = x + (int64_t)r * ld;
        float amax = 0.0f;
        for (int c = 0; c < C; ++c) {
            float v = fabsf(bf16_bits_to_float(row[c]));
            if (v > amax) amax = v;
        }
        float scale = amax > 0.0f ? amax / 448.0f : 1.0f;
        scales[r] = scale;
        for (int c = 0; c < C; ++c)
            codes[(int64_t)r * C + c] = oracle_f32_to_e4m3(bf16_bits_to_float(row[c]) / scale);
    }
    return ORACLE_OK;
}

/* out[m, n] = a_scale[m] * w_scale[n] * sum_k E4M3(a[m,k]) * E4M3(w[n,k]) (fp64 sum,
 * rounded once to fp32).  a: [M, K] codes, w: [N, K] codes. */
int oracle_gemm_fp8(const uint8_t *a, const float *a_scale, int M, const uint8_t *w,
                    const float *w_scale, int64_t N, int K, float *out) {
    if (M < 0 || N < 1 || K < 1 || !a || !a_scale || !w || !w_scale || !out) return ORACLE_ERR_ARG;
    double lut[256];
    for (int c = 0; c < 256; ++c) lut[c] = (double)oracle_e4m3_to_f32((uint8_t)c);
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n) {
        const uint8_t *wrow = w + n * K;
        for (int m = 0; m < M; ++m) {
            const uint8_t *arow = a + (int64_t)m * K;
            double acc = 0.0;
            for (int c = 0; c < K; ++c) acc += lut[arow[c]] * lut[wrow[c]];
            out[(int64_t)m * N + n] = (float)(acc * (double)a_scale[m] * (double)w_scale[n]);
        }
    }
    return ORACLE_OK;
}

/* Element-wise bf16 rounding of an fp32 array (as oracle_f32_to_bf16). */
void oracle_f32_to_bf16_n(const float *x, int64_t n, uint16_t *out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f32_to_bf16(x[i]);
}
