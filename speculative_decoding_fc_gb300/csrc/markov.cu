// Semi-autoregressive Markov-biased greedy drafting and confidence truncation.
//
// "Qwen3.8-27B DFlash drafter recipe" page, DSpark port description:
// VanillaMarkov = markov_w1 embedding [V, r] + markov_w2 projection r -> V;
// _greedy_sample adds the full-vocab bigram bias position by position, each
// position conditioned on the previous position's biased argmax, position 0
// on the accepted bonus token that propose() captured; AcceptRatePredictor +
// _truncate_by_confidence shorten the block.
//
// One launch per block position (the argmax of position i is the context of
// position i+1, a grid-wide dependency).  Each CTA owns a 512-entry slice of
// the vocabulary for every request: it reads the slice of markov_w2 once per
// group of 8 requests, adds the bias to the logits in place, and reduces a
// (value, lowest index) argmax key and the softmax statistics of the slice.
// The last CTA to finish (atomic ticket, nobody waits) merges the slices in a
// fixed order and writes the draft token, which the next launch reads.
#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace dspark {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kVPT = 2;                       // vocab entries per thread
constexpr int kChunk = kThreads * kVPT;       // vocab entries per CTA
constexpr int kGroup = 8;                     // requests per register group

struct __align__(16) ChainPartial {
  unsigned long long key;
  float m;
  float s;
};

template <int G>
__global__ void __launch_bounds__(kThreads) markov_chain_kernel(
    float *__restrict__ logits, const uint16_t *__restrict__ w1, const uint16_t *__restrict__ w2,
    int r, const int32_t *prev_src, int prev_stride, int32_t *draft_tokens, float *q_stats,
    int32_t *draft_len_fill, int B, int k, int V, int pos, int nchunks,
    ChainPartial *__restrict__ partials, int *counter, int *status) {
  __shared__ __align__(16) float e_s[kGroup * kMaxRank];
  __shared__ ChainPartial red[kGroup][kWarps];
  __shared__ int is_last;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int chunk = blockIdx.x;
  const bool biased = (w1 != nullptr);

  for (int g0 = 0; g0 < B; g0 += G) {
    const int gb = min(G, B - g0);
    if (biased) {
      // e_g[t] = markov_w1[prev_g, t]; requests past the group end get zeros.
      for (int idx = tid; idx < G * r; idx += kThreads) {
        const int g = idx / r;
        const int t = idx - g * r;
        float e = 0.0f;
        if (g < gb) {
          const int prev = prev_src[static_cast<long long>(g0 + g) * prev_stride];
          if (prev >= 0 && prev < V) {
            e = __uint_as_float(static_cast<uint32_t>(w1[static_cast<long long>(prev) * r + t]) << 16);
          } else if (t == 0 && chunk == 0) {
            record_error(status, DSPARK_ERR_BAD_TOKEN);
          }
        }
        e_s[idx] = e;
      }
      __syncthreads();
    }

    float acc[kVPT][G];
#pragma unroll
    for (int j = 0; j < kVPT; ++j)
#pragma unroll
      for (int g = 0; g < G; ++g) acc[j][g] = 0.0f;

    if (biased) {
      // bias[v] = sequential fp32 fma chain over t = 0..r-1, 64 ranks at a time; every
      // markov_w2 load of the thread for those ranks is issued before the first fma.
      for (int tc = 0; tc < r; tc += 64) {
        const int n8 = min(8, (r - tc) >> 3);
        uint4 wq[kVPT][8];
#pragma unroll
        for (int j = 0; j < kVPT; ++j) {
          const int v = chunk * kChunk + j * kThreads + tid;
          const uint4 *wrow =
              reinterpret_cast<const uint4 *>(w2 + static_cast<long long>(v < V ? v : 0) * r + tc);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            if (q < n8) wq[j][q] = __ldg(wrow + q);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          if (q < n8) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
              const float4 ea = *reinterpret_cast<const float4 *>(&e_s[g * r + tc + q * 8]);
              const float4 eb = *reinterpret_cast<const float4 *>(&e_s[g * r + tc + q * 8 + 4]);
#pragma unroll
              for (int j = 0; j < kVPT; ++j) {
                const uint4 w = wq[j][q];
                float x = acc[j][g];
                x = __fmaf_rn(bf16_lo(w.x), ea.x, x);
                x = __fmaf_rn(bf16_hi(w.x), ea.y, x);
                x = __fmaf_rn(bf16_lo(w.y), ea.z, x);
                x = __fmaf_rn(bf16_hi(w.y), ea.w, x);
                x = __fmaf_rn(bf16_lo(w.z), eb.x, x);
                x = __fmaf_rn(bf16_hi(w.z), eb.y, x);
                x = __fmaf_rn(bf16_lo(w.w), eb.z, x);
                x = __fmaf_rn(bf16_hi(w.w), eb.w, x);
                acc[j][g] = x;
              }
            }
          }
        }
      }
    }

    unsigned long long best[G];
    SoftStat st[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      best[g] = 0ull;
      st[g] = SoftStat{-INFINITY, 0.0f};
    }
#pragma unroll
    for (int j = 0; j < kVPT; ++j) {
      const int v = chunk * kChunk + j * kThreads + tid;
      if (v < V) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          if (g < gb) {
            float *rowp = logits + (static_cast<long long>(g0 + g) * k + pos) * V;
            float z = rowp[v];
            if (biased) {
              z = __fadd_rn(z, acc[j][g]);
              rowp[v] = z;
            }
            const unsigned long long key = argmax_key(z, static_cast<uint32_t>(v));
            best[g] = key > best[g] ? key : best[g];
            softstat_add(st[g], z);
          }
        }
      }
    }

#pragma unroll
    for (int g = 0; g < G; ++g) {
      if (g < gb) {
        const unsigned long long kmax = warp_max_u64(best[g]);
        const SoftStat ws = warp_softstat(st[g]);
        if (lane == 0) red[g][warp] = ChainPartial{kmax, ws.m, ws.s};
      }
    }
    __syncthreads();
    if (tid < gb) {
      ChainPartial acc2 = red[tid][0];
      SoftStat sacc{acc2.m, acc2.s};
      for (int w = 1; w < kWarps; ++w) {
        const ChainPartial o = red[tid][w];
        acc2.key = o.key > acc2.key ? o.key : acc2.key;
        sacc = softstat_merge(sacc, SoftStat{o.m, o.s});
      }
      acc2.m = sacc.m;
      acc2.s = sacc.s;
      partials[static_cast<long long>(g0 + tid) * nchunks + chunk] = acc2;
    }
    __syncthreads();
  }

  // ---------------------------------------------------------------- last CTA merges
  __threadfence();
  __syncthreads();
  if (tid == 0) is_last = (atomicAdd(counter, 1) == nchunks - 1) ? 1 : 0;
  __syncthreads();
  if (!is_last) return;
  __threadfence();

  for (int b = warp; b < B; b += kWarps) {
    const ChainPartial *pb = partials + static_cast<long long>(b) * nchunks;
    unsigned long long kb = 0ull;
    float mmax = -INFINITY;
    for (int c = lane; c < nchunks; c += 32) {
      const ulonglong2 raw = __ldcg(reinterpret_cast<const ulonglong2 *>(pb + c));
      kb = raw.x > kb ? raw.x : kb;
      mmax = fmaxf(mmax, __uint_as_float(static_cast<uint32_t>(raw.y)));
    }
    kb = warp_max_u64(kb);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mmax = fmaxf(mmax, __shfl_xor_sync(0xffffffffu, mmax, o));
    double s = 0.0;
    if (mmax != -INFINITY) {
      for (int c = lane; c < nchunks; c += 32) {
        const ulonglong2 raw = __ldcg(reinterpret_cast<const ulonglong2 *>(pb + c));
        const float cm = __uint_as_float(static_cast<uint32_t>(raw.y));
        const float cs = __uint_as_float(static_cast<uint32_t>(raw.y >> 32));
        if (cm != -INFINITY) s += static_cast<double>(cs) * static_cast<double>(expf(cm - mmax));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) {
      const long long at = static_cast<long long>(b) * k + pos;
      draft_tokens[at] = static_cast<int32_t>(key_index(kb));
      if (q_stats) {
        q_stats[2 * at] = mmax;
        q_stats[2 * at + 1] = static_cast<float>(s);
      }
      if (draft_len_fill && pos == k - 1) draft_len_fill[b] = k;
    }
  }
  if (tid == 0) *counter = 0;
}

// c[b, i] = sigmoid(w . h[b*k+i] + bias); draft_len[b] = first i whose logit
// falls below thr = logit(tau); later drafts are replaced by -1.
constexpr int kConfThreads = 256;

__global__ void __launch_bounds__(kConfThreads) confidence_kernel(
    const uint16_t *__restrict__ h, const uint16_t *__restrict__ conf_w, float conf_b, float thr,
    int32_t *draft_tokens, int32_t *draft_len, float *conf_out, int k, int H) {
  __shared__ float red[kConfThreads / 32];
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  int len = k;
  for (int i = 0; i < k; ++i) {
    const uint4 *hrow = reinterpret_cast<const uint4 *>(h + (static_cast<long long>(b) * k + i) * H);
    const uint4 *wrow = reinterpret_cast<const uint4 *>(conf_w);
    float acc = 0.0f;
    for (int c = tid; c < H / 8; c += kConfThreads) {
      const uint4 hv = __ldg(hrow + c);
      const uint4 wv = __ldg(wrow + c);
      acc = __fmaf_rn(bf16_lo(wv.x), bf16_lo(hv.x), acc);
      acc = __fmaf_rn(bf16_hi(wv.x), bf16_hi(hv.x), acc);
      acc = __fmaf_rn(bf16_lo(wv.y), bf16_lo(hv.y), acc);
      acc = __fmaf_rn(bf16_hi(wv.y), bf16_hi(hv.y), acc);
      acc = __fmaf_rn(bf16_lo(wv.z), bf16_lo(hv.z), acc);
      acc = __fmaf_rn(bf16_hi(wv.z), bf16_hi(hv.z), acc);
      acc = __fmaf_rn(bf16_lo(wv.w), bf16_lo(hv.w), acc);
      acc = __fmaf_rn(bf16_hi(wv.w), bf16_hi(hv.w), acc);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) red[warp] = acc;
    __syncthreads();
    if (tid == 0) {
      float zc = 0.0f;
      for (int w = 0; w < kConfThreads / 32; ++w) zc += red[w];
      zc += conf_b;
      if (conf_out) conf_out[static_cast<long long>(b) * k + i] = 1.0f / (1.0f + expf(-zc));
      if (len == k && !(zc >= thr)) len = i;
    }
    __syncthreads();
  }
  if (tid == 0) {
    draft_len[b] = len;
    for (int i = len; i < k; ++i) draft_tokens[static_cast<long long>(b) * k + i] = -1;
  }
}

}  // namespace

size_t chain_workspace_size(int B, int k, int V) {
  (void)k;
  const int nchunks = (V + kChunk - 1) / kChunk;
  return kWsAlign + align_up(static_cast<size_t>(B) * nchunks * sizeof(ChainPartial), kWsAlign);
}

dspark_status_t chain_launch(float *logits, const uint16_t *w1, const uint16_t *w2, int r,
                             const int32_t *prev_token, int32_t *draft_tokens, float *q_stats,
                             int32_t *draft_len_fill, int B, int k, int V, void *ws,
                             int *status, cudaStream_t stream) {
  const int nchunks = (V + kChunk - 1) / kChunk;
  int *counter = reinterpret_cast<int *>(ws);
  ChainPartial *partials = reinterpret_cast<ChainPartial *>(static_cast<char *>(ws) + kWsAlign);
  for (int pos = 0; pos < k; ++pos) {
    const int32_t *prev_src = pos == 0 ? prev_token : draft_tokens + (pos - 1);
    const int prev_stride = pos == 0 ? 1 : k;
    auto kern = B >= 8 ? markov_chain_kernel<8>
                       : (B >= 4 ? markov_chain_kernel<4>
                                 : (B >= 2 ? markov_chain_kernel<2> : markov_chain_kernel<1>));
    kern<<<nchunks, kThreads, 0, stream>>>(logits, w1, w2, r, prev_src, prev_stride, draft_tokens,
                                           q_stats, draft_len_fill, B, k, V, pos, nchunks,
                                           partials, counter, status);
    if (cudaGetLastError() != cudaSuccess) return DSPARK_ERR_CUDA;
  }
  return DSPARK_OK;
}

dspark_status_t confidence_launch(const uint16_t *h, const uint16_t *conf_w, float conf_b,
                                  float conf_tau, int32_t *draft_tokens, int32_t *draft_len,
                                  float *conf_out, int B, int k, int H, cudaStream_t stream) {
  float thr;
  if (conf_tau <= 0.0f)
    thr = -INFINITY;
  else if (conf_tau >= 1.0f)
    thr = INFINITY;
  else
    thr = static_cast<float>(log(static_cast<double>(conf_tau)) - log1p(-static_cast<double>(conf_tau)));
  confidence_kernel<<<B, kConfThreads, 0, stream>>>(h, conf_w, conf_b, thr, draft_tokens,
                                                    draft_len, conf_out, k, H);
  return cudaGetLastError() == cudaSuccess ? DSPARK_OK : DSPARK_ERR_CUDA;
}

}  // namespace dspark
