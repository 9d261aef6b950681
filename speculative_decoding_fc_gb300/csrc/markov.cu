// Semi-autoregressive Markov-biased greedy drafting and confidence truncation.
//
// "Qwen3.8-27B DFlash drafter recipe" page, DSpark port description:
// VanillaMarkov = markov_w1 embedding [V, r] + markov_w2 projection r -> V;
// _greedy_sample adds the full-vocab bigram bias position by position, each
// position conditioned on the previous position's biased argmax, position 0
// on the accepted bonus token that propose() captured; AcceptRatePredictor +
// _truncate_by_confidence shorten the block.
//
// The argmax of position i is the context of position i+1: a grid-wide
// dependency between positions.  Two implementations:
//
//  * markov_chain_persistent (default): ONE cooperative launch, one CTA per
//    SM.  Each CTA owns a contiguous slice of the vocabulary for all k
//    positions and keeps its slice of markov_w2 in shared memory (XOR-swizzled
//    16-byte chunks, bank-conflict free), so the weight is read from memory
//    once per step instead of once per position (r <= 64; at r = 128 the slice
//    is prefetched into L2 and read from there at every position).  Positions are separated by
//    tagged 64-bit words: every CTA publishes, per request, one word holding a
//    tag of (call, position) and its slice's argmax key, and every CTA polls all
//    CTAs' words until they carry the current tag.  The polled words are the data
//    (their max is the draft token), so no fence is needed between positions;
//    all CTAs take the same max and agree without a second barrier.
//  * markov_chain_kernel (fallback when a cooperative launch is not possible):
//    one launch per position; the last CTA to finish (atomic ticket, nobody
//    waits) merges the slices and writes the token the next launch reads.
//
// Each CTA reduces, per request, a (value, lowest index) argmax key and the
// softmax statistics (max, sum exp) of its slice of the biased logits.
#include <cuda_runtime.h>
#include <math.h>
#include <stdlib.h>

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
  pdl_wait();
  pdl_release();  // one wave: the next position's kernel may be scheduled

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

// ---------------------------------------------------------------- persistent chain
constexpr int kPThreads = 256;
constexpr int kPWarps = kPThreads / 32;
constexpr int kMaxPGrid = kMaxGemmCtas;       // CTAs of the persistent chain (<= SMs)
constexpr long long kBarrierCycles = 2000000000LL;  // ~1 s at 2 GHz

struct ChainPArgs {
  float *logits;
  const uint16_t *w1;
  const uint16_t *w2;
  const int32_t *prev_token;
  int32_t *draft_tokens;
  float *q_stats;
  int32_t *draft_len_fill;
  ChainPartial *partials;   // [k][B][grid]: softmax statistics of each CTA's slice
  unsigned long long *words;  // [k][B][grid]: tagged argmax word of each CTA's slice
  int *epoch;               // call counter: the words of call e carry tags of epoch e
  int *done;                // exit counter (the last CTA advances the epoch)
  int *abort_flag;          // set when a wait gives up; later calls then do nothing
  int *status;
  int r, B, k, V;
  int rows_per_cta;         // vocabulary rows owned by one CTA
  int w2_smem_bytes;        // shared memory reserved for the markov_w2 slice (0: read via L2)
  long long wait_cycles;    // budget of one wait for the other CTAs' words (clock64 cycles)
  int vec;                  // logits rows 16-byte aligned and slices multiples of 4 rows
};

__device__ __forceinline__ int ld_acquire(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ int ld_relaxed(const int *p) {
  int v;
  asm volatile("ld.relaxed.gpu.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release(int *p, int v) {
  asm volatile("st.release.gpu.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed_u64(unsigned long long *p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void st_release_u64(unsigned long long *p, unsigned long long v) {
  asm volatile("st.release.gpu.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// 16-byte chunk q of local row `row` of the shared-memory markov_w2 slice is
// stored at chunk q ^ ((row / 4) & mask): a thread owns four consecutive rows, so
// the eight threads of a shared-memory phase read rows 4 apart at the same q and hit
// eight different bank groups (128-byte rows; shorter rows share bank groups).
__device__ __forceinline__ int w2_swizzle(int row, int q, int chunks_per_row) {
  const int mask = chunks_per_row < 8 ? chunks_per_row - 1 : 7;
  return q ^ ((row >> 2) & mask);
}

// Position words.  Bits 58-63: tag in [1, 63] of (call epoch, position); two
// consecutive calls give a position different tags (16 or 15 apart mod 63), and 0
// (a cleared workspace) is never a tag, so a word shows by itself whether it was
// written in this call.  Bits 26-57: the ordered value bits of the slice's argmax
// key; bits 0-25: 2^26 - 1 - index (V <= 2^26).  Among words of one tag a larger
// word is a larger value, then a lower index, exactly as for argmax_key.
__device__ __forceinline__ uint32_t word_tag(int epoch, int pos) {
  return 1u + ((static_cast<uint32_t>(epoch) % 63u) * 16u + static_cast<uint32_t>(pos)) % 63u;
}

__device__ __forceinline__ unsigned long long pack_word(unsigned long long key, uint32_t tag) {
  return (static_cast<unsigned long long>(tag) << 58) | ((key >> 32) << 26) | (key & 0x3ffffffull);
}

__device__ __forceinline__ int word_index(unsigned long long w) {
  return static_cast<int>(0x3ffffffu - static_cast<uint32_t>(w & 0x3ffffffull));
}

// Rows of the vocabulary a thread of the persistent chain owns: 4 rows x up to 8
// requests = 32 independent fma chains per thread.
constexpr int kPRows = 4;
constexpr int kGather = 8;    // markov_w1 elements a thread loads at once
constexpr int kPollReq = 4;   // requests a warp polls at once
constexpr int kPSmemMax = 225 * 1024;  // dynamic shared memory of the persistent chain
constexpr int kPollWords = (kMaxPGrid + 31) / 32;  // words of one request per lane

// Two fp32 fused multiply-adds in one instruction: lane i of d = a_i * b_i + c_i,
// each rounded to nearest once (the same IEEE operation as fmaf on each lane).
__device__ __forceinline__ unsigned long long fma_f32x2(unsigned long long a, unsigned long long b,
                                                       unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ unsigned long long pack_f32x2(float lo, float hi) {
  unsigned long long d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(lo), "f"(hi));
  return d;
}

__device__ __forceinline__ void unpack_f32x2(unsigned long long v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

// Asynchronous copies of this thread's logits of requests g0 .. g0 + G - 1 (those
// below B) at position pos into lg_s[(g * kPThreads + tid) * kPRows + j]: issued a
// group ahead, they land while the fma chains run and hold no registers meanwhile.
// vec4: the thread's four rows are consecutive, in range and 16-byte aligned (one
// 16-byte copy per request).
template <int G>
__device__ __forceinline__ void issue_logits_copy(float *lg_s, const float *logits,
                                                  const int (&vrow)[kPRows], bool vec4, int g0,
                                                  int pos, int B, int k, int V, int tid) {
#pragma unroll
  for (int g = 0; g < G; ++g) {
    if (g0 + g < B) {
      const float *src = logits + (static_cast<long long>(g0 + g) * k + pos) * V;
      float *dst0 = &lg_s[(g * kPThreads + tid) * kPRows];
      if (vec4) {
        asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(
                         __cvta_generic_to_shared(dst0))),
                     "l"(src + vrow[0])
                     : "memory");
      } else {
#pragma unroll
        for (int j = 0; j < kPRows; ++j)
          asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(static_cast<uint32_t>(
                           __cvta_generic_to_shared(dst0 + j))),
                       "l"(src + vrow[j])
                       : "memory");
      }
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// Stores this thread's biased logits of one request row: one 16-byte store when vec4,
// else one per row in range.
__device__ __forceinline__ void store_row4(float *row, const int (&vrow)[kPRows],
                                           const bool (&valid)[kPRows], bool vec4, float z0,
                                           float z1, float z2, float z3) {
  if (vec4) {
    *reinterpret_cast<float4 *>(row + vrow[0]) = make_float4(z0, z1, z2, z3);
  } else {
    if (valid[0]) row[vrow[0]] = z0;
    if (valid[1]) row[vrow[1]] = z1;
    if (valid[2]) row[vrow[2]] = z2;
    if (valid[3]) row[vrow[3]] = z3;
  }
}

// This thread's logits of one request row (four rows of the vocabulary): one 16-byte
// load when vec4, else four.
__device__ __forceinline__ void load_row4(const float *row, const int (&vrow)[kPRows], bool vec4,
                                          float (&out)[kPRows]) {
  if (vec4) {
    const float4 v = *reinterpret_cast<const float4 *>(row + vrow[0]);
    out[0] = v.x; out[1] = v.y; out[2] = v.z; out[3] = v.w;
  } else {
#pragma unroll
    for (int j = 0; j < kPRows; ++j) out[j] = row[vrow[j]];
  }
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Warp-wide (key max, softmax stats) of one value pair per thread, with one exp per
// thread: the max first, then the sum of s * exp(m - max).
__device__ __forceinline__ void warp_key_stats(unsigned long long &key, float &m, float &s) {
  key = warp_max_u64(key);
  float mm = m;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, o));
  // __fmul_rn: the rescaled sum is rounded before the shuffle sum (no fused
  // multiply-add), so every chain kernel gives the same bits
  float ss = (m == -INFINITY) ? 0.0f : __fmul_rn(s, expf(m - mm));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  m = mm;
  s = ss;
}

// kStats: also reduce the softmax statistics of q (max z, sum exp(z - max)) for
// q_stats; without it only the argmax keys are reduced.
// kW2Smem: the CTA's markov_w2 slice is copied to shared memory once (r <= 64);
// otherwise (r = 128: 38.9 MB, more than the SMs' shared memory together) the slice
// is prefetched into L2 and read from there at every position.
template <int G, int CPR, bool kStats, bool kW2Smem>
__global__ void __launch_bounds__(kPThreads, 1) markov_chain_persistent(const ChainPArgs a) {
  static_assert(G <= kPWarps, "one combining warp per request of a group");
  __shared__ ChainPartial red[G][kPWarps];
  __shared__ int stop_s, epoch_s;
  extern __shared__ __align__(16) uint8_t psmem[];
  // dynamic shared memory: markov_w2 slice [rows][CPR] (1024-byte aligned), then the
  // contexts e of all requests (G = 1: [B][r]; G >= 2: request pairs interleaved,
  // [B/2][r][2], the odd request's partner zero), then prev tokens [B] (padded to 16
  // bytes), then (G = 8) one request group's logits [G][kPRows][kPThreads]
  uint4 *w2_s = reinterpret_cast<uint4 *>(psmem);
  const size_t e_bytes = static_cast<size_t>((a.B + 1) & ~1) * CPR * 32;
  float *e_s = reinterpret_cast<float *>(psmem + a.w2_smem_bytes);
  int *prev_s = reinterpret_cast<int *>(psmem + a.w2_smem_bytes + e_bytes);
  float *lg_s = reinterpret_cast<float *>(psmem + a.w2_smem_bytes + e_bytes +
                                          ((static_cast<size_t>(a.B) * 4 + 15) & ~static_cast<size_t>(15)));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int grid = gridDim.x, cta = blockIdx.x;
  const int B = a.B, k = a.k, V = a.V;
  constexpr int r = CPR * 8;
  const bool biased = (a.w1 != nullptr);
  const int v_lo = cta * a.rows_per_cta;
  const int v_hi = min(V, v_lo + a.rows_per_cta);
  const int nrows = max(0, v_hi - v_lo);
  // this thread's rows: kPRows * tid + j of the slice, j < kPRows (clamped; results
  // of the clamped copies are discarded).  vec4: all four in range, and the logits
  // rows 16-byte aligned (the slice starts on a multiple of 4, V % 4 == 0): logits
  // move as one 16-byte access per request.
  bool valid[kPRows];
  int vrow[kPRows];
#pragma unroll
  for (int j = 0; j < kPRows; ++j) {
    const int row = kPRows * tid + j;
    valid[j] = row < nrows;
    // a CTA past the vocabulary's end (nrows == 0) points its copies at row 0
    vrow[j] = nrows > 0 ? v_lo + (row < nrows ? row : nrows - 1) : 0;
  }
  const bool vec4 = a.vec != 0 && kPRows * tid + kPRows <= nrows;

  // markov_w2 is a weight that no kernel of the step writes, so the CTA's slice is
  // fetched before the wait for the previous kernel (this CTA runs as soon as the
  // previous kernel's CTA on its SM has exited): into shared memory by asynchronous
  // copies (16-byte chunks XOR-swizzled by row so that 8 consecutive rows read at the
  // same chunk hit 8 bank groups), all in flight together; or, when the slice is read
  // through L2 at every position, as a bulk prefetch into L2.
  if (biased && nrows > 0) {
    if constexpr (kW2Smem) {
      const uint4 *src = reinterpret_cast<const uint4 *>(a.w2 + static_cast<long long>(v_lo) * r);
      for (int i = tid; i < nrows * CPR; i += kPThreads) {
        const int row = i / CPR, q = i - row * CPR;
        const uint32_t dst = static_cast<uint32_t>(
            __cvta_generic_to_shared(&w2_s[row * CPR + w2_swizzle(row, q, CPR)]));
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src + i)
                     : "memory");
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    } else {
      // 16 KB pieces, one per thread (the slice is at most 1024 rows x 256 bytes)
      const char *src = reinterpret_cast<const char *>(a.w2 + static_cast<long long>(v_lo) * r);
      const uint32_t bytes = static_cast<uint32_t>(nrows) * CPR * 16u;
      const uint32_t off = static_cast<uint32_t>(tid) * 16384u;
      if (off < bytes) {
        const uint32_t n = bytes - off < 16384u ? bytes - off : 16384u;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src + off), "r"(n) : "memory");
      }
    }
  }
  pdl_wait();
  pdl_release();
  if (tid == 0) {
    stop_s = ld_acquire(a.abort_flag);
    epoch_s = ld_acquire(a.epoch);
    if (stop_s && cta == 0) record_error(a.status, DSPARK_ERR_DEVICE_TIMEOUT);
  }
  for (int b = tid; b < B; b += kPThreads) {
    int p = a.prev_token[b];
    if (biased && (p < 0 || p >= V)) {
      if (cta == 0) record_error(a.status, DSPARK_ERR_BAD_TOKEN);
      p = -1;
    }
    prev_s[b] = p;
  }
  if (biased && kW2Smem) asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  if (stop_s) return;
  const int epoch = epoch_s;
  int lrow[kPRows];  // local (slice) row of each of this thread's rows, clamped
#pragma unroll
  for (int j = 0; j < kPRows; ++j) lrow[j] = nrows > 0 ? vrow[j] - v_lo : 0;

  // Logits of the first request group at position 0.  Groups of 8 requests stage
  // them in shared memory through asynchronous copies issued a group ahead; smaller
  // groups (latency-bound) hold them in registers, loaded a group ahead.
  constexpr bool kStage = (G >= 8);
  float lg_next[kPRows][G];
  if constexpr (kStage) {
    issue_logits_copy<G>(lg_s, a.logits, vrow, vec4, 0, 0, B, k, V, tid);
  } else {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      float t4[kPRows] = {0.0f, 0.0f, 0.0f, 0.0f};
      if (g < B) load_row4(a.logits + (static_cast<long long>(g) * k) * V, vrow, vec4, t4);
#pragma unroll
      for (int j = 0; j < kPRows; ++j) lg_next[j][g] = t4[j];
    }
  }

  // e_b = markov_w1[prev_b] of every request for position 0 (the poll below gathers
  // those of the later positions): each thread's loads (up to kGather) are all issued
  // before its stores, one round trip
  if (biased) {
    const int bpad = (G >= 2) ? ((B + 1) & ~1) : B;
    for (int i0 = 0; i0 < bpad * r; i0 += kPThreads * kGather) {
      uint32_t ev[kGather];
#pragma unroll
      for (int u = 0; u < kGather; ++u) {
        const int idx = i0 + u * kPThreads + tid;
        const int b = idx / r, t = idx - b * r;
        const int p = (idx < bpad * r && b < B) ? prev_s[b] : -1;
        ev[u] = p >= 0 ? static_cast<uint32_t>(a.w1[static_cast<long long>(p) * r + t]) << 16 : 0u;
      }
#pragma unroll
      for (int u = 0; u < kGather; ++u) {
        const int idx = i0 + u * kPThreads + tid;
        const int b = idx / r, t = idx - b * r;
        if (idx < bpad * r)
          e_s[(G >= 2) ? (((b >> 1) * r + t) << 1) + (b & 1) : idx] = __uint_as_float(ev[u]);
      }
    }
    __syncthreads();
  }

  float acc[kPRows][G];  // bias, then the biased logit, of this thread's rows
  for (int pos = 0; pos < k; ++pos) {
    for (int g0 = 0; g0 < B; g0 += G) {
      const int gb = min(G, B - g0);
      if (!kStage && g0 > 0) {
        // later groups: their logits, loaded before the fma loop hides the latency
#pragma unroll
        for (int g = 0; g < G; ++g) {
          float t4[kPRows] = {0.0f, 0.0f, 0.0f, 0.0f};
          if (g < gb) load_row4(a.logits + (static_cast<long long>(g0 + g) * k + pos) * V, vrow, vec4, t4);
#pragma unroll
          for (int j = 0; j < kPRows; ++j) lg_next[j][g] = t4[j];
        }
      }
      // bias[v] = sequential fp32 fma chain over t = 0..r-1 (the chain of each
      // (row, request) is one thread's, in t order; chains interleave for ILP)
#pragma unroll
      for (int j = 0; j < kPRows; ++j)
#pragma unroll
        for (int g = 0; g < G; ++g) acc[j][g] = 0.0f;
      if (biased && G >= 2) {
        // The chains of requests 2i and 2i+1 advance together in one fma.rn.f32x2:
        // each lane is the same fp32 fma, in the same t order, as the chain alone.
        unsigned long long acc2[kPRows][(G + 1) / 2];
#pragma unroll
        for (int j = 0; j < kPRows; ++j)
#pragma unroll
          for (int gp = 0; gp < G / 2; ++gp) acc2[j][gp] = 0ull;  // +0.0f in both lanes
#pragma unroll
        for (int q = 0; q < CPR; ++q) {
          float w[kPRows][8];
#pragma unroll
          for (int j = 0; j < kPRows; ++j) {
            uint4 c;
            if constexpr (kW2Smem) {
              c = w2_s[lrow[j] * CPR + w2_swizzle(lrow[j], q, CPR)];
            } else {
              c = __ldg(reinterpret_cast<const uint4 *>(a.w2 + static_cast<long long>(vrow[j]) * r) + q);
            }
            w[j][0] = bf16_lo(c.x); w[j][1] = bf16_hi(c.x);
            w[j][2] = bf16_lo(c.y); w[j][3] = bf16_hi(c.y);
            w[j][4] = bf16_lo(c.z); w[j][5] = bf16_hi(c.z);
            w[j][6] = bf16_lo(c.w); w[j][7] = bf16_hi(c.w);
          }
          unsigned long long e2[(G + 1) / 2][8];
#pragma unroll
          for (int gp = 0; gp < G / 2; ++gp) {
            // pairs past the batch end read pair 0 (results unused)
            const int pair = (2 * gp < gb) ? (g0 >> 1) + gp : 0;
            const float4 *ep = reinterpret_cast<const float4 *>(&e_s[(pair * r + q * 8) * 2]);
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const float4 v = ep[h];
              e2[gp][2 * h] = pack_f32x2(v.x, v.y);
              e2[gp][2 * h + 1] = pack_f32x2(v.z, v.w);
            }
          }
#pragma unroll
          for (int t = 0; t < 8; ++t)
#pragma unroll
            for (int j = 0; j < kPRows; ++j) {
              const unsigned long long wd = pack_f32x2(w[j][t], w[j][t]);
#pragma unroll
              for (int gp = 0; gp < G / 2; ++gp) acc2[j][gp] = fma_f32x2(wd, e2[gp][t], acc2[j][gp]);
            }
        }
#pragma unroll
        for (int j = 0; j < kPRows; ++j)
#pragma unroll
          for (int gp = 0; gp < G / 2; ++gp) unpack_f32x2(acc2[j][gp], acc[j][2 * gp], acc[j][2 * gp + 1]);
      } else if (biased) {
#pragma unroll
        for (int q = 0; q < CPR; ++q) {
          float w[kPRows][8];
#pragma unroll
          for (int j = 0; j < kPRows; ++j) {
            uint4 c;
            if constexpr (kW2Smem) {
              c = w2_s[lrow[j] * CPR + w2_swizzle(lrow[j], q, CPR)];
            } else {
              c = __ldg(reinterpret_cast<const uint4 *>(a.w2 + static_cast<long long>(vrow[j]) * r) + q);
            }
            w[j][0] = bf16_lo(c.x); w[j][1] = bf16_hi(c.x);
            w[j][2] = bf16_lo(c.y); w[j][3] = bf16_hi(c.y);
            w[j][4] = bf16_lo(c.z); w[j][5] = bf16_hi(c.z);
            w[j][6] = bf16_lo(c.w); w[j][7] = bf16_hi(c.w);
          }
          float e[G][8];
#pragma unroll
          for (int g = 0; g < G; ++g) {
            // requests past the batch end read request 0's context (results unused)
            const int gg = (g < gb) ? g0 + g : 0;
            const float4 ea = *reinterpret_cast<const float4 *>(&e_s[gg * r + q * 8]);
            const float4 eb = *reinterpret_cast<const float4 *>(&e_s[gg * r + q * 8 + 4]);
            e[g][0] = ea.x; e[g][1] = ea.y; e[g][2] = ea.z; e[g][3] = ea.w;
            e[g][4] = eb.x; e[g][5] = eb.y; e[g][6] = eb.z; e[g][7] = eb.w;
          }
          // rank t of every (row, request) chain, then rank t + 1: all G x kPRows
          // chains advance together
#pragma unroll
          for (int t = 0; t < 8; ++t)
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
              for (int j = 0; j < kPRows; ++j) acc[j][g] = __fmaf_rn(w[j][t], e[g][t], acc[j][g]);
        }
      }
      // Per thread: argmax key (and statistics) of its rows for every request of the
      // group; then warp reductions, one shuffle round for all requests at a time so
      // that the requests' shuffle latencies overlap.
      // The key of a row is (ordered value, inverted index): per thread the best
      // ordered value with the lowest index holding it (rows ascend), then per warp
      // the max ordered value and the lowest index among the lanes holding it.
      unsigned long long key[G];
      float mx[G], sm[G];
      uint32_t bo[G], bi[G];
      if (kStage) cp_async_wait_all();  // this thread's logits of the group are in lg_s
#pragma unroll
      for (int g = 0; g < G; ++g) {
        bo[g] = 0u;             // NaN and "no row" order lowest
        bi[g] = 0xffffffffu;
        mx[g] = -INFINITY;
        sm[g] = 0.0f;
        float zv[kPRows];
        float lg4[kPRows];
        if (kStage) {
          const float4 v = *reinterpret_cast<const float4 *>(&lg_s[(g * kPThreads + tid) * kPRows]);
          lg4[0] = v.x; lg4[1] = v.y; lg4[2] = v.z; lg4[3] = v.w;
        } else {
#pragma unroll
          for (int j = 0; j < kPRows; ++j) lg4[j] = lg_next[j][g];
        }
#pragma unroll
        for (int j = 0; j < kPRows; ++j) {
          float z = lg4[j];
          if (biased) z = __fadd_rn(z, acc[j][g]);
          zv[j] = z;
          acc[j][g] = z;  // kept for the write-back after this position's words
        }
        if (kPRows * tid + kPRows <= nrows) {
          // all four rows in range: the max by fmaxf (which passes over NaN like the
          // strict compare), then the first row holding it; the value and index of the
          // ordered-key scan below.  All NaN: the first row with the lowest key.
          const float m = fmaxf(fmaxf(zv[0], zv[1]), fmaxf(zv[2], zv[3]));
          int jj = 0;
#pragma unroll
          for (int j = kPRows - 1; j >= 0; --j)
            if (zv[j] == m) jj = j;
          if (g < gb) {
            bo[g] = ordered_bits(m);
            bi[g] = static_cast<uint32_t>(vrow[0] + jj);  // the four rows are consecutive
            if (kStats && m == m && m != -INFINITY) mx[g] = m;
          }
        } else {
#pragma unroll
          for (int j = 0; j < kPRows; ++j) {
            const float z = zv[j];
            if (valid[j] && g < gb) {
              const uint32_t o = ordered_bits(z);
              if (o > bo[g] || bi[g] == 0xffffffffu) {
                bo[g] = o;
                bi[g] = static_cast<uint32_t>(vrow[j]);
              }
              if (kStats && z == z && z != -INFINITY) mx[g] = fmaxf(mx[g], z);
            }
          }
        }
        if (kStats) {
#pragma unroll
          for (int j = 0; j < kPRows; ++j)
            if (valid[j] && g < gb && mx[g] != -INFINITY && zv[j] == zv[j] && zv[j] != -INFINITY)
              sm[g] += __expf(zv[j] - mx[g]);  // x <= 0: relative error ~2^-21
        }
      }
      // lg_s is consumed: the next group's logits (this position's, else the next's)
      if (kStage) {
        if (g0 + G < B)
          issue_logits_copy<G>(lg_s, a.logits, vrow, vec4, g0 + G, pos, B, k, V, tid);
        else if (pos + 1 < k)
          issue_logits_copy<G>(lg_s, a.logits, vrow, vec4, 0, pos + 1, B, k, V, tid);
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const uint32_t mo = __reduce_max_sync(0xffffffffu, bo[g]);
        const uint32_t mi = __reduce_min_sync(0xffffffffu, bo[g] == mo ? bi[g] : 0xffffffffu);
        key[g] = (static_cast<unsigned long long>(mo) << 32) | (0xffffffffu - mi);
      }
      if (kStats) {
        float mm[G];
#pragma unroll
        for (int g = 0; g < G; ++g) mm[g] = mx[g];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
          for (int g = 0; g < G; ++g) mm[g] = fmaxf(mm[g], __shfl_xor_sync(0xffffffffu, mm[g], o));
#pragma unroll
        for (int g = 0; g < G; ++g) sm[g] = (mx[g] == -INFINITY) ? 0.0f : __fmul_rn(sm[g], expf(mx[g] - mm[g]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
          for (int g = 0; g < G; ++g) sm[g] += __shfl_xor_sync(0xffffffffu, sm[g], o);
#pragma unroll
        for (int g = 0; g < G; ++g) mx[g] = mm[g];
      }
      if (lane == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g)
          if (g < gb) red[g][warp] = ChainPartial{key[g], mx[g], sm[g]};
      }
      __syncthreads();
      // one warp per request of the group combines the kPWarps warp partials (warp w
      // takes requests w and w + kPWarps of the group)
      for (int g = warp; g < gb; g += kPWarps) {
        unsigned long long key = 0ull;
        float m = -INFINITY, sum = 0.0f;
        if (lane < kPWarps) {
          const ChainPartial c0 = red[g][lane];
          key = c0.key;
          m = c0.m;
          sum = c0.s;
        }
        if (kStats)
          warp_key_stats(key, m, sum);
        else
          key = warp_max_u64(key);
        if (lane == 0) {
          const long long at = (static_cast<long long>(pos) * B + g0 + g) * grid + cta;
          if (kStats) a.partials[at] = ChainPartial{key, m, sum};
          // This thread wrote every partial of this request (the combining warp of a
          // request is fixed), so the release on the last position's word makes all
          // of them visible to whoever sees that word.
          const unsigned long long wd = pack_word(key, word_tag(epoch, pos));
          if (pos + 1 < k)
            st_relaxed_u64(a.words + at, wd);
          else
            st_release_u64(a.words + at, wd);
          // the global winner is one of the CTA winners: warm L2 with this one's
          // markov_w1 row for the next position's gather
          const int kidx = static_cast<int>(key_index(key));
          if (biased && pos + 1 < k && kidx >= 0 && kidx < V)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(a.w1 + static_cast<long long>(kidx) * r));
        }
      }
      if (biased && B > G) {
        // several groups share acc: store this group's biased logits now
#pragma unroll
        for (int g = 0; g < G; ++g)
          if (g < gb)
            store_row4(a.logits + (static_cast<long long>(g0 + g) * k + pos) * V, vrow, valid, vec4,
                       acc[0][g], acc[1][g], acc[2][g], acc[3][g]);
      }
      __syncthreads();
    }

    // This CTA's words of `pos` are published (above).  While the other CTAs finish,
    // store the biased logits and load the next position's logits (register path).
    if (biased && B <= G) {
#pragma unroll
      for (int g = 0; g < G; ++g)
        if (g < B)
          store_row4(a.logits + (static_cast<long long>(g) * k + pos) * V, vrow, valid, vec4,
                     acc[0][g], acc[1][g], acc[2][g], acc[3][g]);
    }
    if (!kStage && pos + 1 < k) {
#pragma unroll
      for (int g = 0; g < G; ++g) {
        float t4[kPRows] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (g < B) load_row4(a.logits + (static_cast<long long>(g) * k + pos + 1) * V, vrow, vec4, t4);
#pragma unroll
        for (int j = 0; j < kPRows; ++j) lg_next[j][g] = t4[j];
      }
    }
    // Wait for every CTA's word of each request (warp w polls requests w, w + 8, ...,
    // up to kPollReq of them at once);
    // the max of the words is the draft token.  Relaxed loads suffice: nothing else is
    // read on the strength of a word, except after the last position, where an acquire
    // fence pairs with the words' release stores before the statistics are merged.
    {
      const uint32_t tg = word_tag(epoch, pos);
      const long long t0 = clock64();
      for (int b0 = warp; b0 < B; b0 += kPWarps * kPollReq) {
        // requests b0 + i * kPWarps (i < kPollReq): their words are loaded together,
        // one round trip per pass for all of them
        unsigned long long best[kPollReq];
        bool done[kPollReq];  // warp-uniform
#pragma unroll
        for (int i = 0; i < kPollReq; ++i) {
          best[i] = 0ull;
          done[i] = b0 + i * kPWarps >= B;
        }
        int stop = 0;
        while (true) {
          unsigned long long w[kPollReq][kPollWords];
#pragma unroll
          for (int i = 0; i < kPollReq; ++i) {
            const unsigned long long *wb =
                a.words + (static_cast<long long>(pos) * B + b0 + i * kPWarps) * grid;
#pragma unroll
            for (int c = 0; c < kPollWords; ++c) {
              const int cc = lane + 32 * c;
              w[i][c] = (!done[i] && cc < grid) ? ld_relaxed_u64(wb + cc) : 0ull;
            }
          }
          bool all_done = true;
#pragma unroll
          for (int i = 0; i < kPollReq; ++i) {
            if (done[i]) continue;
            unsigned long long mx = 0ull;
            int missing = 0;
#pragma unroll
            for (int c = 0; c < kPollWords; ++c) {
              if (lane + 32 * c < grid) {
                missing += (static_cast<uint32_t>(w[i][c] >> 58) != tg) ? 1 : 0;
                mx = w[i][c] > mx ? w[i][c] : mx;
              }
            }
            if (__all_sync(0xffffffffu, missing == 0)) {
              best[i] = warp_max_u64(mx);
              done[i] = true;
            } else {
              all_done = false;
            }
          }
          if (all_done) break;
          int give_up = 0;
          if (lane == 0)
            give_up = (ld_relaxed(a.abort_flag) != 0 || clock64() - t0 > a.wait_cycles) ? 1 : 0;
          if (__shfl_sync(0xffffffffu, give_up, 0)) {
            if (lane == 0 && atomicExch(a.abort_flag, 1) == 0)
              record_error(a.status, DSPARK_ERR_DEVICE_TIMEOUT);
            stop = 1;
            break;
          }
          __nanosleep(20);
        }
        if (stop) {
          if (lane == 0) stop_s = 1;
          break;
        }
        if (lane == 0) {
#pragma unroll
          for (int i = 0; i < kPollReq; ++i) {
            const int b = b0 + i * kPWarps;
            if (b < B) {
              const int d = word_index(best[i]);
              prev_s[b] = d;
              if (cta == 0) a.draft_tokens[static_cast<long long>(b) * k + pos] = d;
            }
          }
        }
        // the next position's context of these requests: markov_w1[draft], gathered
        // by the warp that found it (loads first, then stores)
        if (biased && pos + 1 < k) {
          constexpr int kPerLane = (r + 31) / 32;
          uint32_t ev[kPollReq][kPerLane];
#pragma unroll
          for (int i = 0; i < kPollReq; ++i) {
            const int b = b0 + i * kPWarps;
            const int d = word_index(best[i]);
            const bool ok = b < B && d >= 0 && d < V;
#pragma unroll
            for (int u = 0; u < kPerLane; ++u) {
              const int t = lane + 32 * u;
              ev[i][u] = (ok && t < r) ? static_cast<uint32_t>(a.w1[static_cast<long long>(d) * r + t]) << 16 : 0u;
            }
          }
#pragma unroll
          for (int i = 0; i < kPollReq; ++i) {
            const int b = b0 + i * kPWarps;
            if (b < B) {
#pragma unroll
              for (int u = 0; u < kPerLane; ++u) {
                const int t = lane + 32 * u;
                if (t < r) e_s[(G >= 2) ? (((b >> 1) * r + t) << 1) + (b & 1) : b * r + t] = __uint_as_float(ev[i][u]);
              }
            }
          }
        }
      }
      if (pos + 1 == k) asm volatile("fence.acq_rel.gpu;" ::: "memory");
    }
    __syncthreads();
    if (stop_s) {
      cp_async_wait_all();  // the next group's logits copies land before the CTA exits
      return;
    }
  }

  if (!kStats && a.draft_len_fill && cta == 0)
    for (int b = tid; b < B; b += kPThreads) a.draft_len_fill[b] = k;
  // Off the critical path: softmax statistics of q for every (position, request),
  // spread over the CTAs, one warp each.
  if (kStats) {
    const int pairs = k * B;
    for (int pr = cta * kPWarps + warp; pr < pairs; pr += grid * kPWarps) {
      const int pos = pr / B, b = pr - pos * B;
      const ChainPartial *pb = a.partials + (static_cast<long long>(pos) * B + b) * grid;
      float mmax = -INFINITY;
      for (int c = lane; c < grid; c += 32)
        mmax = fmaxf(mmax, __ldcg(reinterpret_cast<const float *>(pb + c) + 2));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mmax = fmaxf(mmax, __shfl_xor_sync(0xffffffffu, mmax, o));
      double sd = 0.0;
      if (mmax != -INFINITY) {
        for (int c = lane; c < grid; c += 32) {
          const float cm = __ldcg(reinterpret_cast<const float *>(pb + c) + 2);
          const float cs = __ldcg(reinterpret_cast<const float *>(pb + c) + 3);
          if (cm != -INFINITY) sd += static_cast<double>(cs) * static_cast<double>(expf(cm - mmax));
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sd += __shfl_xor_sync(0xffffffffu, sd, o);
      if (lane == 0) {
        const long long at = static_cast<long long>(b) * k + pos;
        if (a.q_stats) {
          a.q_stats[2 * at] = mmax;
          a.q_stats[2 * at + 1] = static_cast<float>(sd);
        }
        if (a.draft_len_fill && pos == k - 1) a.draft_len_fill[b] = k;
      }
    }
  }

  // The last CTA out advances the epoch for the next call.
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(a.done, 1) == grid - 1) {
      *a.done = 0;
      __threadfence();
      st_release(a.epoch, epoch + 1);
    }
  }
}

// ------------------------------------------------- persistent chain, two halves
// Batches of more than 8 requests (r <= 64): 512 threads per CTA in two halves of
// 256.  Half h owns request groups h, h + 2, h + 4, ... (8 requests each) and covers
// the CTA's whole vocabulary slice for them, four rows per thread as above.  The
// halves take turns on the fp32 FMA pipe: half 1 starts the fma chains of a group
// when half 0 has finished those of its group, and the other way round, so that
// while one half takes its argmax, publishes its words and waits for the other CTAs'
// words, the other half's chains run alone on the pipe.  Each (row, request) chain is
// the same sequential fp32 fma chain in rank order as in the kernel above.
//
// Barriers: 1 + h synchronises half h (256 threads); 3 (half 0 arrives, half 1
// waits) and 4 (half 1 arrives, half 0 waits) pass the pipe between the halves.
// Both halves run the same number of group slots (empty slots past the batch end
// keep the barrier sequence), and a half that gives up waiting keeps the sequence
// too, doing no work: every barrier is reached the same number of times by both.
constexpr int kSThreads = 512;
constexpr int kSGroup = 8;

__device__ __forceinline__ void half_sync(int h) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + h), "r"(kPThreads) : "memory");
}
__device__ __forceinline__ void pipe_pass(int h) {  // this half's fma chains are done
  asm volatile("bar.arrive %0, %1;" ::"r"(3 + h), "r"(kSThreads) : "memory");
}
__device__ __forceinline__ void pipe_take(int h) {  // wait for the other half's chains
  asm volatile("bar.sync %0, %1;" ::"r"(4 - h), "r"(kSThreads) : "memory");
}

// kW2Smem: the CTA's markov_w2 slice in shared memory (r <= 64); otherwise (r = 128) it
// is read through L2 at every position after a bulk L2 prefetch, as in the kernel above.
template <int CPR, bool kStats, bool kW2Smem>
__global__ void __launch_bounds__(kSThreads, 1) markov_chain_split(const ChainPArgs a) {
  constexpr int G = kSGroup;
  __shared__ ChainPartial red[2][G][kPWarps];
  __shared__ int stop_s[2], epoch_s, abort0_s;
  extern __shared__ __align__(16) uint8_t psmem[];
  // dynamic shared memory: markov_w2 slice [rows][CPR] (1024-byte aligned), then the
  // contexts e [r][npair4][2] (request pairs, npair4 a multiple of 4), then prev
  // tokens [B] (padded to 16 bytes), then each half's staged logits [G][kPThreads][kPRows]
  const int B = a.B, k = a.k, V = a.V;
  const int npair4 = ((B + 1) / 2 + 3) & ~3;
  constexpr int r = CPR * 8;
  uint4 *w2_s = reinterpret_cast<uint4 *>(psmem);
  const size_t e_bytes = static_cast<size_t>(r) * npair4 * 8;
  float *e_s = reinterpret_cast<float *>(psmem + a.w2_smem_bytes);
  int *prev_s = reinterpret_cast<int *>(psmem + a.w2_smem_bytes + e_bytes);

  const int tid = threadIdx.x, lane = tid & 31;
  const int h = tid >> 8, ht = tid & (kPThreads - 1), hw = ht >> 5;
  float *lg_s = reinterpret_cast<float *>(psmem + a.w2_smem_bytes + e_bytes +
                                          ((static_cast<size_t>(B) * 4 + 15) & ~static_cast<size_t>(15))) +
                static_cast<size_t>(h) * G * kPThreads * kPRows;
  const int grid = gridDim.x, cta = blockIdx.x;
  const bool biased = (a.w1 != nullptr);
  const int v_lo = cta * a.rows_per_cta;
  const int v_hi = min(V, v_lo + a.rows_per_cta);
  const int nrows = max(0, v_hi - v_lo);
  bool valid[kPRows];
  int vrow[kPRows], lrow[kPRows];
#pragma unroll
  for (int j = 0; j < kPRows; ++j) {
    const int row = kPRows * ht + j;
    valid[j] = row < nrows;
    // a CTA past the vocabulary's end (nrows == 0) points its copies at row 0
    vrow[j] = nrows > 0 ? v_lo + (row < nrows ? row : nrows - 1) : 0;
    lrow[j] = nrows > 0 ? vrow[j] - v_lo : 0;
  }
  const bool vec4 = a.vec != 0 && kPRows * ht + kPRows <= nrows;

  // markov_w2 slice into shared memory (or L2) before the wait for the previous kernel
  // (no kernel of the step writes it), 16-byte chunks swizzled as above
  if (biased && nrows > 0) {
    if constexpr (kW2Smem) {
      const uint4 *src = reinterpret_cast<const uint4 *>(a.w2 + static_cast<long long>(v_lo) * r);
      for (int i = tid; i < nrows * CPR; i += kSThreads) {
        const int row = i / CPR, q = i - row * CPR;
        const uint32_t dst = static_cast<uint32_t>(
            __cvta_generic_to_shared(&w2_s[row * CPR + w2_swizzle(row, q, CPR)]));
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src + i) : "memory");
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    } else {
      // 16 KB pieces, one per thread (the slice is at most 1024 rows x 256 bytes)
      const char *src = reinterpret_cast<const char *>(a.w2 + static_cast<long long>(v_lo) * r);
      const uint32_t bytes = static_cast<uint32_t>(nrows) * CPR * 16u;
      const uint32_t off = static_cast<uint32_t>(tid) * 16384u;
      if (off < bytes) {
        const uint32_t n = bytes - off < 16384u ? bytes - off : 16384u;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src + off), "r"(n) : "memory");
      }
    }
  }
  pdl_wait();
  pdl_release();
  if (tid == 0) {
    abort0_s = ld_acquire(a.abort_flag);
    epoch_s = ld_acquire(a.epoch);
    stop_s[0] = stop_s[1] = 0;
    if (abort0_s && cta == 0) record_error(a.status, DSPARK_ERR_DEVICE_TIMEOUT);
  }
  for (int b = tid; b < B; b += kSThreads) {
    int p = a.prev_token[b];
    if (biased && (p < 0 || p >= V)) {
      if (cta == 0) record_error(a.status, DSPARK_ERR_BAD_TOKEN);
      p = -1;
    }
    prev_s[b] = p;
  }
  if (biased && kW2Smem) asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  if (abort0_s) return;
  const int epoch = epoch_s;
  const int ngroups = (B + G - 1) / G;
  const int nslots = (ngroups + 1) / 2;  // group slots per half (the same for both)

  // this half's first group's logits at position 0
  if (h < ngroups) issue_logits_copy<G>(lg_s, a.logits, vrow, vec4, h * G, 0, B, k, V, ht);

  // e_b = markov_w1[prev_b] for position 0, all requests, by the whole CTA
  if (biased) {
    for (int i0 = 0; i0 < B * r; i0 += kSThreads * kGather) {
      uint32_t ev[kGather];
#pragma unroll
      for (int u = 0; u < kGather; ++u) {
        const int idx = i0 + u * kSThreads + tid;
        const int b = idx / r, t = idx - b * r;
        const int p = idx < B * r ? prev_s[b] : -1;
        ev[u] = p >= 0 ? static_cast<uint32_t>(a.w1[static_cast<long long>(p) * r + t]) << 16 : 0u;
      }
#pragma unroll
      for (int u = 0; u < kGather; ++u) {
        const int idx = i0 + u * kSThreads + tid;
        const int b = idx / r, t = idx - b * r;
        if (idx < B * r) e_s[(t * npair4 + (b >> 1)) * 2 + (b & 1)] = __uint_as_float(ev[u]);
      }
    }
  }
  __syncthreads();

  float acc[kPRows][G];
  bool first_fma = true;
  for (int pos = 0; pos < k; ++pos) {
    for (int s = 0; s < nslots; ++s) {
      const int g0 = (2 * s + h) * G;
      const bool active = g0 < B && stop_s[h] == 0;
      const int gb = active ? min(G, B - g0) : 0;
      // the pipe: half 0 waits for half 1's previous chains (none before its first),
      // half 1 for half 0's chains of this slot
      if (h == 1 || !first_fma) pipe_take(h);
      first_fma = false;
#pragma unroll
      for (int j = 0; j < kPRows; ++j)
#pragma unroll
        for (int g = 0; g < G; ++g) acc[j][g] = 0.0f;
      if (biased && active) {
        unsigned long long acc2[kPRows][G / 2];
#pragma unroll
        for (int j = 0; j < kPRows; ++j)
#pragma unroll
          for (int gp = 0; gp < G / 2; ++gp) acc2[j][gp] = 0ull;
        const float *eg = e_s + static_cast<size_t>(g0 >> 1) * 2;
#pragma unroll
        for (int q = 0; q < CPR; ++q) {
          uint4 c[kPRows];
#pragma unroll
          for (int j = 0; j < kPRows; ++j) {
            if constexpr (kW2Smem)
              c[j] = w2_s[lrow[j] * CPR + w2_swizzle(lrow[j], q, CPR)];
            else
              c[j] = __ldg(reinterpret_cast<const uint4 *>(a.w2 + static_cast<long long>(vrow[j]) * r) + q);
          }
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            // contexts of the group's four request pairs at rank 8q + t (32 bytes)
            const float4 *ep = reinterpret_cast<const float4 *>(eg + static_cast<size_t>(q * 8 + t) * npair4 * 2);
            const float4 e01 = ep[0], e23 = ep[1];
            const unsigned long long e2[4] = {pack_f32x2(e01.x, e01.y), pack_f32x2(e01.z, e01.w),
                                              pack_f32x2(e23.x, e23.y), pack_f32x2(e23.z, e23.w)};
#pragma unroll
            for (int j = 0; j < kPRows; ++j) {
              const uint32_t word = (t >> 1) == 0 ? c[j].x : (t >> 1) == 1 ? c[j].y : (t >> 1) == 2 ? c[j].z : c[j].w;
              const float w = (t & 1) ? bf16_hi(word) : bf16_lo(word);
              const unsigned long long wd = pack_f32x2(w, w);
#pragma unroll
              for (int gp = 0; gp < G / 2; ++gp) acc2[j][gp] = fma_f32x2(wd, e2[gp], acc2[j][gp]);
            }
          }
        }
#pragma unroll
        for (int j = 0; j < kPRows; ++j)
#pragma unroll
          for (int gp = 0; gp < G / 2; ++gp) unpack_f32x2(acc2[j][gp], acc[j][2 * gp], acc[j][2 * gp + 1]);
      }
      pipe_pass(h);

      unsigned long long key[G];
      float mx[G], sm[G];
      uint32_t bo[G], bi[G];
      cp_async_wait_all();  // this thread's logits of the group are in lg_s
#pragma unroll
      for (int g = 0; g < G; ++g) {
        bo[g] = 0u;
        bi[g] = 0xffffffffu;
        mx[g] = -INFINITY;
        sm[g] = 0.0f;
        const float4 v = *reinterpret_cast<const float4 *>(&lg_s[(g * kPThreads + ht) * kPRows]);
        float zv[kPRows] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < kPRows; ++j) {
          if (biased) zv[j] = __fadd_rn(zv[j], acc[j][g]);
          acc[j][g] = zv[j];
        }
        if (kPRows * ht + kPRows <= nrows) {
          const float m = fmaxf(fmaxf(zv[0], zv[1]), fmaxf(zv[2], zv[3]));
          int jj = 0;
#pragma unroll
          for (int j = kPRows - 1; j >= 0; --j)
            if (zv[j] == m) jj = j;
          if (g < gb) {
            bo[g] = ordered_bits(m);
            bi[g] = static_cast<uint32_t>(vrow[0] + jj);
            if (kStats && m == m && m != -INFINITY) mx[g] = m;
          }
        } else {
#pragma unroll
          for (int j = 0; j < kPRows; ++j) {
            const float z = zv[j];
            if (valid[j] && g < gb) {
              const uint32_t o = ordered_bits(z);
              if (o > bo[g] || bi[g] == 0xffffffffu) {
                bo[g] = o;
                bi[g] = static_cast<uint32_t>(vrow[j]);
              }
              if (kStats && z == z && z != -INFINITY) mx[g] = fmaxf(mx[g], z);
            }
          }
        }
        if (kStats) {
#pragma unroll
          for (int j = 0; j < kPRows; ++j)
            if (valid[j] && g < gb && mx[g] != -INFINITY && zv[j] == zv[j] && zv[j] != -INFINITY)
              sm[g] += __expf(zv[j] - mx[g]);
        }
      }
      // lg_s is consumed: this half's next group (this position's, else the next's)
      {
        const int gn = g0 + 2 * G;
        if (s + 1 < nslots) {
          if (gn < B) issue_logits_copy<G>(lg_s, a.logits, vrow, vec4, gn, pos, B, k, V, ht);
        } else if (pos + 1 < k && h * G < B) {
          issue_logits_copy<G>(lg_s, a.logits, vrow, vec4, h * G, pos + 1, B, k, V, ht);
        }
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const uint32_t mo = __reduce_max_sync(0xffffffffu, bo[g]);
        const uint32_t mi = __reduce_min_sync(0xffffffffu, bo[g] == mo ? bi[g] : 0xffffffffu);
        key[g] = (static_cast<unsigned long long>(mo) << 32) | (0xffffffffu - mi);
      }
      if (kStats) {
        float mm[G];
#pragma unroll
        for (int g = 0; g < G; ++g) mm[g] = mx[g];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
          for (int g = 0; g < G; ++g) mm[g] = fmaxf(mm[g], __shfl_xor_sync(0xffffffffu, mm[g], o));
#pragma unroll
        for (int g = 0; g < G; ++g) sm[g] = (mx[g] == -INFINITY) ? 0.0f : __fmul_rn(sm[g], expf(mx[g] - mm[g]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
          for (int g = 0; g < G; ++g) sm[g] += __shfl_xor_sync(0xffffffffu, sm[g], o);
#pragma unroll
        for (int g = 0; g < G; ++g) mx[g] = mm[g];
      }
      if (lane == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g)
          if (g < gb) red[h][g][hw] = ChainPartial{key[g], mx[g], sm[g]};
      }
      half_sync(h);
      // warp w of the half combines request w of the group and publishes its word
      if (hw < gb) {
        const int g = hw;
        unsigned long long kk = 0ull;
        float m = -INFINITY, sum = 0.0f;
        if (lane < kPWarps) {
          const ChainPartial c0 = red[h][g][lane];
          kk = c0.key;
          m = c0.m;
          sum = c0.s;
        }
        if (kStats)
          warp_key_stats(kk, m, sum);
        else
          kk = warp_max_u64(kk);
        if (lane == 0) {
          const long long at = (static_cast<long long>(pos) * B + g0 + g) * grid + cta;
          if (kStats) a.partials[at] = ChainPartial{kk, m, sum};
          const unsigned long long wd = pack_word(kk, word_tag(epoch, pos));
          if (pos + 1 < k)
            st_relaxed_u64(a.words + at, wd);
          else
            st_release_u64(a.words + at, wd);
          const int kidx = static_cast<int>(key_index(kk));
          if (biased && pos + 1 < k && kidx >= 0 && kidx < V)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(a.w1 + static_cast<long long>(kidx) * r));
        }
      }
      if (biased) {
#pragma unroll
        for (int g = 0; g < G; ++g)
          if (g < gb)
            store_row4(a.logits + (static_cast<long long>(g0 + g) * k + pos) * V, vrow, valid, vec4,
                       acc[0][g], acc[1][g], acc[2][g], acc[3][g]);
      }
      half_sync(h);  // red[h] is free again
    }

    // Wait for every CTA's word of this half's requests at `pos`: warp w of the half
    // polls request w of each of the half's groups, up to kPollReq at once; the max
    // of the words is the draft token, whose markov_w1 row the warp then gathers.
    if (stop_s[h] == 0) {
      const uint32_t tg = word_tag(epoch, pos);
      const long long t0 = clock64();
      for (int s0 = 0; s0 < nslots; s0 += kPollReq) {
        unsigned long long best[kPollReq];
        bool done[kPollReq];
        int req[kPollReq];
#pragma unroll
        for (int i = 0; i < kPollReq; ++i) {
          req[i] = (2 * (s0 + i) + h) * G + hw;
          best[i] = 0ull;
          done[i] = s0 + i >= nslots || req[i] >= B;
        }
        int stop = 0;
        while (true) {
          unsigned long long w[kPollReq][kPollWords];
#pragma unroll
          for (int i = 0; i < kPollReq; ++i) {
            const unsigned long long *wb = a.words + (static_cast<long long>(pos) * B + (done[i] ? 0 : req[i])) * grid;
#pragma unroll
            for (int c = 0; c < kPollWords; ++c) {
              const int cc = lane + 32 * c;
              w[i][c] = (!done[i] && cc < grid) ? ld_relaxed_u64(wb + cc) : 0ull;
            }
          }
          bool all_done = true;
#pragma unroll
          for (int i = 0; i < kPollReq; ++i) {
            if (done[i]) continue;
            unsigned long long mxw = 0ull;
            int missing = 0;
#pragma unroll
            for (int c = 0; c < kPollWords; ++c) {
              if (lane + 32 * c < grid) {
                missing += (static_cast<uint32_t>(w[i][c] >> 58) != tg) ? 1 : 0;
                mxw = w[i][c] > mxw ? w[i][c] : mxw;
              }
            }
            if (__all_sync(0xffffffffu, missing == 0)) {
              best[i] = warp_max_u64(mxw);
              done[i] = true;
            } else {
              all_done = false;
            }
          }
          if (all_done) break;
          int give_up = 0;
          if (lane == 0)
            give_up = (ld_relaxed(a.abort_flag) != 0 || clock64() - t0 > a.wait_cycles) ? 1 : 0;
          if (__shfl_sync(0xffffffffu, give_up, 0)) {
            if (lane == 0 && atomicExch(a.abort_flag, 1) == 0)
              record_error(a.status, DSPARK_ERR_DEVICE_TIMEOUT);
            stop = 1;
            break;
          }
          __nanosleep(20);
        }
        if (stop) {
          if (lane == 0) stop_s[h] = 1;
          break;
        }
        if (lane == 0) {
#pragma unroll
          for (int i = 0; i < kPollReq; ++i) {
            if (s0 + i < nslots && req[i] < B) {
              const int d = word_index(best[i]);
              prev_s[req[i]] = d;
              if (cta == 0) a.draft_tokens[static_cast<long long>(req[i]) * k + pos] = d;
            }
          }
        }
        if (biased && pos + 1 < k) {
          constexpr int kPerLane = (r + 31) / 32;
          uint32_t ev[kPollReq][kPerLane];
#pragma unroll
          for (int i = 0; i < kPollReq; ++i) {
            const int d = word_index(best[i]);
            const bool ok = s0 + i < nslots && req[i] < B && d >= 0 && d < V;
#pragma unroll
            for (int u = 0; u < kPerLane; ++u) {
              const int t = lane + 32 * u;
              ev[i][u] = (ok && t < r) ? static_cast<uint32_t>(a.w1[static_cast<long long>(d) * r + t]) << 16 : 0u;
            }
          }
#pragma unroll
          for (int i = 0; i < kPollReq; ++i) {
            const int b = req[i];
            if (s0 + i < nslots && b < B) {
#pragma unroll
              for (int u = 0; u < kPerLane; ++u) {
                const int t = lane + 32 * u;
                if (t < r) e_s[(t * npair4 + (b >> 1)) * 2 + (b & 1)] = __uint_as_float(ev[i][u]);
              }
            }
          }
        }
      }
      if (pos + 1 == k) asm volatile("fence.acq_rel.gpu;" ::: "memory");
    }
    half_sync(h);
  }
  // the pipe's last hand-over (half 1's final chains) completes the barrier sequence
  if (h == 0) pipe_take(h);
  cp_async_wait_all();
  __syncthreads();
  if (stop_s[0] || stop_s[1]) return;

  if (!kStats && a.draft_len_fill && cta == 0)
    for (int b = tid; b < B; b += kSThreads) a.draft_len_fill[b] = k;
  if (kStats) {
    constexpr int kSWarps = kSThreads / 32;
    const int warp = tid >> 5;
    const int pairs = k * B;
    for (int pr = cta * kSWarps + warp; pr < pairs; pr += grid * kSWarps) {
      const int pos = pr / B, b = pr - pos * B;
      const ChainPartial *pb = a.partials + (static_cast<long long>(pos) * B + b) * grid;
      float mmax = -INFINITY;
      for (int c = lane; c < grid; c += 32)
        mmax = fmaxf(mmax, __ldcg(reinterpret_cast<const float *>(pb + c) + 2));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mmax = fmaxf(mmax, __shfl_xor_sync(0xffffffffu, mmax, o));
      double sd = 0.0;
      if (mmax != -INFINITY) {
        for (int c = lane; c < grid; c += 32) {
          const float cm = __ldcg(reinterpret_cast<const float *>(pb + c) + 2);
          const float cs = __ldcg(reinterpret_cast<const float *>(pb + c) + 3);
          if (cm != -INFINITY) sd += static_cast<double>(cs) * static_cast<double>(expf(cm - mmax));
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sd += __shfl_xor_sync(0xffffffffu, sd, o);
      if (lane == 0) {
        const long long at = static_cast<long long>(b) * k + pos;
        if (a.q_stats) {
          a.q_stats[2 * at] = mmax;
          a.q_stats[2 * at + 1] = static_cast<float>(sd);
        }
        if (a.draft_len_fill && pos == k - 1) a.draft_len_fill[b] = k;
      }
    }
  }

  if (tid == 0) {
    __threadfence();
    if (atomicAdd(a.done, 1) == grid - 1) {
      *a.done = 0;
      __threadfence();
      st_release(a.epoch, epoch + 1);
    }
  }
}

// c[b, i] = sigmoid(zc[b, i]), zc = w . h[b*k+i] (+ w_m . markov_w1[ctx_i] when the head
// sees the Markov context) + bias; draft_len[b] = first i that fails the truncation rule
// (per position: zc < thr = logit(tau); cumulative: the running sum of log sigmoid(zc)
// falls below log tau); later drafts are replaced by -1.  One CTA per request; wpp warps
// per block position (all k dot products at once, each split over wpp warps, the warps'
// sums added in warp order; the first warp of a position also takes the Markov term).
constexpr int kConfMaxWarps = 32;

struct ConfArgs {
  const uint16_t *h, *conf_w;
  const uint16_t *w1;         // markov_w1 [V, r] or null (plain head)
  const int32_t *prev_token;  // context of position 0 (with w1)
  int32_t *draft_tokens, *draft_len;
  float *conf_out;
  int *status;
  float conf_b, thr;          // thr: logit(tau) (per position) or log(tau) (cumulative)
  int cumulative, r, V, k, H, wpp;
};

__device__ __forceinline__ float log_sigmoid_f(float z) {
  return z >= 0.0f ? -log1pf(expf(-z)) : z - log1pf(expf(z));
}

__global__ void __launch_bounds__(32 * kConfMaxWarps) confidence_kernel(const ConfArgs a) {
  __shared__ float part_s[kConfMaxWarps];
  __shared__ float zc_s[kMaxK];
  __shared__ int len_s;
  pdl_wait();
  pdl_release();  // one CTA per request: one wave
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int k = a.k, H = a.H;
  const int pos = warp / a.wpp, part = warp - pos * a.wpp;
  if (pos < k) {
    const uint4 *hrow = reinterpret_cast<const uint4 *>(a.h + (static_cast<long long>(b) * k + pos) * H);
    const uint4 *wrow = reinterpret_cast<const uint4 *>(a.conf_w);
    float acc = 0.0f;
#pragma unroll 4
    for (int c = part * 32 + lane; c < H / 8; c += 32 * a.wpp) {
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
    if (a.w1 && part == 0) {
      // the Markov context of this position: the bonus token for position 0, else the
      // draft of the position before (read before any draft is overwritten below)
      const int ctx = pos == 0 ? a.prev_token[b] : a.draft_tokens[static_cast<long long>(b) * k + pos - 1];
      if (ctx >= 0 && ctx < a.V) {
        for (int t = lane; t < a.r; t += 32)
          acc = __fmaf_rn(bf16_lo(static_cast<uint32_t>(a.conf_w[H + t])),
                          bf16_lo(static_cast<uint32_t>(a.w1[static_cast<long long>(ctx) * a.r + t])), acc);
      } else if (lane == 0) {
        record_error(a.status, DSPARK_ERR_BAD_TOKEN);
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) part_s[warp] = acc;
  }
  __syncthreads();
  if (threadIdx.x < k) {
    const int i = threadIdx.x;
    float zc = 0.0f;
    for (int w = 0; w < a.wpp; ++w) zc += part_s[i * a.wpp + w];
    zc += a.conf_b;
    zc_s[i] = zc;
    if (a.conf_out) a.conf_out[static_cast<long long>(b) * k + i] = 1.0f / (1.0f + expf(-zc));
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int len = k;
    float cum = 0.0f;
    for (int i = 0; i < k; ++i) {
      bool keep;
      if (a.cumulative) {
        cum += log_sigmoid_f(zc_s[i]);
        keep = cum >= a.thr;
      } else {
        keep = zc_s[i] >= a.thr;
      }
      if (!keep) {
        len = i;
        break;
      }
    }
    len_s = len;
    a.draft_len[b] = len;
  }
  __syncthreads();
  if (threadIdx.x < k && threadIdx.x >= len_s)
    a.draft_tokens[static_cast<long long>(b) * k + threadIdx.x] = -1;
}

}  // namespace

// Chain workspace: [0] ticket of the per-position kernel, [4] epoch, [8] exit
// count, [12] abort flag; position words from byte 256 (k x B x kMaxPGrid u64,
// zero = not written); partials after them.
size_t chain_words_bytes(int B, int k) {
  return align_up(static_cast<size_t>(k) * B * kMaxPGrid * sizeof(unsigned long long), kWsAlign);
}

size_t chain_counter_bytes(int B, int k) { return kWsAlign + chain_words_bytes(B, k); }

size_t chain_workspace_size(int B, int k, int V) {
  const int nchunks = (V + kChunk - 1) / kChunk;
  const size_t per_pos = static_cast<size_t>(B) * nchunks * sizeof(ChainPartial);
  const size_t persistent = static_cast<size_t>(k) * B * kMaxPGrid * sizeof(ChainPartial);
  return kWsAlign + chain_words_bytes(B, k) +
         align_up(per_pos > persistent ? per_pos : persistent, kWsAlign);
}

namespace {

// Cooperative launch of a persistent chain kernel (all CTAs resident together: they
// wait on each other), with programmatic dependent launch when enabled (without it if
// the combination is refused).  The opt-in dynamic shared memory is raised to what
// this launch needs (the kernel's static shared memory plus the dynamic part must
// stay within the per-CTA limit, so not to a fixed maximum).
// attr_bytes: the attribute already set per device, one table per kernel (the caller's
// static: every chain kernel has the same function type).
template <typename Kern>
bool launch_chain_coop(Kern kern, size_t (&attr_bytes)[64], int grid, int threads, size_t smem,
                       const ChainPArgs &a, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  if (attr_bytes[dev] < smem) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    attr_bytes[dev] = smem;
  }
  if (pdl_enabled()) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, kern, a) == cudaSuccess) return true;
    cudaGetLastError();
  }
  void *params[] = {const_cast<ChainPArgs *>(&a)};
  if (cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(kern), dim3(grid), dim3(threads),
                                  params, smem, stream) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return true;
}

// Grid and slice of the persistent chains: one CTA per SM (at most kMaxPGrid), at
// least 256 rows per CTA, slices a multiple of kPRows rows; false if a slice would
// exceed kPRows x kPThreads rows.
bool chain_grid(int V, int &grid, int &rows) {
  const int sms = device_sm_count();
  if (sms <= 0) return false;
  grid = sms < kMaxPGrid ? sms : kMaxPGrid;
  const int by_rows = (V + 255) / 256;
  if (grid > by_rows) grid = by_rows;
  rows = ((V + grid - 1) / grid + kPRows - 1) / kPRows * kPRows;
  return rows <= kPRows * kPThreads;
}

template <int G, int CPR, bool kStats, bool kW2Smem>
bool try_persistent_r(const ChainPArgs &args0, int B, int V, cudaStream_t stream) {
  int grid = 0, rows = 0;
  if (!chain_grid(V, grid, rows)) return false;
  ChainPArgs a = args0;
  a.rows_per_cta = rows;
  a.vec = ((V % kPRows) == 0 && (reinterpret_cast<uintptr_t>(a.logits) & 15u) == 0) ? 1 : 0;
  a.w2_smem_bytes =
      kW2Smem ? static_cast<int>(align_up(static_cast<size_t>(rows) * CPR * 16, 1024)) : 0;
  const size_t smem = static_cast<size_t>(a.w2_smem_bytes) +
                      static_cast<size_t>((B + 1) & ~1) * CPR * 32 +
                      ((static_cast<size_t>(B) * sizeof(int) + 15) & ~static_cast<size_t>(15)) +
                      (G >= 8 ? static_cast<size_t>(G) * kPRows * kPThreads * sizeof(float) : 0);
  if (smem > kPSmemMax) return false;
  static size_t attr_bytes[64] = {};
  return launch_chain_coop(markov_chain_persistent<G, CPR, kStats, kW2Smem>, attr_bytes, grid, kPThreads,
                           smem, a, stream);
}

template <int CPR, bool kStats, bool kW2Smem>
bool try_split_r(const ChainPArgs &args0, int B, int V, cudaStream_t stream) {
  int grid = 0, rows = 0;
  if (!chain_grid(V, grid, rows)) return false;
  ChainPArgs a = args0;
  a.rows_per_cta = rows;
  a.vec = ((V % kPRows) == 0 && (reinterpret_cast<uintptr_t>(a.logits) & 15u) == 0) ? 1 : 0;
  a.w2_smem_bytes = kW2Smem ? static_cast<int>(align_up(static_cast<size_t>(rows) * CPR * 16, 1024)) : 0;
  const size_t npair4 = static_cast<size_t>(((B + 1) / 2 + 3) & ~3);
  const size_t smem = static_cast<size_t>(a.w2_smem_bytes) + npair4 * CPR * 64 +
                      ((static_cast<size_t>(B) * sizeof(int) + 15) & ~static_cast<size_t>(15)) +
                      2 * static_cast<size_t>(kSGroup) * kPRows * kPThreads * sizeof(float);
  if (smem > kPSmemMax) return false;
  static size_t attr_bytes[64] = {};
  return launch_chain_coop(markov_chain_split<CPR, kStats, kW2Smem>, attr_bytes, grid, kSThreads, smem, a,
                           stream);
}

template <bool kStats>
bool try_split_s(const ChainPArgs &a, int r, int B, int V, cudaStream_t stream) {
  switch (r) {
    case 16: return try_split_r<2, kStats, true>(a, B, V, stream);
    case 32: return try_split_r<4, kStats, true>(a, B, V, stream);
    case 64: return try_split_r<8, kStats, true>(a, B, V, stream);
    case 128: return try_split_r<16, kStats, false>(a, B, V, stream);
    default: return false;
  }
}

template <int G, bool kStats>
bool try_persistent_s(const ChainPArgs &a, int r, int B, int V, cudaStream_t stream) {
  switch (r) {
    case 0: return try_persistent_r<G, 1, kStats, true>(a, B, V, stream);  // no bias: rank unused
    case 16: return try_persistent_r<G, 2, kStats, true>(a, B, V, stream);
    case 32: return try_persistent_r<G, 4, kStats, true>(a, B, V, stream);
    case 64: return try_persistent_r<G, 8, kStats, true>(a, B, V, stream);
    case 128: return try_persistent_r<G, 16, kStats, false>(a, B, V, stream);
    default: return false;  // other ranks: per-position kernels
  }
}

template <int G>
bool try_persistent(const ChainPArgs &a, int r, int B, int V, cudaStream_t stream) {
  return a.q_stats ? try_persistent_s<G, true>(a, r, B, V, stream)
                   : try_persistent_s<G, false>(a, r, B, V, stream);
}

}  // namespace

dspark_status_t chain_launch(float *logits, const uint16_t *w1, const uint16_t *w2, int r,
                             const int32_t *prev_token, int32_t *draft_tokens, float *q_stats,
                             int32_t *draft_len_fill, int B, int k, int V, void *ws,
                             int *status, cudaStream_t stream) {
  int *ctrl = reinterpret_cast<int *>(ws);
  unsigned long long *words =
      reinterpret_cast<unsigned long long *>(static_cast<char *>(ws) + kWsAlign);
  ChainPartial *partials = reinterpret_cast<ChainPartial *>(static_cast<char *>(ws) + kWsAlign +
                                                           chain_words_bytes(B, k));

  ChainPArgs pa;
  pa.logits = logits;
  pa.w1 = w1;
  pa.w2 = w2;
  pa.prev_token = prev_token;
  pa.draft_tokens = draft_tokens;
  pa.q_stats = q_stats;
  pa.draft_len_fill = draft_len_fill;
  pa.partials = partials;
  pa.words = words;
  pa.epoch = ctrl + 1;
  pa.done = ctrl + 2;
  pa.abort_flag = ctrl + 3;
  pa.status = status;
  pa.r = w1 ? r : 0;
  pa.B = B;
  pa.k = k;
  pa.V = V;
  pa.rows_per_cta = 0;
  pa.w2_smem_bytes = 0;
  // DSPARK_CHAIN_PER_POSITION=1 selects the per-position kernels (same results).
  const char *env = getenv("DSPARK_CHAIN_PER_POSITION");
  const bool per_position = env && env[0] == '1';
  // DSPARK_CHAIN_WAIT_CYCLES: budget of each wait for the other CTAs' words (default
  // about a second); a tiny budget makes the waits give up (a failure-path test).
  pa.wait_cycles = kBarrierCycles;
  if (const char *wc = getenv("DSPARK_CHAIN_WAIT_CYCLES")) {
    const long long v = atoll(wc);
    if (v >= 0) pa.wait_cycles = v;
  }
  // Batches of more than 8 requests: the two-halves kernel, unless
  // DSPARK_CHAIN_SPLIT=0 (same results).
  const char *senv = getenv("DSPARK_CHAIN_SPLIT");
  const bool split = !per_position && B > 8 && !(senv && senv[0] == '0');
  bool split_ok = false;
  if (split)
    split_ok = pa.q_stats ? try_split_s<true>(pa, pa.r, B, V, stream)
                          : try_split_s<false>(pa, pa.r, B, V, stream);
  const bool ok = per_position ? false
                  : split_ok ? true
                  : B >= 8 ? try_persistent<8>(pa, pa.r, B, V, stream)
                  : B >= 4 ? try_persistent<4>(pa, pa.r, B, V, stream)
                  : B >= 2 ? try_persistent<2>(pa, pa.r, B, V, stream)
                           : try_persistent<1>(pa, pa.r, B, V, stream);
  if (ok) {
    count_launches(1);
    return DSPARK_OK;
  }

  const int nchunks = (V + kChunk - 1) / kChunk;
  int *counter = ctrl;
  for (int pos = 0; pos < k; ++pos) {
    const int32_t *prev_src = pos == 0 ? prev_token : draft_tokens + (pos - 1);
    const int prev_stride = pos == 0 ? 1 : k;
    auto kern = B >= 8 ? markov_chain_kernel<8>
                       : (B >= 4 ? markov_chain_kernel<4>
                                 : (B >= 2 ? markov_chain_kernel<2> : markov_chain_kernel<1>));
    if (launch_pdl(kern, dim3(nchunks), dim3(kThreads), 0, stream, logits, w1, w2, r, prev_src,
                   prev_stride, draft_tokens, q_stats, draft_len_fill, B, k, V, pos, nchunks,
                   partials, counter, status) != cudaSuccess)
      return DSPARK_ERR_CUDA;
    count_launches(1);
  }
  return DSPARK_OK;
}

dspark_status_t confidence_launch(const uint16_t *h, const uint16_t *conf_w, float conf_b,
                                  float conf_tau, int cumulative, const uint16_t *w1, int r, int V,
                                  const int32_t *prev_token, int32_t *draft_tokens,
                                  int32_t *draft_len, float *conf_out, int B, int k, int H,
                                  int *status, cudaStream_t stream) {
  ConfArgs a;
  a.h = h;
  a.conf_w = conf_w;
  a.w1 = w1;
  a.prev_token = prev_token;
  a.draft_tokens = draft_tokens;
  a.draft_len = draft_len;
  a.conf_out = conf_out;
  a.status = status;
  a.conf_b = conf_b;
  a.cumulative = cumulative ? 1 : 0;
  a.r = w1 ? r : 0;
  a.V = V;
  a.k = k;
  a.H = H;
  // thresholds: tau <= 0 keeps every position, tau >= 1 keeps none
  if (conf_tau <= 0.0f)
    a.thr = -INFINITY;
  else if (conf_tau >= 1.0f)
    a.thr = INFINITY;
  else if (cumulative)
    a.thr = static_cast<float>(log(static_cast<double>(conf_tau)));
  else
    a.thr = static_cast<float>(log(static_cast<double>(conf_tau)) - log1p(-static_cast<double>(conf_tau)));
  // warps per position: as many as fit in 32 warps, no more than the 16-byte chunks of
  // a row over 32 lanes
  int wpp = kConfMaxWarps / k;
  const int chunks_per_lane_min = 2;
  while (wpp > 1 && (H / 8) / (32 * wpp) < chunks_per_lane_min) --wpp;
  a.wpp = wpp;
  if (launch_pdl(confidence_kernel, dim3(B), dim3(32 * wpp * k), 0, stream, a) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  count_launches(1);
  return DSPARK_OK;
}

}  // namespace dspark
