// Verification of one draft block per request: greedy exact match or
// probabilistic rejection sampling.
//
// Pages: "Qwen3.8-27B DFlash drafter recipe" ("greedy spec decode is lossless
// by construction"), the "Qwen3.8-27B-DSpark-vLLM" card ("draft_sample_method":
// "probabilistic"), "Qwen4Exp DFlash2 hidden-state capture" ("verified by
// rejection sampling"; acceptance length = accepted tokens per verification
// step).  Rejection rule: accept d with probability min(1, p(d)/q(d)); at the
// first rejection draw from max(0, p - q) normalised; after a fully accepted
// block draw the bonus token from p.
//
// Two stages.
//
// Row statistics (row_stats_kernel): one streaming read of a set of fp32 rows
// with 128-bit loads.  Each CTA reduces a 16384-entry slice of one row to
// (argmax key, max, sum exp(x - max)); the last CTA of a row (atomic ticket,
// nobody waits) merges the slices in a fixed order and stores the row's
// (max, sum) and argmax.  Applied to the target rows it depends on nothing but
// the target logits, so it can run as soon as they exist (in a serving loop:
// right after the target forward, beside the next block's fc and LM head, which
// also need only the target forward's outputs).  Applied to the draft-logit
// rows it yields q's statistics when the drafting kernel did not supply them.
//
// Decision and draw (verify_draw_kernel, probabilistic; verify_greedy_kernel,
// greedy): with the row statistics known, the accept/reject tests of a request
// need only its drafted tokens and two gathered logits per position.  Every CTA
// of the draw grid takes its request's decision itself (a handful of loads,
// identical in every CTA), then reduces one slice (1024 entries per Philox block
// per thread; 1 to 4 blocks per thread, fewer CTAs for larger batches) of the row
// that needs a draw.  The draw is the Gumbel-max rule: the index maximising
// log w_v + G_v, G_v = -log(-log U_v) with U_v from Philox counter (request,
// row, step, 1 + v/4).  That samples exactly from w normalised and makes the
// draw an argmax, reduced like every other argmax here (per-CTA 64-bit keys,
// merged by the request's last CTA).  One launch after the drafts exist.
#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace dspark {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kPer = 64;                    // entries per thread per slice (row statistics),
                                            // all loaded before any is used
constexpr int kSlice = kThreads * kPer;     // 16384 entries (64 KB) per CTA (row statistics)
constexpr int kDrawSlice = kThreads * 4;    // 1024 entries per draw block: one Philox block per thread

struct __align__(16) RowPartial {
  unsigned long long key;
  float m;
  float s;
};

enum SampleKind { kNone = 0, kResidual = 1, kResidualOneHot = 2, kFromP = 3 };

struct __align__(16) SampleJob {
  int row;     // block row of the target (and draft) logits to draw from
  int kind;
  int d;       // draft token removed by the one-hot residual
  int acc_len;
  double cp;   // log-normaliser of the target row: max + log(sum exp)
  double cq;   // log-normaliser of the draft row (kResidual)
};

struct __align__(16) SamplePartial {
  unsigned long long best_r;  // argmax key of log w + G over the slice
  unsigned long long best_p;  // argmax key of log p + G (fallback: residual all zero)
};

// Atomic ticket `t`: true for the CTA that arrives last (of `count`), which then
// resets the ticket.  Block-wide.
// The CTA's partial was stored by thread 0; thread 0's ticket increment is an
// acquire-release atomic, so the partial is visible before the ticket moves, and the
// last CTA's thread 0 sees every other CTA's partial; the CTA barrier then orders the
// reads of the other threads after that acquire.  (A fence in every thread of every
// CTA cost about a microsecond per CTA wave.)
__device__ __forceinline__ bool last_arrival(int *t, int count, int *flag_s) {
  if (threadIdx.x == 0) {
    int old;
    asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;" : "=r"(old) : "l"(t) : "memory");
    const bool last = (old == count - 1);
    if (last) *t = 0;
    *flag_s = last ? 1 : 0;
  }
  __syncthreads();
  const bool last = *flag_s != 0;
  if (last) __threadfence();  // the last CTA only: its threads read the others' partials
  return last;
}

__device__ __forceinline__ int clamp_len(const int32_t *draft_len, int b, int k, int *status) {
  int L = draft_len ? draft_len[b] : k;
  if (L < 0 || L > k) {
    if (status) record_error(status, DSPARK_ERR_INVALID_ARG);
    L = L < 0 ? 0 : k;
  }
  return L;
}

// ------------------------------------------------------------------ row statistics
// One set of rows reduced by a row-statistics launch (a launch reduces one or two sets,
// e.g. the target rows and the draft-logit rows of a verify).
struct RowSet {
  const float *rows;      // [nrows, V]
  float *ms;              // [nrows, 2]: (max, sum exp(x - max)); may be null
  int32_t *argmax;        // [nrows]; may be null
  RowPartial *parts;      // [nrows, nslices]
  int *tickets;           // [nrows]
  const int32_t *len;     // optional: row rho = g * group + j is read only if j <= len[g] + len_off
  int group, len_off;
  long long nrows;
  int vec;                // 1 when rows start on 16-byte boundaries (128-bit loads)
};

struct RowStatsArgs {
  RowSet set[2];
  long long blocks0;      // CTAs of set 0 (nrows * nslices); set 1's follow
  int k;                  // the cap of len, for the clamp
  int V;
  int nslices;
};

// This thread's KP entries of slice `slice` of `row`: entry e has index
// base + (e/4)*1024 + 4*tid + e%4 (vector loads) or base + e*256 + tid; -inf past V.
template <int KP>
__device__ __forceinline__ void load_slice(const float *row, int V, int slice, int vec, float (&x)[KP]) {
  const int tid = threadIdx.x;
  const int base = slice * (kThreads * KP);
  if (vec) {
#pragma unroll
    for (int it = 0; it < KP / 4; ++it) {
      const int v = base + it * (kThreads * 4) + tid * 4;
      const float4 q = v < V ? __ldcs(reinterpret_cast<const float4 *>(row + v))
                             : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      x[4 * it] = q.x; x[4 * it + 1] = q.y; x[4 * it + 2] = q.z; x[4 * it + 3] = q.w;
    }
  } else {
#pragma unroll
    for (int it = 0; it < KP; ++it) {
      const int v = base + it * kThreads + tid;
      x[it] = v < V ? __ldcs(row + v) : -INFINITY;
    }
  }
}

// (argmax key, max, sum exp) of one slice whose entries this thread holds in x; thread
// 0 stores it in *dst.  Block-wide; `red` is shared scratch of kWarps entries.
template <int KP, bool kSums>
__device__ void slice_stats(const float (&x)[KP], int V, int slice, int vec, RowPartial *red,
                            RowPartial *dst) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int base = slice * (kThreads * KP);
  auto index_of = [&](int e) {
    return vec ? base + (e >> 2) * (kThreads * 4) + tid * 4 + (e & 3) : base + e * kThreads + tid;
  };
  // A slice wholly inside the row (every slice but a row's last): the max by fmaxf
  // (which passes over NaN like the strict compare), then the first entry holding it
  // (ascending index); the same value and index as the strict-compare scan below.
  const bool full = base + kThreads * KP <= V;
  float bv = -INFINITY;
  int bi = -1;
  if (full) {
    float m = -INFINITY;
#pragma unroll
    for (int e = 0; e < KP; ++e) m = fmaxf(m, x[e]);
    if (m != -INFINITY) {
#pragma unroll
      for (int e = KP - 1; e >= 0; --e) {
        if (x[e] == m) {  // the last hit is the lowest index
          bv = x[e];
          bi = index_of(e);
        }
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < KP; ++e) {
      const int xi = index_of(e);
      if (xi < V && x[e] > bv) {
        bv = x[e];
        bi = xi;
      }
    }
  }
  const int x0 = index_of(0);
  unsigned long long best = bi >= 0 ? argmax_key(bv, static_cast<uint32_t>(bi))
                                    : (x0 < V ? argmax_key(-INFINITY, static_cast<uint32_t>(x0)) : 0ull);
  SoftStat st{-INFINITY, 0.0f};
  if (kSums && bi >= 0 && bv != INFINITY) {
    float sum = 0.0f;
    if (full) {
      // every entry in range; -inf adds exp(-inf) = +0 and NaN adds +0, both exact
      // no-ops on a sum that starts at +0, so the sum is the one of the scan below
#pragma unroll
      for (int e = 0; e < KP; ++e) sum += (x[e] == x[e]) ? __expf(x[e] - bv) : 0.0f;
    } else {
#pragma unroll
      for (int e = 0; e < KP; ++e)
        if (index_of(e) < V && x[e] == x[e] && x[e] != -INFINITY) sum += __expf(x[e] - bv);
    }
    st = SoftStat{bv, sum};
  }
  best = warp_max_u64(best);
  if (kSums) {
    // warp (max, sum): the max first, then the sum of s * exp(m - max)
    float mm = st.m;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mm = fmaxf(mm, __shfl_xor_sync(0xffffffffu, mm, o));
    float ss = (st.m == -INFINITY) ? 0.0f : st.s * __expf(st.m - mm);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    st = SoftStat{mm, ss};
  }
  if (lane == 0) red[warp] = RowPartial{best, st.m, st.s};
  __syncthreads();
  if (tid == 0) {
    RowPartial acc = red[0];
    SoftStat sacc{acc.m, acc.s};
    for (int w = 1; w < kWarps; ++w) {
      acc.key = red[w].key > acc.key ? red[w].key : acc.key;
      sacc = softstat_merge(sacc, SoftStat{red[w].m, red[w].s});
    }
    acc.m = sacc.m;
    acc.s = sacc.s;
    *dst = acc;
  }
}

// Warp 0 of a row's last CTA: merges the slice partials (max first, then the sum of
// s * exp(m - max) in fp64, one pass with online rescaling) and stores the row's
// statistics.
template <bool kSums>
__device__ void merge_row(const RowSet &a, int nslices, long long rho) {
  const int lane = threadIdx.x & 31;
  const RowPartial *pr = a.parts + rho * nslices;
  unsigned long long kb = 0ull;
  float mm = -INFINITY;
  double s = 0.0;
  for (int c = lane; c < nslices; c += 32) {
    const ulonglong2 raw = __ldcg(reinterpret_cast<const ulonglong2 *>(pr + c));
    kb = raw.x > kb ? raw.x : kb;
    const float cm = __uint_as_float(static_cast<uint32_t>(raw.y));
    const float cs = __uint_as_float(static_cast<uint32_t>(raw.y >> 32));
    if (kSums && cm != -INFINITY) {
      if (cm > mm) {
        s = (mm == -INFINITY) ? static_cast<double>(cs)
                              : s * static_cast<double>(expf(mm - cm)) + static_cast<double>(cs);
        mm = cm;
      } else {
        s += static_cast<double>(cs) * static_cast<double>(expf(cm - mm));
      }
    }
  }
  kb = warp_max_u64(kb);
  if (kSums) {
    float wm = mm;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
    s = (mm == -INFINITY) ? 0.0 : s * static_cast<double>(expf(mm - wm));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    mm = wm;
  }
  if (lane == 0) {
    if (a.ms) {
      a.ms[2 * rho] = mm;
      a.ms[2 * rho + 1] = static_cast<float>(s);
    }
    if (a.argmax) a.argmax[rho] = static_cast<int32_t>(key_index(kb));
  }
}

// One CTA per (row, slice): the slice's KP entries per thread are loaded together,
// reduced, and the row's last CTA to arrive merges the slices.  Rows past a request's
// draft length are skipped (every slice of such a row returns at once, so its ticket
// never moves).
template <int KP, bool kSums>
__global__ void __launch_bounds__(kThreads) row_stats_kernel(const __grid_constant__ RowStatsArgs a) {
  __shared__ RowPartial red[kWarps];
  __shared__ int flag_s;
  // 1-D grid (rows can exceed the 65535 limit of gridDim.y): block = row * nslices + slice,
  // set 0's blocks first
  const bool second = blockIdx.x >= a.blocks0;
  const RowSet &rs = second ? a.set[1] : a.set[0];
  const long long bid = second ? blockIdx.x - a.blocks0 : blockIdx.x;
  const int slice = static_cast<int>(bid % a.nslices);
  const long long rho = bid / a.nslices;
  pdl_wait();
  if (rs.len) {
    const int g = static_cast<int>(rho / rs.group), j = static_cast<int>(rho - static_cast<long long>(g) * rs.group);
    if (j > clamp_len(rs.len, g, a.k, nullptr) + rs.len_off) {
      pdl_release();
      return;
    }
  }
  float x[KP];
  load_slice<KP>(rs.rows + rho * a.V, a.V, slice, rs.vec, x);
  slice_stats<KP, kSums>(x, a.V, slice, rs.vec, red, rs.parts + rho * a.nslices + slice);
  pdl_release();  // after this CTA's pass: the grid may span many waves
  if (!last_arrival(rs.tickets + rho, a.nslices, &flag_s)) return;
  if (threadIdx.x < 32) merge_row<kSums>(rs, a.nslices, rho);
}

// ------------------------------------------------------------------ decision and draw
struct DrawArgs {
  const float *target;      // [B, k+1, V]
  const float *t_ms;        // [B, k+1, 2] target row (max, sum exp)
  const int32_t *t_arg;     // [B, k+1] target row argmax (greedy)
  const int32_t *drafts;    // [B, k]
  const int32_t *draft_len; // [B] or null (= k)
  const float *zlog;        // [B, k, V] draft logits, or null (one-hot q)
  const float *q_ms;        // [B, k, 2] draft row (max, sum exp) when zlog is given
  const uint32_t *request_id;
  int32_t *accepted_len;
  int32_t *next_token;
  SamplePartial *sparts;    // [B, ndraw]
  int *tickets;             // [B]
  int *status;
  unsigned long long seed;
  unsigned int step;
  int B, k, V;
  int ndraw;
  int vec;
};

// Warp 0: the accept/reject decisions of request b (lane j takes block position j)
// and the draw job they leave.  Every CTA of the request computes the same job.
// p(d)/q(d) = exp((T_d - M) - (z_d - m)) * s / S: the exponent is formed exactly in
// fp64, the exponential in fp32 (relative error ~1e-7).
__device__ void decide_request(const DrawArgs &a, int b, SampleJob *job_s, bool record) {
  const int lane = threadIdx.x & 31;
  const int k = a.k, V = a.V;
  const int L = clamp_len(a.draft_len, b, k, record ? a.status : nullptr);
  const long long drow = static_cast<long long>(b) * k;
  const long long trow = static_cast<long long>(b) * (k + 1);
  const uint32_t req = a.request_id ? a.request_id[b] : static_cast<uint32_t>(b);
  int dt = -1;
  bool bad = false, stop = false;
  if (lane < L) {
    dt = a.drafts[drow + lane];
    bad = (dt < 0 || dt >= V);
    double ratio = 0.0;
    if (!bad) {
      const float tT = a.target[(trow + lane) * V + dt];
      const float2 tm = *reinterpret_cast<const float2 *>(a.t_ms + 2 * (trow + lane));
      double ex = static_cast<double>(tT) - static_cast<double>(tm.x);
      double sc = 1.0 / static_cast<double>(tm.y);
      if (a.zlog) {
        const float zd = a.zlog[(drow + lane) * V + dt];
        const float2 qm = *reinterpret_cast<const float2 *>(a.q_ms + 2 * (drow + lane));
        ex -= static_cast<double>(zd) - static_cast<double>(qm.x);
        sc *= static_cast<double>(qm.y);
      }
      ratio = static_cast<double>(expf(static_cast<float>(ex))) * sc;
    }
    double ua, us;
    verify_uniforms(a.seed, req, static_cast<uint32_t>(lane), a.step, ua, us);
    stop = bad || !(ua < ratio);
  }
  const unsigned stops = __ballot_sync(0xffffffffu, stop);
  const int acc = stops ? __ffs(stops) - 1 : L;
  const int stop_bad = __shfl_sync(0xffffffffu, bad ? 1 : 0, acc & 31);
  const int dsel = __shfl_sync(0xffffffffu, dt, acc & 31);
  if (lane == 0) {
    SampleJob job;
    job.row = acc;
    job.acc_len = acc;
    job.d = -1;
    job.cq = 0.0;
    if (acc < L && stop_bad) {
      if (record) record_error(a.status, DSPARK_ERR_BAD_TOKEN);
      job.kind = kFromP;
    } else if (acc < L) {
      job.kind = a.zlog ? kResidual : kResidualOneHot;
      job.d = dsel;
      if (a.zlog) {
        const float2 qm = *reinterpret_cast<const float2 *>(a.q_ms + 2 * (drow + acc));
        job.cq = static_cast<double>(qm.x) + log(static_cast<double>(qm.y));
      }
    } else {
      job.kind = kFromP;
    }
    const float2 tm = *reinterpret_cast<const float2 *>(a.t_ms + 2 * (trow + acc));
    job.cp = static_cast<double>(tm.x) + log(static_cast<double>(tm.y));
    *job_s = job;
  }
}

// Noise of entry v of a draw at block row `row`: Philox4x32-10 counter
// (request, row, step, 1 + v/4), word v mod 4; U = (2 (w >> 9) + 1) 2^-24 is an
// odd multiple of 2^-24, exact in fp32 and strictly inside (0, 1).
// The inner logarithm is the accurate one (-log u is tiny when u is near 1,
// where an approximate log would lose all relative precision); the outer one is
// the fast intrinsic (absolute error ~2^-21 relative to |G| + 1).
__device__ __forceinline__ float gumbel_from_word(uint32_t w) {
  const float u = static_cast<float>(2u * (w >> 9) + 1u) * (1.0f / 16777216.0f);
  return -__logf(-logf(u));
}

// Gumbel-max keys of one slice (NB blocks of 1024 entries, one Philox block of 4 entries
// per thread in each) of the draw row of request b -> draw partial (block-wide).
// `red_r`, `red_p` are shared scratch of kWarps.
template <int NB>
__device__ void draw_slice(const DrawArgs &a, const SampleJob &job, int b, int slice,
                           unsigned long long *red_r, unsigned long long *red_p) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k = a.k, V = a.V;
  const uint32_t req = a.request_id ? a.request_id[b] : static_cast<uint32_t>(b);
  const uint32_t k0 = static_cast<uint32_t>(a.seed & 0xffffffffull);
  const uint32_t k1 = static_cast<uint32_t>(a.seed >> 32);
  const float *trow = a.target + (static_cast<long long>(b) * (k + 1) + job.row) * V;
  const float *zrow = (job.kind == kResidual)
                          ? a.zlog + (static_cast<long long>(b) * k + job.row) * V
                          : nullptr;
  const float cpf = static_cast<float>(job.cp);
  const float cqf = static_cast<float>(job.cq);

  unsigned long long best_r = 0ull, best_p = 0ull;
  // every block's row values first (loads in flight together), then the arithmetic
  float tv[NB][4], zv[NB][4];
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    const int vg = (slice * NB + nb) * kDrawSlice + tid * 4;
    if (a.vec && vg + 4 <= V) {
      const float4 t4 = __ldcs(reinterpret_cast<const float4 *>(trow + vg));
      tv[nb][0] = t4.x; tv[nb][1] = t4.y; tv[nb][2] = t4.z; tv[nb][3] = t4.w;
      if (zrow) {
        const float4 z4 = __ldcs(reinterpret_cast<const float4 *>(zrow + vg));
        zv[nb][0] = z4.x; zv[nb][1] = z4.y; zv[nb][2] = z4.z; zv[nb][3] = z4.w;
      } else {
        zv[nb][0] = zv[nb][1] = zv[nb][2] = zv[nb][3] = 0.0f;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        tv[nb][e] = vg + e < V ? trow[vg + e] : 0.0f;
        zv[nb][e] = (zrow && vg + e < V) ? zrow[vg + e] : 0.0f;
      }
    }
  }
#pragma unroll
  for (int nb = 0; nb < NB; ++nb) {
    const int vg = (slice * NB + nb) * kDrawSlice + tid * 4;
    if (vg < V) {
      const U4 w = philox4x32_10(U4{req, static_cast<uint32_t>(job.row), a.step,
                                    1u + static_cast<uint32_t>(vg >> 2)},
                                 k0, k1);
      const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int v = vg + e;
        if (v < V) {
          const float g = gumbel_from_word(words[e]);
          const float t = tv[nb][e];
          const float kp = t + g;
          float kr;
          if (job.kind == kResidual) {
            const float av = t - cpf;
            const float bv = zv[nb][e] - cqf;
            kr = (av > bv) ? av + log1pf(-expf(bv - av)) + g : -INFINITY;
          } else if (job.kind == kResidualOneHot) {
            kr = (v == job.d) ? -INFINITY : kp;
          } else {
            kr = kp;
          }
          const unsigned long long keyr = argmax_key(kr, static_cast<uint32_t>(v));
          const unsigned long long keyp = argmax_key(kp, static_cast<uint32_t>(v));
          best_r = keyr > best_r ? keyr : best_r;
          best_p = keyp > best_p ? keyp : best_p;
        }
      }
    }
  }
  best_r = warp_max_u64(best_r);
  best_p = warp_max_u64(best_p);
  if (lane == 0) {
    red_r[warp] = best_r;
    red_p[warp] = best_p;
  }
  __syncthreads();
  if (tid == 0) {
    unsigned long long br = red_r[0], bp = red_p[0];
    for (int w2 = 1; w2 < kWarps; ++w2) {
      br = red_r[w2] > br ? red_r[w2] : br;
      bp = red_p[w2] > bp ? red_p[w2] : bp;
    }
    a.sparts[static_cast<long long>(b) * a.ndraw + slice] = SamplePartial{br, bp};
  }
}

// Warp 0 of a request's last CTA: merges the draw partials and stores the results.
__device__ void finish_draw(const DrawArgs &a, const SampleJob &job, int b) {
  const int lane = threadIdx.x & 31;
  const SamplePartial *sp = a.sparts + static_cast<long long>(b) * a.ndraw;
  unsigned long long br = 0ull, bp = 0ull;
  for (int c = lane; c < a.ndraw; c += 32) {
    const ulonglong2 raw = __ldcg(reinterpret_cast<const ulonglong2 *>(sp + c));
    br = raw.x > br ? raw.x : br;
    bp = raw.y > bp ? raw.y : bp;
  }
  br = warp_max_u64(br);
  bp = warp_max_u64(bp);
  if (lane == 0) {
    // The residual is empty only if p <= q everywhere (then draw from p).
    const float vr = key_value(br);
    const bool has_r = br != 0ull && vr != -INFINITY && vr == vr;
    a.next_token[b] = static_cast<int32_t>(key_index(has_r ? br : bp));
    a.accepted_len[b] = job.acc_len;
  }
}

template <int NB>
__global__ void __launch_bounds__(kThreads) verify_draw_kernel(const DrawArgs a) {
  __shared__ unsigned long long red_r[kWarps], red_p[kWarps];
  __shared__ SampleJob job_s;
  __shared__ int flag_s;
  const int slice = static_cast<int>(blockIdx.x % static_cast<unsigned>(a.ndraw));
  const int b = static_cast<int>(blockIdx.x / static_cast<unsigned>(a.ndraw));
  pdl_wait();
  if (threadIdx.x < 32) decide_request(a, b, &job_s, slice == 0);
  __syncthreads();
  const SampleJob job = job_s;
  draw_slice<NB>(a, job, b, slice, red_r, red_p);
  pdl_release();
  if (!last_arrival(a.tickets + b, a.ndraw, &flag_s)) return;
  if (threadIdx.x < 32) finish_draw(a, job, b);
}

// Greedy: one warp per request; lane j compares draft j with the target argmax of
// row j.  accepted_len = first mismatch (draft_len if none), next = argmax of that row.
__global__ void __launch_bounds__(kThreads) verify_greedy_kernel(const DrawArgs a) {
  const int lane = threadIdx.x & 31;
  const int b = blockIdx.x * kWarps + (threadIdx.x >> 5);
  pdl_wait();
  pdl_release();
  if (b >= a.B) return;
  const int k = a.k;
  const int L = clamp_len(a.draft_len, b, k, a.status);
  const long long trow = static_cast<long long>(b) * (k + 1);
  const int t = lane <= L ? a.t_arg[trow + lane] : -1;
  const bool miss = lane < L && a.drafts[static_cast<long long>(b) * k + lane] != t;
  const unsigned m = __ballot_sync(0xffffffffu, miss);
  const int acc = m ? __ffs(m) - 1 : L;
  const int next = __shfl_sync(0xffffffffu, t, acc & 31);
  if (lane == 0) {
    a.accepted_len[b] = acc;
    a.next_token[b] = next;
  }
}

int nslices_of(int V) { return (V + kSlice - 1) / kSlice; }
int ndraw_of(int V) { return (V + kDrawSlice - 1) / kDrawSlice; }

bool rows_vec(const float *p, int V) { return (V & 3) == 0 && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

RowSet row_set(const float *rows, long long nrows, int V, float *ms, int32_t *argmax,
               RowPartial *parts, int *tickets, const int32_t *len, int group, int len_off) {
  RowSet r;
  r.rows = rows;
  r.ms = ms;
  r.argmax = argmax;
  r.parts = parts;
  r.tickets = tickets;
  r.len = len;
  r.group = group;
  r.len_off = len_off;
  r.nrows = nrows;
  r.vec = rows_vec(rows, V) ? 1 : 0;
  return r;
}

// One launch over one or two row sets (n = 1 or 2).
dspark_status_t launch_row_stats(const RowSet *sets, int n, int V, int k, bool sums,
                                 cudaStream_t stream) {
  RowStatsArgs a;
  a.set[0] = sets[0];
  a.set[1] = n > 1 ? sets[1] : sets[0];
  a.k = k;
  a.V = V;
  a.nslices = nslices_of(V);
  a.blocks0 = sets[0].nrows * a.nslices;
  // 16384 entries (64 KB) per CTA: each CTA's fixed cost (scheduling, reduction,
  // ticket) is spread over 64 loads in flight per thread.
  const long long g = a.blocks0 + (n > 1 ? sets[1].nrows * a.nslices : 0);
  if (g > 0x7fffffffLL) return DSPARK_ERR_UNSUPPORTED_SHAPE;
  const cudaError_t e =
      sums ? launch_pdl(row_stats_kernel<kPer, true>, dim3(static_cast<unsigned>(g)), dim3(kThreads), 0, stream, a)
           : launch_pdl(row_stats_kernel<kPer, false>, dim3(static_cast<unsigned>(g)), dim3(kThreads), 0, stream, a);
  if (e != cudaSuccess) return DSPARK_ERR_CUDA;
  count_launches(1);
  return DSPARK_OK;
}

dspark_status_t launch_decision(const DrawArgs &a, int mode, cudaStream_t stream) {
  if (mode == 0) {
    if (launch_pdl(verify_greedy_kernel, dim3((a.B + kWarps - 1) / kWarps), dim3(kThreads), 0, stream,
                   a) != cudaSuccess)
      return DSPARK_ERR_CUDA;
  } else {
    // Philox blocks per thread: 1 while the grid stays within about four CTAs per SM,
    // else 2 or 4 (fewer CTAs, each with its decision taken once, at larger batches)
    const int sms = device_sm_count() > 0 ? device_sm_count() : 1;
    DrawArgs d = a;
    int nb = 1;
    while (nb < 4 && static_cast<long long>(a.B) * ((a.V + kDrawSlice * nb - 1) / (kDrawSlice * nb)) > 4LL * sms)
      nb *= 2;
    d.ndraw = (a.V + kDrawSlice * nb - 1) / (kDrawSlice * nb);
    const long long g = static_cast<long long>(a.B) * d.ndraw;
    if (g > 0x7fffffffLL) return DSPARK_ERR_UNSUPPORTED_SHAPE;
    cudaError_t e;
    if (nb == 1)
      e = launch_pdl(verify_draw_kernel<1>, dim3(static_cast<unsigned>(g)), dim3(kThreads), 0, stream, d);
    else if (nb == 2)
      e = launch_pdl(verify_draw_kernel<2>, dim3(static_cast<unsigned>(g)), dim3(kThreads), 0, stream, d);
    else
      e = launch_pdl(verify_draw_kernel<4>, dim3(static_cast<unsigned>(g)), dim3(kThreads), 0, stream, d);
    if (e != cudaSuccess) return DSPARK_ERR_CUDA;
  }
  count_launches(1);
  return DSPARK_OK;
}

// Workspace layouts (offsets from the start of the caller's workspace, whose first
// kWsAlign bytes hold the status word).
struct RowStatsLayout {
  size_t tickets, parts, total;
};

RowStatsLayout row_stats_layout(long long nrows, int V) {
  RowStatsLayout L;
  size_t off = kWsAlign;
  L.tickets = off;
  off += align_up(static_cast<size_t>(nrows) * sizeof(int), kWsAlign);
  L.parts = off;
  off += align_up(static_cast<size_t>(nrows) * nslices_of(V) * sizeof(RowPartial), kWsAlign);
  L.total = off;
  return L;
}

struct DrawLayout {
  size_t tickets, sparts, total;
};

DrawLayout draw_layout(int B, int V, size_t start) {
  DrawLayout L;
  size_t off = start;
  L.tickets = off;
  off += align_up(static_cast<size_t>(B) * sizeof(int), kWsAlign);
  L.sparts = off;
  off += align_up(static_cast<size_t>(B) * ndraw_of(V) * sizeof(SamplePartial), kWsAlign);
  L.total = off;
  return L;
}

// The whole verify in one workspace: [status | target-row tickets | draft-row tickets
// | draw tickets | target partials | draft partials | target (max, sum) | target
// argmax | draft (max, sum) | draw partials].
struct VerifyLayout {
  size_t t_tickets, z_tickets, d_tickets, t_parts, z_parts, t_ms, t_arg, q_ms, sparts, total;
};

VerifyLayout verify_layout(int B, int k, int V) {
  VerifyLayout L;
  const size_t tr = static_cast<size_t>(B) * (k + 1), zr = static_cast<size_t>(B) * k;
  const size_t ns = nslices_of(V);
  size_t off = kWsAlign;
  L.t_tickets = off;
  off += align_up(tr * sizeof(int), kWsAlign);
  L.z_tickets = off;
  off += align_up(zr * sizeof(int), kWsAlign);
  L.d_tickets = off;
  off += align_up(static_cast<size_t>(B) * sizeof(int), kWsAlign);
  L.t_parts = off;
  off += align_up(tr * ns * sizeof(RowPartial), kWsAlign);
  L.z_parts = off;
  off += align_up(zr * ns * sizeof(RowPartial), kWsAlign);
  L.t_ms = off;
  off += align_up(tr * 2 * sizeof(float), kWsAlign);
  L.t_arg = off;
  off += align_up(tr * sizeof(int32_t), kWsAlign);
  L.q_ms = off;
  off += align_up(zr * 2 * sizeof(float), kWsAlign);
  L.sparts = off;
  off += align_up(static_cast<size_t>(B) * ndraw_of(V) * sizeof(SamplePartial), kWsAlign);
  L.total = off;
  return L;
}

DrawArgs draw_args(int mode, const float *target, const float *t_ms, const int32_t *t_arg,
                   const int32_t *drafts, const int32_t *draft_len, const float *zlog,
                   const float *q_ms, uint64_t seed, const uint32_t *request_id, uint32_t step,
                   int32_t *accepted_len, int32_t *next_token, int B, int k, int V,
                   SamplePartial *sparts, int *tickets, int *status) {
  DrawArgs a;
  a.target = target;
  a.t_ms = t_ms;
  a.t_arg = t_arg;
  a.drafts = drafts;
  a.draft_len = draft_len;
  a.zlog = (mode == 1) ? zlog : nullptr;
  a.q_ms = q_ms;
  a.request_id = request_id;
  a.accepted_len = accepted_len;
  a.next_token = next_token;
  a.sparts = sparts;
  a.tickets = tickets;
  a.status = status;
  a.seed = seed;
  a.step = step;
  a.B = B;
  a.k = k;
  a.V = V;
  a.ndraw = ndraw_of(V);
  a.vec = (rows_vec(target, V) && (a.zlog == nullptr || rows_vec(a.zlog, V))) ? 1 : 0;
  return a;
}

}  // namespace

size_t row_stats_workspace_size(long long nrows, int V) { return row_stats_layout(nrows, V).total; }
size_t row_stats_counter_bytes(long long nrows, int V) { return row_stats_layout(nrows, V).parts; }

dspark_status_t row_stats_launch(const float *rows, long long nrows, int V, float *ms,
                                 int32_t *argmax, void *ws, int *status, cudaStream_t stream) {
  (void)status;
  const RowStatsLayout L = row_stats_layout(nrows, V);
  char *w = static_cast<char *>(ws);
  const RowSet rs = row_set(rows, nrows, V, ms, argmax, reinterpret_cast<RowPartial *>(w + L.parts),
                            reinterpret_cast<int *>(w + L.tickets), nullptr, 1, 0);
  return launch_row_stats(&rs, 1, V, 0, ms != nullptr, stream);
}

size_t verify_from_stats_workspace_size(int B, int V) { return draw_layout(B, V, kWsAlign).total; }
size_t verify_from_stats_counter_bytes(int B, int V) { return draw_layout(B, V, kWsAlign).sparts; }

dspark_status_t verify_from_stats_launch(int mode, const float *target, const float *t_ms,
                                         const int32_t *t_arg, const int32_t *drafts,
                                         const int32_t *draft_len, const float *zlog,
                                         const float *q_ms, uint64_t seed,
                                         const uint32_t *request_id, uint32_t step,
                                         int32_t *accepted_len, int32_t *next_token, int B, int k,
                                         int V, void *ws, int *status, cudaStream_t stream) {
  const DrawLayout L = draw_layout(B, V, kWsAlign);
  char *w = static_cast<char *>(ws);
  const DrawArgs a = draw_args(mode, target, t_ms, t_arg, drafts, draft_len, zlog, q_ms, seed,
                               request_id, step, accepted_len, next_token, B, k, V,
                               reinterpret_cast<SamplePartial *>(w + L.sparts),
                               reinterpret_cast<int *>(w + L.tickets), status);
  return launch_decision(a, mode, stream);
}

size_t verify_workspace_size(int B, int k, int V) { return verify_layout(B, k, V).total; }

size_t verify_counter_bytes(int B, int k, int V) { return verify_layout(B, k, V).t_parts; }

dspark_status_t verify_launch(int mode, const float *target, const int32_t *drafts,
                              const int32_t *draft_len, const float *zlog, const float *q_stats,
                              uint64_t seed, const uint32_t *request_id, uint32_t step,
                              int32_t *accepted_len, int32_t *next_token, int B, int k, int V,
                              void *ws, int *status, cudaStream_t stream) {
  const VerifyLayout L = verify_layout(B, k, V);
  char *w = static_cast<char *>(ws);
  float *t_ms = reinterpret_cast<float *>(w + L.t_ms);
  int32_t *t_arg = reinterpret_cast<int32_t *>(w + L.t_arg);
  // One launch over the target rows 0 .. draft_len of every request (greedy needs only
  // their argmax) and, when q's statistics are not given, the draft-logit rows
  // 0 .. draft_len - 1.
  RowSet sets[2];
  sets[0] = row_set(target, static_cast<long long>(B) * (k + 1), V, t_ms, t_arg,
                    reinterpret_cast<RowPartial *>(w + L.t_parts),
                    reinterpret_cast<int *>(w + L.t_tickets), draft_len, k + 1, 0);
  int nsets = 1;
  const float *q_ms = q_stats;
  if (mode == 1 && zlog != nullptr && q_stats == nullptr) {
    float *qw = reinterpret_cast<float *>(w + L.q_ms);
    sets[1] = row_set(zlog, static_cast<long long>(B) * k, V, qw, nullptr,
                      reinterpret_cast<RowPartial *>(w + L.z_parts),
                      reinterpret_cast<int *>(w + L.z_tickets), draft_len, k, -1);
    nsets = 2;
    q_ms = qw;
  }
  dspark_status_t st = launch_row_stats(sets, nsets, V, k, mode == 1, stream);
  if (st != DSPARK_OK) return st;
  const DrawArgs a = draw_args(mode, target, t_ms, t_arg, drafts, draft_len, zlog, q_ms, seed,
                               request_id, step, accepted_len, next_token, B, k, V,
                               reinterpret_cast<SamplePartial *>(w + L.sparts),
                               reinterpret_cast<int *>(w + L.d_tickets), status);
  return launch_decision(a, mode, stream);
}

}  // namespace dspark
