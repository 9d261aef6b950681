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
// Phase 1 (row statistics): one streaming read of every needed row (target
// rows 0..draft_len, and the draft-logit rows when their softmax statistics
// were not supplied) with 128-bit loads; each CTA reduces a 16384-entry slice to
// (argmax key, max, sum exp).
// Decision: the slices of a request are merged in a fixed order, then the
// accept/reject tests run with Philox uniforms.
// Phase 2 (draw, probabilistic only): the one row per request that needs a draw
// is re-read.  The draw is the Gumbel-max rule: the index maximising
// log w_v + G_v, G_v = -log(-log U_v) with U_v from Philox counter (request,
// row, step, 1 + v/4).  That samples exactly from w normalised and makes the
// draw an argmax, reduced like every other argmax here (per-CTA 64-bit keys,
// merged by the request's last CTA).
//
// verify_stats_kernel does phase 1 and its last CTA per request (atomic
// ticket, nobody waits) takes the decisions; verify_sample_kernel does phase 2
// and its last CTA per request merges the draw.
#include <cuda_runtime.h>
#include <math.h>

#include "common.cuh"
#include "internal.h"

namespace dspark {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kPer = 64;                    // entries per thread per slice (pass 1), all
                                            // loaded before any is used
constexpr int kSlice = kThreads * kPer;     // 16384 entries per CTA (pass 1)
constexpr int kDrawSlice = kThreads * 4;    // 1024 entries per CTA (pass 2): one Philox block per thread

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
  int pad;
  double cp;   // log-normaliser of the target row: max + log(sum exp)
  double cq;   // log-normaliser of the draft row (kResidual)
};

struct __align__(16) SamplePartial {
  unsigned long long best_r;  // argmax key of log w + G over the slice
  unsigned long long best_p;  // argmax key of log p + G (fallback: residual all zero)
};

struct VerifyArgs {
  const float *target;
  const int32_t *drafts;
  const int32_t *draft_len;
  const float *zlog;
  const float *q_stats;
  const uint32_t *request_id;
  int32_t *accepted_len;
  int32_t *next_token;
  RowPartial *rows;
  SampleJob *jobs;
  SamplePartial *sparts;
  int *req_ticket;
  int *samp_ticket;
  int *status;
  unsigned long long seed;
  unsigned int step;
  int mode;
  int B, k, V;
  int nslices;
  int ndraw;      // slices of the draw pass
  int zrows;      // 1 when draft-logit statistics are computed here
  int vec;        // 1 when every row starts on a 16-byte boundary (128-bit loads)
};

__device__ __forceinline__ int request_len(const VerifyArgs &a, int b, bool record) {
  int L = a.draft_len ? a.draft_len[b] : a.k;
  if (L < 0 || L > a.k) {
    if (record) record_error(a.status, DSPARK_ERR_INVALID_ARG);
    L = L < 0 ? 0 : a.k;
  }
  return L;
}

// ------------------------------------------------------------------ shared pieces

// Row index rho -> (request, block row, draft-logit row?).
struct RowRef {
  int b, j;
  bool is_z;
};

__device__ __forceinline__ RowRef row_ref(const VerifyArgs &a, int rho) {
  const int trows = a.B * (a.k + 1);
  RowRef r;
  r.is_z = rho >= trows;
  r.b = r.is_z ? (rho - trows) / a.k : rho / (a.k + 1);
  r.j = r.is_z ? (rho - trows) - r.b * a.k : rho - r.b * (a.k + 1);
  return r;
}

__device__ __forceinline__ bool row_needed(const VerifyArgs &a, const RowRef &r) {
  const int L = request_len(a, r.b, false);
  return r.is_z ? (a.mode == 1 && r.j < L) : (r.j <= L);
}

// (argmax key, max, sum exp) of one slice of row rho (KP entries per thread) -> rows
// partial.  Block-wide; `red` is shared scratch of kWarps entries.
template <int KP>
__device__ void stats_item(const VerifyArgs &a, int rho, int slice, RowPartial *red) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k = a.k, V = a.V;
  const RowRef rr = row_ref(a, rho);
  const bool want_stats = (a.mode == 1);
  const float *row = rr.is_z ? a.zlog + (static_cast<long long>(rr.b) * k + rr.j) * V
                             : a.target + (static_cast<long long>(rr.b) * (k + 1) + rr.j) * V;
  const int base = slice * (kThreads * KP);
  // This thread's KP entries, all loaded before any is used, in ascending index
  // order: the argmax by strict float compare (first index wins ties, -0 == +0, NaN
  // never wins), then the max and the sum of exp(x - max) from registers.  Entry e
  // has index base + (e/4)*1024 + 4*tid + e%4 (vector loads) or base + e*256 + tid.
  float x[KP];
  if (a.vec) {
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
  auto index_of = [&](int e) {
    return a.vec ? base + (e >> 2) * (kThreads * 4) + tid * 4 + (e & 3) : base + e * kThreads + tid;
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
  if (want_stats && bi >= 0 && bv != INFINITY) {
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
  if (want_stats) {
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
    a.rows[static_cast<long long>(rho) * a.nslices + slice] = acc;
  }
  __syncthreads();
}

// Decision state of one request, in shared memory.
struct Decision {
  unsigned long long tkey[kMaxK + 1];
  double tM[kMaxK + 1], tS[kMaxK + 1];
  double zM[kMaxK], zS[kMaxK];
  double ratio[kMaxK], ua[kMaxK];
  int bad[kMaxK];
  SampleJob job;
  int acc_len;
  int next;  // greedy: the next token
};

// Merges the row partials of request b and takes its decisions (block-wide).
// Greedy: acc_len and next.  Probabilistic: acc_len and the draw job.
__device__ void decide_request(const VerifyArgs &a, int b, Decision &d, bool record) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k = a.k, V = a.V;
  const int trows = a.B * (k + 1);
  const int L = request_len(a, b, record);
  const bool want_stats = (a.mode == 1);
  const int n_t = L + 1;
  const int n_z = a.zrows ? L : 0;
  // Loads that do not need the row statistics go first: each position's drafted
  // token and its target / draft logit (thread j takes position j).
  const long long drow = static_cast<long long>(b) * k;
  int pre_dt = -1;
  float pre_t = 0.0f, pre_z = 0.0f;
  if (a.mode == 1 && tid < L) {
    pre_dt = a.drafts[drow + tid];
    if (pre_dt >= 0 && pre_dt < V) {
      pre_t = a.target[(static_cast<long long>(b) * (k + 1) + tid) * V + pre_dt];
      if (a.zlog) pre_z = a.zlog[(drow + tid) * V + pre_dt];
    }
  }
  for (int q = warp; q < n_t + n_z; q += kWarps) {
    const bool qz = q >= n_t;
    const int jj = qz ? q - n_t : q;
    const int r_idx = qz ? trows + b * k + jj : b * (k + 1) + jj;
    const RowPartial *pr = a.rows + static_cast<long long>(r_idx) * a.nslices;
    // one pass: each lane merges its slices online (fp64 sums), then the warp
    unsigned long long kb = 0ull;
    float mm = -INFINITY;
    double s = 0.0;
    for (int c = lane; c < a.nslices; c += 32) {
      const ulonglong2 raw = __ldcg(reinterpret_cast<const ulonglong2 *>(pr + c));
      kb = raw.x > kb ? raw.x : kb;
      const float cm = __uint_as_float(static_cast<uint32_t>(raw.y));
      const float cs = __uint_as_float(static_cast<uint32_t>(raw.y >> 32));
      if (want_stats && cm != -INFINITY) {
        if (cm > mm) {
          s = (mm == -INFINITY) ? static_cast<double>(cs)
                                : s * static_cast<double>(expf(mm - cm)) + static_cast<double>(cs);
          mm = cm;
        } else {
          s += static_cast<double>(cs) * static_cast<double>(expf(cm - mm));
        }
      } else if (!want_stats) {
        mm = fmaxf(mm, cm);
      }
    }
    kb = warp_max_u64(kb);
    float wm = mm;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) wm = fmaxf(wm, __shfl_xor_sync(0xffffffffu, wm, o));
    if (want_stats) {
      s = (mm == -INFINITY) ? 0.0 : s * static_cast<double>(expf(mm - wm));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    }
    mm = wm;
    if (lane == 0) {
      if (qz) {
        d.zM[jj] = mm;
        d.zS[jj] = s;
      } else {
        d.tkey[jj] = kb;
        d.tM[jj] = mm;
        d.tS[jj] = s;
      }
    }
  }
  __syncthreads();

  // Probabilistic: every position's ratio p(d)/q(d) and accept uniform, in parallel
  // (thread j takes position j); the sequential accept loop below only compares.
  if (a.mode == 1 && tid < L) {
    const int jj = tid;
    const uint32_t req = a.request_id ? a.request_id[b] : static_cast<uint32_t>(b);
    const int dt = pre_dt;
    double ua, us;
    verify_uniforms(a.seed, req, static_cast<uint32_t>(jj), a.step, ua, us);
    d.ua[jj] = ua;
    d.bad[jj] = (dt < 0 || dt >= V) ? 1 : 0;
    double ratio = 0.0;
    if (!d.bad[jj]) {
      // p(d)/q(d) = exp((T_d - M) - (z_d - m)) * s / S: the exponent is formed
      // exactly in fp64, the exponential in fp32 (relative error ~1e-7)
      const double tT = pre_t;
      double ex = tT - d.tM[jj], sc = 1.0 / d.tS[jj];
      if (a.zlog) {
        const double qm = a.zrows ? d.zM[jj] : static_cast<double>(a.q_stats[2 * (drow + jj)]);
        const double qs = a.zrows ? d.zS[jj] : static_cast<double>(a.q_stats[2 * (drow + jj) + 1]);
        const double zd = pre_z;
        ex -= zd - qm;
        sc *= qs;
      }
      ratio = static_cast<double>(expf(static_cast<float>(ex))) * sc;
    }
    d.ratio[jj] = ratio;
  }
  __syncthreads();

  if (tid == 0) {
    int acc_len = 0;
    if (a.mode == 0) {
      while (acc_len < L &&
             a.drafts[drow + acc_len] == static_cast<int32_t>(key_index(d.tkey[acc_len])))
        ++acc_len;
      d.next = static_cast<int32_t>(key_index(d.tkey[acc_len]));
    } else {
      SampleJob job;
      job.kind = kNone;
      job.d = -1;
      job.pad = 0;
      job.cq = 0.0;
      for (; acc_len < L; ++acc_len) {
        const int jj = acc_len;
        if (d.bad[jj]) {
          if (record) record_error(a.status, DSPARK_ERR_BAD_TOKEN);
          job.row = jj;
          job.kind = kFromP;
          job.cp = d.tM[jj] + log(d.tS[jj]);
          break;
        }
        if (d.ua[jj] < d.ratio[jj]) continue;
        double qm = 0.0, qs = 1.0;
        if (a.zlog) {
          qm = a.zrows ? d.zM[jj] : static_cast<double>(a.q_stats[2 * (drow + jj)]);
          qs = a.zrows ? d.zS[jj] : static_cast<double>(a.q_stats[2 * (drow + jj) + 1]);
        }
        job.row = jj;
        job.kind = a.zlog ? kResidual : kResidualOneHot;
        job.d = a.drafts[drow + jj];
        job.cp = d.tM[jj] + log(d.tS[jj]);
        job.cq = qm + log(qs);
        break;
      }
      if (job.kind == kNone) {
        job.row = L;
        job.kind = kFromP;
        job.cp = d.tM[L] + log(d.tS[L]);
      }
      d.job = job;
    }
    d.acc_len = acc_len;
  }
  __syncthreads();
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

// Gumbel-max keys of one 1024-entry slice of the draw row of request b ->
// draw partial (block-wide).  `red_r`, `red_p` are shared scratch of kWarps.
__device__ void draw_item(const VerifyArgs &a, const SampleJob &job, int b, int slice,
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
  const int vg = slice * kDrawSlice + tid * 4;   // this thread's 4 entries: one Philox block
  if (vg < V) {
    const U4 w = philox4x32_10(U4{req, static_cast<uint32_t>(job.row), a.step,
                                  1u + static_cast<uint32_t>(vg >> 2)},
                               k0, k1);
    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
    float tv[4], zv[4];
    if (a.vec && vg + 4 <= V) {
      const float4 t4 = __ldcs(reinterpret_cast<const float4 *>(trow + vg));
      tv[0] = t4.x; tv[1] = t4.y; tv[2] = t4.z; tv[3] = t4.w;
      if (zrow) {
        const float4 z4 = __ldcs(reinterpret_cast<const float4 *>(zrow + vg));
        zv[0] = z4.x; zv[1] = z4.y; zv[2] = z4.z; zv[3] = z4.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        tv[e] = vg + e < V ? trow[vg + e] : 0.0f;
        zv[e] = (zrow && vg + e < V) ? zrow[vg + e] : 0.0f;
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int v = vg + e;
      if (v < V) {
        const float g = gumbel_from_word(words[e]);
        const float t = tv[e];
        const float kp = t + g;
        float kr;
        if (job.kind == kResidual) {
          const float av = t - cpf;
          const float bv = zv[e] - cqf;
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
  __syncthreads();
}

// Warp 0 merges the draw partials of request b and stores the next token.
__device__ void finish_draw(const VerifyArgs &a, int b) {
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
  }
}

// Atomic ticket of request b in `tickets`: true for the CTA that arrives last
// (of `count`), which then resets the ticket.  Block-wide.
// The CTA's partial was stored by thread 0; thread 0's ticket increment is an
// acquire-release atomic, so the partial is visible before the ticket moves, and the
// last CTA's thread 0 sees every other CTA's partial; the CTA barrier then orders the
// reads of the other threads after that acquire.  (A fence in every thread of every
// CTA cost about a microsecond per CTA wave.)
__device__ __forceinline__ bool last_arrival(int *tickets, int b, int count, int *flag_s) {
  if (threadIdx.x == 0) {
    int old;
    asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;" : "=r"(old) : "l"(tickets + b) : "memory");
    const bool last = (old == count - 1);
    if (last) tickets[b] = 0;
    *flag_s = last ? 1 : 0;
  }
  __syncthreads();
  const bool last = *flag_s != 0;
  if (last) __threadfence();  // the last CTA only: its threads read the others' partials
  return last;
}

// ------------------------------------------------------------------ two-launch path
__global__ void __launch_bounds__(kThreads) verify_stats_kernel(const VerifyArgs a) {
  __shared__ RowPartial red[kWarps];
  __shared__ int flag_s;
  __shared__ Decision dec;
  // 1-D grid (rows can exceed the 65535 limit of gridDim.y): block = row * nslices + slice
  const int slice = static_cast<int>(blockIdx.x % static_cast<unsigned>(a.nslices));
  const int rho = static_cast<int>(blockIdx.x / static_cast<unsigned>(a.nslices));
  const RowRef rr = row_ref(a, rho);
  pdl_wait();
  if (row_needed(a, rr)) stats_item<kPer>(a, rho, slice, red);
  pdl_release();  // after this CTA's pass: the grid may span many waves
  const int rows_per_req = (a.k + 1) + (a.zrows ? a.k : 0);
  if (!last_arrival(a.req_ticket, rr.b, rows_per_req * a.nslices, &flag_s)) return;
  decide_request(a, rr.b, dec, true);
  if (threadIdx.x == 0) {
    a.accepted_len[rr.b] = dec.acc_len;
    if (a.mode == 0)
      a.next_token[rr.b] = dec.next;
    else
      a.jobs[rr.b] = dec.job;
  }
}

__global__ void __launch_bounds__(kThreads) verify_sample_kernel(const VerifyArgs a) {
  __shared__ unsigned long long red_r[kWarps], red_p[kWarps];
  __shared__ int flag_s;
  const int slice = static_cast<int>(blockIdx.x % static_cast<unsigned>(a.ndraw));
  const int b = static_cast<int>(blockIdx.x / static_cast<unsigned>(a.ndraw));
  pdl_wait();
  const SampleJob job = a.jobs[b];
  draw_item(a, job, b, slice, red_r, red_p);
  pdl_release();
  if (!last_arrival(a.samp_ticket, b, a.ndraw, &flag_s)) return;
  if (threadIdx.x < 32) finish_draw(a, b);
}

struct VerifyLayout {
  size_t req_ticket, samp_ticket, rows, jobs, sparts, total;
  int nslices, ndraw;
};

VerifyLayout layout(int B, int k, int V) {
  VerifyLayout L;
  L.nslices = (V + kSlice - 1) / kSlice;
  L.ndraw = (V + kDrawSlice - 1) / kDrawSlice;
  size_t off = kWsAlign;
  L.req_ticket = off;
  off += align_up(static_cast<size_t>(B) * sizeof(int), kWsAlign);
  L.samp_ticket = off;
  off += align_up(static_cast<size_t>(B) * sizeof(int), kWsAlign);
  L.rows = off;
  off += align_up(static_cast<size_t>(B) * (2 * k + 1) * L.nslices * sizeof(RowPartial), kWsAlign);
  L.jobs = off;
  off += align_up(static_cast<size_t>(B) * sizeof(SampleJob), kWsAlign);
  L.sparts = off;
  off += align_up(static_cast<size_t>(B) * L.ndraw * sizeof(SamplePartial), kWsAlign);
  L.total = off;
  return L;
}

}  // namespace

size_t verify_workspace_size(int B, int k, int V) { return layout(B, k, V).total; }

size_t verify_counter_bytes(int B, int k, int V) { return layout(B, k, V).rows; }

dspark_status_t verify_launch(int mode, const float *target, const int32_t *drafts,
                              const int32_t *draft_len, const float *zlog, const float *q_stats,
                              uint64_t seed, const uint32_t *request_id, uint32_t step,
                              int32_t *accepted_len, int32_t *next_token, int B, int k, int V,
                              void *ws, int *status, cudaStream_t stream) {
  const VerifyLayout L = layout(B, k, V);
  char *w = static_cast<char *>(ws);
  VerifyArgs a;
  a.target = target;
  a.drafts = drafts;
  a.draft_len = draft_len;
  a.zlog = (mode == 1) ? zlog : nullptr;
  a.q_stats = q_stats;
  a.request_id = request_id;
  a.accepted_len = accepted_len;
  a.next_token = next_token;
  a.rows = reinterpret_cast<RowPartial *>(w + L.rows);
  a.jobs = reinterpret_cast<SampleJob *>(w + L.jobs);
  a.sparts = reinterpret_cast<SamplePartial *>(w + L.sparts);
  a.req_ticket = reinterpret_cast<int *>(w + L.req_ticket);
  a.samp_ticket = reinterpret_cast<int *>(w + L.samp_ticket);
  a.status = status;
  a.seed = seed;
  a.step = step;
  a.mode = mode;
  a.B = B;
  a.k = k;
  a.V = V;
  a.nslices = L.nslices;
  a.ndraw = L.ndraw;
  a.zrows = (mode == 1 && zlog != nullptr && q_stats == nullptr) ? 1 : 0;
  a.vec = ((V & 3) == 0 && (reinterpret_cast<uintptr_t>(target) & 15u) == 0 &&
           (a.zlog == nullptr || (reinterpret_cast<uintptr_t>(a.zlog) & 15u) == 0))
              ? 1
              : 0;
  const long long nrows = static_cast<long long>(B) * (k + 1) + (a.zrows ? static_cast<long long>(B) * k : 0);
  // 16384 entries (64 KB) per CTA: each CTA's fixed cost (scheduling, reduction,
  // ticket) is spread over 64 loads in flight per thread; at batch 1 the 27B rows
  // make one wave of CTAs.
  const long long g1 = nrows * a.nslices;
  if (launch_pdl(verify_stats_kernel, dim3(static_cast<unsigned>(g1)), dim3(kThreads), 0, stream, a) !=
      cudaSuccess)
    return DSPARK_ERR_CUDA;
  count_launches(1);
  if (mode == 1) {
    const long long g2 = static_cast<long long>(B) * L.ndraw;
    if (g2 > 0x7fffffffLL) return DSPARK_ERR_UNSUPPORTED_SHAPE;
    if (launch_pdl(verify_sample_kernel, dim3(static_cast<unsigned>(g2)), dim3(kThreads), 0, stream,
                   a) != cudaSuccess)
      return DSPARK_ERR_CUDA;
    count_launches(1);
  }
  return DSPARK_OK;
}

}  // namespace dspark
