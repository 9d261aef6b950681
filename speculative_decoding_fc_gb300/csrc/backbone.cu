// Drafter backbone kernels: the Qwen3-form decoder layers that run the draft block
// (the anchor token and k mask tokens) over the fc'd context before the LM head
// ([PR620] DSparkDraftModel(DFlashQwen3ForCausalLM), "the DFlash backbone"; [CARD]
// config fields layer_types, head_dim, mask_token_id; the forward pass itself is a
// reading, see norm_rows_kernel .. silu_mul_kernel below).  The projections are the
// library's tcgen05 GEMM (dspark_linear); these kernels are the memory- and
// latency-bound pieces between them:
//   * norm_rows_kernel: RMSNorm of rows, after a residual add (x += delta), after an
//     embedding gather (x = table[token]) or of a plain bf16 input; bf16 output,
//     optionally leaving out the first row of every group (the block's anchor).
//   * qk_norm_rope_kernel: per-head RMSNorm of q and k, NeoX rotary embedding at each
//     row's position, q to its buffer and k, v to the key/value cache.
//   * attention_kernel + attention_merge_kernel: grouped-query attention of the block
//     rows over the cache, split over 64-key slices (one CTA per request, kv head and
//     slice), then one warp per query row combining the slices.
//   * silu_mul_kernel: act = silu(gate) * up.
// All arithmetic fp32, bf16 stores rounded to nearest even.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace dspark {
namespace {

constexpr int kNormThreads = 256;
constexpr int kNormMaxChunks = 4;     // 16-byte chunks per thread: H <= 8 * 256 * 4
constexpr int kHeadDim = 128;
constexpr int kAttnKeys = 64;         // keys per attention CTA
constexpr int kAttnThreads = 256;
constexpr float kNormEps = 1e-6f;

__device__ __forceinline__ uint16_t f2bf(float x) { return __bfloat16_as_ushort(__float2bfloat16_rn(x)); }
__device__ __forceinline__ float bf2f(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }

__device__ __forceinline__ void unpack8(const uint4 &c, float (&v)[8]) {
  v[0] = bf16_lo(c.x); v[1] = bf16_hi(c.x); v[2] = bf16_lo(c.y); v[3] = bf16_hi(c.y);
  v[4] = bf16_lo(c.z); v[5] = bf16_hi(c.z); v[6] = bf16_lo(c.w); v[7] = bf16_hi(c.w);
}

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  return static_cast<uint32_t>(f2bf(lo)) | (static_cast<uint32_t>(f2bf(hi)) << 16);
}

// ------------------------------------------------------------------ RMSNorm rows
struct NormArgs {
  float *x;                  // fp32 residual rows [rows, H] (updated), or null
  const uint16_t *delta;     // bf16 rows added to x first (null: none)
  int64_t ld_delta;
  const uint16_t *table;     // bf16 [V, H]: x = table[token] (null: none)
  const int32_t *tok;
  int V;
  const uint16_t *in;        // bf16 input rows when x is null
  int64_t ld_in;
  const uint16_t *w;         // [H] norm weight
  uint16_t *out;             // bf16 output rows
  int64_t ld_out;
  int group;                 // > 0: the first row of each group of `group` rows is not written
  int rows, H;
  int *status;
};

// out = bf16(v / sqrt(mean(v^2) + eps) * w) of the row's values v (after the add or
// gather, which also land in x).  One CTA per row; each thread keeps its (at most 4)
// 16-byte chunks in registers between the sum of squares and the output.
__global__ void __launch_bounds__(kNormThreads) norm_rows_kernel(const NormArgs a) {
  __shared__ float red[kNormThreads / 32];
  pdl_wait();
  pdl_release();
  const int row = blockIdx.x;
  const int H = a.H, nc = H / 8;
  const int tid = threadIdx.x;
  float v[kNormMaxChunks][8];
  float ss = 0.0f;
  int tok = 0;
  if (a.table) {
    tok = a.tok[row];
    if (tok < 0 || tok >= a.V) {
      if (tid == 0) record_error(a.status, DSPARK_ERR_BAD_TOKEN);
      tok = tok < 0 ? 0 : a.V - 1;
    }
  }
#pragma unroll
  for (int u = 0; u < kNormMaxChunks; ++u) {
    const int c = tid + u * kNormThreads;
    if (c >= nc) break;
    if (a.x) {
      float4 *xp = reinterpret_cast<float4 *>(a.x + static_cast<int64_t>(row) * H) + 2 * c;
      if (a.table) {
        unpack8(*reinterpret_cast<const uint4 *>(a.table + static_cast<int64_t>(tok) * H + 8 * c), v[u]);
      } else {
        const float4 x0 = xp[0], x1 = xp[1];
        v[u][0] = x0.x; v[u][1] = x0.y; v[u][2] = x0.z; v[u][3] = x0.w;
        v[u][4] = x1.x; v[u][5] = x1.y; v[u][6] = x1.z; v[u][7] = x1.w;
        if (a.delta) {
          float d[8];
          unpack8(*reinterpret_cast<const uint4 *>(a.delta + static_cast<int64_t>(row) * a.ld_delta + 8 * c), d);
#pragma unroll
          for (int i = 0; i < 8; ++i) v[u][i] = __fadd_rn(v[u][i], d[i]);
        }
      }
      xp[0] = make_float4(v[u][0], v[u][1], v[u][2], v[u][3]);
      xp[1] = make_float4(v[u][4], v[u][5], v[u][6], v[u][7]);
    } else {
      unpack8(*reinterpret_cast<const uint4 *>(a.in + static_cast<int64_t>(row) * a.ld_in + 8 * c), v[u]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) ss = __fmaf_rn(v[u][i], v[u][i], ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((tid & 31) == 0) red[tid >> 5] = ss;
  __syncthreads();
  float tot = 0.0f;
#pragma unroll
  for (int w = 0; w < kNormThreads / 32; ++w) tot += red[w];
  const float inv = 1.0f / sqrtf(tot / static_cast<float>(H) + kNormEps);

  int orow = row;
  if (a.group > 0) {
    const int i = row % a.group;
    if (i == 0) return;
    orow = (row / a.group) * (a.group - 1) + i - 1;
  }
#pragma unroll
  for (int u = 0; u < kNormMaxChunks; ++u) {
    const int c = tid + u * kNormThreads;
    if (c >= nc) break;
    float wv[8];
    unpack8(*reinterpret_cast<const uint4 *>(a.w + 8 * c), wv);
    uint4 o;
    o.x = pack2(v[u][0] * inv * wv[0], v[u][1] * inv * wv[1]);
    o.y = pack2(v[u][2] * inv * wv[2], v[u][3] * inv * wv[3]);
    o.z = pack2(v[u][4] * inv * wv[4], v[u][5] * inv * wv[5]);
    o.w = pack2(v[u][6] * inv * wv[6], v[u][7] * inv * wv[7]);
    *reinterpret_cast<uint4 *>(a.out + static_cast<int64_t>(orow) * a.ld_out + 8 * c) = o;
  }
}

// ------------------------------------------------------------------ q/k norm + rotary
struct RopeArgs {
  const uint16_t *qkv;       // rows [rows, ld]: [q heads (nq > 0) | k heads | v heads] x 128
  int64_t ld;
  int nq, nkv;
  const uint16_t *wq, *wk;   // [128] per-head norm weights
  uint16_t *q_out;           // [rows, nq, 128]
  uint16_t *k_cache, *v_cache;  // [B, cache_len, nkv, 128]
  int cache_len, rows_per_req, pos0, rows;
  double log2_theta;
};

// One warp per (row, head), 4 dims per lane (lanes 0-15 the first half of the head,
// 16-31 the second, so the rotary partner of a lane's dims is lane ^ 16).
__global__ void __launch_bounds__(256) qk_norm_rope_kernel(const RopeArgs a) {
  // the inverse frequencies theta^(-2d/128) in fp64, once per CTA
  __shared__ double inv_freq[kHeadDim / 2];
  if (threadIdx.x < kHeadDim / 2)
    inv_freq[threadIdx.x] = exp2(-(2.0 * threadIdx.x / kHeadDim) * a.log2_theta);
  __syncthreads();
  pdl_wait();
  pdl_release();
  const int nh = a.nq + 2 * a.nkv;
  const long long wid = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (wid >= static_cast<long long>(a.rows) * nh) return;
  const int lane = threadIdx.x & 31;
  const int row = static_cast<int>(wid / nh), h = static_cast<int>(wid % nh);
  const int b = row / a.rows_per_req;
  const int pos = a.pos0 + row % a.rows_per_req;
  const uint2 raw = *reinterpret_cast<const uint2 *>(a.qkv + static_cast<int64_t>(row) * a.ld + h * kHeadDim + 4 * lane);
  if (h >= a.nq + a.nkv) {  // value head: to the cache as it is
    const int g = h - a.nq - a.nkv;
    *reinterpret_cast<uint2 *>(a.v_cache + ((static_cast<int64_t>(b) * a.cache_len + pos) * a.nkv + g) * kHeadDim +
                               4 * lane) = raw;
    return;
  }
  float x[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
  float ss = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) ss = __fmaf_rn(x[i], x[i], ss);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float inv = 1.0f / sqrtf(ss / static_cast<float>(kHeadDim) + kNormEps);
  const uint16_t *w = h < a.nq ? a.wq : a.wk;
  const uint2 wr = *reinterpret_cast<const uint2 *>(w + 4 * lane);
  const float wv[4] = {bf16_lo(wr.x), bf16_hi(wr.x), bf16_lo(wr.y), bf16_hi(wr.y)};
  float y[4], r[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) y[i] = x[i] * inv * wv[i];
  const bool second = lane >= 16;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float other = __shfl_xor_sync(0xffffffffu, y[i], 16);
    const int d = (lane & 15) * 4 + i;  // frequency index 0..63
    // the angle in fp64, reduced to [0, 2 pi) before the fp32 sine and cosine (an fp32
    // angle of ~1000 rad would carry an error of ~1e-4 rad)
    const double ang = static_cast<double>(pos) * inv_freq[d];
    const double two_pi = 6.283185307179586;
    float s, c;
    sincosf(static_cast<float>(ang - two_pi * floor(ang / two_pi)), &s, &c);
    r[i] = second ? (y[i] * c + other * s) : (y[i] * c - other * s);
  }
  uint2 o;
  o.x = pack2(r[0], r[1]);
  o.y = pack2(r[2], r[3]);
  if (h < a.nq) {
    *reinterpret_cast<uint2 *>(a.q_out + (static_cast<int64_t>(row) * a.nq + h) * kHeadDim + 4 * lane) = o;
  } else {
    const int g = h - a.nq;
    *reinterpret_cast<uint2 *>(a.k_cache + ((static_cast<int64_t>(b) * a.cache_len + pos) * a.nkv + g) * kHeadDim +
                               4 * lane) = o;
  }
}

// ------------------------------------------------------------------ attention
struct AttnArgs {
  const uint16_t *q;         // [B, nr, nq, 128]
  const uint16_t *k_cache, *v_cache;  // [B, cache_len, nkv, 128]
  float *part_o;             // [B, nkv, nsplit, nqry, 128]
  float *part_ml;            // [B, nkv, nsplit, nqry, 2]
  uint16_t *out;             // [B, nr, nq, 128]
  int B, nr, nq, nkv, cache_len, nkeys, nsplit, nqry;
  float scale;
};

// CTA (split s, kv head g, request b): keys s*64 .. s*64+63 (those below nkeys) for
// the nqry = nr * (nq / nkv) query rows of the group (query qi = block row
// qi / grp, head g * grp + qi % grp).  Scores by one key per lane (the key row in
// registers, the scaled queries in shared memory), softmax per query row over the
// slice (its max and sum kept for the merge), then P.V with 4 dims per lane.
__global__ void __launch_bounds__(kAttnThreads) attention_kernel(const AttnArgs a) {
  extern __shared__ __align__(16) float attn_smem[];
  const int nqry = a.nqry;
  uint16_t *vs = reinterpret_cast<uint16_t *>(attn_smem);              // [64][128] bf16
  float *qs = attn_smem + kAttnKeys * kHeadDim / 2;                    // [nqry][128]
  float *sc = qs + nqry * kHeadDim;             // [nqry][64]
  float *ml = sc + nqry * kAttnKeys;            // [nqry][2]
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int grp = a.nq / a.nkv;
  const int kend = min(kAttnKeys, a.nkeys - split * kAttnKeys);
  pdl_wait();
  pdl_release();
  // the slice's value rows into shared memory, in flight while the scores are computed
  for (int e = tid; e < kend * (kHeadDim / 8); e += kAttnThreads) {
    const int kl = e / (kHeadDim / 8), c = e % (kHeadDim / 8);
    const uint16_t *src =
        a.v_cache + ((static_cast<int64_t>(b) * a.cache_len + split * kAttnKeys + kl) * a.nkv + g) * kHeadDim + 8 * c;
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(
                     __cvta_generic_to_shared(vs + kl * kHeadDim + 8 * c))),
                 "l"(src)
                 : "memory");
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  for (int e = tid; e < nqry * (kHeadDim / 8); e += kAttnThreads) {
    const int qi = e / (kHeadDim / 8), c = e % (kHeadDim / 8);
    const int i = qi / grp, head = g * grp + qi % grp;
    float v[8];
    unpack8(*reinterpret_cast<const uint4 *>(a.q + ((static_cast<int64_t>(b) * a.nr + i) * a.nq + head) * kHeadDim + 8 * c), v);
#pragma unroll
    for (int t = 0; t < 8; ++t) qs[qi * kHeadDim + 8 * c + t] = v[t] * a.scale;
  }
  __syncthreads();

  // scores: warp w takes keys 32 * (w & 1) + lane and query rows of quarter w >> 1
  {
    const int kl = 32 * (warp & 1) + lane;
    const int key = split * kAttnKeys + kl;
    const bool valid = key < a.nkeys;
    const int qpw = (nqry + 3) / 4;
    const int q0 = (warp >> 1) * qpw, q1 = min(nqry, q0 + qpw);
    uint4 kr[kHeadDim / 8];
    const uint4 *kp = reinterpret_cast<const uint4 *>(
        a.k_cache + ((static_cast<int64_t>(b) * a.cache_len + (valid ? key : 0)) * a.nkv + g) * kHeadDim);
#pragma unroll
    for (int c = 0; c < kHeadDim / 8; ++c) kr[c] = valid ? kp[c] : make_uint4(0u, 0u, 0u, 0u);
    for (int qi = q0; qi < q1; ++qi) {
      const float4 *qv = reinterpret_cast<const float4 *>(qs + qi * kHeadDim);
      float s = 0.0f;
#pragma unroll
      for (int c = 0; c < kHeadDim / 8; ++c) {
        float kv[8];
        unpack8(kr[c], kv);
        const float4 qa = qv[2 * c], qb = qv[2 * c + 1];
        s = __fmaf_rn(qa.x, kv[0], s); s = __fmaf_rn(qa.y, kv[1], s);
        s = __fmaf_rn(qa.z, kv[2], s); s = __fmaf_rn(qa.w, kv[3], s);
        s = __fmaf_rn(qb.x, kv[4], s); s = __fmaf_rn(qb.y, kv[5], s);
        s = __fmaf_rn(qb.z, kv[6], s); s = __fmaf_rn(qb.w, kv[7], s);
      }
      sc[qi * kAttnKeys + kl] = valid ? s : -INFINITY;
    }
  }
  __syncthreads();

  // softmax over the slice per query row (two keys per lane)
  for (int qi = warp; qi < nqry; qi += kAttnThreads / 32) {
    const float s0 = sc[qi * kAttnKeys + lane], s1 = sc[qi * kAttnKeys + 32 + lane];
    float m = fmaxf(s0, s1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float p0 = m == -INFINITY ? 0.0f : expf(s0 - m);
    const float p1 = m == -INFINITY ? 0.0f : expf(s1 - m);
    float l = p0 + p1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    sc[qi * kAttnKeys + lane] = p0;
    sc[qi * kAttnKeys + 32 + lane] = p1;
    if (lane == 0) {
      ml[2 * qi] = m;
      ml[2 * qi + 1] = l;
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();

  // P.V: warp w takes query rows w, w + 8, ...; lane dims 4 * lane .. + 3
  constexpr int kRowsPerWarp = 8;  // nqry <= 64
  float acc[kRowsPerWarp][4];
#pragma unroll
  for (int t = 0; t < kRowsPerWarp; ++t)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[t][i] = 0.0f;
#pragma unroll 4
  for (int kl = 0; kl < kend; ++kl) {
    const uint2 vr = *reinterpret_cast<const uint2 *>(vs + kl * kHeadDim + 4 * lane);
    const float v[4] = {bf16_lo(vr.x), bf16_hi(vr.x), bf16_lo(vr.y), bf16_hi(vr.y)};
#pragma unroll
    for (int t = 0; t < kRowsPerWarp; ++t) {
      const int qi = warp + 8 * t;
      if (qi < nqry) {
        const float p = sc[qi * kAttnKeys + kl];
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[t][i] = __fmaf_rn(p, v[i], acc[t][i]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kRowsPerWarp; ++t) {
    const int qi = warp + 8 * t;
    if (qi < nqry) {
      const int64_t base = ((static_cast<int64_t>(b) * a.nkv + g) * a.nsplit + split) * nqry + qi;
      *reinterpret_cast<float4 *>(a.part_o + base * kHeadDim + 4 * lane) =
          make_float4(acc[t][0], acc[t][1], acc[t][2], acc[t][3]);
      if (lane == 0) {
        a.part_ml[2 * base] = ml[2 * qi];
        a.part_ml[2 * base + 1] = ml[2 * qi + 1];
      }
    }
  }
}

// One warp per (request, kv head, query row): out = sum_s e^(m_s - M) o_s / sum_s e^(m_s - M) l_s.
__global__ void __launch_bounds__(256) attention_merge_kernel(const AttnArgs a) {
  pdl_wait();
  pdl_release();
  const long long wid = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  const long long total = static_cast<long long>(a.B) * a.nkv * a.nqry;
  if (wid >= total) return;
  const int lane = threadIdx.x & 31;
  const int qi = static_cast<int>(wid % a.nqry);
  const int g = static_cast<int>((wid / a.nqry) % a.nkv);
  const int b = static_cast<int>(wid / (static_cast<long long>(a.nqry) * a.nkv));
  const int grp = a.nq / a.nkv;
  const int64_t base0 = ((static_cast<int64_t>(b) * a.nkv + g) * a.nsplit) * a.nqry + qi;
  // the slices' maxima, one slice per lane
  float M = -INFINITY;
  for (int s = lane; s < a.nsplit; s += 32) M = fmaxf(M, a.part_ml[2 * (base0 + static_cast<int64_t>(s) * a.nqry)]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float o4[4] = {0.0f, 0.0f, 0.0f, 0.0f}, L = 0.0f;
  if (M != -INFINITY) {
    for (int s0 = 0; s0 < a.nsplit; s0 += 32) {
      // lane s0 + j: the weight e^(m - M) of slice s0 + j (0 for an empty slice)
      const int s = s0 + lane;
      float e = 0.0f;
      if (s < a.nsplit) {
        const int64_t base = base0 + static_cast<int64_t>(s) * a.nqry;
        const float m = a.part_ml[2 * base];
        if (m != -INFINITY) {
          e = expf(m - M);
          L = __fmaf_rn(e, a.part_ml[2 * base + 1], L);
        }
      }
      const int n = min(32, a.nsplit - s0);
#pragma unroll 4
      for (int j = 0; j < n; ++j) {
        const float ej = __shfl_sync(0xffffffffu, e, j);
        const float4 po = *reinterpret_cast<const float4 *>(
            a.part_o + (base0 + static_cast<int64_t>(s0 + j) * a.nqry) * kHeadDim + 4 * lane);
        o4[0] = __fmaf_rn(ej, po.x, o4[0]); o4[1] = __fmaf_rn(ej, po.y, o4[1]);
        o4[2] = __fmaf_rn(ej, po.z, o4[2]); o4[3] = __fmaf_rn(ej, po.w, o4[3]);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
  const float inv = L > 0.0f ? 1.0f / L : 0.0f;
  const int i = qi / grp, head = g * grp + qi % grp;
  uint2 r;
  r.x = pack2(o4[0] * inv, o4[1] * inv);
  r.y = pack2(o4[2] * inv, o4[3] * inv);
  *reinterpret_cast<uint2 *>(a.out + ((static_cast<int64_t>(b) * a.nr + i) * a.nq + head) * kHeadDim + 4 * lane) = r;
}

// ------------------------------------------------------------------ SiLU(gate) * up
// gu rows [M, 2I] = [gate | up]; act[m, c] = bf16(silu(g) * u), 8 entries per thread.
__global__ void __launch_bounds__(256) silu_mul_kernel(const uint16_t *gu, uint16_t *act, int M, int I) {
  pdl_wait();
  pdl_release();
  const long long n8 = static_cast<long long>(M) * (I / 8);
  for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < n8;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int m = static_cast<int>(e / (I / 8)), c = static_cast<int>(e % (I / 8));
    float gv[8], uv[8];
    unpack8(*reinterpret_cast<const uint4 *>(gu + static_cast<int64_t>(m) * 2 * I + 8 * c), gv);
    unpack8(*reinterpret_cast<const uint4 *>(gu + static_cast<int64_t>(m) * 2 * I + I + 8 * c), uv);
    float y[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) y[t] = gv[t] / (1.0f + expf(-gv[t])) * uv[t];
    uint4 o;
    o.x = pack2(y[0], y[1]);
    o.y = pack2(y[2], y[3]);
    o.z = pack2(y[4], y[5]);
    o.w = pack2(y[6], y[7]);
    *reinterpret_cast<uint4 *>(act + static_cast<int64_t>(m) * I + 8 * c) = o;
  }
}

}  // namespace

dspark_status_t norm_rows_launch(float *x, const uint16_t *delta, int64_t ld_delta, const uint16_t *table,
                                 const int32_t *tok, int V, const uint16_t *in, int64_t ld_in,
                                 const uint16_t *w, uint16_t *out, int64_t ld_out, int group, int rows,
                                 int H, int *status, cudaStream_t stream) {
  NormArgs a;
  a.x = x;
  a.delta = delta;
  a.ld_delta = ld_delta;
  a.table = table;
  a.tok = tok;
  a.V = V;
  a.in = in;
  a.ld_in = ld_in;
  a.w = w;
  a.out = out;
  a.ld_out = ld_out;
  a.group = group;
  a.rows = rows;
  a.H = H;
  a.status = status;
  if (launch_pdl(norm_rows_kernel, dim3(static_cast<unsigned>(rows)), dim3(kNormThreads), 0, stream, a) !=
      cudaSuccess)
    return DSPARK_ERR_CUDA;
  count_launches(1);
  return DSPARK_OK;
}

dspark_status_t qk_norm_rope_launch(const uint16_t *qkv, int64_t ld, int nq, int nkv, const uint16_t *wq,
                                    const uint16_t *wk, float theta, uint16_t *q_out, uint16_t *k_cache,
                                    uint16_t *v_cache, int cache_len, int rows_per_req, int pos0, int rows,
                                    cudaStream_t stream) {
  RopeArgs a;
  a.qkv = qkv;
  a.ld = ld;
  a.nq = nq;
  a.nkv = nkv;
  a.wq = wq;
  a.wk = wk;
  a.q_out = q_out;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.cache_len = cache_len;
  a.rows_per_req = rows_per_req;
  a.pos0 = pos0;
  a.rows = rows;
  a.log2_theta = log2(static_cast<double>(theta));
  const long long warps = static_cast<long long>(rows) * (nq + 2 * nkv);
  if (launch_pdl(qk_norm_rope_kernel, dim3(static_cast<unsigned>((warps + 7) / 8)), dim3(256), 0, stream, a) !=
      cudaSuccess)
    return DSPARK_ERR_CUDA;
  count_launches(1);
  return DSPARK_OK;
}

int attention_splits(int nkeys) { return (nkeys + kAttnKeys - 1) / kAttnKeys; }

size_t attention_workspace_bytes(int B, int nr, int nq, int nkv, int nkeys) {
  const size_t nqry = static_cast<size_t>(nr) * (nq / nkv);
  const size_t parts = static_cast<size_t>(B) * nkv * attention_splits(nkeys) * nqry;
  return align_up(parts * kHeadDim * sizeof(float), kWsAlign) + align_up(parts * 2 * sizeof(float), kWsAlign);
}

dspark_status_t attention_launch(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                                 uint16_t *out, int B, int nr, int nq, int nkv, int cache_len, int nkeys,
                                 void *ws, cudaStream_t stream) {
  AttnArgs a;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.out = out;
  a.B = B;
  a.nr = nr;
  a.nq = nq;
  a.nkv = nkv;
  a.cache_len = cache_len;
  a.nkeys = nkeys;
  a.nsplit = attention_splits(nkeys);
  a.nqry = nr * (nq / nkv);
  a.scale = static_cast<float>(1.0 / sqrt(static_cast<double>(kHeadDim)));
  const size_t parts = static_cast<size_t>(B) * nkv * a.nsplit * a.nqry;
  a.part_o = static_cast<float *>(ws);
  a.part_ml = reinterpret_cast<float *>(static_cast<char *>(ws) + align_up(parts * kHeadDim * sizeof(float), kWsAlign));
  const size_t smem = static_cast<size_t>(kAttnKeys) * kHeadDim * 2 +
                      static_cast<size_t>(a.nqry) * (kHeadDim + kAttnKeys + 2) * sizeof(float);
  static size_t attr_bytes[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DSPARK_ERR_CUDA;
  if (attr_bytes[dev] < smem) {
    if (cudaFuncSetAttribute(attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess)
      return DSPARK_ERR_CUDA;
    attr_bytes[dev] = smem;
  }
  if (launch_pdl(attention_kernel, dim3(static_cast<unsigned>(a.nsplit), static_cast<unsigned>(nkv),
                                        static_cast<unsigned>(B)),
                 dim3(kAttnThreads), smem, stream, a) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  const long long warps = static_cast<long long>(B) * nkv * a.nqry;
  if (launch_pdl(attention_merge_kernel, dim3(static_cast<unsigned>((warps + 7) / 8)), dim3(256), 0, stream, a) !=
      cudaSuccess)
    return DSPARK_ERR_CUDA;
  count_launches(2);
  return DSPARK_OK;
}

dspark_status_t silu_mul_launch(const uint16_t *gu, uint16_t *act, int M, int I, cudaStream_t stream) {
  const long long n8 = static_cast<long long>(M) * (I / 8);
  long long blocks = (n8 + 255) / 256;
  const long long cap = static_cast<long long>(device_sm_count() > 0 ? device_sm_count() : 1) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (launch_pdl(silu_mul_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, gu, act, M, I) !=
      cudaSuccess)
    return DSPARK_ERR_CUDA;
  count_launches(1);
  return DSPARK_OK;
}

}  // namespace dspark
