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

// ------------------------------------------------------------------ GEMM output pieces
// W consecutive outputs (m, n0 .. n0 + W - 1) of a GEMM that left its split tiles as
// pieces (PieceView; W divides 128 and n0): the bf16 values the GEMM's own fix-up
// would have stored (pieces added in CTA order from 0, rounded to bf16), as floats.
// The schedule's index arithmetic runs in 32 bits: the host uses a PieceView only when
// units * grid < 2^31.
template <int W>
__device__ __forceinline__ void view_vals(const PieceView &v, int m, int n0, float (&o)[W]) {
  const int n_tile = n0 / 128, m_tile = m / v.BN;
  const int tile = n_tile * v.tiles_m + m_tile;
  const uint32_t units = static_cast<uint32_t>(v.units), grid = static_cast<uint32_t>(v.grid);
  const uint32_t kbt = static_cast<uint32_t>(v.kb_total);
  const uint32_t t_first = static_cast<uint32_t>(tile) * kbt;
  const int c_first = static_cast<int>(((t_first + 1) * grid - 1) / units);
  const int c_last = static_cast<int>(((t_first + kbt) * grid - 1) / units);
  if (c_first == c_last) {  // the tile was stored whole
    const uint16_t *src = v.out + static_cast<int64_t>(m) * v.ldo + n0;
    if (W == 8) {
      float t[8];
      unpack8(*reinterpret_cast<const uint4 *>(src), t);
#pragma unroll
      for (int j = 0; j < W; ++j) o[j] = t[j];
    } else {
      const uint2 r = *reinterpret_cast<const uint2 *>(src);
      const float t[4] = {bf16_lo(r.x), bf16_hi(r.x), bf16_lo(r.y), bf16_hi(r.y)};
#pragma unroll
      for (int j = 0; j < W; ++j) o[j] = t[j];
    }
    return;
  }
  float acc[W];
#pragma unroll
  for (int j = 0; j < W; ++j) acc[j] = 0.0f;
  const int off = (m - m_tile * v.BN) * 128 + (n0 - n_tile * 128);
#pragma unroll 4
  for (int c = c_first; c <= c_last; ++c) {
    const int tile_c = static_cast<int>((units * static_cast<uint32_t>(c) / grid) / kbt);
    const float *src = v.partials + (static_cast<size_t>(c) * 2 + (tile == tile_c ? 0 : 1)) * v.BN * 128 + off;
#pragma unroll
    for (int j = 0; j < W; j += 4) {
      const float4 q = __ldcg(reinterpret_cast<const float4 *>(src + j));
      acc[j] += q.x;
      acc[j + 1] += q.y;
      acc[j + 2] += q.z;
      acc[j + 3] += q.w;
    }
  }
#pragma unroll
  for (int j = 0; j < W; ++j) o[j] = bf2f(f2bf(acc[j]));
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
  int rows, H;               // rows of the first part (the grid may add in2's rows)
  const uint16_t *in2;       // second part: plain bf16 rows (out rows rows, rows + 1, ...)
  int64_t ld_in2;
  int *status;
  int delta_view;            // the delta rows are rows 0 .. rows - 1 of dv (not `delta`)
  PieceView dv;
};

// out = bf16(v / sqrt(mean(v^2) + eps) * w) of the row's values v (after the add or
// gather, which also land in x).  One CTA per row; each thread keeps its (at most 4)
// 16-byte chunks in registers between the sum of squares and the output.  CTAs past
// the first part's rows norm the second part's plain rows (the context rows beside
// the block rows: one launch for both).
__global__ void __launch_bounds__(kNormThreads) norm_rows_kernel(const NormArgs a) {
  __shared__ float red[kNormThreads / 32];
  pdl_wait();
  pdl_release();
  const int row = blockIdx.x;
  const bool second = row >= a.rows;
  float *const xrow = (!second && a.x) ? a.x + static_cast<int64_t>(row) * a.H : nullptr;
  const uint16_t *const table = second ? nullptr : a.table;
  const uint16_t *const delta = second ? nullptr : a.delta;
  const bool dview = !second && a.delta_view;
  const uint16_t *const inrow = second ? a.in2 + static_cast<int64_t>(row - a.rows) * a.ld_in2
                                       : (a.in ? a.in + static_cast<int64_t>(row) * a.ld_in : nullptr);
  const int H = a.H, nc = H / 8;
  const int tid = threadIdx.x;
  float v[kNormMaxChunks][8];
  float ss = 0.0f;
  int tok = 0;
  if (table) {
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
    if (xrow) {
      float4 *xp = reinterpret_cast<float4 *>(xrow) + 2 * c;
      if (table) {
        unpack8(*reinterpret_cast<const uint4 *>(table + static_cast<int64_t>(tok) * H + 8 * c), v[u]);
      } else {
        const float4 x0 = xp[0], x1 = xp[1];
        v[u][0] = x0.x; v[u][1] = x0.y; v[u][2] = x0.z; v[u][3] = x0.w;
        v[u][4] = x1.x; v[u][5] = x1.y; v[u][6] = x1.z; v[u][7] = x1.w;
        if (dview) {
          float d[8];
          view_vals<8>(a.dv, row, 8 * c, d);
#pragma unroll
          for (int i = 0; i < 8; ++i) v[u][i] = __fadd_rn(v[u][i], d[i]);
        } else if (delta) {
          float d[8];
          unpack8(*reinterpret_cast<const uint4 *>(delta + static_cast<int64_t>(row) * a.ld_delta + 8 * c), d);
#pragma unroll
          for (int i = 0; i < 8; ++i) v[u][i] = __fadd_rn(v[u][i], d[i]);
        }
      }
      xp[0] = make_float4(v[u][0], v[u][1], v[u][2], v[u][3]);
      xp[1] = make_float4(v[u][4], v[u][5], v[u][6], v[u][7]);
    } else {
      unpack8(*reinterpret_cast<const uint4 *>(inrow + 8 * c), v[u]);
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
  if (a.group > 0 && !second) {
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
  // a second group of rows holding key and value heads only (the context rows beside
  // the block rows, one launch for both): [rows2, ld2] = [k heads | v heads] x 128
  const uint16_t *kv2;
  int64_t ld2;
  int rows_per_req2, pos02, rows2;
  int qkv_view;              // read rows (block rows, then the second group's) from qv
  PieceView qv;
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
  const long long n1 = static_cast<long long>(a.rows) * nh;
  const int lane = threadIdx.x & 31;
  int h, b, pos, row = 0, vrow = 0;
  const uint16_t *src;
  if (wid < n1) {
    row = static_cast<int>(wid / nh);
    h = static_cast<int>(wid % nh);
    b = row / a.rows_per_req;
    pos = a.pos0 + row % a.rows_per_req;
    src = a.qkv + static_cast<int64_t>(row) * a.ld + h * kHeadDim;
    vrow = row;
  } else {
    const long long w2 = wid - n1;
    if (w2 >= static_cast<long long>(a.rows2) * 2 * a.nkv) return;
    const int row2 = static_cast<int>(w2 / (2 * a.nkv)), h2 = static_cast<int>(w2 % (2 * a.nkv));
    h = a.nq + h2;   // a key or value head: no q row
    b = row2 / a.rows_per_req2;
    pos = a.pos02 + row2 % a.rows_per_req2;
    src = a.kv2 + static_cast<int64_t>(row2) * a.ld2 + h2 * kHeadDim;
    vrow = a.rows + row2;
  }
  uint2 raw;
  if (a.qkv_view) {   // the GEMM's pieces: column h * 128 + 4 lane of view row vrow
    float t[4];
    view_vals<4>(a.qv, vrow, h * kHeadDim + 4 * lane, t);
    raw.x = pack2(t[0], t[1]);
    raw.y = pack2(t[2], t[3]);
  } else {
    raw = *reinterpret_cast<const uint2 *>(src + 4 * lane);
  }
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
// the nqry = nr * (nq / nkv) query rows of the group (query qi = block row qi / grp,
// head g * grp + qi % grp).  The two contractions of a slice (scores 48 x 64 x 128,
// P.V 48 x 128 x 64 with the query rows padded to 48) are warp-level bf16 MMAs with
// fp32 accumulation (mma.sync m16n8k16; at this size an allocation of tensor memory
// and its descriptors would cost more than the products): scores from the bf16 q and
// k rows, scaled by 1/sqrt(128) after the sum; softmax per query row over the slice in
// fp32 (its max and sum kept for the merge); the weights p enter P.V as two bf16 parts
// hi = bf16(p), lo = bf16(p - hi) (p to about 2^-17 relative), the value rows exact.
constexpr int kAttnQPad = 48;                 // query rows per CTA (3 tiles of 16)
constexpr int kAttnRow = kHeadDim + 8;        // bf16 per staged row: 272 B, conflict-free ldmatrix
constexpr int kAttnPRow = kAttnKeys + 4;      // fp32 per score row

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t &r0, uint32_t &r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
// d += a . b (m16 x k16 bf16 row-major a, k16 x n8 bf16 b, fp32 d)
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
// the hi and lo bf16 parts of two fp32 weights, packed (first weight in the low half)
__device__ __forceinline__ void split2(float x0, float x1, uint32_t &hi, uint32_t &lo) {
  const uint16_t h0 = f2bf(x0), h1 = f2bf(x1);
  hi = static_cast<uint32_t>(h0) | (static_cast<uint32_t>(h1) << 16);
  lo = pack2(x0 - bf2f(h0), x1 - bf2f(h1));
}

size_t attention_smem_bytes() {
  return static_cast<size_t>(kAttnQPad + 2 * kAttnKeys) * kAttnRow * 2 +
         static_cast<size_t>(kAttnQPad) * (kAttnPRow + 2) * sizeof(float);
}

__global__ void __launch_bounds__(kAttnThreads) attention_kernel(const AttnArgs a) {
  extern __shared__ __align__(16) float attn_smem[];
  uint16_t *qs = reinterpret_cast<uint16_t *>(attn_smem);     // [48][136] bf16
  uint16_t *ks = qs + kAttnQPad * kAttnRow;                    // [64][136]
  uint16_t *vs = ks + kAttnKeys * kAttnRow;                    // [64][136]
  float *ps = reinterpret_cast<float *>(vs + kAttnKeys * kAttnRow);  // [48][68] scores, then weights
  float *ml = ps + kAttnQPad * kAttnPRow;                      // [48][2]
  const int nqry = a.nqry;
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int grp = a.nq / a.nkv;
  const int kend = min(kAttnKeys, a.nkeys - split * kAttnKeys);
  pdl_wait();
  pdl_release();
  // stage the slice's key and value rows and the group's query rows (16-byte chunks);
  // rows past the slice's keys or the group's queries are zero
  constexpr int kChunks = kHeadDim / 8;
  for (int e = tid; e < (2 * kAttnKeys + kAttnQPad) * kChunks; e += kAttnThreads) {
    const int r = e / kChunks, c = e % kChunks;
    uint16_t *dst;
    const uint16_t *src = nullptr;
    if (r < 2 * kAttnKeys) {
      const int kl = r < kAttnKeys ? r : r - kAttnKeys;
      dst = (r < kAttnKeys ? ks : vs) + kl * kAttnRow + 8 * c;
      if (kl < kend)
        src = (r < kAttnKeys ? a.k_cache : a.v_cache) +
              ((static_cast<int64_t>(b) * a.cache_len + split * kAttnKeys + kl) * a.nkv + g) * kHeadDim + 8 * c;
    } else {
      const int qi = r - 2 * kAttnKeys;
      dst = qs + qi * kAttnRow + 8 * c;
      if (qi < nqry) {
        const int i = qi / grp, head = g * grp + qi % grp;
        src = a.q + ((static_cast<int64_t>(b) * a.nr + i) * a.nq + head) * kHeadDim + 8 * c;
      }
    }
    if (src) {
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(static_cast<uint32_t>(
                       __cvta_generic_to_shared(dst))),
                   "l"(src)
                   : "memory");
    } else {
      *reinterpret_cast<uint4 *>(dst) = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();

  const int gq = lane >> 2, tq = lane & 3;   // the mma fragment's row group and column pair
  const uint32_t qs_a = static_cast<uint32_t>(__cvta_generic_to_shared(qs));
  const uint32_t ks_a = static_cast<uint32_t>(__cvta_generic_to_shared(ks));
  const uint32_t vs_a = static_cast<uint32_t>(__cvta_generic_to_shared(vs));
  // scores: warp w takes keys 8w .. 8w + 7 for the three query tiles
  {
    float acc[3][4];
#pragma unroll
    for (int m = 0; m < 3; ++m)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[m][i] = 0.0f;
#pragma unroll
    for (int kk = 0; kk < kHeadDim / 16; ++kk) {
      uint32_t b0, b1;
      ldsm_x2(ks_a + ((8 * warp + (lane & 7)) * kAttnRow + 16 * kk + ((lane >> 3) & 1) * 8) * 2, b0, b1);
#pragma unroll
      for (int m = 0; m < 3; ++m) {
        uint32_t a0, a1, a2, a3;
        ldsm_x4(qs_a + ((16 * m + (lane & 15)) * kAttnRow + 16 * kk + (lane >> 4) * 8) * 2, a0, a1, a2, a3);
        mma_bf16(acc[m], a0, a1, a2, a3, b0, b1);
      }
    }
    const int key0 = 8 * warp + 2 * tq;
    const bool v0 = key0 < kend, v1 = key0 + 1 < kend;
#pragma unroll
    for (int m = 0; m < 3; ++m) {
      const int r0 = 16 * m + gq;
      *reinterpret_cast<float2 *>(ps + r0 * kAttnPRow + key0) =
          make_float2(v0 ? acc[m][0] * a.scale : -INFINITY, v1 ? acc[m][1] * a.scale : -INFINITY);
      *reinterpret_cast<float2 *>(ps + (r0 + 8) * kAttnPRow + key0) =
          make_float2(v0 ? acc[m][2] * a.scale : -INFINITY, v1 ? acc[m][3] * a.scale : -INFINITY);
    }
  }
  __syncthreads();

  // softmax over the slice per query row (two keys per lane); padded rows get weights 0
  for (int qi = warp; qi < kAttnQPad; qi += kAttnThreads / 32) {
    float *row = ps + qi * kAttnPRow;
    if (qi >= nqry) {
      row[lane] = 0.0f;
      row[32 + lane] = 0.0f;
      continue;
    }
    const float s0 = row[lane], s1 = row[32 + lane];
    float m = fmaxf(s0, s1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float p0 = m == -INFINITY ? 0.0f : expf(s0 - m);
    const float p1 = m == -INFINITY ? 0.0f : expf(s1 - m);
    float l = p0 + p1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    row[lane] = p0;
    row[32 + lane] = p1;
    if (lane == 0) {
      ml[2 * qi] = m;
      ml[2 * qi + 1] = l;
    }
  }
  __syncthreads();

  // P.V: warp w takes dims 16w .. 16w + 15 (two n-tiles) for the three query tiles
  float acc[3][2][4];
#pragma unroll
  for (int m = 0; m < 3; ++m)
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[m][j][i] = 0.0f;
#pragma unroll
  for (int kk = 0; kk < kAttnKeys / 16; ++kk) {
    uint32_t b00, b01, b10, b11;   // [n-tile][k half]
    ldsm_x4_t(vs_a + ((16 * kk + (lane & 15)) * kAttnRow + 16 * warp + (lane >> 4) * 8) * 2, b00, b01, b10, b11);
#pragma unroll
    for (int m = 0; m < 3; ++m) {
      const float *r0 = ps + (16 * m + gq) * kAttnPRow + 16 * kk + 2 * tq;
      const float *r1 = r0 + 8 * kAttnPRow;
      const float2 x0 = *reinterpret_cast<const float2 *>(r0);
      const float2 x1 = *reinterpret_cast<const float2 *>(r1);
      const float2 x2 = *reinterpret_cast<const float2 *>(r0 + 8);
      const float2 x3 = *reinterpret_cast<const float2 *>(r1 + 8);
      uint32_t h0, h1, h2, h3, l0, l1, l2, l3;
      split2(x0.x, x0.y, h0, l0);
      split2(x1.x, x1.y, h1, l1);
      split2(x2.x, x2.y, h2, l2);
      split2(x3.x, x3.y, h3, l3);
      mma_bf16(acc[m][0], h0, h1, h2, h3, b00, b01);
      mma_bf16(acc[m][0], l0, l1, l2, l3, b00, b01);
      mma_bf16(acc[m][1], h0, h1, h2, h3, b10, b11);
      mma_bf16(acc[m][1], l0, l1, l2, l3, b10, b11);
    }
  }
#pragma unroll
  for (int m = 0; m < 3; ++m) {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int qi = 16 * m + gq + 8 * half;
      if (qi < nqry) {
        const int64_t base = ((static_cast<int64_t>(b) * a.nkv + g) * a.nsplit + split) * nqry + qi;
#pragma unroll
        for (int j = 0; j < 2; ++j)
          *reinterpret_cast<float2 *>(a.part_o + base * kHeadDim + 16 * warp + 8 * j + 2 * tq) =
              make_float2(acc[m][j][2 * half], acc[m][j][2 * half + 1]);
        if (tq == 0 && warp == 0) {
          a.part_ml[2 * base] = ml[2 * qi];
          a.part_ml[2 * base + 1] = ml[2 * qi + 1];
        }
      }
    }
  }
}

// One warp per (request, kv head, query row): out = sum_s e^(m_s - M) o_s / sum_s e^(m_s - M) l_s.
// Slices go 16 at a time: lane j (j < 16) loads slice s0 + j's (m, l) while every lane
// loads its 4 dims of the 16 slices' o rows, all in flight together; the weights are
// then passed from lane to lane.  Slices are added in order.
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
  constexpr int kBatch = 16;
  float M = -INFINITY, L = 0.0f;
  float o4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  for (int s0 = 0; s0 < a.nsplit; s0 += kBatch) {
    const int n = min(kBatch, a.nsplit - s0);
    float2 mlv = make_float2(-INFINITY, 0.0f);
    if (lane < n) mlv = *reinterpret_cast<const float2 *>(a.part_ml + 2 * (base0 + static_cast<int64_t>(s0 + lane) * a.nqry));
    float4 po[kBatch];
#pragma unroll
    for (int j = 0; j < kBatch; ++j)
      po[j] = j < n ? *reinterpret_cast<const float4 *>(a.part_o + (base0 + static_cast<int64_t>(s0 + j) * a.nqry) * kHeadDim +
                                                        4 * lane)
                    : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    // the running maximum over the slices so far; earlier sums are rescaled to it
    float mb = mlv.x;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, o));
    const float Mn = fmaxf(M, mb);
    if (Mn != -INFINITY) {
      const float r = M == -INFINITY ? 0.0f : expf(M - Mn);
      L *= r;
#pragma unroll
      for (int i = 0; i < 4; ++i) o4[i] *= r;
      const float e = (lane < n && mlv.x != -INFINITY) ? expf(mlv.x - Mn) : 0.0f;
      float le = e * mlv.y;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) le += __shfl_xor_sync(0xffffffffu, le, o);
      L += le;
#pragma unroll
      for (int j = 0; j < kBatch; ++j) {
        const float ej = __shfl_sync(0xffffffffu, e, j);
        o4[0] = __fmaf_rn(ej, po[j].x, o4[0]); o4[1] = __fmaf_rn(ej, po[j].y, o4[1]);
        o4[2] = __fmaf_rn(ej, po[j].z, o4[2]); o4[3] = __fmaf_rn(ej, po[j].w, o4[3]);
      }
      M = Mn;
    }
  }
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

// silu_mul_kernel reading the gate|up GEMM's pieces.
__global__ void __launch_bounds__(256) silu_mul_view_kernel(const PieceView gv, uint16_t *act, int M, int I) {
  pdl_wait();
  pdl_release();
  const long long n8 = static_cast<long long>(M) * (I / 8);
  for (long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; e < n8;
       e += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int m = static_cast<int>(e / (I / 8)), c = static_cast<int>(e % (I / 8));
    float gv8[8], uv[8];
    view_vals<8>(gv, m, 8 * c, gv8);
    view_vals<8>(gv, m, I + 8 * c, uv);
    float y[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) y[t] = gv8[t] / (1.0f + expf(-gv8[t])) * uv[t];
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
                                 int H, int *status, cudaStream_t stream, const uint16_t *in2, int64_t ld_in2,
                                 int rows2, const PieceView *dv) {
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
  a.in2 = in2;
  a.ld_in2 = ld_in2;
  a.status = status;
  a.delta_view = dv ? 1 : 0;
  if (dv) a.dv = *dv;
  if (launch_pdl(norm_rows_kernel, dim3(static_cast<unsigned>(rows + (in2 ? rows2 : 0))), dim3(kNormThreads), 0,
                 stream, a) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  count_launches(1);
  return DSPARK_OK;
}

dspark_status_t qk_norm_rope_launch(const uint16_t *qkv, int64_t ld, int nq, int nkv, const uint16_t *wq,
                                    const uint16_t *wk, float theta, uint16_t *q_out, uint16_t *k_cache,
                                    uint16_t *v_cache, int cache_len, int rows_per_req, int pos0, int rows,
                                    cudaStream_t stream, const uint16_t *kv2, int64_t ld2, int rows_per_req2,
                                    int pos02, int rows2, const PieceView *qv) {
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
  a.kv2 = kv2;
  a.ld2 = ld2;
  a.rows_per_req2 = rows_per_req2 > 0 ? rows_per_req2 : 1;
  a.pos02 = pos02;
  a.rows2 = (kv2 || qv) ? rows2 : 0;
  a.qkv_view = qv ? 1 : 0;
  if (qv) a.qv = *qv;
  const long long warps = static_cast<long long>(rows) * (nq + 2 * nkv) + static_cast<long long>(a.rows2) * 2 * nkv;
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
  const size_t smem = attention_smem_bytes();
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

dspark_status_t silu_mul_view_launch(const PieceView &gv, uint16_t *act, int M, int I, cudaStream_t stream) {
  const long long n8 = static_cast<long long>(M) * (I / 8);
  long long blocks = (n8 + 255) / 256;
  const long long cap = static_cast<long long>(device_sm_count() > 0 ? device_sm_count() : 1) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  if (launch_pdl(silu_mul_view_kernel, dim3(static_cast<unsigned>(blocks)), dim3(256), 0, stream, gv, act, M, I) !=
      cudaSuccess)
    return DSPARK_ERR_CUDA;
  count_launches(1);
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
