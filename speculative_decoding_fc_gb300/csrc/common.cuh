// Device-side helpers shared by the DSpark kernels (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "dspark.h"

namespace dspark {

// Records the first device-side error of a call in the workspace status word.
__device__ __forceinline__ void record_error(int *status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------- argmax keys
// A 64-bit key whose unsigned order is (value ascending, then index
// descending): the maximum key is the largest value at its lowest index.
// -0 is folded onto +0 so the two compare equal; NaN maps below every
// number so it never wins.
// Programmatic dependent launch.  Every kernel of the library is launched so that it
// may start while the previous kernel on the stream is still finishing: it calls
// pdl_wait() before its first access to global memory that an earlier kernel may
// have written (and before any global write), and pdl_release() once the next
// kernel may be scheduled.  Both are no-ops for a kernel launched without the
// attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint32_t ordered_bits(float x) {
  uint32_t u = __float_as_uint(x);
  if ((u & 0x7fffffffu) == 0u) u = 0u;                       // -0 -> +0
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu)) // NaN
    return 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ uint64_t argmax_key(float x, uint32_t idx) {
  return ((uint64_t)ordered_bits(x) << 32) | (uint64_t)(0xffffffffu - idx);
}

__device__ __forceinline__ uint32_t key_index(uint64_t key) {
  return 0xffffffffu - (uint32_t)(key & 0xffffffffu);
}

__device__ __forceinline__ float key_value(uint64_t key) {
  uint32_t o = (uint32_t)(key >> 32);
  uint32_t u = (o & 0x80000000u) ? (o & 0x7fffffffu) : ~o;
  return __uint_as_float(u);
}

// Max over the warp of a 64-bit key: the max of the high words, then the max of
// the low words of the lanes holding it (two warp reductions, no shuffles).
__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
  const uint32_t hi = static_cast<uint32_t>(v >> 32), lo = static_cast<uint32_t>(v);
  const uint32_t mh = __reduce_max_sync(0xffffffffu, hi);
  const uint32_t ml = __reduce_max_sync(0xffffffffu, hi == mh ? lo : 0u);
  return (static_cast<uint64_t>(mh) << 32) | ml;
}

// ---------------------------------------------------------------- softmax stats
// Running (max, sum of exp(x - max)) pairs.  Merging is exact in the max and
// rounds only in the sum.
struct SoftStat {
  float m;
  float s;
};

__device__ __forceinline__ SoftStat softstat_merge(SoftStat a, SoftStat b) {
  if (a.m == -INFINITY) return b;
  if (b.m == -INFINITY) return a;
  if (a.m >= b.m) return {a.m, a.s + b.s * expf(b.m - a.m)};
  return {b.m, b.s + a.s * expf(a.m - b.m)};
}

__device__ __forceinline__ void softstat_add(SoftStat &st, float x) {
  if (x == -INFINITY || x != x) return;
  if (x > st.m) {
    st.s = (st.m == -INFINITY) ? 1.0f : st.s * expf(st.m - x) + 1.0f;
    st.m = x;
  } else {
    st.s += expf(x - st.m);
  }
}

__device__ __forceinline__ SoftStat warp_softstat(SoftStat st) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    SoftStat w;
    w.m = __shfl_xor_sync(0xffffffffu, st.m, o);
    w.s = __shfl_xor_sync(0xffffffffu, st.s, o);
    st = softstat_merge(st, w);
  }
  return st;
}

// ---------------------------------------------------------------- Philox4x32-10
// Counter-based generator of Salmon, Moraes, Dror and Shaw (SC'11): ten
// rounds, each multiplying counter words 0 and 2 by fixed odd constants and
// mixing the 32-bit halves of the products with words 1 and 3 and the key;
// the key advances by two Weyl increments between rounds.
struct U4 {
  uint32_t x, y, z, w;
};

__device__ __forceinline__ U4 philox4x32_10(U4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint32_t a = 0xD2511F53u * c.x;
    const uint32_t ah = __umulhi(0xD2511F53u, c.x);
    const uint32_t b = 0xCD9E8D57u * c.z;
    const uint32_t bh = __umulhi(0xCD9E8D57u, c.z);
    c = U4{bh ^ c.y ^ k0, b, ah ^ c.w ^ k1, a};
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

// Uniforms of verify position `pos` of request `req` at decode step `step`:
// word 0 -> accept test, word 1 -> resample, each (w >> 8) * 2^-24.
__device__ __forceinline__ void verify_uniforms(uint64_t seed, uint32_t req, uint32_t pos,
                                                uint32_t step, double &ua, double &us) {
  U4 w = philox4x32_10(U4{req, pos, step, 0u}, (uint32_t)(seed & 0xffffffffu),
                       (uint32_t)(seed >> 32));
  ua = (double)(w.x >> 8) * (1.0 / 16777216.0);
  us = (double)(w.y >> 8) * (1.0 / 16777216.0);
}

__device__ __forceinline__ float bf16_lo(uint32_t pair) { return __uint_as_float(pair << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t pair) {
  return __uint_as_float(pair & 0xffff0000u);
}

}  // namespace dspark
