// Per-row FP8 (E4M3) quantisation for the FP8 drafter weights and activations.
//
// "Qwen3.8-27B DFlash drafter recipe - 72.2 tok/s on Arc Pro B70" ships FP8
// drafters (drafter-fp8-v5, qwen3.8-27b-dflash-drafter-fp8-b70) without giving
// the scheme.  The reading taken: one fp32 scale per row, scale = amax / 448
// (1 for an all-zero row), codes = E4M3(x / scale) rounded to nearest even and
// saturated to +-448.  Both divisions are the IEEE ones, so the codes are
// bit-identical to any exact implementation of the same rule.
#include <cuda_runtime.h>

#include "common.cuh"
#include "internal.h"

namespace dspark {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxSegs = kMaxTaps;

struct QuantArgs {
  const uint16_t *segs[kMaxSegs];
  int64_t seg_ld;
  int nseg;
  int seg_cols;
  uint8_t *codes;
  float *scales;
};

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  // cvt packs (hi, lo): the first source lands in the upper byte
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
  return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

// One CTA per row: the row max over every segment, then the codes.
__global__ void __launch_bounds__(kThreads) quantize_rows_kernel(const __grid_constant__ QuantArgs a) {
  __shared__ float red[kThreads / 32];
  __shared__ float scale_s;
  const int row = blockIdx.x;
  const int tid = threadIdx.x;
  const int c8 = a.seg_cols / 8;  // 16-byte chunks of a segment row
  pdl_wait();
  float amax = 0.0f;
  for (int sgi = 0; sgi < a.nseg; ++sgi) {
    const uint4 *src = reinterpret_cast<const uint4 *>(a.segs[sgi] + row * a.seg_ld);
    for (int i = tid; i < c8; i += kThreads) {
      const uint4 q = __ldg(src + i);
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int e = 0; e < 4; ++e)
        amax = fmaxf(amax, fmaxf(fabsf(bf16_lo(w[e])), fabsf(bf16_hi(w[e]))));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((tid & 31) == 0) red[tid >> 5] = amax;
  __syncthreads();
  if (tid == 0) {
    float m = red[0];
    for (int w = 1; w < kThreads / 32; ++w) m = fmaxf(m, red[w]);
    const float sc = m > 0.0f ? __fdiv_rn(m, 448.0f) : 1.0f;
    scale_s = sc;
    a.scales[row] = sc;
  }
  __syncthreads();
  const float sc = scale_s;
  const long long out_row = static_cast<long long>(row) * a.nseg * a.seg_cols;
  for (int sgi = 0; sgi < a.nseg; ++sgi) {
    const uint4 *src = reinterpret_cast<const uint4 *>(a.segs[sgi] + row * a.seg_ld);
    uint2 *dst = reinterpret_cast<uint2 *>(a.codes + out_row + static_cast<long long>(sgi) * a.seg_cols);
    for (int i = tid; i < c8; i += kThreads) {
      const uint4 q = __ldg(src + i);
      float f[8] = {bf16_lo(q.x), bf16_hi(q.x), bf16_lo(q.y), bf16_hi(q.y),
                    bf16_lo(q.z), bf16_hi(q.z), bf16_lo(q.w), bf16_hi(q.w)};
#pragma unroll
      for (int e = 0; e < 8; ++e) f[e] = __fdiv_rn(f[e], sc);
      dst[i] = make_uint2(e4m3x4(f[0], f[1], f[2], f[3]), e4m3x4(f[4], f[5], f[6], f[7]));
    }
  }
  pdl_release();  // after this CTA's work: the grid may span many waves
}

}  // namespace

dspark_status_t quantize_fp8_launch(const uint16_t *const *segs, int nseg, int64_t seg_ld,
                                    int rows, int seg_cols, uint8_t *codes, float *scales,
                                    cudaStream_t stream) {
  QuantArgs a;
  for (int i = 0; i < kMaxSegs; ++i) a.segs[i] = i < nseg ? segs[i] : nullptr;
  a.seg_ld = seg_ld;
  a.nseg = nseg;
  a.seg_cols = seg_cols;
  a.codes = codes;
  a.scales = scales;
  if (launch_pdl(quantize_rows_kernel, dim3(rows), dim3(kThreads), 0, stream, a) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  count_launches(1);
  return DSPARK_OK;
}

}  // namespace dspark
