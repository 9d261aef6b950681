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

// ---------------------------------------------------------------- cluster variant
// For a few long rows (the activation rows of one step): a cluster of C CTAs per
// row, CTA rank r taking the r-th contiguous range of the row's 16-byte chunks.
// Each CTA keeps up to kHold chunks per thread in registers, takes their max, the
// cluster combines the C maxima through distributed shared memory (the max does not
// depend on the order), and each CTA writes its codes; rank 0 writes the scale.
constexpr int kHold = 4;
constexpr int kMaxCluster = 8;

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ float dsmem_load(const float *local, uint32_t rank) {
  const uint32_t la = static_cast<uint32_t>(__cvta_generic_to_shared(local));
  uint32_t ra;
  float v;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(ra) : "r"(la), "r"(rank));
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(ra) : "memory");
  return v;
}

__device__ __forceinline__ float amax8(const uint4 q, float m) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) m = fmaxf(m, fmaxf(fabsf(bf16_lo(w[e])), fabsf(bf16_hi(w[e]))));
  return m;
}

__device__ __forceinline__ uint2 codes8(const uint4 q, float sc) {
  float f[8] = {bf16_lo(q.x), bf16_hi(q.x), bf16_lo(q.y), bf16_hi(q.y),
                bf16_lo(q.z), bf16_hi(q.z), bf16_lo(q.w), bf16_hi(q.w)};
#pragma unroll
  for (int e = 0; e < 8; ++e) f[e] = __fdiv_rn(f[e], sc);
  return make_uint2(e4m3x4(f[0], f[1], f[2], f[3]), e4m3x4(f[4], f[5], f[6], f[7]));
}

__global__ void __launch_bounds__(kThreads) quantize_rows_cluster_kernel(
    const __grid_constant__ QuantArgs a, int csize) {
  __shared__ float red[kThreads / 32];
  __shared__ float part_s, scale_s;
  const uint32_t rank = cluster_rank();
  const int row = blockIdx.x / csize;
  const int tid = threadIdx.x;
  const int c8 = a.seg_cols / 8;       // chunks of one segment row
  const int chunks = a.nseg * c8;      // chunks of the concatenated row
  const int per = (chunks + csize - 1) / csize;
  const int lo = static_cast<int>(rank) * per;
  const int hi = min(chunks, lo + per);
  pdl_wait();
  uint4 held[kHold];
  float amax = 0.0f;
#pragma unroll
  for (int h = 0; h < kHold; ++h) {
    const int ch = lo + tid + h * kThreads;
    held[h] = make_uint4(0u, 0u, 0u, 0u);
    if (ch < hi) {
      const int sg = ch / c8;
      held[h] = __ldg(reinterpret_cast<const uint4 *>(a.segs[sg] + row * a.seg_ld) + (ch - sg * c8));
      amax = amax8(held[h], amax);
    }
  }
  for (int ch = lo + tid + kHold * kThreads; ch < hi; ch += kThreads) {  // long ranges
    const int sg = ch / c8;
    amax = amax8(__ldg(reinterpret_cast<const uint4 *>(a.segs[sg] + row * a.seg_ld) + (ch - sg * c8)),
                 amax);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((tid & 31) == 0) red[tid >> 5] = amax;
  __syncthreads();
  if (tid == 0) {
    float m = red[0];
    for (int w = 1; w < kThreads / 32; ++w) m = fmaxf(m, red[w]);
    part_s = m;
  }
  // every CTA's partial max is in its shared memory
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
  if (tid == 0) {
    float m = 0.0f;
    for (int r = 0; r < csize; ++r) m = fmaxf(m, dsmem_load(&part_s, static_cast<uint32_t>(r)));
    const float sc = m > 0.0f ? __fdiv_rn(m, 448.0f) : 1.0f;
    scale_s = sc;
    if (rank == 0) a.scales[row] = sc;
  }
  __syncthreads();
  // this CTA is done reading its peers' shared memory; it waits for them before exit
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
  const float sc = scale_s;
  uint2 *dst = reinterpret_cast<uint2 *>(a.codes + static_cast<long long>(row) * chunks * 8);
#pragma unroll
  for (int h = 0; h < kHold; ++h) {
    const int ch = lo + tid + h * kThreads;
    if (ch < hi) dst[ch] = codes8(held[h], sc);
  }
  for (int ch = lo + tid + kHold * kThreads; ch < hi; ch += kThreads) {
    const int sg = ch / c8;
    dst[ch] = codes8(__ldg(reinterpret_cast<const uint4 *>(a.segs[sg] + row * a.seg_ld) + (ch - sg * c8)),
                     sc);
  }
  pdl_release();
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
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
  // Few rows (activations): a cluster of up to 8 CTAs per row, about 512 chunks of
  // 16 bytes per CTA.  Many rows (weights): one CTA per row.
  const long long chunks = static_cast<long long>(nseg) * seg_cols / 8;
  const int sms = device_sm_count();
  int csize = 1;
  if (sms > 0 && rows < 2 * sms)
    while (csize < kMaxCluster && chunks > static_cast<long long>(csize) * 2 * kThreads) csize *= 2;
  if (csize > 1 && static_cast<long long>(rows) * csize <= 0x7fffffffLL) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(rows * csize));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(csize);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 2 : 1;
    if (cudaLaunchKernelEx(&cfg, quantize_rows_cluster_kernel, a, csize) == cudaSuccess) {
      count_launches(1);
      return DSPARK_OK;
    }
    cudaGetLastError();  // refused: one CTA per row below
  }
  if (launch_pdl(quantize_rows_kernel, dim3(rows), dim3(kThreads), 0, stream, a) != cudaSuccess)
    return DSPARK_ERR_CUDA;
  count_launches(1);
  return DSPARK_OK;
}

}  // namespace dspark
