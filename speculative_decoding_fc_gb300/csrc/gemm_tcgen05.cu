// Dense bf16 GEMM on the 5th-generation tensor cores (sm_103a):
//   out[m, n] = sum_k X[m, k] * W[n, k]        fp32 accumulate in TMEM
//
// Serves both contractions of the drafter readout:
//   - fc projection: W = fc.weight [H, T*H], X = the T tapped hidden-state
//     tensors, read as T consecutive K segments (the concatenation is never
//     materialised); out = h, bf16.
//   - LM head: W = lm_head.weight [V, H], X = h [B*k, H]; out = fp32 logits.
//
// Design (GB300-first):
//   * "Swap-AB": the weight supplies the 128-row M side of tcgen05.mma and the
//     (few) activation rows the N side, so a decode batch of B*k = 7 rows is a
//     legal N = 16 tile and the kernel streams the weight exactly once.
//   * Persistent grid of one CTA per SM, 192 threads, warp-specialised:
//     warp 0 issues TMA loads into a ring of shared-memory stages, warp 1 issues
//     tcgen05.mma (one thread) into one of two TMEM accumulators, warps 2-5
//     drain TMEM with tcgen05.ld and store the tile.
//   * Work is split "stream-K": the (tile, k-block) units are cut into equal
//     contiguous ranges, one per CTA, so every SM streams the same number of
//     weight bytes whatever the tile count.  A tile cut between CTAs is
//     finished by the last CTA to arrive (atomic ticket, no spinning), which
//     adds the fp32 partials in CTA order: results do not depend on timing.
//     The fix-up keeps up to four pieces' loads in flight at once (one L2 round
//     trip per 16 columns for up to four pieces).
//   * Operands are 128-byte-swizzled K-major tiles (64 bf16 of K per row) as
//     TMA writes them; the UMMA shared-memory descriptors describe exactly that
//     layout.  Weights are loaded with an L2 evict-first policy, activations
//     with evict-last, and so are the outputs (the next kernel reads them).
//   * FP8 variant (kind::f8f6f4, E4M3 x E4M3): the same 128-byte rows hold 128
//     codes, each MMA consumes K = 32, and the epilogue multiplies by the
//     activation-row and weight-row scales.
//   * Every wait on an mbarrier is bounded: on timeout the CTA records
//     DSPARK_ERR_DEVICE_TIMEOUT, stops issuing, waits (bounded) for its own
//     copies and MMAs in flight, frees its TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace dspark {
namespace {

constexpr int kThreads = 192;
constexpr int kBM = 128;          // weight rows per tile (UMMA M)
constexpr int kBK = 64;           // bf16 K per stage: one 128-byte swizzle row
constexpr int kRowBytes = 128;    // bytes of K per operand row and stage (both kinds)
constexpr int kMaxStages = 12;
constexpr uint32_t kABytes = kBM * kBK * 2;
constexpr long long kWaitCycles = 2000000000LL;  // ~1 s at 2 GHz

// One GEMM of a launch.  A launch runs one phase, or two (the fc projection, then
// the LM head on its output h): the second phase's activation loads wait until
// the first phase has stored every output tile, its weight loads do not.
struct GemmPhase {
  CUtensorMap tm_w;
  CUtensorMap tm_x[kMaxTaps];
  const float *a_scale;   // FP8: scale of each activation row (else null)
  const float *w_scale;   // FP8: scale of each weight row (else null)
  void *out;
  float *partials;
  int *tickets;
  long long ldo;
  long long units;
  int kb_per_seg;
  int kb_total;
  int N;
  int out_bf16;
  int tiles;              // output tiles of the phase
};

struct GemmParams {
  GemmPhase ph[2];
  int nphase;
  int *sync;              // two phases: [0] phase-0 tiles stored, [1] CTAs finished
  int *status;
  int M;
  int BN;
  int tiles_m;
  int stages;
  uint32_t tmem_cols;
  uint32_t idesc;
  int defer_fixup;        // split tiles are added up by gemm_reduce_kernel, not here
};

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase of the given parity to complete.  Returns false
// (without waiting further) once the CTA's abort flag is set or the budget
// runs out; the latter sets the flag and records the timeout.
__device__ __noinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                      int *status) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if (clock64() - t0 > kWaitCycles) {
      *abort_flag = 1;
      record_error(status, DSPARK_ERR_DEVICE_TIMEOUT);
      return false;
    }
  }
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void prefetch_map(const CUtensorMap *map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major, 128-byte-swizzled operand
// tile: rows of 128 bytes, groups of 8 rows 1024 bytes apart (stride byte
// offset); the leading byte offset is unused by this layout.  Bits 46-48 hold
// the descriptor version 1, bits 61-63 the swizzle mode (2 = 128 bytes).
__device__ __forceinline__ uint64_t sdesc_k_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1) << 16;
  d |= static_cast<uint64_t>(1024 >> 4) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tc_mma_e4m3(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void tc_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void epi_bar_sync() {
  asm volatile("bar.sync 1, 128;" ::: "memory");
}

// ------------------------------------------------------------------ schedule
struct Range {
  long long begin, end;
};

__device__ __forceinline__ Range cta_range(long long units, int cta, int grid) {
  return {units * cta / grid, units * (cta + 1) / grid};
}

// The pieces ("segments") of a CTA's unit range, each within one tile: k-blocks kb0 ..
// kb1 - 1 of `tile`.  In range order segment 0 starts at begin and the last one ends at
// end.  A single-phase launch processes the last segment first when it is a partial
// tile and the range holds whole tiles too: the next CTA holds the rest of that tile
// and processes its own piece first, so every shared tile's pieces are done early and
// its fix-up runs while whole tiles are still streaming (in range order the piece would
// come last and the fix-ups of all shared tiles would trail the kernel).  Pieces and
// their fix-up order are the same in either order, so are the results.
struct Seg {
  int tile, kb0, kb1;
};

__device__ __forceinline__ int seg_count(Range rg, int kbt) {
  if (rg.end <= rg.begin) return 0;
  return static_cast<int>((rg.end - 1) / kbt - rg.begin / kbt) + 1;
}

__device__ __forceinline__ Seg seg_at(Range rg, int kbt, int i, int n, bool last_first) {
  int j = i;
  if (last_first && n >= 3 && (rg.end % kbt) != 0) j = (i == 0) ? n - 1 : i - 1;
  const long long tile = rg.begin / kbt + j;
  const long long lo = rg.begin > tile * kbt ? rg.begin : tile * kbt;
  const long long hi = rg.end < (tile + 1) * kbt ? rg.end : (tile + 1) * kbt;
  return {static_cast<int>(tile), static_cast<int>(lo - tile * kbt), static_cast<int>(hi - tile * kbt)};
}

// CTA whose range holds unit x: the largest c with floor(U*c/G) <= x.
__device__ __forceinline__ int cta_of_unit(long long x, long long units, int grid) {
  return static_cast<int>(((x + 1) * grid - 1) / units);
}

// The output side of a phase, copied into registers once per phase (fields read
// through a reference into the parameter block would be re-read after every store).
struct OutDesc {
  void *out;
  const float *a_scale;
  const float *w_scale;
  long long ldo;
  int N;
  int out_bf16;
  uint64_t pol;  // L2 policy of the output stores (evict-last: the next kernel reads them)
};

__device__ __forceinline__ OutDesc out_desc(const GemmPhase &P) {
  OutDesc o;
  o.out = P.out;
  o.a_scale = P.a_scale;
  o.w_scale = P.w_scale;
  o.ldo = P.ldo;
  o.N = P.N;
  o.out_bf16 = P.out_bf16;
  o.pol = policy_evict_last();
  return o;
}

__device__ __forceinline__ void store_out(const OutDesc &o, int M, int m, int n, float v) {
  if (m >= M || n >= o.N) return;
  if (o.w_scale) v *= __ldg(o.a_scale + m) * __ldg(o.w_scale + n);
  const long long off = static_cast<long long>(m) * o.ldo + n;
  if (o.out_bf16) {
    const unsigned short b = __bfloat16_as_ushort(__float2bfloat16_rn(v));
    asm volatile("st.global.L2::cache_hint.b16 [%0], %1, %2;" ::"l"(reinterpret_cast<unsigned short *>(o.out) + off),
                 "h"(b), "l"(o.pol)
                 : "memory");
  } else {
    asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(reinterpret_cast<float *>(o.out) + off), "f"(v),
                 "l"(o.pol)
                 : "memory");
  }
}

__device__ __forceinline__ int ld_relaxed_s32(const int *ptr) {
  int v;
  asm volatile("ld.relaxed.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(ptr) : "memory");
  return v;
}

// After observing (with a relaxed load) that phase 0 has stored all its tiles: an
// acquire fence for those stores, then a proxy fence so that this thread's TMA
// loads (async proxy) of h see them.
__device__ __forceinline__ void acquire_for_tma() {
  asm volatile("fence.acq_rel.gpu;" ::: "memory");
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Activation loads of n consecutive units from unit u (ring stages from `stage`).
__device__ __noinline__ void issue_x_pending(const GemmParams &p, const CUtensorMap *tmx, int kps,
                                             int kbt, int elem_k, long long u, int n, int stage,
                                             uint32_t base, uint32_t stage_bytes, uint32_t full0,
                                             int S, uint64_t pol_x) {
  for (int i = 0; i < n; ++i, ++u) {
    const int tile = static_cast<int>(u / kbt);
    const int kb = static_cast<int>(u - static_cast<long long>(tile) * kbt);
    const int m_tile = tile % p.tiles_m;
    const int seg = kb / kps;
    const int xk = (kb - seg * kps) * elem_k;
    tma_load_2d(base + stage * stage_bytes + kABytes, tmx + seg, xk, m_tile * p.BN,
                full0 + 8u * stage, pol_x);
    if (++stage == S) stage = 0;
  }
}

// Adds the pieces of a split tile (CTAs c_first .. c_first + nseg - 1, in CTA order,
// from 0) for output columns [c0, c0 + kC) of the row this thread holds, the loads of
// kP pieces in flight at a time, and stores them.  The GEMM's own fix-up takes 16
// columns of 4 pieces (8 columns of 8 pieces as well raised the kernel from 190 to 254
// registers; 8 of 8 alone made the 15-row projections' two column halves two rounds);
// the separate fix-up kernel takes 8 columns of 8 pieces for tiles of at most 8
// activation rows (the batch-1 fc's 4-5 way splits in one round of loads).  The sums
// are the same in either.
template <int kP, int kC>
__device__ __forceinline__ void add_pieces(const float *partials, int BN, long long units, int grid, int kbt,
                                           int tile, int c_first, int nseg, int c0, int mcount, int row, int n,
                                           int m_base, int M, const OutDesc &od) {
  float acc[kC];
#pragma unroll
  for (int j = 0; j < kC; ++j) acc[j] = 0.0f;
  for (int s0 = 0; s0 < nseg; s0 += kP) {
    float v[kP][kC];
#pragma unroll
    for (int q = 0; q < kP; ++q) {
      if (s0 + q < nseg) {
        const int c2 = c_first + s0 + q;
        const int tile_c2 = static_cast<int>((units * c2 / grid) / kbt);
        const int slot = (tile == tile_c2) ? 0 : 1;
        const float *src = partials + (static_cast<size_t>(c2) * 2 + slot) * static_cast<size_t>(BN) * kBM;
#pragma unroll
        for (int j = 0; j < kC; ++j) v[q][j] = (c0 + j < mcount) ? __ldcg(src + (c0 + j) * kBM + row) : 0.0f;
      }
    }
#pragma unroll
    for (int q = 0; q < kP; ++q)
      if (s0 + q < nseg)
#pragma unroll
        for (int j = 0; j < kC; ++j) acc[j] += v[q][j];
  }
#pragma unroll
  for (int j = 0; j < kC; ++j)
    if (c0 + j < mcount) store_out(od, M, m_base + c0 + j, n, acc[j]);
}

// ------------------------------------------------------------------ kernel
template <bool kFP8>
__global__ void __launch_bounds__(kThreads, 1) gemm_tcgen05_kernel(const __grid_constant__ GemmParams p) {
  constexpr int kElemK = kFP8 ? 128 : kBK;  // K elements per stage row
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *sbase = smem_raw + (base - raw);
  const uint32_t b_bytes = static_cast<uint32_t>(p.BN) * kRowBytes;
  const uint32_t stage_bytes = kABytes + b_bytes;
  const int S = p.stages;

  uint64_t *bars = reinterpret_cast<uint64_t *>(sbase + S * stage_bytes);
  const uint32_t full0 = smem_u32(bars);
  const uint32_t empty0 = full0 + 8u * S;
  const uint32_t tfull0 = empty0 + 8u * S;
  const uint32_t tempty0 = tfull0 + 16u;
  const uint32_t drain_bar = tempty0 + 16u;
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 2 * S + 5);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_holder + 1);
  volatile int *ticket_slot = reinterpret_cast<volatile int *>(tmem_holder + 2);
  volatile int *ok_slot = reinterpret_cast<volatile int *>(tmem_holder + 3);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int grid = gridDim.x;
  const int cta = blockIdx.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(full0 + 8u * s, 1);
      mbar_init(empty0 + 8u * s, 1);
    }
    mbar_init(tfull0, 1);
    mbar_init(tfull0 + 8u, 1);
    mbar_init(tempty0, 4);
    mbar_init(tempty0 + 8u, 4);
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    for (int ph = 0; ph < p.nphase; ++ph) prefetch_map(&p.ph[ph].tm_w);
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_holder)),
                 "r"(p.tmem_cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_holder;
  // Everything above touched only shared and tensor memory: from here on the
  // previous kernel's results are needed.  One wave of persistent CTAs: the next
  // kernel may be scheduled right away (its CTAs take SMs as these exit).
  pdl_wait();
  pdl_release();

  if (warp == 0) {
    // ---------------------------------------------------------------- TMA producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      long long issued = 0;
      bool ok = true;
      for (int ph = 0; ph < p.nphase && ok; ++ph) {
        const GemmPhase &P = p.ph[ph];
        const CUtensorMap *tmw = &P.tm_w;
        const CUtensorMap *tmx = &P.tm_x[0];
        const int kps = P.kb_per_seg;
        const Range rg = cta_range(P.units, cta, grid);
        const int kbt = P.kb_total;
        long long u = rg.begin;
        if (ph == 1) {
          // Phase 1 reads phase 0's output.  Until every phase-0 tile is stored,
          // only weight tiles are loaded (up to one ring of stages); their
          // activation loads follow once phase 0 is complete.
          const int need = p.ph[0].tiles;
          int seen = ld_relaxed_s32(p.sync);
          const long long u0 = u;
          const int stage0 = stage;
          int nq = 0;
          while (seen < need && nq < S && u < rg.end && ok) {
            const int tile = static_cast<int>(u / kbt);
            const int kb = static_cast<int>(u - static_cast<long long>(tile) * kbt);
            if (!wait_bar(empty0 + 8u * stage, phase ^ 1u, abort_flag, p.status)) {
              ok = false;
              break;
            }
            const uint32_t fb = full0 + 8u * stage;
            mbar_expect_tx(fb, stage_bytes);
            tma_load_2d(base + stage * stage_bytes, tmw, kb * kElemK, (tile / p.tiles_m) * kBM, fb,
                        pol_w);
            ++nq;
            ++u;
            ++issued;
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
            if ((nq & 3) == 0) seen = ld_relaxed_s32(p.sync);  // a round trip every 4 tiles
          }
          const long long t0 = clock64();
          while (seen < need) {
            if (*abort_flag || clock64() - t0 > kWaitCycles) break;
            __nanosleep(64);
            seen = ld_relaxed_s32(p.sync);
          }
          if (seen < need) {
            if (!*abort_flag) {
              *abort_flag = 1;
              record_error(p.status, DSPARK_ERR_DEVICE_TIMEOUT);
            }
            ok = false;
          }
          acquire_for_tma();
          // (on failure the launch's status is set; the stages are still completed
          // so that every issued copy lands)
          issue_x_pending(p, tmx, kps, kbt, kElemK, u0, nq, stage0, base, stage_bytes, full0, S,
                          pol_x);
          if (!ok) break;
        }
        // (a two-phase launch keeps range order from where phase 1's prefix stopped)
        const bool last_first = p.nphase == 1;
        const int nsg = last_first ? seg_count(rg, kbt) : 0;
        for (int si = 0; (last_first ? si < nsg : u < rg.end) && ok; ++si) {
          int tile, kb0, kb1;
          if (last_first) {
            const Seg sg = seg_at(rg, kbt, si, nsg, true);
            tile = sg.tile;
            kb0 = sg.kb0;
            kb1 = sg.kb1;
          } else {
            tile = static_cast<int>(u / kbt);
            kb0 = static_cast<int>(u - static_cast<long long>(tile) * kbt);
            const long long left = rg.end - u;
            kb1 = left < (kbt - kb0) ? kb0 + static_cast<int>(left) : kbt;
          }
          const int n_tile = tile / p.tiles_m;
          const int m_tile = tile - n_tile * p.tiles_m;
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!wait_bar(empty0 + 8u * stage, phase ^ 1u, abort_flag, p.status)) {
              ok = false;
              break;
            }
            const uint32_t fb = full0 + 8u * stage;
            mbar_expect_tx(fb, stage_bytes);
            const uint32_t sa = base + stage * stage_bytes;
            tma_load_2d(sa, tmw, kb * kElemK, n_tile * kBM, fb, pol_w);
            const int seg = kb / kps;
            const int xk = (kb - seg * kps) * kElemK;
            tma_load_2d(sa + kABytes, tmx + seg, xk, m_tile * p.BN, fb, pol_x);
            ++issued;
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
          }
          u += kb1 - kb0;
        }
      }
      if (!ok) {
        // Let the copies already issued land before the CTA exits.
        const long long first = issued > S ? issued - S : 0;
        for (long long j = first; j < issued; ++j) {
          const int s = static_cast<int>(j % S);
          const uint32_t par = static_cast<uint32_t>((j / S) & 1);
          const long long t0 = clock64();
          while (!mbar_try_wait(full0 + 8u * s, par) && clock64() - t0 < kWaitCycles) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int ph = 0; ph < p.nphase && ok; ++ph) {
        const Range rg = cta_range(p.ph[ph].units, cta, grid);
        const int kbt = p.ph[ph].kb_total;
        const int nsg = seg_count(rg, kbt);
        for (int si = 0; si < nsg && ok; ++si) {
          const Seg sg = seg_at(rg, kbt, si, nsg, p.nphase == 1);
          const int kb0 = sg.kb0, kb1 = sg.kb1;
          if (!wait_bar(tempty0 + 8u * acc, acc_phase ^ 1u, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * p.BN);
          for (int kb = kb0; kb < kb1; ++kb) {
            if (!wait_bar(full0 + 8u * stage, phase, abort_flag, p.status)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sa = base + stage * stage_bytes;
            const uint32_t sb = sa + kABytes;
            // 4 MMAs per stage, each over 32 bytes of K (16 bf16 or 32 E4M3)
#pragma unroll
            for (int kk = 0; kk < kRowBytes / 32; ++kk) {
              if constexpr (kFP8)
                tc_mma_e4m3(d_tmem, sdesc_k_sw128(sa + kk * 32), sdesc_k_sw128(sb + kk * 32),
                            p.idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
              else
                tc_mma_bf16(d_tmem, sdesc_k_sw128(sa + kk * 32), sdesc_k_sw128(sb + kk * 32),
                            p.idesc, (kb > kb0 || kk > 0) ? 1u : 0u);
            }
            tc_commit(empty0 + 8u * stage);
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          tc_commit(tfull0 + 8u * acc);
          acc ^= 1;
          if (acc == 0) acc_phase ^= 1u;
        }
      }
      // Every MMA issued by this thread has completed once this arrives.
      tc_commit(drain_bar);
      const long long t0 = clock64();
      while (!mbar_try_wait(drain_bar, 0) && clock64() - t0 < kWaitCycles) {
      }
    }
  } else {
    // ---------------------------------------------------------------- epilogue
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
    int acc = 0;
    uint32_t acc_phase = 0;
    bool alive = true;
    for (int ph = 0; ph < p.nphase && alive; ++ph) {
      const GemmPhase &P = p.ph[ph];
      const OutDesc od = out_desc(P);
      float *const partials = P.partials;
      int *const tickets = P.tickets;
      const long long units = P.units;
      const Range rg = cta_range(units, cta, grid);
      const int kbt = P.kb_total;
      const int first_tile = static_cast<int>(rg.begin / kbt);
      // phase 0 of a two-phase launch counts its stored tiles for phase 1
      const bool signal = (p.nphase == 2 && ph == 0);
      const int nsg = seg_count(rg, kbt);
      for (int si = 0; si < nsg; ++si) {
        const Seg sg = seg_at(rg, kbt, si, nsg, p.nphase == 1);
        const int tile = sg.tile, kb0 = sg.kb0, kb1 = sg.kb1;
        const int n_tile = tile / p.tiles_m;
        const int m_tile = tile - n_tile * p.tiles_m;
        const int n = n_tile * kBM + row;
        const int m_base = m_tile * p.BN;
        const bool whole = (kb0 == 0 && kb1 == kbt);

        // One thread waits for the accumulator; the decision is shared by all
        // four epilogue warps so that they leave the loop together on abort.
        if (threadIdx.x == 64)
          *ok_slot = wait_bar(tfull0 + 8u * acc, acc_phase, abort_flag, p.status) ? 1 : 0;
        epi_bar_sync();
        const int ok = *ok_slot;
        epi_bar_sync();
        if (!ok) {
          alive = false;
          break;
        }
        tc_fence_after();

        float *part = nullptr;
        if (!whole) {
          const int slot = (tile == first_tile) ? 0 : 1;
          part = partials + (static_cast<size_t>(cta) * 2 + slot) * static_cast<size_t>(p.BN) * kBM;
        }
        for (int cc = 0; cc < p.BN; cc += 16) {
          uint32_t r[16];
          tmem_ld16(lane_addr + static_cast<uint32_t>(acc * p.BN + cc), r);
          if (whole) {
            if (m_base + cc < p.M) {
#pragma unroll
              for (int j = 0; j < 16; ++j) store_out(od, p.M, m_base + cc + j, n, __uint_as_float(r[j]));
            }
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) part[(cc + j) * kBM + row] = __uint_as_float(r[j]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty0 + 8u * acc);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;

        if (whole && signal) {
          // the tile is stored: publish it (the barrier orders the four warps'
          // stores before thread 64's fence)
          epi_bar_sync();
          if (threadIdx.x == 64) {
            __threadfence();
            atomicAdd(p.sync, 1);
          }
        }
        if (!whole && !p.defer_fixup) {
          // Stream-K fix-up: the last CTA to finish a piece of this tile adds the
          // pieces in CTA order and stores the tile.
          __threadfence();
          epi_bar_sync();
          if (threadIdx.x == 64) *ticket_slot = atomicAdd(&tickets[tile], 1);
          epi_bar_sync();
          const int ticket = *ticket_slot;
          const long long t_first = static_cast<long long>(tile) * kbt;
          const int c_first = cta_of_unit(t_first, units, grid);
          const int c_last = cta_of_unit(t_first + kbt - 1, units, grid);
          const int nseg = c_last - c_first + 1;
          if (ticket == nseg - 1) {
            __threadfence();
            const int mcount = min(p.BN, p.M - m_base);
            // (24 columns, 96 loads in flight, took the batch-112 fc's fix-up tail down
            // by 2 us but the kernel to 244 registers and every other shape up by about
            // 0.5 us.)
            for (int c0 = 0; c0 < mcount; c0 += 16)
              add_pieces<4, 16>(partials, p.BN, units, grid, kbt, tile, c_first, nseg, c0, mcount, row, n, m_base,
                                p.M, od);
            if (threadIdx.x == 64) tickets[tile] = 0;
            if (signal) {
              epi_bar_sync();
              if (threadIdx.x == 64) {
                __threadfence();
                atomicAdd(p.sync, 1);
              }
            }
          }
          epi_bar_sync();
        }
      }
    }
  }

  // The producer and MMA warps ran their loops on one lane: converge each warp
  // before the CTA barrier so that every warp arrives whole, and only then free
  // the tensor memory the epilogue warps read.
  __syncwarp();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                 "r"(p.tmem_cols)
                 : "memory");
  }
  // A two-phase launch: the last CTA out clears the tile counter for the next one.
  if (p.nphase == 2 && threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.sync + 1, 1) == grid - 1) {
      p.sync[0] = 0;
      p.sync[1] = 0;
    }
  }
}

// ------------------------------------------------------------------ deferred fix-up
// When every tile is split across CTAs (fewer tiles than CTAs: the fc, the small
// projections), each tile's last arriver would add its pieces at the very end of the
// GEMM, one CTA per tile, after that CTA's own last piece.  Instead the GEMM only
// writes its pieces and this kernel adds them for all tiles at once: CTA (tile, 16
// columns), one thread per weight row, pieces added in CTA order from 0 exactly as
// the in-kernel fix-up does (the same bits).  A tile held whole by one CTA was stored
// by the GEMM and is skipped.
struct ReduceArgs {
  float *partials;
  void *out;
  const float *a_scale, *w_scale;
  long long ldo, units;
  int kb_total, N, out_bf16, M, BN, tiles_m, grid;
};

__global__ void __launch_bounds__(kBM) gemm_reduce_kernel(const ReduceArgs a) {
  pdl_wait();
  pdl_release();
  const int tile = blockIdx.x;
  const int c0 = blockIdx.y * 16;
  const int row = threadIdx.x;
  const int n_tile = tile / a.tiles_m;
  const int m_base = (tile - n_tile * a.tiles_m) * a.BN;
  const int n = n_tile * kBM + row;
  const long long t_first = static_cast<long long>(tile) * a.kb_total;
  const int c_first = cta_of_unit(t_first, a.units, a.grid);
  const int c_last = cta_of_unit(t_first + a.kb_total - 1, a.units, a.grid);
  const int mcount = min(a.BN, a.M - m_base);
  if (c_first == c_last || c0 >= mcount) return;
  OutDesc od;
  od.out = a.out;
  od.a_scale = a.a_scale;
  od.w_scale = a.w_scale;
  od.ldo = a.ldo;
  od.N = a.N;
  od.out_bf16 = a.out_bf16;
  od.pol = policy_evict_last();
  const int nseg = c_last - c_first + 1;
  if (mcount - c0 <= 8)
    add_pieces<8, 8>(a.partials, a.BN, a.units, a.grid, a.kb_total, tile, c_first, nseg, c0, mcount, row, n, m_base,
                     a.M, od);
  else
    add_pieces<4, 16>(a.partials, a.BN, a.units, a.grid, a.kb_total, tile, c_first, nseg, c0,
                      c0 + 16 < mcount ? c0 + 16 : mcount, row, n, m_base, a.M, od);
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// 2-D bf16 tensor [rows, inner] with the given row stride, read in boxes of
// 64 (one 128-byte swizzle row) x box_rows.
bool make_map(CUtensorMap *map, const void *ptr, uint64_t inner, uint64_t rows,
              uint64_t row_stride_bytes, uint32_t box_rows, bool fp8) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(fp8 ? kRowBytes : kBK), box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                   const_cast<void *>(ptr), dims,
                   strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

struct Tiling {
  int BN, tiles_m, tiles_n, kb_total, stages;
  long long units;
  uint32_t tmem_cols;
  size_t smem;
};

// K is counted in elements; esize = bytes per element (2 bf16, 1 E4M3).
Tiling plan(int M, int N, int K, int esize = 2) {
  Tiling t;
  t.tiles_m = (M + 255) / 256;
  int bn = (M + t.tiles_m - 1) / t.tiles_m;
  bn = (bn + 15) / 16 * 16;
  if (bn < 16) bn = 16;
  t.BN = bn;
  t.tiles_n = (N + kBM - 1) / kBM;
  t.kb_total = K * esize / kRowBytes;
  t.units = static_cast<long long>(t.tiles_m) * t.tiles_n * t.kb_total;
  uint32_t cols = 32;
  while (cols < static_cast<uint32_t>(2 * bn)) cols <<= 1;
  t.tmem_cols = cols;
  const size_t stage = kABytes + static_cast<size_t>(bn) * kRowBytes;
  const size_t budget = 227 * 1024 - 1024 - 256;
  int st = static_cast<int>(budget / stage);
  if (st > kMaxStages) st = kMaxStages;
  t.stages = st;
  t.smem = 1024 + stage * st + 256;
  return t;
}

size_t partial_bytes(const Tiling &t) {
  return static_cast<size_t>(kMaxGemmCtas) * 2 * t.BN * kBM * sizeof(float);
}

}  // namespace

size_t gemm_counter_bytes(int M, int N, int K) {
  if (M < 1 || N < 1 || K < kBK) return 0;
  Tiling t = plan(M, N, K);  // the tile grid does not depend on the element size
  return align_up(static_cast<size_t>(t.tiles_m) * t.tiles_n * sizeof(int), kWsAlign);
}

size_t gemm_workspace_size(int M, int N, int K) {
  if (M < 1 || N < 1 || K < kBK) return 0;
  Tiling t = plan(M, N, K);
  const size_t tickets = align_up(static_cast<size_t>(t.tiles_m) * t.tiles_n * sizeof(int), kWsAlign);
  return tickets + align_up(partial_bytes(t), kWsAlign);
}

// The tile grid and the partial tiles do not depend on the element size.
size_t gemm_workspace_size_fp8(int M, int N, int K) { return gemm_workspace_size(M, N, K); }

namespace {

// Tensor maps, scales, outputs and the stream-K schedule of one phase; ws holds the
// phase's tile tickets then its partial tiles.
bool fill_phase(GemmPhase &P, const GemmProblem &pr, const Tiling &t, void *ws) {
  const int K = pr.n_seg * pr.seg_k;
  const int esize = pr.fp8 ? 1 : 2;
  if (!make_map(&P.tm_w, pr.w, static_cast<uint64_t>(K), static_cast<uint64_t>(pr.N),
                static_cast<uint64_t>(K) * esize, kBM, pr.fp8))
    return false;
  for (int s = 0; s < pr.n_seg; ++s) {
    if (!make_map(&P.tm_x[s], pr.x[s], static_cast<uint64_t>(pr.seg_k),
                  static_cast<uint64_t>(pr.M), static_cast<uint64_t>(pr.x_ld[s]) * esize,
                  static_cast<uint32_t>(t.BN), pr.fp8))
      return false;
  }
  P.a_scale = pr.a_scale;
  P.w_scale = pr.w_scale;
  const size_t tickets = align_up(static_cast<size_t>(t.tiles_m) * t.tiles_n * sizeof(int), kWsAlign);
  P.tickets = reinterpret_cast<int *>(ws);
  P.partials = reinterpret_cast<float *>(static_cast<char *>(ws) + tickets);
  P.out = pr.out;
  P.ldo = pr.ldo;
  P.units = t.units;
  P.kb_per_seg = pr.seg_k * esize / kRowBytes;
  P.kb_total = t.kb_total;
  P.N = pr.N;
  P.out_bf16 = pr.out_bf16 ? 1 : 0;
  P.tiles = t.tiles_m * t.tiles_n;
  return true;
}

void fill_common(GemmParams &p, const Tiling &t, int M, bool fp8, int *status) {
  p.status = status;
  p.M = M;
  p.BN = t.BN;
  p.tiles_m = t.tiles_m;
  p.stages = t.stages;
  p.tmem_cols = t.tmem_cols;
  // Instruction descriptor: D fp32 (bits 4-5 = 1); A and B format at bits 7-9 and
  // 10-12 (kind::f16: 1 = bf16; kind::f8f6f4: 0 = E4M3); both K-major; N >> 3 at
  // bits 17-22, M >> 4 at bits 24-28.
  const uint32_t fmt = fp8 ? 0u : 1u;
  p.idesc = (1u << 4) | (fmt << 7) | (fmt << 10) | (static_cast<uint32_t>(t.BN >> 3) << 17) |
            (static_cast<uint32_t>(kBM >> 4) << 24);
}

bool configure(bool fp8) {
  static bool configured[2][64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (dev >= 0 && dev < 64 && configured[fp8 ? 1 : 0][dev]) return true;
  auto kern = fp8 ? gemm_tcgen05_kernel<true> : gemm_tcgen05_kernel<false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024) !=
      cudaSuccess)
    return false;
  if (dev >= 0 && dev < 64) configured[fp8 ? 1 : 0][dev] = true;
  return true;
}

}  // namespace

dspark_status_t gemm_launch(const GemmProblem &pr, void *ws, size_t ws_bytes, int *status,
                            cudaStream_t stream, PieceView *view) {
  const int K = pr.n_seg * pr.seg_k;
  const int esize = pr.fp8 ? 1 : 2;
  Tiling t = plan(pr.M, pr.N, K, esize);
  if (ws_bytes < gemm_workspace_size(pr.M, pr.N, K)) return DSPARK_ERR_WORKSPACE;
  const int sms = device_sm_count();
  if (sms <= 0) return DSPARK_ERR_NO_DEVICE;

  GemmParams p;
  memset(&p, 0, sizeof(p));
  if (!fill_phase(p.ph[0], pr, t, ws)) return DSPARK_ERR_CUDA;
  p.nphase = 1;
  fill_common(p, t, pr.M, pr.fp8, status);

  long long grid = sms < kMaxGemmCtas ? sms : kMaxGemmCtas;
  const long long by_work = t.units / 4 > 0 ? t.units / 4 : 1;
  if (grid > by_work) grid = by_work;
  // Fewer tiles than CTAs: every tile is split.  Where its fix-up is heavy (tiles of 32
  // or more activation rows, or K of 320 k-blocks and more, split about four ways:
  // the fc), the pieces are added by a second kernel; for the small projections the
  // in-kernel fix-up is cheaper than one more launch.  (Measured: the batch-112 fc 67
  // -> 51 us; the 8- and 15-row backbone projections about 1 us slower deferred.)
  bool defer = static_cast<long long>(t.tiles_m) * t.tiles_n < grid && (t.BN >= 32 || t.kb_total >= 320);
  if (pr.pieces_only) {
    // the reader adds the pieces: the kernel only writes them, no fix-up launch
    if (pr.fp8 || !pr.out_bf16 || !view) return DSPARK_ERR_INVALID_ARG;
    if (t.units * grid >= (1LL << 31)) return DSPARK_ERR_UNSUPPORTED_SHAPE;  // readers index in 32 bits
    p.defer_fixup = 1;
    defer = false;
    view->partials = p.ph[0].partials;
    view->out = static_cast<const uint16_t *>(pr.out);
    view->ldo = pr.ldo;
    view->units = t.units;
    view->kb_total = t.kb_total;
    view->grid = static_cast<int>(grid);
    view->BN = t.BN;
    view->tiles_m = t.tiles_m;
    view->M = pr.M;
  } else {
    p.defer_fixup = defer ? 1 : 0;
  }
  if (!configure(pr.fp8)) return DSPARK_ERR_CUDA;
  auto kern = pr.fp8 ? gemm_tcgen05_kernel<true> : gemm_tcgen05_kernel<false>;
  if (launch_pdl(kern, dim3(static_cast<unsigned>(grid)), dim3(kThreads), t.smem, stream, p) !=
      cudaSuccess)
    return DSPARK_ERR_CUDA;
  count_launches(1);
  if (defer) {
    ReduceArgs r;
    r.partials = p.ph[0].partials;
    r.out = p.ph[0].out;
    r.a_scale = p.ph[0].a_scale;
    r.w_scale = p.ph[0].w_scale;
    r.ldo = p.ph[0].ldo;
    r.units = p.ph[0].units;
    r.kb_total = p.ph[0].kb_total;
    r.N = p.ph[0].N;
    r.out_bf16 = p.ph[0].out_bf16;
    r.M = p.M;
    r.BN = p.BN;
    r.tiles_m = p.tiles_m;
    r.grid = static_cast<int>(grid);
    const dim3 rgrid(static_cast<unsigned>(t.tiles_m * t.tiles_n), static_cast<unsigned>((t.BN + 15) / 16));
    if (launch_pdl(gemm_reduce_kernel, rgrid, dim3(kBM), 0, stream, r) != cudaSuccess) return DSPARK_ERR_CUDA;
    count_launches(1);
  }
  return DSPARK_OK;
}

// Two GEMMs in one launch: [256 B: tile counter, exit counter][phase 0][phase 1].
size_t gemm2_workspace_size(int M, int N0, int K0, int N1, int K1) {
  const size_t a = gemm_workspace_size(M, N0, K0), b = gemm_workspace_size(M, N1, K1);
  if (!a || !b) return 0;
  return kWsAlign + align_up(a, kWsAlign) + b;
}

size_t gemm2_phase1_offset(int M, int N0, int K0) {
  return kWsAlign + align_up(gemm_workspace_size(M, N0, K0), kWsAlign);
}

dspark_status_t gemm_launch2(const GemmProblem &pr0, const GemmProblem &pr1, void *ws,
                             size_t ws_bytes, int *status, cudaStream_t stream) {
  const int K0 = pr0.n_seg * pr0.seg_k, K1 = pr1.n_seg * pr1.seg_k;
  if (pr0.M != pr1.M || pr0.fp8 != pr1.fp8) return DSPARK_ERR_INVALID_ARG;
  const int esize = pr0.fp8 ? 1 : 2;
  Tiling t0 = plan(pr0.M, pr0.N, K0, esize), t1 = plan(pr1.M, pr1.N, K1, esize);
  if (ws_bytes < gemm2_workspace_size(pr0.M, pr0.N, K0, pr1.N, K1)) return DSPARK_ERR_WORKSPACE;
  const int sms = device_sm_count();
  if (sms <= 0) return DSPARK_ERR_NO_DEVICE;

  char *w = static_cast<char *>(ws);
  GemmParams p;
  memset(&p, 0, sizeof(p));
  p.sync = reinterpret_cast<int *>(w);
  if (!fill_phase(p.ph[0], pr0, t0, w + kWsAlign)) return DSPARK_ERR_CUDA;
  if (!fill_phase(p.ph[1], pr1, t1, w + gemm2_phase1_offset(pr0.M, pr0.N, K0)))
    return DSPARK_ERR_CUDA;
  p.nphase = 2;
  fill_common(p, t0, pr0.M, pr0.fp8, status);  // same M: same tile width and ring

  // every CTA must be resident (phase 1 waits for tiles stored by all CTAs): a
  // cooperative launch, with programmatic dependent launch when enabled
  long long grid = sms < kMaxGemmCtas ? sms : kMaxGemmCtas;
  const long long small = (t0.units < t1.units ? t0.units : t1.units) / 4;
  if (grid > small) grid = small > 0 ? small : 1;
  if (!configure(pr0.fp8)) return DSPARK_ERR_CUDA;
  auto kern = pr0.fp8 ? gemm_tcgen05_kernel<true> : gemm_tcgen05_kernel<false>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = t0.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess && cfg.numAttrs == 2) {
    cudaGetLastError();
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, p);
  }
  if (e != cudaSuccess) {
    cudaGetLastError();
    return DSPARK_ERR_CUDA;
  }
  count_launches(1);
  return DSPARK_OK;
}

}  // namespace dspark
