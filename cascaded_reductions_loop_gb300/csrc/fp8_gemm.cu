// fp8_gemm.cu -- dynamic FP8 quantised GEMM: row absmax -> E4M3 quantisation
// -> FP8 GEMM -> dequantisation ([E] §4.3, read per row of X).
//
// The cascade has a hard dependency: no element can be rounded before the
// max of its whole row is known, and the rounding is not linear, so the max
// cannot be folded into the GEMM loop incrementally the way the softmax max
// can ([S] Methodologie 1: the round has no invertible dependent factor).
// The two stages therefore cooperate inside one persistent kernel
// (fp8_gemm_kernel), at the granularity of 128-row blocks of X ([E] §3.3,
// the inter-block level):
//   * quantiser warps (eight per CTA) take rows of X in increasing order, a
//     batch of eight per CTA at a time from a global counter (the next batch
//     is claimed while the current one is processed); one warp holds a whole
//     row in registers, reduces |x|
//     to the row max, sets sx = max / 448 (IEEE fp32 division), writes the
//     E4M3 codes of the correctly rounded x / sx (cvt.rn.satfinite) and then
//     counts the row into its 128-row block's readiness counter (release);
//   * the GEMM part runs on CTA pairs (2-CTA clusters, tcgen05 cta_group::2):
//     a pair computes a 256 x 256 output tile (or, in the last round, a
//     256 x 128 half tile, so that the leftover tiles spread over every
//     pair), each CTA loading with TMA its own 128 rows of the codes and its
//     own half of the tile's Wq rows into its own shared memory; one thread
//     of rank 0 issues the M = 256 MMAs
//     (kind::f8f6f4, E4M3 x E4M3 -> fp32 in tensor memory), so each SM reads
//     only its half of the B tile from its shared memory.  A CTA's TMA
//     producer waits (acquire) for its row block to be complete before it
//     loads codes from it, so the first tiles start while later rows are
//     still being quantised.  Four epilogue warps per CTA apply sx[m]*sw[n]
//     and round to bf16.
// The standalone absmax_quant_regs_kernel / absmax_quant_long_kernel compute
// the first two steps alone (rf_absmax_quant_fp8).
#include <math.h>

#include <vector>

#include "rf_device.cuh"
#include "rf_internal.h"

namespace rf {
namespace {

// ------------------------------------------------------------------ quantisation

constexpr int kQuantWarps = 4;
constexpr int kVecPerLaneMax = 16;   // rows up to 32 * 16 * 8 = 4096 elements stay in registers
constexpr int kRegRowMax = 32 * kVecPerLaneMax * 8;

__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// x / s correctly rounded to fp32, given r = RN(1/s) for the row: q0 = RN(x r)
// is within one ulp of x / s, the residual x - s q0 is exact under an FMA,
// and one more FMA step q0 + r (x - s q0) rounds to RN(x / s) (Markstein's
// correction, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990).  Done on pairs of
// elements with the packed f32x2 FMA/MUL (each lane rounds as the scalar
// instruction would).  The correction can turn a negative zero quotient into
// +0, so the sign bit of every code is then OR-ed in from x's own sign bit
// (a nonzero negative quotient already carries it; x >= 0 adds nothing).
// Rows with a tiny scale use IEEE division instead (see row_scale).
// tests/test_gpu_fp8.py checks the codes against an IEEE fp32 division over
// every (bf16 x, bf16 row max) pair.
__device__ __forceinline__ uint32_t quant2_recip(uint32_t w, uint64_t neg_s2, uint64_t r2) {
  const uint64_t x2 = f2(bf16lo(w), bf16hi(w));
  const uint64_t q0 = fmul2(x2, r2);
  const uint64_t e = ffma2(q0, neg_s2, x2);          // x - s q0, exact
  float lo, hi;
  f2_split(ffma2(e, r2, q0), lo, hi);
  return cvt_e4m3x2(lo, hi);
}

// 8 bf16 (one 16-byte vector) -> 8 E4M3 codes (little-endian in a uint2).
template <bool kRecip>
__device__ __forceinline__ uint2 quant8(const uint4 v, float s, float r) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t c[4];
  if constexpr (kRecip) {
    const uint64_t neg_s2 = f2(-s, -s), r2 = f2(r, r);
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = quant2_recip(w[i], neg_s2, r2);
    // byte k of a code word is element k; its sign is bit 7 of byte 1 or 3
    // of the bf16 word holding it
    const uint32_t sg0 = __byte_perm(w[0], w[1], 0x7531) & 0x80808080u;
    const uint32_t sg1 = __byte_perm(w[2], w[3], 0x7531) & 0x80808080u;
    return make_uint2(__byte_perm(c[0], c[1], 0x5410) | sg0, __byte_perm(c[2], c[3], 0x5410) | sg1);
  } else {
    (void)r;
#pragma unroll
    for (int i = 0; i < 4; ++i)
      c[i] = cvt_e4m3x2(__fdiv_rn(bf16lo(w[i]), s), __fdiv_rn(bf16hi(w[i]), s));
    return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
  }
}

__device__ __forceinline__ uint32_t absmax_bits(const uint4 v) {
  // |bf16| ordering equals the ordering of its bits with the sign cleared;
  // __vmaxu2 takes the max of each 16-bit half separately
  const uint32_t a = __vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu);
  const uint32_t b = __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu);
  const uint32_t c = __vmaxu2(a, b);
  return max(c & 0xFFFFu, c >> 16);
}

struct RowScale {
  float s, r;
  bool recip;
};

__device__ __forceinline__ RowScale row_scale(uint32_t amax_bits) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    amax_bits = max(amax_bits, __shfl_xor_sync(0xffffffffu, amax_bits, o));
  RowScale rs;
  rs.s = __fdiv_rn(__uint_as_float(amax_bits << 16), 448.0f);
  rs.r = __frcp_rn(rs.s);
  // The reciprocal route needs the residual x - s q0 to be exact.  It is a
  // multiple of 2^(e_x - 46) below 2^(e_x - 22) (e_x = exponent of x), hence
  // representable whenever |x| >= 2^-103; smaller |x| only matter when
  // |x / s| >= 2^-10 (below that every code is a signed zero), i.e. when
  // s < 2^-93.  Rows with s < 2^-90 therefore use IEEE division.
  rs.recip = rs.s >= 8.07793567e-28f;   // 2^-90
  return rs;
}

template <bool kStream>
__device__ __forceinline__ void store_codes(uint2* p, uint2 v) {
  if constexpr (kStream) __stcs(p, v);
  else *p = v;
}

// One warp quantises one row of nvec 16-byte vectors (nvec <= 32 *
// kVecPerLaneMax) held in registers: X is read from memory once.  kStream
// marks the codes as streamed (evict-first) when nothing reads them soon.
template <bool kStream>
__device__ __forceinline__ void quant_row_regs(const uint4* __restrict__ xr, uint2* __restrict__ qr,
                                               float* __restrict__ sxp, int nvec, int lane) {
  uint4 cur[kVecPerLaneMax];
#pragma unroll
  for (int i = 0; i < kVecPerLaneMax; ++i) {
    const int j = lane + 32 * i;
    cur[i] = j < nvec ? __ldcs(xr + j) : make_uint4(0, 0, 0, 0);
  }
  uint32_t amax = 0;
#pragma unroll
  for (int i = 0; i < kVecPerLaneMax; ++i) amax = max(amax, absmax_bits(cur[i]));
  const RowScale rs = row_scale(amax);
  if (lane == 0) *sxp = rs.s;
  if (rs.s == 0.f) {                                // all-zero row: codes 0x00
#pragma unroll
    for (int i = 0; i < kVecPerLaneMax; ++i)
      if (lane + 32 * i < nvec) store_codes<kStream>(qr + lane + 32 * i, make_uint2(0, 0));
  } else if (rs.recip) {
#pragma unroll
    for (int i = 0; i < kVecPerLaneMax; ++i)
      if (lane + 32 * i < nvec)
        store_codes<kStream>(qr + lane + 32 * i, quant8<true>(cur[i], rs.s, rs.r));
  } else {
#pragma unroll
    for (int i = 0; i < kVecPerLaneMax; ++i)
      if (lane + 32 * i < nvec)
        store_codes<kStream>(qr + lane + 32 * i, quant8<false>(cur[i], rs.s, rs.r));
  }
}

// Longer rows: two passes over the row (the second one mostly hits L2).
__device__ __forceinline__ void quant_row_long(const uint4* __restrict__ xr, uint2* __restrict__ qr,
                                               float* __restrict__ sxp, int nvec, int lane) {
  uint32_t amax = 0;
  for (int j = lane; j < nvec; j += 32) amax = max(amax, absmax_bits(__ldg(xr + j)));
  const RowScale rs = row_scale(amax);
  if (lane == 0) *sxp = rs.s;
  for (int j = lane; j < nvec; j += 32) {
    if (rs.s == 0.f)
      qr[j] = make_uint2(0, 0);
    else
      qr[j] = rs.recip ? quant8<true>(__ldg(xr + j), rs.s, rs.r)
                       : quant8<false>(__ldg(xr + j), rs.s, rs.r);
  }
}

// Standalone quantisation, rows up to kRegRowMax elements: one warp per row.
// Memory parallelism comes from occupancy: four 4-warp CTAs per SM, each
// warp with its whole row in flight.
__global__ void __launch_bounds__(kQuantWarps * 32, 4)
    absmax_quant_regs_kernel(const uint4* __restrict__ X, uint8_t* __restrict__ Xq,
                             float* __restrict__ sx, int M, int K, unsigned* err) {
  const int lane = threadIdx.x & 31;
  const int nw = gridDim.x * kQuantWarps;
  const int nvec = K >> 3;
  for (int row = blockIdx.x * kQuantWarps + (threadIdx.x >> 5); row < M; row += nw)
    if (RF_IN(err, row, M))
      quant_row_regs<true>(X + (size_t)row * nvec, reinterpret_cast<uint2*>(Xq + (size_t)row * K),
                           sx + row, nvec, lane);
}

__global__ void __launch_bounds__(kQuantWarps * 32)
    absmax_quant_long_kernel(const uint4* __restrict__ X, uint8_t* __restrict__ Xq,
                             float* __restrict__ sx, int M, int K, unsigned* err) {
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kQuantWarps + (threadIdx.x >> 5);
  if (row >= M || !RF_IN(err, row, M)) return;
  const int nvec = K >> 3;
  quant_row_long(X + (size_t)row * nvec, reinterpret_cast<uint2*>(Xq + (size_t)row * K), sx + row,
                 nvec, lane);
}

// ------------------------------------------------------------------ fused kernel

constexpr int BM = 128;                          // rows of A per CTA (256 per pair)
constexpr int BN = 256;                          // output columns per pair tile
constexpr int BK = 128;                          // bytes of K per stage = one 128-byte swizzle row
constexpr int kStages = 6;
constexpr int kABytes = BM * BK;                 // this CTA's 128 rows of codes
constexpr int kBBytes = (BN / 2) * BK;           // this CTA's half of the B tile (full tiles)
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kPairStageBytes = 2 * kStageBytes; // what lands on rank 0's barrier per stage
constexpr int kEpiWarps = 4;
constexpr int kFusedQuantWarps = 8;
constexpr int kFirstEpiWarp = 2, kFirstQuantWarp = kFirstEpiWarp + kEpiWarps;
constexpr int kGemmThreads = 32 * (kFirstQuantWarp + kFusedQuantWarps);   // 448
constexpr int kAccCols = BN;                     // one fp32 accumulator tile in TMEM
constexpr int kTmemCols = 2 * kAccCols;          // two: epilogue of tile i overlaps tile i+1
constexpr int kGemmSmem = kStages * kStageBytes + 1024 /*align*/ + 256 /*bars*/;
constexpr uint32_t kIdescPair = make_idesc(2 * BM, BN, /*e4m3*/ 0, 0, 0);
constexpr uint32_t kIdescPairHalf = make_idesc(2 * BM, BN / 2, /*e4m3*/ 0, 0, 0);

// Output tile t of the schedule.  Tiles t < n_full are 256 x 256 tiles in
// row-major order of the tile grid; the next n_half are 256 x 128 halves of
// the remaining tiles (full tile n_full + h / 2, column half h % 2).
struct Tile {
  int m0;      // first output row of the pair
  int n0;      // first output column
  int ncols;   // 256 or 128
};

__host__ __device__ __forceinline__ Tile tile_of(int t, int tiles_n, int n_full) {
  Tile w;
  if (t < n_full) {
    w.m0 = (t / tiles_n) * (2 * BM);
    w.n0 = (t % tiles_n) * BN;
    w.ncols = BN;
  } else {
    const int h = t - n_full, f = n_full + (h >> 1);
    w.m0 = (f / tiles_n) * (2 * BM);
    w.n0 = (f % tiles_n) * BN + (h & 1) * (BN / 2);
    w.ncols = BN / 2;
  }
  return w;
}
static_assert(kStages * kStageBytes + 256 + 1024 <= 227 * 1024, "shared memory");

// The tile schedule of a launch over `clusters` CTA pairs: whole rounds of
// 256 x 256 tiles first; the tiles left for a last, partial round are split
// in column halves when that spreads them over the pairs.  Tiles t < n_full
// are full, the rest halves; cluster c takes tiles c, c + clusters, ...
struct Schedule {
  int tiles_n;      // 256-column tiles per row of tiles
  int64_t pairs;    // full tiles of the output
  int n_full;       // of them, scheduled whole
  int n_tiles;      // scheduled tiles, halves counted one by one
};
inline Schedule make_schedule(int M, int N, int clusters) {
  Schedule sc;
  sc.tiles_n = (N + BN - 1) / BN;
  sc.pairs = (int64_t)sc.tiles_n * ((M + 2 * BM - 1) / (2 * BM));
  const int full_rounds = (int)(sc.pairs / clusters);
  const int left = (int)(sc.pairs - (int64_t)full_rounds * clusters);
  sc.n_full = (left > 0 && 2 * left <= clusters) ? full_rounds * clusters : (int)sc.pairs;
  sc.n_tiles = sc.n_full + 2 * ((int)sc.pairs - sc.n_full);
  return sc;
}

struct GemmBars {
  uint64_t full[kStages];    // rank 0: both CTAs' tiles of a stage have landed
  uint64_t empty[kStages];   // each CTA: the pair's MMAs have read its slot
  uint64_t acc_full[2];      // each CTA: its accumulator rows of a tile are complete
  uint64_t acc_empty[2];     // rank 0: both CTAs' epilogues have drained a buffer
  uint64_t drain;            // rank 0: every MMA has completed
  uint32_t tmem;
  int abort;
  int qbase[2];              // first row of the quantisers' current / next batch
};

// Readiness of one 128-row block of codes: bounded wait (acquire) until all
// its rows below M have been counted in.
__device__ __forceinline__ bool wait_rows_ready(const unsigned* ready, int m0, int M) {
  if (m0 >= M) return true;                       // rows past M: TMA fills zeros
  const unsigned need = (unsigned)min(BM, M - m0);
  const unsigned* c = ready + m0 / BM;
  if (ld_acquire_u32(c) < need) {
    const uint64_t t0 = globaltimer_ns();
    while (ld_acquire_u32(c) < need) {
      if (globaltimer_ns() - t0 > kDefaultWaitNs) return false;
      __nanosleep(128);
    }
  }
  fence_proxy_async_global();                     // the codes are then read by TMA
  return true;
}

// Persistent: 2-CTA clusters, one CTA per SM, 448 threads.
//   warp 0      TMA producer (both CTAs)
//   warp 1      TMEM allocation (both CTAs); MMA issuer (rank 0, one thread)
//   warps 2-5   epilogue (TMEM lane quarter = warp % 4)
//   warps 6-13  quantisers
// Tile t (tile_of) covers output rows m0 .. m0 + 255 (CTA r: + 128 r) and
// columns n0 .. n0 + ncols - 1 (CTA r loads B rows n0 + r ncols / 2 ..,
// through tmB for full tiles and tmBh, with boxes of 64 rows, for halves);
// cluster c takes tiles c, c + nclusters, ...  Rank 0's MMA thread
// accumulates tile i into TMEM buffer i % 2 of both CTAs while the epilogues
// drain buffer (i - 1) % 2.  Counters (zeroed by the host before the launch):
// ctr[0] is the next row to quantise, ctr[1 + b] the rows of block b done.
__global__ void __launch_bounds__(kGemmThreads, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmBh, const uint4* __restrict__ X,
                    uint8_t* __restrict__ Xq, float* __restrict__ sx, const float* __restrict__ sw,
                    __nv_bfloat16* __restrict__ Y, int M, int N, int K, int tiles_n, int n_full,
                    int n_tiles, unsigned* __restrict__ ctr, unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  GemmBars* bars = reinterpret_cast<GemmBars*>(smem + kStages * kStageBytes);
  volatile int* abort_flag = &bars->abort;
  const unsigned* ready = ctr + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int crank = (int)cluster_ctarank();
  const bool leader = crank == 0;
  const int cid = (int)blockIdx.x >> 1, ncl = (int)gridDim.x >> 1;
  const int nk = (K + BK - 1) / BK;
  const int my_tiles = n_tiles > cid ? (n_tiles - cid + ncl - 1) / ncl : 0;

  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    prefetch_tmap(&tmBh);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&bars->full[i]), 1);
      mbar_init(smem_u32(&bars->empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars->acc_full[i]), 1);
      mbar_init(smem_u32(&bars->acc_empty[i]), 2 * kEpiWarps);
    }
    mbar_init(smem_u32(&bars->drain), 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(&bars->tmem), kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();            // both CTAs' barriers and TMEM exist before any cross-CTA use
  tc_fence_after();
  const uint32_t tmem = bars->tmem;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer: this CTA's A rows and B half, counted
      // on rank 0's full barrier
      int it = 0;
      bool ok = true;
      for (int i = 0; ok && i < my_tiles && !*abort_flag; ++i) {
        const Tile w = tile_of(cid + i * ncl, tiles_n, n_full);
        const int m0 = w.m0 + crank * BM;
        const int nb0 = w.n0 + crank * (w.ncols / 2);
        const bool half = w.ncols != BN;
        if (!wait_rows_ready(ready, m0, M)) {
          ok = false;
          break;
        }
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int slot = it % kStages;
          if (it >= kStages &&
              !mbar_wait_cluster(smem_u32(&bars->empty[slot]), (uint32_t)(((it / kStages) + 1) & 1))) {
            ok = false;
            break;
          }
          if (*abort_flag) {
            ok = false;
            break;
          }
          uint8_t* a = smem + slot * kStageBytes;
          const uint32_t full0 = mapa_shared(smem_u32(&bars->full[slot]), 0);
          if (leader)
            mbar_arrive_expect_tx(smem_u32(&bars->full[slot]),
                                  half ? 2 * (kABytes + kBBytes / 2) : kPairStageBytes);
          tma_load_2d_pair(smem_u32(a), &tmA, full0, kb * BK, m0);
          tma_load_2d_pair(smem_u32(a + kABytes), half ? &tmBh : &tmB, full0, kb * BK, nb0);
        }
      }
      if (!ok) {
        raise_error(err, kDevErrTimeout);
        *abort_flag = 1;
      }
      // the last stages' release arrives from the peer's MMA thread: take
      // them before this CTA may exit (bounded)
      for (int j = it - kStages < 0 ? 0 : it - kStages; j < it; ++j)
        ok = mbar_wait_cluster(smem_u32(&bars->empty[j % kStages]), (uint32_t)((j / kStages) & 1),
                               ok ? kDefaultWaitNs : 1000000ull) && ok;
    }
  } else if (warp == 1) {
    if (leader && lane == 0) {
      // ---------------- MMA issuer (one thread of rank 0)
      int it = 0;
      bool ok = true;
      for (int i = 0; ok && i < my_tiles; ++i) {
        const int a = i & 1;
        if (i >= 2 &&
            !mbar_wait_cluster(smem_u32(&bars->acc_empty[a]), (uint32_t)(((i >> 1) + 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + a * kAccCols;
        const uint32_t idesc =
            tile_of(cid + i * ncl, tiles_n, n_full).ncols == BN ? kIdescPair : kIdescPairHalf;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int slot = it % kStages;
          if (!mbar_wait_cluster(smem_u32(&bars->full[slot]), (uint32_t)((it / kStages) & 1)) ||
              *abort_flag) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + slot * kStageBytes);
          const uint32_t sb = sa + kABytes;
#pragma unroll
          for (int k = 0; k < BK / 32; ++k)
            mma_f8_pair(d, sw128_desc(sa + k * 32, 1024, 16), sw128_desc(sb + k * 32, 1024, 16),
                        idesc, (kb | k) != 0);
          mma_commit_pair(smem_u32(&bars->empty[slot]));
          mma_commit_pair(mapa_shared(smem_u32(&bars->empty[slot]), 1));
        }
        if (ok) {
          mma_commit_pair(smem_u32(&bars->acc_full[a]));
          mma_commit_pair(mapa_shared(smem_u32(&bars->acc_full[a]), 1));
        }
      }
      if (!ok) {
        raise_error(err, kDevErrTimeout);
        *abort_flag = 1;
      }
      // nothing may still run on the tensor core when TMEM is released
      mma_commit_pair(smem_u32(&bars->drain));
      (void)mbar_wait(smem_u32(&bars->drain), 0, 1000000000ull);
    }
  } else if (warp < kFirstQuantWarp) {
    // ---------------- epilogue: TMEM -> registers -> scale -> bf16 -> global
    const int sub = warp & 3;                    // TMEM lane quarter of this warp
    const uint32_t lane_off = (uint32_t)(sub * 32) << 16;
    const bool vec_ok = (N % 8) == 0;
    // 32-byte stores (whole L2 sectors) when every chunk start is 32-byte aligned
    const bool v8_ok = (N % 16) == 0 && (reinterpret_cast<uintptr_t>(Y) & 31) == 0;
    for (int i = 0; i < my_tiles; ++i) {
      const int a = i & 1;
      const Tile w = tile_of(cid + i * ncl, tiles_n, n_full);
      const int m0 = w.m0 + crank * BM, n0 = w.n0;
      const int row = m0 + sub * 32 + lane;
      const bool got = mbar_wait_cluster(smem_u32(&bars->acc_full[a]), (uint32_t)((i >> 1) & 1)) &&
                       wait_rows_ready(ready, m0, M);
      if (!__all_sync(0xffffffffu, got && !*abort_flag)) {
        raise_error(err, kDevErrTimeout);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const bool row_in = row < M && RF_IN(err, (int64_t)row * N + N - 1, (int64_t)M * N);
      const float srow = row_in ? sx[row] : 0.f;
#pragma unroll 1
      for (int c0 = 0; c0 < w.ncols; c0 += 32) {
        if (n0 + c0 >= N) break;
        uint32_t r[32];
        tmem_ld32(tmem + a * kAccCols + lane_off + c0, r);
        tmem_ld_wait();
        const bool full_chunk = n0 + c0 + 32 <= N;
        float swv[32];
        if (full_chunk) {
          const float4* s4 = reinterpret_cast<const float4*>(sw + n0 + c0);
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 f = __ldg(s4 + q);
            swv[4 * q] = f.x;
            swv[4 * q + 1] = f.y;
            swv[4 * q + 2] = f.z;
            swv[4 * q + 3] = f.w;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) swv[j] = (n0 + c0 + j < N) ? __ldg(sw + n0 + c0 + j) : 0.f;
        }
        uint32_t packed[16];
#pragma unroll
        for (int j = 0; j < 16; ++j)
          packed[j] = pack_bf16x2(__uint_as_float(r[2 * j]) * srow * swv[2 * j],
                                  __uint_as_float(r[2 * j + 1]) * srow * swv[2 * j + 1]);
        if (row_in) {
          __nv_bfloat16* yp = Y + (size_t)row * N + n0 + c0;
          if (v8_ok && full_chunk) {
#pragma unroll
            for (int q = 0; q < 2; ++q)
              st_global_v8(yp + 16 * q, &packed[8 * q]);
          } else if (vec_ok && full_chunk) {
            uint4* y4 = reinterpret_cast<uint4*>(yp);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              y4[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2],
                                 packed[4 * q + 3]);
          } else {
            uint16_t* yh = reinterpret_cast<uint16_t*>(yp);
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (n0 + c0 + j < N)
                yh[j] = (j & 1) ? (uint16_t)(packed[j >> 1] >> 16) : (uint16_t)(packed[j >> 1] & 0xFFFF);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {                             // buffer a may be overwritten
        if (leader) mbar_arrive(smem_u32(&bars->acc_empty[a]));
        else mbar_arrive_remote(mapa_shared(smem_u32(&bars->acc_empty[a]), 0));
      }
    }
  } else {
    // ---------------- quantisers: batches of rows in increasing order from ctr[0]
    const int qw = warp - kFirstQuantWarp;
    const int nvec = K >> 3;
    if (qw == 0 && lane == 0) bars->qbase[0] = (int)atomicAdd(ctr, (unsigned)kFusedQuantWarps);
    named_bar_sync(1, 32 * kFusedQuantWarps);
    for (int k = 0;; ++k) {
      const int base = *reinterpret_cast<volatile int*>(&bars->qbase[k & 1]);
      if (base >= M) break;                        // the same for every quantiser warp
      if (qw == 0 && lane == 0)                    // claim the next batch early
        bars->qbase[(k + 1) & 1] = (int)atomicAdd(ctr, (unsigned)kFusedQuantWarps);
      const int row = base + qw;
      if (row < M && RF_IN(err, row, M)) {
        const uint4* xr = X + (size_t)row * nvec;
        uint2* qr = reinterpret_cast<uint2*>(Xq + (size_t)row * K);
        if (K <= kRegRowMax) quant_row_regs<false>(xr, qr, sx + row, nvec, lane);
        else quant_row_long(xr, qr, sx + row, nvec, lane);
        fence_proxy_async_global();                // codes are read by TMA
        __syncwarp();                              // the row's stores before the release below
        if (lane == 0) red_release_add(ctr + 1 + row / BM, 1u);
      }
      // the next batch's base is visible, and every warp has read this one
      // before it is overwritten two batches on
      named_bar_sync(1, 32 * kFusedQuantWarps);
    }
  }

  tc_fence_before();
  __syncthreads();
  // rank 0 has drained its MMAs and each CTA has taken its last barrier
  // arrivals from the peer; neither CTA's shared or tensor memory is used by
  // the other after this
  cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// Pairs of CTAs of fp8_gemm_kernel that can be resident at once (cached per
// device): at most one per two SMs.
int gemm_clusters(int sms, cudaLaunchConfig_t cfg) {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!cached[dev]) {
    cfg.gridDim = dim3(sms & ~1, 1, 1);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, fp8_gemm_kernel, &cfg) != cudaSuccess || n < 1) return 0;
    cached[dev] = n < sms / 2 ? n : sms / 2;
  }
  return cached[dev];
}

}  // namespace

size_t fp8_counter_bytes(int M) {
  return ((size_t)(1 + (M + BM - 1) / BM) * sizeof(unsigned) + 255) & ~(size_t)255;
}

size_t fp8_workspace_bytes(int M, int N, int K, bool need_xq, bool need_sx) {
  (void)N;
  size_t b = fp8_counter_bytes(M);
  if (need_xq) b += ((size_t)M * K + 255) & ~(size_t)255;
  if (need_sx) b += (size_t)M * sizeof(float);
  return b;
}

cudaError_t launch_absmax_quant(const void* X, int M, int K, float* sx, uint8_t* xq,
                                unsigned* err, cudaStream_t s) {
  const int qblocks = (M + kQuantWarps - 1) / kQuantWarps;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidValue;
  if (K <= kRegRowMax) {
    const int resident = 4 * sms;                      // four 4-warp CTAs per SM
    absmax_quant_regs_kernel<<<qblocks < resident ? qblocks : resident, kQuantWarps * 32, 0, s>>>(
        static_cast<const uint4*>(X), xq, sx, M, K, err);
  } else {
    absmax_quant_long_kernel<<<qblocks, kQuantWarps * 32, 0, s>>>(static_cast<const uint4*>(X), xq,
                                                                   sx, M, K, err);
  }
  return cudaGetLastError();
}

cudaError_t launch_absmax_fp8_gemm(const void* X, const uint8_t* Wq, const float* sw, void* Y,
                                   int M, int N, int K, float* sx, uint8_t* xq, void* workspace,
                                   unsigned* err, cudaStream_t s) {
  const int sms = sm_count();
  if (sms < 2) return cudaErrorInvalidValue;
  // workspace: counters first, then (when the caller keeps no copy) the codes
  // and the row scales
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  unsigned* ctr = reinterpret_cast<unsigned*>(ws);
  size_t off = fp8_counter_bytes(M);
  if (!xq) {
    xq = ws + off;
    off += ((size_t)M * K + 255) & ~(size_t)255;
  }
  if (!sx) sx = reinterpret_cast<float*>(ws + off);

  CUtensorMap tmA, tmB, tmBh;
  if (!encode_tmap_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, (uint64_t)K, (uint64_t)M,
                      (uint64_t)K, BK, BM, true) ||
      !encode_tmap_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, Wq, (uint64_t)K, (uint64_t)N,
                      (uint64_t)K, BK, BN / 2, true) ||
      !encode_tmap_2d(&tmBh, CU_TENSOR_MAP_DATA_TYPE_UINT8, Wq, (uint64_t)K, (uint64_t)N,
                      (uint64_t)K, BK, BN / 4, true))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaMemsetAsync(ctr, 0, (size_t)(1 + (M + BM - 1) / BM) * sizeof(unsigned), s);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(fp8_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
  if (e != cudaSuccess) return e;
  if ((int64_t)((N + BN - 1) / BN) * ((M + 2 * BM - 1) / (2 * BM)) >= (1ll << 29))
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = kGemmSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // every CTA also quantises, so the grid fills the GPU even when there are
  // fewer tiles than pairs of SMs; it is sized to the clusters that can be
  // resident together
  const int clusters = gemm_clusters(sms, cfg);
  if (clusters < 1) return cudaErrorInvalidConfiguration;
  cfg.gridDim = dim3(2 * clusters, 1, 1);
  const Schedule sc = make_schedule(M, N, clusters);
  return cudaLaunchKernelEx(&cfg, fp8_gemm_kernel, tmA, tmB, tmBh, static_cast<const uint4*>(X), xq,
                            sx, sw, static_cast<__nv_bfloat16*>(Y), M, N, K, sc.tiles_n, sc.n_full,
                            sc.n_tiles, ctr, err);
}

// Host-side check of the tile schedule (make_schedule, tile_of and the
// kernel's per-cluster tile count) for an M x N output on `clusters` pairs.
// Returns 0 when it holds, -1 for refused sizes, else the number of the
// first check that fails:
//   1 the per-cluster tile counts add up to the scheduled tiles;
//   2 every tile is a full tile or a column half, on the 256 x 128 grid;
//   3 every 256-row x 128-column block of the output is computed once.
int fp8_schedule_selfcheck(int M, int N, int clusters) {
  if (M < 1 || N < 1 || clusters < 1 || clusters > 4096) return -1;
  const Schedule sc = make_schedule(M, N, clusters);
  if (sc.pairs >= (1ll << 24)) return -1;          // keeps the coverage map small
  int64_t counted = 0;
  for (int c = 0; c < clusters; ++c)
    counted += sc.n_tiles > c ? (sc.n_tiles - c + clusters - 1) / clusters : 0;
  if (counted != sc.n_tiles) return 1;
  const int rows = (M + 2 * BM - 1) / (2 * BM);
  std::vector<unsigned char> cover((size_t)rows * sc.tiles_n * 2, 0);
  for (int t = 0; t < sc.n_tiles; ++t) {
    const Tile w = tile_of(t, sc.tiles_n, sc.n_full);
    if (w.ncols != BN && w.ncols != BN / 2) return 2;
    if (w.m0 % (2 * BM) != 0 || w.n0 % (BN / 2) != 0 || (w.ncols == BN && w.n0 % BN != 0)) return 2;
    const int r = w.m0 / (2 * BM), h0 = w.n0 / (BN / 2);
    if (r >= rows || h0 + w.ncols / (BN / 2) > 2 * sc.tiles_n) return 2;
    for (int h = h0; h < h0 + w.ncols / (BN / 2); ++h)
      if (cover[(size_t)r * 2 * sc.tiles_n + h]++) return 3;
  }
  for (unsigned char v : cover)
    if (v != 1) return 3;
  return 0;
}

}  // namespace rf
