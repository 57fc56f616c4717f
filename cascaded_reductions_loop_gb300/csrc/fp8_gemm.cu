// fp8_gemm.cu -- dynamic FP8 quantised GEMM: row absmax -> E4M3 quantisation
// -> FP8 GEMM -> dequantisation ([E] §4.3, read per row of X).
//
// The cascade has a hard dependency: no element can be rounded before the
// max of its whole row is known, and the rounding is not linear, so the max
// cannot be folded into the GEMM loop incrementally the way the softmax max
// can.  It therefore runs as two cooperating kernels ([E] §3.3 multi-kernel
// level):
//   1. absmax_quant_regs_kernel (rows up to 4096 elements; longer rows use
//      absmax_quant_long_kernel, which reads each row twice): one warp per
//      row of X reads the row once into registers, reduces |x| to the row
//      max, sets sx = max / 448 (IEEE fp32 division) and writes the E4M3
//      codes of the correctly rounded x / sx (cvt.rn.satfinite) plus sx.
//      X is read from HBM once.
//   2. fp8_gemm_kernel: a tcgen05 GEMM (kind::f8f6f4, E4M3 x E4M3 -> fp32 in
//      tensor memory) over TMA-staged 128-byte-swizzled tiles, warp
//      specialised (TMA producer warp, single-thread MMA issuer, four
//      epilogue warps), whose epilogue applies sx[m] * sw[n] and rounds to
//      bf16.  It is launched as a programmatic dependent of kernel 1.  The
//      codes travel through memory as 1 byte per element, half the size of
//      the bf16 input, so the pair moves as many bytes as a fused kernel
//      that re-reads X would.
#include <math.h>

#include "rf_device.cuh"
#include "rf_internal.h"

namespace rf {
namespace {

// ------------------------------------------------------------------ kernel 1

constexpr int kQuantWarps = 4;
constexpr int kVecPerLaneMax = 16;   // rows up to 32 * 16 * 8 = 4096 elements stay in registers

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

// Rows of up to 4096 elements: one warp per row, the row held in registers
// (16 x 16-byte loads per lane).  Memory parallelism comes from occupancy:
// four 4-warp CTAs per SM, each warp with its whole row in flight.
__global__ void __launch_bounds__(kQuantWarps * 32, 4)
    absmax_quant_regs_kernel(const uint4* __restrict__ X, uint8_t* __restrict__ Xq,
                             float* __restrict__ sx, int M, int K) {
  // the GEMM (a programmatic dependent) may be scheduled onto SMs this grid
  // leaves; it waits for this grid to finish before reading Xq or sx
  asm volatile("griddepcontrol.launch_dependents;");
  const int lane = threadIdx.x & 31;
  const int nw = gridDim.x * kQuantWarps;
  const int nvec = K >> 3;
  int row = blockIdx.x * kQuantWarps + (threadIdx.x >> 5);
  uint4 cur[kVecPerLaneMax];
  auto load = [&](uint4 (&v)[kVecPerLaneMax], int rr) {
    const uint4* xr = X + (size_t)rr * nvec;
#pragma unroll
    for (int i = 0; i < kVecPerLaneMax; ++i) {
      const int j = lane + 32 * i;
      v[i] = j < nvec ? __ldcs(xr + j) : make_uint4(0, 0, 0, 0);
    }
  };
  for (; row < M; row += nw) {
    load(cur, row);
    uint32_t amax = 0;
#pragma unroll
    for (int i = 0; i < kVecPerLaneMax; ++i) amax = max(amax, absmax_bits(cur[i]));
    const RowScale rs = row_scale(amax);
    if (lane == 0) sx[row] = rs.s;
    uint2* qr = reinterpret_cast<uint2*>(Xq + (size_t)row * K);
    if (rs.s == 0.f) {                                // all-zero row: codes 0x00
#pragma unroll
      for (int i = 0; i < kVecPerLaneMax; ++i)
        if (lane + 32 * i < nvec) qr[lane + 32 * i] = make_uint2(0, 0);
    } else if (rs.recip) {
#pragma unroll
      for (int i = 0; i < kVecPerLaneMax; ++i)
        if (lane + 32 * i < nvec) __stcs(qr + lane + 32 * i, quant8<true>(cur[i], rs.s, rs.r));
    } else {
#pragma unroll
      for (int i = 0; i < kVecPerLaneMax; ++i)
        if (lane + 32 * i < nvec) __stcs(qr + lane + 32 * i, quant8<false>(cur[i], rs.s, rs.r));
    }
  }
}

// Longer rows: two passes over the row (the second one hits L2).
__global__ void __launch_bounds__(kQuantWarps * 32)
    absmax_quant_long_kernel(const uint4* __restrict__ X, uint8_t* __restrict__ Xq,
                             float* __restrict__ sx, int M, int K) {
  asm volatile("griddepcontrol.launch_dependents;");
  const int lane = threadIdx.x & 31;
  const int row = blockIdx.x * kQuantWarps + (threadIdx.x >> 5);
  if (row >= M) return;
  const int nvec = K >> 3;
  const uint4* xr = X + (size_t)row * nvec;
  uint2* qr = reinterpret_cast<uint2*>(Xq + (size_t)row * K);
  uint32_t amax = 0;
  for (int j = lane; j < nvec; j += 32) amax = max(amax, absmax_bits(__ldg(xr + j)));
  const RowScale rs = row_scale(amax);
  if (lane == 0) sx[row] = rs.s;
  for (int j = lane; j < nvec; j += 32) {
    if (rs.s == 0.f)
      qr[j] = make_uint2(0, 0);
    else
      qr[j] = rs.recip ? quant8<true>(__ldg(xr + j), rs.s, rs.r)
                       : quant8<false>(__ldg(xr + j), rs.s, rs.r);
  }
}

// ------------------------------------------------------------------ kernel 2

constexpr int BM = 128, BN = 256, BK = 128;      // BK bytes = one 128-byte swizzle row
constexpr int kStages = 4;
constexpr int kABytes = BM * BK, kBBytes = BN * BK, kStageBytes = kABytes + kBBytes;
constexpr int kBHalfBytes = kBBytes / 2;         // the part of B one CTA of a pair loads
constexpr int kGemmThreads = 192;                // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kEpiThreads = 128;
constexpr int kAccCols = BN;                     // one fp32 accumulator tile in TMEM
constexpr int kTmemCols = 2 * kAccCols;          // two: epilogue of tile i overlaps tile i+1
constexpr int kGemmSmem = kStages * kStageBytes + 1024 /*align*/ + 256 /*bars*/;
constexpr uint32_t kIdescF8 = make_idesc(BM, BN, /*e4m3*/ 0, 0, 0);
constexpr uint16_t kPairMask = 0x3;

struct GemmBars {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint32_t tmem;
  int abort;
};

// Persistent, clusters of two CTAs.  The pair shares each 256-column B tile:
// CTA r loads B rows n0 + 128 r .. + 127 and multicasts them to both CTAs, so
// each SM pulls 32 KB (A 16 KB + half of B) per k-block from L2 instead of
// 48 KB.  Pair p of the tile grid covers output rows 256 mp .. + 255 (CTA r
// takes rows 256 mp + 128 r) and columns 256 nb; cluster c handles pairs
// c, c + nclusters, ...  The MMA thread accumulates tile i into TMEM buffer
// i % 2 while the epilogue warps drain buffer (i - 1) % 2.  A stage is
// refilled only after the MMAs of both CTAs have read it (each MMA thread
// commits to the "empty" barrier of both CTAs).
__global__ void __launch_bounds__(kGemmThreads, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const float* __restrict__ sx, const float* __restrict__ sw,
                    __nv_bfloat16* __restrict__ Y, int M, int N, int K, int tiles_n, int num_pairs,
                    unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  GemmBars* bars = reinterpret_cast<GemmBars*>(smem + kStages * kStageBytes);
  volatile int* abort_flag = &bars->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int crank = (int)cluster_ctarank();
  const int cid = (int)blockIdx.x >> 1, ncl = (int)gridDim.x >> 1;
  const int nk = (K + BK - 1) / BK;
  const int my_tiles = num_pairs > cid ? (num_pairs - cid + ncl - 1) / ncl : 0;

  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&bars->full[i]), 1);
      mbar_init(smem_u32(&bars->empty[i]), 2);      // both CTAs' MMAs release a stage
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars->acc_full[i]), 1);
      mbar_init(smem_u32(&bars->acc_empty[i]), kEpiThreads);
    }
    mbar_init(smem_u32(&bars->drain), 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&bars->tmem), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync();            // both CTAs' barriers exist before any multicast
  tc_fence_after();
  const uint32_t tmem = bars->tmem;
  // launched as a programmatic dependent of the quantisation kernel: the
  // prologue above overlapped its tail; Xq and sx are read only after this
  asm volatile("griddepcontrol.wait;" ::: "memory");

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      int it = 0;
      for (int i = 0; i < my_tiles && !*abort_flag; ++i) {
        const int p = cid + i * ncl;
        const int m0 = (p / tiles_n) * (2 * BM) + crank * BM, n0 = (p % tiles_n) * BN;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int slot = it % kStages;
          if (it >= kStages &&
              !mbar_wait(smem_u32(&bars->empty[slot]), (uint32_t)(((it / kStages) + 1) & 1))) {
            raise_error(err, kDevErrTimeout);
            *abort_flag = 1;
            break;
          }
          if (*abort_flag) break;
          uint8_t* a = smem + slot * kStageBytes;
          const uint32_t bar = smem_u32(&bars->full[slot]);
          mbar_arrive_expect_tx(bar, kStageBytes);   // A + both halves of B
          tma_load_2d(smem_u32(a), &tmA, bar, kb * BK, m0);
          tma_load_2d_mc(smem_u32(a + kABytes + crank * kBHalfBytes), &tmB, bar, kb * BK,
                         n0 + crank * (BN / 2), kPairMask);
        }
      }
      if (*abort_flag)   // let the copies this CTA waits for land before smem is released
        for (int j = it - kStages < 0 ? 0 : it - kStages; j < it; ++j)
          (void)mbar_wait(smem_u32(&bars->full[j % kStages]), (uint32_t)((j / kStages) & 1),
                          1000000ull);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer (one thread)
      int it = 0;
      bool ok = true;
      for (int i = 0; ok && i < my_tiles; ++i) {
        const int a = i & 1;
        if (i >= 2 && !mbar_wait(smem_u32(&bars->acc_empty[a]), (uint32_t)(((i >> 1) + 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + a * kAccCols;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int slot = it % kStages;
          if (!mbar_wait(smem_u32(&bars->full[slot]), (uint32_t)((it / kStages) & 1)) ||
              *abort_flag) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + slot * kStageBytes);
          const uint32_t sb = sa + kABytes;
#pragma unroll
          for (int k = 0; k < BK / 32; ++k)
            mma_f8_ss(d, sw128_desc(sa + k * 32, 1024, 16), sw128_desc(sb + k * 32, 1024, 16),
                      kIdescF8, (kb | k) != 0);
          mma_commit_mc(smem_u32(&bars->empty[slot]), kPairMask);
        }
        if (ok) mma_commit(smem_u32(&bars->acc_full[a]));
      }
      if (!ok) {
        raise_error(err, kDevErrTimeout);
        *abort_flag = 1;
      }
      // nothing may still run on the tensor core when TMEM is released
      mma_commit(smem_u32(&bars->drain));
      (void)mbar_wait(smem_u32(&bars->drain), 0, 1000000000ull);
    }
  } else {
    // ---------------- epilogue: TMEM -> registers -> scale -> bf16 -> global
    const int sub = warp & 3;                    // TMEM lane quarter of this warp
    const uint32_t lane_off = (uint32_t)(sub * 32) << 16;
    const bool vec_ok = (N % 8) == 0;
    for (int i = 0; i < my_tiles; ++i) {
      const int a = i & 1;
      const int p = cid + i * ncl;
      const int m0 = (p / tiles_n) * (2 * BM) + crank * BM, n0 = (p % tiles_n) * BN;
      const int row = m0 + sub * 32 + lane;
      const bool got = mbar_wait(smem_u32(&bars->acc_full[a]), (uint32_t)((i >> 1) & 1));
      if (!__all_sync(0xffffffffu, got && !*abort_flag)) {
        raise_error(err, kDevErrTimeout);
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const float srow = (row < M) ? sx[row] : 0.f;
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
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
        if (row < M) {
          __nv_bfloat16* yp = Y + (size_t)row * N + n0 + c0;
          if (vec_ok && full_chunk) {
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
      mbar_arrive(smem_u32(&bars->acc_empty[a]));   // buffer a may be overwritten
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  // the peer may still multicast into this CTA or arrive on its barriers
  // until both are done
  cluster_sync();
}

}  // namespace

size_t fp8_workspace_bytes(int M, int N, int K) {
  (void)N;
  const size_t xq = ((size_t)M * K + 255) & ~(size_t)255;
  return xq + (size_t)M * sizeof(float);
}

cudaError_t launch_absmax_fp8_gemm(const void* X, const uint8_t* Wq, const float* sw, void* Y,
                                   int M, int N, int K, float* sx, uint8_t* xq, unsigned* err,
                                   cudaStream_t s) {
  // kernel 1: absmax + quantisation
  const int qblocks = (M + kQuantWarps - 1) / kQuantWarps;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidValue;
  if (K <= 32 * kVecPerLaneMax * 8) {
    const int resident = 4 * sms;                      // four 4-warp CTAs per SM
    absmax_quant_regs_kernel<<<qblocks < resident ? qblocks : resident, kQuantWarps * 32, 0, s>>>(
        static_cast<const uint4*>(X), xq, sx, M, K);
  } else {
    absmax_quant_long_kernel<<<qblocks, kQuantWarps * 32, 0, s>>>(
        static_cast<const uint4*>(X), xq, sx, M, K);
  }
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  // kernel 2: FP8 GEMM with dequantising epilogue
  CUtensorMap tmA, tmB;
  if (!encode_tmap_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, (uint64_t)K, (uint64_t)M,
                      (uint64_t)K, BK, BM, true) ||
      !encode_tmap_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, Wq, (uint64_t)K, (uint64_t)N,
                      (uint64_t)K, BK, BN / 2, true))
    return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(fp8_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
  if (e != cudaSuccess) return e;
  const int tiles_n = (N + BN - 1) / BN;
  const int64_t pairs = (int64_t)tiles_n * ((M + 2 * BM - 1) / (2 * BM));
  if (pairs >= (1ll << 30)) return cudaErrorInvalidValue;
  const int clusters = (int)(pairs < sms / 2 ? pairs : sms / 2);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * (clusters > 0 ? clusters : 1), 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = kGemmSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, fp8_gemm_kernel, tmA, tmB, static_cast<const float*>(sx), sw,
                            static_cast<__nv_bfloat16*>(Y), M, N, K, tiles_n, (int)pairs, err);
}

}  // namespace rf
