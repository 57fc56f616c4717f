// fp8_gemm.cu -- dynamic FP8 quantised GEMM: row absmax -> E4M3 quantisation
// -> FP8 GEMM -> dequantisation ([E] §4.3, read per row of X).
//
// The cascade has a hard dependency: no element can be rounded before the
// max of its whole row is known, and the rounding is not linear, so the max
// cannot be folded into the GEMM loop incrementally the way the softmax max
// can.  It therefore runs as two cooperating kernels ([E] §3.3 multi-kernel
// level):
//   1. absmax_quant_kernel: one warp per row of X reads the row once into
//      registers, reduces |x| to the row max, sets sx = max / 448 (IEEE fp32
//      division) and writes the E4M3 codes of x / sx (IEEE division, then
//      cvt.rn.satfinite) plus sx.  X is read from HBM once.
//   2. fp8_gemm_kernel: a tcgen05 GEMM (kind::f8f6f4, E4M3 x E4M3 -> fp32 in
//      tensor memory) over TMA-staged 128-byte-swizzled tiles, warp
//      specialised (TMA producer warp, single-thread MMA issuer, four
//      epilogue warps), whose epilogue applies sx[m] * sw[n] and rounds to
//      bf16.  The codes travel through HBM as 1 byte per element, half the
//      size of the bf16 input, so the pair moves as many bytes as a fused
//      kernel that re-reads X would.
#include <math.h>

#include "rf_device.cuh"
#include "rf_internal.h"

namespace rf {
namespace {

// ------------------------------------------------------------------ kernel 1

constexpr int kQuantWarps = 8;
constexpr int kVecPerLaneMax = 16;   // rows up to 32 * 16 * 8 = 4096 elements stay in registers

__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// 8 bf16 (one 16-byte vector) -> 8 E4M3 codes (little-endian in a uint2).
__device__ __forceinline__ uint2 quant8(const uint4 v, float s) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t c[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) c[i] = cvt_e4m3x2(__fdiv_rn(bf16lo(w[i]), s), __fdiv_rn(bf16hi(w[i]), s));
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

__device__ __forceinline__ uint32_t absmax_bits(const uint4 v) {
  // |bf16| ordering equals the ordering of its bits with the sign cleared;
  // __vmaxu2 takes the max of each 16-bit half separately
  const uint32_t a = __vmaxu2(v.x & 0x7FFF7FFFu, v.y & 0x7FFF7FFFu);
  const uint32_t b = __vmaxu2(v.z & 0x7FFF7FFFu, v.w & 0x7FFF7FFFu);
  const uint32_t c = __vmaxu2(a, b);
  return max(c & 0xFFFFu, c >> 16);
}

template <bool kInRegs>
__global__ void __launch_bounds__(kQuantWarps * 32)
    absmax_quant_kernel(const uint4* __restrict__ X, uint8_t* __restrict__ Xq,
                        float* __restrict__ sx, int M, int K) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kQuantWarps + warp;
  if (row >= M) return;
  const int nvec = K >> 3;
  const uint4* xr = X + (size_t)row * nvec;
  uint2* qr = reinterpret_cast<uint2*>(Xq + (size_t)row * K);

  uint32_t amax = 0;
  uint4 v[kInRegs ? kVecPerLaneMax : 1];
  if (kInRegs) {
#pragma unroll
    for (int i = 0; i < kVecPerLaneMax; ++i) {
      const int j = lane + 32 * i;
      v[i] = j < nvec ? __ldcs(xr + j) : make_uint4(0, 0, 0, 0);
      amax = max(amax, absmax_bits(v[i]));
    }
  } else {
    for (int j = lane; j < nvec; j += 32) amax = max(amax, absmax_bits(__ldg(xr + j)));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, o));

  const float a = __uint_as_float(amax << 16);
  const float s = __fdiv_rn(a, 448.0f);
  if (lane == 0) sx[row] = s;

  if (s == 0.f) {   // all-zero row: codes 0x00
    for (int j = lane; j < nvec; j += 32) qr[j] = make_uint2(0, 0);
    return;
  }
  if (kInRegs) {
#pragma unroll
    for (int i = 0; i < kVecPerLaneMax; ++i) {
      const int j = lane + 32 * i;
      if (j < nvec) qr[j] = quant8(v[i], s);
    }
  } else {
    for (int j = lane; j < nvec; j += 32) qr[j] = quant8(__ldg(xr + j), s);
  }
}

// ------------------------------------------------------------------ kernel 2

constexpr int BM = 128, BN = 256, BK = 128;      // BK bytes = one 128-byte swizzle row
constexpr int kStages = 4;
constexpr int kABytes = BM * BK, kBBytes = BN * BK, kStageBytes = kABytes + kBBytes;
constexpr int kGemmThreads = 192;                // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kTmemCols = 256;
constexpr int kGemmSmem = kStages * kStageBytes + 1024 /*align*/ + 256 /*bars*/ + BN * 4;
constexpr uint32_t kIdescF8 = make_idesc(BM, BN, /*e4m3*/ 0, 0, 0);

__global__ void __launch_bounds__(kGemmThreads, 1)
    fp8_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const float* __restrict__ sx, const float* __restrict__ sw,
                    __nv_bfloat16* __restrict__ Y, int M, int N, int K, unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* accum = empty + kStages;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(accum + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  float* sw_s = reinterpret_cast<float*>(smem + kStages * kStageBytes + 256);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * BN, m0 = blockIdx.y * BM;
  const int nk = (K + BK - 1) / BK;

  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 1);
    }
    mbar_init(smem_u32(accum), 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), kTmemCols);
    tmem_relinquish();
  }
  if (warp >= 2) {
    for (int j = threadIdx.x - 64; j < BN; j += 128) sw_s[j] = (n0 + j < N) ? sw[n0 + j] : 0.f;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------- TMA producer
      int kb = 0;
      for (; kb < nk; ++kb) {
        const int slot = kb % kStages;
        if (kb >= kStages &&
            !mbar_wait(smem_u32(&empty[slot]), (uint32_t)(((kb / kStages) + 1) & 1))) {
          raise_error(err, kDevErrTimeout);
          *abort_flag = 1;
          break;
        }
        if (*abort_flag) break;
        uint8_t* a = smem + slot * kStageBytes;
        const uint32_t bar = smem_u32(&full[slot]);
        mbar_arrive_expect_tx(bar, kStageBytes);
        tma_load_2d(smem_u32(a), &tmA, bar, kb * BK, m0);
        tma_load_2d(smem_u32(a + kABytes), &tmB, bar, kb * BK, n0);
      }
      if (*abort_flag) {
        // let the copies this thread issued land before shared memory is released
        for (int j = kb - kStages < 0 ? 0 : kb - kStages; j < kb; ++j)
          (void)mbar_wait(smem_u32(&full[j % kStages]), (uint32_t)((j / kStages) & 1), 1000000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------- MMA issuer (one thread)
      int kb = 0;
      for (; kb < nk; ++kb) {
        const int slot = kb % kStages;
        if (!mbar_wait(smem_u32(&full[slot]), (uint32_t)((kb / kStages) & 1))) {
          raise_error(err, kDevErrTimeout);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t a = smem_u32(smem + slot * kStageBytes);
        const uint32_t b = a + kABytes;
#pragma unroll
        for (int k = 0; k < BK / 32; ++k) {
          const uint64_t ad = sw128_desc(a + k * 32, 1024, 16);
          const uint64_t bd = sw128_desc(b + k * 32, 1024, 16);
          mma_f8_ss(tmem, ad, bd, kIdescF8, (kb | k) != 0);
        }
        mma_commit(smem_u32(&empty[slot]));
      }
      // signals the epilogue once every MMA issued above has completed (also
      // after an abort, so that nothing is in flight when TMEM is released)
      mma_commit(smem_u32(accum));
    }
  } else {
    // ---------------- epilogue: TMEM -> registers -> scale -> bf16 -> global
    const int sub = warp & 3;                    // TMEM lane quarter of this warp
    const int row = m0 + sub * 32 + lane;
    const bool ok = mbar_wait(smem_u32(accum), 0);
    if (!ok) {
      raise_error(err, kDevErrTimeout);
      *abort_flag = 1;
    }
    tc_fence_after();
    const float srow = (row < M) ? sx[row] : 0.f;
    const bool vec_ok = (N % 8) == 0;
    if (ok && !*abort_flag) {
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        if (n0 + c0 >= N) break;
        uint32_t r[32];
        tmem_ld32(tmem + ((uint32_t)(sub * 32) << 16) + c0, r);
        tmem_ld_wait();
        uint32_t packed[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float y0 = __uint_as_float(r[2 * j]) * srow * sw_s[c0 + 2 * j];
          const float y1 = __uint_as_float(r[2 * j + 1]) * srow * sw_s[c0 + 2 * j + 1];
          packed[j] = pack_bf16x2(y0, y1);
        }
        if (row < M) {
          __nv_bfloat16* yp = Y + (size_t)row * N + n0 + c0;
          if (vec_ok && n0 + c0 + 32 <= N) {
            uint4* y4 = reinterpret_cast<uint4*>(yp);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              y4[q] = make_uint4(packed[4 * q], packed[4 * q + 1], packed[4 * q + 2],
                                 packed[4 * q + 3]);
          } else {
            for (int j = 0; j < 32 && n0 + c0 + j < N; ++j) {
              const uint32_t w = packed[j >> 1];
              const uint16_t h = (j & 1) ? (uint16_t)(w >> 16) : (uint16_t)(w & 0xFFFF);
              reinterpret_cast<uint16_t*>(yp)[j] = h;
            }
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
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
  if (K <= 32 * kVecPerLaneMax * 8)
    absmax_quant_kernel<true><<<qblocks, kQuantWarps * 32, 0, s>>>(
        static_cast<const uint4*>(X), xq, sx, M, K);
  else
    absmax_quant_kernel<false><<<qblocks, kQuantWarps * 32, 0, s>>>(
        static_cast<const uint4*>(X), xq, sx, M, K);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  // kernel 2: FP8 GEMM with dequantising epilogue
  CUtensorMap tmA, tmB;
  if (!encode_tmap_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, xq, (uint64_t)K, (uint64_t)M,
                      (uint64_t)K, BK, BM, true) ||
      !encode_tmap_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, Wq, (uint64_t)K, (uint64_t)N,
                      (uint64_t)K, BK, BN, true))
    return cudaErrorInvalidValue;
  e = cudaFuncSetAttribute(fp8_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
  if (e != cudaSuccess) return e;
  dim3 grid((N + BN - 1) / BN, (M + BM - 1) / BM);
  if (grid.y > 65535u) return cudaErrorInvalidValue;
  fp8_gemm_kernel<<<grid, kGemmThreads, kGemmSmem, s>>>(tmA, tmB, sx, sw,
                                                        static_cast<__nv_bfloat16*>(Y), M, N, K,
                                                        err);
  return cudaGetLastError();
}

}  // namespace rf
