// attn_two_pass_tc.cu -- single-segment attention in the non-incremental
// (two-pass) form on the tcgen05 tensor cores: bf16 in, fp32 accumulation and
// softmax state, bf16 out, d = 64, at most 256 keys.
//
// Safe-softmax cascade ([E] §2.2) without the incremental rescaling: [E] §5.2
// reports that short reductions are better served without the incremental
// form.  With at most two key tiles every score of a row fits in tensor
// memory at once, so the exact row maximum is taken over all keys first and
// every P is formed against it; O needs no rescale and is read from tensor
// memory once.
//
// One CTA per work item: 128 query rows of one (batch, head) against all of
// its key tiles of 128 (one or two).  Roles:
//   warp 0, one thread: TMA of the Q tile and of every K and V tile of the
//     item (no ring: each tile has a slot of its own);
//   warp 1, one thread: S_j = Q K_j^T (tcgen05 kind::f16, M=128, N=128, fp32
//     in tensor memory columns 128 j ..); once P is written, O = sum_j P_j V_j
//     (M=128, N=64, K=128; V as the MN-major B operand) into columns 0-63,
//     which S_0 no longer holds anything needed;
//   warps 2-5: one thread per query row: the row max over both S tiles, then
//     P = 2^(S c - m) (c = scale * log2 e) as bf16 in 128-byte-swizzled
//     K-major tiles (P_0 in a buffer of its own, P_1 over the K tiles, which
//     the S products have finished reading) and the row sum l; after the P.V
//     products, o / l as bf16 to global memory.
// Causal mask: row i reads keys j <= i + (Lk - Lq); a query tile walks only
// the key tiles its last row reads, keys past a row's diagonal get P = 0, a
// row that reads no key is written as zero, and within each (batch, head) the
// query tiles with the most key tiles are launched first.
//
// Every wait is bounded.  On a timeout the kernel records it in the device
// error word; before the CTA ends, thread 0 then waits (bounded) for the
// copies it issued, and tensor memory is released.
#include <math.h>

#include "rf_device.cuh"
#include "rf_internal.h"

namespace rf {
namespace {

constexpr int kD = 64;
constexpr int BQ = 128, BKV = 128;
constexpr int kMaxKv = 2;                             // key tiles of one item at most
constexpr int kTileBytes = 128 * kD * 2;              // 16 KB: 128 rows x 128 B
constexpr int kQOff = 0;
constexpr int kKOff = kQOff + kTileBytes;             // K_0, K_1; later P_1
constexpr int kVOff = kKOff + kMaxKv * kTileBytes;
constexpr int kPOff = kVOff + kMaxKv * kTileBytes;    // P_0: keys 0-63, 64-127 (16 KB each)
constexpr int kBarOff = kPOff + 2 * kTileBytes;
constexpr int kSmem = kBarOff + 256;
constexpr int kThreads = 192;                         // warp 0 TMA, 1 MMA, 2-5 softmax
constexpr int kTmemCols = 256;                        // S_0: 0-127 (later O: 0-63), S_1: 128-255
constexpr uint32_t kIdescS = make_idesc(BQ, BKV, /*bf16*/ 1, 0, 0);
constexpr uint32_t kIdescO = make_idesc(BQ, kD, /*bf16*/ 1, 0, /*V MN-major*/ 1);

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct Bars {
  uint64_t q_full;
  uint64_t k_full[kMaxKv], v_full[kMaxKv];
  uint64_t s_full[kMaxKv];  // S_j in tensor memory
  uint64_t p_full;          // every row's P written (count BQ)
  uint64_t o_full;          // O = sum_j P_j V_j in tensor memory
  uint64_t drain;
  uint32_t tmem;
  int abort;
};
static_assert(sizeof(Bars) <= 256, "barriers fit their slot");

// Work item it = slot * n_bh + bh: query tile qt of (batch, head) bh, with
// qt = slot (causal: the last tile first).  Rows are 2-D coordinates of the
// [B*H*L][64] tensor maps (row = bh * L + i).
struct Item {
  int qt;
  int nkv;                    // key tiles the tile's rows read (0: only zero rows)
  int32_t q_row0, kv_row0;    // first query row, first key row
};

template <bool kCausal>
__device__ __forceinline__ Item item_of(int it, int n_bh, int nq, int Lq, int Lk) {
  const int slot = it / n_bh, bh = it % n_bh;
  Item w;
  w.qt = kCausal ? nq - 1 - slot : slot;
  int keys = Lk;
  if (kCausal) {
    const int last_row = min(w.qt * BQ + BQ - 1, Lq - 1);
    keys = max(0, min(Lk, last_row + (Lk - Lq) + 1));
  }
  w.nkv = (keys + BKV - 1) / BKV;
  w.q_row0 = (int32_t)((int64_t)bh * Lq) + w.qt * BQ;
  w.kv_row0 = (int32_t)((int64_t)bh * Lk);
  return w;
}

template <bool kCausal>
__global__ void __launch_bounds__(kThreads, 2)
    attn_two_pass_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ O,
                         int Lq, int Lk, float c_log2, int n_bh, int nq, unsigned* err) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Bars* bars = reinterpret_cast<Bars*>(smem + kBarOff);
  volatile int* abort_flag = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Item w = item_of<kCausal>(blockIdx.x, n_bh, nq, Lq, Lk);
  const int nkv = w.nkv;

  if ((smem_u32(smem) & 1023u) != 0) {   // swizzled tiles need 1 KB alignment
    if (threadIdx.x == 0) raise_error(err, kDevErrLayout);
    return;
  }

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    mbar_init(smem_u32(&bars->q_full), 1);
    for (int i = 0; i < kMaxKv; ++i) {
      mbar_init(smem_u32(&bars->k_full[i]), 1);
      mbar_init(smem_u32(&bars->v_full[i]), 1);
      mbar_init(smem_u32(&bars->s_full[i]), 1);
    }
    mbar_init(smem_u32(&bars->p_full), BQ);
    mbar_init(smem_u32(&bars->o_full), 1);
    mbar_init(smem_u32(&bars->drain), 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&bars->tmem), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;

  if (warp == 0) {
    if (lane == 0 && nkv > 0) {
      // ------------------------------------------------ TMA producer
      const uint64_t pol_kv = policy_evict_last();   // K/V tiles are read by Lq/128 CTAs
      mbar_arrive_expect_tx(smem_u32(&bars->q_full), kTileBytes);
      tma_load_2d(smem_u32(smem + kQOff), &tmQ, smem_u32(&bars->q_full), 0, w.q_row0);
      for (int j = 0; j < nkv; ++j) {
        mbar_arrive_expect_tx(smem_u32(&bars->k_full[j]), kTileBytes);
        tma_load_2d_hint(smem_u32(smem + kKOff + j * kTileBytes), &tmK, smem_u32(&bars->k_full[j]),
                         0, w.kv_row0 + j * BKV, pol_kv);
        mbar_arrive_expect_tx(smem_u32(&bars->v_full[j]), kTileBytes);
        tma_load_2d_hint(smem_u32(smem + kVOff + j * kTileBytes), &tmV, smem_u32(&bars->v_full[j]),
                         0, w.kv_row0 + j * BKV, pol_kv);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && nkv > 0) {
      // ------------------------------------------------ MMA issuer
      const uint32_t q_addr = smem_u32(smem + kQOff);
      const uint32_t p_addr = smem_u32(smem + kPOff);
      bool ok = mbar_wait(smem_u32(&bars->q_full), 0);
      // every S tile first (S_j in columns 128 j ..)
      for (int j = 0; ok && j < nkv; ++j) {
        if (!mbar_wait(smem_u32(&bars->k_full[j]), 0)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t k_addr = smem_u32(smem + kKOff + j * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_bf16_ss(tmem + j * BKV, sw128_desc(q_addr + kk * 32, 1024, 16),
                      sw128_desc(k_addr + kk * 32, 1024, 16), kIdescS, kk != 0);
        mma_commit(smem_u32(&bars->s_full[j]));
      }
      // once the softmax warps have turned S into P: both P.V products into
      // one O accumulator in columns 0-63 (P_1 lies over the K tiles)
      if (ok) ok = mbar_wait(smem_u32(&bars->p_full), 0);
      for (int j = 0; ok && j < nkv; ++j) {
        if (!mbar_wait(smem_u32(&bars->v_full[j]), 0)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t pj = j == 0 ? p_addr : smem_u32(smem + kKOff);
        const uint32_t v_addr = smem_u32(smem + kVOff + j * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < BKV / 16; ++kk)
          mma_bf16_ss(tmem, sw128_desc(pj + (kk >> 2) * kTileBytes + (kk & 3) * 32, 1024, 16),
                      sw128_desc(v_addr + kk * 16 * 128, 1024, kTileBytes), kIdescO,
                      (j | kk) != 0);
      }
      if (ok) mma_commit(smem_u32(&bars->o_full));
      if (!ok) {
        raise_error(err, kDevErrTimeout);
        *abort_flag = 1;
      }
      // drain: nothing may still be running on the tensor core when tensor
      // memory and shared memory are released
      mma_commit(smem_u32(&bars->drain));
      (void)mbar_wait(smem_u32(&bars->drain), 0, 1000000000ull);
    }
  } else {
    // ------------------------------------------------ softmax / epilogue
    const int sub = warp & 3;
    const int r = sub * 32 + lane;                     // query row within the tile
    const uint32_t lane_off = (uint32_t)(sub * 32) << 16;
    const int qt = w.qt;
    const int off = Lk - Lq;                           // causal: row i reads keys <= i + off
    const uint64_t c2 = f2(c_log2, c_log2);
    uint64_t o2[kD / 2];                               // o as fp32 pairs
#pragma unroll
    for (int i = 0; i < kD / 2; ++i) o2[i] = 0ull;
    float l_run = 0.f;
    bool ok = true;
    if (nkv > 0) {
      // warp-uniform decisions: the tensor-memory loads are warp-collective
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->s_full[0]), 0) &&
                                       (nkv < 2 || mbar_wait(smem_u32(&bars->s_full[1]), 0)) &&
                                       !*abort_flag);
      if (ok) {
        tc_fence_after();
        // keys of tile j this row reads: a prefix of `valid[j]`; `full[j]`
        // (uniform over the CTA) when every row reads the whole tile
        int valid[kMaxKv];
        bool full[kMaxKv];
        // pass 1: the exact row max over every key the row reads
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < kMaxKv; ++j) {
          if (j >= nkv) break;
          valid[j] = min(BKV, Lk - j * BKV);
          full[j] = valid[j] == BKV;
          if (kCausal) {
            full[j] = full[j] && qt * BQ + off + 1 - j * BKV >= BKV;
            valid[j] = max(0, min(valid[j], qt * BQ + r + off + 1 - j * BKV));
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_off + j * BKV + q * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (full[j] || q * 32 + i < valid[j]) mx = fmaxf(mx, __uint_as_float(v[i]));
          }
        }
        const float m = mx * c_log2;
        const float m_use = m == -INFINITY ? 0.f : m;  // a row without keys: P = 0, not NaN
        const uint64_t negm2 = f2(-m_use, -m_use);
        // pass 2: P = 2^(S c - m) as swizzled bf16 tiles, row sum
        uint64_t sum2 = 0ull;
#pragma unroll
        for (int j = 0; j < kMaxKv; ++j) {
          if (j >= nkv) break;
          uint8_t* pr = smem + (j == 0 ? kPOff : kKOff) + r * 128;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_off + j * BKV + q * 32, v);
            tmem_ld_wait();
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float t0, t1;
              f2_split(ffma2(f2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])), c2,
                             negm2),
                       t0, t1);
              float p0 = ex2(t0), p1 = ex2(t1);
              if (!full[j]) {
                const int c0 = q * 32 + 2 * i;
                p0 = c0 < valid[j] ? p0 : 0.f;
                p1 = c0 + 1 < valid[j] ? p1 : 0.f;
              }
              sum2 = fadd2(sum2, f2(p0, p1));
              pk[i] = pack_bf16x2(p0, p1);
            }
            // keys 32q .. 32q+31 = block q/2, 16-byte chunks (q%2)*4 .. +3
            uint8_t* blk = pr + (q >> 1) * kTileBytes;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int chunk = (q & 1) * 4 + c;
              *reinterpret_cast<uint4*>(blk + ((chunk ^ (r & 7)) << 4)) =
                  make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            }
          }
        }
        float s_lo, s_hi;
        f2_split(sum2, s_lo, s_hi);
        l_run = s_lo + s_hi;
        fence_proxy_async_smem();                      // P visible to the tensor core
        tc_fence_before();                             // S reads ordered before the arrive
        mbar_arrive(smem_u32(&bars->p_full));
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->o_full), 0) && !*abort_flag);
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t v[32];
            tmem_ld32(tmem + lane_off + h * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 16; ++i)
              o2[h * 16 + i] = f2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
          }
        }
      }
    }
    const int row = qt * BQ + r;
    const int64_t o_first = ((int64_t)w.q_row0 + r) * kD;
    if (ok && row < Lq && RF_IN(err, o_first + kD - 1, (int64_t)n_bh * Lq * kD)) {
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;   // no key read: O = 0
      uint4* dst = reinterpret_cast<uint4*>(O + o_first);
#pragma unroll
      for (int c = 0; c < kD / 8; ++c) {
        float o[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) f2_split(o2[4 * c + e], o[2 * e], o[2 * e + 1]);
        dst[c] = make_uint4(pack_bf16x2(o[0] * inv, o[1] * inv), pack_bf16x2(o[2] * inv, o[3] * inv),
                            pack_bf16x2(o[4] * inv, o[5] * inv), pack_bf16x2(o[6] * inv, o[7] * inv));
      }
    }
    if (!ok) {
      raise_error(err, kDevErrTimeout);
      *abort_flag = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *abort_flag && nkv > 0) {
    // a wait gave up: the copies this CTA issued land (bounded) before its
    // shared memory is released
    (void)mbar_wait(smem_u32(&bars->q_full), 0, 1000000ull);
    for (int j = 0; j < nkv; ++j) {
      (void)mbar_wait(smem_u32(&bars->k_full[j]), 0, 1000000ull);
      (void)mbar_wait(smem_u32(&bars->v_full[j]), 0, 1000000ull);
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_attn_two_pass_tc(const void* Q, const void* K, const void* V, void* O, int B,
                                    int H, int Lq, int Lk, float scale, int causal, unsigned* err,
                                    cudaStream_t s) {
  if (Lk > kMaxKv * BKV) return cudaErrorInvalidValue;
  CUtensorMap tmQ, tmK, tmV;
  const uint64_t q_rows = (uint64_t)B * H * Lq, kv_rows = (uint64_t)B * H * Lk;
  if (!encode_tmap_2d(&tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Q, kD, q_rows, kD * 2, kD, BQ, true) ||
      !encode_tmap_2d(&tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, kD, kv_rows, kD * 2, kD, BKV, true) ||
      !encode_tmap_2d(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, V, kD, kv_rows, kD * 2, kD, BKV, true))
    return cudaErrorInvalidValue;
  auto kern = causal ? attn_two_pass_kernel<true> : attn_two_pass_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  const int nq = (Lq + BQ - 1) / BQ, n_bh = B * H;
  const int64_t items = (int64_t)nq * n_bh;             // one CTA each
  if (items <= 0 || items >= (1ll << 31)) return cudaErrorInvalidValue;
  const float c_log2 = scale * 1.4426950408889634f;
  kern<<<(int)items, kThreads, kSmem, s>>>(tmQ, tmK, tmV, static_cast<__nv_bfloat16*>(O), Lq, Lk,
                                           c_log2, n_bh, nq, err);
  return cudaGetLastError();
}

}  // namespace rf
