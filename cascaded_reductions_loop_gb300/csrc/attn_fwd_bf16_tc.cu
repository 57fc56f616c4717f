// attn_fwd_bf16_tc.cu -- single-segment fused attention on the tcgen05 tensor
// cores (bf16 in, fp32 accumulation and softmax state, bf16 out), d = 64.
//
// Safe-softmax cascade ([E] §2.2) in the single-loop incremental form ([E]
// §2.3, §4.1; [S] Methodologie 2, single-segment strategy of Methodologie 3):
// one CTA owns 128 query rows of one (batch, head) and walks all key tiles of
// 128 once.  Per tile j:
//   1. MMA warp:      S = Q K_j^T            (tcgen05 kind::f16, M=128, N=128,
//                                            fp32 in tensor memory)
//   2. softmax warps: one thread per query row reads its S row from TMEM,
//                     m' = max(m, rowmax), alpha = 2^(m - m'),
//                     P = 2^(S*c - m') (c = scale*log2 e), l' = alpha*l + sum P,
//                     and writes P as bf16 into a 128-byte-swizzled K-major
//                     shared tile (the A operand of the next MMA)
//   3. MMA warp:      O_j = P V_j            (M=128, N=64, K=128; V is the
//                                            MN-major B operand)
//   4. softmax warps: o = alpha*o + O_j in registers.
// After the last tile each thread writes o / l as bf16.  S and P never
// leave the SM.  A TMA warp streams Q once and K and V tiles through two
// 2-stage rings (a K slot is refilled as soon as its S product is done, a V
// slot after its P.V product); every wait is bounded.
//
// Pipelining: S is double-buffered in TMEM (tile j in columns 128 (j % 2) ..),
// and O_j is written into the first 64 columns of S_j's buffer once the
// softmax warps have read S_j.  The softmax warps fold O_{j-1} into o right
// after the max pass of tile j, so the tensor core computes P_{j-1} V_{j-1}
// during that pass, and S_{j+1} = Q K_{j+1}^T as soon as O_{j-1} has been
// read, while the exp pass of tile j runs.
//
// Causal mask: row i reads keys j <= i + (Lk - Lq).  A CTA walks only the
// key tiles its rows can read; tiles below the diagonal take the unmasked
// path, the diagonal tiles mask per element, and within each (batch, head)
// the query tiles with the most key tiles are launched first.  A row that
// reads no key is written as zero.
//
// Non-incremental (two-pass) mode, for Lk <= 256 ([E] §5.2 reports that short
// reductions are better served without the incremental form): both S tiles
// are computed into TMEM first, the exact row max over all keys is taken,
// then every P is formed against it, so O needs no rescale and is read from
// TMEM once.  P of the second tile is written over the K tiles, which the S
// products have finished reading.
//
// Two layouts: fixed-length [B][H][L][64] (2-D tensor maps over rows of 128
// bytes), and packed variable-length sequences [total][H][64] delimited by
// cumulative lengths cu_seqlens[B + 1] (3-D tensor maps over (dim, head,
// token) with a box of 64 x 1 x 128, which lands in shared memory exactly
// like the 2-D box).  Tiles that run past a sequence read the next
// sequence's tokens (or zeros past the end of the tensor) and are masked.
#include <math.h>

#include "rf_device.cuh"
#include "rf_internal.h"

namespace rf {
namespace {

constexpr int kD = 64;
constexpr int BQ = 128, BKV = 128;
constexpr int kKV = 2;                                // K/V ring depth
constexpr int kTileBytes = 128 * kD * 2;              // 16 KB: 128 rows x 128 B
constexpr int kQOff = 0;
constexpr int kKOff = kQOff + kTileBytes;
constexpr int kVOff = kKOff + kKV * kTileBytes;
constexpr int kPOff = kVOff + kKV * kTileBytes;       // two 16 KB blocks (keys 0-63, 64-127)
constexpr int kBarOff = kPOff + 2 * kTileBytes;
constexpr int kSmem = kBarOff + 256;
constexpr int kThreads = 192;                         // warp 0 TMA, 1 MMA, 2-5 softmax
constexpr int kTmemCols = 256;                        // S: cols 0-127, O_j: cols 128-191
constexpr uint32_t kIdescS = make_idesc(BQ, BKV, /*bf16*/ 1, 0, 0);
constexpr uint32_t kIdescO = make_idesc(BQ, kD, /*bf16*/ 1, 0, /*V MN-major*/ 1);

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct Bars {
  uint64_t q_full;
  uint64_t k_full[kKV], v_full[kKV];
  uint64_t k_empty[kKV], v_empty[kKV];
  uint64_t s_full[2];     // S_j in TMEM buffer j % 2
  uint64_t o_full[2];     // O_j in TMEM buffer j % 2 (columns 0-63)
  uint64_t o_free[2];     // O_j read by the softmax warps: the buffer may take S_{j+2}
  uint64_t p_full;        // P_j in shared memory
  uint64_t drain;
  uint32_t tmem;
  int abort;
};

// Sizes and addressing of the (sequence, head) a CTA works on.  Fixed
// layout: tile rows are 2-D coordinates (row = bh * L + i).  Varlen: 3-D
// coordinates (dim, head, token); sizes that contradict the host-side totals
// are reported and the sequence is skipped.
struct Seq {
  int Lq, Lk, h;
  int32_t q0, k0;       // first row (fixed) or first token (varlen)
  bool ok;
};

__device__ __forceinline__ Seq seq_of_cta(int Lq_, int Lk_, const int* cu_q, const int* cu_k,
                                          int H, int total_q, int total_k, unsigned* err) {
  Seq q;
  if (!cu_q) {
    const int64_t bh = blockIdx.y;
    q = {Lq_, Lk_, 0, (int32_t)(bh * Lq_), (int32_t)(bh * Lk_), true};
    return q;
  }
  const int b = blockIdx.y / H, h = blockIdx.y % H;
  const int q0 = cu_q[b], q1 = cu_q[b + 1], k0 = cu_k[b], k1 = cu_k[b + 1];
  q.ok = 0 <= q0 && q0 <= q1 && q1 <= total_q && q1 - q0 <= Lq_ && 0 <= k0 && k0 <= k1 &&
         k1 <= total_k;
  if (!q.ok) {
    if (threadIdx.x == 0 && blockIdx.x == 0) raise_error(err, kDevErrInput);
    return q;
  }
  q.Lq = q1 - q0;
  q.Lk = k1 - k0;
  q.h = h;
  q.q0 = q0;
  q.k0 = k0;
  return q;
}

// Output row `row` of the CTA's sequence (recomputed at the end rather than
// kept live through the key loop).
template <bool kVarlen>
__device__ __forceinline__ __nv_bfloat16* out_row(__nv_bfloat16* O, const int* cu_q, int Lq_,
                                                  int H, int row) {
  if (kVarlen) {
    const int b = blockIdx.y / H, h = blockIdx.y % H;
    return O + ((int64_t)(cu_q[b] + row) * H + h) * kD;
  }
  return O + ((int64_t)blockIdx.y * Lq_ + row) * kD;
}

template <bool kVarlen, bool kTwoPass, bool causal>
__global__ void __launch_bounds__(kThreads, 2)
    attn_fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ O,
                         int Lq_, int Lk_, float c_log2, const int* __restrict__ cu_q,
                         const int* __restrict__ cu_k, int H, int total_q, int total_k,
                         unsigned* err) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Bars* bars = reinterpret_cast<Bars*>(smem + kBarOff);
  volatile int* abort_flag = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // causal: heavier query tiles (more key tiles) first
  const int qt = causal ? (int)(gridDim.x - 1 - blockIdx.x) : (int)blockIdx.x;
  const Seq sq = seq_of_cta(Lq_, Lk_, kVarlen ? cu_q : nullptr, cu_k, H, total_q, total_k, err);
  if (!sq.ok || qt * BQ >= sq.Lq) return;           // uniform over the CTA, before any barrier
  const int Lq = sq.Lq, Lk = sq.Lk;
  const int off = Lk - Lq;                          // causal: row i reads keys <= i + off
  int nkv = (Lk + BKV - 1) / BKV;
  if (causal) {
    const int last_row = min(qt * BQ + BQ - 1, Lq - 1);
    const int keys = max(0, min(Lk, last_row + off + 1));
    nkv = (keys + BKV - 1) / BKV;
  }
  const int32_t q_row0 = sq.q0 + qt * BQ;           // row (fixed) or token (varlen)
  const int32_t kv_row0 = sq.k0;

  if ((smem_u32(smem) & 1023u) != 0) {   // swizzled tiles need 1 KB alignment
    if (threadIdx.x == 0) raise_error(err, kDevErrTimeout);
    return;
  }

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    mbar_init(smem_u32(&bars->q_full), 1);
    for (int i = 0; i < kKV; ++i) {
      mbar_init(smem_u32(&bars->k_full[i]), 1);
      mbar_init(smem_u32(&bars->v_full[i]), 1);
      mbar_init(smem_u32(&bars->k_empty[i]), 1);
      mbar_init(smem_u32(&bars->v_empty[i]), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars->s_full[i]), 1);
      mbar_init(smem_u32(&bars->o_full[i]), 1);
      mbar_init(smem_u32(&bars->o_free[i]), BQ);
    }
    mbar_init(smem_u32(&bars->p_full), BQ);
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
  const uint32_t tmem_s = tmem;                     // buffer b at columns 128 b

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      const uint64_t pol_kv = policy_evict_last();   // K/V tiles are read by Lq/128 CTAs
      mbar_arrive_expect_tx(smem_u32(&bars->q_full), kTileBytes);
      if (kVarlen)
        tma_load_3d(smem_u32(smem + kQOff), &tmQ, smem_u32(&bars->q_full), 0, sq.h, q_row0);
      else
        tma_load_2d(smem_u32(smem + kQOff), &tmQ, smem_u32(&bars->q_full), 0, q_row0);
      // one K or V tile of key tile j into ring slot j % kKV
      auto load = [&](const CUtensorMap* tm, int off, uint64_t* full, int j) {
        const int slot = j % kKV;
        const uint32_t bar = smem_u32(&full[slot]);
        mbar_arrive_expect_tx(bar, kTileBytes);
        if (kVarlen)
          tma_load_3d_hint(smem_u32(smem + off + slot * kTileBytes), tm, bar, 0, sq.h,
                           kv_row0 + j * BKV, pol_kv);
        else
          tma_load_2d_hint(smem_u32(smem + off + slot * kTileBytes), tm, bar, 0,
                           kv_row0 + j * BKV, pol_kv);
      };
      int nk = 0, nv = 0;                              // K / V tiles issued
      for (int j = 0; j < nkv && !*abort_flag; ++j) {
        const uint32_t ph = (uint32_t)(((j / kKV) + 1) & 1);
        if (j >= kKV && !mbar_wait(smem_u32(&bars->k_empty[j % kKV]), ph)) {
          *abort_flag = 1;
          break;
        }
        load(&tmK, kKOff, bars->k_full, j);
        ++nk;
        if (j >= kKV && !mbar_wait(smem_u32(&bars->v_empty[j % kKV]), ph)) {
          *abort_flag = 1;
          break;
        }
        load(&tmV, kVOff, bars->v_full, j);
        ++nv;
      }
      if (*abort_flag) {
        raise_error(err, kDevErrTimeout);
        // let the copies still in flight land before shared memory is released
        (void)mbar_wait(smem_u32(&bars->q_full), 0, 1000000ull);
        for (int i = nk - kKV < 0 ? 0 : nk - kKV; i < nk; ++i)
          (void)mbar_wait(smem_u32(&bars->k_full[i % kKV]), (uint32_t)((i / kKV) & 1), 1000000ull);
        for (int i = nv - kKV < 0 ? 0 : nv - kKV; i < nv; ++i)
          (void)mbar_wait(smem_u32(&bars->v_full[i % kKV]), (uint32_t)((i / kKV) & 1), 1000000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      const uint32_t q_addr = smem_u32(smem + kQOff);
      const uint32_t p_addr = smem_u32(smem + kPOff);
      // S_j = Q K_j^T into TMEM buffer j % 2; frees K slot j % kKV when done
      auto issue_s = [&](int j) -> bool {
        const int slot = j % kKV;
        if (!mbar_wait(smem_u32(&bars->k_full[slot]), (uint32_t)((j / kKV) & 1))) return false;
        tc_fence_after();
        const uint32_t k_addr = smem_u32(smem + kKOff + slot * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_bf16_ss(tmem_s + (j & 1) * BKV, sw128_desc(q_addr + kk * 32, 1024, 16),
                      sw128_desc(k_addr + kk * 32, 1024, 16), kIdescS, kk != 0);
        mma_commit(smem_u32(&bars->s_full[j & 1]));
        mma_commit(smem_u32(&bars->k_empty[slot]));
        return true;
      };
      bool ok = mbar_wait(smem_u32(&bars->q_full), 0);
      if constexpr (kTwoPass) {
        // every S tile first (tile j in TMEM columns 128 j ..), then, once the
        // softmax warps have turned S into P, both P.V products into one O
        // accumulator in columns 0-63 (S is no longer read by then)
        for (int j = 0; ok && j < nkv; ++j) ok = issue_s(j);
        if (ok && nkv > 0) {
          ok = mbar_wait(smem_u32(&bars->p_full), 0);
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
              mma_bf16_ss(tmem_s, sw128_desc(pj + (kk >> 2) * kTileBytes + (kk & 3) * 32, 1024, 16),
                          sw128_desc(v_addr + kk * 16 * 128, 1024, kTileBytes), kIdescO,
                          (j | kk) != 0);
          }
          if (ok) mma_commit(smem_u32(&bars->o_full[0]));
        }
      } else {
        if (nkv > 0) ok = ok && issue_s(0);
        if (nkv > 1) ok = ok && issue_s(1);
        for (int j = 0; ok && j < nkv; ++j) {
          const int slot = j % kKV;
          if (!mbar_wait(smem_u32(&bars->p_full), (uint32_t)(j & 1)) ||
              !mbar_wait(smem_u32(&bars->v_full[slot]), (uint32_t)((j / kKV) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          // O_j = P_j V_j into the first 64 columns of S_j's buffer (S_j has been read)
          const uint32_t v_addr = smem_u32(smem + kVOff + slot * kTileBytes);
#pragma unroll
          for (int kk = 0; kk < BKV / 16; ++kk)
            mma_bf16_ss(tmem_s + (j & 1) * BKV,
                        sw128_desc(p_addr + (kk >> 2) * kTileBytes + (kk & 3) * 32, 1024, 16),
                        sw128_desc(v_addr + kk * 16 * 128, 1024, kTileBytes), kIdescO, kk != 0);
          mma_commit(smem_u32(&bars->o_full[j & 1]));
          mma_commit(smem_u32(&bars->v_empty[slot]));
          if (j + 2 < nkv) {
            // the buffer takes S_{j+2} once the softmax warps have read O_j
            if (!mbar_wait(smem_u32(&bars->o_free[j & 1]), (uint32_t)((j >> 1) & 1))) {
              ok = false;
              break;
            }
            tc_fence_after();
            ok = issue_s(j + 2);
          }
        }
      }
      if (!ok) {
        raise_error(err, kDevErrTimeout);
        *abort_flag = 1;
      }
      // drain: nothing may still be running on the tensor core when TMEM and
      // shared memory are released
      mma_commit(smem_u32(&bars->drain));
      (void)mbar_wait(smem_u32(&bars->drain), 0, 1000000000ull);
    }
  } else {
    // ------------------------------------------------ softmax / epilogue
    const int sub = warp & 3;
    const int r = sub * 32 + lane;                     // query row within the tile
    const uint32_t lane_off = (uint32_t)(sub * 32) << 16;
    uint8_t* prow = smem + kPOff + r * 128;
    uint64_t o2[kD / 2];                               // o as fp32 pairs
#pragma unroll
    for (int i = 0; i < kD / 2; ++i) o2[i] = 0ull;
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    const uint64_t c2 = f2(c_log2, c_log2);

    if constexpr (kTwoPass) {
      // Non-incremental form for at most two key tiles: the exact row max over
      // every key first, then P = 2^(S c - m) for all keys (P of tile 0 in the
      // P buffer, of tile 1 over the consumed K tiles), one O with no rescale.
      if (nkv > 0) {
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->s_full[0]), 0) &&
                                         (nkv < 2 || mbar_wait(smem_u32(&bars->s_full[1]), 0)) &&
                                         !*abort_flag);
        if (ok) {
          tc_fence_after();
          int valid[2];
          bool full[2];
          float mx = -INFINITY;
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            if (j >= nkv) break;
            valid[j] = min(BKV, Lk - j * BKV);
            full[j] = valid[j] == BKV;
            if (causal) {
              full[j] = full[j] && qt * BQ + off + 1 - j * BKV >= BKV;
              valid[j] = max(0, min(valid[j], qt * BQ + r + off + 1 - j * BKV));
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t v[32];
              tmem_ld32(tmem_s + lane_off + j * BKV + q * 32, v);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i)
                if (full[j] || q * 32 + i < valid[j]) mx = fmaxf(mx, __uint_as_float(v[i]));
            }
          }
          const float m = mx * c_log2;
          const float m_use = m == -INFINITY ? 0.f : m;      // a row without keys
          const uint64_t negm2 = f2(-m_use, -m_use);
          uint64_t sum2 = 0ull;
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            if (j >= nkv) break;
            uint8_t* pr = smem + (j == 0 ? kPOff : kKOff) + r * 128;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              uint32_t v[32];
              tmem_ld32(tmem_s + lane_off + j * BKV + q * 32, v);
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
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->o_full[0]), 0) && !*abort_flag);
          if (ok) {
            tc_fence_after();
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              uint32_t v[32];
              tmem_ld32(tmem_s + lane_off + h * 32, v);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 16; ++i)
                o2[h * 16 + i] = f2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
            }
          }
        }
      }
    }

    // o = alpha * o + O_t for the tile t whose P.V product is in buffer t % 2
    auto fold_o = [&](int t, float alpha) -> bool {
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->o_full[t & 1]), (uint32_t)((t >> 1) & 1)) &&
                                       !*abort_flag))
        return false;
      tc_fence_after();
      const uint64_t a2 = f2(alpha, alpha);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t v[32];
        tmem_ld32(tmem_s + (t & 1) * BKV + lane_off + h * 32, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 16; ++i)
          o2[h * 16 + i] =
              ffma2(o2[h * 16 + i], a2, f2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])));
      }
      return true;
    };
    float alpha_prev = 0.f;
    for (int j = 0; !kTwoPass && j < nkv; ++j) {
      // warp-uniform decision: the TMEM loads below are warp-collective
      if (!__all_sync(0xffffffffu,
                      mbar_wait(smem_u32(&bars->s_full[j & 1]), (uint32_t)((j >> 1) & 1)) &&
                          !*abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t sbuf = tmem_s + (j & 1) * BKV + lane_off;
      int valid = min(BKV, Lk - j * BKV);              // keys of this tile that exist
      bool full = valid == BKV;                        // uniform over the CTA
      if (causal) {
        // every row of the CTA reads the whole tile iff its first row does
        full = full && qt * BQ + off + 1 - j * BKV >= BKV;
        valid = max(0, min(valid, qt * BQ + r + off + 1 - j * BKV));   // per row
      }
      // pass 1: row max of the raw scores (four independent max chains)
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t v[32];
        tmem_ld32(sbuf + q * 32, v);
        tmem_ld_wait();
        if (full) {
#pragma unroll
          for (int i = 0; i < 32; i += 2)
            mx4[(i >> 1) & 3] = fmax3(mx4[(i >> 1) & 3], __uint_as_float(v[i]), __uint_as_float(v[i + 1]));
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (q * 32 + i < valid) mx4[i & 3] = fmaxf(mx4[i & 3], __uint_as_float(v[i]));
        }
      }
      const float mx = fmaxf(fmax3(mx4[0], mx4[1], mx4[2]), mx4[3]);
      const float m_new = fmaxf(m_run, mx * c_log2);
      // -inf only while the row has read no key (a causal row above the
      // first visible key): then every P is masked to 0 and alpha is 0
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = ex2(m_run - m_use);          // 0 on the first tile
      const uint64_t negm2 = f2(-m_use, -m_use);
      // O_{j-1} (its P.V ran during the max pass); then its buffer may take
      // S_{j+1}, and P_{j-1} has been read, so P_j may overwrite it
      if (j > 0) {
        if (!fold_o(j - 1, alpha_prev)) {
          ok = false;
          break;
        }
        tc_fence_before();
        mbar_arrive(smem_u32(&bars->o_free[(j - 1) & 1]));
      }
      // pass 2: P = 2^(S c - m'), row sum (four independent chains), P ->
      // swizzled bf16 tile
      uint64_t sum4[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t v[32];
        tmem_ld32(sbuf + q * 32, v);
        tmem_ld_wait();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float t0, t1;
          f2_split(ffma2(f2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1])), c2, negm2),
                   t0, t1);
          float p0 = ex2(t0), p1 = ex2(t1);
          if (!full) {
            const int c0 = q * 32 + 2 * i;
            p0 = c0 < valid ? p0 : 0.f;
            p1 = c0 + 1 < valid ? p1 : 0.f;
          }
          sum4[i & 3] = fadd2(sum4[i & 3], f2(p0, p1));
          pk[i] = pack_bf16x2(p0, p1);
        }
        // keys 32q..32q+31 = block q/2, 16-byte chunks (q%2)*4 .. +3
        uint8_t* blk = prow + (q >> 1) * kTileBytes;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int chunk = (q & 1) * 4 + c;
          *reinterpret_cast<uint4*>(blk + ((chunk ^ (r & 7)) << 4)) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
      }
      float s_lo, s_hi;
      f2_split(fadd2(fadd2(sum4[0], sum4[1]), fadd2(sum4[2], sum4[3])), s_lo, s_hi);
      l_run = l_run * alpha + (s_lo + s_hi);
      m_run = m_new;
      alpha_prev = alpha;
      fence_proxy_async_smem();                        // P visible to the tensor core
      tc_fence_before();                               // S reads ordered before the arrive
      mbar_arrive(smem_u32(&bars->p_full));
    }
    if (!kTwoPass && ok && nkv > 0 && !fold_o(nkv - 1, alpha_prev)) ok = false;
    if (!ok) {
      raise_error(err, kDevErrTimeout);
      *abort_flag = 1;
    } else if (qt * BQ + r < Lq) {
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;   // no key read: O = 0
      uint4* dst = reinterpret_cast<uint4*>(out_row<kVarlen>(O, cu_q, Lq_, H, qt * BQ + r));
#pragma unroll
      for (int c = 0; c < kD / 8; ++c) {
        float o[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) f2_split(o2[4 * c + e], o[2 * e], o[2 * e + 1]);
        dst[c] = make_uint4(pack_bf16x2(o[0] * inv, o[1] * inv), pack_bf16x2(o[2] * inv, o[3] * inv),
                            pack_bf16x2(o[4] * inv, o[5] * inv), pack_bf16x2(o[6] * inv, o[7] * inv));
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

cudaError_t launch_attn_fwd_bf16_tc(const void* Q, const void* K, const void* V, void* O, int B,
                                    int H, int Lq, int Lk, int d, float scale, int causal,
                                    int two_pass, unsigned* err, cudaStream_t s) {
  (void)d;
  CUtensorMap tmQ, tmK, tmV;
  const uint64_t q_rows = (uint64_t)B * H * Lq, kv_rows = (uint64_t)B * H * Lk;
  if (!encode_tmap_2d(&tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Q, kD, q_rows, kD * 2, kD, BQ, true) ||
      !encode_tmap_2d(&tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, kD, kv_rows, kD * 2, kD, BKV, true) ||
      !encode_tmap_2d(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, V, kD, kv_rows, kD * 2, kD, BKV, true))
    return cudaErrorInvalidValue;
  if (two_pass && Lk > kKV * BKV) return cudaErrorInvalidValue;
  auto kern = two_pass ? (causal ? attn_fwd_bf16_kernel<false, true, true>
                                 : attn_fwd_bf16_kernel<false, true, false>)
                       : (causal ? attn_fwd_bf16_kernel<false, false, true>
                                 : attn_fwd_bf16_kernel<false, false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  dim3 grid((Lq + BQ - 1) / BQ, B * H);
  if (grid.y > 65535u) return cudaErrorInvalidValue;
  const float c_log2 = scale * 1.4426950408889634f;
  kern<<<grid, kThreads, kSmem, s>>>(tmQ, tmK, tmV, static_cast<__nv_bfloat16*>(O), Lq, Lk, c_log2,
                                     nullptr, nullptr, H, 0, 0, err);
  return cudaGetLastError();
}

cudaError_t launch_attn_fwd_bf16_tc_varlen(const void* Q, const void* K, const void* V, void* O,
                                           const int* cu_q, const int* cu_k, int B, int H,
                                           int max_q, int total_q, int total_k, float scale,
                                           int causal, unsigned* err, cudaStream_t s) {
  CUtensorMap tmQ, tmK, tmV;
  const uint64_t pitch = (uint64_t)H * kD * 2;     // bytes between tokens
  if (!encode_tmap_3d(&tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Q, kD, H, total_q, kD * 2, pitch,
                      kD, 1, BQ, true) ||
      !encode_tmap_3d(&tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, kD, H, total_k, kD * 2, pitch,
                      kD, 1, BKV, true) ||
      !encode_tmap_3d(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, V, kD, H, total_k, kD * 2, pitch,
                      kD, 1, BKV, true))
    return cudaErrorInvalidValue;
  auto kern = causal ? attn_fwd_bf16_kernel<true, false, true>
                     : attn_fwd_bf16_kernel<true, false, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  dim3 grid((max_q + BQ - 1) / BQ, B * H);
  if (grid.y > 65535u) return cudaErrorInvalidValue;
  const float c_log2 = scale * 1.4426950408889634f;
  kern<<<grid, kThreads, kSmem, s>>>(tmQ, tmK, tmV, static_cast<__nv_bfloat16*>(O), max_q, 0,
                                     c_log2, cu_q, cu_k, H, total_q, total_k, err);
  return cudaGetLastError();
}

}  // namespace rf
