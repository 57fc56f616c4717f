// attn_fwd_bf16_tc.cu -- single-segment fused attention on the tcgen05 tensor
// cores (bf16 in, fp32 accumulation and softmax state, bf16 out), d = 64.
//
// The calls it serves: the non-incremental (two-pass) mode below.  The
// single-pass calls, fixed-length and packed, with or without the causal
// mask, go to attn_prefill_kernel (attn_prefill_tc.cu), which keeps two
// query tiles per CTA and issues their products from one thread each; the
// incremental path of this kernel (which the two-pass mode is built on) and
// its packed layout are no longer launched.
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
  uint64_t q_empty;       // every S product of the item has read Q
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

// A work item is one 128-row query tile of one (sequence, head): item it
// covers query tile qt of (sequence, head) bh, with it = slot * n_bh + bh and
// qt = slot (causal: the last tile first, so that the longest items start
// first).  Fixed layout: tile rows are 2-D coordinates (row = bh * L + i).
// Varlen: 3-D coordinates (dim, head, token); sizes that contradict the
// host-side totals are reported and the item is skipped.
struct Item {
  int Lq, Lk, h, qt, nkv;
  int32_t q_row0, kv_row0;   // first query row / first key row (fixed) or token (varlen)
  int64_t o_row0, o_stride;  // element offset of the item's first output row, row stride
  bool ok;                   // the item has rows to compute
};

template <bool kVarlen, bool causal>
__device__ __forceinline__ Item item_of(int it, int n_bh, int nq, int Lq_, int Lk_,
                                        const int* cu_q, const int* cu_k, int H, int total_q,
                                        int total_k, unsigned* err) {
  const int slot = it / n_bh, bh = it % n_bh;
  Item w;
  w.qt = causal ? nq - 1 - slot : slot;
  int32_t q0, k0;
  if (!kVarlen) {
    w.Lq = Lq_;
    w.Lk = Lk_;
    w.h = 0;
    q0 = (int32_t)((int64_t)bh * Lq_);
    k0 = (int32_t)((int64_t)bh * Lk_);
    w.o_row0 = (int64_t)q0 * kD;
    w.o_stride = kD;
    w.ok = true;
  } else {
    const int b = bh / H, h = bh % H;
    const bool cu_ok = RF_IN(err, b + 1, n_bh / H + 1);     // cu_q, cu_k have B + 1 entries
    const int a0 = cu_ok ? cu_q[b] : 0, a1 = cu_ok ? cu_q[b + 1] : 0;
    const int c0 = cu_ok ? cu_k[b] : 0, c1 = cu_ok ? cu_k[b + 1] : 0;
    w.ok = cu_ok && 0 <= a0 && a0 <= a1 && a1 <= total_q && a1 - a0 <= Lq_ && 0 <= c0 &&
           c0 <= c1 && c1 <= total_k;
    if (!w.ok) {
      if (threadIdx.x == 0 && w.qt == 0) raise_error(err, kDevErrInput);
      w.Lq = w.Lk = w.nkv = 0;
      return w;
    }
    w.Lq = a1 - a0;
    w.Lk = c1 - c0;
    w.h = h;
    q0 = a0;
    k0 = c0;
    w.o_row0 = ((int64_t)a0 * H + h) * kD;
    w.o_stride = (int64_t)H * kD;
  }
  w.ok = w.ok && w.qt * BQ < w.Lq;                 // a tile past the sequence has no rows
  w.nkv = (w.Lk + BKV - 1) / BKV;
  if (causal) {
    const int last_row = min(w.qt * BQ + BQ - 1, w.Lq - 1);
    const int keys = max(0, min(w.Lk, last_row + (w.Lk - w.Lq) + 1));
    w.nkv = (keys + BKV - 1) / BKV;
  }
  if (!w.ok) w.nkv = 0;
  w.q_row0 = q0 + w.qt * BQ;
  w.kv_row0 = k0;
  return w;
}

// Persistent: CTA c takes items c, c + gridDim.x, ...  Every role walks the
// same item sequence; K/V ring slots, S/O buffers and their barriers are
// indexed by a tile counter that runs on across items, so the pipeline does
// not drain between items, and the next item's Q is loaded as soon as the
// last S product of the current item has read Q.
template <bool kVarlen, bool kTwoPass, bool causal>
__global__ void __launch_bounds__(kThreads, 2)
    attn_fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmQ,
                         const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ O,
                         int Lq_, int Lk_, float c_log2, const int* __restrict__ cu_q,
                         const int* __restrict__ cu_k, int H, int total_q, int total_k,
                         int n_bh, int nq, unsigned* err) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Bars* bars = reinterpret_cast<Bars*>(smem + kBarOff);
  volatile int* abort_flag = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = n_bh * nq;
  auto item = [&](int it) {
    return item_of<kVarlen, causal>(it, n_bh, nq, Lq_, Lk_, cu_q, cu_k, H, total_q, total_k, err);
  };

  if ((smem_u32(smem) & 1023u) != 0) {   // swizzled tiles need 1 KB alignment
    if (threadIdx.x == 0) raise_error(err, kDevErrLayout);
    return;
  }

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    mbar_init(smem_u32(&bars->q_full), 1);
    mbar_init(smem_u32(&bars->q_empty), 1);
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
      int h = 0, kv_row0 = 0;
      // one K or V tile (global tile counter g, key tile j of the item) into slot g % kKV
      auto load = [&](const CUtensorMap* tm, int off, uint64_t* full, int g, int j) {
        const int slot = g % kKV;
        const uint32_t bar = smem_u32(&full[slot]);
        mbar_arrive_expect_tx(bar, kTileBytes);
        if (kVarlen)
          tma_load_3d_hint(smem_u32(smem + off + slot * kTileBytes), tm, bar, 0, h,
                           kv_row0 + j * BKV, pol_kv);
        else
          tma_load_2d_hint(smem_u32(smem + off + slot * kTileBytes), tm, bar, 0,
                           kv_row0 + j * BKV, pol_kv);
      };
      int nk = 0, nv = 0, nqi = 0;                     // K / V tiles and Q tiles issued
      for (int it = blockIdx.x; it < n_items && !*abort_flag; it += gridDim.x) {
        const Item w = item(it);
        if (w.nkv == 0) continue;
        // Q is the A operand of every S product of the previous item
        if (nqi > 0 && !mbar_wait(smem_u32(&bars->q_empty), (uint32_t)((nqi - 1) & 1))) {
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(smem_u32(&bars->q_full), kTileBytes);
        if (kVarlen)
          tma_load_3d(smem_u32(smem + kQOff), &tmQ, smem_u32(&bars->q_full), 0, w.h, w.q_row0);
        else
          tma_load_2d(smem_u32(smem + kQOff), &tmQ, smem_u32(&bars->q_full), 0, w.q_row0);
        ++nqi;
        h = w.h;
        kv_row0 = w.kv_row0;
        for (int j = 0; j < w.nkv; ++j) {
          const int g = nk;                            // == nv here
          const uint32_t ph = (uint32_t)(((g / kKV) + 1) & 1);
          if (g >= kKV && !mbar_wait(smem_u32(&bars->k_empty[g % kKV]), ph)) {
            *abort_flag = 1;
            break;
          }
          load(&tmK, kKOff, bars->k_full, g, j);
          ++nk;
          if (g >= kKV && !mbar_wait(smem_u32(&bars->v_empty[g % kKV]), ph)) {
            *abort_flag = 1;
            break;
          }
          load(&tmV, kVOff, bars->v_full, g, j);
          ++nv;
        }
      }
      if (*abort_flag) {
        raise_error(err, kDevErrTimeout);
        // let the copies still in flight land before shared memory is released
        if (nqi > 0) (void)mbar_wait(smem_u32(&bars->q_full), (uint32_t)((nqi - 1) & 1), 1000000ull);
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
      // S_g = Q K_g^T into TMEM buffer g % 2 (g: global tile counter) once the
      // buffer's previous O (tile g - 2) has been read; frees K slot g % kKV
      auto issue_s = [&](int g) -> bool {
        const int slot = g % kKV;
        if (g >= 2 && !mbar_wait(smem_u32(&bars->o_free[g & 1]), (uint32_t)(((g - 2) >> 1) & 1)))
          return false;
        if (!mbar_wait(smem_u32(&bars->k_full[slot]), (uint32_t)((g / kKV) & 1))) return false;
        tc_fence_after();
        const uint32_t k_addr = smem_u32(smem + kKOff + slot * kTileBytes);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_bf16_ss(tmem_s + (g & 1) * BKV, sw128_desc(q_addr + kk * 32, 1024, 16),
                      sw128_desc(k_addr + kk * 32, 1024, 16), kIdescS, kk != 0);
        mma_commit(smem_u32(&bars->s_full[g & 1]));
        mma_commit(smem_u32(&bars->k_empty[slot]));
        return true;
      };
      bool ok = true;
      int gk = 0, nqi = 0;
      for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
        const Item w = item(it);
        const int nkv = w.nkv;
        if (nkv == 0) continue;
        ok = mbar_wait(smem_u32(&bars->q_full), (uint32_t)(nqi & 1));
        ++nqi;
        if constexpr (kTwoPass) {
          // (one item per CTA) every S tile first (tile j in TMEM columns
          // 128 j ..), then, once the softmax warps have turned S into P,
          // both P.V products into one O accumulator in columns 0-63
          for (int j = 0; ok && j < nkv; ++j) ok = issue_s(j);
          if (ok) mma_commit(smem_u32(&bars->q_empty));
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
              mma_bf16_ss(tmem_s, sw128_desc(pj + (kk >> 2) * kTileBytes + (kk & 3) * 32, 1024, 16),
                          sw128_desc(v_addr + kk * 16 * 128, 1024, kTileBytes), kIdescO,
                          (j | kk) != 0);
          }
          if (ok) mma_commit(smem_u32(&bars->o_full[0]));
          gk += nkv;
        } else {
          const int g_last = gk + nkv - 1;
          if (ok) ok = issue_s(gk);
          if (ok && nkv > 1) ok = issue_s(gk + 1);
          if (ok && g_last <= gk + 1) mma_commit(smem_u32(&bars->q_empty));   // last S issued
          for (int j = 0; ok && j < nkv; ++j) {
            const int g = gk + j, slot = g % kKV;
            if (!mbar_wait(smem_u32(&bars->p_full), (uint32_t)(g & 1)) ||
                !mbar_wait(smem_u32(&bars->v_full[slot]), (uint32_t)((g / kKV) & 1))) {
              ok = false;
              break;
            }
            tc_fence_after();
            // O_g = P_g V_g into the first 64 columns of S_g's buffer (S_g has been read)
            const uint32_t v_addr = smem_u32(smem + kVOff + slot * kTileBytes);
#pragma unroll
            for (int kk = 0; kk < BKV / 16; ++kk)
              mma_bf16_ss(tmem_s + (g & 1) * BKV,
                          sw128_desc(p_addr + (kk >> 2) * kTileBytes + (kk & 3) * 32, 1024, 16),
                          sw128_desc(v_addr + kk * 16 * 128, 1024, kTileBytes), kIdescO, kk != 0);
            mma_commit(smem_u32(&bars->o_full[g & 1]));
            mma_commit(smem_u32(&bars->v_empty[slot]));
            if (j + 2 < nkv) {
              ok = issue_s(g + 2);
              if (ok && g + 2 == g_last) mma_commit(smem_u32(&bars->q_empty));
            }
          }
          gk += nkv;
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
    const uint64_t c2 = f2(c_log2, c_log2);
    bool ok = true;
    int gk = 0;
    for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
      const Item w = item(it);
      if (!w.ok) continue;
      const int nkv = w.nkv, Lk = w.Lk, qt = w.qt;
      const int off = w.Lk - w.Lq;                     // causal: row i reads keys <= i + off
      uint64_t o2[kD / 2];                             // o as fp32 pairs
#pragma unroll
      for (int i = 0; i < kD / 2; ++i) o2[i] = 0ull;
      float m_run = -INFINITY, l_run = 0.f;
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
        uint32_t v[2][32];                               // both halves in flight together
        tmem_ld32(tmem_s + (t & 1) * BKV + lane_off, v[0]);
        tmem_ld32(tmem_s + (t & 1) * BKV + lane_off + 32, v[1]);
        tmem_ld_wait();
  #pragma unroll
        for (int h = 0; h < 2; ++h) {
  #pragma unroll
          for (int i = 0; i < 16; ++i)
            o2[h * 16 + i] = ffma2(o2[h * 16 + i], a2,
                                   f2(__uint_as_float(v[h][2 * i]), __uint_as_float(v[h][2 * i + 1])));
        }
        return true;
      };
      float alpha_prev = 0.f;
      for (int j = 0; !kTwoPass && j < nkv; ++j) {
        // warp-uniform decision: the TMEM loads below are warp-collective
        const int g = gk + j;                            // tile counter across items
        if (!__all_sync(0xffffffffu,
                        mbar_wait(smem_u32(&bars->s_full[g & 1]), (uint32_t)((g >> 1) & 1)) &&
                            !*abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sbuf = tmem_s + (g & 1) * BKV + lane_off;
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
        for (int qq = 0; qq < 2; ++qq) {
          uint32_t v[2][32];                             // two 32-key blocks in flight together
          tmem_ld32(sbuf + (2 * qq) * 32, v[0]);
          tmem_ld32(sbuf + (2 * qq + 1) * 32, v[1]);
          tmem_ld_wait();
  #pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int q = 2 * qq + h;
            if (full) {
  #pragma unroll
              for (int i = 0; i < 32; i += 2)
                mx4[(i >> 1) & 3] =
                    fmax3(mx4[(i >> 1) & 3], __uint_as_float(v[h][i]), __uint_as_float(v[h][i + 1]));
            } else {
  #pragma unroll
              for (int i = 0; i < 32; ++i)
                if (q * 32 + i < valid) mx4[i & 3] = fmaxf(mx4[i & 3], __uint_as_float(v[h][i]));
            }
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
          if (!fold_o(g - 1, alpha_prev)) {
            ok = false;
            break;
          }
          tc_fence_before();
          mbar_arrive(smem_u32(&bars->o_free[(g - 1) & 1]));
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
      // O of the item's last tile; its buffer may then take the next item's S
      if (!kTwoPass && ok && nkv > 0) {
        if (!fold_o(gk + nkv - 1, alpha_prev)) {
          ok = false;
        } else {
          tc_fence_before();
          mbar_arrive(smem_u32(&bars->o_free[(gk + nkv - 1) & 1]));
        }
      }
      gk += nkv;
      if (!ok) break;
      const int64_t o_first = w.o_row0 + (int64_t)(qt * BQ + r) * w.o_stride;
      const int64_t n_o = kVarlen ? (int64_t)total_q * H * kD : (int64_t)n_bh * Lq_ * kD;
      if (qt * BQ + r < w.Lq && RF_IN(err, o_first + kD - 1, n_o)) {
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
    }
    if (!ok) {
      raise_error(err, kDevErrTimeout);
      *abort_flag = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Grid of the persistent kernel: two CTAs per SM; the items are spread so
// that every CTA takes the same number (ceil(items / slots)), which uses no
// more CTAs than needed.  (Fixed-length items have equal cost, or with the
// causal mask are paired heavy with light by the item order.)  The two-pass
// form and the variable-length layout take one item per CTA.
int persistent_grid(int64_t items, bool one_per_cta) {
  if (items <= 0 || items >= (1ll << 31)) return 0;
  if (one_per_cta) return (int)items;
  const int sms = sm_count();
  if (sms <= 0) return 0;
  const int64_t slots = 2ll * sms;
  const int64_t per_cta = (items + slots - 1) / slots;
  return (int)((items + per_cta - 1) / per_cta);
}

}  // namespace

cudaError_t launch_attn_fwd_bf16_tc(const void* Q, const void* K, const void* V, void* O, int B,
                                    int H, int Lq, int Lk, int d, float scale, int causal,
                                    int two_pass, unsigned* err, cudaStream_t s) {
  (void)d;
  if (!two_pass) return launch_attn_prefill_tc(Q, K, V, O, B, H, Lq, Lk, scale, causal, err, s);
  CUtensorMap tmQ, tmK, tmV;
  const uint64_t q_rows = (uint64_t)B * H * Lq, kv_rows = (uint64_t)B * H * Lk;
  if (!encode_tmap_2d(&tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Q, kD, q_rows, kD * 2, kD, BQ, true) ||
      !encode_tmap_2d(&tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, kD, kv_rows, kD * 2, kD, BKV, true) ||
      !encode_tmap_2d(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, V, kD, kv_rows, kD * 2, kD, BKV, true))
    return cudaErrorInvalidValue;
  if (Lk > kKV * BKV) return cudaErrorInvalidValue;
  auto kern = causal ? attn_fwd_bf16_kernel<false, true, true> : attn_fwd_bf16_kernel<false, true, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  const int nq = (Lq + BQ - 1) / BQ, n_bh = B * H;
  const int grid = persistent_grid((int64_t)nq * n_bh, two_pass != 0);
  if (grid <= 0) return cudaErrorInvalidValue;
  const float c_log2 = scale * 1.4426950408889634f;
  kern<<<grid, kThreads, kSmem, s>>>(tmQ, tmK, tmV, static_cast<__nv_bfloat16*>(O), Lq, Lk, c_log2,
                                     nullptr, nullptr, H, 0, 0, n_bh, nq, err);
  return cudaGetLastError();
}

cudaError_t launch_attn_fwd_bf16_tc_varlen(const void* Q, const void* K, const void* V, void* O,
                                           const int* cu_q, const int* cu_k, int B, int H,
                                           int max_q, int total_q, int total_k, float scale,
                                           int causal, unsigned* err, cudaStream_t s) {
  return launch_attn_prefill_tc_varlen(Q, K, V, O, cu_q, cu_k, B, H, max_q, total_q, total_k, scale,
                                       causal, err, s);
}

}  // namespace rf
