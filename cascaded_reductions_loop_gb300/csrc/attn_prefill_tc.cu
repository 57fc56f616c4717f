// attn_prefill_tc.cu -- single-segment fused attention, fixed-length layout
// [B][H][L][64], no mask: the BERT-style prefill path (bf16 in, fp32
// accumulation and softmax state, bf16 out).
//
// Safe-softmax cascade ([E] §2.2) in the single-loop incremental form ([E]
// §2.3, §4.1; [S] Methodologie 2, single-segment strategy of Methodologie 3).
// One CTA per SM takes a pair of 128-row query tiles (a, b) of one (batch,
// head) at a time; both tiles read every key/value tile of that head, so K
// and V are loaded once for 256 query rows.  Per key tile j and query tile x:
//   1. MMA warp:   S_x = Q_x K_j^T              (tcgen05 kind::f16, M=128,
//                                               N=128, fp32 in tensor memory)
//   2. softmax warpgroup x (thread = query row): row max of its S_x row (read
//      from tensor memory); the running reference m moves only when the
//      tile's max exceeds it by more than kLazy (log2 units), and then O_x and
//      l are rescaled by 2^(m - m'); P = 2^(S*c - m) (c = scale * log2 e),
//      l += sum P; P is written as bf16 pairs over the first 64 columns of S_x
//   3. MMA warp:   O_x += P_x V_j               (M=128, N=64, K=128; P is the
//                                               tensor-memory A operand, V the
//                                               MN-major shared-memory B operand)
// After the last key tile the warpgroup reads O_x from tensor memory and
// writes O_x / l as bf16.  S, P and O never leave the SM.
//
// The MMA warp issues S_a, S_b, then for each tile P_a V, S_a(next), P_b V,
// S_b(next): the tensor core computes one query tile's products while the
// other warpgroup runs its exponentials.  The tensor core executes one
// thread's MMAs in issue order, so S_x(next) overwrites P_x only after P_x V
// has read it, and a completed S_x(j) implies a completed P_x V(j - 1).  Any
// reference m gives the same result ([S] Methodologie 1: the dependent
// factor 2^-m is invertible); with m at least the true running max minus
// kLazy, every P is at most 2^kLazy.
//
// A TMA warp loads the pair's Q tiles (two slots, so the next item's Q lands
// while the current one runs) and streams K and V tiles through kStages-deep
// rings.  Every wait is bounded.
#include <math.h>

#include "rf_device.cuh"
#include "rf_internal.h"

namespace rf {
namespace {

constexpr int kD = 64;
constexpr int BQ = 128, BKV = 128;
constexpr int kStages = 3;                            // K and V ring depth
constexpr int kTile = 128 * kD * 2;                   // 16 KB: 128 rows x 128 B
constexpr int kQOff = 0;                              // [slot][x] Q tiles
constexpr int kKOff = kQOff + 4 * kTile;
constexpr int kVOff = kKOff + kStages * kTile;
constexpr int kBarOff = kVOff + kStages * kTile;
constexpr int kSmem = kBarOff + 256 + 1024;           // + alignment slack
constexpr int kThreads = 320;                         // warp 0 TMA, 1 MMA, 2-5 / 6-9 softmax a / b
constexpr int kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128;          // S_x, fp32 (P_x as bf16 pairs in its first 64)
constexpr uint32_t kColO0 = 256, kColO1 = 320;        // O_x, fp32
constexpr uint32_t kIdescS = make_idesc(BQ, BKV, /*bf16*/ 1, 0, 0);
constexpr uint32_t kIdescO = make_idesc(BQ, kD, /*bf16*/ 1, 0, /*V MN-major*/ 1);
constexpr float kLazy = 8.f;                          // reference may trail the max by 2^8
static_assert(kSmem <= 227 * 1024, "shared memory");

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t col_s(int x) { return x ? kColS1 : kColS0; }
__device__ __forceinline__ uint32_t col_o(int x) { return x ? kColO1 : kColO0; }

struct Bars {
  uint64_t q_full[2], q_empty[2];                    // per Q slot (both tiles of an item)
  uint64_t k_full[kStages], k_empty[kStages];
  uint64_t v_full[kStages], v_empty[kStages];
  uint64_t s_full[2];                                // per query tile x: S_x complete
  uint64_t p_full[2];                                // per x: P_x written (128 arrivals)
  uint64_t o_done[2];                                // per x: the item's last P_x V complete
  uint64_t drain;
  uint32_t tmem;
  int abort;
};

// Item it = pair * n_bh + bh: query tiles 2 pair and 2 pair + 1 of (b, h) = bh.
struct Item {
  int bh, qa;
  bool has_b;
};

__device__ __forceinline__ Item item_of(int it, int n_bh, int nq) {
  Item w;
  w.bh = it % n_bh;
  w.qa = 2 * (it / n_bh);
  w.has_b = w.qa + 1 < nq;
  return w;
}

__global__ void __launch_bounds__(kThreads, 1)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, __nv_bfloat16* __restrict__ O,
                        int Lq, int Lk, float c_log2, int n_bh, int nq, unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + kBarOff);
  volatile int* abort_flag = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = n_bh * ((nq + 1) / 2);
  const int nkv = (Lk + BKV - 1) / BKV;

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars->q_full[i]), 1);
      mbar_init(smem_u32(&bars->q_empty[i]), 1);
      mbar_init(smem_u32(&bars->s_full[i]), 1);
      mbar_init(smem_u32(&bars->p_full[i]), BQ);
      mbar_init(smem_u32(&bars->o_done[i]), 1);
    }
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&bars->k_full[i]), 1);
      mbar_init(smem_u32(&bars->k_empty[i]), 1);
      mbar_init(smem_u32(&bars->v_full[i]), 1);
      mbar_init(smem_u32(&bars->v_empty[i]), 1);
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
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer
      const uint64_t pol_kv = policy_evict_last();   // K/V are read by every pair of the head
      bool ok = true;
      int ni = 0, g = 0;                             // items and K/V tiles issued
      for (int it = blockIdx.x; ok && it < n_items && !*abort_flag; it += gridDim.x, ++ni) {
        const Item w = item_of(it, n_bh, nq);
        const int slot = ni & 1;
        if (ni >= 2 &&
            !mbar_wait(smem_u32(&bars->q_empty[slot]), (uint32_t)(((ni >> 1) - 1) & 1))) {
          ok = false;
          break;
        }
        const uint32_t qb = smem_u32(&bars->q_full[slot]);
        mbar_arrive_expect_tx(qb, (w.has_b ? 2 : 1) * kTile);
        const int q_row = w.bh * Lq + w.qa * BQ;
        tma_load_2d(smem_u32(smem + kQOff + (2 * slot) * kTile), &tmQ, qb, 0, q_row);
        if (w.has_b) tma_load_2d(smem_u32(smem + kQOff + (2 * slot + 1) * kTile), &tmQ, qb, 0, q_row + BQ);
        const int kv_row = w.bh * Lk;
        for (int j = 0; j < nkv; ++j, ++g) {
          const int st = g % kStages;
          const uint32_t ph = (uint32_t)(((g / kStages) + 1) & 1);
          if (g >= kStages && !mbar_wait(smem_u32(&bars->k_empty[st]), ph)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(smem_u32(&bars->k_full[st]), kTile);
          tma_load_2d_hint(smem_u32(smem + kKOff + st * kTile), &tmK, smem_u32(&bars->k_full[st]), 0,
                           kv_row + j * BKV, pol_kv);
          if (g >= kStages && !mbar_wait(smem_u32(&bars->v_empty[st]), ph)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(smem_u32(&bars->v_full[st]), kTile);
          tma_load_2d_hint(smem_u32(smem + kVOff + st * kTile), &tmV, smem_u32(&bars->v_full[st]), 0,
                           kv_row + j * BKV, pol_kv);
        }
      }
      if (!ok || *abort_flag) {
        raise_error(err, kDevErrTimeout);
        *abort_flag = 1;
        // let the copies still in flight land before shared memory is released
        for (int i = ni - 2 < 0 ? 0 : ni - 2; i <= ni && i >= 0; ++i)
          (void)mbar_wait(smem_u32(&bars->q_full[i & 1]), (uint32_t)((i >> 1) & 1), 1000000ull);
        for (int i = g - kStages < 0 ? 0 : g - kStages; i < g; ++i) {
          (void)mbar_wait(smem_u32(&bars->k_full[i % kStages]), (uint32_t)((i / kStages) & 1), 1000000ull);
          (void)mbar_wait(smem_u32(&bars->v_full[i % kStages]), (uint32_t)((i / kStages) & 1), 1000000ull);
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      bool ok = true;
      int np[2] = {0, 0};                            // P tiles consumed per query tile
      // S_x(g) = Q_x K_g^T, Q from slot qs
      auto issue_s = [&](int x, int g, int qs) {
        const uint32_t qa = smem_u32(smem + kQOff + (2 * qs + x) * kTile);
        const uint32_t ka = smem_u32(smem + kKOff + (g % kStages) * kTile);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_bf16_ss(tmem + col_s(x), sw128_desc(qa + kk * 32, 1024, 16),
                      sw128_desc(ka + kk * 32, 1024, 16), kIdescS, kk != 0);
        mma_commit(smem_u32(&bars->s_full[x]));
      };
      // the softmax warpgroup has written P_x (and read S_x)
      auto wait_p = [&](int x) -> bool {
        if (!mbar_wait(smem_u32(&bars->p_full[x]), (uint32_t)(np[x] & 1))) return false;
        tc_fence_after();
        ++np[x];
        return true;
      };
      // O_x (+)= P_x V_g, P_x from the first 64 columns of S_x
      auto issue_pv = [&](int x, int g, bool first) {
        const uint32_t va = smem_u32(smem + kVOff + (g % kStages) * kTile);
#pragma unroll
        for (int kk = 0; kk < BKV / 16; ++kk)
          mma_bf16_ts(tmem + col_o(x), tmem + col_s(x) + kk * 8,
                      sw128_desc(va + kk * 16 * 128, 1024, kTile), kIdescO, (!first || kk != 0));
      };
      auto wait_kv = [&](uint64_t* full, int g) -> bool {
        if (!mbar_wait(smem_u32(&full[g % kStages]), (uint32_t)((g / kStages) & 1))) return false;
        tc_fence_after();
        return true;
      };
      int ni = 0, g = 0;
      int it = blockIdx.x;
      Item w = item_of(it, n_bh, nq);
      if (it < n_items) {
        ok = mbar_wait(smem_u32(&bars->q_full[0]), 0) && wait_kv(bars->k_full, 0);
        if (ok) {
          tc_fence_after();
          issue_s(0, 0, 0);
          if (w.has_b) issue_s(1, 0, 0);
          mma_commit(smem_u32(&bars->k_empty[0]));
        }
      }
      for (; ok && it < n_items; it += gridDim.x, ++ni) {
        const int qs = ni & 1;
        const int it_next = it + gridDim.x;
        const Item wn = item_of(it_next, n_bh, nq);
        for (int j = 0; ok && j < nkv; ++j, ++g) {
          const bool last = j == nkv - 1;
          // next tile: the same item's, or the next item's first
          const bool has_next = !last || it_next < n_items;
          const int qs_next = last ? qs ^ 1 : qs;
          const bool next_b = last ? wn.has_b : w.has_b;
          if (has_next && last &&
              !(ok = mbar_wait(smem_u32(&bars->q_full[qs_next]), (uint32_t)(((ni + 1) >> 1) & 1))))
            break;
          // query tile a: P.V, then its next S (which overwrites P_a)
          if (!(ok = wait_p(0) && wait_kv(bars->v_full, g))) break;
          issue_pv(0, g, j == 0);
          if (last) mma_commit(smem_u32(&bars->o_done[0]));
          if (has_next) {
            if (!(ok = wait_kv(bars->k_full, g + 1))) break;
            issue_s(0, g + 1, qs_next);
          }
          // query tile b likewise
          if (w.has_b) {
            if (!(ok = wait_p(1))) break;
            issue_pv(1, g, j == 0);
            if (last) mma_commit(smem_u32(&bars->o_done[1]));
          }
          if (has_next && next_b) issue_s(1, g + 1, qs_next);
          mma_commit(smem_u32(&bars->v_empty[g % kStages]));
          if (has_next) mma_commit(smem_u32(&bars->k_empty[(g + 1) % kStages]));
          if (last) mma_commit(smem_u32(&bars->q_empty[qs]));   // every S of the item issued
        }
        w = wn;
      }
      if (!ok) {
        raise_error(err, kDevErrTimeout);
        *abort_flag = 1;
      }
      // nothing may still run on the tensor core when TMEM and shared memory
      // are released
      mma_commit(smem_u32(&bars->drain));
      (void)mbar_wait(smem_u32(&bars->drain), 0, 1000000000ull);
    }
  } else {
    // ------------------------------------------------ softmax warpgroups
    const int x = warp >= 6 ? 1 : 0;                   // query tile of this warpgroup
    const int sub = warp & 3;                          // TMEM lane quarter
    const int r = sub * 32 + lane;                     // query row within the tile
    const uint32_t lane_off = (uint32_t)(sub * 32) << 16;
    const uint32_t s_addr = tmem + lane_off + col_s(x);
    const uint32_t o_addr = tmem + lane_off + col_o(x);
    const uint64_t c2 = f2(c_log2, c_log2);
    bool ok = true;
    int cnt = 0, icnt = 0;                             // tiles and items of this warpgroup
    for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
      const Item w = item_of(it, n_bh, nq);
      if (x == 1 && !w.has_b) continue;
      float m_ref = -INFINITY, l_run = 0.f;
      for (int j = 0; j < nkv; ++j, ++cnt) {
        // warp-uniform decision: the TMEM loads below are warp-collective
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->s_full[x]), (uint32_t)(cnt & 1)) &&
                                         !*abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int valid = min(BKV, Lk - j * BKV);      // keys of this tile that exist
        const bool full = valid == BKV;
        // the row's 128 scores read from tensor memory once (four loads in
        // flight together) and kept in registers for both passes
        uint32_t v[4][32];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld32(s_addr + q * 32, v[q]);
        tmem_ld_wait();
        // pass 1: row max (four independent chains)
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (full) {
#pragma unroll
            for (int i = 0; i < 32; i += 2)
              mx4[(i >> 1) & 3] =
                  fmax3(mx4[(i >> 1) & 3], __uint_as_float(v[q][i]), __uint_as_float(v[q][i + 1]));
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
              if (q * 32 + i < valid) mx4[i & 3] = fmaxf(mx4[i & 3], __uint_as_float(v[q][i]));
          }
        }
        const float mt = fmaxf(fmax3(mx4[0], mx4[1], mx4[2]), mx4[3]) * c_log2;
        float alpha = 1.f;
        bool need = false;
        if (j == 0) {
          m_ref = mt;                                   // P.V of tile 0 overwrites O
        } else if (mt > m_ref + kLazy) {
          alpha = ex2(m_ref - mt);
          l_run *= alpha;
          m_ref = mt;
          need = true;
        }
        const uint64_t negm2 = f2(-m_ref, -m_ref);
        // pass 2: P = 2^(S c - m) as bf16 pairs, row sum (four chains); P
        // goes over S columns 0-63, all of S being in registers by now
        uint64_t sum4[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t pk[32];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int q = 2 * hh + h;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              float t0, t1;
              f2_split(ffma2(f2(__uint_as_float(v[q][2 * i]), __uint_as_float(v[q][2 * i + 1])), c2,
                             negm2),
                       t0, t1);
              float p0 = ex2(t0), p1 = ex2(t1);
              if (!full) {
                const int c0 = q * 32 + 2 * i;
                p0 = c0 < valid ? p0 : 0.f;
                p1 = c0 + 1 < valid ? p1 : 0.f;
              }
              sum4[i & 3] = fadd2(sum4[i & 3], f2(p0, p1));
              pk[h * 16 + i] = pack_bf16x2(p0, p1);
            }
          }
          tmem_st32(s_addr + hh * 32, pk);
        }
        float s_lo, s_hi;
        f2_split(fadd2(fadd2(sum4[0], sum4[1]), fadd2(sum4[2], sum4[3])), s_lo, s_hi);
        l_run += s_lo + s_hi;
        // a moved reference: O_x (complete through the previous tile, since
        // S_x of this tile is) is rescaled before this tile's P.V adds to it
        if (__any_sync(0xffffffffu, need)) {
          uint32_t o[2][32];
          tmem_ld32(o_addr, o[0]);
          tmem_ld32(o_addr + 32, o[1]);
          tmem_ld_wait();
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int i = 0; i < 32; ++i) o[h][i] = __float_as_uint(__uint_as_float(o[h][i]) * alpha);
          tmem_st32(o_addr, o[0]);
          tmem_st32(o_addr + 32, o[1]);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(&bars->p_full[x]));
      }
      if (!ok) break;
      // epilogue: O_x / l -> bf16
      if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->o_done[x]), (uint32_t)(icnt & 1)) &&
                                       !*abort_flag)) {
        ok = false;
        break;
      }
      ++icnt;
      tc_fence_after();
      uint32_t v[2][32];
      tmem_ld32(o_addr, v[0]);
      tmem_ld32(o_addr + 32, v[1]);
      tmem_ld_wait();
      tc_fence_before();                               // O read before the next P.V may overwrite it
      const int row = (w.qa + x) * BQ + r;
      const int64_t o_first = ((int64_t)w.bh * Lq + row) * kD;
      if (row < Lq && RF_IN(err, o_first + kD - 1, (int64_t)n_bh * Lq * kD)) {
        const float inv = 1.f / l_run;
        uint4* dst = reinterpret_cast<uint4*>(O + o_first);
#pragma unroll
        for (int c = 0; c < kD / 8; ++c) {
          const uint32_t* u = &v[c >> 2][(c & 3) * 8];
          dst[c] = make_uint4(
              pack_bf16x2(__uint_as_float(u[0]) * inv, __uint_as_float(u[1]) * inv),
              pack_bf16x2(__uint_as_float(u[2]) * inv, __uint_as_float(u[3]) * inv),
              pack_bf16x2(__uint_as_float(u[4]) * inv, __uint_as_float(u[5]) * inv),
              pack_bf16x2(__uint_as_float(u[6]) * inv, __uint_as_float(u[7]) * inv));
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

}  // namespace

cudaError_t launch_attn_prefill_tc(const void* Q, const void* K, const void* V, void* O, int B,
                                   int H, int Lq, int Lk, float scale, unsigned* err,
                                   cudaStream_t s) {
  CUtensorMap tmQ, tmK, tmV;
  const uint64_t q_rows = (uint64_t)B * H * Lq, kv_rows = (uint64_t)B * H * Lk;
  if (!encode_tmap_2d(&tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Q, kD, q_rows, kD * 2, kD, BQ, true) ||
      !encode_tmap_2d(&tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, kD, kv_rows, kD * 2, kD, BKV, true) ||
      !encode_tmap_2d(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, V, kD, kv_rows, kD * 2, kD, BKV, true))
    return cudaErrorInvalidValue;
  cudaError_t e =
      cudaFuncSetAttribute(attn_prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  const int nq = (Lq + BQ - 1) / BQ, n_bh = B * H;
  const int64_t items = (int64_t)n_bh * ((nq + 1) / 2);
  const int sms = sm_count();
  if (sms <= 0 || items <= 0 || items >= (1ll << 31)) return cudaErrorInvalidValue;
  // persistent, one CTA per SM; every CTA takes the same number of items
  const int64_t per_cta = (items + sms - 1) / sms;
  const int grid = (int)((items + per_cta - 1) / per_cta);
  const float c_log2 = scale * 1.4426950408889634f;
  attn_prefill_kernel<<<grid, kThreads, kSmem, s>>>(tmQ, tmK, tmV, static_cast<__nv_bfloat16*>(O),
                                                    Lq, Lk, c_log2, n_bh, nq, err);
  return cudaGetLastError();
}

}  // namespace rf
