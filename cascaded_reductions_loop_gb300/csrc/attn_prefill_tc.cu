// attn_prefill_tc.cu -- single-segment fused attention, single pass, bf16 in,
// fp32 accumulation and softmax state, bf16 out: the BERT-style prefill path.
// Two layouts: fixed-length [B][H][L][64], and packed variable-length
// sequences [total][H][64] delimited by cumulative lengths (3-D tensor maps
// over (dim, head, token); one CTA per item, since items differ in cost).
// Under the causal mask row i reads keys j <= i + Lk - Lq of its sequence;
// each query tile reads only the key tiles its last row needs, scores of keys
// a row does not read are set to -inf (their P is 0), and a row that reads no
// key is written as zeros.
//
// Safe-softmax cascade ([E] §2.2) in the single-loop incremental form ([E]
// §2.3, §4.1; [S] Methodologie 2, single-segment strategy of Methodologie 3).
// One CTA per SM takes a pair of 128-row query tiles (a, b) of one (batch,
// head) at a time; both tiles read every key/value tile of that head, so K
// and V are loaded once for 256 query rows.  Per key tile j and query tile x:
//   1. MMA thread x: S_x = Q_x K_j^T           (tcgen05 kind::f16, M=128,
//                                               N=128, fp32 in tensor memory)
//   2. softmax warpgroup x (thread = query row): reads its 128 scores of S_x
//      into registers once (the MMA thread may then compute S_x(j+1) into
//      the same columns), takes the row max; the running reference m moves
//      only when the tile's max exceeds it by more than kLazy (log2 units),
//      and then O_x and l are rescaled by 2^(m - m'); P = 2^(S*c - m)
//      (c = scale * log2 e), l += sum P; P is written as bf16 pairs to
//      tensor-memory columns of its own once the previous P_x V has read them
//   3. MMA thread x: O_x += P_x V_j            (M=128, N=64, K=128; P is the
//                                               tensor-memory A operand, V the
//                                               MN-major shared-memory B operand)
// After the last key tile the warpgroup reads O_x from tensor memory, stages
// O_x / l as bf16 in shared memory and writes it with one bulk tensor store
// (a packed sequence's partial last tile: each thread stores its own row,
// since the box would run into the next sequence).  S, P and O never leave
// the SM.
//
// Each query tile has an MMA-issuing thread of its own, so one tile's
// products never wait behind the other tile's softmax; within a tile the
// next S is issued as soon as the current one has been read, the P.V as soon
// as P is written (at a pair's last key tile the P.V first, so O is complete
// early).  Tile b starts once tile a's softmax has taken its first row
// maxima, so the two softmax warpgroups run out of phase.  Any reference m
// gives the same result ([S] Methodologie 1: the dependent factor 2^-m is
// invertible); with m at least the true running max minus kLazy, every P is
// at most 2^kLazy.
//
// A TMA warp loads the pair's Q tiles (two slots, so the next item's Q lands
// while the current one runs) and streams K and V tiles through kStages-deep
// rings; both MMA threads release each stage.  Every wait is bounded.
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
constexpr int kStOff = kVOff + kStages * kTile;       // [x] O tiles staged for the bulk store
constexpr int kBarOff = kStOff + 2 * kTile;
constexpr int kSmem = kBarOff + 512 + 1024;           // + alignment slack
constexpr int kThreads = 352;   // warp 0 TMA, 1 / 10 MMA of tile a / b, 2-5 / 6-9 softmax a / b
constexpr int kMmaWarpB = 10;
constexpr int kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128;          // S_x, fp32
constexpr uint32_t kColO0 = 256, kColO1 = 320;        // O_x, fp32
constexpr uint32_t kColP0 = 384, kColP1 = 448;        // P_x, bf16 pairs
constexpr uint32_t kIdescS = make_idesc(BQ, BKV, /*bf16*/ 1, 0, 0);
constexpr uint32_t kIdescO = make_idesc(BQ, kD, /*bf16*/ 1, 0, /*V MN-major*/ 1);
constexpr float kLazy = 8.f;                          // reference may trail the max by 2^8
static_assert(kSmem <= 227 * 1024, "shared memory");
static_assert(kStOff % 1024 == 0, "staged O tiles on 1 KB (swizzle atom) boundaries");

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t col_s(int x) { return x ? kColS1 : kColS0; }
__device__ __forceinline__ uint32_t col_o(int x) { return x ? kColO1 : kColO0; }
__device__ __forceinline__ uint32_t col_p(int x) { return x ? kColP1 : kColP0; }

struct Bars {
  uint64_t q_full[2], q_empty[2];                    // per Q slot (both tiles of an item)
  uint64_t k_full[kStages], k_empty[kStages];
  uint64_t v_full[kStages], v_empty[kStages];
  uint64_t s_full[2];                                // per query tile x: S_x complete
  uint64_t s_read[2];                                // per x: S_x is in the softmax registers (4 warps)
  uint64_t p_full[2];                                // per x: P_x written (128 arrivals)
  uint64_t pv_done[2];                               // per x: the last P_x V has completed
  uint64_t o_done[2];                                // per x: the item's last P_x V complete
  uint64_t drain[2];                                 // per issuer: its MMAs have completed
  uint64_t st_full[2];                               // per x: the staged O tile is written (4 warps)
  uint64_t st_free[2];                               // per x: the last bulk store has read it
  uint64_t a_max0;                                   // tile a's first row maxima are taken (4 warps)
  uint32_t tmem;
  int abort;
};

// Item it = pair * n_bh + bh: query tiles 2 pair and 2 pair + 1 of (b, h) = bh.
__host__ __device__ __forceinline__ int n_items_of(int n_bh, int nq) {
  return n_bh * ((nq + 1) / 2);
}

struct Item {
  int bh, h;               // (batch or sequence, head); head (packed layout)
  int qa;                  // query tile of a (tile b is qa + 1)
  bool has_a, has_b;       // the tiles have rows (has_a: the item exists)
  int nkv_a, nkv_b, nkv;   // key tiles tile a / tile b read; key tiles loaded for the pair
  int lq, lk;              // the sequence's query / key lengths
  int q0, k0;              // fixed layout: rows bh * Lq / bh * Lk of the 2-D maps;
                           // packed layout: the sequence's first query / key token
};

// Keys the last row of query tile qt may read (all lk without the causal
// mask; with it, keys j <= i + lk - lq of row i, clamped to 0..lk), as a
// count of 128-key tiles, at least one: a tile whose rows read no key still
// runs one fully masked key tile and writes zeros.
__device__ __forceinline__ int tiles_of(int qt, int lq, int lk, bool causal) {
  int end = lk;
  if (causal) end = max(0, min(lk, min((qt + 1) * BQ, lq) + (lk - lq)));
  return max(1, (end + BKV - 1) / BKV);
}

// Item it: pair p = it / n_bh of query tiles (2p, 2p + 1) of (batch, head)
// bh = it % n_bh.  Fixed layout [B*H][L][64]: every item exists.  Packed
// layout (tokens [total][H][64], sequence b = bh / H owns query tokens
// cu_q[b] .. cu_q[b + 1] - 1 and key tokens cu_k[b] ..): an item whose first
// tile lies past its sequence does not exist; lengths that contradict the
// host-side totals are reported and the sequence skipped; with the causal
// mask the heaviest pairs come first (one CTA per item, started in order).
template <bool kCausal, bool kVarlen>
__device__ __forceinline__ Item item_of(int it, int n_bh, int nq, int Lq, int Lk, const int* cu_q,
                                        const int* cu_k, int H, int total_q, int total_k,
                                        unsigned* err) {
  Item w;
  const int npairs = (nq + 1) / 2;
  int p = it / n_bh;
  w.bh = it % n_bh;
  if (kCausal && kVarlen) p = npairs - 1 - p;
  w.qa = 2 * p;
  bool ok = it < n_items_of(n_bh, nq);
  if (!kVarlen) {
    w.h = 0;
    w.lq = Lq;
    w.lk = Lk;
    w.q0 = w.bh * Lq;
    w.k0 = w.bh * Lk;
  } else {
    const int b = w.bh / H;
    w.h = w.bh % H;
    const bool cu_ok = ok && RF_IN(err, b + 1, n_bh / H + 1);   // cu_q, cu_k have B + 1 entries
    const int a0 = cu_ok ? cu_q[b] : 0, a1 = cu_ok ? cu_q[b + 1] : 0;
    const int c0 = cu_ok ? cu_k[b] : 0, c1 = cu_ok ? cu_k[b + 1] : 0;
    const bool len_ok = cu_ok && 0 <= a0 && a0 <= a1 && a1 <= total_q && a1 - a0 <= Lq &&
                        0 <= c0 && c0 <= c1 && c1 <= total_k;
    if (cu_ok && !len_ok && p == 0 && threadIdx.x == 0) raise_error(err, kDevErrInput);
    ok = len_ok;
    w.lq = ok ? a1 - a0 : 0;
    w.lk = ok ? c1 - c0 : 0;
    w.q0 = a0;
    w.k0 = c0;
  }
  w.has_a = ok && w.qa * BQ < w.lq;
  w.has_b = ok && (w.qa + 1) * BQ < w.lq;
  w.nkv_a = w.has_a ? tiles_of(w.qa, w.lq, w.lk, kCausal) : 0;
  w.nkv_b = w.has_b ? tiles_of((w.qa + 1), w.lq, w.lk, kCausal) : 0;
  w.nkv = max(w.nkv_a, w.nkv_b);
  return w;
}

// Fixed layout: tmQ/tmK/tmV are 2-D maps over rows [B*H*L][64] and tmO a
// 3-D map [B*H][Lq][64].  Packed layout: all four are 3-D maps
// [total][H][64]; Lq is the longest sequence (max_q) and Lk unused.
template <bool kCausal, bool kVarlen>
__global__ void __launch_bounds__(kThreads, 1)
    attn_prefill_kernel(const __grid_constant__ CUtensorMap tmQ,
                        const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV,
                        const __grid_constant__ CUtensorMap tmO, __nv_bfloat16* __restrict__ O,
                        int Lq, int Lk, float c_log2, int n_bh, int nq, const int* __restrict__ cu_q,
                        const int* __restrict__ cu_k, int H, int total_q, int total_k,
                        unsigned* err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + kBarOff);
  volatile int* abort_flag = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_items = n_items_of(n_bh, nq);
  auto item = [&](int it) {
    return item_of<kCausal, kVarlen>(it, n_bh, nq, Lq, Lk, cu_q, cu_k, H, total_q, total_k, err);
  };
  // the next item of this CTA from `it` on that has rows (n_items if none)
  auto next_item = [&](int it) {
    while (it < n_items && !item(it).has_a) it += gridDim.x;
    return it;
  };
  // TMA loads of 128 rows (query tile or key tile) of head h starting at
  // row / token r0 of the map
  auto load_rows = [&](uint32_t dst, const CUtensorMap* m, uint32_t bar, int h, int r0,
                       uint64_t pol) {
    if (kVarlen) tma_load_3d_hint(dst, m, bar, 0, h, r0, pol);
    else tma_load_2d_hint(dst, m, bar, 0, r0, pol);
  };

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmQ);
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    prefetch_tmap(&tmO);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars->q_full[i]), 1);
      mbar_init(smem_u32(&bars->q_empty[i]), 2);     // one commit per issuer
      mbar_init(smem_u32(&bars->s_full[i]), 1);
      mbar_init(smem_u32(&bars->s_read[i]), 4);
      mbar_init(smem_u32(&bars->p_full[i]), BQ);
      mbar_init(smem_u32(&bars->pv_done[i]), 1);
      mbar_init(smem_u32(&bars->o_done[i]), 1);
      mbar_init(smem_u32(&bars->st_full[i]), 4);
      mbar_init(smem_u32(&bars->st_free[i]), 1);
    }
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&bars->k_full[i]), 1);
      mbar_init(smem_u32(&bars->k_empty[i]), 2);
      mbar_init(smem_u32(&bars->v_full[i]), 1);
      mbar_init(smem_u32(&bars->v_empty[i]), 2);
    }
    mbar_init(smem_u32(&bars->a_max0), 4);
    mbar_init(smem_u32(&bars->drain[0]), 1);
    mbar_init(smem_u32(&bars->drain[1]), 1);
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
      const uint64_t pol_q = policy_evict_first();   // each Q tile is read once
      bool ok = true;
      int ni = 0, g = 0;                             // items and K/V tiles issued
      for (int it = next_item(blockIdx.x); ok && it < n_items && !*abort_flag;
           it = next_item(it + gridDim.x), ++ni) {
        const Item w = item(it);
        const int slot = ni & 1;
        if (ni >= 2 &&
            !mbar_wait(smem_u32(&bars->q_empty[slot]), (uint32_t)(((ni >> 1) - 1) & 1))) {
          ok = false;
          break;
        }
        const uint32_t qb = smem_u32(&bars->q_full[slot]);
        mbar_arrive_expect_tx(qb, (w.has_b ? 2 : 1) * kTile);
        load_rows(smem_u32(smem + kQOff + (2 * slot) * kTile), &tmQ, qb, w.h, w.q0 + w.qa * BQ,
                  pol_q);
        if (w.has_b)
          load_rows(smem_u32(smem + kQOff + (2 * slot + 1) * kTile), &tmQ, qb, w.h,
                    w.q0 + (w.qa + 1) * BQ, pol_q);
        for (int j = 0; j < w.nkv; ++j, ++g) {
          const int st = g % kStages;
          const uint32_t ph = (uint32_t)(((g / kStages) + 1) & 1);
          if (g >= kStages && !mbar_wait(smem_u32(&bars->k_empty[st]), ph)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(smem_u32(&bars->k_full[st]), kTile);
          load_rows(smem_u32(smem + kKOff + st * kTile), &tmK, smem_u32(&bars->k_full[st]), w.h,
                    w.k0 + j * BKV, pol_kv);
          if (g >= kStages && !mbar_wait(smem_u32(&bars->v_empty[st]), ph)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(smem_u32(&bars->v_full[st]), kTile);
          load_rows(smem_u32(smem + kVOff + st * kTile), &tmV, smem_u32(&bars->v_full[st]), w.h,
                    w.k0 + j * BKV, pol_kv);
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
  } else if (warp == 1 || warp == kMmaWarpB) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuers, one per query tile
      // Thread x issues its tile's products in the tile's own order: S_x(j+1)
      // as soon as the softmax warps have read S_x(j), P_x V(j) once P_x(j)
      // is written; neither tile waits behind the other's events.  Both
      // threads release every K/V stage and Q slot (barrier counts 2), each
      // after waiting for that stage itself, so neither runs a phase ahead.
      const int x = warp == 1 ? 0 : 1;
      bool ok = true;
      int np = 0;                                    // P tiles consumed
      int nsr = 0;                                   // S reads waited for
      bool unread = false;                           // an issued S_x not yet known to be read
      // S_x(g) = Q_x K_g^T, Q from slot qs; S_x's columns are free once the
      // softmax warps have read the previous S_x into registers
      auto issue_s = [&](int g, int qs) -> bool {
        if (unread) {
          if (!mbar_wait(smem_u32(&bars->s_read[x]), (uint32_t)(nsr & 1))) return false;
          ++nsr;
          tc_fence_after();
        }
        const uint32_t qa = smem_u32(smem + kQOff + (2 * qs + x) * kTile);
        const uint32_t ka = smem_u32(smem + kKOff + (g % kStages) * kTile);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk)
          mma_bf16_ss(tmem + col_s(x), sw128_desc(qa + kk * 32, 1024, 16),
                      sw128_desc(ka + kk * 32, 1024, 16), kIdescS, kk != 0);
        mma_commit(smem_u32(&bars->s_full[x]));
        unread = true;
        return true;
      };
      // O_x (+)= P_x V_g, P_x from its own columns; pv_done[x] tells the
      // softmax warps when P_x may be overwritten and O_x is up to date
      auto issue_pv = [&](int g, bool first) {
        const uint32_t va = smem_u32(smem + kVOff + (g % kStages) * kTile);
#pragma unroll
        for (int kk = 0; kk < BKV / 16; ++kk)
          mma_bf16_ts(tmem + col_o(x), tmem + col_p(x) + kk * 8,
                      sw128_desc(va + kk * 16 * 128, 1024, kTile), kIdescO, (!first || kk != 0));
        mma_commit(smem_u32(&bars->pv_done[x]));
      };
      auto wait_kv = [&](uint64_t* full, int g) -> bool {
        if (!mbar_wait(smem_u32(&full[g % kStages]), (uint32_t)((g / kStages) & 1))) return false;
        tc_fence_after();
        return true;
      };
      int ni = 0, g = 0;
      int it = next_item(blockIdx.x);
      Item w = item(it);
      if (it < n_items) {
        ok = mbar_wait(smem_u32(&bars->q_full[0]), 0) && wait_kv(bars->k_full, 0);
        // tile b starts once tile a's softmax has taken its first row maxima,
        // so that the two softmax warpgroups run out of phase (one's
        // exponentials beside the other's max pass) rather than both loading
        // the MUFU at once
        if (ok && x == 1 && w.has_b) ok = mbar_wait(smem_u32(&bars->a_max0), 0);
        if (ok && (x == 0 || w.has_b)) ok = issue_s(0, 0);
        if (ok) mma_commit(smem_u32(&bars->k_empty[0]));
      }
      for (; ok && it < n_items; ++ni) {
        const int qs = ni & 1;
        const int it_next = next_item(it + gridDim.x);
        const bool next_has_b = it_next < n_items && item(it_next).has_b;
        // key tiles this query tile reads (0 for a missing tile b); the
        // pair's loaded tiles may run past them under the causal mask
        const int nkv_x = x == 0 ? w.nkv_a : w.nkv_b;
        for (int j = 0; ok && j < w.nkv; ++j, ++g) {
          const bool last = j == w.nkv - 1;            // the pair's last key tile
          const bool mine = j < nkv_x;
          // next tile: the same item's, or the next item's first
          const bool has_next = !last || it_next < n_items;
          const int qs_next = last ? qs ^ 1 : qs;
          const bool next_mine = last ? (x == 0 || next_has_b) : j + 1 < nkv_x;
          // the next S, as soon as the softmax warps have read the current
          // one (their exponentials then overlap this product)
          auto next_s = [&]() -> bool {
            if (!has_next) return true;
            if (last && !mbar_wait(smem_u32(&bars->q_full[qs_next]), (uint32_t)(((ni + 1) >> 1) & 1)))
              return false;
            if (!wait_kv(bars->k_full, g + 1)) return false;
            if (next_mine && !issue_s(g + 1, qs_next)) return false;
            mma_commit(smem_u32(&bars->k_empty[(g + 1) % kStages]));
            return true;
          };
          // this key tile's P.V
          auto this_pv = [&]() -> bool {
            if (!wait_kv(bars->v_full, g)) return false;
            if (mine) {
              if (!mbar_wait(smem_u32(&bars->p_full[x]), (uint32_t)(np & 1))) return false;
              tc_fence_after();
              ++np;
              issue_pv(g, j == 0);
              if (j == nkv_x - 1) mma_commit(smem_u32(&bars->o_done[x]));
            }
            mma_commit(smem_u32(&bars->v_empty[g % kStages]));
            if (last) mma_commit(smem_u32(&bars->q_empty[qs]));   // every S of the item issued
            return true;
          };
          // within an item the next S goes first; at its last key tile the
          // P.V goes first, so the epilogue's O is complete as early as
          // possible (the softmax warps store O before they read the next S)
          ok = last ? (this_pv() && next_s()) : (next_s() && this_pv());
        }
        it = it_next;
        w = item(it);
      }
      if (!ok) {
        raise_error(err, kDevErrTimeout);
        *abort_flag = 1;
      }
      // nothing may still run on the tensor core when TMEM and shared memory
      // are released
      mma_commit(smem_u32(&bars->drain[x]));
      (void)mbar_wait(smem_u32(&bars->drain[x]), 0, 1000000000ull);
    }
  } else {
    // ------------------------------------------------ softmax warpgroups
    const int x = warp >= 6 ? 1 : 0;                   // query tile of this warpgroup
    const int sub = warp & 3;                          // TMEM lane quarter
    const int r = sub * 32 + lane;                     // query row within the tile
    const uint32_t lane_off = (uint32_t)(sub * 32) << 16;
    const uint32_t s_addr = tmem + lane_off + col_s(x);
    const uint32_t o_addr = tmem + lane_off + col_o(x);
    static_assert(kColP1 - kColO1 == kColP0 - kColO0, "P_x at a fixed offset from O_x");
    const uint32_t p_addr = o_addr + (kColP0 - kColO0);
    const uint64_t c2 = f2(c_log2, c_log2);
    bool ok = true;
    int cnt = 0, icnt = 0;                             // tiles and items of this warpgroup
    int ns = 0;                                        // of those, O tiles written by bulk store
    for (int it = blockIdx.x; ok && it < n_items; it += gridDim.x) {
      const Item w = item(it);
      if (!w.has_a || (x == 1 && !w.has_b)) continue;
      const int nkv_x = x == 0 ? w.nkv_a : w.nkv_b;
      const int row0 = (w.qa + x) * BQ;                   // first row of this query tile
      // keys this row reads: all lk, or under the causal mask j <= i + lk - lq
      const int kv_row =
          kCausal ? max(0, min(w.lk, row0 + r + (w.lk - w.lq) + 1)) : w.lk;
      float m_ref = -INFINITY, l_run = 0.f;
      for (int j = 0; j < nkv_x; ++j, ++cnt) {
        // warp-uniform decision: the TMEM loads below are warp-collective
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->s_full[x]), (uint32_t)(cnt & 1)) &&
                                         !*abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // keys of this tile the row reads (a prefix; 0 for a row that reads
        // none: its P is all zero and its output row zero)
        const int valid = max(0, min(BKV, kv_row - j * BKV));
        const bool full = valid == BKV;
        // the row's 128 scores read from tensor memory once (four loads in
        // flight together) and kept in registers for both passes
        uint32_t v[4][32];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld32(s_addr + q * 32, v[q]);
        tmem_ld_wait();
        // S_x is in registers: the MMA warp may compute the next S_x into
        // the same columns while this tile's exponentials run
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&bars->s_read[x]));
        // keys the row does not read score -inf: their P is 2^-inf = 0, so
        // both passes below run without per-key tests
        if (!full) {
#pragma unroll
          for (int q = 0; q < 4; ++q)
#pragma unroll
            for (int i = 0; i < 32; ++i)
              v[q][i] = q * 32 + i < valid ? v[q][i] : 0xff800000u;
        }
        // pass 1: row max (four independent chains)
        float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int i = 0; i < 32; i += 2)
            mx4[(i >> 1) & 3] =
                fmax3(mx4[(i >> 1) & 3], __uint_as_float(v[q][i]), __uint_as_float(v[q][i + 1]));
        const float mt = fmaxf(fmax3(mx4[0], mx4[1], mx4[2]), mx4[3]) * c_log2;
        if (x == 0 && cnt == 0) {
          __syncwarp();
          if (lane == 0) mbar_arrive(smem_u32(&bars->a_max0));
        }
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
        // a row that has read no key yet (m = -inf) takes 0 as its reference:
        // its P is then 2^-inf = 0, not NaN
        const float m_use = m_ref == -INFINITY ? 0.f : m_ref;
        const uint64_t negm2 = f2(-m_use, -m_use);
        // pass 2: P = 2^(S c - m) as bf16 pairs, row sum (four chains),
        // written to P_x half by half; before the first half, the previous
        // P_x V must have completed: P_x may then be overwritten and O_x
        // holds every earlier tile (warp-uniform: the TMEM accesses are
        // warp-collective)
        uint64_t sum4[4] = {0ull, 0ull, 0ull, 0ull};
        bool pv_ok = true;
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
              const float p0 = ex2(t0), p1 = ex2(t1);
              sum4[i & 3] = fadd2(sum4[i & 3], f2(p0, p1));
              pk[h * 16 + i] = pack_bf16x2(p0, p1);
            }
          }
          if (hh == 0 && cnt > 0) {
            pv_ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->pv_done[x]),
                                                      (uint32_t)((cnt - 1) & 1)));
            if (!pv_ok) break;
            tc_fence_after();
          }
          tmem_st32(p_addr + hh * 32, pk);
        }
        if (!pv_ok) {
          ok = false;
          break;
        }
        float s_lo, s_hi;
        f2_split(fadd2(fadd2(sum4[0], sum4[1]), fadd2(sum4[2], sum4[3])), s_lo, s_hi);
        l_run += s_lo + s_hi;
        // a moved reference: O_x (complete through the previous tile, since
        // its P.V is) is rescaled before this tile's P.V adds to it
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
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;   // a row that read no key: zeros
      auto out8 = [&](int c) {                         // 16-byte chunk c of the row's bf16 O
        const uint32_t* u = &v[c >> 2][(c & 3) * 8];
        return make_uint4(pack_bf16x2(__uint_as_float(u[0]) * inv, __uint_as_float(u[1]) * inv),
                          pack_bf16x2(__uint_as_float(u[2]) * inv, __uint_as_float(u[3]) * inv),
                          pack_bf16x2(__uint_as_float(u[4]) * inv, __uint_as_float(u[5]) * inv),
                          pack_bf16x2(__uint_as_float(u[6]) * inv, __uint_as_float(u[7]) * inv));
      };
      if (kVarlen && row0 + BQ > w.lq) {
        // the sequence's last, partial tile: a bulk store would run into the
        // next sequence's rows, so each thread stores its own row
        const int row = row0 + r;
        const int64_t o_first = ((int64_t)(w.q0 + row) * H + w.h) * kD;
        if (row < w.lq && RF_IN(err, o_first + kD - 1, (int64_t)total_q * H * kD)) {
          uint4* dst = reinterpret_cast<uint4*>(O + o_first);
#pragma unroll
          for (int c = 0; c < kD / 8; ++c) dst[c] = out8(c);
        }
        continue;
      }
      // O_x / l as bf16, staged in shared memory as 128-byte swizzled rows
      // and written by one bulk tensor store per tile (fixed layout: rows
      // past Lq are outside the tensor map and are not written).  The
      // staging tile is reused once the previous store has read it.
      const int e = ns++;
      const bool issuer = sub == 0 && lane == 0;
      if (e > 0) {
        if (issuer) {
          bulk_wait_group_read0();
          mbar_arrive(smem_u32(&bars->st_free[x]));
        }
        if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars->st_free[x]), (uint32_t)((e - 1) & 1)))) {
          ok = false;
          break;
        }
      }
      uint8_t* st = smem + kStOff + x * kTile + r * 128;
#pragma unroll
      for (int c = 0; c < kD / 8; ++c) *reinterpret_cast<uint4*>(st + ((c ^ (r & 7)) << 4)) = out8(c);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->st_full[x]));
      bool st_ok = true;
      if (issuer) {
        st_ok = mbar_wait(smem_u32(&bars->st_full[x]), (uint32_t)(e & 1)) && RF_IN(err, w.bh, n_bh) &&
                RF_IN(err, row0, Lq);
        if (st_ok) {
          const uint32_t src = smem_u32(smem + kStOff + x * kTile);
          if (kVarlen) tma_store_3d(&tmO, src, 0, w.h, w.q0 + row0);
          else tma_store_3d(&tmO, src, 0, row0, w.bh);
          bulk_commit_group();
        }
      }
      if (!__shfl_sync(0xffffffffu, st_ok, 0)) {
        ok = false;
        break;
      }
    }
    // every bulk store of this warpgroup has completed before the CTA exits
    if (sub == 0 && lane == 0 && ns > 0) bulk_wait_group0();
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
                                   int H, int Lq, int Lk, float scale, int causal, unsigned* err,
                                   cudaStream_t s) {
  CUtensorMap tmQ, tmK, tmV, tmO;
  const uint64_t q_rows = (uint64_t)B * H * Lq, kv_rows = (uint64_t)B * H * Lk;
  // O as [B*H][Lq][64]: a store box of 128 rows is clipped at its head's Lq
  if (!encode_tmap_2d(&tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Q, kD, q_rows, kD * 2, kD, BQ, true) ||
      !encode_tmap_3d(&tmO, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, O, kD, (uint64_t)Lq, (uint64_t)B * H,
                      kD * 2, (uint64_t)Lq * kD * 2, kD, BQ, 1, true) ||
      !encode_tmap_2d(&tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, kD, kv_rows, kD * 2, kD, BKV, true) ||
      !encode_tmap_2d(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, V, kD, kv_rows, kD * 2, kD, BKV, true))
    return cudaErrorInvalidValue;
  auto kern = causal ? attn_prefill_kernel<true, false> : attn_prefill_kernel<false, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  const int nq = (Lq + BQ - 1) / BQ, n_bh = B * H;
  const int64_t items = (int64_t)n_bh * ((nq + 1) / 2);
  const int sms = sm_count();
  if (sms <= 0 || items <= 0 || items >= (1ll << 31)) return cudaErrorInvalidValue;
  // persistent, one CTA per SM; every CTA takes the same number of items
  const int64_t per_cta = (items + sms - 1) / sms;
  const int grid = (int)((items + per_cta - 1) / per_cta);
  const float c_log2 = scale * 1.4426950408889634f;
  kern<<<grid, kThreads, kSmem, s>>>(tmQ, tmK, tmV, tmO, static_cast<__nv_bfloat16*>(O), Lq, Lk,
                                     c_log2, n_bh, nq, nullptr, nullptr, H, 0, 0, err);
  return cudaGetLastError();
}

cudaError_t launch_attn_prefill_tc_varlen(const void* Q, const void* K, const void* V, void* O,
                                          const int* cu_q, const int* cu_k, int B, int H,
                                          int max_q, int total_q, int total_k, float scale,
                                          int causal, unsigned* err, cudaStream_t s) {
  // [total][H][64] tokens: one head's 128 consecutive tokens are a box of
  // 64 x 1 x 128 (coordinates: dim, head, token)
  CUtensorMap tmQ, tmK, tmV, tmO;
  const uint64_t pitch = (uint64_t)H * kD * 2;     // bytes between tokens
  if (!encode_tmap_3d(&tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Q, kD, H, total_q, kD * 2, pitch,
                      kD, 1, BQ, true) ||
      !encode_tmap_3d(&tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, kD, H, total_k, kD * 2, pitch,
                      kD, 1, BKV, true) ||
      !encode_tmap_3d(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, V, kD, H, total_k, kD * 2, pitch,
                      kD, 1, BKV, true) ||
      !encode_tmap_3d(&tmO, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, O, kD, H, total_q, kD * 2, pitch,
                      kD, 1, BQ, true))
    return cudaErrorInvalidValue;
  auto kern = causal ? attn_prefill_kernel<true, true> : attn_prefill_kernel<false, true>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  const int nq = (max_q + BQ - 1) / BQ, n_bh = B * H;
  const int64_t items = (int64_t)n_items_of(n_bh, nq);
  if (items <= 0 || items >= (1ll << 31)) return cudaErrorInvalidValue;
  // items of very different cost (sequence lengths vary, and pairs past a
  // short sequence are empty): one CTA per item, so that the hardware's CTA
  // scheduler balances them
  const float c_log2 = scale * 1.4426950408889634f;
  kern<<<(int)items, kThreads, kSmem, s>>>(tmQ, tmK, tmV, tmO, static_cast<__nv_bfloat16*>(O), max_q,
                                           0, c_log2, n_bh, nq, cu_q, cu_k, H, total_q, total_k, err);
  return cudaGetLastError();
}

}  // namespace rf
