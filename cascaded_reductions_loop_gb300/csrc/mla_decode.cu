// mla_decode.cu -- latent-KV (multi-latent attention) decode in its absorbed
// form on the tcgen05 tensor cores: bf16 query and latent cache, fp32 scores,
// softmax state and accumulation, bf16 output.
//
// For batch b every one of the Hq (<= 128) query heads attends to the same
// latent cache rows C_b [Lk, 576]: s = scale * q . c over all 576 dims (512
// latent + 64 positional) and o = softmax(s) . C_b[:, 0:512].  This is the
// safe-softmax cascade ([E] §2.2) in the single-loop incremental form ([E]
// §2.3, §4.1; [S] Methodologie 2) over tiles of 64 cache rows, and, when the
// rows of a batch are cut into segments, the multi-segment form with a merge
// kernel ([S] Methodologie 3; [E] §3.3).
//
// Work split.  The state of one (batch, segment) -- O for 128 heads x 512
// dims in fp32 -- is 256 KB, all of one SM's tensor memory, so two SMs share
// it: a cluster of two CTAs, CTA r owning the value dims 256 r .. 256 r + 255.
// Each CTA loads only its own 64-dim blocks of every cache row (CTA 0: blocks
// 0-3 and the positional block 8; CTA 1: blocks 4-7) and computes a partial
// score tile over them.  The two fp32 partial tiles (128 heads x 64 rows) are
// swapped through distributed shared memory (bulk copies, whose bytes complete
// a barrier in the receiving CTA), and both CTAs form s = S_0 + S_1 -- the same
// bits on both sides, as a + b = b + a exactly -- so they run the identical
// softmax: the same maxima, the same P, the same l.  The value block of a CTA
// is the latent part of what it loaded, so P . V needs no further exchange.
//
// Per CTA: its Q dims sit in tensor memory (written once by the softmax
// warps) as the A operand of the score products, and so does P (bf16) for the
// P . V products; the cache rows stream by TMA through a 4-stage ring (64 rows
// x 64 dims per block, 128-byte swizzle; prefetching further tiles into L2
// measured slower); S has one buffer in tensor memory, O accumulates there.
// Two threads issue the products: one the score products (S_t once the
// softmax warps have taken S_{t-1} and the tile has landed), one the P . V
// products (P_j V_j once P_j is written), so that a ready P . V enters the
// tensor core between score products instead of after all of them.
//
// Exchange, one tile ahead: at tile j the softmax warps add the peer's
// partial S_j to their own, then at once take their own S_{j+1} out of tensor
// memory (freeing it for S_{j+2}) and ship it, so its copy runs under the
// softmax of tile j.  Each CTA has two 32 KB slots, each in turn the landing
// place of a peer tile and the staging place of an own tile: S_{j+1} is
// staged in slot j % 2, whose peer tile S_j each thread has just read (its own
// row), and each warp bulk-copies its 32 rows to the peer's slot (j + 1) % 2.
// Each row is read and written by the warp of the same number on both sides,
// so the slots are tracked per warp (one barrier per slot and warp, 8 KB):
// a warp waits only for its own rows.  Ordering needs no extra messages: the
// peer's S_j landing here shows that
// the peer has read our S_{j-1} from its slot (j + 1) % 2; the peer ships its
// S_{j+2} into the slot our S_{j+1} was staged in only after our S_{j+1} has
// landed there, i.e. after the copy has read it.
//
// Lazy rescaling: a row's reference maximum m moves only when a tile's
// maximum exceeds it by more than 8 (log2 units); only then are O (in tensor
// memory) and l multiplied by 2^(m_old - m_new).  The cascade's invertible
// dependent factor makes the result independent of the reference chosen ([S]
// Methodologie 1), and P <= 2^8 keeps bf16 P and fp32 sums far from overflow.
//
// Tensor memory (512 columns): O 0-255, S 256-319, P 320-351, Q 352-511.
#include <math.h>

#include "rf_device.cuh"
#include "rf_internal.h"

namespace rf {
namespace {

constexpr int kDqk = 576, kDv = 512;
constexpr int BH = 128;                            // head rows (MMA M)
constexpr int BN = 64;                             // cache rows per tile
constexpr int kMaxBlk = 5;                         // 64-dim blocks per CTA
constexpr int kStages = 4;
constexpr int kChBytes = BN * 128;                 // one 64-dim block of a tile: 8 KB
constexpr int kStageBytes = kMaxBlk * kChBytes;    // 40 KB
constexpr int kXBytes = BH * BN * 4;               // one partial score tile: 32 KB
constexpr int kNX = 2;                             // exchange slots
constexpr int kStOff = 0;
constexpr int kXOff = kStOff + kStages * kStageBytes;   // 160 KB
constexpr int kBarOff = kXOff + kNX * kXBytes;          // 224 KB
constexpr int kSmem = kBarOff + 512;
constexpr int kThreads = 224;                      // warp 0 TMA, 1 MMA (S), 2-5 softmax, 6 MMA (P.V)
constexpr int kPvWarp = 6;
constexpr int kTmemCols = 512;
constexpr int kTmemS = 256, kTmemP = 320, kTmemQ = 352;
constexpr float kLazy = 8.f;
constexpr uint32_t kIdescS = make_idesc(BH, BN, /*bf16*/ 1, 0, 0);
// P . V: N = 256 value dims in one product; the four 64-dim blocks of a stage
// are 8 KB apart, the stride between 64-element blocks of an MN-major operand
constexpr uint32_t kIdescO = make_idesc(BH, 256, /*bf16*/ 1, 0, /*V MN-major*/ 1);
constexpr int kMergeThreads = 128;                 // 4 dims per thread

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

struct Bars {
  uint64_t q_full;                  // Q in tensor memory (128 softmax threads)
  uint64_t full[kStages], empty[kStages];
  uint64_t s_full;                  // own partial S_t in tensor memory
  uint64_t s_free;                  // S_t taken by the softmax warps
  uint64_t p_full;                  // P_j in tensor memory
  uint64_t pv_done;                 // P_j V_j accumulated into O (P_j read)
  uint64_t x_full[kNX][4];          // rows 32 w .. of the peer's partial S_t in slot t % 2
  uint64_t drain, drain_pv;         // every MMA of the S / P.V issuer has completed
  uint32_t tmem;
  int abort;
};
static_assert(sizeof(Bars) <= 512, "barrier block");
static_assert(kSmem <= 232448, "shared memory per CTA");

// 64-dim block held by CTA `rank` as its c-th block.
__device__ __forceinline__ int dim_block(int rank, int c) {
  return rank == 0 ? (c < 4 ? c : 8) : 4 + c;
}

// One cluster of two CTAs per work item (batch b, segment seg); the segment
// covers cache tiles seg * tps .. of batch b.
__global__ void __launch_bounds__(kThreads, 1)
    mla_decode_kernel(const __grid_constant__ CUtensorMap tmC, const __nv_bfloat16* __restrict__ Q,
                      __nv_bfloat16* __restrict__ O, float* __restrict__ part_o,
                      float* __restrict__ part_ml, int Hq, int Lk, int S, int tps, float c_log2,
                      unsigned* err) {
  extern __shared__ __align__(1024) uint8_t smem[];
  Bars* bars = reinterpret_cast<Bars*>(smem + kBarOff);
  volatile int* abort_flag = &bars->abort;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rank = (int)cluster_ctarank(), peer = rank ^ 1;
  const int item = blockIdx.x >> 1;
  const int b = item / S, seg = item % S;
  const int64_t n_bat = (int64_t)(gridDim.x >> 1) / S;   // batches (debug-build bounds checks)
  const int ntiles = (Lk + BN - 1) / BN;
  const int t0 = seg * tps;
  int nt = min(tps, ntiles - t0);
  const int lo = t0 * BN, hi = min(Lk, (t0 + nt) * BN);
  const int nblk = rank == 0 ? 5 : 4;
  if ((smem_u32(smem) & 1023u) != 0 || nt < 1) {   // both CTAs of the cluster agree
    if (threadIdx.x == 0) raise_error(err, nt < 1 ? kDevErrInput : kDevErrLayout);
    nt = 0;
  }

  if (threadIdx.x == 0) {
    prefetch_tmap(&tmC);
    mbar_init(smem_u32(&bars->q_full), BH);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&bars->full[i]), 1);
      mbar_init(smem_u32(&bars->empty[i]), 1);
    }
    mbar_init(smem_u32(&bars->s_full), 1);
    mbar_init(smem_u32(&bars->s_free), BH);
    mbar_init(smem_u32(&bars->p_full), BH);
    mbar_init(smem_u32(&bars->pv_done), 1);
    for (int i = 0; i < kNX; ++i)
      for (int w = 0; w < 4; ++w) mbar_init(smem_u32(&bars->x_full[i][w]), 1);
    mbar_init(smem_u32(&bars->drain), 1);
    mbar_init(smem_u32(&bars->drain_pv), 1);
    bars->abort = 0;
    fence_mbar_init();
    // armed for the peer's first two partial tiles; re-armed as slots are read
    for (int i = 0; i < kNX && i < nt; ++i)
      for (int w = 0; w < 4; ++w) mbar_arrive_expect_tx(smem_u32(&bars->x_full[i][w]), kXBytes / 4);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&bars->tmem), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync();            // both CTAs' barriers are armed before any exchange
  tc_fence_after();
  const uint32_t tm = bars->tmem;
  // a merge kernel may be scheduled now; it waits for this grid to finish
  asm volatile("griddepcontrol.launch_dependents;");

  if (warp == 0) {
    if (lane == 0 && nt > 0) {
      // ------------------------------------------------ TMA producer
      const uint64_t pol = policy_evict_first();       // every cache row is read once
      const int32_t row0 = b * Lk + lo;
      int issued = 0;
      for (int t = 0; t < nt && !*abort_flag; ++t) {
        const int st = t % kStages;
        if (t >= kStages &&
            !mbar_wait(smem_u32(&bars->empty[st]), (uint32_t)(((t / kStages) - 1) & 1))) {
          *abort_flag = 1;
          break;
        }
        const uint32_t bar = smem_u32(&bars->full[st]);
        mbar_arrive_expect_tx(bar, nblk * kChBytes);
        const uint32_t dst = smem_u32(smem + kStOff + st * kStageBytes);
        for (int c = 0; c < nblk; ++c)
          tma_load_2d_hint(dst + c * kChBytes, &tmC, bar, 64 * dim_block(rank, c), row0 + t * BN,
                           pol);
        ++issued;
      }
      if (*abort_flag) {
        raise_error(err, kDevErrTimeout);
        for (int i = issued - kStages < 0 ? 0 : issued - kStages; i < issued; ++i)
          (void)mbar_wait(smem_u32(&bars->full[i % kStages]), (uint32_t)((i / kStages) & 1),
                          1000000ull);
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && nt > 0) {
      // ------------------------------------------------ MMA issuer: score products
      bool ok = mbar_wait(smem_u32(&bars->q_full), 0);
      for (int ns = 0; ok && ns < nt; ++ns) {
        // S_t once the softmax warps have taken S_{t-1} and the tile has landed
        ok = (ns == 0 || mbar_wait(smem_u32(&bars->s_free), (uint32_t)((ns - 1) & 1))) &&
             mbar_wait(smem_u32(&bars->full[ns % kStages]), (uint32_t)((ns / kStages) & 1)) &&
             !*abort_flag;
        if (!ok) break;
        // partial S_t = Q_r C_t,r^T over this CTA's dims
        tc_fence_after();
        const uint32_t sb = smem_u32(smem + kStOff + (ns % kStages) * kStageBytes);
        for (int c = 0; c < nblk; ++c) {
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_bf16_ts(tm + kTmemS, tm + kTmemQ + c * 32 + kk * 8,
                        sw128_desc(sb + c * kChBytes + kk * 32, 1024, 16), kIdescS, (c | kk) != 0);
        }
        mma_commit(smem_u32(&bars->s_full));
      }
      if (!ok) {
        raise_error(err, kDevErrTimeout);
        *abort_flag = 1;
      }
      mma_commit(smem_u32(&bars->drain));
      (void)mbar_wait(smem_u32(&bars->drain), 0, 1000000000ull);
    }
  } else if (warp == kPvWarp) {
    if (lane == 0 && nt > 0) {
      // ------------------------------------------------ MMA issuer: P.V products
      // A thread of its own, so that a ready P.V does not wait behind the
      // issue of a later tile's score products.  S_j has completed before
      // P_j exists (the softmax warps read it first), so the stage release
      // committed after P_j V_j covers both products that read the stage.
      bool ok = true;
      for (int npv = 0; ok && npv < nt; ++npv) {
        ok = mbar_wait(smem_u32(&bars->p_full), (uint32_t)(npv & 1)) && !*abort_flag;
        if (!ok) break;
        // O (+)= P_j V_j over all 256 value dims, P_j from tensor memory
        tc_fence_after();
        const int st = npv % kStages;
        const uint32_t sb = smem_u32(smem + kStOff + st * kStageBytes);
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_bf16_ts(tm, tm + kTmemP + kk * 8, sw128_desc(sb + kk * 16 * 128, 1024, kChBytes),
                      kIdescO, (npv | kk) != 0);
        mma_commit(smem_u32(&bars->pv_done));
        mma_commit(smem_u32(&bars->empty[st]));
      }
      if (!ok) {
        raise_error(err, kDevErrTimeout);
        *abort_flag = 1;
      }
      mma_commit(smem_u32(&bars->drain_pv));
      (void)mbar_wait(smem_u32(&bars->drain_pv), 0, 1000000000ull);
    }
  } else if (nt > 0) {
    // ------------------------------------------------ softmax / exchange / epilogue
    const int sub = warp & 3;
    const int r = sub * 32 + lane;                      // head row
    const int swz = r & 7;
    const uint32_t lane_off = (uint32_t)(sub * 32) << 16;
    const uint32_t x_peer = mapa_shared(smem_u32(smem + kXOff), (uint32_t)peer);
    const bool row_ok = r < Hq;
    const int64_t bh = (int64_t)b * Hq + r;

    // Q row r (this CTA's blocks) into tensor memory; rows past Hq are zero.
    // All loads are issued before the first store, so that the row's blocks
    // are fetched together rather than one round trip per block.
    {
      const uint4* qrow = reinterpret_cast<const uint4*>(Q + (row_ok ? bh : 0) * kDqk);
      const bool q_ok = row_ok && RF_IN(err, bh * kDqk + kDqk - 1, n_bat * Hq * kDqk);
      uint4 w[kMaxBlk][8];
#pragma unroll
      for (int c = 0; c < kMaxBlk; ++c) {
        const int db = dim_block(rank, c);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          w[c][i] = q_ok && c < nblk ? qrow[db * 8 + i] : make_uint4(0u, 0u, 0u, 0u);
      }
#pragma unroll
      for (int c = 0; c < kMaxBlk; ++c) {
        if (c >= nblk) break;                          // uniform over the CTA
        uint32_t v[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          v[4 * i] = w[c][i].x;
          v[4 * i + 1] = w[c][i].y;
          v[4 * i + 2] = w[c][i].z;
          v[4 * i + 3] = w[c][i].w;
        }
        tmem_st32(tm + lane_off + kTmemQ + c * 32, v);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&bars->q_full));
    }

    // own partial S_t out of tensor memory, which may then take S_{t+1}
    auto take = [&](int t, float (&own)[BN]) -> bool {
      if (!__all_sync(0xffffffffu,
                      mbar_wait(smem_u32(&bars->s_full), (uint32_t)(t & 1)) && !*abort_flag))
        return false;
      tc_fence_after();
      uint32_t v[32];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        tmem_ld32(tm + lane_off + kTmemS + 32 * h, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) own[32 * h + i] = __uint_as_float(v[i]);
      }
      tc_fence_before();
      mbar_arrive(smem_u32(&bars->s_free));
      return true;
    };
    // S_t staged in this CTA's slot (t + 1) % 2, then each warp bulk-copies
    // its 32 rows (8 KB) to the peer's slot t % 2 once the peer's S_{t-1} has
    // landed here (t >= 1; observed already by the caller)
    auto ship = [&](int t, const float (&own)[BN]) -> bool {
      uint8_t* stage = smem + kXOff + ((t + 1) % kNX) * kXBytes;
#pragma unroll
      for (int c = 0; c < BN / 4; ++c)
        *reinterpret_cast<uint4*>(stage + r * (BN * 4) + ((c ^ swz) << 4)) =
            make_uint4(__float_as_uint(own[4 * c]), __float_as_uint(own[4 * c + 1]),
                       __float_as_uint(own[4 * c + 2]), __float_as_uint(own[4 * c + 3]));
      fence_proxy_async_smem();                      // rows visible to the copy engine
      if (t >= 1 && !__all_sync(0xffffffffu,
                                mbar_wait_cluster(smem_u32(&bars->x_full[(t - 1) % kNX][sub]),
                                                  (uint32_t)(((t - 1) / kNX) & 1)) &&
                                    !*abort_flag))
        return false;
      __syncwarp();
      if (lane == 0) {
        const uint32_t blk = (uint32_t)(sub * 32 * BN * 4);   // this warp's 32 rows
        bulk_copy_to_peer(x_peer + (t % kNX) * kXBytes + blk, smem_u32(stage) + blk, 32 * BN * 4,
                          mapa_shared(smem_u32(&bars->x_full[t % kNX][sub]), (uint32_t)peer));
      }
      return true;
    };

    float m_run = -INFINITY, l_run = 0.f;
    const uint64_t c2 = f2(c_log2, c_log2);
    float own_a[BN], own_b[BN];                       // own partial S_j and S_{j+1}, in turn
    bool ok = take(0, own_a) && ship(0, own_a);
    // tile j with cur = own S_j and nxt = own S_{j+1} (taken here)
    auto step = [&](int j, float (&cur)[BN], float (&nxt)[BN]) -> bool {
      // (a) s = own + the peer's partial scores of tile j
      if (!__all_sync(0xffffffffu, mbar_wait_cluster(smem_u32(&bars->x_full[j % kNX][sub]),
                                                     (uint32_t)((j / kNX) & 1)) &&
                                       !*abort_flag))
        return false;
      // armed for the peer's S_{j+2}, which its warp ships only after our
      // warp's S_{j+1} rows have reached it (this phase is complete by then)
      if (lane == 0 && j + kNX < nt)
        mbar_arrive_expect_tx(smem_u32(&bars->x_full[j % kNX][sub]), kXBytes / 4);
      float (&sc)[BN] = cur;
      {
        const uint8_t* src = smem + kXOff + (j % kNX) * kXBytes + r * (BN * 4);
#pragma unroll
        for (int c = 0; c < BN / 4; ++c) {
          const uint4 w = *reinterpret_cast<const uint4*>(src + ((c ^ swz) << 4));
          sc[4 * c] += __uint_as_float(w.x);
          sc[4 * c + 1] += __uint_as_float(w.y);
          sc[4 * c + 2] += __uint_as_float(w.z);
          sc[4 * c + 3] += __uint_as_float(w.w);
        }
      }
      // own S_{j+1} out and to the peer, under this tile's softmax
      if (j + 1 < nt && !(take(j + 1, nxt) && ship(j + 1, nxt))) return false;

      // (b) online softmax with a lazily moved reference maximum
      const int valid = min(BN, hi - (lo + j * BN));   // rows of this tile in the segment
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      if (valid == BN) {
#pragma unroll
        for (int i = 0; i < BN; i += 2)
          mx4[(i >> 1) & 3] = fmax3(mx4[(i >> 1) & 3], sc[i], sc[i + 1]);
      } else {
#pragma unroll
        for (int i = 0; i < BN; ++i)
          if (i < valid) mx4[i & 3] = fmaxf(mx4[i & 3], sc[i]);
      }
      const float mt = fmaxf(fmax3(mx4[0], mx4[1], mx4[2]), mx4[3]) * c_log2;
      float alpha = 1.f;
      bool need = false;
      if (j == 0) {
        m_run = mt;
      } else if (mt > m_run + kLazy) {
        alpha = ex2(m_run - mt);
        l_run *= alpha;
        m_run = mt;
        need = true;
      }
      const uint64_t negm2 = f2(-m_run, -m_run);
      uint32_t pk[BN / 2];
      uint64_t sum4[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
      for (int i = 0; i < BN / 2; ++i) {
        float e0, e1;
        f2_split(ffma2(f2(sc[2 * i], sc[2 * i + 1]), c2, negm2), e0, e1);
        float p0 = ex2(e0), p1 = ex2(e1);
        if (valid != BN) {
          p0 = 2 * i < valid ? p0 : 0.f;
          p1 = 2 * i + 1 < valid ? p1 : 0.f;
        }
        sum4[i & 3] = fadd2(sum4[i & 3], f2(p0, p1));
        pk[i] = pack_bf16x2(p0, p1);
      }
      float s_lo, s_hi;
      f2_split(fadd2(fadd2(sum4[0], sum4[1]), fadd2(sum4[2], sum4[3])), s_lo, s_hi);
      l_run += s_lo + s_hi;

      // P_{j-1} V_{j-1} done: its P columns are free, and O may be rescaled
      if (j >= 1 && !__all_sync(0xffffffffu,
                                mbar_wait(smem_u32(&bars->pv_done), (uint32_t)((j - 1) & 1)) &&
                                    !*abort_flag))
        return false;
      tc_fence_after();
      if (__any_sync(0xffffffffu, need)) {
#pragma unroll 1
        for (int blk = 0; blk < 8; ++blk) {
          uint32_t v[32];
          tmem_ld32(tm + lane_off + 32 * blk, v);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
          tmem_st32(tm + lane_off + 32 * blk, v);
        }
      }
      tmem_st32(tm + lane_off + kTmemP, pk);            // keys 2c, 2c+1 in column c
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&bars->p_full));

      return true;
    };
    for (int j = 0; ok && j < nt; ++j) ok = (j & 1) ? step(j, own_b, own_a) : step(j, own_a, own_b);

    // epilogue: O of this CTA's 256 dims, normalised (one segment) or as a
    // partial state (o unnormalised, m in log2 units, l) for the merge
    if (ok) {
      const int jl = nt - 1;
      if (!__all_sync(0xffffffffu,
                      mbar_wait(smem_u32(&bars->pv_done), (uint32_t)(jl & 1)) && !*abort_flag)) {
        ok = false;
      } else {
        tc_fence_after();
        if (S == 1) {
          const float inv = 1.f / l_run;
          uint4* dst = reinterpret_cast<uint4*>(O + bh * kDv + 256 * rank);
          const bool o_ok = row_ok && RF_IN(err, bh * kDv + 256 * rank + 255, n_bat * Hq * kDv);
#pragma unroll 1
          for (int blk = 0; blk < 8; ++blk) {
            uint32_t v[32];
            tmem_ld32(tm + lane_off + 32 * blk, v);
            tmem_ld_wait();
            if (o_ok) {
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                const float* f = reinterpret_cast<const float*>(v + 8 * c);
                dst[blk * 4 + c] = make_uint4(pack_bf16x2(f[0] * inv, f[1] * inv),
                                              pack_bf16x2(f[2] * inv, f[3] * inv),
                                              pack_bf16x2(f[4] * inv, f[5] * inv),
                                              pack_bf16x2(f[6] * inv, f[7] * inv));
              }
            }
          }
        } else {
          const int64_t ps = bh * S + seg;
          uint4* dst = reinterpret_cast<uint4*>(part_o + ps * kDv + 256 * rank);
          const bool p_ok = row_ok && RF_IN(err, ps, n_bat * Hq * S);
#pragma unroll 1
          for (int blk = 0; blk < 8; ++blk) {
            uint32_t v[32];
            tmem_ld32(tm + lane_off + 32 * blk, v);
            tmem_ld_wait();
            if (p_ok) {
#pragma unroll
              for (int c = 0; c < 8; ++c)
                dst[blk * 8 + c] = make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
            }
          }
          if (rank == 0 && p_ok)
            reinterpret_cast<float2*>(part_ml)[ps] = make_float2(m_run, l_run);
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
    tmem_dealloc(tm, kTmemCols);
  }
  // the peer may still write into this CTA's exchange slots until both CTAs
  // are done
  cluster_sync();
}

// Merge of the S partial states of every (batch, head): M = max m_j,
// L = sum l_j 2^(m_j - M), O = sum o_j 2^(m_j - M) / L.  One CTA per (batch,
// head), thread t = dims 4t .. 4t+3.  Launched as a programmatic dependent of
// the partial kernel; waits for it (griddepcontrol.wait) before reading.
__global__ void __launch_bounds__(kMergeThreads)
    mla_merge_kernel(const float* __restrict__ part_o, const float* __restrict__ part_ml,
                     __nv_bfloat16* __restrict__ O, int S, unsigned* err) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int64_t bh = blockIdx.x;
  // every state of this (batch, head) and its output row lie in the buffers
  if (!RF_IN(err, bh * S + S - 1, (int64_t)gridDim.x * S)) return;
  const float2* ml = reinterpret_cast<const float2*>(part_ml) + bh * S;
  const float4* po = reinterpret_cast<const float4*>(part_o + bh * S * kDv) + threadIdx.x;
  float M = -INFINITY;
  for (int j = 0; j < S; ++j) M = fmaxf(M, ml[j].x);
  float L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j = 0; j < S; ++j) {
    const float2 v = ml[j];
    const float w = exp2f(v.x - M);
    L += v.y * w;
    const float4 o = po[(int64_t)j * (kDv / 4)];
    acc.x = fmaf(o.x, w, acc.x);
    acc.y = fmaf(o.y, w, acc.y);
    acc.z = fmaf(o.z, w, acc.z);
    acc.w = fmaf(o.w, w, acc.w);
  }
  const float inv = 1.f / L;
  uint2 out;
  out.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  out.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  reinterpret_cast<uint2*>(O + bh * kDv)[threadIdx.x] = out;
}

}  // namespace

// Segments per batch.  A cluster (two SMs) takes one (batch, segment); the
// cost of a choice is modelled in units of one tile's time per cluster:
// waves * (tiles per segment + ~4 of start-up + ~2 to write a partial state)
// plus the merge's reads of every partial state (at HBM rate, ~8 tiles per
// 16 MB).  Segments hold whole tiles, and no segment is empty.
int mla_num_splits(int B, int Hq, int Lk, int requested) {
  const int ntiles = (Lk + BN - 1) / BN;
  auto fix = [&](int s) {          // the segment count that tps = ceil(ntiles / s) yields
    const int tps = (ntiles + s - 1) / s;
    return (ntiles + tps - 1) / tps;
  };
  if (requested > 0) return fix(requested < ntiles ? requested : ntiles);
  const int sms = sm_count();
  if (sms < 2) return 0;
  const int64_t pairs = sms / 2;
  double best = 1e300;
  int best_s = 1;
  for (int s = 1; s <= ntiles && s <= 64; ++s) {
    const int se = fix(s);
    if (se != s) continue;
    const int64_t tps = (ntiles + s - 1) / s;
    const int64_t clusters = (int64_t)B * s;
    const int64_t waves = (clusters + pairs - 1) / pairs;
    double cost = (double)waves * (double)(tps + 4 + (s > 1 ? 2 : 0));
    if (s > 1) cost += 8.0 * (double)B * Hq * s * kDv * 4 / (16.0 * (1 << 20));
    if (cost < best) {
      best = cost;
      best_s = s;
    }
  }
  return best_s;
}

size_t mla_workspace_bytes(int B, int Hq, int S) {
  if (S <= 1) return 0;
  const size_t n = (size_t)B * Hq * S;
  const size_t o_bytes = (n * kDv * sizeof(float) + 255) & ~(size_t)255;
  return o_bytes + n * 2 * sizeof(float);
}

cudaError_t launch_mla_decode(const void* Q, const void* CKV, void* O, int B, int Hq, int Lk,
                              float scale, int S, void* workspace, unsigned* err, cudaStream_t s) {
  CUtensorMap tmC;
  if (!encode_tmap_2d(&tmC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, CKV, kDqk, (uint64_t)B * Lk,
                      kDqk * 2, 64, BN, true))
    return cudaErrorInvalidValue;
  const int ntiles = (Lk + BN - 1) / BN;
  const int tps = (ntiles + S - 1) / S;
  if (S < 1 || (int64_t)(S - 1) * tps >= ntiles) return cudaErrorInvalidValue;
  const int64_t clusters = (int64_t)B * S;
  if (clusters * 2 >= (1ll << 31)) return cudaErrorInvalidValue;
  float* part_o = nullptr;
  float* part_ml = nullptr;
  if (S > 1) {
    const size_t n = (size_t)B * Hq * S;
    part_o = static_cast<float*>(workspace);
    part_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                       ((n * kDv * sizeof(float) + 255) & ~(size_t)255));
  }
  cudaError_t e = cudaFuncSetAttribute(mla_decode_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * clusters), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const float c_log2 = scale * 1.4426950408889634f;
  e = cudaLaunchKernelEx(&cfg, mla_decode_kernel, tmC, static_cast<const __nv_bfloat16*>(Q),
                         static_cast<__nv_bfloat16*>(O), part_o, part_ml, Hq, Lk, S, tps, c_log2,
                         err);
  if (e != cudaSuccess || S == 1) return e;
  cudaLaunchConfig_t mcfg = {};
  mcfg.gridDim = dim3((unsigned)((int64_t)B * Hq), 1, 1);
  mcfg.blockDim = dim3(kMergeThreads, 1, 1);
  mcfg.stream = s;
  cudaLaunchAttribute mattr[1];
  mattr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  mattr[0].val.programmaticStreamSerializationAllowed = 1;
  mcfg.attrs = mattr;
  mcfg.numAttrs = 1;
  return cudaLaunchKernelEx(&mcfg, mla_merge_kernel, (const float*)part_o, (const float*)part_ml,
                            static_cast<__nv_bfloat16*>(O), S, err);
}

}  // namespace rf
