// moe_gate.cu -- fused MoE gate: scores = x . W_gate^T -> top-k -> softmax of
// the selected scores ([E] §4.2), one kernel, no score matrix in HBM.
//
// Each CTA owns a tile of bm <= 128 tokens (bm chosen on the host so that the
// tiles fill the SMs evenly) and one slice of the reduction dimension D; the
// CTAs covering the slices of the same tile form a thread-block cluster
// (split-K).  Per CTA: a TMA producer warp streams bm x 64 tiles of x and
// the matching 64-dim slices of W_gate (128-byte swizzled) through a ring of
// stages (for E <= 64 two adjacent tiles of each per stage, so that every
// row's 256 bytes are fetched together).  W_gate may be expert-major, [E][D]
// (a K-major B operand: E rows of 64 dims per slice), or dim-major, [D][E]
// (an MN-major B operand: per slice, 64 rows of D, each 64 experts wide, one
// 8 KB box per 64 experts); one thread issues tcgen05.mma
// kind::f16 (bf16 x bf16 -> fp32, M = 128, N = NE, the expert count rounded
// up to 32, 64, 128 or 256) into tensor memory.  The epilogue warps copy the
// partial score tile out of TMEM: after a cluster barrier (every peer's ring
// is then free) each row is stored straight into the shared memory of the
// peer that finalises it -- CTA c owns rows [c*rows_per, (c+1)*rows_per) and
// receives one slot per peer -- with fire-and-forget distributed-shared-memory
// stores; after a second cluster barrier the top-k threads read the sum of
// the slots.  1-8 threads per token select the top k of the E scores (descending
// score, ties to the lower expert index) and compute the softmax over the k
// selected scores.  Accumulator columns E..NE-1 and rows bm..127 come from
// unused parts of the operand tiles and are never read.
#include <math.h>

#include "rf_device.cuh"
#include "rf_internal.h"

namespace rf {
namespace {

constexpr int BM = 128;            // the MMA's M: the largest tile of tokens
constexpr int BK = 64;             // bf16 elements per TMA box (one 128-byte swizzle row)
constexpr int kThreads = 192;      // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kRing = 200 * 1024;    // stages (runtime count) and, afterwards, the score tile
constexpr int kRingPad = 16 * 1024;  // the MMA reads 128 A rows / NE B rows past a short box
constexpr int kMaxStages = 8;

// Tile configuration for an MMA width of NE experts (32, 64, 128 or 256).
// A stage holds kBoxes x-boxes of bm rows, then kBoxes W-boxes of E rows
// (E rounded up to 8), each a 128-byte-swizzled box of 64 bf16 per row; the
// ring holds as many stages as fit (up to 8), so short tiles keep more
// bytes in flight.  The MMA always reads 128 x rows and NE W rows from a
// box's start: rows past the box are other boxes' data (or padding) and only
// feed accumulator rows / columns that are never read.
template <int NE>
struct GateCfg {
  static constexpr int kBoxes = NE <= 64 ? 2 : 1;          // boxes per stage
  static constexpr int KB = BK * kBoxes;                   // bf16 elements per k-block
  static constexpr int kRedStride = NE + 4;                // padded fp32 row of the score tile
  static constexpr int kRedBytes = (BM + 8) * kRedStride * 4;   // cs slots of ceil(bm/cs) rows
  static constexpr int kSmem = kRing + kRingPad + 1024 + 256;
  static constexpr int kTmemCols = NE;
  static constexpr uint32_t kIdesc = make_idesc(BM, NE, /*bf16*/ 1, 0, 0);
  static_assert(kRedBytes <= kRing, "score tile fits in the ring");
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

// Ring layout for a launch (the same on host and device).
struct Ring {
  int a_box, w_box, stage, stages;
};
template <int NE>
__host__ __device__ inline Ring ring_layout(int bm, int E) {
  using C = GateCfg<NE>;
  Ring r;
  r.a_box = bm * BK * 2;
  r.w_box = ((E + 7) / 8) * 8 * BK * 2;
  r.stage = C::kBoxes * (r.a_box + r.w_box);
  r.stages = kRing / r.stage > kMaxStages ? kMaxStages : kRing / r.stage;
  return r;
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
__device__ __forceinline__ uint32_t map_peer(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

// Top-k under the total order (score descending, expert index ascending).
// A list holds KT entries in that order.  insert() adds (cv, ce) when every
// entry of equal score already in the list has a lower index -- true for a
// scan in ascending expert order, and for merging a list of higher experts
// into one of lower experts -- so (cv, ce) ranks above entry j exactly when
// cv > v[j].  Branch-free: each slot takes the previous slot's entry, the new
// one, or keeps its own.
template <int KT>
__device__ __forceinline__ void topk_insert(float (&v)[KT], int (&ix)[KT], float cv, int ce) {
#pragma unroll
  for (int j = KT - 1; j > 0; --j) {
    const bool above_prev = cv > v[j - 1];
    const bool above = cv > v[j];
    v[j] = above_prev ? v[j - 1] : (above ? cv : v[j]);
    ix[j] = above_prev ? ix[j - 1] : (above ? ce : ix[j]);
  }
  const bool above0 = cv > v[0];
  v[0] = above0 ? cv : v[0];
  ix[0] = above0 ? ce : ix[0];
}

// insert() into four independent lists at once, one element each, written
// slot by slot across the lists so that the four compare/select chains are
// interleaved instruction by instruction.
template <int KT>
__device__ __forceinline__ void topk_insert4(float (&v)[4][KT], int (&ix)[4][KT],
                                             const float (&cv)[4], const int (&ce)[4]) {
#pragma unroll
  for (int j = KT - 1; j > 0; --j) {
    bool above_prev[4], above[4];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      above_prev[c] = cv[c] > v[c][j - 1];
      above[c] = cv[c] > v[c][j];
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      v[c][j] = above_prev[c] ? v[c][j - 1] : (above[c] ? cv[c] : v[c][j]);
      ix[c][j] = above_prev[c] ? ix[c][j - 1] : (above[c] ? ce[c] : ix[c][j]);
    }
  }
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const bool above0 = cv[c] > v[c][0];
    v[c][0] = above0 ? cv[c] : v[c][0];
    ix[c][0] = above0 ? ce[c] : ix[c][0];
  }
}

// Top-KT and softmax of one token row (the sum of its nslots partial rows,
// slot_floats apart), split over tpr (1, 2, 4 or 8) consecutive lanes: lane
// `part` takes experts [part*chunk, (part+1)*chunk)
// and scans them as four contiguous runs kept in four independent lists (so
// that four insertions are in flight at once), merges the lists (each run's
// list into the one of the run before it), then log2(tpr) butterfly rounds
// merge the partners' lists (the list of the lower experts is the base).
// Every lane of the warp must call this (shuffles); `live` marks lanes whose
// row exists.
template <int KT>
__device__ __forceinline__ void topk_softmax_row(const float* srow, int nslots, int slot_floats,
                                                 int E, int tpr, int part, bool live,
                                                 int32_t* idx_out, float* w_out) {
  float v[4][KT];
  int ix[4][KT];
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int j = 0; j < KT; ++j) {
      v[c][j] = -INFINITY;
      ix[c][j] = E;
    }
  const int chunk = (E + tpr - 1) / tpr;
  const int e0 = part * chunk, e1 = min(E, e0 + chunk);
  const int run = (chunk + 3) / 4;
  // Blocks of 4 elements per run: the 16 loads are issued unconditionally
  // (an index past the run reads at most a few floats beyond the row, still
  // inside the score tile's shared memory) and masked to -inf, which is never
  // inserted.
  for (int i0 = 0; i0 < run; i0 += 4) {
    float cv[4][4];
#pragma unroll
    for (int c = 0; c < 4; ++c)
#pragma unroll
      for (int u = 0; u < 4; ++u) cv[c][u] = srow[e0 + c * run + i0 + u];
    for (int sl = 1; sl < nslots; ++sl)          // split-K partial sums of the cluster
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int u = 0; u < 4; ++u) cv[c][u] += srow[sl * slot_floats + e0 + c * run + i0 + u];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float x[4];
      int xe[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        xe[c] = e0 + c * run + i0 + u;
        x[c] = (i0 + u < run && xe[c] < e1) ? cv[c][u] : -INFINITY;
      }
      topk_insert4(v, ix, x, xe);
    }
  }
#pragma unroll
  for (int j = 0; j < KT; ++j) {
    topk_insert(v[0], ix[0], v[1][j], ix[1][j]);
    topk_insert(v[2], ix[2], v[3][j], ix[3][j]);
  }
#pragma unroll
  for (int j = 0; j < KT; ++j) topk_insert(v[0], ix[0], v[2][j], ix[2][j]);
  for (int s = 1; s < tpr; s <<= 1) {
    const bool upper = (part & s) != 0;
    float a[KT], b[KT];
    int ai[KT], bi[KT];
#pragma unroll
    for (int j = 0; j < KT; ++j) {
      const float pv = __shfl_xor_sync(0xffffffffu, v[0][j], s);
      const int pi = __shfl_xor_sync(0xffffffffu, ix[0][j], s);
      a[j] = upper ? pv : v[0][j];
      ai[j] = upper ? pi : ix[0][j];
      b[j] = upper ? v[0][j] : pv;
      bi[j] = upper ? ix[0][j] : pi;
    }
#pragma unroll
    for (int j = 0; j < KT; ++j) topk_insert(a, ai, b[j], bi[j]);
#pragma unroll
    for (int j = 0; j < KT; ++j) {
      v[0][j] = a[j];
      ix[0][j] = ai[j];
    }
  }
  if (!live || part != 0) return;
  // softmax over the selected scores (v[0][0] is their max)
  float ex[KT], sum = 0.f;
#pragma unroll
  for (int j = 0; j < KT; ++j) {
    ex[j] = expf(v[0][j] - v[0][0]);
    sum += ex[j];
  }
#pragma unroll
  for (int j = 0; j < KT; ++j) {
    idx_out[j] = ix[0][j];
    w_out[j] = ex[j] / sum;
  }
}

__device__ __forceinline__ void st_peer_v4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1,%2,%3,%4};" ::"r"(addr), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}

// DE: W_gate is [D][E] (E a multiple of 64); else [E][D].
template <int NE, bool DE>
__global__ void __launch_bounds__(kThreads, 1)
    moe_gate_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                    int T, int D, int E, int k, int bm, int32_t* __restrict__ idx_out,
                    float* __restrict__ w_out, unsigned* err) {
  using C = GateCfg<NE>;
  // [D][E]: the MN-major B operand; its 64-expert atoms are 8 KB apart
  constexpr uint32_t kIdesc = DE ? make_idesc(BM, NE, /*bf16*/ 1, 0, /*B MN-major*/ 1) : C::kIdesc;
  constexpr int kAtom = 64 * BK * 2;               // 64 experts x 64 dims, bf16
  constexpr int KB = C::KB, kRedStride = C::kRedStride;
  const Ring rg = ring_layout<NE>(bm, E);
  const int nst = rg.stages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kRing + kRingPad);
  uint64_t* empty = full + kMaxStages;
  uint64_t* accum = empty + kMaxStages;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(accum + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  float* red = reinterpret_cast<float*>(smem);     // [BM][kRedStride], reuses the ring

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_rank(), csize = cluster_size();
  const int m0 = blockIdx.y * bm;                  // bm (<= 128) token rows per tile
  // k-blocks crank, crank + csize, ...: the peers of a cluster walk each
  // token row side by side, so their requests for a row arrive close together
  const int nkb_total = (D + KB - 1) / KB;
  const int nk = nkb_total > (int)crank ? (nkb_total - (int)crank + (int)csize - 1) / (int)csize : 0;
  const uint32_t stage_tx = (uint32_t)(C::kBoxes * (bm + E) * BK * 2);
  const uint64_t pol_x = policy_evict_first();     // x is streamed once
  const uint64_t pol_w = policy_evict_last();      // W_gate is re-read by every token tile
  // stage i: x rows m0 .. m0+bm-1 (the rest of the 128-row A tile is unused),
  // all E rows of W_gate, k-block crank + i * csize
  auto issue_stage = [&](int i) {
    const int slot = i % nst;
    uint8_t* a = smem + slot * rg.stage;
    const uint32_t bar = smem_u32(&full[slot]);
    mbar_arrive_expect_tx(bar, stage_tx);
#pragma unroll
    for (int bx = 0; bx < C::kBoxes; ++bx) {
      const int x = ((int)crank + i * (int)csize) * KB + bx * BK;
      tma_load_2d_hint(smem_u32(a + bx * rg.a_box), &tmX, bar, x, m0, pol_x);
      uint8_t* wb = a + C::kBoxes * rg.a_box + bx * rg.w_box;
      if (DE) {
        for (int e0 = 0; e0 < E; e0 += 64)       // box: 64 experts x 64 rows of D
          tma_load_2d_hint(smem_u32(wb + (e0 / 64) * kAtom), &tmW, bar, e0, x, pol_w);
      } else {
        tma_load_2d_hint(smem_u32(wb), &tmW, bar, x, 0, pol_w);
      }
    }
  };

  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW);
    for (int i = 0; i < nst; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 1);
    }
    mbar_init(smem_u32(accum), 1);
    *abort_flag = 0;
    fence_mbar_init();
    // the ring starts filling while TMEM is allocated and the CTA syncs
    for (int i = 0; i < nst && i < nk; ++i) issue_stage(i);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_holder), C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 0) {
    if (lane == 0) {
      int i = nst < nk ? nst : nk;
      for (; i < nk; ++i) {
        const int slot = i % nst;
        if (!mbar_wait(smem_u32(&empty[slot]), (uint32_t)(((i / nst) + 1) & 1))) {
          raise_error(err, kDevErrTimeout);
          *abort_flag = 1;
          break;
        }
        if (*abort_flag) break;
        issue_stage(i);
      }
      if (*abort_flag)
        for (int j = i - nst < 0 ? 0 : i - nst; j < i; ++j)
          (void)mbar_wait(smem_u32(&full[j % nst]), (uint32_t)((j / nst) & 1), 1000000ull);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int i = 0; i < nk; ++i) {
        const int slot = i % nst;
        if (!mbar_wait(smem_u32(&full[slot]), (uint32_t)((i / nst) & 1))) {
          raise_error(err, kDevErrTimeout);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t a = smem_u32(smem + slot * rg.stage);
        const uint32_t b = a + C::kBoxes * rg.a_box;
#pragma unroll
        for (int kk = 0; kk < KB / 16; ++kk) {
          const uint32_t ao = (kk / (BK / 16)) * rg.a_box + (kk % (BK / 16)) * 32;
          // K-major: 16 dims = 32 bytes along a row; MN-major: 16 rows of D
          const uint32_t bo = (kk / (BK / 16)) * rg.w_box + (kk % (BK / 16)) * (DE ? 16 * 128 : 32);
          mma_bf16_ss(tmem, sw128_desc(a + ao, 1024, 16),
                      sw128_desc(b + bo, 1024, DE ? (uint32_t)kAtom : 16u), kIdesc, (i | kk) != 0);
        }
        mma_commit(smem_u32(&empty[slot]));
      }
      mma_commit(smem_u32(accum));
    }
  } else {
    if (!mbar_wait(smem_u32(accum), 0)) {
      raise_error(err, kDevErrTimeout);
      *abort_flag = 1;
    }
  }

  // This CTA finalises rows [r_lo, r_lo + rows_fin) of the tile's bm rows.
  // Receive area (in the ring, free once every peer's MMAs are done): slot c
  // = CTA c's partial scores of those rows, [rows_per][kRedStride] fp32.
  const int rows_per = (bm + (int)csize - 1) / (int)csize;
  const int r_lo = (int)crank * rows_per;
  const int rows_fin = max(0, min(bm, r_lo + rows_per) - r_lo);
  const int slot_floats = rows_per * kRedStride;
  tc_fence_before();
  if (csize > 1) cluster_sync_all();   // every peer's ring is free: pushes may land
  if (warp >= 2) {
    tc_fence_after();
    const int sub = warp & 3;
    const int r = sub * 32 + lane;                // TMEM lane = row of the tile
    const int dst_cta = r / rows_per;
    const bool mine = r < bm;
    const uint32_t dst = smem_u32(red + crank * slot_floats + (r - dst_cta * rows_per) * kRedStride);
    const uint32_t raddr = (csize > 1 && mine) ? map_peer(dst, (uint32_t)dst_cta) : dst;
#pragma unroll 1
    for (int c0 = 0; c0 < NE; c0 += 32) {
      uint32_t v[32];
      tmem_ld32(tmem + ((uint32_t)(sub * 32) << 16) + c0, v);   // warp-collective
      tmem_ld_wait();
      if (!mine) continue;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float4 f;
        f.x = nk > 0 ? __uint_as_float(v[4 * q]) : 0.f;
        f.y = nk > 0 ? __uint_as_float(v[4 * q + 1]) : 0.f;
        f.z = nk > 0 ? __uint_as_float(v[4 * q + 2]) : 0.f;
        f.w = nk > 0 ? __uint_as_float(v[4 * q + 3]) : 0.f;
        if (csize > 1)
          st_peer_v4(raddr + (c0 + 4 * q) * 4, f);
        else
          reinterpret_cast<float4*>(red + (size_t)r * kRedStride + c0)[q] = f;
      }
    }
  }
  if (csize > 1)
    cluster_sync_all();                 // all pushes have landed; no remote access after this
  else
    __syncthreads();

  if (warp >= 2 && !*abort_flag) {
    // tpr (1, 2, 4 or 8) threads per row: as many as the 128 threads allow
    const int t = threadIdx.x - 64;
    int tpr = 1;
    while (tpr < 8 && 2 * tpr * rows_fin <= 128) tpr *= 2;
    const int row = t / tpr, part = t % tpr;
    const int tok = m0 + r_lo + row;
    const bool live = row < rows_fin && tok < T && RF_IN(err, (int64_t)tok * k + k - 1, (int64_t)T * k);
    const float* srow = red + (live ? row : 0) * kRedStride;
    const int ns = (int)csize;
    int32_t* io = idx_out + (size_t)(live ? tok : 0) * k;
    float* wo = w_out + (size_t)(live ? tok : 0) * k;
    switch (k) {
      case 1: topk_softmax_row<1>(srow, ns, slot_floats, E, tpr, part, live, io, wo); break;
      case 2: topk_softmax_row<2>(srow, ns, slot_floats, E, tpr, part, live, io, wo); break;
      case 3: topk_softmax_row<3>(srow, ns, slot_floats, E, tpr, part, live, io, wo); break;
      case 4: topk_softmax_row<4>(srow, ns, slot_floats, E, tpr, part, live, io, wo); break;
      case 5: topk_softmax_row<5>(srow, ns, slot_floats, E, tpr, part, live, io, wo); break;
      case 6: topk_softmax_row<6>(srow, ns, slot_floats, E, tpr, part, live, io, wo); break;
      case 7: topk_softmax_row<7>(srow, ns, slot_floats, E, tpr, part, live, io, wo); break;
      default: topk_softmax_row<8>(srow, ns, slot_floats, E, tpr, part, live, io, wo); break;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// The tile plan of a launch on `sms` SMs.
// Tile shape: a cluster of cs CTAs (one per SM) splits the D reduction of
// a tile of bm token rows.  For each cs in {1, 2, 4, 8}, bm is the multiple
// of 8 (<= 128) that spreads the tokens evenly over whole waves of clusters.
// Cost = waves x (k-blocks per CTA x time per k-block + a fixed per-CTA cost
// of about three k-blocks, plus one for the cluster reduction when cs > 1),
// in units of the HBM time of a 128-row k-block at an even share of the
// bandwidth.  Time per k-block = max(bm / 128, MMA time) + a fixed 0.35 for
// the stage's barrier round trip and its W tile (fitted to a sweep of cs and
// bm on GB300 at T = 8192, D = 4096, E in {8, 64, 256}: halving the rows
// per CTA does not halve the k-block time).  The MMA always covers 128
// rows; at an even HBM share (~24 B/clk per SM) its N = NE product takes
// about NE * 3 / 1024 of the unit.
struct GatePlan {
  int cs;      // CTAs per cluster (split of D)
  int bm;      // token rows per tile (a multiple of 8, <= 128)
  int tiles;   // clusters: ceil(T / bm)
};
template <int NE>
GatePlan gate_plan(int T, int D, int sms) {
  constexpr double kMmaPerKb = NE * 3.0 / 1024.0;
  constexpr double kStageFixed = 0.35;
  const int nkb = (D + GateCfg<NE>::KB - 1) / GateCfg<NE>::KB;
  int cs = 1, bm = BM;
  double best = -1.0;
  for (int c = 1; c <= 8; c *= 2) {
    if (c > nkb || c > sms) break;
    const int64_t per_wave = sms / c;                        // clusters per wave
    const int64_t waves = (T + per_wave * BM - 1) / (per_wave * BM);
    int b = (int)((T + waves * per_wave - 1) / (waves * per_wave));
    b = b < 8 ? 8 : ((b + 7) / 8) * 8;
    if (b > BM) b = BM;
    const double per_kb =
        ((double)b / BM > kMmaPerKb ? (double)b / BM : kMmaPerKb) + kStageFixed;
    const double cost = (double)waves * (per_kb * ((nkb + c - 1) / c) + 3 + (c > 1));
    if (best < 0 || cost < best) {
      best = cost;
      cs = c;
      bm = b;
    }
  }
  GatePlan gp;
  gp.cs = cs;
  gp.bm = bm;
  gp.tiles = (int)(((int64_t)T + bm - 1) / bm);
  return gp;
}

// Host side: tensor maps, the cluster split and the launch for one width.
template <int NE, bool DE>
cudaError_t launch_ne(const void* X, const void* Wg, int T, int D, int E, int k, int32_t* idx,
                      float* w, unsigned* err, cudaStream_t s) {
  using C = GateCfg<NE>;
  CUtensorMap tmX, tmW;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidValue;
  const GatePlan gp = gate_plan<NE>(T, D, sms);
  const int cs = gp.cs, bm = gp.bm;
  const int tiles = gp.tiles;
  if (tiles > 65535) return cudaErrorInvalidValue;
  if (!encode_tmap_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, (uint64_t)D, (uint64_t)T,
                      (uint64_t)D * 2, BK, (uint32_t)bm, true) ||
      !(DE ? encode_tmap_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Wg, (uint64_t)E, (uint64_t)D,
                            (uint64_t)E * 2, 64, BK, true)
           : encode_tmap_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Wg, (uint64_t)D, (uint64_t)E,
                            (uint64_t)D * 2, BK, (uint32_t)E, true)))
    return cudaErrorInvalidValue;

  cudaError_t e = cudaFuncSetAttribute(moe_gate_kernel<NE, DE>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs, tiles, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, moe_gate_kernel<NE, DE>, tmX, tmW, T, D, E, k, bm, idx, w, err);
}

}  // namespace

cudaError_t launch_moe_gate(const void* X, const void* Wg, int T, int D, int E, int k,
                            bool w_de, int32_t* idx, float* w, unsigned* err, cudaStream_t s) {
  if (w_de) {                                      // [D][E]: E % 64 == 0, checked by the caller
    if (E == 64) return launch_ne<64, true>(X, Wg, T, D, E, k, idx, w, err, s);
    if (E == 128) return launch_ne<128, true>(X, Wg, T, D, E, k, idx, w, err, s);
    if (E == 192 || E == 256) return launch_ne<256, true>(X, Wg, T, D, E, k, idx, w, err, s);
    return cudaErrorInvalidValue;
  }
  if (E <= 32) return launch_ne<32, false>(X, Wg, T, D, E, k, idx, w, err, s);
  if (E <= 64) return launch_ne<64, false>(X, Wg, T, D, E, k, idx, w, err, s);
  if (E <= 128) return launch_ne<128, false>(X, Wg, T, D, E, k, idx, w, err, s);
  if (E <= 256) return launch_ne<256, false>(X, Wg, T, D, E, k, idx, w, err, s);
  return cudaErrorInvalidValue;
}

// Host-side check of the tile plan (gate_plan, with the width the launcher
// picks for E) for T tokens of D dims on `sms` SMs.  Returns 0 when it
// holds, -1 for sizes the call refuses, else the number of the first check
// that fails:
//   1 the cluster size is 1, 2, 4 or 8 and at most the k-blocks and the SMs;
//   2 the tile height is a multiple of 8 in 8..128;
//   3 the tiles hold every token once and none is empty;
//   4 the tiles fit the grid's y extent (65535) whenever T <= 65535 * 120;
//   5 the cluster's CTAs share the k-blocks with none left out or idle;
//   6 the epilogue's rows (ceil(bm / cs) per CTA) cover the tile.
int moe_plan_selfcheck(int T, int D, int E, int sms) {
  if (T < 1 || D < 1 || D % 8 != 0 || E < 1 || E > 256 || sms < 1) return -1;
  GatePlan gp;
  int kb;
  if (E <= 32) {
    gp = gate_plan<32>(T, D, sms);
    kb = GateCfg<32>::KB;
  } else if (E <= 64) {
    gp = gate_plan<64>(T, D, sms);
    kb = GateCfg<64>::KB;
  } else if (E <= 128) {
    gp = gate_plan<128>(T, D, sms);
    kb = GateCfg<128>::KB;
  } else {
    gp = gate_plan<256>(T, D, sms);
    kb = GateCfg<256>::KB;
  }
  const int nkb = (D + kb - 1) / kb;
  const int cs = gp.cs, bm = gp.bm;
  if ((cs != 1 && cs != 2 && cs != 4 && cs != 8) || cs > nkb || cs > sms) return 1;
  if (bm % 8 != 0 || bm < 8 || bm > BM) return 2;
  if ((int64_t)gp.tiles * bm < T || (int64_t)(gp.tiles - 1) * bm >= T) return 3;
  if (T <= 65535 * 120 && gp.tiles > 65535) return 4;
  int shared = 0;
  for (int r = 0; r < cs; ++r) {
    const int nk = nkb > r ? (nkb - r + cs - 1) / cs : 0;
    if (nk < 1) return 5;
    shared += nk;
  }
  if (shared != nkb) return 5;
  if (((bm + cs - 1) / cs) * cs < bm) return 6;
  return 0;
}

}  // namespace rf
