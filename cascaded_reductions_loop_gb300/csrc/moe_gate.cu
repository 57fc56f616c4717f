// moe_gate.cu -- fused MoE gate: scores = x . W_gate^T -> top-k -> softmax of
// the selected scores ([E] §4.2), one kernel, no score matrix in HBM.
//
// Each CTA owns 128 tokens and one slice of the reduction dimension D; the
// CTAs covering the slices of the same 128 tokens form a thread-block
// cluster (split-K).  Per CTA: a TMA producer warp streams 128x64 tiles of x
// and Ex64 tiles of W_gate (both K-major, 128-byte swizzled) through a ring
// of stages (for E <= 64 two adjacent tiles of each per stage, so that every
// row's 256 bytes are fetched together); one thread issues tcgen05.mma
// kind::f16 (bf16 x bf16 -> fp32, M = 128, N = NE, the expert count rounded
// up to 32, 64, 128 or 256) into tensor memory.  The epilogue warps copy the
// partial 128 x NE score tile from TMEM to shared memory; after a cluster
// barrier each CTA sums its share of the rows over all cluster peers through
// distributed shared memory, in place (a CTA only ever writes the rows it
// finalises, which no peer reads), then one thread per token selects the top
// k of the E scores (descending score, ties to the lower expert index) and
// computes the softmax over the k selected scores.  Accumulator columns
// E..NE-1 come from unused rows of the W tile and are never read.
#include <math.h>

#include "rf_device.cuh"
#include "rf_internal.h"

namespace rf {
namespace {

constexpr int BM = 128;            // tokens per CTA
constexpr int BK = 64;             // bf16 elements per TMA box (one 128-byte swizzle row)
constexpr int kThreads = 192;      // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kXBox = BM * BK * 2;
constexpr int kRingBudget = 200 * 1024;

// Tile configuration for an MMA width of NE experts (32, 64, 128 or 256).
template <int NE>
struct GateCfg {
  static constexpr int kBoxes = NE <= 64 ? 2 : 1;          // boxes per stage
  static constexpr int KB = BK * kBoxes;                   // bf16 elements per k-block
  static constexpr int kWBox = NE * BK * 2;                // room for NE rows of W
  static constexpr int kABytes = kBoxes * kXBox;
  static constexpr int kStageBytes = kABytes + kBoxes * kWBox;
  static constexpr int kStages = kRingBudget / kStageBytes > 8 ? 8 : kRingBudget / kStageBytes;
  static constexpr int kRedStride = NE + 4;                // padded fp32 row of the score tile
  static constexpr int kRedBytes = BM * kRedStride * 4;
  static constexpr int kRing =
      kStages * kStageBytes > kRedBytes ? kStages * kStageBytes : kRedBytes;
  static constexpr int kSmem = kRing + 1024 + 256;
  static constexpr int kTmemCols = NE;
  static constexpr uint32_t kIdesc = make_idesc(BM, NE, /*bf16*/ 1, 0, 0);
  static_assert(kStages >= 2, "ring depth");
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

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
__device__ __forceinline__ float4 ld_peer_v4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// Top-KT of a row of E scores: a sorted insertion scan in expert order under
// the total order (score descending, expert index ascending).  An entry
// pushed down by a larger score carries its (lower) index, so it must also
// displace an equal score with a higher index further down.
template <int KT>
__device__ __forceinline__ void topk_softmax_row(const float* srow, int E, int32_t* idx_out,
                                                 float* w_out) {
  float v[KT];
  int ix[KT];
#pragma unroll
  for (int j = 0; j < KT; ++j) {
    v[j] = -INFINITY;
    ix[j] = E;
  }
#pragma unroll 4
  for (int e = 0; e < E; ++e) {
    float cv = srow[e];
    int ce = e;
#pragma unroll
    for (int j = 0; j < KT; ++j) {
      if (cv > v[j] || (cv == v[j] && ce < ix[j])) {
        const float tv = v[j];
        const int te = ix[j];
        v[j] = cv;
        ix[j] = ce;
        cv = tv;
        ce = te;
      }
    }
  }
  // softmax over the selected scores (v[0] is their max)
  float ex[KT], sum = 0.f;
#pragma unroll
  for (int j = 0; j < KT; ++j) {
    ex[j] = expf(v[j] - v[0]);
    sum += ex[j];
  }
#pragma unroll
  for (int j = 0; j < KT; ++j) {
    idx_out[j] = ix[j];
    w_out[j] = ex[j] / sum;
  }
}

template <int NE>
__global__ void __launch_bounds__(kThreads, 1)
    moe_gate_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                    int T, int D, int E, int k, int kb_per_cta, int32_t* __restrict__ idx_out,
                    float* __restrict__ w_out, unsigned* err) {
  using C = GateCfg<NE>;
  constexpr int kStages = C::kStages, KB = C::KB, kRedStride = C::kRedStride;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kRing);
  uint64_t* empty = full + kStages;
  uint64_t* accum = empty + kStages;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(accum + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  float* red = reinterpret_cast<float*>(smem);     // [BM][kRedStride], reuses the ring

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t crank = cluster_rank(), csize = cluster_size();
  const int m0 = blockIdx.y * BM;
  const int nkb_total = (D + KB - 1) / KB;
  const int kb0 = (int)crank * kb_per_cta;
  int nk = nkb_total - kb0;
  nk = nk < 0 ? 0 : (nk > kb_per_cta ? kb_per_cta : nk);
  const uint32_t stage_tx = (uint32_t)(C::kBoxes * (kXBox + E * BK * 2));

  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmX);
    prefetch_tmap(&tmW);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(smem_u32(&full[i]), 1);
      mbar_init(smem_u32(&empty[i]), 1);
    }
    mbar_init(smem_u32(accum), 1);
    *abort_flag = 0;
    fence_mbar_init();
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
      const uint64_t pol_x = policy_evict_first();   // x is streamed once
      const uint64_t pol_w = policy_evict_last();    // W_gate is re-read by every token tile
      int i = 0;
      for (; i < nk; ++i) {
        const int slot = i % kStages;
        if (i >= kStages &&
            !mbar_wait(smem_u32(&empty[slot]), (uint32_t)(((i / kStages) + 1) & 1))) {
          raise_error(err, kDevErrTimeout);
          *abort_flag = 1;
          break;
        }
        if (*abort_flag) break;
        uint8_t* a = smem + slot * C::kStageBytes;
        const uint32_t bar = smem_u32(&full[slot]);
        mbar_arrive_expect_tx(bar, stage_tx);
#pragma unroll
        for (int bx = 0; bx < C::kBoxes; ++bx) {
          const int x = (kb0 + i) * KB + bx * BK;
          tma_load_2d_hint(smem_u32(a + bx * kXBox), &tmX, bar, x, m0, pol_x);
          tma_load_2d_hint(smem_u32(a + C::kABytes + bx * C::kWBox), &tmW, bar, x, 0, pol_w);
        }
      }
      if (*abort_flag)
        for (int j = i - kStages < 0 ? 0 : i - kStages; j < i; ++j)
          (void)mbar_wait(smem_u32(&full[j % kStages]), (uint32_t)((j / kStages) & 1), 1000000ull);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      for (int i = 0; i < nk; ++i) {
        const int slot = i % kStages;
        if (!mbar_wait(smem_u32(&full[slot]), (uint32_t)((i / kStages) & 1))) {
          raise_error(err, kDevErrTimeout);
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t a = smem_u32(smem + slot * C::kStageBytes);
        const uint32_t b = a + C::kABytes;
#pragma unroll
        for (int kk = 0; kk < KB / 16; ++kk) {
          const uint32_t ao = (kk / (BK / 16)) * kXBox + (kk % (BK / 16)) * 32;
          const uint32_t bo = (kk / (BK / 16)) * C::kWBox + (kk % (BK / 16)) * 32;
          mma_bf16_ss(tmem, sw128_desc(a + ao, 1024, 16), sw128_desc(b + bo, 1024, 16), C::kIdesc,
                      (i | kk) != 0);
        }
        mma_commit(smem_u32(&empty[slot]));
      }
      mma_commit(smem_u32(accum));
    }
  } else {
    // partial scores: TMEM -> padded shared tile (row = token)
    const int sub = warp & 3;
    const int r = sub * 32 + lane;
    if (!mbar_wait(smem_u32(accum), 0)) {
      raise_error(err, kDevErrTimeout);
      *abort_flag = 1;
    }
    tc_fence_after();
#pragma unroll 1
    for (int c0 = 0; c0 < NE; c0 += 32) {
      uint32_t v[32];
      tmem_ld32(tmem + ((uint32_t)(sub * 32) << 16) + c0, v);
      tmem_ld_wait();
      float4* dst = reinterpret_cast<float4*>(red + r * kRedStride + c0);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float4 f;
        f.x = nk > 0 ? __uint_as_float(v[4 * q]) : 0.f;
        f.y = nk > 0 ? __uint_as_float(v[4 * q + 1]) : 0.f;
        f.z = nk > 0 ? __uint_as_float(v[4 * q + 2]) : 0.f;
        f.w = nk > 0 ? __uint_as_float(v[4 * q + 3]) : 0.f;
        dst[q] = f;
      }
    }
  }

  tc_fence_before();
  cluster_sync_all();        // every peer's partial tile is complete and visible

  // Split-K reduction: this CTA finalises rows [r_lo, r_hi) of the 128,
  // summing them over every cluster peer's partial tile, in place.
  const int rows_per = (BM + (int)csize - 1) / (int)csize;
  const int r_lo = (int)crank * rows_per;
  const int r_hi = min(BM, r_lo + rows_per);
  if (csize > 1 && warp >= 2) {
    constexpr int kCols = NE / 4;             // 4 threads per row
    const int t = threadIdx.x - 64;
    const int c0 = (t & 3) * kCols;
    for (int row = r_lo + (t >> 2); row < r_hi; row += 32) {
      float4 acc[kCols / 4];
#pragma unroll
      for (int q = 0; q < kCols / 4; ++q) acc[q] = make_float4(0.f, 0.f, 0.f, 0.f);
      const uint32_t local = smem_u32(red + row * kRedStride + c0);
      for (uint32_t p = 0; p < csize; ++p) {
        const uint32_t raddr = map_peer(local, p);
#pragma unroll
        for (int q = 0; q < kCols / 4; ++q) {
          const float4 f = ld_peer_v4(raddr + q * 16);
          acc[q].x += f.x;
          acc[q].y += f.y;
          acc[q].z += f.z;
          acc[q].w += f.w;
        }
      }
      float4* dst = reinterpret_cast<float4*>(red + row * kRedStride + c0);
#pragma unroll
      for (int q = 0; q < kCols / 4; ++q) dst[q] = acc[q];
    }
  }
  __syncthreads();
  if (warp >= 2 && !*abort_flag) {
    for (int row = r_lo + (threadIdx.x - 64); row < r_hi; row += 128) {
      const int tok = m0 + row;
      if (tok >= T) break;
      const float* srow = red + row * kRedStride;
      int32_t* io = idx_out + (size_t)tok * k;
      float* wo = w_out + (size_t)tok * k;
      switch (k) {
        case 1: topk_softmax_row<1>(srow, E, io, wo); break;
        case 2: topk_softmax_row<2>(srow, E, io, wo); break;
        case 3: topk_softmax_row<3>(srow, E, io, wo); break;
        case 4: topk_softmax_row<4>(srow, E, io, wo); break;
        case 5: topk_softmax_row<5>(srow, E, io, wo); break;
        case 6: topk_softmax_row<6>(srow, E, io, wo); break;
        case 7: topk_softmax_row<7>(srow, E, io, wo); break;
        default: topk_softmax_row<8>(srow, E, io, wo); break;
      }
    }
  }
  cluster_sync_all();        // no peer reads this CTA's tile any more

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Host side: tensor maps, the cluster split and the launch for one width.
template <int NE>
cudaError_t launch_ne(const void* X, const void* Wg, int T, int D, int E, int k, int32_t* idx,
                      float* w, unsigned* err, cudaStream_t s) {
  using C = GateCfg<NE>;
  CUtensorMap tmX, tmW;
  if (!encode_tmap_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, (uint64_t)D, (uint64_t)T,
                      (uint64_t)D * 2, BK, BM, true) ||
      !encode_tmap_2d(&tmW, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Wg, (uint64_t)D, (uint64_t)E,
                      (uint64_t)D * 2, BK, (uint32_t)E, true))
    return cudaErrorInvalidValue;
  // Split the reduction over a cluster of cs CTAs (one CTA per SM): pick the
  // cs in {1, 2, 4, 8} that minimises waves x (k-blocks per CTA + a fixed
  // per-CTA cost of about three k-blocks for start-up and epilogue).
  const int nkb = (D + C::KB - 1) / C::KB;
  const int tiles = (T + BM - 1) / BM;
  if (tiles > 65535) return cudaErrorInvalidValue;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidValue;
  int cs = 1;
  int64_t best = -1;
  for (int c = 1; c <= 8; c *= 2) {
    if (c > nkb) break;
    const int64_t waves = ((int64_t)tiles * c + sms - 1) / sms;
    const int64_t cost = waves * ((nkb + c - 1) / c + 3);
    if (best < 0 || cost < best) {
      best = cost;
      cs = c;
    }
  }
  const int kb_per = (nkb + cs - 1) / cs;

  cudaError_t e = cudaFuncSetAttribute(moe_gate_kernel<NE>,
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
  return cudaLaunchKernelEx(&cfg, moe_gate_kernel<NE>, tmX, tmW, T, D, E, k, kb_per, idx, w, err);
}

}  // namespace

cudaError_t launch_moe_gate(const void* X, const void* Wg, int T, int D, int E, int k,
                            int32_t* idx, float* w, unsigned* err, cudaStream_t s) {
  if (E <= 32) return launch_ne<32>(X, Wg, T, D, E, k, idx, w, err, s);
  if (E <= 64) return launch_ne<64>(X, Wg, T, D, E, k, idx, w, err, s);
  if (E <= 128) return launch_ne<128>(X, Wg, T, D, E, k, idx, w, err, s);
  if (E <= 256) return launch_ne<256>(X, Wg, T, D, E, k, idx, w, err, s);
  return cudaErrorInvalidValue;
}

}  // namespace rf
