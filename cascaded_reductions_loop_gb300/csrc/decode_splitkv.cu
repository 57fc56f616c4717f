// decode_splitkv.cu -- multi-segment (split-KV) fused decode attention.
//
// Multi-segment strategy ([S] Methodologie 3; [E] §3.3 inter-block merge and
// multi-kernel cooperation): the keys of every (batch, kv head) are cut into
// S segments.  Kernel 1 (decode_partial_kernel, a persistent grid of one CTA
// per SM) takes the segments as work items; the four warps of the CTA that
// takes an item each run the incremental safe-softmax loop ([E] §2.3, §4.1)
// over every fourth chunk of the segment and write their partial state
// (m, l, o) -- o unnormalised, m in log2 units -- for each of the G query heads
// that share the kv head.  Kernel 2 (decode_merge_kernel, launched as a
// programmatic dependent of kernel 1) combines the 4 S partial states of
// every (batch, query head): M = max m_j,
// L = sum l_j 2^(m_j - M), O = sum o_j 2^(m_j - M) / L.  (Merging inside
// kernel 1, by the last warp to finish a group, was measured slower: each
// warp must make its states visible with a fence before taking a ticket, and
// the merging warp falls behind the others.)
//
// Data movement: K and V stream from HBM exactly once, by TMA into 128-byte
// swizzled shared-memory tiles (chunks of 32 keys x 128 dims, two 64-dim
// boxes each), one private ring of stages per warp.  The G (<= 8) query rows
// of a kv head form the M = 16 side of mma.sync m16n8k16 bf16 tiles with fp32
// accumulation: S = Q K^T, then O += P V with P rounded to bf16; the row max,
// exp2 and sums stay in registers (quad shuffles).
#include <math.h>

#include <mutex>

#include "rf_device.cuh"
#include "rf_internal.h"

namespace rf {
namespace {

constexpr int kD = 128;          // head dim
constexpr int kCK = 32;          // keys per chunk
constexpr int kStages = 2;       // ring depth per warp
constexpr int kWarps = 4;        // consumer warps per CTA
constexpr int kBoxBytes = kCK * 128;             // one 64-dim box of kCK rows
constexpr int kStageBytes = 4 * kBoxBytes;       // K box0, K box1, V box0, V box1
constexpr int kSmemBytes = kWarps * kStages * kStageBytes + 1024 + 256;

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// Byte offset of 16-byte chunk c (0..15, i.e. dims 8c..8c+7) of key row r in
// a K or V stage (two 64-dim boxes, each 128-byte swizzled).
__device__ __forceinline__ uint32_t sw_off(int r, int c) {
  return (uint32_t)((c >> 3) * kBoxBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// A work item is one key segment of one (batch, kv head): item = (b * Hkv +
// kvh) * S + seg.  The grid is persistent: CTA c takes items c, c + gridDim.x,
// ...  Within a CTA, warp w takes chunks w, w + kWarps, ... of each item in
// turn; its private ring is refilled across item boundaries, so the next
// item's keys are already in flight while the current item's partial state
// is merged and written.
struct DecodeItem {
  int b, kvh, seg;
  int64_t lo, hi, row_base;
  int nchunks;
};

__device__ __forceinline__ DecodeItem decode_item(int item, int Hkv, int Lk, int S) {
  DecodeItem it;
  it.seg = item % S;
  const int pair = item / S;
  it.kvh = pair % Hkv;
  it.b = pair / Hkv;
  it.lo = (int64_t)it.seg * Lk / S;
  it.hi = (int64_t)(it.seg + 1) * Lk / S;
  it.row_base = (int64_t)pair * Lk;
  it.nchunks = (int)((it.hi - it.lo + kCK - 1) / kCK);
  return it;
}

template <int G>
__global__ void __launch_bounds__(kWarps * 32)
    decode_partial_kernel(const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV,
                          const __nv_bfloat16* __restrict__ Q, float* __restrict__ part_o,
                          float* __restrict__ part_ml, int Hq, int Hkv, int Lk, int S, int items,
                          float qk_scale_log2, unsigned* err) {
  static_assert(G >= 1 && G <= 8, "query heads per kv head");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kWarps * kStages * kStageBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int my_items =
      items > (int)blockIdx.x ? (items - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x : 0;
  uint8_t* my_stage = smem + warp * kStages * kStageBytes;
  uint64_t* my_full = bars + warp * kStages;

  if (lane == 0) {
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
#pragma unroll
    for (int i = 0; i < kStages; ++i) mbar_init(smem_u32(&my_full[i]), 1);
    fence_mbar_init();
  }
  __syncwarp();

  // producer cursor over this warp's chunk stream (lane 0 only)
  int pk = 0, pci = warp, issued = 0;
  DecodeItem pit = decode_item(my_items > 0 ? (int)blockIdx.x : 0, Hkv, Lk, S);
  auto skip_empty = [&]() {
    while (pk < my_items && pci >= pit.nchunks) {
      ++pk;
      pci = warp;
      if (pk < my_items) pit = decode_item((int)blockIdx.x + pk * (int)gridDim.x, Hkv, Lk, S);
    }
  };
  auto issue_next = [&]() {
    skip_empty();
    if (pk >= my_items) return;
    const int slot = issued % kStages;
    const int32_t row = (int32_t)(pit.row_base + pit.lo + (int64_t)pci * kCK);
    const uint32_t dst = smem_u32(my_stage + slot * kStageBytes);
    const uint32_t bar = smem_u32(&my_full[slot]);
    mbar_arrive_expect_tx(bar, kStageBytes);
    tma_load_2d(dst, &tmK, bar, 0, row);
    tma_load_2d(dst + kBoxBytes, &tmK, bar, 64, row);
    tma_load_2d(dst + 2 * kBoxBytes, &tmV, bar, 0, row);
    tma_load_2d(dst + 3 * kBoxBytes, &tmV, bar, 64, row);
    ++issued;
    pci += kWarps;
  };
  if (lane == 0)
    for (int i = 0; i < kStages; ++i) issue_next();
  // the merge kernel may be scheduled now; it waits for this grid to finish
  asm volatile("griddepcontrol.launch_dependents;");

  const int hrow = lane >> 2;           // head of this lane's accumulator rows
  const int kq = (lane & 3) * 2;        // first of this lane's two columns
  const int mi = lane >> 3, mr = lane & 7;   // ldmatrix: matrix, row within it
  int consumed = 0;
  bool failed = false;

  // Q of the G query heads as the A operand (rows zero-padded to 16); the
  // next item's Q is loaded while the current item runs.
  auto load_q = [&](int k, uint32_t (&q)[8][2]) {
    if (k >= my_items) return;
    const DecodeItem it = decode_item((int)blockIdx.x + k * (int)gridDim.x, Hkv, Lk, S);
    const uint32_t* qp = reinterpret_cast<const uint32_t*>(
        Q + ((int64_t)it.b * Hq + (int64_t)it.kvh * G + (hrow < G ? hrow : 0)) * kD);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      q[ks][0] = hrow < G ? __ldg(qp + ((ks * 16 + kq) >> 1)) : 0u;
      q[ks][1] = hrow < G ? __ldg(qp + ((ks * 16 + kq + 8) >> 1)) : 0u;
    }
  };
  uint32_t qa[8][2], qn[8][2];
  load_q(0, qn);

  for (int k = 0; k < my_items && !failed; ++k) {
    const DecodeItem it = decode_item((int)blockIdx.x + k * (int)gridDim.x, Hkv, Lk, S);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      qa[ks][0] = qn[ks][0];
      qa[ks][1] = qn[ks][1];
    }
    load_q(k + 1, qn);
    float oacc[16][4];
#pragma unroll
    for (int j = 0; j < 16; ++j) oacc[j][0] = oacc[j][1] = oacc[j][2] = oacc[j][3] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;

    for (int ci = warp; ci < it.nchunks; ci += kWarps) {
      const int slot = consumed % kStages;
      bool ok = mbar_wait(smem_u32(&my_full[slot]), (uint32_t)((consumed / kStages) & 1));
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        failed = true;
        break;
      }
      const uint32_t kbase = smem_u32(my_stage + slot * kStageBytes);
      const uint32_t vbase = kbase + 2 * kBoxBytes;
      const int64_t key0 = it.lo + (int64_t)ci * kCK;   // first key of the chunk

      // ---- S = Q K^T for 32 keys: two 16-key sub-blocks x two 8-key n-blocks
      float sc[2][2][4];
#pragma unroll
      for (int sb = 0; sb < 2; ++sb) {
        sc[sb][0][0] = sc[sb][0][1] = sc[sb][0][2] = sc[sb][0][3] = 0.f;
        sc[sb][1][0] = sc[sb][1][1] = sc[sb][1][2] = sc[sb][1][3] = 0.f;
        const int krow = sb * 16 + (mi >> 1) * 8 + mr;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          uint32_t r0, r1, r2, r3;
          ldsm_x4(kbase + sw_off(krow, 2 * ks + (mi & 1)), r0, r1, r2, r3);
          const uint32_t a[4] = {qa[ks][0], 0u, qa[ks][1], 0u};
          mma16816(sc[sb][0], a, r0, r1);
          mma16816(sc[sb][1], a, r2, r3);
        }
      }

      // ---- online softmax for head hrow over this chunk (log2 domain)
      float mx = -INFINITY;
#pragma unroll
      for (int sb = 0; sb < 2; ++sb)
#pragma unroll
        for (int nb = 0; nb < 2; ++nb)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int64_t key = key0 + sb * 16 + nb * 8 + kq + e;
            const float v = key < it.hi ? sc[sb][nb][e] * qk_scale_log2 : -INFINITY;
            sc[sb][nb][e] = v;
            mx = fmaxf(mx, v);
          }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run, mx);          // finite: every chunk has a valid key
      const float alpha = exp2f(m_run - m_new);      // 0 on the first chunk
      float psum = 0.f;
      uint32_t pa[2][2];
#pragma unroll
      for (int sb = 0; sb < 2; ++sb)
#pragma unroll
        for (int nb = 0; nb < 2; ++nb) {
          const float p0 = exp2f(sc[sb][nb][0] - m_new);
          const float p1 = exp2f(sc[sb][nb][1] - m_new);
          psum += p0 + p1;
          pa[sb][nb] = pack_bf16x2(p0, p1);
        }
      l_run = l_run * alpha + psum;
      m_run = m_new;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        oacc[j][0] *= alpha;
        oacc[j][1] *= alpha;
      }

      // ---- O += P V: A = P (16 rows x 16 keys), B = V (16 keys x 8 dims)
#pragma unroll
      for (int sb = 0; sb < 2; ++sb) {
        const uint32_t a[4] = {pa[sb][0], 0u, pa[sb][1], 0u};
        const int vrow = sb * 16 + (mi & 1) * 8 + mr;
#pragma unroll
        for (int j = 0; j < 16; j += 2) {
          uint32_t r0, r1, r2, r3;
          ldsm_x4_t(vbase + sw_off(vrow, j + (mi >> 1)), r0, r1, r2, r3);
          mma16816(oacc[j], a, r0, r1);
          mma16816(oacc[j + 1], a, r2, r3);
        }
      }

      __syncwarp();
      ++consumed;
      if (lane == 0) issue_next();               // refill the slot just freed
    }
    if (failed) break;

    // ---- this warp's partial state of the item (o unnormalised, m in log2
    // units); a warp without keys in the item writes (-inf, 0, 0)
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    if (hrow < G) {
      const int64_t pidx =
          (((int64_t)it.b * Hq + (int64_t)it.kvh * G + hrow) * S + it.seg) * kWarps + warp;
      float2* po = reinterpret_cast<float2*>(part_o + pidx * kD);
#pragma unroll
      for (int j = 0; j < 16; ++j) po[(j * 8 + kq) >> 1] = make_float2(oacc[j][0], oacc[j][1]);
      if ((lane & 3) == 0) reinterpret_cast<float2*>(part_ml)[pidx] = make_float2(m_run, l_run);
    }
  }

  if (failed) {
    raise_error(err, kDevErrTimeout);
    // let this warp's copies still in flight land before shared memory is released
    if (lane == 0)
      for (int c = consumed; c < issued; ++c)
        (void)mbar_wait(smem_u32(&my_full[c % kStages]), (uint32_t)((c / kStages) & 1), 1000000ull);
  }
}

// Merge kernel: one warp per (batch, query head), lane = 4 consecutive dims.
// Lane j holds the (m, l) of state j of each block of 32 states and hands its
// weight 2^(m_j - M) to the other lanes by shuffle; o is read 16 states at a
// time so that those loads are in flight together.  It is launched as a
// programmatic dependent of the partial kernel: its CTAs may start while the
// partial kernel drains and wait (griddepcontrol.wait) until that grid has
// finished and its writes are visible.
constexpr int kMergeWarps = 4;

__device__ __forceinline__ float4 o_block16(const float4* po, int j0, int n, float w,
                                            float4 acc) {
  float4 o[16];
  if (n >= 16) {                     // common case: no per-load condition
#pragma unroll
    for (int u = 0; u < 16; ++u) o[u] = po[(int64_t)(j0 + u) * (kD / 4)];
  } else {
#pragma unroll
    for (int u = 0; u < 16; ++u)
      o[u] = u < n ? po[(int64_t)(j0 + u) * (kD / 4)] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int u = 0; u < 16; ++u) {
    const float wu = __shfl_sync(0xffffffffu, w, (j0 + u) & 31);
    acc.x = fmaf(o[u].x, wu, acc.x);
    acc.y = fmaf(o[u].y, wu, acc.y);
    acc.z = fmaf(o[u].z, wu, acc.z);
    acc.w = fmaf(o[u].w, wu, acc.w);
  }
  return acc;
}

__global__ void __launch_bounds__(kMergeWarps * 32)
    decode_merge_kernel(const float* __restrict__ part_o, const float* __restrict__ part_ml,
                        __nv_bfloat16* __restrict__ O, int n_heads, int P) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int64_t bh = (int64_t)blockIdx.x * kMergeWarps + (threadIdx.x >> 5);
  if (bh >= n_heads) return;
  const float2* ml = reinterpret_cast<const float2*>(part_ml) + bh * P;
  const float4* po = reinterpret_cast<const float4*>(part_o + bh * P * kD) + lane;
  float M = -INFINITY;
  for (int j = lane; j < P; j += 32) M = fmaxf(M, ml[j].x);
  M = warp_max(M);                                 // finite: some segment has keys
  float L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int j0 = 0; j0 < P; j0 += 32) {
    const float2 v = j0 + lane < P ? ml[j0 + lane] : make_float2(-INFINITY, 0.f);
    const float w = exp2f(v.x - M);                // 0 for empty states
    L += v.y * w;
    acc = o_block16(po, j0, P - j0, w, acc);
    if (P - j0 > 16) acc = o_block16(po, j0 + 16, P - j0 - 16, w, acc);
  }
  const float inv = 1.f / warp_sum(L);
  uint2 out;
  out.x = pack_bf16x2(acc.x * inv, acc.y * inv);
  out.y = pack_bf16x2(acc.z * inv, acc.w * inv);
  reinterpret_cast<uint2*>(O + bh * kD)[lane] = out;
}

template <int G>
cudaError_t launch_g(const CUtensorMap& tmK, const CUtensorMap& tmV, const void* Q, void* O,
                     int B, int Hq, int Hkv, int Lk, float scale, int S, float* part_o,
                     float* part_ml, unsigned* err, cudaStream_t s) {
  auto kern = decode_partial_kernel<G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
  const int64_t items = (int64_t)B * Hkv * S;
  if (items >= (1ll << 31)) return cudaErrorInvalidValue;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidValue;
  const int grid = (int)(items < sms ? items : sms);        // one CTA per SM, persistent
  const float qk_scale_log2 = scale * 1.4426950408889634f;
  kern<<<grid, kWarps * 32, kSmemBytes, s>>>(tmK, tmV, static_cast<const __nv_bfloat16*>(Q),
                                             part_o, part_ml, Hq, Hkv, Lk, S, (int)items,
                                             qk_scale_log2, err);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int n_heads = B * Hq;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((n_heads + kMergeWarps - 1) / kMergeWarps, 1, 1);
  cfg.blockDim = dim3(kMergeWarps * 32, 1, 1);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_merge_kernel, (const float*)part_o,
                            (const float*)part_ml, static_cast<__nv_bfloat16*>(O), n_heads,
                            S * kWarps);
}

}  // namespace

int decode_num_splits(int B, int Hq, int Hkv, int Lk, int d, int requested) {
  (void)Hq;
  (void)d;
  if (requested > 0) return requested;
  const int sms = sm_count();
  if (sms <= 0) return 0;
  // The persistent grid has one CTA per SM.  Take the smallest S whose items
  // (B * Hkv * S) keep the SMs at least 95 % busy (items / (rounds * SMs)),
  // with segments of at least 128 keys (one chunk per warp); else the best S.
  const int64_t pairs = (int64_t)B * Hkv;
  const int64_t max_s = (Lk + 127) / 128 < 1 ? 1 : (Lk + 127) / 128;
  int best_s = 1;
  double best_eff = -1.0;
  for (int64_t S = 1; S <= max_s && S <= 4096; ++S) {
    const int64_t items = pairs * S;
    const int64_t rounds = (items + sms - 1) / sms;
    const double eff = (double)items / (double)(rounds * sms);
    if (eff >= 0.95) return (int)S;
    if (eff > best_eff) {
      best_eff = eff;
      best_s = (int)S;
    }
  }
  return best_s;
}

size_t decode_workspace_bytes(int B, int Hq, int d, int S) {
  const size_t n = (size_t)B * Hq * S * kWarps;       // one partial state per warp
  const size_t o_bytes = (n * d * sizeof(float) + 255) & ~(size_t)255;
  return o_bytes + n * 2 * sizeof(float);
}

cudaError_t launch_decode_splitkv(const void* Q, const void* K, const void* V, void* O, int B,
                                  int Hq, int Hkv, int Lk, int d, float scale, int S,
                                  void* workspace, unsigned* err, cudaStream_t s) {
  const uint64_t rows = (uint64_t)B * Hkv * Lk;
  CUtensorMap tmK, tmV;
  if (!encode_tmap_2d(&tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, kD, rows, kD * 2, 64, kCK, true) ||
      !encode_tmap_2d(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, V, kD, rows, kD * 2, 64, kCK, true))
    return cudaErrorInvalidValue;
  const size_t n = (size_t)B * Hq * S * kWarps;
  float* part_o = static_cast<float*>(workspace);
  float* part_ml = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                            ((n * d * sizeof(float) + 255) & ~(size_t)255));
  switch (Hq / Hkv) {
    case 1: return launch_g<1>(tmK, tmV, Q, O, B, Hq, Hkv, Lk, scale, S, part_o, part_ml, err, s);
    case 2: return launch_g<2>(tmK, tmV, Q, O, B, Hq, Hkv, Lk, scale, S, part_o, part_ml, err, s);
    case 4: return launch_g<4>(tmK, tmV, Q, O, B, Hq, Hkv, Lk, scale, S, part_o, part_ml, err, s);
    case 8: return launch_g<8>(tmK, tmV, Q, O, B, Hq, Hkv, Lk, scale, S, part_o, part_ml, err, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace rf

// ====================================================================
// Allocation-free variant of rf_attn_decode_splitkv.
//
// Some callers cannot hand this library a device buffer: a plugin reached
// through a fixed C interface that carries no workspace argument, a serving
// loop that forbids device allocation after start-up (cudaMalloc can
// synchronise the device and stall the loop), or a host framework whose pool
// allocator already holds nearly all device memory, so that a direct
// cudaMalloc would fail or fragment it.  For them the partial states live in
// the file-scope array below, which every GPU that loads the library keeps
// for the life of the process.
// ====================================================================

namespace rf {
namespace {

// Scratch for the partial (m, l, o) states of the split-KV decode.  Its size
// is part of the ABI (RF_DECODE_NOALLOC_SCRATCH_BYTES in rf.h).
constexpr size_t kNoAllocScratchBytes = RF_DECODE_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) uint8_t g_decode_scratch[kNoAllocScratchBytes];

constexpr int kMaxScratchDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxScratchDevices] = {};
void* g_scratch_ctx[kMaxScratchDevices] = {};

// Device address of g_decode_scratch on the current device.  In host code the
// array's name is only a host-side handle, so the address is looked up once
// per device (with that device current) and cached together with the CUDA
// context it belongs to; if the context changes (a device reset makes the
// runtime create a new one, with its own copy of the array), it is looked up
// again.  Returns nullptr on error.
void* decode_scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices) return nullptr;
  void* ctx = current_cu_context();
  {
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (g_scratch_ptr[dev] && ctx && ctx == g_scratch_ctx[dev]) return g_scratch_ptr[dev];
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return nullptr;
  ctx = current_cu_context();        // the lookup above creates the context if needed
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  g_scratch_ptr[dev] = p;
  g_scratch_ctx[dev] = ctx;
  return p;
}

}  // namespace
}  // namespace rf

extern "C" rf_status rf_attn_decode_splitkv_noalloc(const void* Q, const void* K, const void* V,
                                                    void* O, int B, int Hq, int Hkv, int Lk,
                                                    int d, float scale, int num_splits,
                                                    rf_stream_t stream) {
  // Nothing in the scratch has to start at zero: the partial kernel writes
  // every (batch, head, segment) state that the merge kernel reads.
  void* scratch = rf::decode_scratch_address();
  if (!scratch) return RF_ERR_CUDA;
  return rf_attn_decode_splitkv(Q, K, V, O, B, Hq, Hkv, Lk, d, scale, num_splits, scratch,
                                rf::kNoAllocScratchBytes, stream);
}

