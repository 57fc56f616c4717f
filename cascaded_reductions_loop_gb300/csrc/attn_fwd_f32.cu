// attn_fwd_f32.cu -- single-segment fused attention in exact fp32 on the CUDA
// cores (no tensor cores, no approximate exponentials).
//
// Safe-softmax cascade ([E] §2.2) fused into one loop with the incremental
// form ([E] §2.3, §4.1; [S] Methodologie 2): each warp owns one query row and
// walks the key tiles once, keeping (m, l, o) in registers; when a tile
// raises the running max from m to m', the earlier l and o are multiplied by
// exp(m - m').  K/V tiles of 32 keys are staged in shared memory and shared
// by the CTA's four warps.
#include <math.h>

#include "rf_device.cuh"
#include "rf_internal.h"

namespace rf {
namespace {

constexpr int kWarps = 4;
constexpr int kTileKeys = 32;

template <int D>
__global__ void __launch_bounds__(kWarps * 32)
    attn_fwd_f32_kernel(const float* __restrict__ Q, const float* __restrict__ K,
                        const float* __restrict__ V, float* __restrict__ O, int Lq, int Lk,
                        float scale) {
  static_assert(D % 32 == 0, "head dim must be a multiple of 32");
  constexpr int C = D / 32;                   // output columns per lane
  __shared__ float ks[kTileKeys][D + 1];      // +1: lane j reads row j conflict-free
  __shared__ float vs[kTileKeys][D];
  __shared__ float qs[kWarps][D];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t bh = blockIdx.y;
  const int row = blockIdx.x * kWarps + warp;
  const bool active = row < Lq;
  const float* Kp = K + bh * (size_t)Lk * D;
  const float* Vp = V + bh * (size_t)Lk * D;

  const float* Qp = Q + (bh * (size_t)Lq + (active ? row : 0)) * D;
  for (int i = lane; i < D; i += 32) qs[warp][i] = Qp[i];

  float m = -INFINITY, l = 0.f, o[C];
#pragma unroll
  for (int c = 0; c < C; ++c) o[c] = 0.f;

  for (int t0 = 0; t0 < Lk; t0 += kTileKeys) {
    __syncthreads();                           // previous tile fully consumed
    for (int i = threadIdx.x; i < kTileKeys * D; i += kWarps * 32) {
      const int r = i / D, cidx = i % D;
      const bool ok = t0 + r < Lk;
      ks[r][cidx] = ok ? Kp[(size_t)(t0 + r) * D + cidx] : 0.f;
      vs[r][cidx] = ok ? Vp[(size_t)(t0 + r) * D + cidx] : 0.f;
    }
    __syncthreads();

    // scores of this tile: lane j -> key t0 + j
    const bool valid = t0 + lane < Lk;
    float acc = 0.f;
#pragma unroll 8
    for (int i = 0; i < D; ++i) acc = fmaf(qs[warp][i], ks[lane][i], acc);
    const float s = valid ? acc * scale : -INFINITY;

    // running max, rescale factor, weights and running sum
    const float m_new = fmaxf(m, warp_max(s));
    const float alpha = expf(m - m_new);      // 0 on the first tile (m = -inf)
    const float p = valid ? expf(s - m_new) : 0.f;
    l = l * alpha + warp_sum(p);

#pragma unroll
    for (int c = 0; c < C; ++c) o[c] *= alpha;
    for (int j = 0; j < kTileKeys; ++j) {
      const float pj = __shfl_sync(0xffffffffu, p, j);
#pragma unroll
      for (int c = 0; c < C; ++c) o[c] = fmaf(pj, vs[j][c * 32 + lane], o[c]);
    }
    m = m_new;
  }

  if (active) {
    float* Op = O + (bh * (size_t)Lq + row) * D;
#pragma unroll
    for (int c = 0; c < C; ++c) Op[c * 32 + lane] = o[c] / l;
  }
}

}  // namespace

cudaError_t launch_attn_fwd_f32(const float* Q, const float* K, const float* V, float* O, int B,
                                int H, int Lq, int Lk, int d, float scale, cudaStream_t s) {
  dim3 grid((Lq + kWarps - 1) / kWarps, B * H);
  if (grid.y > 65535u) return cudaErrorInvalidValue;
  if (d == 64)
    attn_fwd_f32_kernel<64><<<grid, kWarps * 32, 0, s>>>(Q, K, V, O, Lq, Lk, scale);
  else
    attn_fwd_f32_kernel<128><<<grid, kWarps * 32, 0, s>>>(Q, K, V, O, Lq, Lk, scale);
  return cudaGetLastError();
}

}  // namespace rf
