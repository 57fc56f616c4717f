// attn_fwd_f32.cu -- single-segment fused attention in exact fp32 on the CUDA
// cores (no tensor cores, no approximate exponentials).
//
// Safe-softmax cascade ([E] §2.2) fused into one loop with the incremental
// form ([E] §2.3, §4.1; [S] Methodologie 2): each warp owns one query row and
// walks the key tiles once, keeping (m, l, o) in registers; when a tile
// raises the running max from m to m', the earlier l and o are multiplied by
// exp(m - m').  K/V tiles of 32 keys are staged in shared memory and shared
// by the CTA's four warps.  With the causal mask, row i reads keys
// j <= i + (Lk - Lq) only; the CTA stops after the last tile any of its rows
// can read, and a row that reads no key is written as zero.
//
// Two layouts: fixed-length [B][H][L][D], and packed variable-length
// sequences [total][H][D] delimited by cumulative lengths cu_seqlens[B + 1]
// (sequence b holds tokens cu[b] .. cu[b+1]-1); rows of one head are then H*D
// floats apart.
#include <math.h>

#include "rf_device.cuh"
#include "rf_internal.h"

namespace rf {
namespace {

constexpr int kWarps = 4;
constexpr int kTileKeys = 32;

// Where the rows of one (sequence, head) live: row i of Q/O at qo + i *
// stride, key j of K/V at kv + j * stride (offsets in elements).
struct Rows {
  int Lq, Lk;
  size_t qo, kv, stride;
  bool ok;
};

__device__ __forceinline__ Rows fixed_rows(int Lq, int Lk, int D) {
  const size_t bh = blockIdx.y;
  return {Lq, Lk, bh * (size_t)Lq * D, bh * (size_t)Lk * D, (size_t)D, true};
}

// Varlen: blockIdx.y = b * H + h.  Sizes that contradict the host-side totals
// are reported and the sequence is skipped (nothing out of bounds is touched).
__device__ __forceinline__ Rows varlen_rows(const int* cu_q, const int* cu_k, int H, int max_q,
                                            int total_q, int total_k, int D, unsigned* err) {
  const int b = blockIdx.y / H, h = blockIdx.y % H;
  const bool cu_ok = RF_IN(err, b + 1, gridDim.y / H + 1);  // cu_q, cu_k have B + 1 entries
  const int q0 = cu_ok ? cu_q[b] : 0, q1 = cu_ok ? cu_q[b + 1] : 0;
  const int k0 = cu_ok ? cu_k[b] : 0, k1 = cu_ok ? cu_k[b + 1] : 0;
  Rows r;
  r.ok = cu_ok && 0 <= q0 && q0 <= q1 && q1 <= total_q && q1 - q0 <= max_q && 0 <= k0 &&
         k0 <= k1 && k1 <= total_k;
  if (!r.ok) {
    if (threadIdx.x == 0 && blockIdx.x == 0) raise_error(err, kDevErrInput);
    return r;
  }
  r.Lq = q1 - q0;
  r.Lk = k1 - k0;
  r.qo = ((size_t)q0 * H + h) * D;
  r.kv = ((size_t)k0 * H + h) * D;
  r.stride = (size_t)H * D;
  return r;
}

template <int D>
__global__ void __launch_bounds__(kWarps * 32)
    attn_fwd_f32_kernel(const float* __restrict__ Q, const float* __restrict__ K,
                        const float* __restrict__ V, float* __restrict__ O, int Lq_, int Lk_,
                        float scale, int causal, const int* __restrict__ cu_q,
                        const int* __restrict__ cu_k, int H, int total_q, int total_k,
                        unsigned* err) {
  static_assert(D % 32 == 0, "head dim must be a multiple of 32");
  constexpr int C = D / 32;                   // output columns per lane
  __shared__ float ks[kTileKeys][D + 1];      // +1: lane j reads row j conflict-free
  __shared__ float vs[kTileKeys][D];
  __shared__ float qs[kWarps][D];

  const Rows g = cu_q ? varlen_rows(cu_q, cu_k, H, Lq_, total_q, total_k, D, err)
                      : fixed_rows(Lq_, Lk_, D);
  // elements of Q/O and of K/V (debug-build bounds checks)
  const int64_t n_q = cu_q ? (int64_t)total_q * H * D : (int64_t)gridDim.y * Lq_ * D;
  const int64_t n_k = cu_q ? (int64_t)total_k * H * D : (int64_t)gridDim.y * Lk_ * D;
  if (!g.ok || (int)blockIdx.x * kWarps >= g.Lq) return;   // uniform over the CTA
  const int Lq = g.Lq, Lk = g.Lk;
  const size_t st = g.stride;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * kWarps + warp;
  const bool active = row < Lq;
  const float* Kp = K + g.kv;
  const float* Vp = V + g.kv;

  const float* Qp = Q + g.qo + (size_t)(active ? row : 0) * st;
  for (int i = lane; i < D; i += 32) qs[warp][i] = RF_IN(err, Qp + i - Q, n_q) ? Qp[i] : 0.f;

  // keys this row reads, and keys any row of the CTA reads
  const int off = Lk - Lq;
  const int last_row = min((int)blockIdx.x * kWarps + kWarps - 1, Lq - 1);
  const int lim_row = !active ? 0 : causal ? max(0, min(Lk, row + off + 1)) : Lk;
  const int lim_cta = causal ? max(0, min(Lk, last_row + off + 1)) : Lk;

  float m = -INFINITY, l = 0.f, o[C];
#pragma unroll
  for (int c = 0; c < C; ++c) o[c] = 0.f;

  for (int t0 = 0; t0 < lim_cta; t0 += kTileKeys) {
    __syncthreads();                           // previous tile fully consumed
    for (int i = threadIdx.x; i < kTileKeys * D; i += kWarps * 32) {
      const int r = i / D, cidx = i % D;
      const bool ok = t0 + r < Lk;
      const int64_t kv_i = Kp + (size_t)(t0 + r) * st + cidx - K;
      ks[r][cidx] = ok && RF_IN(err, kv_i, n_k) ? Kp[(size_t)(t0 + r) * st + cidx] : 0.f;
      vs[r][cidx] = ok && RF_IN(err, kv_i, n_k) ? Vp[(size_t)(t0 + r) * st + cidx] : 0.f;
    }
    __syncthreads();

    // scores of this tile: lane j -> key t0 + j
    const bool valid = t0 + lane < lim_row;
    float acc = 0.f;
#pragma unroll 8
    for (int i = 0; i < D; ++i) acc = fmaf(qs[warp][i], ks[lane][i], acc);
    const float s = valid ? acc * scale : -INFINITY;

    // running max, rescale factor, weights and running sum; m_new stays
    // -inf only while the row has read no key (then l = o = 0 and alpha = 0)
    const float m_new = fmaxf(m, warp_max(s));
    const float m_use = m_new == -INFINITY ? 0.f : m_new;
    const float alpha = expf(m - m_use);      // 0 on the first tile (m = -inf)
    const float p = valid ? expf(s - m_use) : 0.f;
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
    float* Op = O + g.qo + (size_t)row * st;
#pragma unroll
    for (int c = 0; c < C; ++c)
      if (RF_IN(err, Op + c * 32 + lane - O, n_q)) Op[c * 32 + lane] = l > 0.f ? o[c] / l : 0.f;
  }
}

}  // namespace

cudaError_t launch_attn_fwd_f32(const float* Q, const float* K, const float* V, float* O, int B,
                                int H, int Lq, int Lk, int d, float scale, int causal,
                                unsigned* err, cudaStream_t s) {
  dim3 grid((Lq + kWarps - 1) / kWarps, B * H);
  if (grid.y > 65535u) return cudaErrorInvalidValue;
  if (d == 64)
    attn_fwd_f32_kernel<64><<<grid, kWarps * 32, 0, s>>>(Q, K, V, O, Lq, Lk, scale, causal,
                                                         nullptr, nullptr, H, 0, 0, err);
  else
    attn_fwd_f32_kernel<128><<<grid, kWarps * 32, 0, s>>>(Q, K, V, O, Lq, Lk, scale, causal,
                                                          nullptr, nullptr, H, 0, 0, err);
  return cudaGetLastError();
}

cudaError_t launch_attn_fwd_f32_varlen(const float* Q, const float* K, const float* V, float* O,
                                       const int* cu_q, const int* cu_k, int B, int H,
                                       int max_q, int total_q, int total_k, int d, float scale,
                                       int causal, unsigned* err, cudaStream_t s) {
  dim3 grid((max_q + kWarps - 1) / kWarps, B * H);
  if (grid.y > 65535u) return cudaErrorInvalidValue;
  if (d == 64)
    attn_fwd_f32_kernel<64><<<grid, kWarps * 32, 0, s>>>(Q, K, V, O, max_q, 0, scale, causal,
                                                         cu_q, cu_k, H, total_q, total_k, err);
  else
    attn_fwd_f32_kernel<128><<<grid, kWarps * 32, 0, s>>>(Q, K, V, O, max_q, 0, scale, causal,
                                                          cu_q, cu_k, H, total_q, total_k, err);
  return cudaGetLastError();
}

}  // namespace rf
