// decode_splitkv.cu -- multi-segment (split-KV) fused decode attention with
// the merge of the segments' partial states done inside the same kernel.
//
// Multi-segment strategy ([S] Methodologie 3; [E] §3.3 inter-block merge):
// the keys of every (batch, kv head) sequence are cut into segments, each
// reduced by one CTA with the incremental safe-softmax loop ([E] §2.3, §4.1)
// into a partial state (m, l, o) -- o unnormalised, m in log2 units -- for
// each of the G query heads that share the kv head; the states of a sequence
// are then merged: M = max m_j, L = sum l_j 2^(m_j - M),
// O = sum o_j 2^(m_j - M) / L.
//
// Partition.  Automatic (num_splits = 0): the 32-key chunks of all B * Hkv
// sequences, laid end to end, are cut into one contiguous range per CTA of a
// persistent grid of one CTA per SM, so every CTA streams the same number of
// chunks (within one).  A range covers whole sequences and the ends of one or
// two others; a sequence is cut into as many segments as ranges touch it.
// Explicit (num_splits = S): each sequence is cut into S equal key segments,
// and CTA c takes segments c, c + grid, ... in turn.  Either way a CTA works
// through a list of "pieces" (a sequence and a key range of it).
//
// Inside a CTA: four consumer warps take every fourth chunk of the current
// piece, each with a private 2-stage TMA ring that is refilled across piece
// boundaries (the next piece's keys are in flight while the current one
// ends); the G (<= 8) query rows form the M = 16 side (zero-padded) of
// mma.sync m16n8k16 bf16 tiles with fp32 accumulation: S = Q K^T, online
// softmax in registers (quad shuffles), O += P V with P rounded to bf16.  At
// the end of a piece each consumer warp drops its state into a hand-off
// buffer in shared memory (two buffers, taken in turn) and goes on with the
// next piece at once; a fifth warp, the merge warp, combines the four states
// (inter-warp level of the merge) and then
//   - for a piece that is a whole sequence, writes O = o / l in bf16;
//   - otherwise writes the piece's partial state to the workspace, and takes
//     a ticket on the sequence's counter (a fence before the atomic makes the
//     state visible first); the CTA that draws the last ticket reads the
//     other pieces' states back from L2 and merges them (inter-block level),
//     always in the pieces' key order, so the result has the same bits
//     whichever CTA finishes last.
// The ticket counters are zeroed by a small memset on the same stream just
// before the kernel, so the workspace never needs initialising.  (Zeroing
// them inside the kernel needs a grid-wide barrier before the first ticket,
// i.e. a cooperative launch; measured, that barrier cost ~1 us more than the
// memset.)
//
// Data movement: K and V stream from HBM exactly once, by TMA into 128-byte
// swizzled shared-memory tiles (chunks of 32 keys x 128 dims, two 64-dim
// boxes each).  The partial states are a few hundred KB, read back from L2.
#include <math.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "rf_device.cuh"
#include "rf_internal.h"

namespace rf {
namespace {

constexpr int kD = 128;          // head dim
constexpr int kCK = 32;          // keys per chunk
constexpr int kStages = 2;       // ring depth per consumer warp
constexpr int kWarps = 4;        // consumer warps per CTA
constexpr int kThreads = (kWarps + 1) * 32;      // + the merge warp
constexpr int kBoxBytes = kCK * 128;             // one 64-dim box of kCK rows
constexpr int kStageBytes = 4 * kBoxBytes;       // K box0, K box1, V box0, V box1
constexpr int kRingBytes = kWarps * kStages * kStageBytes;
// Hand-off buffer: o of each consumer warp and head, rows padded to 136
// floats (so the eight head rows a warp writes at once fall in different
// banks), then (m, l) of each warp and head.
constexpr int kRowF = 136;
constexpr int kHandOBytes = kWarps * 8 * kRowF * 4;
constexpr int kHandBytes = kHandOBytes + kWarps * 8 * 8;
constexpr int kSmemBytes = kRingBytes + 2 * kHandBytes + 256 + 1024;

// The partition of the keys into pieces, the same on the host and the device.
// Every count here is below 2^31 (B * Hkv * Lk < 2^31), so the automatic
// partition needs 32-bit arithmetic only.
struct DecodePlan {
  uint32_t T;      // automatic: chunks of all sequences (P * nck)
  uint32_t q;      // T / grid: every CTA owns q or q + 1 chunks
  uint32_t rem;    // T % grid: CTAs c < rem own q + 1
  uint32_t nck;    // chunks per sequence, ceil(Lk / kCK)
  int Lk;
  int S;           // explicit segments per sequence, 0 = automatic
  int P;           // sequences, B * Hkv
  int grid;        // CTAs
};

struct DecodePiece {
  int p;           // sequence (b * Hkv + kv head)
  int lo, hi;      // keys [lo, hi) of the sequence
  int slot;        // workspace slot of its partial state (when npieces > 1)
  int npieces;     // pieces the sequence is cut into
};

// grid = min(SMs, units) so that no CTA is left without work.
__host__ __device__ inline void plan_init(DecodePlan* pl, int P, int Lk, int S, int sms) {
  pl->P = P;
  pl->Lk = Lk;
  pl->S = S;
  pl->nck = (uint32_t)(((int64_t)Lk + kCK - 1) / kCK);   // Lk up to 2^31 - 1
  pl->T = (uint32_t)P * pl->nck;
  const int64_t units = S > 0 ? (int64_t)P * S : (int64_t)pl->T;
  pl->grid = (int)(units < sms ? units : sms);
  pl->q = pl->T / (uint32_t)pl->grid;
  pl->rem = pl->T % (uint32_t)pl->grid;
}

// Automatic partition: CTA c owns chunks [start(c), start(c + 1)).
__host__ __device__ __forceinline__ uint32_t plan_start(const DecodePlan& pl, int c) {
  const uint32_t uc = (uint32_t)c;
  return uc * pl.q + (uc < pl.rem ? uc : pl.rem);
}
// The CTA whose range holds chunk x.
__host__ __device__ __forceinline__ int plan_owner(const DecodePlan& pl, uint32_t x) {
  const uint32_t big = pl.rem * (pl.q + 1);          // chunks of the CTAs with q + 1
  return (int)(x < big ? x / (pl.q + 1) : pl.rem + (x - big) / pl.q);
}

__host__ __device__ __forceinline__ int plan_num_pieces(const DecodePlan& pl, int c) {
  if (pl.S > 0) {
    const uint32_t items = (uint32_t)pl.P * (uint32_t)pl.S;
    return items > (uint32_t)c ? (int)((items - c + pl.grid - 1) / pl.grid) : 0;
  }
  const uint32_t r0 = plan_start(pl, c), r1 = plan_start(pl, c + 1);
  return r1 > r0 ? (int)((r1 - 1) / pl.nck - r0 / pl.nck + 1) : 0;
}

// Piece k (0 ..) of CTA c.  In the automatic partition the slot of a piece
// is 2c for the CTA's first piece and 2c + 1 for its last; only those two
// can be parts of a longer sequence.
__host__ __device__ __forceinline__ DecodePiece plan_piece(const DecodePlan& pl, int c, int k) {
  DecodePiece pc;
  if (pl.S > 0) {
    const uint32_t item = (uint32_t)c + (uint32_t)k * (uint32_t)pl.grid;
    const int seg = (int)(item % (uint32_t)pl.S);
    pc.p = (int)(item / (uint32_t)pl.S);
    pc.lo = (int)((int64_t)seg * pl.Lk / pl.S);
    pc.hi = (int)((int64_t)(seg + 1) * pl.Lk / pl.S);
    pc.slot = (int)item;
    pc.npieces = pl.S;
    return pc;
  }
  const uint32_t r0 = plan_start(pl, c), r1 = plan_start(pl, c + 1);
  const uint32_t p = r0 / pl.nck + (uint32_t)k;
  const uint32_t s0 = p * pl.nck, s1 = s0 + pl.nck;
  const uint32_t a = (r0 > s0 ? r0 : s0) - s0, b = (r1 < s1 ? r1 : s1) - s0;
  const uint32_t hi = b * kCK;                      // up to 2^31: unsigned
  pc.p = (int)p;
  pc.lo = (int)(a * kCK);
  pc.hi = hi < (uint32_t)pl.Lk ? (int)hi : pl.Lk;
  pc.slot = 2 * c + (k == 0 ? 0 : 1);
  // a piece strictly inside the range is a whole sequence
  pc.npieces = (s0 >= r0 && s1 <= r1) ? 1 : plan_owner(pl, s1 - 1) - plan_owner(pl, s0) + 1;
  return pc;
}

// Workspace slot of the j-th piece (in key order) of sequence p.
__host__ __device__ __forceinline__ int plan_slot(const DecodePlan& pl, int p, int j) {
  if (pl.S > 0) return p * pl.S + j;
  const int c = plan_owner(pl, (uint32_t)p * pl.nck) + j;
  return 2 * c + (plan_start(pl, c) / pl.nck == (uint32_t)p ? 0 : 1);
}

__host__ __device__ __forceinline__ int64_t plan_slots(const DecodePlan& pl) {
  return pl.S > 0 ? (int64_t)pl.P * pl.S : 2 * (int64_t)pl.grid;
}

// The order in which a CTA works through its np pieces: in the automatic
// partition its two partial pieces (first and last) come before the whole
// sequences between them, so the neighbours' matching pieces are done early
// and the merges across CTAs happen while the keys still stream, not at the
// end of the kernel.
__host__ __device__ __forceinline__ int plan_order(const DecodePlan& pl, int np, int k) {
  if (pl.S > 0 || np < 3) return k;
  return k == 0 ? 0 : (k == 1 ? np - 1 : k - 1);
}

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

__device__ __forceinline__ int piece_chunks(const DecodePiece& pc) {
  return (int)(((int64_t)pc.hi - pc.lo + kCK - 1) / kCK);
}

// Adds state (m, l, o) into the running merge (M, L, O) whose reference is
// the final maximum Mx (so every weight is 2^(m - Mx) <= 1).
__device__ __forceinline__ void merge_into(float Mx, float m, float l, float4 o, float& L,
                                           float4& O) {
  const float w = exp2f(m - Mx);     // 0 for an empty state (m = -inf)
  L = fmaf(l, w, L);
  O.x = fmaf(o.x, w, O.x);
  O.y = fmaf(o.y, w, O.y);
  O.z = fmaf(o.z, w, O.z);
  O.w = fmaf(o.w, w, O.w);
}

__device__ __forceinline__ void store_out(__nv_bfloat16* O, int64_t row, int lane, float L,
                                          float4 o, int64_t n_o, unsigned* err) {
  if (!RF_IN(err, row * kD + 4 * lane + 3, n_o)) return;
  const float inv = 1.f / L;
  uint2 out;
  out.x = pack_bf16x2(o.x * inv, o.y * inv);
  out.y = pack_bf16x2(o.z * inv, o.w * inv);
  reinterpret_cast<uint2*>(O + row * kD)[lane] = out;
}

// Bounded wait that sleeps between polls: for the merge warp, which idles
// for most of a piece and would otherwise take issue slots from the consumer
// warp it shares a scheduler with.
__device__ __forceinline__ bool mbar_wait_sleep(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_test_wait(bar, parity)) {
    __nanosleep(256);
    if (globaltimer_ns() - t0 > kDefaultWaitNs) return false;
  }
  return true;
}

struct Bars {
  uint64_t full[kWarps][kStages];   // TMA ring of each consumer warp
  uint64_t hand_full[2];            // the four consumer states of a piece are in buffer i
  uint64_t hand_free[2];            // the merge warp has read buffer i
};
static_assert(sizeof(Bars) <= 256, "barrier block");

template <int G>
__global__ void __launch_bounds__(kThreads, 1)
    decode_splitkv_kernel(const __grid_constant__ CUtensorMap tmK,
                          const __grid_constant__ CUtensorMap tmV,
                          const __nv_bfloat16* __restrict__ Q, __nv_bfloat16* __restrict__ O,
                          float* __restrict__ ws_o, float2* __restrict__ ws_ml,
                          unsigned* __restrict__ tickets, const DecodePlan pl,
                          float qk_scale_log2, unsigned* err) {
  static_assert(G >= 1 && G <= 8, "query heads per kv head");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* hand = smem + kRingBytes;
  Bars* bars = reinterpret_cast<Bars*>(hand + 2 * kHandBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = (int)blockIdx.x;
  const int np = plan_num_pieces(pl, cta);
  // elements of Q and O, of the partial-state slots (debug-build bounds checks)
  const int64_t n_qo = (int64_t)pl.P * G * kD;
  const int64_t n_ml = plan_slots(pl) * G;
  const bool consumer = warp < kWarps;

  if (threadIdx.x == 0) {
    for (int w = 0; w < kWarps; ++w)
      for (int i = 0; i < kStages; ++i) mbar_init(smem_u32(&bars->full[w][i]), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&bars->hand_full[i]), kWarps);
      mbar_init(smem_u32(&bars->hand_free[i]), 1);
    }
    fence_mbar_init();
  }
  __syncthreads();

  // producer cursor over this warp's chunk stream (lane 0 of a consumer warp)
  uint8_t* my_stage = smem + (consumer ? warp : 0) * kStages * kStageBytes;
  uint64_t* my_full = bars->full[consumer ? warp : 0];
  int pk = 0, pci = warp, issued = 0;
  DecodePiece pp = plan_piece(pl, cta, plan_order(pl, np, 0));
  auto skip_empty = [&]() {
    while (pk < np && pci >= piece_chunks(pp)) {
      ++pk;
      pci = warp;
      if (pk < np) pp = plan_piece(pl, cta, plan_order(pl, np, pk));
    }
  };
  auto issue_next = [&]() {
    skip_empty();
    if (pk >= np) return;
    const int slot = issued % kStages;
    const int32_t row = (int32_t)((int64_t)pp.p * pl.Lk + pp.lo + (int64_t)pci * kCK);
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
  if (consumer && lane == 0) {
    prefetch_tmap(&tmK);
    prefetch_tmap(&tmV);
    for (int i = 0; i < kStages; ++i) issue_next();
  }

  if (!consumer) {
    // ------------------------------------------------------------ merge warp
    for (int k = 0; k < np; ++k) {
      const DecodePiece pc = plan_piece(pl, cta, plan_order(pl, np, k));
      const int buf = k & 1;
      bool ok = mbar_wait_sleep(smem_u32(&bars->hand_full[buf]), (uint32_t)((k >> 1) & 1));
      if (!__all_sync(0xffffffffu, ok)) {
        raise_error(err, kDevErrTimeout);
        return;
      }
      const float* ho = reinterpret_cast<const float*>(hand + buf * kHandBytes);
      const float2* hml = reinterpret_cast<const float2*>(hand + buf * kHandBytes + kHandOBytes);
      float Mh[G], Lh[G];
      float4 Oh[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float m[kWarps], l[kWarps];
        float Mx = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
          const float2 v = hml[w * 8 + h];
          m[w] = v.x;
          l[w] = v.y;
          Mx = fmaxf(Mx, v.x);
        }
        float L = 0.f;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        if (Mx != -INFINITY) {       // else no key of the piece reached this CTA's warps
#pragma unroll
          for (int w = 0; w < kWarps; ++w)
            merge_into(Mx, m[w], l[w],
                       *reinterpret_cast<const float4*>(ho + (w * 8 + h) * kRowF + 4 * lane), L,
                       o);
        }
        Mh[h] = Mx;
        Lh[h] = L;
        Oh[h] = o;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&bars->hand_free[buf]));   // release: reads done

      if (pc.npieces == 1) {
#pragma unroll
        for (int h = 0; h < G; ++h) store_out(O, (int64_t)pc.p * G + h, lane, Lh[h], Oh[h], n_qo, err);
        continue;
      }
      // partial state of the piece -> workspace; ticket on the sequence
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const int64_t sh = (int64_t)pc.slot * G + h;
        if (RF_IN(err, sh, n_ml)) {
          reinterpret_cast<float4*>(ws_o + sh * kD)[lane] = Oh[h];
          if (lane == 0) ws_ml[sh] = make_float2(Mh[h], Lh[h]);
        }
      }
      __threadfence();
      __syncwarp();
      unsigned t = 0;
      if (lane == 0 && RF_IN(err, pc.p, pl.P)) t = atomicAdd(&tickets[pc.p], 1u);
      t = __shfl_sync(0xffffffffu, t, 0);
      if (t != (unsigned)(pc.npieces - 1)) continue;
      __threadfence();               // the other pieces' states are visible now
      // Last piece to finish: merge all pieces of the sequence, one after
      // another in key order (this CTA's own piece from registers: the same
      // values it stored), so the bits do not depend on which CTA is last.
      // The loads of a batch of kBatch pieces are issued together.
      constexpr int kBatch = G <= 2 ? 4 : (G == 4 ? 2 : 1);
      float Mt[G], Lt[G];
      float4 Ot[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        Mt[h] = -INFINITY;
        Lt[h] = 0.f;
        Ot[h] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      for (int j0 = 0; j0 < pc.npieces; j0 += kBatch) {
        float2 ml[kBatch][G];
        float4 oj[kBatch][G];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
          const int j = j0 + u;
          const int sj = j < pc.npieces ? plan_slot(pl, pc.p, j) : -1;
#pragma unroll
          for (int h = 0; h < G; ++h) {
            if (sj == pc.slot) {
              ml[u][h] = make_float2(Mh[h], Lh[h]);
              oj[u][h] = Oh[h];
            } else if (sj >= 0 && RF_IN(err, (int64_t)sj * G + h, n_ml)) {
              ml[u][h] = __ldcg(&ws_ml[(int64_t)sj * G + h]);
              oj[u][h] =
                  __ldcg(reinterpret_cast<const float4*>(ws_o + ((int64_t)sj * G + h) * kD) + lane);
            } else {
              ml[u][h] = make_float2(-INFINITY, 0.f);
              oj[u][h] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
          }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u)
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float m = ml[u][h].x;
            if (m == -INFINITY) continue;          // a piece without keys adds nothing
            const float Mn = fmaxf(Mt[h], m);
            const float a = exp2f(Mt[h] - Mn);     // 0 while nothing has been added
            const float w = exp2f(m - Mn);
            Lt[h] = fmaf(ml[u][h].y, w, Lt[h] * a);
            Ot[h].x = fmaf(oj[u][h].x, w, Ot[h].x * a);
            Ot[h].y = fmaf(oj[u][h].y, w, Ot[h].y * a);
            Ot[h].z = fmaf(oj[u][h].z, w, Ot[h].z * a);
            Ot[h].w = fmaf(oj[u][h].w, w, Ot[h].w * a);
            Mt[h] = Mn;
          }
      }
#pragma unroll
      for (int h = 0; h < G; ++h) store_out(O, (int64_t)pc.p * G + h, lane, Lt[h], Ot[h], n_qo, err);
    }
    return;
  }

  // ------------------------------------------------------------ consumer warps
  const int hrow = lane >> 2;           // head of this lane's accumulator rows
  const int kq = (lane & 3) * 2;        // first of this lane's two columns
  const int mi = lane >> 3, mr = lane & 7;   // ldmatrix: matrix, row within it
  int consumed = 0;
  bool failed = false;

  // Q of the G query heads as the A operand (rows zero-padded to 16); the
  // next piece's Q is loaded while the current piece runs.
  auto load_q = [&](int k, uint32_t (&q)[8][2]) {
    if (k >= np) return;
    const DecodePiece pc = plan_piece(pl, cta, plan_order(pl, np, k));
    const int64_t q_row = ((int64_t)pc.p * G + (hrow < G ? hrow : 0)) * kD;
    const uint32_t* qp = reinterpret_cast<const uint32_t*>(Q + q_row);
    const bool q_ok = hrow < G && RF_IN(err, q_row + kD - 1, n_qo);
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      q[ks][0] = q_ok ? __ldg(qp + ((ks * 16 + kq) >> 1)) : 0u;
      q[ks][1] = q_ok ? __ldg(qp + ((ks * 16 + kq + 8) >> 1)) : 0u;
    }
  };
  uint32_t qa[8][2], qn[8][2];
  load_q(0, qn);

  for (int k = 0; k < np && !failed; ++k) {
    const DecodePiece pc = plan_piece(pl, cta, plan_order(pl, np, k));
    const int nchunks = piece_chunks(pc);
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

    for (int ci = warp; ci < nchunks; ci += kWarps) {
      const int slot = consumed % kStages;
      bool ok = mbar_wait(smem_u32(&my_full[slot]), (uint32_t)((consumed / kStages) & 1));
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) {
        failed = true;
        break;
      }
      const uint32_t kbase = smem_u32(my_stage + slot * kStageBytes);
      const uint32_t vbase = kbase + 2 * kBoxBytes;
      const int key0 = pc.lo + ci * kCK;   // first key of the chunk

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
            const int key = key0 + sb * 16 + nb * 8 + kq + e;
            const float v = key < pc.hi ? sc[sb][nb][e] * qk_scale_log2 : -INFINITY;
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

    // ---- this warp's state of the piece -> hand-off buffer k % 2 (a warp
    // without keys in the piece hands over (-inf, 0, 0))
    const int buf = k & 1;
    if (k >= 2) {
      bool ok = mbar_wait(smem_u32(&bars->hand_free[buf]), (uint32_t)(((k >> 1) - 1) & 1));
      if (!__all_sync(0xffffffffu, ok)) {
        failed = true;
        break;
      }
    }
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    if (hrow < G) {
      float* ho = reinterpret_cast<float*>(hand + buf * kHandBytes) + (warp * 8 + hrow) * kRowF;
#pragma unroll
      for (int j = 0; j < 16; ++j)
        *reinterpret_cast<float2*>(ho + j * 8 + kq) = make_float2(oacc[j][0], oacc[j][1]);
      if ((lane & 3) == 0)
        reinterpret_cast<float2*>(hand + buf * kHandBytes + kHandOBytes)[warp * 8 + hrow] =
            make_float2(m_run, l_run);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&bars->hand_full[buf]));
  }

  if (failed) {
    raise_error(err, kDevErrTimeout);
    // let this warp's copies still in flight land before shared memory is released
    if (lane == 0)
      for (int c = consumed; c < issued; ++c)
        (void)mbar_wait(smem_u32(&my_full[c % kStages]), (uint32_t)((c / kStages) & 1), 1000000ull);
  }
}

template <int G>
cudaError_t launch_g(const CUtensorMap& tmK, const CUtensorMap& tmV, const void* Q, void* O,
                     const DecodePlan& pl, float scale, float* ws_o, float2* ws_ml,
                     unsigned* tickets, unsigned* err, cudaStream_t s) {
  auto kern = decode_splitkv_kernel<G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e != cudaSuccess) return e;
  const float qk_scale_log2 = scale * 1.4426950408889634f;
  // the ticket counters start at zero (one small memset; a sequence of one
  // piece takes no ticket, so with S = 1 none is needed)
  if (pl.S != 1) {
    e = cudaMemsetAsync(tickets, 0, (size_t)pl.P * sizeof(unsigned), s);
    if (e != cudaSuccess) return e;
  }
  kern<<<pl.grid, kThreads, kSmemBytes, s>>>(tmK, tmV, static_cast<const __nv_bfloat16*>(Q),
                                             static_cast<__nv_bfloat16*>(O), ws_o, ws_ml,
                                             tickets, pl, qk_scale_log2, err);
  return cudaGetLastError();
}

// The partition for a shape; false if the device's SM count cannot be read.
bool make_plan(int B, int Hkv, int Lk, int requested, DecodePlan* pl) {
  const int sms = sm_count();
  if (sms <= 0) return false;
  plan_init(pl, B * Hkv, Lk, requested, sms);
  return true;
}

// Workspace layout: ticket counters [P] (padded to 256 bytes), partial o
// [slots][G][128] fp32 (padded to 256 bytes), partial (m, l) [slots][G].
size_t ws_tickets_bytes(const DecodePlan& pl) {
  return ((size_t)pl.P * sizeof(unsigned) + 255) & ~(size_t)255;
}
size_t ws_o_bytes(const DecodePlan& pl, int G) {
  return ((size_t)plan_slots(pl) * G * kD * sizeof(float) + 255) & ~(size_t)255;
}

}  // namespace

// Host-side check of the partition the kernel follows (the plan_* functions
// above, shared by host and device), for P = B * Hkv sequences of Lk keys,
// S explicit segments (0 = automatic) and a grid of at most `sms` CTAs.
// Returns 0 when every invariant holds, -1 for a shape the decode call
// refuses, else the number of the first invariant that fails:
//   1 every CTA has at least one piece;
//   2 plan_order visits each of a CTA's pieces once;
//   3 every piece is a non-empty key range [lo, hi) of a sequence;
//   4 pieces of split sequences have distinct workspace slots in range;
//   5 the pieces of each sequence tile [0, Lk) with no gap or overlap;
//   6 every piece knows how many pieces its sequence has;
//   7 plan_slot lists a split sequence's slots in key order, which is the
//     order the merge reads them in.
int decode_plan_selfcheck(int P, int Lk, int S, int sms) {
  if (P < 1 || Lk < 1 || S < 0 || S > Lk || sms < 1 || (int64_t)P * Lk >= (1ll << 31)) return -1;
  DecodePlan pl;
  plan_init(&pl, P, Lk, S, sms);
  struct Rec {
    int p, lo, hi, slot, np;
  };
  std::vector<Rec> all;
  std::vector<unsigned char> used((size_t)plan_slots(pl), 0);
  for (int c = 0; c < pl.grid; ++c) {
    const int np = plan_num_pieces(pl, c);
    if (np < 1) return 1;
    std::vector<unsigned char> seen((size_t)np, 0);
    for (int k = 0; k < np; ++k) {
      const int o = plan_order(pl, np, k);
      if (o < 0 || o >= np || seen[(size_t)o]++) return 2;
    }
    for (int k = 0; k < np; ++k) {
      const DecodePiece pc = plan_piece(pl, c, k);
      if (pc.p < 0 || pc.p >= P || pc.lo < 0 || pc.lo >= pc.hi || pc.hi > Lk) return 3;
      if (pc.npieces > 1 && (pc.slot < 0 || pc.slot >= plan_slots(pl) || used[(size_t)pc.slot]++))
        return 4;
      all.push_back({pc.p, pc.lo, pc.hi, pc.slot, pc.npieces});
    }
  }
  std::sort(all.begin(), all.end(),
            [](const Rec& a, const Rec& b) { return a.p != b.p ? a.p < b.p : a.lo < b.lo; });
  size_t i = 0;
  for (int p = 0; p < P; ++p) {
    size_t j = i;
    int end = 0;
    for (; j < all.size() && all[j].p == p; ++j) {
      if (all[j].lo != end) return 5;
      end = all[j].hi;
    }
    if (end != Lk) return 5;
    const int n = (int)(j - i);
    for (size_t t = i; t < j; ++t) {
      if (all[t].np != n) return 6;
      if (n > 1 && plan_slot(pl, p, (int)(t - i)) != all[t].slot) return 7;
    }
    i = j;
  }
  return i == all.size() ? 0 : 5;
}

int decode_num_splits(int B, int Hq, int Hkv, int Lk, int d, int requested) {
  (void)Hq;
  (void)d;
  if (requested > 0) return requested;
  DecodePlan pl;
  if (!make_plan(B, Hkv, Lk, 0, &pl)) return 0;
  // The automatic partition cuts a sequence of nck chunks into at most
  // ceil((nck - 1) / q) + 1 segments, q = the fewest chunks of any range.
  const int64_t most = ((int64_t)pl.nck - 1 + pl.q - 1) / pl.q + 1;
  return (int)(most < pl.grid ? most : pl.grid);
}

size_t decode_workspace_bytes(int B, int Hq, int Hkv, int Lk, int d, int requested) {
  (void)d;
  DecodePlan pl;
  if (!make_plan(B, Hkv, Lk, requested, &pl)) {
    if (requested <= 0) return 0;
    plan_init(&pl, B * Hkv, Lk, requested, 1);    // explicit S: independent of the device
  }
  const int G = Hq / Hkv;
  return ws_tickets_bytes(pl) + ws_o_bytes(pl, G) + (size_t)plan_slots(pl) * G * sizeof(float2);
}

cudaError_t launch_decode_splitkv(const void* Q, const void* K, const void* V, void* O, int B,
                                  int Hq, int Hkv, int Lk, int d, float scale, int requested,
                                  void* workspace, unsigned* err, cudaStream_t s) {
  (void)d;
  DecodePlan pl;
  if (!make_plan(B, Hkv, Lk, requested, &pl)) return cudaErrorInvalidValue;
  const uint64_t rows = (uint64_t)B * Hkv * Lk;
  CUtensorMap tmK, tmV;
  if (!encode_tmap_2d(&tmK, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, K, kD, rows, kD * 2, 64, kCK, true) ||
      !encode_tmap_2d(&tmV, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, V, kD, rows, kD * 2, 64, kCK, true))
    return cudaErrorInvalidValue;
  const int G = Hq / Hkv;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  unsigned* tickets = reinterpret_cast<unsigned*>(ws);
  float* ws_o = reinterpret_cast<float*>(ws + ws_tickets_bytes(pl));
  float2* ws_ml = reinterpret_cast<float2*>(ws + ws_tickets_bytes(pl) + ws_o_bytes(pl, G));
  switch (G) {
    case 1: return launch_g<1>(tmK, tmV, Q, O, pl, scale, ws_o, ws_ml, tickets, err, s);
    case 2: return launch_g<2>(tmK, tmV, Q, O, pl, scale, ws_o, ws_ml, tickets, err, s);
    case 4: return launch_g<4>(tmK, tmV, Q, O, pl, scale, ws_o, ws_ml, tickets, err, s);
    case 8: return launch_g<8>(tmK, tmV, Q, O, pl, scale, ws_o, ws_ml, tickets, err, s);
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
  // Nothing in the scratch has to start at zero: the launcher zeroes the
  // ticket counters, and every partial state is written before it is read.
  void* scratch = rf::decode_scratch_address();
  if (!scratch) return RF_ERR_CUDA;
  return rf_attn_decode_splitkv(Q, K, V, O, B, Hq, Hkv, Lk, d, scale, num_splits, scratch,
                                rf::kNoAllocScratchBytes, stream);
}

