// rf_internal.h -- host-side declarations shared by the library's translation
// units (launchers called from api.cu after argument validation).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/rf.h"

namespace rf {

// The current CUDA context (driver handle), or nullptr if there is none yet.
void* current_cu_context();

// Device address of the per-device error word (looked up once per device and
// context).  Returns nullptr if the address could not be obtained.
unsigned* device_error_word();

// SM count of the current device (cached per device).
int sm_count();

// Encodes a 2-D tiled tensor map: inner dimension `inner` elements (contiguous),
// `outer` rows with a row pitch of `row_bytes`; box = box_inner x box_outer;
// 128-byte swizzle when swizzle128 is set.  Returns false on failure.
bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base,
                    uint64_t inner, uint64_t outer, uint64_t row_bytes, uint32_t box_inner,
                    uint32_t box_outer, bool swizzle128);

// 3-D tiled tensor map: extents d0 (contiguous), d1, d2 with byte strides of
// dims 1 and 2; box b0 x b1 x b2.  Returns false on failure.
bool encode_tmap_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t d0,
                    uint64_t d1, uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes,
                    uint32_t b0, uint32_t b1, uint32_t b2, bool swizzle128);

// ---------------------------------------------------------------- launchers
// Each returns cudaSuccess or the launch error.  Arguments are pre-validated.

// causal = 1: query row i reads keys j <= i + (Lk - Lq) only.
cudaError_t launch_attn_fwd_f32(const float* Q, const float* K, const float* V, float* O, int B,
                                int H, int Lq, int Lk, int d, float scale, int causal,
                                unsigned* err, cudaStream_t s);

// bf16, d = 64, the non-incremental (two-pass) form: Lk <= 256, one CTA per
// 128 query rows.
cudaError_t launch_attn_two_pass_tc(const void* Q, const void* K, const void* V, void* O, int B,
                                    int H, int Lq, int Lk, float scale, int causal, unsigned* err,
                                    cudaStream_t s);

// bf16, d = 64, the incremental single-pass form (the BERT-style prefill
// path): two query tiles per CTA, one MMA-issuing thread each, P and O in
// tensor memory; fixed-length [B][H][L][64] or packed variable-length
// [total][H][64] (sequence b = tokens cu_q[b] .. cu_q[b+1]-1, device arrays
// of B + 1 int32), with or without the causal mask.
cudaError_t launch_attn_prefill_tc(const void* Q, const void* K, const void* V, void* O, int B,
                                   int H, int Lq, int Lk, float scale, int causal, unsigned* err,
                                   cudaStream_t s);
cudaError_t launch_attn_prefill_tc_varlen(const void* Q, const void* K, const void* V, void* O,
                                          const int* cu_q, const int* cu_k, int B, int H,
                                          int max_q, int total_q, int total_k, float scale,
                                          int causal, unsigned* err, cudaStream_t s);

// Packed variable-length layout: Q/O [total_q][H][d], K/V [total_k][H][d],
// sequence b = tokens cu_q[b] .. cu_q[b+1]-1 (device arrays of B + 1 int32).
cudaError_t launch_attn_fwd_f32_varlen(const float* Q, const float* K, const float* V, float* O,
                                       const int* cu_q, const int* cu_k, int B, int H,
                                       int max_q, int total_q, int total_k, int d, float scale,
                                       int causal, unsigned* err, cudaStream_t s);

int decode_num_splits(int B, int Hq, int Hkv, int Lk, int d, int requested);
// host only: 0 when the split-KV partition of P sequences is consistent
int decode_plan_selfcheck(int P, int Lk, int S, int sms);
// host only: 0 when the FP8 GEMM's tile schedule covers an M x N output once
int fp8_schedule_selfcheck(int M, int N, int clusters);
// host only: 0 when the MoE gate's tile plan is consistent
int moe_plan_selfcheck(int T, int D, int E, int sms);
size_t decode_workspace_bytes(int B, int Hq, int Hkv, int Lk, int d, int requested);
cudaError_t launch_decode_splitkv(const void* Q, const void* K, const void* V, void* O, int B,
                                  int Hq, int Hkv, int Lk, int d, float scale, int requested,
                                  void* workspace, unsigned* err, cudaStream_t s);

// Latent-KV decode: Q [B][Hq][576], CKV [B][Lk][576], O [B][Hq][512] (bf16).
int mla_num_splits(int B, int Hq, int Lk, int requested);
size_t mla_workspace_bytes(int B, int Hq, int S);
cudaError_t launch_mla_decode(const void* Q, const void* CKV, void* O, int B, int Hq, int Lk,
                              float scale, int S, void* workspace, unsigned* err, cudaStream_t s);

// w_de: W_gate is [D][E] (E in {64, 128, 192, 256}); else [E][D].
cudaError_t launch_moe_gate(const void* X, const void* Wg, int T, int D, int E, int k,
                            bool w_de, int32_t* idx, float* w, unsigned* err, cudaStream_t s);

// FP8: the workspace holds the kernel's row counters, then (when the caller
// keeps no copy) the codes and the row scales.
size_t fp8_counter_bytes(int M);
size_t fp8_workspace_bytes(int M, int N, int K, bool need_xq, bool need_sx);
cudaError_t launch_absmax_quant(const void* X, int M, int K, float* sx, uint8_t* xq,
                                unsigned* err, cudaStream_t s);
cudaError_t launch_absmax_fp8_gemm(const void* X, const uint8_t* Wq, const float* sw, void* Y,
                                   int M, int N, int K, float* sx, uint8_t* xq, void* workspace,
                                   unsigned* err, cudaStream_t s);

cudaError_t launch_selftest_wait_timeout(int timeout_us, unsigned* err, cudaStream_t s);

}  // namespace rf
