// api.cu -- the C ABI: argument validation, dispatch to the kernels, the
// device-side error word, tensor-map encoding and the wait-timeout self-test.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdio.h>

#include <mutex>

#include "rf_device.cuh"
#include "rf_internal.h"

#define RF_VERSION_NUM 10000

namespace rf {

// One error word per device: kernels OR kDevErr* bits into it when a bounded
// wait runs out; rf_get_device_status reads and clears it.
static __device__ unsigned g_error_word;

namespace {
constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned* g_err_ptr[kMaxDevices] = {};
void* g_err_ctx[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
PFN_cuCtxGetCurrent_v4000 g_ctx_get = nullptr;

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}
}  // namespace

void* current_cu_context() {
  PFN_cuCtxGetCurrent_v4000 get = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_ctx_get) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        return nullptr;
      g_ctx_get = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    }
    get = g_ctx_get;
  }
  CUcontext ctx = nullptr;
  return get(&ctx) == CUDA_SUCCESS ? static_cast<void*>(ctx) : nullptr;
}

// The address is cached together with the context it belongs to: after a
// device reset the runtime creates a new context whose copy of the word
// lives elsewhere, and the lookup is then repeated.
unsigned* device_error_word() {
  const int dev = current_device();
  if (dev < 0) return nullptr;
  void* ctx = current_cu_context();
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_err_ptr[dev] && ctx && ctx == g_err_ctx[dev]) return g_err_ptr[dev];
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess || !p) return nullptr;
  ctx = current_cu_context();        // the lookup above creates the context if needed
  std::lock_guard<std::mutex> lk(g_mu);
  g_err_ptr[dev] = static_cast<unsigned*>(p);
  g_err_ctx[dev] = ctx;
  return g_err_ptr[dev];
}

int sm_count() {
  const int dev = current_device();
  if (dev < 0) return 0;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_sm_count[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

// cuTensorMapEncodeTiled, looked up once through the runtime (no libcuda link).
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return nullptr;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  return g_encode;
}

bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                    uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                    bool swizzle128) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE,
                      swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool encode_tmap_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t d0,
                    uint64_t d1, uint64_t d2, uint64_t stride1_bytes, uint64_t stride2_bytes,
                    uint32_t b0, uint32_t b1, uint32_t b2, bool swizzle128) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return false;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  const cuuint32_t box[3] = {b0, b1, b2};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = encode(map, dtype, 3, const_cast<void*>(base), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE,
                      swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// ------------------------------------------------------------ self-test

// One thread waits on a barrier that expects two arrivals but only ever
// receives one, with a short limit; on timeout it records the error bit and
// returns.  Exercises the bounded-wait path without hanging or faulting.
__global__ void selftest_wait_kernel(uint64_t limit_ns, unsigned* err) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t b = smem_u32(&bar);
  if (threadIdx.x == 0) {
    mbar_init(b, 2);
    fence_mbar_init();
    mbar_arrive(b);                 // one of two arrivals: the phase never completes
    if (!mbar_wait(b, 0, limit_ns)) raise_error(err, kDevErrTimeout);
  }
}

cudaError_t launch_selftest_wait_timeout(int timeout_us, unsigned* err, cudaStream_t s) {
  selftest_wait_kernel<<<1, 32, 0, s>>>((uint64_t)timeout_us * 1000ull, err);
  return cudaGetLastError();
}

#ifdef RF_DEBUG_BOUNDS
// Asks the bounds check about an index one past the end of a 16-element
// tensor: it records kDevErrBounds and the (never made) access is skipped.
__global__ void selftest_bounds_kernel(unsigned* err, int64_t n, unsigned* sink) {
  if (RF_IN(err, n, n)) *sink = 1u;
}
#endif

}  // namespace rf

// ================================================================ C ABI

using namespace rf;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool ptr_ok(const void* p) { return p != nullptr && aligned16(p); }

thread_local char g_last_cuda_error[160] = "none";

rf_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return RF_OK;
  snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s", cudaGetErrorName(e),
           cudaGetErrorString(e));
  return RF_ERR_CUDA;
}

}  // namespace

extern "C" {

const char* rf_status_string(int status) {
  switch (status) {
    case RF_OK: return "RF_OK";
    case RF_ERR_INVALID_ARG: return "RF_ERR_INVALID_ARG: invalid argument";
    case RF_ERR_UNSUPPORTED: return "RF_ERR_UNSUPPORTED: shape or option not supported";
    case RF_ERR_WORKSPACE: return "RF_ERR_WORKSPACE: workspace missing or too small";
    case RF_ERR_CUDA: return "RF_ERR_CUDA: CUDA runtime call or kernel launch failed";
    case RF_ERR_DEVICE_TIMEOUT: return "RF_ERR_DEVICE_TIMEOUT: a kernel's bounded wait ran out";
    case RF_ERR_DEVICE_INPUT:
      return "RF_ERR_DEVICE_INPUT: device-side sizes (cu_seqlens) were inconsistent";
    case RF_ERR_DEVICE_LAYOUT:
      return "RF_ERR_DEVICE_LAYOUT: a kernel's shared memory was not aligned as its tiles need";
    case RF_ERR_DEVICE_BOUNDS:
      return "RF_ERR_DEVICE_BOUNDS: a global access fell outside its tensor (bounds-checked build)";
    default: return "unknown rf_status";
  }
}

int rf_version(void) { return RF_VERSION_NUM; }

const char* rf_last_cuda_error(void) { return g_last_cuda_error; }

rf_status rf_get_device_status(rf_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return RF_ERR_CUDA;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof(v)) != cudaSuccess) return RF_ERR_CUDA;
  if (v != 0) {
    const unsigned zero = 0;
    if (cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero)) != cudaSuccess) return RF_ERR_CUDA;
  }
  if (v & kDevErrTimeout) return RF_ERR_DEVICE_TIMEOUT;
  if (v & kDevErrBounds) return RF_ERR_DEVICE_BOUNDS;
  if (v & kDevErrLayout) return RF_ERR_DEVICE_LAYOUT;
  return (v & kDevErrInput) ? RF_ERR_DEVICE_INPUT : RF_OK;
}

// Longest key sequence for which RF_ATTN_AUTO takes the non-incremental
// (two-pass) bf16 kernel; 0 = always incremental (the incremental kernel
// measured faster: 15.7 against 16.8 us at Lq = Lk = 128 and 14.8 against
// 22.7 us at 256, 65536 query rows of d = 64 each).
static constexpr int kAutoTwoPassMaxLk = 0;

rf_status rf_attn_fwd(int dtype, const void* Q, const void* K, const void* V, void* O, int B,
                      int H, int Lq, int Lk, int d, float scale, int causal, rf_stream_t stream) {
  return rf_attn_fwd_ex(dtype, Q, K, V, O, B, H, Lq, Lk, d, scale, causal, RF_ATTN_AUTO, stream);
}

rf_status rf_attn_fwd_ex(int dtype, const void* Q, const void* K, const void* V, void* O, int B,
                         int H, int Lq, int Lk, int d, float scale, int causal, int mode,
                         rf_stream_t stream) {
  if (dtype != RF_F32 && dtype != RF_BF16) return RF_ERR_INVALID_ARG;
  if (mode != RF_ATTN_AUTO && mode != RF_ATTN_INCREMENTAL && mode != RF_ATTN_TWO_PASS)
    return RF_ERR_INVALID_ARG;
  if (!ptr_ok(Q) || !ptr_ok(K) || !ptr_ok(V) || !ptr_ok(O)) return RF_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || Lq < 1 || Lk < 1 || d < 1 || (causal != 0 && causal != 1))
    return RF_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !(scale < INFINITY)) return RF_ERR_INVALID_ARG;
  if ((int64_t)B * H * Lq >= (1ll << 31) || (int64_t)B * H * Lk >= (1ll << 31))
    return RF_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (dtype == RF_F32) {
    if (d != 64 && d != 128) return RF_ERR_UNSUPPORTED;
    if (mode == RF_ATTN_TWO_PASS) return RF_ERR_UNSUPPORTED;
    if ((int64_t)B * H > 65535) return RF_ERR_INVALID_ARG;     // the grid's y extent
    unsigned* err = device_error_word();
    if (!err) return RF_ERR_CUDA;
    return from_cuda(launch_attn_fwd_f32(static_cast<const float*>(Q),
                                         static_cast<const float*>(K),
                                         static_cast<const float*>(V), static_cast<float*>(O), B,
                                         H, Lq, Lk, d, scale, causal, err, s));
  }
  if (d != 64) return RF_ERR_UNSUPPORTED;
  if (mode == RF_ATTN_TWO_PASS && Lk > 256) return RF_ERR_UNSUPPORTED;
  const int two_pass = mode == RF_ATTN_TWO_PASS || (mode == RF_ATTN_AUTO && Lk <= kAutoTwoPassMaxLk);
  unsigned* err = device_error_word();
  if (!err) return RF_ERR_CUDA;
  return from_cuda(two_pass
                       ? launch_attn_two_pass_tc(Q, K, V, O, B, H, Lq, Lk, scale, causal, err, s)
                       : launch_attn_prefill_tc(Q, K, V, O, B, H, Lq, Lk, scale, causal, err, s));
}

rf_status rf_attn_fwd_varlen(int dtype, const void* Q, const void* K, const void* V, void* O,
                             const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int B,
                             int H, int max_seqlen_q, int total_q, int total_k, int d,
                             float scale, int causal, rf_stream_t stream) {
  if (dtype != RF_F32 && dtype != RF_BF16) return RF_ERR_INVALID_ARG;
  if (!ptr_ok(Q) || !ptr_ok(K) || !ptr_ok(V) || !ptr_ok(O)) return RF_ERR_INVALID_ARG;
  if (!cu_seqlens_q || !cu_seqlens_k || (reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3) ||
      (reinterpret_cast<uintptr_t>(cu_seqlens_k) & 3))
    return RF_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || max_seqlen_q < 1 || total_q < 1 || total_k < 1 || d < 1 ||
      (causal != 0 && causal != 1))
    return RF_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !(scale < INFINITY)) return RF_ERR_INVALID_ARG;
  if ((int64_t)total_q * H >= (1ll << 31) || (int64_t)total_k * H >= (1ll << 31) ||
      (int64_t)B * H > 65535)
    return RF_ERR_INVALID_ARG;
  if (dtype == RF_F32 ? (d != 64 && d != 128) : d != 64) return RF_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  unsigned* err = device_error_word();
  if (!err) return RF_ERR_CUDA;
  if (dtype == RF_F32) {
    return from_cuda(launch_attn_fwd_f32_varlen(
        static_cast<const float*>(Q), static_cast<const float*>(K), static_cast<const float*>(V),
        static_cast<float*>(O), cu_seqlens_q, cu_seqlens_k, B, H, max_seqlen_q, total_q, total_k,
        d, scale, causal, err, s));
  }
  return from_cuda(launch_attn_prefill_tc_varlen(Q, K, V, O, cu_seqlens_q, cu_seqlens_k, B, H,
                                                 max_seqlen_q, total_q, total_k, scale, causal,
                                                 err, s));
}

static rf_status decode_shape_check(int B, int Hq, int Hkv, int Lk, int d, int num_splits) {
  if (B < 1 || Hq < 1 || Hkv < 1 || Lk < 1 || d < 1 || num_splits < 0) return RF_ERR_INVALID_ARG;
  if (Hq % Hkv != 0) return RF_ERR_INVALID_ARG;
  if (num_splits > Lk) return RF_ERR_INVALID_ARG;
  if ((int64_t)B * Hkv * Lk >= (1ll << 31)) return RF_ERR_INVALID_ARG;
  const int G = Hq / Hkv;
  if (d != 128 || (G != 1 && G != 2 && G != 4 && G != 8)) return RF_ERR_UNSUPPORTED;
  return RF_OK;
}

int rf_attn_decode_splitkv_num_splits(int B, int Hq, int Hkv, int Lk, int d, int num_splits) {
  if (decode_shape_check(B, Hq, Hkv, Lk, d, num_splits) != RF_OK) return 0;
  return decode_num_splits(B, Hq, Hkv, Lk, d, num_splits);
}

size_t rf_attn_decode_splitkv_workspace_size(int B, int Hq, int Hkv, int Lk, int d,
                                             int num_splits) {
  if (decode_shape_check(B, Hq, Hkv, Lk, d, num_splits) != RF_OK) return 0;
  return decode_workspace_bytes(B, Hq, Hkv, Lk, d, num_splits);
}

rf_status rf_attn_decode_splitkv(const void* Q, const void* K, const void* V, void* O, int B,
                                 int Hq, int Hkv, int Lk, int d, float scale, int num_splits,
                                 void* workspace, size_t workspace_bytes, rf_stream_t stream) {
  if (!ptr_ok(Q) || !ptr_ok(K) || !ptr_ok(V) || !ptr_ok(O)) return RF_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !(scale < INFINITY)) return RF_ERR_INVALID_ARG;
  rf_status st = decode_shape_check(B, Hq, Hkv, Lk, d, num_splits);
  if (st != RF_OK) return st;
  const size_t need = decode_workspace_bytes(B, Hq, Hkv, Lk, d, num_splits);
  if (need == 0) return RF_ERR_CUDA;   // the automatic partition needs the device's SM count
  if (!workspace || !aligned16(workspace) || workspace_bytes < need) return RF_ERR_WORKSPACE;
  unsigned* err = device_error_word();
  if (!err) return RF_ERR_CUDA;
  return from_cuda(launch_decode_splitkv(Q, K, V, O, B, Hq, Hkv, Lk, d, scale, num_splits,
                                         workspace, err, reinterpret_cast<cudaStream_t>(stream)));
}

static rf_status mla_shape_check(int B, int Hq, int Lk, int d_qk, int d_v, int num_splits) {
  if (B < 1 || Hq < 1 || Lk < 1 || d_qk < 1 || d_v < 1 || num_splits < 0)
    return RF_ERR_INVALID_ARG;
  if ((int64_t)B * Lk >= (1ll << 31) || (int64_t)B * Hq >= (1ll << 31)) return RF_ERR_INVALID_ARG;
  if (d_qk != 576 || d_v != 512 || Hq > 128) return RF_ERR_UNSUPPORTED;
  return RF_OK;
}

int rf_mla_decode_num_splits(int B, int Hq, int Lk, int d_qk, int d_v, int num_splits) {
  if (mla_shape_check(B, Hq, Lk, d_qk, d_v, num_splits) != RF_OK) return 0;
  const int S = mla_num_splits(B, Hq, Lk, num_splits);
  if (S < 1 || (int64_t)B * S * 2 >= (1ll << 31)) return 0;
  return S;
}

size_t rf_mla_decode_workspace_size(int B, int Hq, int Lk, int d_qk, int d_v, int num_splits) {
  const int S = rf_mla_decode_num_splits(B, Hq, Lk, d_qk, d_v, num_splits);
  return S < 1 ? 0 : mla_workspace_bytes(B, Hq, S);
}

rf_status rf_mla_decode(const void* Q, const void* CKV, void* O, int B, int Hq, int Lk, int d_qk,
                        int d_v, float scale, int num_splits, void* workspace,
                        size_t workspace_bytes, rf_stream_t stream) {
  if (!ptr_ok(Q) || !ptr_ok(CKV) || !ptr_ok(O)) return RF_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !(scale < INFINITY)) return RF_ERR_INVALID_ARG;
  rf_status st = mla_shape_check(B, Hq, Lk, d_qk, d_v, num_splits);
  if (st != RF_OK) return st;
  const int S = rf_mla_decode_num_splits(B, Hq, Lk, d_qk, d_v, num_splits);
  if (S < 1) return RF_ERR_CUDA;   // the automatic choice needs the device's SM count
  const size_t need = mla_workspace_bytes(B, Hq, S);
  if (need > 0 && (!workspace || !aligned16(workspace) || workspace_bytes < need))
    return RF_ERR_WORKSPACE;
  unsigned* err = device_error_word();
  if (!err) return RF_ERR_CUDA;
  return from_cuda(launch_mla_decode(Q, CKV, O, B, Hq, Lk, scale, S, workspace, err,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

rf_status rf_moe_gate_topk_softmax_ex(const void* X, const void* Wg, int T, int D, int E, int k,
                                      int w_layout, int32_t* idx, float* w, rf_stream_t stream) {
  if (!ptr_ok(X) || !ptr_ok(Wg) || !ptr_ok(idx) || !ptr_ok(w)) return RF_ERR_INVALID_ARG;
  if (T < 1 || D < 1 || E < 1 || k < 1 || k > E) return RF_ERR_INVALID_ARG;
  if (D % 8 != 0) return RF_ERR_INVALID_ARG;   // 16-byte row pitch for TMA
  if (w_layout != RF_GATE_W_ED && w_layout != RF_GATE_W_DE) return RF_ERR_INVALID_ARG;
  if (E > 256 || k > 8) return RF_ERR_UNSUPPORTED;
  // the tiles lie along the grid's y extent (at most 65535); the host plan
  // makes at most T / 128 + (SMs per cluster wave) of them, within that limit
  // for T <= 65535 * 120
  if (T > 65535 * 120) return RF_ERR_UNSUPPORTED;
  if (w_layout == RF_GATE_W_DE && E % 64 != 0) return RF_ERR_UNSUPPORTED;
  unsigned* err = device_error_word();
  if (!err) return RF_ERR_CUDA;
  return from_cuda(launch_moe_gate(X, Wg, T, D, E, k, w_layout == RF_GATE_W_DE, idx, w, err,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

rf_status rf_moe_gate_topk_softmax(const void* X, const void* Wg, int T, int D, int E, int k,
                                   int32_t* idx, float* w, rf_stream_t stream) {
  return rf_moe_gate_topk_softmax_ex(X, Wg, T, D, E, k, RF_GATE_W_ED, idx, w, stream);
}

size_t rf_absmax_fp8_gemm_workspace_size(int M, int N, int K) {
  if (M < 1 || N < 1 || K < 16 || K % 16 != 0) return 0;
  return fp8_workspace_bytes(M, N, K, true, true);
}

rf_status rf_absmax_fp8_gemm(const void* X, const uint8_t* Wq, const float* sw, void* Y, int M,
                             int N, int K, float* sx_out, uint8_t* xq_out, void* workspace,
                             size_t workspace_bytes, rf_stream_t stream) {
  if (!ptr_ok(X) || !ptr_ok(Wq) || !ptr_ok(sw) || !ptr_ok(Y)) return RF_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 16 || K % 16 != 0) return RF_ERR_INVALID_ARG;
  if ((int64_t)M * K >= (1ll << 40) || (int64_t)N * K >= (1ll << 40)) return RF_ERR_INVALID_ARG;
  if ((sx_out && !aligned16(sx_out)) || (xq_out && !aligned16(xq_out))) return RF_ERR_INVALID_ARG;
  if (!workspace || !aligned16(workspace) ||
      workspace_bytes < fp8_workspace_bytes(M, N, K, !xq_out, !sx_out))
    return RF_ERR_WORKSPACE;
  unsigned* err = device_error_word();
  if (!err) return RF_ERR_CUDA;
  return from_cuda(launch_absmax_fp8_gemm(X, Wq, sw, Y, M, N, K, sx_out, xq_out, workspace, err,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

rf_status rf_absmax_quant_fp8(const void* X, int M, int K, float* sx_out, uint8_t* xq_out,
                              rf_stream_t stream) {
  if (!ptr_ok(X) || !ptr_ok(sx_out) || !ptr_ok(xq_out)) return RF_ERR_INVALID_ARG;
  if (M < 1 || K < 16 || K % 16 != 0) return RF_ERR_INVALID_ARG;
  if ((int64_t)M * K >= (1ll << 40)) return RF_ERR_INVALID_ARG;
  unsigned* err = device_error_word();
  if (!err) return RF_ERR_CUDA;
  return from_cuda(launch_absmax_quant(X, M, K, sx_out, xq_out, err,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

rf_status rf_selftest_wait_timeout(int timeout_us, rf_stream_t stream) {
  if (timeout_us < 1 || timeout_us > 1000000) return RF_ERR_INVALID_ARG;
  unsigned* err = device_error_word();
  if (!err) return RF_ERR_CUDA;
  return from_cuda(launch_selftest_wait_timeout(timeout_us, err,
                                                reinterpret_cast<cudaStream_t>(stream)));
}

int rf_selftest_decode_plan(int B, int Hkv, int Lk, int num_splits, int sms) {
  if (B < 1 || Hkv < 1 || Lk < 1 || (int64_t)B * Hkv * Lk >= (1ll << 31)) return -1;
  return decode_plan_selfcheck(B * Hkv, Lk, num_splits, sms);
}

int rf_selftest_fp8_schedule(int M, int N, int clusters) {
  return fp8_schedule_selfcheck(M, N, clusters);
}

int rf_selftest_moe_plan(int T, int D, int E, int sms) {
  return moe_plan_selfcheck(T, D, E, sms);
}

rf_status rf_selftest_bounds(rf_stream_t stream) {
#ifdef RF_DEBUG_BOUNDS
  unsigned* err = device_error_word();
  if (!err) return RF_ERR_CUDA;
  selftest_bounds_kernel<<<1, 1, 0, reinterpret_cast<cudaStream_t>(stream)>>>(err, 16, err);
  return from_cuda(cudaGetLastError());
#else
  (void)stream;
  return RF_ERR_UNSUPPORTED;
#endif
}

}  // extern "C"
