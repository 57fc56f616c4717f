/*
 * rf.h -- C ABI of the fused cascaded-reduction kernels for GB300 (sm_103a).
 *
 * A cascaded reduction is a chain of reductions in which each step needs the
 * result of the previous one (safe softmax: max, then sum of exp(x - max),
 * then the weighted sum with V).  The kernels behind this header run each
 * chain as one pass over its input, keeping a small running state on chip
 * and rescaling it as each tile arrives ("incremental computation form").
 *
 * Sources of the operations (cited by title and section):
 *  [A] "RedFuser: An Automatic Operator Fusion Framework for Cascaded
 *      Reductions on AI Accelerators", ASPLOS 2026, abstract.
 *  [E] "RedFuser框架：AI加速器中的算子融合技术解析" (explainer article),
 *      §2.2 softmax cascade, §2.3 incremental form, §3.3 execution hierarchy,
 *      §4.1 fused attention, §4.2 MoE routing, §4.3 FP8 quantised GEMM.
 *  [S] gist.science technical summary of [A], "Methodologie" 1-3
 *      (fusion conditions, incremental form, single-/multi-segment code).
 *
 * Conventions for every entry point:
 *  - Tensor arguments are DEVICE pointers on the current CUDA device, owned
 *    by the caller; the library never allocates, frees or synchronises
 *    (except rf_get_device_status, which synchronises the given stream).
 *  - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default).
 *  - Layouts are dense row-major (C order) with the shapes given.
 *  - Pointers must be 16-byte aligned.
 *  - Arguments are validated on the host before anything is launched; a bad
 *    argument returns an error code and enqueues nothing.  Launch failures
 *    return RF_ERR_CUDA.  Asynchronous device-side problems (a bounded wait
 *    that ran out) are reported by rf_get_device_status.
 *  - The functions are reentrant; calls on one stream execute in order, and
 *    concurrent calls on different streams must not share output buffers
 *    or workspaces.
 */
#ifndef RF_H_
#define RF_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st* rf_stream_t;

typedef enum {
  RF_OK = 0,
  RF_ERR_INVALID_ARG = 1,     /* null / misaligned pointer, bad size       */
  RF_ERR_UNSUPPORTED = 2,     /* valid request this build does not cover    */
  RF_ERR_WORKSPACE = 3,       /* workspace missing or too small             */
  RF_ERR_CUDA = 4,            /* a CUDA runtime call or launch failed       */
  RF_ERR_DEVICE_TIMEOUT = 5,  /* a kernel's bounded wait ran out            */
  RF_ERR_DEVICE_INPUT = 6,    /* device-resident sizes were inconsistent    */
  RF_ERR_DEVICE_LAYOUT = 7,   /* a kernel's shared memory was misaligned    */
  RF_ERR_DEVICE_BOUNDS = 8    /* debug build: an access outside its tensor  */
} rf_status;

typedef enum { RF_F32 = 0, RF_BF16 = 1 } rf_dtype;

/* Human-readable name of a status code (static string, never NULL). */
const char* rf_status_string(int status);

/* Library version as major*10000 + minor*100 + patch. */
int rf_version(void);

/*
 * Name and description of the last CUDA error that made an entry point
 * return RF_ERR_CUDA in the calling host thread ("none" if there was none).
 * The string is owned by the library and stays valid until the thread's next
 * call.  (An interface aid; the paper has no counterpart.)
 */
const char* rf_last_cuda_error(void);

/*
 * Synchronises `stream`, then reads and clears the device-side error word of
 * the current device.  Returns RF_OK, RF_ERR_DEVICE_TIMEOUT (some kernel gave
 * up on a bounded wait and returned early; its outputs are incomplete),
 * RF_ERR_DEVICE_INPUT (a kernel found device-resident sizes, such as the
 * cumulative sequence lengths of rf_attn_fwd_varlen, inconsistent with the
 * host-side sizes; it skipped that work and wrote nothing out of bounds),
 * RF_ERR_DEVICE_LAYOUT (a kernel found its dynamic shared memory not aligned
 * as its swizzled tiles need; it did no work), RF_ERR_DEVICE_BOUNDS (only in
 * the bounds-checked debug build of the library, librf_gb300_dbg.so: a
 * thread's global load or store would have fallen outside its tensor; it was
 * skipped) or RF_ERR_CUDA (the synchronisation itself failed).  When several
 * kinds occurred, the first of TIMEOUT, BOUNDS, LAYOUT, INPUT in that order is
 * returned.
 */
rf_status rf_get_device_status(rf_stream_t stream);

/*
 * Single-segment fused attention ([E] §2.2, §4.1; [S] Methodologie 2 and the
 * single-segment strategy of Methodologie 3): for every (b, h, query row),
 *     s_j = scale * q . k_j,  m = max_j s_j,  l = sum_j exp(s_j - m),
 *     o   = sum_j exp(s_j - m) / l * v_j,
 * computed by one CTA per block of query rows in a single loop over key
 * tiles with the running (m, l, o) rescaled per tile; S and P never reach
 * global memory.
 *   dtype   RF_F32: Q/K/V/O fp32, exact-fp32 SIMT path (no tensor cores).
 *           RF_BF16: Q/K/V/O bf16, tcgen05 tensor-core path, fp32
 *           accumulation and softmax state, P rounded to bf16 for P.V.
 *   Q, O    [B][H][Lq][d];  K, V  [B][H][Lk][d]  (multi-head: one K/V head
 *           per query head).
 *   Sizes   B, H, Lq, Lk >= 1 (B*H*Lq and B*H*Lk below 2^31; for RF_F32
 *           also B*H <= 65535); d = 64 (both dtypes) or 128 (RF_F32 only).
 *   scale   finite and > 0 (the usual 1/sqrt(d)).
 *   causal  0: every row reads every key.  1: autoregressive mask aligned
 *           to the end of the keys (the pages define no mask; this is the
 *           usual reading): row i reads keys j <= i + (Lk - Lq) only, so the
 *           last row reads all Lk keys; a row that reads no key (possible
 *           only when Lq > Lk) is written as zeros.
 * Errors: RF_ERR_INVALID_ARG (null/misaligned pointer, size < 1 or beyond
 * the limits above, causal not 0 or 1, bad dtype), RF_ERR_UNSUPPORTED (d not
 * covered), RF_ERR_CUDA.
 */
rf_status rf_attn_fwd(int dtype, const void* Q, const void* K, const void* V, void* O,
                      int B, int H, int Lq, int Lk, int d, float scale, int causal,
                      rf_stream_t stream);

/* Evaluation order of the softmax cascade for rf_attn_fwd_ex. */
typedef enum {
  RF_ATTN_AUTO = 0,          /* the library's choice (what rf_attn_fwd uses): the
                                incremental order, which measured faster on this
                                GPU at Lk = 128 and 256 as well                  */
  RF_ATTN_INCREMENTAL = 1,   /* one loop over key tiles, running (m, l, o)
                                rescaled per tile ([E] §2.3; [S] Methodologie 2) */
  RF_ATTN_TWO_PASS = 2       /* non-incremental: exact row max over all keys,
                                then P and O with no rescale; Lk <= 256, bf16
                                only ([E] §5.2: short reductions)                */
} rf_attn_mode;

/*
 * rf_attn_fwd with an explicit evaluation order `mode` (an rf_attn_mode).
 * Both orders compute the same cascade; they differ in rounding only.
 * Errors as rf_attn_fwd, plus RF_ERR_INVALID_ARG for an unknown mode and
 * RF_ERR_UNSUPPORTED for RF_ATTN_TWO_PASS with RF_F32 or with Lk > 256.
 */
rf_status rf_attn_fwd_ex(int dtype, const void* Q, const void* K, const void* V, void* O,
                         int B, int H, int Lq, int Lk, int d, float scale, int causal, int mode,
                         rf_stream_t stream);

/*
 * rf_attn_fwd over a batch of sequences of different lengths, packed
 * token-major without padding (the same computation per sequence and head,
 * including the causal option):
 *   Q, O   [total_q][H][d];  K, V  [total_k][H][d]  (bf16 or fp32 as dtype).
 *   cu_seqlens_q, cu_seqlens_k   DEVICE int32 arrays of B + 1 cumulative
 *          lengths: sequence b owns query tokens cu_seqlens_q[b] ..
 *          cu_seqlens_q[b+1]-1 and key tokens cu_seqlens_k[b] ..
 *          cu_seqlens_k[b+1]-1; entry 0 is 0, entries never decrease, the
 *          last equals total_q (total_k).  Lengths may be 0; a sequence with
 *          no keys gives zero rows.
 *   max_seqlen_q   >= every query length (sizes the grid).
 *   total_q, total_k >= 1; B * H <= 65535; total_q * H, total_k * H < 2^31.
 *   d = 64 (both dtypes) or 128 (RF_F32 only).
 * The host does not read the device arrays.  A kernel that finds them
 * inconsistent with max_seqlen_q / total_q / total_k skips that sequence,
 * touches nothing out of bounds and makes rf_get_device_status report
 * RF_ERR_DEVICE_INPUT.
 * Errors: RF_ERR_INVALID_ARG, RF_ERR_UNSUPPORTED, RF_ERR_CUDA.
 */
rf_status rf_attn_fwd_varlen(int dtype, const void* Q, const void* K, const void* V, void* O,
                             const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int B,
                             int H, int max_seqlen_q, int total_q, int total_k, int d,
                             float scale, int causal, rf_stream_t stream);

/*
 * Number of key segments rf_attn_decode_splitkv cuts a (b, kv head) sequence
 * into for this shape when its num_splits argument is `num_splits`: that
 * number itself when it is > 0; for 0 (the automatic partition, sized to the
 * device's SM count) the most segments any one sequence can be cut into.
 * Returns 0 for an invalid shape, or for 0 when no device can be queried.
 */
int rf_attn_decode_splitkv_num_splits(int B, int Hq, int Hkv, int Lk, int d, int num_splits);

/* Workspace bytes rf_attn_decode_splitkv needs for the same arguments (for
 * num_splits = 0 it depends on the current device's SM count). */
size_t rf_attn_decode_splitkv_workspace_size(int B, int Hq, int Hkv, int Lk, int d,
                                             int num_splits);

/*
 * Multi-segment (split-KV) fused decode attention ([S] Methodologie 3,
 * multi-segment strategy; [E] §3.3 inter-block merge).  One query token per
 * (b, query head):
 *   Q   [B][Hq][d] bf16;  K, V  [B][Hkv][Lk][d] bf16;  O  [B][Hq][d] bf16.
 * Grouped-query attention: query head hq reads K/V head hq / (Hq / Hkv).
 * One kernel (a persistent grid of at most one CTA per SM) cuts the
 * (b, kv head) sequences into key segments, reduces each segment to a
 * partial state (m, l, o) per query head (o unnormalised, m in log2 units)
 * and merges the segments of a sequence: M = max m_j,
 * L = sum l_j 2^(m_j - M), O = sum o_j 2^(m_j - M) / L.  The merge is done
 * by the CTA that finishes a sequence's last segment, always in key order,
 * so the result does not depend on which CTA that is.
 *   Sizes   B, Lk >= 1; d = 128; Hq / Hkv in {1, 2, 4, 8}; scale finite, > 0.
 *   num_splits  0 = automatic: the 32-key chunks of all sequences, end to
 *               end, are cut into one equal range per CTA (a sequence may be
 *               cut into several segments, another lie within one range);
 *               1..Lk = each sequence cut into that many equal segments
 *               (the segments are handed to the CTAs round-robin; every
 *               segment adds a fence, a ticket and a merge step, so large
 *               counts are much slower than the automatic partition and
 *               are meant for exercising the merge).
 *   workspace   device buffer of at least
 *               rf_attn_decode_splitkv_workspace_size(...) bytes, 16-byte
 *               aligned, owned by the caller; holds a ticket counter per
 *               sequence (zeroed by a memset on `stream` before the kernel)
 *               and the partial states of segments.  Its contents need not
 *               be initialised and are unspecified on return.
 * Errors: RF_ERR_INVALID_ARG, RF_ERR_UNSUPPORTED, RF_ERR_WORKSPACE, RF_ERR_CUDA.
 */
rf_status rf_attn_decode_splitkv(const void* Q, const void* K, const void* V, void* O,
                                 int B, int Hq, int Hkv, int Lk, int d, float scale,
                                 int num_splits, void* workspace, size_t workspace_bytes,
                                 rf_stream_t stream);

/* Size in bytes of the built-in scratch of rf_attn_decode_splitkv_noalloc. */
#define RF_DECODE_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * Allocation-free form of rf_attn_decode_splitkv (the paper has no
 * counterpart: this is an interface convenience).  For callers that cannot
 * provide device memory -- a plugin behind a fixed C interface with no
 * workspace argument, a serving loop that must not allocate after start-up,
 * or a host framework whose own pool allocator owns the device memory.
 * Same arguments, computation and results as rf_attn_decode_splitkv, but the
 * partial states go to a 16 MiB scratch array built into the library (a
 * file-scope __device__ array that every GPU loading the library keeps
 * until the process exits); the function never allocates or frees memory.
 *   - Returns RF_ERR_WORKSPACE when the partial states of the request,
 *     rf_attn_decode_splitkv_workspace_size(...), exceed
 *     RF_DECODE_NOALLOC_SCRATCH_BYTES (lower num_splits, or use
 *     rf_attn_decode_splitkv with a caller workspace).
 *   - The first call on a device looks up the scratch's device address (one
 *     cudaGetSymbolAddress with that device current) and caches it with the
 *     device's current CUDA context; make that first call before any stream
 *     capture on the device.  After a device reset the runtime creates a new
 *     context, and the next call looks the address up again (so, again,
 *     before any capture).
 *   - All calls on a device share the one scratch, which keeps the last
 *     call's contents (nothing in it needs to start at zero).  Calls that
 *     may overlap on the GPU -- on different streams without ordering, or
 *     from several host threads -- race on it; serialise them on one stream.
 */
rf_status rf_attn_decode_splitkv_noalloc(const void* Q, const void* K, const void* V, void* O,
                                         int B, int Hq, int Hkv, int Lk, int d, float scale,
                                         int num_splits, rf_stream_t stream);

/*
 * Number of key segments per batch that rf_mla_decode uses for this shape
 * when its num_splits argument is `num_splits` (0 = automatic: one segment
 * unless the batches alone leave most SMs idle).  Returns 0 for an invalid
 * or unsupported shape.
 */
int rf_mla_decode_num_splits(int B, int Hq, int Lk, int d_qk, int d_v, int num_splits);

/* Workspace bytes rf_mla_decode needs for the same arguments (0 when it
 * uses one segment per batch). */
size_t rf_mla_decode_workspace_size(int B, int Hq, int Lk, int d_qk, int d_v, int num_splits);

/*
 * Latent-KV (multi-latent attention) decode, absorbed form -- the
 * technical summary's MLA workload ([S] "Resultaten"), whose operation the
 * pages do not define; the public definition is used.  One query token per
 * (b, head); every head of batch b attends to the one latent cache of b:
 *   Q    [B][Hq][d_qk] bf16   (latent part, then positional part)
 *   CKV  [B][Lk][d_qk] bf16   (cache rows: the first d_v dims are the latent
 *                              vector, which also serves as the value)
 *   O    [B][Hq][d_v]  bf16
 *   s_j = scale * Q[b,h,:] . CKV[b,j,:]   (all d_qk dims)
 *   O[b,h,:] = sum_j softmax(s)_j CKV[b,j,0:d_v]
 * computed as the safe-softmax cascade in one incremental loop over tiles
 * of 64 cache rows ([E] §2.3, §4.1), on a cluster of two CTAs per (batch,
 * segment) that exchange partial scores; with more than one segment, the
 * partial states (m, l, o) of the segments are merged by a second kernel
 * ([S] Methodologie 3).
 *   Sizes   B, Lk >= 1; 1 <= Hq <= 128; d_qk = 576 and d_v = 512 (else
 *           RF_ERR_UNSUPPORTED); scale finite, > 0.
 *   num_splits  0 = automatic, else the requested number of segments
 *           (clamped to whole 64-row tiles: rf_mla_decode_num_splits tells
 *           the count used).
 *   workspace   device buffer of at least rf_mla_decode_workspace_size(...)
 *           bytes, 16-byte aligned, owned by the caller; may be NULL when
 *           that size is 0.  Contents need not be initialised and are
 *           unspecified on return.
 * All pointers are device pointers, 16-byte aligned.
 * Errors: RF_ERR_INVALID_ARG, RF_ERR_UNSUPPORTED, RF_ERR_WORKSPACE,
 * RF_ERR_CUDA; a bounded wait that runs out on the device (or cluster peer)
 * is reported by rf_get_device_status as RF_ERR_DEVICE_TIMEOUT.
 */
rf_status rf_mla_decode(const void* Q, const void* CKV, void* O, int B, int Hq, int Lk, int d_qk,
                        int d_v, float scale, int num_splits, void* workspace,
                        size_t workspace_bytes, rf_stream_t stream);

/*
 * Fused MoE gate ([E] §4.2): scores = x . W_gate^T, top-k experts per token,
 * softmax over the k selected scores; the score matrix never reaches
 * global memory.
 *   X      [T][D] bf16 (token activations).
 *   Wg     [E][D] bf16 (gate weight, expert-major: a linear layer's weight).
 *   idx    [T][k] int32 out: selected experts by descending score, equal
 *          scores by ascending expert index.
 *   w      [T][k] fp32 out: softmax of the selected scores (same order).
 *   Sizes  1 <= T <= 7864200 (65535 x 120: tiles of up to 128 tokens are
 *          the grid's y extent); D >= 1 with D % 8 == 0; 1 <= E <= 256;
 *          1 <= k <= min(8, E).
 * Scores are accumulated in fp32 on the tensor cores (exact when every
 * partial sum is an integer below 2^24, e.g. small-integer inputs).
 * Errors: RF_ERR_INVALID_ARG (null/misaligned pointer, size < 1, k > E,
 * D % 8 != 0), RF_ERR_UNSUPPORTED (E > 256, k > 8 or T > 7864200),
 * RF_ERR_CUDA.
 */
rf_status rf_moe_gate_topk_softmax(const void* X, const void* Wg, int T, int D, int E, int k,
                                   int32_t* idx, float* w, rf_stream_t stream);

/* Layouts of W_gate for rf_moe_gate_topk_softmax_ex. */
#define RF_GATE_W_ED 0 /* [E][D]: expert-major, a linear layer's weight  */
#define RF_GATE_W_DE 1 /* [D][E]: dim-major, scores = X . W_gate           */

/*
 * rf_moe_gate_topk_softmax with the layout of W_gate given: the same
 * computation, arguments and errors, with
 *   w_layout  RF_GATE_W_ED: Wg [E][D] (as rf_moe_gate_topk_softmax);
 *             RF_GATE_W_DE: Wg [D][E] bf16, scores[t][e] = sum_d X[t][d]
 *             Wg[d][e] ([E] §4.2 writes the gate as x . W_gate); E must be
 *             64, 128, 192 or 256 (else RF_ERR_UNSUPPORTED); any other
 *             w_layout value: RF_ERR_INVALID_ARG.
 */
rf_status rf_moe_gate_topk_softmax_ex(const void* X, const void* Wg, int T, int D, int E, int k,
                                      int w_layout, int32_t* idx, float* w, rf_stream_t stream);

/*
 * Workspace bytes rf_absmax_fp8_gemm needs when neither sx_out nor xq_out is
 * given (0 for an invalid shape).  With both outputs given it needs only the
 * row counters at the start of this size: 4 * (1 + ceil(M / 128)) bytes,
 * rounded up to 256.
 */
size_t rf_absmax_fp8_gemm_workspace_size(int M, int N, int K);

/*
 * Dynamic FP8 quantised GEMM ([E] §4.3), read per row of X:
 *   sx[m]    = fp32(max_k |X[m,k]| / 448)                     (row absmax)
 *   Xq[m,k]  = E4M3(fp32(X[m,k] / sx[m])), round-to-nearest-even,
 *              saturating to +-448; rows with sx = 0 give code 0x00, and a
 *              negative value that rounds to zero gives 0x80
 *   Y[m,n]   = bf16( (sum_k Xq[m,k] * Wq[n,k]) * sx[m] * sw[n] )
 * The division is an IEEE fp32 division; the sum is accumulated in fp32 on
 * the tensor cores (tcgen05 kind::f8f6f4); Y is rounded to nearest even.
 * One persistent kernel does both stages: quantiser warps read each row of X
 * once (absmax and quantisation from registers), and the GEMM of a 128-row
 * block of X starts as soon as that block's codes are written.
 *   X       [M][K] bf16.
 *   Wq      [N][K] uint8 E4M3 codes (pre-quantised weight; K contiguous).
 *   sw      [N] fp32 per-output-column weight scales.
 *   Y       [M][N] bf16 out.
 *   sx_out  [M] fp32 out, or NULL (then kept in the workspace).
 *   xq_out  [M][K] uint8 out, or NULL (then kept in the workspace).
 *   workspace  device buffer, 16-byte aligned, always required: the
 *              kernel's row counters (reset by the call itself, with a
 *              memset on `stream`), plus the codes and scales the caller
 *              does not keep.  rf_absmax_fp8_gemm_workspace_size(M,N,K)
 *              bytes always suffice.  Calls that overlap on the GPU must
 *              not share a workspace.
 *   Sizes   M, N >= 1; K >= 16 with K % 16 == 0.
 * Errors: RF_ERR_INVALID_ARG, RF_ERR_WORKSPACE (missing, misaligned or too
 * small), RF_ERR_CUDA.
 */
rf_status rf_absmax_fp8_gemm(const void* X, const uint8_t* Wq, const float* sw, void* Y,
                             int M, int N, int K, float* sx_out, uint8_t* xq_out,
                             void* workspace, size_t workspace_bytes, rf_stream_t stream);

/*
 * The first two steps of the FP8 cascade alone ([E] §4.3): row absmax and
 * E4M3 quantisation, with the same arithmetic and bits as
 * rf_absmax_fp8_gemm (sx[m] = fp32(max_k |X[m,k]| / 448), Xq = E4M3(fp32(X /
 * sx)) round-to-nearest-even, satfinite, signed zero kept).  Used, for
 * example, to quantise a weight per output column (rows of Wq [N][K]).
 *   X       [M][K] bf16.
 *   sx_out  [M] fp32 out.
 *   xq_out  [M][K] uint8 E4M3 codes out.
 *   Sizes   M >= 1; K >= 16 with K % 16 == 0.
 * Errors: RF_ERR_INVALID_ARG, RF_ERR_CUDA.
 */
rf_status rf_absmax_quant_fp8(const void* X, int M, int K, float* sx_out, uint8_t* xq_out,
                              rf_stream_t stream);

/*
 * Failure-detection self-test (no counterpart in the paper).  Launches one
 * CTA that waits on an mbarrier nothing ever completes, with a wait limit of
 * `timeout_us` microseconds (1..1000000).  The kernel gives up, records
 * RF_ERR_DEVICE_TIMEOUT in the device error word and returns, leaving the
 * context usable; rf_get_device_status then reports it.
 */
rf_status rf_selftest_wait_timeout(int timeout_us, rf_stream_t stream);

/*
 * Bounds-check self-test (no counterpart in the paper).  In the
 * bounds-checked debug build (librf_gb300_dbg.so, built with
 * RF_DEBUG_BOUNDS) it launches one thread that asks the kernels' bounds check
 * about an element index one past the end of a 16-element tensor: the check
 * records it, the access is never made, and rf_get_device_status then reports
 * RF_ERR_DEVICE_BOUNDS.  In the normal build it returns RF_ERR_UNSUPPORTED
 * and launches nothing.
 */
rf_status rf_selftest_bounds(rf_stream_t stream);

/*
 * Host-side check of the split-KV decode partition (no counterpart in the
 * paper; no GPU needed, no CUDA call made).  For B * Hkv sequences of Lk keys,
 * num_splits as in rf_attn_decode_splitkv (0 = automatic) and a device of
 * `sms` SMs, it walks the pieces every CTA would take and checks that every
 * CTA has work, that the pieces of each sequence cover its keys exactly once,
 * that the workspace slots of split sequences are distinct and in range, and
 * that the merge would read a sequence's slots in key order.  Returns 0 when
 * all of that holds, -1 for a shape rf_attn_decode_splitkv refuses (sizes
 * < 1, num_splits outside 0..Lk, B * Hkv * Lk >= 2^31, sms < 1), else the
 * number (1..7) of the first check that fails.
 */
int rf_selftest_decode_plan(int B, int Hkv, int Lk, int num_splits, int sms);

/*
 * Host-side check of the tile schedule of rf_absmax_fp8_gemm (no
 * counterpart in the paper; no GPU needed, no CUDA call made).  For an
 * M x N output computed by `clusters` CTA pairs (1..4096) it checks that the
 * pairs' tile counts add up, that every scheduled tile is a 256 x 256 tile
 * or a 256 x 128 column half on that grid, and that every 256-row x
 * 128-column block of the output is computed exactly once.  Returns 0 when
 * all of that holds, -1 for sizes < 1, clusters outside 1..4096 or more than
 * 2^24 tiles, else the number (1..3) of the first check that fails.
 */
int rf_selftest_fp8_schedule(int M, int N, int clusters);

/*
 * Host-side check of the tile plan of rf_moe_gate_topk_softmax (no
 * counterpart in the paper; no GPU needed, no CUDA call made).  For T tokens
 * of D dims, E experts and a device of `sms` SMs it checks that the chosen
 * cluster size (1, 2, 4 or 8 CTAs splitting D) and tile height (a multiple
 * of 8 up to 128 tokens) are valid, that the tiles hold every token once and
 * fit the grid (for T <= 7864200), that the cluster's CTAs share the
 * k-blocks with none idle, and that the epilogue's rows cover each tile.
 * Returns 0 when all of that holds, -1 for refused sizes (T, D, E < 1,
 * D % 8 != 0, E > 256, sms < 1), else the number (1..6) of the first check
 * that fails.
 */
int rf_selftest_moe_plan(int T, int D, int E, int sms);

#ifdef __cplusplus
}
#endif

#endif /* RF_H_ */
