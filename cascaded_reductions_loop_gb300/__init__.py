"""Python binding of librf_gb300.so, the fused cascaded-reduction kernels for
GB300 (sm_103a).

Argument marshalling only: each function below checks tensor shapes and
dtypes, then calls the C entry point of the same name (declared in
``include/rf.h``) with raw device pointers and the current torch CUDA
stream.  Every step of the computation runs in the library's CUDA kernels;
there is no other implementation behind these names.  If the library is
missing, importing this package raises: build it first with
``python __graft_entry__.py`` (or ``python cascaded_reductions_loop_gb300/_build.py``).
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

__all__ = [
    "RFError", "lib", "rf_status_string", "rf_version", "rf_get_device_status", "rf_last_cuda_error",
    "rf_attn_fwd", "rf_attn_fwd_ex", "rf_attn_fwd_varlen", "rf_attn_decode_splitkv",
    "rf_attn_decode_splitkv_num_splits",
    "rf_attn_decode_splitkv_workspace_size", "rf_attn_decode_splitkv_noalloc",
    "RF_DECODE_NOALLOC_SCRATCH_BYTES", "rf_mla_decode", "rf_mla_decode_num_splits",
    "rf_mla_decode_workspace_size", "rf_moe_gate_topk_softmax", "rf_moe_gate_topk_softmax_ex",
    "rf_absmax_fp8_gemm", "rf_absmax_fp8_gemm_workspace_size", "rf_absmax_quant_fp8",
    "rf_selftest_wait_timeout", "rf_selftest_bounds", "rf_selftest_decode_plan",
    "rf_selftest_fp8_schedule", "rf_selftest_moe_plan",
    "RF_OK", "RF_ERR_INVALID_ARG", "RF_ERR_UNSUPPORTED", "RF_ERR_WORKSPACE", "RF_ERR_CUDA",
    "RF_ERR_DEVICE_TIMEOUT", "RF_ERR_DEVICE_INPUT", "RF_ERR_DEVICE_LAYOUT", "RF_ERR_DEVICE_BOUNDS",
    "RF_F32", "RF_BF16",
    "RF_ATTN_AUTO", "RF_ATTN_INCREMENTAL", "RF_ATTN_TWO_PASS", "RF_GATE_W_ED", "RF_GATE_W_DE",
]

RF_OK, RF_ERR_INVALID_ARG, RF_ERR_UNSUPPORTED, RF_ERR_WORKSPACE, RF_ERR_CUDA, \
    RF_ERR_DEVICE_TIMEOUT, RF_ERR_DEVICE_INPUT, RF_ERR_DEVICE_LAYOUT, RF_ERR_DEVICE_BOUNDS = range(9)
RF_F32, RF_BF16 = 0, 1
RF_ATTN_AUTO, RF_ATTN_INCREMENTAL, RF_ATTN_TWO_PASS = 0, 1, 2
RF_GATE_W_ED, RF_GATE_W_DE = 0, 1                # layouts of W_gate: [E][D], [D][E]
RF_DECODE_NOALLOC_SCRATCH_BYTES = 16 << 20   # as in rf.h

# RF_GB300_LIB=debug selects the bounds-checked debug build of the same library
LIB_PATH = _build.DEBUG_LIB_PATH if os.environ.get("RF_GB300_LIB") == "debug" else _build.LIB_PATH

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: the CUDA library must be built first "
        "(python __graft_entry__.py); there is no fallback path")

_c = ctypes
_P = _c.c_void_p
_I = _c.c_int
_F = _c.c_float
_Z = _c.c_size_t

lib = _c.CDLL(LIB_PATH)

_SIGS = {
    "rf_status_string": (_c.c_char_p, [_I]),
    "rf_last_cuda_error": (_c.c_char_p, []),
    "rf_version": (_I, []),
    "rf_get_device_status": (_I, [_P]),
    "rf_attn_fwd": (_I, [_I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P]),
    "rf_attn_fwd_ex": (_I, [_I, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _I, _P]),
    "rf_attn_fwd_varlen": (_I, [_I, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P]),
    "rf_attn_decode_splitkv_num_splits": (_I, [_I, _I, _I, _I, _I, _I]),
    "rf_attn_decode_splitkv_workspace_size": (_Z, [_I, _I, _I, _I, _I, _I]),
    "rf_attn_decode_splitkv": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _Z, _P]),
    "rf_attn_decode_splitkv_noalloc": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P]),
    "rf_mla_decode_num_splits": (_I, [_I, _I, _I, _I, _I, _I]),
    "rf_mla_decode_workspace_size": (_Z, [_I, _I, _I, _I, _I, _I]),
    "rf_mla_decode": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _F, _I, _P, _Z, _P]),
    "rf_moe_gate_topk_softmax": (_I, [_P, _P, _I, _I, _I, _I, _P, _P, _P]),
    "rf_moe_gate_topk_softmax_ex": (_I, [_P, _P, _I, _I, _I, _I, _I, _P, _P, _P]),
    "rf_absmax_fp8_gemm_workspace_size": (_Z, [_I, _I, _I]),
    "rf_absmax_fp8_gemm": (_I, [_P, _P, _P, _P, _I, _I, _I, _P, _P, _P, _Z, _P]),
    "rf_absmax_quant_fp8": (_I, [_P, _I, _I, _P, _P, _P]),
    "rf_selftest_wait_timeout": (_I, [_I, _P]),
    "rf_selftest_bounds": (_I, [_P]),
    "rf_selftest_decode_plan": (_I, [_I, _I, _I, _I, _I]),
    "rf_selftest_fp8_schedule": (_I, [_I, _I, _I]),
    "rf_selftest_moe_plan": (_I, [_I, _I, _I, _I]),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(lib, _name)
    _fn.restype = _res
    _fn.argtypes = _args


class RFError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {rf_status_string(status)}"
        if status == RF_ERR_CUDA:
            msg += f" ({lib.rf_last_cuda_error().decode()})"
        super().__init__(msg)


def _check(status: int, where: str) -> None:
    if status != RF_OK:
        raise RFError(status, where)


def _ptr(t):
    return None if t is None else _c.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return _c.c_void_p(stream.cuda_stream)


def _need(t, dtype, shape, name):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


# ------------------------------------------------------------------ entry points


def rf_status_string(status: int) -> str:
    return lib.rf_status_string(int(status)).decode()


def rf_version() -> int:
    return lib.rf_version()


def rf_last_cuda_error() -> str:
    return lib.rf_last_cuda_error().decode()


def rf_get_device_status(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device status."""
    return lib.rf_get_device_status(_stream(stream))


def rf_attn_fwd(q, k, v, o, scale: float, causal: int = 0, stream=None) -> None:
    """Single-segment fused attention.  q, o: [B,H,Lq,d]; k, v: [B,H,Lk,d];
    all fp32 (exact SIMT path) or all bf16 (tcgen05 path)."""
    _attn_fwd(q, k, v, o, scale, causal, None, stream)


def rf_attn_fwd_ex(q, k, v, o, scale: float, causal: int, mode: int, stream=None) -> None:
    """rf_attn_fwd with an explicit evaluation order: RF_ATTN_AUTO,
    RF_ATTN_INCREMENTAL or RF_ATTN_TWO_PASS (bf16, Lk <= 256)."""
    _attn_fwd(q, k, v, o, scale, causal, mode, stream)


def _attn_fwd(q, k, v, o, scale, causal, mode, stream):
    B, H, Lq, d = q.shape
    Lk = k.shape[2]
    dt = q.dtype
    if dt not in (torch.float32, torch.bfloat16):
        raise ValueError("q must be float32 or bfloat16")
    _need(q, dt, (B, H, Lq, d), "q")
    _need(k, dt, (B, H, Lk, d), "k")
    _need(v, dt, (B, H, Lk, d), "v")
    _need(o, dt, (B, H, Lq, d), "o")
    code = RF_F32 if dt == torch.float32 else RF_BF16
    if mode is None:
        _check(lib.rf_attn_fwd(code, _ptr(q), _ptr(k), _ptr(v), _ptr(o), B, H, Lq, Lk, d,
                               float(scale), int(causal), _stream(stream)), "rf_attn_fwd")
    else:
        _check(lib.rf_attn_fwd_ex(code, _ptr(q), _ptr(k), _ptr(v), _ptr(o), B, H, Lq, Lk, d,
                                  float(scale), int(causal), int(mode), _stream(stream)),
               "rf_attn_fwd_ex")


def rf_attn_fwd_varlen(q, k, v, o, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, scale: float,
                       causal: int = 0, stream=None) -> None:
    """Fused attention over packed variable-length sequences.  q, o:
    [total_q,H,d]; k, v: [total_k,H,d]; cu_seqlens_q/k: int32 CUDA tensors
    of B+1 cumulative lengths (not read on the host)."""
    total_q, H, d = q.shape
    total_k = k.shape[0]
    B = cu_seqlens_q.shape[0] - 1
    dt = q.dtype
    if dt not in (torch.float32, torch.bfloat16):
        raise ValueError("q must be float32 or bfloat16")
    _need(q, dt, (total_q, H, d), "q")
    _need(k, dt, (total_k, H, d), "k")
    _need(v, dt, (total_k, H, d), "v")
    _need(o, dt, (total_q, H, d), "o")
    _need(cu_seqlens_q, torch.int32, (B + 1,), "cu_seqlens_q")
    _need(cu_seqlens_k, torch.int32, (B + 1,), "cu_seqlens_k")
    code = RF_F32 if dt == torch.float32 else RF_BF16
    _check(lib.rf_attn_fwd_varlen(code, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(cu_seqlens_q),
                                  _ptr(cu_seqlens_k), B, H, int(max_seqlen_q), total_q, total_k,
                                  d, float(scale), int(causal), _stream(stream)),
           "rf_attn_fwd_varlen")


def rf_attn_decode_splitkv_num_splits(B, Hq, Hkv, Lk, d, num_splits=0) -> int:
    return lib.rf_attn_decode_splitkv_num_splits(B, Hq, Hkv, Lk, d, num_splits)


def rf_attn_decode_splitkv_workspace_size(B, Hq, Hkv, Lk, d, num_splits=0) -> int:
    return lib.rf_attn_decode_splitkv_workspace_size(B, Hq, Hkv, Lk, d, num_splits)


def rf_attn_decode_splitkv(q, k, v, o, scale: float, workspace, num_splits: int = 0,
                           stream=None) -> None:
    """Multi-segment decode attention.  q, o: [B,Hq,d] bf16; k, v:
    [B,Hkv,Lk,d] bf16; workspace: a uint8 CUDA tensor of at least
    rf_attn_decode_splitkv_workspace_size(...) bytes."""
    B, Hq, d = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    _need(q, torch.bfloat16, (B, Hq, d), "q")
    _need(k, torch.bfloat16, (B, Hkv, Lk, d), "k")
    _need(v, torch.bfloat16, (B, Hkv, Lk, d), "v")
    _need(o, torch.bfloat16, (B, Hq, d), "o")
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.rf_attn_decode_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, Hq, Hkv, Lk, d,
                                      float(scale), int(num_splits), _ptr(workspace), ws_bytes,
                                      _stream(stream)), "rf_attn_decode_splitkv")


def rf_attn_decode_splitkv_noalloc(q, k, v, o, scale: float, num_splits: int = 0,
                                   stream=None) -> None:
    """rf_attn_decode_splitkv with the library's built-in scratch instead of a
    caller workspace, for callers that cannot provide device memory.  The
    first call on a device must come before any stream capture; calls that
    overlap on the GPU race on the shared scratch."""
    B, Hq, d = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    _need(q, torch.bfloat16, (B, Hq, d), "q")
    _need(k, torch.bfloat16, (B, Hkv, Lk, d), "k")
    _need(v, torch.bfloat16, (B, Hkv, Lk, d), "v")
    _need(o, torch.bfloat16, (B, Hq, d), "o")
    _check(lib.rf_attn_decode_splitkv_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), B, Hq, Hkv, Lk,
                                              d, float(scale), int(num_splits), _stream(stream)),
           "rf_attn_decode_splitkv_noalloc")


def rf_mla_decode_num_splits(B, Hq, Lk, d_qk=576, d_v=512, num_splits=0) -> int:
    return lib.rf_mla_decode_num_splits(B, Hq, Lk, d_qk, d_v, num_splits)


def rf_mla_decode_workspace_size(B, Hq, Lk, d_qk=576, d_v=512, num_splits=0) -> int:
    return lib.rf_mla_decode_workspace_size(B, Hq, Lk, d_qk, d_v, num_splits)


def rf_mla_decode(q, ckv, o, scale: float, workspace=None, num_splits: int = 0,
                  stream=None) -> None:
    """Latent-KV (multi-latent attention) decode.  q: [B,Hq,d_qk] bf16; ckv:
    [B,Lk,d_qk] bf16 latent cache (its first d_v dims are the values); o:
    [B,Hq,d_v] bf16 out; workspace: a uint8 CUDA tensor of at least
    rf_mla_decode_workspace_size(...) bytes, or None when that size is 0."""
    B, Hq, d_qk = q.shape
    Lk = ckv.shape[1]
    d_v = o.shape[2]
    _need(q, torch.bfloat16, (B, Hq, d_qk), "q")
    _need(ckv, torch.bfloat16, (B, Lk, d_qk), "ckv")
    _need(o, torch.bfloat16, (B, Hq, d_v), "o")
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.rf_mla_decode(_ptr(q), _ptr(ckv), _ptr(o), B, Hq, Lk, d_qk, d_v, float(scale),
                             int(num_splits), _ptr(workspace), ws_bytes, _stream(stream)),
           "rf_mla_decode")


def rf_moe_gate_topk_softmax(x, w_gate, k: int, idx, weights, stream=None) -> None:
    """Fused MoE gate.  x: [T,D] bf16; w_gate: [E,D] bf16 (expert-major);
    idx: [T,k] int32 out; weights: [T,k] fp32 out."""
    T, D = x.shape
    E = w_gate.shape[0]
    _need(x, torch.bfloat16, (T, D), "x")
    _need(w_gate, torch.bfloat16, (E, D), "w_gate")
    _need(idx, torch.int32, (T, k), "idx")
    _need(weights, torch.float32, (T, k), "weights")
    _check(lib.rf_moe_gate_topk_softmax(_ptr(x), _ptr(w_gate), T, D, E, int(k), _ptr(idx),
                                        _ptr(weights), _stream(stream)),
           "rf_moe_gate_topk_softmax")


def rf_moe_gate_topk_softmax_ex(x, w_gate, k: int, w_layout: int, idx, weights,
                                stream=None) -> None:
    """Fused MoE gate with the layout of W_gate given.  x: [T,D] bf16;
    w_gate: [E,D] bf16 (RF_GATE_W_ED) or [D,E] bf16 (RF_GATE_W_DE, E a
    multiple of 64, at most 256); idx: [T,k] int32 out; weights: [T,k] fp32 out."""
    T, D = x.shape
    if w_layout == RF_GATE_W_DE:
        E = w_gate.shape[1]
        _need(w_gate, torch.bfloat16, (D, E), "w_gate")
    else:
        E = w_gate.shape[0]
        _need(w_gate, torch.bfloat16, (E, D), "w_gate")
    _need(x, torch.bfloat16, (T, D), "x")
    _need(idx, torch.int32, (T, k), "idx")
    _need(weights, torch.float32, (T, k), "weights")
    _check(lib.rf_moe_gate_topk_softmax_ex(_ptr(x), _ptr(w_gate), T, D, E, int(k), int(w_layout),
                                           _ptr(idx), _ptr(weights), _stream(stream)),
           "rf_moe_gate_topk_softmax_ex")


def rf_absmax_fp8_gemm_workspace_size(M, N, K) -> int:
    return lib.rf_absmax_fp8_gemm_workspace_size(M, N, K)


def rf_absmax_fp8_gemm(x, wq, sw, y, workspace, sx_out=None, xq_out=None, stream=None) -> None:
    """Row absmax -> E4M3 quantisation -> FP8 GEMM -> dequantisation.
    x: [M,K] bf16; wq: [N,K] uint8 E4M3 codes; sw: [N] fp32; y: [M,N] bf16
    out; workspace: uint8 CUDA tensor of at least
    rf_absmax_fp8_gemm_workspace_size(M, N, K) bytes (always required: it
    holds the kernel's row counters); sx_out: [M] fp32 out or None; xq_out:
    [M,K] uint8 out or None."""
    M, K = x.shape
    N = wq.shape[0]
    _need(x, torch.bfloat16, (M, K), "x")
    _need(wq, torch.uint8, (N, K), "wq")
    _need(sw, torch.float32, (N,), "sw")
    _need(y, torch.bfloat16, (M, N), "y")
    if sx_out is not None:
        _need(sx_out, torch.float32, (M,), "sx_out")
    if xq_out is not None:
        _need(xq_out, torch.uint8, (M, K), "xq_out")
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib.rf_absmax_fp8_gemm(_ptr(x), _ptr(wq), _ptr(sw), _ptr(y), M, N, K, _ptr(sx_out),
                                  _ptr(xq_out), _ptr(workspace), ws_bytes, _stream(stream)),
           "rf_absmax_fp8_gemm")


def rf_absmax_quant_fp8(x, sx_out, xq_out, stream=None) -> None:
    """Row absmax and E4M3 quantisation alone.  x: [M,K] bf16; sx_out: [M]
    fp32 out; xq_out: [M,K] uint8 out (same bits as rf_absmax_fp8_gemm)."""
    M, K = x.shape
    _need(x, torch.bfloat16, (M, K), "x")
    _need(sx_out, torch.float32, (M,), "sx_out")
    _need(xq_out, torch.uint8, (M, K), "xq_out")
    _check(lib.rf_absmax_quant_fp8(_ptr(x), M, K, _ptr(sx_out), _ptr(xq_out), _stream(stream)),
           "rf_absmax_quant_fp8")


def rf_selftest_wait_timeout(timeout_us: int, stream=None) -> None:
    _check(lib.rf_selftest_wait_timeout(int(timeout_us), _stream(stream)),
           "rf_selftest_wait_timeout")


def rf_selftest_bounds(stream=None) -> int:
    """Bounds-check self-test: in the debug build, one thread asks the bounds
    check about an index past a tensor's end (reported as
    RF_ERR_DEVICE_BOUNDS by rf_get_device_status, the access never made);
    returns the call's status (RF_ERR_UNSUPPORTED in the normal build)."""
    return lib.rf_selftest_bounds(_stream(stream))


def rf_selftest_decode_plan(B: int, Hkv: int, Lk: int, num_splits: int, sms: int) -> int:
    """Host-side check of the split-KV decode partition (no GPU needed):
    0 when it is consistent, -1 for a refused shape, else the number of the
    first failed check (see include/rf.h)."""
    return lib.rf_selftest_decode_plan(int(B), int(Hkv), int(Lk), int(num_splits), int(sms))


def rf_selftest_fp8_schedule(M: int, N: int, clusters: int) -> int:
    """Host-side check of the FP8 GEMM's tile schedule (no GPU needed): 0
    when every block of the M x N output is computed once by the pairs'
    tiles, -1 for refused sizes, else the number of the first failed check."""
    return lib.rf_selftest_fp8_schedule(int(M), int(N), int(clusters))


def rf_selftest_moe_plan(T: int, D: int, E: int, sms: int) -> int:
    """Host-side check of the MoE gate's tile plan (no GPU needed): 0 when it
    is consistent, -1 for refused sizes, else the number of the first failed
    check."""
    return lib.rf_selftest_moe_plan(int(T), int(D), int(E), int(sms))
