"""The C-ABI library builds, loads and exports every function include/rf.h
declares; host-side argument validation rejects bad calls before any CUDA
work (these calls need no GPU)."""
import ctypes
import os
import re

import pytest

import __graft_entry__

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_build = __graft_entry__._load_build_module()


@pytest.fixture(scope="module")
def rf():
    _build.build()
    import cascaded_reductions_loop_gb300 as m
    return m


def _declared():
    text = open(os.path.join(ROOT, "include", "rf.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rf_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("rf_attn_fwd", "rf_attn_decode_splitkv", "rf_mla_decode", "rf_moe_gate_topk_softmax",
              "rf_absmax_fp8_gemm", "rf_status_string", "rf_get_device_status"):
        assert n in names


def test_library_exports_every_declared_symbol(rf):
    lib = ctypes.CDLL(_build.LIB_PATH)
    for n in _declared():
        assert hasattr(lib, n), f"{n} declared in rf.h but not exported"
        assert hasattr(rf, n), f"{n} has no Python binding"


def test_debug_build_exports_the_same_symbols(rf):
    """The bounds-checked debug build is built beside the library and
    exports the same boundary."""
    lib = ctypes.CDLL(_build.DEBUG_LIB_PATH)
    for n in _declared():
        assert hasattr(lib, n), f"{n} not exported by the debug build"


def test_bounds_selftest_only_in_debug_build(rf):
    # the normal build returns before any CUDA call
    assert rf.lib.rf_selftest_bounds(None) == rf.RF_ERR_UNSUPPORTED


def test_status_strings(rf):
    assert rf.rf_status_string(0) == "RF_OK"
    for s in range(1, 9):
        assert rf.rf_status_string(s).startswith("RF_ERR_")
    assert "aligned" in rf.rf_status_string(rf.RF_ERR_DEVICE_LAYOUT)
    assert "unknown" in rf.rf_status_string(99)
    assert rf.rf_version() >= 10000


def test_validation_rejects_bad_arguments_without_a_gpu(rf):
    L = rf.lib
    p = ctypes.c_void_p(1 << 20)        # 16-byte aligned, never dereferenced
    mis = ctypes.c_void_p((1 << 20) + 4)
    null = None
    # attention: null / misaligned pointers, bad sizes, causal, dtype, scale
    assert L.rf_attn_fwd(1, null, p, p, p, 1, 1, 64, 64, 64, 0.125, 0, None) == rf.RF_ERR_INVALID_ARG
    assert L.rf_attn_fwd(1, mis, p, p, p, 1, 1, 64, 64, 64, 0.125, 0, None) == rf.RF_ERR_INVALID_ARG
    assert L.rf_attn_fwd(1, p, p, p, p, 0, 1, 64, 64, 64, 0.125, 0, None) == rf.RF_ERR_INVALID_ARG
    assert L.rf_attn_fwd(1, p, p, p, p, 1, 1, 64, 64, 64, 0.125, 2, None) == rf.RF_ERR_INVALID_ARG
    assert L.rf_attn_fwd(1, p, p, p, p, 1, 1, 64, 64, 64, 0.125, -1, None) == rf.RF_ERR_INVALID_ARG
    assert L.rf_attn_fwd(7, p, p, p, p, 1, 1, 64, 64, 64, 0.125, 0, None) == rf.RF_ERR_INVALID_ARG
    assert L.rf_attn_fwd(1, p, p, p, p, 1, 1, 64, 64, 64, -1.0, 0, None) == rf.RF_ERR_INVALID_ARG
    assert L.rf_attn_fwd(1, p, p, p, p, 1, 1, 64, 64, 96, 0.125, 0, None) == rf.RF_ERR_UNSUPPORTED
    assert L.rf_attn_fwd(0, p, p, p, p, 1, 1, 64, 64, 48, 0.125, 0, None) == rf.RF_ERR_UNSUPPORTED
    # fp32: B * H is the grid's y extent (at most 65535)
    assert L.rf_attn_fwd(0, p, p, p, p, 256, 256, 1, 1, 64, 0.125, 0, None) == rf.RF_ERR_INVALID_ARG
    # explicit evaluation order: unknown mode, two-pass beyond 256 keys or in fp32
    X = L.rf_attn_fwd_ex
    assert X(1, p, p, p, p, 1, 1, 64, 64, 64, 0.125, 0, 3, None) == rf.RF_ERR_INVALID_ARG
    assert X(1, p, p, p, p, 1, 1, 64, 257, 64, 0.125, 0, 2, None) == rf.RF_ERR_UNSUPPORTED
    assert X(0, p, p, p, p, 1, 1, 64, 64, 64, 0.125, 0, 2, None) == rf.RF_ERR_UNSUPPORTED
    # varlen attention: missing cumulative lengths, bad totals, causal, head dim
    V = L.rf_attn_fwd_varlen
    assert V(1, p, p, p, p, null, p, 2, 4, 64, 100, 100, 64, 0.125, 0, None) == rf.RF_ERR_INVALID_ARG
    assert V(1, p, p, p, p, p, p, 2, 4, 64, 0, 100, 64, 0.125, 0, None) == rf.RF_ERR_INVALID_ARG
    assert V(1, p, p, p, p, p, p, 2, 4, 0, 100, 100, 64, 0.125, 0, None) == rf.RF_ERR_INVALID_ARG
    assert V(1, p, p, p, p, p, p, 2, 4, 64, 100, 100, 64, 0.125, 3, None) == rf.RF_ERR_INVALID_ARG
    assert V(1, p, p, p, p, p, p, 2, 4, 64, 100, 100, 128, 0.125, 0, None) == rf.RF_ERR_UNSUPPORTED
    assert V(0, p, p, p, p, p, p, 2, 4, 64, 100, 100, 96, 0.125, 0, None) == rf.RF_ERR_UNSUPPORTED
    # decode: Hq not a multiple of Hkv, unsupported group / head dim, too many splits
    assert L.rf_attn_decode_splitkv(p, p, p, p, 1, 6, 4, 64, 128, 0.1, 0, p, 1 << 20, None) == rf.RF_ERR_INVALID_ARG
    assert L.rf_attn_decode_splitkv(p, p, p, p, 1, 12, 4, 64, 128, 0.1, 0, p, 1 << 20, None) == rf.RF_ERR_UNSUPPORTED
    assert L.rf_attn_decode_splitkv(p, p, p, p, 1, 8, 2, 64, 64, 0.1, 0, p, 1 << 20, None) == rf.RF_ERR_UNSUPPORTED
    assert L.rf_attn_decode_splitkv(p, p, p, p, 1, 8, 2, 64, 128, 0.1, 65, p, 1 << 20, None) == rf.RF_ERR_INVALID_ARG
    # an explicit split count needs no device: a too-small workspace is caught on the host
    assert L.rf_attn_decode_splitkv(p, p, p, p, 1, 8, 2, 64, 128, 0.1, 4, p, 16, None) == rf.RF_ERR_WORKSPACE
    assert L.rf_attn_decode_splitkv(p, p, p, p, 1, 8, 2, 64, 128, 0.1, 4, null, 1 << 20, None) == rf.RF_ERR_WORKSPACE
    # ticket counter per (batch, kv head) padded to 256 bytes, then one (m, l, o)
    # partial state per (batch, query head, segment): o padded to 256 bytes, then (m, l)
    P, G, S = 2 * 2, 8 // 2, 4
    assert rf.rf_attn_decode_splitkv_workspace_size(2, 8, 2, 64, 128, S) == \
        256 + P * S * G * 128 * 4 + P * S * G * 2 * 4
    assert rf.rf_attn_decode_splitkv_num_splits(1, 6, 4, 64, 128, 0) == 0
    # latent-KV decode: sizes, head count, latent widths, workspace of a split request
    M = L.rf_mla_decode
    assert M(null, p, p, 2, 128, 100, 576, 512, 0.1, 1, null, 0, None) == rf.RF_ERR_INVALID_ARG
    assert M(p, mis, p, 2, 128, 100, 576, 512, 0.1, 1, null, 0, None) == rf.RF_ERR_INVALID_ARG
    assert M(p, p, p, 0, 128, 100, 576, 512, 0.1, 1, null, 0, None) == rf.RF_ERR_INVALID_ARG
    assert M(p, p, p, 2, 128, 0, 576, 512, 0.1, 1, null, 0, None) == rf.RF_ERR_INVALID_ARG
    assert M(p, p, p, 2, 128, 100, 576, 512, 0.0, 1, null, 0, None) == rf.RF_ERR_INVALID_ARG
    assert M(p, p, p, 2, 128, 100, 576, 512, 0.1, -1, null, 0, None) == rf.RF_ERR_INVALID_ARG
    assert M(p, p, p, 2, 129, 100, 576, 512, 0.1, 1, null, 0, None) == rf.RF_ERR_UNSUPPORTED
    assert M(p, p, p, 2, 128, 100, 192, 128, 0.1, 1, null, 0, None) == rf.RF_ERR_UNSUPPORTED
    assert M(p, p, p, 2, 128, 100, 576, 512, 0.1, 2, null, 0, None) == rf.RF_ERR_WORKSPACE
    assert M(p, p, p, 2, 128, 100, 576, 512, 0.1, 2, p, 1024, None) == rf.RF_ERR_WORKSPACE
    # segments hold whole 64-row tiles: 300 rows = 5 tiles; a request of 3
    # gives segments of 2 tiles and so 3 segments, of 4 also 3, of 9 five
    assert rf.rf_mla_decode_num_splits(2, 128, 300, 576, 512, 3) == 3
    assert rf.rf_mla_decode_num_splits(2, 128, 300, 576, 512, 4) == 3
    assert rf.rf_mla_decode_num_splits(2, 128, 300, 576, 512, 9) == 5
    assert rf.rf_mla_decode_num_splits(2, 128, 100, 576, 512, 9) == 2
    assert rf.rf_mla_decode_num_splits(2, 128, 100, 576, 512, 1) == 1
    assert rf.rf_mla_decode_workspace_size(2, 128, 100, 576, 512, 1) == 0
    n = 2 * 128 * 2
    assert rf.rf_mla_decode_workspace_size(2, 128, 100, 576, 512, 2) == n * 512 * 4 + n * 2 * 4
    assert rf.rf_mla_decode_num_splits(2, 129, 100, 576, 512, 1) == 0
    # MoE: D not a multiple of 8, k out of range, E not covered
    assert L.rf_moe_gate_topk_softmax(p, p, 16, 100, 64, 2, p, p, None) == rf.RF_ERR_INVALID_ARG
    assert L.rf_moe_gate_topk_softmax(p, p, 16, 128, 64, 0, p, p, None) == rf.RF_ERR_INVALID_ARG
    assert L.rf_moe_gate_topk_softmax(p, p, 16, 128, 257, 2, p, p, None) == rf.RF_ERR_UNSUPPORTED
    assert L.rf_moe_gate_topk_softmax(p, p, 16, 128, 4, 5, p, p, None) == rf.RF_ERR_INVALID_ARG
    assert L.rf_moe_gate_topk_softmax(p, p, 16, 128, 64, 9, p, p, None) == rf.RF_ERR_UNSUPPORTED
    assert L.rf_moe_gate_topk_softmax(p, p, 65535 * 120 + 1, 128, 64, 2, p, p, None) == \
        rf.RF_ERR_UNSUPPORTED
    # W_gate layout: an unknown layout, and [D][E] with E not a multiple of 64
    Mx = L.rf_moe_gate_topk_softmax_ex
    assert Mx(p, p, 16, 128, 64, 2, 2, p, p, None) == rf.RF_ERR_INVALID_ARG
    assert Mx(p, p, 16, 128, 20, 2, rf.RF_GATE_W_DE, p, p, None) == rf.RF_ERR_UNSUPPORTED
    assert Mx(p, p, 16, 128, 320, 2, rf.RF_GATE_W_DE, p, p, None) == rf.RF_ERR_UNSUPPORTED
    assert Mx(p, p, 16, 100, 64, 2, rf.RF_GATE_W_DE, p, p, None) == rf.RF_ERR_INVALID_ARG
    # FP8: K not a multiple of 16, missing workspace
    assert L.rf_absmax_fp8_gemm(p, p, p, p, 16, 16, 40, p, p, null, 0, None) == rf.RF_ERR_INVALID_ARG
    assert L.rf_absmax_fp8_gemm(p, p, p, p, 16, 16, 64, null, null, null, 0, None) == rf.RF_ERR_WORKSPACE
    # the workspace is always needed (row counters), even with both outputs given
    assert L.rf_absmax_fp8_gemm(p, p, p, p, 16, 16, 64, p, p, null, 0, None) == rf.RF_ERR_WORKSPACE
    assert L.rf_absmax_fp8_gemm(p, p, p, p, 16, 16, 64, p, p, p, 255, None) == rf.RF_ERR_WORKSPACE
    # counters (1 + ceil(16 / 128) words, padded to 256) + codes (padded to 256) + scales
    assert rf.rf_absmax_fp8_gemm_workspace_size(16, 16, 64) == 256 + 1024 + 16 * 4
    assert rf.rf_absmax_fp8_gemm_workspace_size(300, 16, 64) == 256 + 19200 + 300 * 4
    # standalone quantiser: K not a multiple of 16, null outputs
    assert L.rf_absmax_quant_fp8(p, 16, 40, p, p, None) == rf.RF_ERR_INVALID_ARG
    assert L.rf_absmax_quant_fp8(p, 16, 64, null, p, None) == rf.RF_ERR_INVALID_ARG
    assert L.rf_absmax_quant_fp8(p, 0, 64, p, p, None) == rf.RF_ERR_INVALID_ARG
    assert rf.rf_absmax_fp8_gemm_workspace_size(16, 16, 40) == 0
    # self-test: out-of-range limit
    assert L.rf_selftest_wait_timeout(0, None) == rf.RF_ERR_INVALID_ARG


def test_every_declaration_is_documented():
    """Each function of the boundary is preceded by its comment block (what
    it computes, argument meaning and layout, ownership, errors)."""
    text = open(os.path.join(ROOT, "include", "rf.h")).read()
    decls = re.finditer(r"^(?:rf_status|int|size_t|const char\*)\s+(rf_[a-z0-9_]+)\s*\(",
                        text, flags=re.M)
    undocumented = [m.group(1) for m in decls if not text[:m.start()].rstrip().endswith("*/")]
    assert not undocumented, undocumented
