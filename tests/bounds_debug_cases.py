"""Ragged cases of every entry point, run against the bounds-checked debug
build of the library (librf_gb300_dbg.so, selected by RF_GB300_LIB=debug).

In that build every global load or store a kernel thread issues is checked
against its tensor; an access outside is skipped and reported through the
device error word as RF_ERR_DEVICE_BOUNDS.  Each case below must leave the
device status RF_OK and still match the oracle.  Run as a script (by
tests/test_gpu_bounds_debug.py, in a process of its own, since the library is
chosen when the package is imported); prints one line per case.
"""
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import workloads as I  # noqa: E402
from oracle import attention as A  # noqa: E402
from oracle import fp8_quant_gemm as F  # noqa: E402
from oracle import moe_gate as G  # noqa: E402
from tests.helpers import (MOE_W_ABS, assert_bf16_close, assert_f32_close,  # noqa: E402
                           assert_fp8_y_close, fp8_weight_gpu, fp8_weight_oracle)


def status_ok(rf, what):
    st = rf.rf_get_device_status()
    assert st == rf.RF_OK, f"{what}: device status {rf.rf_status_string(st)}"
    print(f"ok  {what}", flush=True)


def attention_cases(rf):
    sh = I.AttnShape(1, 2, 2, 64, 200, 64, "f32", seed=11)
    q, k, v = I.attention_inputs(sh)
    o = torch.full_like(q, float("nan")).cuda()
    rf.rf_attn_fwd(q.cuda(), k.cuda(), v.cuda(), o, sh.scale, 1)
    assert_f32_close(o.cpu(), A.attention(q, k, v, sh.scale, causal=True), "f32 causal")
    status_ok(rf, "attention fp32 causal 1x2x64x200")
    for (B, H, Lq, Lk, causal, mode) in [(2, 3, 200, 333, 0, rf.RF_ATTN_AUTO),
                                         (2, 2, 130, 200, 1, rf.RF_ATTN_AUTO),
                                         (1, 2, 100, 200, 0, rf.RF_ATTN_TWO_PASS)]:
        sh = I.AttnShape(B, H, H, Lq, Lk, 64, "bf16", seed=B + H + Lq + Lk)
        q, k, v = I.attention_inputs(sh)
        o = torch.full_like(q, float("nan")).cuda()
        rf.rf_attn_fwd_ex(q.cuda(), k.cuda(), v.cuda(), o, sh.scale, causal, mode)
        assert_bf16_close(o.cpu(), A.attention(q, k, v, sh.scale, causal=bool(causal)), "bf16")
        status_ok(rf, f"attention bf16 {B}x{H}x{Lq}x{Lk} causal={causal} mode={mode}")
    for dtype in ("bf16", "f32"):
        vs = I.VarlenShape(B=4, H=2, d=64, len_lo=1, len_hi=1, dtype=dtype, seed=12,
                           lens=(1, 130, 77, 300))
        q, k, v, cu = I.varlen_inputs(vs)
        o = torch.full_like(q, float("nan")).cuda()
        cud = cu.cuda()
        rf.rf_attn_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), o, cud, cud, 300, vs.scale, 1)
        ref = A.attention_varlen(q, k, v, cu, cu, vs.scale, causal=True)
        (assert_bf16_close if dtype == "bf16" else assert_f32_close)(o.cpu(), ref, "varlen")
        status_ok(rf, f"attention varlen {dtype} lens 1,130,77,300 causal")


def decode_cases(rf):
    for (B, Hq, Hkv, Lk, splits) in [(3, 8, 2, 1000, 0), (2, 16, 4, 777, 5), (1, 8, 1, 20000, 0),
                                     (2, 32, 8, 70, 0)]:
        sh = I.AttnShape(B, Hq, Hkv, 1, Lk, 128, "bf16", seed=B + Hq + Lk + splits)
        q, k, v = I.decode_inputs(sh)
        o = torch.full_like(q, float("nan")).cuda()
        n = rf.rf_attn_decode_splitkv_workspace_size(B, Hq, Hkv, Lk, 128, splits)
        ws = torch.full((n,), 0xFF, dtype=torch.uint8, device="cuda")
        rf.rf_attn_decode_splitkv(q.cuda(), k.cuda(), v.cuda(), o, sh.scale, ws, splits)
        assert_bf16_close(o.cpu(), A.decode_attention(q, k, v, sh.scale), "decode")
        status_ok(rf, f"decode {B}x{Hq}x{Hkv}x{Lk} splits={splits}")
        o2 = torch.full_like(q, float("nan")).cuda()
        rf.rf_attn_decode_splitkv_noalloc(q.cuda(), k.cuda(), v.cuda(), o2, sh.scale, splits)
        assert torch.equal(o, o2), "no-alloc entry point differs"
        status_ok(rf, f"decode no-alloc {B}x{Hq}x{Hkv}x{Lk} splits={splits}")


def mla_cases(rf):
    for (B, Hq, Lk, splits) in [(2, 128, 300, 1), (1, 100, 1000, 3), (2, 128, 65, 2)]:
        sh = I.MLAShape(B, Hq, Lk, seed=B + Hq + Lk)
        q, c = I.mla_inputs(sh)
        o = torch.full((B, Hq, 512), float("nan"), dtype=torch.bfloat16, device="cuda")
        n = rf.rf_mla_decode_workspace_size(B, Hq, Lk, 576, 512, splits)
        ws = torch.empty(max(n, 16), dtype=torch.uint8, device="cuda") if n else None
        rf.rf_mla_decode(q.cuda(), c.cuda(), o, sh.scale, ws, splits)
        assert_bf16_close(o.cpu(), A.mla_decode(q, c, sh.scale, 512), "mla")
        status_ok(rf, f"latent-KV decode {B}x{Hq}x{Lk} splits={splits}")


def moe_cases(rf):
    for (T, D, E, k, layout) in [(300, 256, 64, 2, rf.RF_GATE_W_ED), (129, 1024, 20, 4, rf.RF_GATE_W_ED),
                                 (513, 200, 256, 8, rf.RF_GATE_W_ED), (300, 256, 64, 2, rf.RF_GATE_W_DE),
                                 (129, 1024, 128, 4, rf.RF_GATE_W_DE)]:
        x, w = I.moe_inputs(I.MoEShape(T=T, D=D, E=E, k=k, seed=T + D + E + k))
        idx = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
        wts = torch.full((T, k), float("nan"), dtype=torch.float32, device="cuda")
        wg = w.t().contiguous() if layout == rf.RF_GATE_W_DE else w
        rf.rf_moe_gate_topk_softmax_ex(x.cuda(), wg.cuda(), k, layout, idx, wts)
        ref_idx, ref_w, _ = G.moe_gate(x, w, k)
        assert (idx.cpu().numpy() == ref_idx).all(), "MoE indices"
        assert np.abs(wts.cpu().numpy() - ref_w).max() <= MOE_W_ABS, "MoE weights"
        status_ok(rf, f"MoE gate {T}x{D}x{E} k={k} layout={layout}")


def fp8_cases(rf):
    for (M, N, K) in [(200, 300, 272), (257, 512, 384), (64, 1000, 5008), (1, 16, 16)]:
        x, w = I.fp8_inputs(I.FP8Shape(M=M, N=N, K=K, seed=M + N + K))
        wq_d, sw_d = fp8_weight_gpu(rf, w)
        wq_o, sw_o = fp8_weight_oracle(w)
        assert (wq_d.cpu().numpy() == wq_o).all(), "weight codes"
        ref_sx, ref_xq, ref_y = F.absmax_fp8_gemm(x, wq_o, sw_o)
        for keep in (True, False):
            y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
            sx = torch.empty(M, dtype=torch.float32, device="cuda") if keep else None
            xq = torch.empty(M, K, dtype=torch.uint8, device="cuda") if keep else None
            ws = torch.empty(rf.rf_absmax_fp8_gemm_workspace_size(M, N, K), dtype=torch.uint8,
                             device="cuda")
            rf.rf_absmax_fp8_gemm(x.cuda(), wq_d, sw_d, y, ws, sx_out=sx, xq_out=xq)
            assert_fp8_y_close(y.cpu(), ref_y, "FP8 Y")
            if keep:
                np.testing.assert_array_equal(sx.cpu().numpy().view(np.uint32), ref_sx.view(np.uint32))
                assert (xq.cpu().numpy() == ref_xq).all(), "E4M3 codes"
            status_ok(rf, f"FP8 {M}x{N}x{K} codes {'out' if keep else 'in workspace'}")


def main():
    import cascaded_reductions_loop_gb300 as rf
    assert rf.LIB_PATH.endswith("_dbg.so"), f"not the debug build: {rf.LIB_PATH}"
    assert torch.cuda.is_available()
    # the checker reports: an index past the end is caught (and never used)
    assert rf.rf_selftest_bounds() == rf.RF_OK
    assert rf.rf_get_device_status() == rf.RF_ERR_DEVICE_BOUNDS, "bounds self-test not reported"
    assert rf.rf_get_device_status() == rf.RF_OK, "error word not cleared"
    print("ok  bounds self-test reported RF_ERR_DEVICE_BOUNDS", flush=True)
    for cases in (attention_cases, decode_cases, mla_cases, moe_cases, fp8_cases):
        cases(rf)
    print("bounds-checked build: every case clean", flush=True)


if __name__ == "__main__":
    main()
