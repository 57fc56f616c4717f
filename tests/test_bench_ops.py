"""The roofline arithmetic of bench.py (CPU only): each timed call's
algorithmic bytes and FLOPs, written out here from the workload shapes
independently of bench.py's own formulas, and the roofline time and bound
they give at the fallback peaks."""
import pytest

import bench
import workloads as I

MB = 1e6


def _ops():
    return {op.name: op for op in bench.make_ops() + bench.make_extra_ops()}


def test_step_calls_and_order():
    assert [op.name for op in bench.make_ops()] == [
        "decode_2k", "moe_gate", "fp8_gemm", "bert_prefill", "decode_32k"]


def test_decode_bytes_and_flops():
    ops = _ops()
    # K and V of 32 x 8 kv heads x Lk x 128 dims in bf16, plus Q and O
    for name, lk in (("decode_32k", 32768), ("decode_2k", 2048)):
        kv = 2 * 32 * 8 * lk * 128 * 2
        qo = 2 * 32 * 32 * 128 * 2
        assert ops[name].bytes == kv + qo
        assert ops[name].flops == 2 * 2 * 32 * 32 * lk * 128     # QK^T and PV, every query head
    assert ops["decode_32k"].bytes == pytest.approx(4295.5 * MB, rel=1e-3)


def test_prefill_and_gate_and_fp8():
    ops = _ops()
    assert ops["bert_prefill"].bytes == 4 * 8 * 16 * 512 * 64 * 2          # Q, K, V, O once
    assert ops["bert_prefill"].flops == 8.589934592e9
    causal_pairs = 512 * 513 // 2
    assert ops["bert_prefill_causal"].flops == 2 * 2 * 8 * 16 * causal_pairs * 64
    g = ops["moe_gate"]
    assert g.bytes == 8192 * 4096 * 2 + 64 * 4096 * 2 + 8192 * 2 * (4 + 4)
    assert g.flops == 2 * 8192 * 4096 * 64
    f = ops["fp8_gemm"]
    assert f.bytes == 4096 * 4096 * 2 + 4096 * 4096 + 4096 * 4 + 4096 * 4096 * 2
    assert f.flops == 2 * 4096 ** 3 and f.tc_dtype == "fp8"


def test_latent_decode_bytes_and_flops():
    s = I.MLA_DECODE
    op = _ops()["mla_decode"]
    # the cache once (576 bf16 per row), q in, O out
    assert op.bytes == s.B * s.Lk * 576 * 2 + s.B * s.Hq * 576 * 2 + s.B * s.Hq * 512 * 2
    assert op.bytes == pytest.approx(319.8 * MB, rel=1e-3)
    # scores over 576 dims and P.V over 512 for every (batch, head, row)
    assert op.flops == 2 * s.B * s.Hq * s.Lk * (576 + 512)


def test_roofline_time_and_bound_at_fallback_peaks():
    peaks = {"hbm_gbs": 6800.0, "bf16_tfs": 1900.0, "bf16_tfs_sustained": 1700.0,
             "source": "fallback"}
    ops = _ops()
    d = ops["decode_32k"]
    assert d.bound(peaks) == "hbm"
    assert d.roofline_s(peaks) == pytest.approx(d.bytes / 6.8e12)
    # tensor bounds use the burst peak (kernels run far under a second)
    p = ops["bert_prefill"]
    assert p.bound(peaks) == "hbm"                                  # 4.93 us of HBM vs 4.52 us of tensor
    assert p.roofline_s(peaks) == pytest.approx(p.bytes / 6.8e12)
    assert p.tensor_peak(peaks) == 1900.0
    f = ops["fp8_gemm"]
    assert f.bound(peaks) == "tensor"
    assert f.roofline_s(peaks) == pytest.approx(f.flops / 3.8e15)   # FP8 = 2 x bf16
    m = ops["mla_decode"]
    assert m.bound(peaks) == "hbm"                                  # 47 us of HBM vs 38 us of tensor


def test_workload_config_names_the_calls():
    step = bench.workload_config(bench.make_ops(), 1)
    assert step["workload"] == "decode2k+moe_gate+fp8_gemm+bert_prefill+decode32k"
    assert "exceed" not in step["l2"] and "> 129 MB L2" in step["l2"]
    mla = bench.workload_config([_ops()["mla_decode"]], 1)
    assert mla["workload"] == "mla_decode" and "mla" in mla and "decode" not in mla
