"""GPU parity: single-segment fused attention (fp32 SIMT and bf16 tcgen05)
against the fp64 three-pass oracle, through the C ABI."""
import math

import numpy as np
import pytest
import torch

import workloads as I
from oracle import attention as A
from tests.helpers import Guarded, assert_bf16_close, assert_f32_close, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rf():
    import cascaded_reductions_loop_gb300 as m
    assert torch.cuda.is_available()
    return m


def _run(rf, q, k, v, scale, causal=0):
    """One call with guard bytes around the (NaN-filled) output."""
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = Guarded(tuple(qd.shape), qd.dtype)
    rf.rf_attn_fwd(qd, kd, vd, o.t, scale, causal)
    assert rf.rf_get_device_status() == rf.RF_OK
    o.check("attention output")
    return o.t.cpu()


def test_tiny_fp32_workload(rf):
    s = I.TINY_ATTN
    q, k, v = I.attention_inputs(s)
    o = _run(rf, q, k, v, s.scale)
    assert_f32_close(o, A.attention(q, k, v, s.scale), "tiny fp32")


@pytest.mark.parametrize("shape", [(2, 3, 37, 101, 64), (1, 2, 5, 300, 128), (1, 1, 1, 1, 64),
                                   (1, 1, 33, 32, 64), (1, 1, 4, 1000, 64)])
def test_fp32_ragged(rf, shape):
    B, H, Lq, Lk, d = shape
    sh = I.AttnShape(B, H, H, Lq, Lk, d, "f32", seed=11 + Lk)
    q, k, v = I.attention_inputs(sh)
    o = _run(rf, q, k, v, sh.scale)
    assert_f32_close(o, A.attention(q, k, v, sh.scale), f"fp32 {shape}")


def test_bert_prefill_bf16_full(rf):
    s = I.BERT_PREFILL
    q, k, v = I.attention_inputs(s)
    o = _run(rf, q, k, v, s.scale)
    assert_bf16_close(o, A.attention(q, k, v, s.scale), "BERT prefill")


@pytest.mark.parametrize("shape", [(2, 3, 200, 333, 64), (1, 1, 1, 1, 64), (1, 2, 128, 128, 64),
                                   (1, 1, 129, 257, 64), (3, 1, 64, 1000, 64),
                                   (1, 1, 300, 5, 64)])
def test_bf16_ragged(rf, shape):
    B, H, Lq, Lk, d = shape
    sh = I.AttnShape(B, H, H, Lq, Lk, d, "bf16", seed=100 + Lq + Lk)
    q, k, v = I.attention_inputs(sh)
    o = _run(rf, q, k, v, sh.scale)
    assert_bf16_close(o, A.attention(q, k, v, sh.scale), f"bf16 {shape}")


def test_bf16_single_key_returns_v0(rf):
    sh = I.AttnShape(2, 2, 2, 130, 1, 64, "bf16", seed=7)
    q, k, v = I.attention_inputs(sh)
    o = _run(rf, q, k, v, sh.scale)
    ref = v.float().expand(-1, -1, 130, -1)
    np.testing.assert_array_equal(to64(o), to64(ref.to(torch.bfloat16)))


def test_bf16_large_scores_stay_finite(rf):
    """Scores of magnitude ~200 exercise the running-max rescale (a missing
    rescale overflows exp)."""
    sh = I.AttnShape(1, 2, 2, 128, 512, 64, "bf16", seed=9)
    q, k, v = I.attention_inputs(sh)
    q = (q.float() * 8).to(torch.bfloat16)
    o = _run(rf, q, k, v, 1.0 / math.sqrt(64))
    assert_bf16_close(o, A.attention(q, k, v, 1.0 / math.sqrt(64)), "large scores")


# ------------------------------------------------------------- causal mask
# Row i reads keys j <= i + (Lk - Lq); rows that read no key are zero.


@pytest.mark.parametrize("shape", [(1, 2, 64, 256, 64), (2, 1, 37, 37, 128), (1, 1, 50, 20, 64),
                                   (1, 1, 1, 1, 64), (1, 1, 33, 1000, 64)])
def test_fp32_causal(rf, shape):
    B, H, Lq, Lk, d = shape
    sh = I.AttnShape(B, H, H, Lq, Lk, d, "f32", seed=300 + Lq + Lk)
    q, k, v = I.attention_inputs(sh)
    o = _run(rf, q, k, v, sh.scale, causal=1)
    assert_f32_close(o, A.attention(q, k, v, sh.scale, causal=True), f"fp32 causal {shape}")
    if Lq > Lk:
        assert (o[:, :, :Lq - Lk] == 0).all()


def test_bert_prefill_bf16_causal(rf):
    s = I.BERT_PREFILL
    q, k, v = I.attention_inputs(s)
    o = _run(rf, q, k, v, s.scale, causal=1)
    assert_bf16_close(o, A.attention(q, k, v, s.scale, causal=True), "BERT prefill causal")


@pytest.mark.parametrize("shape", [(2, 3, 200, 333, 64), (1, 2, 300, 300, 64), (1, 1, 500, 130, 64),
                                   (1, 1, 129, 129, 64), (1, 1, 1, 700, 64), (3, 1, 640, 640, 64),
                                   (1, 1, 256, 1, 64)])
def test_bf16_causal_ragged(rf, shape):
    B, H, Lq, Lk, d = shape
    sh = I.AttnShape(B, H, H, Lq, Lk, d, "bf16", seed=400 + Lq + Lk)
    q, k, v = I.attention_inputs(sh)
    o = _run(rf, q, k, v, sh.scale, causal=1)
    assert_bf16_close(o, A.attention(q, k, v, sh.scale, causal=True), f"bf16 causal {shape}")
    if Lq > Lk:
        assert (o[:, :, :Lq - Lk].float() == 0).all()


def test_bf16_causal_last_row_equals_unmasked(rf):
    """The last query row reads every key: the causal kernel's last row
    matches the unmasked oracle, and the unmasked kernel (a different kernel,
    whose running maximum moves lazily) to within bf16 rounding."""
    sh = I.AttnShape(1, 4, 4, 384, 384, 64, "bf16", seed=77)
    q, k, v = I.attention_inputs(sh)
    oc = _run(rf, q, k, v, sh.scale, causal=1)
    on = _run(rf, q, k, v, sh.scale, causal=0)
    ref = A.attention(q, k, v, sh.scale)
    assert_bf16_close(oc[:, :, -1], ref[:, :, -1], "causal last row")
    assert_bf16_close(on[:, :, -1], ref[:, :, -1], "unmasked last row")
    assert np.abs(to64(oc[:, :, -1]) - to64(on[:, :, -1])).max() <= 4e-3


# ----------------------------------------- non-incremental (two-pass) mode
# Lk <= 256: exact row max over all keys first, then P and O, no rescale.


@pytest.mark.parametrize("shape,causal", [((2, 3, 200, 256, 64), 0), ((1, 2, 256, 256, 64), 1),
                                          ((1, 1, 129, 129, 64), 0), ((2, 1, 300, 100, 64), 1),
                                          ((1, 1, 1, 1, 64), 0), ((1, 2, 500, 130, 64), 1),
                                          ((4, 2, 128, 128, 64), 0), ((1, 1, 77, 200, 64), 1)])
def test_bf16_two_pass(rf, shape, causal):
    B, H, Lq, Lk, d = shape
    sh = I.AttnShape(B, H, H, Lq, Lk, d, "bf16", seed=500 + Lq + Lk + causal)
    q, k, v = I.attention_inputs(sh)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = Guarded(tuple(qd.shape), qd.dtype)
    rf.rf_attn_fwd_ex(qd, kd, vd, o.t, sh.scale, causal, rf.RF_ATTN_TWO_PASS)
    assert rf.rf_get_device_status() == rf.RF_OK
    o.check("two-pass output")
    assert_bf16_close(o.t.cpu(), A.attention(q, k, v, sh.scale, causal=bool(causal)),
                      f"two-pass {shape} causal={causal}")


def test_two_pass_short_workloads_and_mode_errors(rf):
    for sh in (I.SHORT_PREFILL_256, I.SHORT_PREFILL_128):
        q, k, v = I.attention_inputs(sh)
        for mode in (rf.RF_ATTN_INCREMENTAL, rf.RF_ATTN_TWO_PASS):
            o = Guarded(tuple(q.shape), q.dtype)
            rf.rf_attn_fwd_ex(q.cuda(), k.cuda(), v.cuda(), o.t, sh.scale, 0, mode)
            assert rf.rf_get_device_status() == rf.RF_OK
            o.check(f"mode {mode} output")
            assert_bf16_close(o.t.cpu(), A.attention(q, k, v, sh.scale), f"mode {mode}")
    x = torch.zeros(1, 1, 64, 64, device="cuda", dtype=torch.bfloat16)
    kk = torch.zeros(1, 1, 300, 64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(rf.RFError):                     # two-pass needs Lk <= 256
        rf.rf_attn_fwd_ex(x, kk, kk, x.clone(), 0.125, 0, rf.RF_ATTN_TWO_PASS)
    xf = torch.zeros(1, 1, 64, 64, device="cuda")
    with pytest.raises(rf.RFError):                     # and the bf16 path
        rf.rf_attn_fwd_ex(xf, xf, xf, xf.clone(), 0.125, 0, rf.RF_ATTN_TWO_PASS)
