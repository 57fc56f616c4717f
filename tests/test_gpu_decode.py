"""GPU parity: multi-segment split-KV decode attention (segment partial
states merged inside the same kernel) against the fp64 three-pass oracle,
through the C ABI."""
import pytest
import torch

import workloads as I
from oracle import attention as A
from tests.helpers import Guarded, assert_bf16_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rf():
    import cascaded_reductions_loop_gb300 as m
    assert torch.cuda.is_available()
    return m


def _run(rf, q, k, v, scale, num_splits=0):
    """One call with guard bytes around the output and the workspace."""
    B, Hq, d = q.shape
    Hkv, Lk = k.shape[1], k.shape[2]
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = Guarded((B, Hq, d), torch.bfloat16)
    nbytes = rf.rf_attn_decode_splitkv_workspace_size(B, Hq, Hkv, Lk, d, num_splits)
    assert nbytes > 0
    ws = Guarded((nbytes,), torch.uint8, fill=0xFF)                    # NaN-filled partials
    rf.rf_attn_decode_splitkv(qd, kd, vd, o.t, scale, ws.t, num_splits)
    assert rf.rf_get_device_status() == rf.RF_OK
    o.check("decode output")
    ws.check("decode workspace")
    return o.t.cpu()


@pytest.mark.parametrize("B,Hq,Hkv,Lk,splits", [
    (2, 8, 2, 300, 0), (2, 8, 2, 300, 1), (2, 8, 2, 300, 3), (2, 8, 2, 300, 7),
    (1, 4, 4, 77, 5), (1, 8, 4, 1000, 0), (3, 8, 1, 513, 2), (1, 32, 8, 1, 0),
    (1, 32, 8, 31, 1), (2, 16, 4, 4096, 16), (1, 4, 1, 300, 300), (5, 24, 3, 2049, 0),
    (1, 16, 2, 129, 4)])
def test_decode_small(rf, B, Hq, Hkv, Lk, splits):
    sh = I.AttnShape(B, Hq, Hkv, 1, Lk, 128, "bf16", seed=1000 + Lk + splits)
    q, k, v = I.decode_inputs(sh)
    o = _run(rf, q, k, v, sh.scale, splits)
    assert_bf16_close(o, A.decode_attention(q, k, v, sh.scale), f"decode {B},{Hq},{Hkv},{Lk},{splits}")


@pytest.mark.parametrize("B,Hq,Hkv,Lk", [
    (1, 8, 1, 20000), (1, 4, 4, 5000), (2, 32, 8, 70), (1, 16, 2, 40000), (3, 8, 8, 33)])
def test_decode_sequence_cut_by_many_ctas(rf, B, Hq, Hkv, Lk):
    """The automatic partition gives every CTA the same number of key chunks,
    so few, long sequences are each cut into many segments (one sequence of
    20000 keys: one per SM), merged by whichever CTA finishes last; and with
    fewer chunks than SMs each CTA gets one chunk."""
    sh = I.AttnShape(B, Hq, Hkv, 1, Lk, 128, "bf16", seed=2000 + Lk)
    q, k, v = I.decode_inputs(sh)
    assert rf.rf_attn_decode_splitkv_num_splits(B, Hq, Hkv, Lk, 128, 0) >= 1
    o = _run(rf, q, k, v, sh.scale)
    assert_bf16_close(o, A.decode_attention(q, k, v, sh.scale), f"decode {B},{Hq},{Hkv},{Lk}")


def test_decode_2k_full(rf):
    s = I.DECODE_2K
    q, k, v = I.decode_inputs(s)
    o = _run(rf, q, k, v, s.scale)
    assert_bf16_close(o, A.decode_attention(q, k, v, s.scale), "decode 2k")


def test_decode_32k_full(rf):
    """The 32768-key workload: every one of the 1024 (batch, head) rows."""
    s = I.DECODE_32K
    q, k, v = I.decode_inputs(s)
    o = _run(rf, q, k, v, s.scale)
    assert_bf16_close(o, A.decode_attention(q, k, v, s.scale), "decode 32k")


def test_segment_count_does_not_change_the_result_much(rf):
    """Any split merges to the same cascade: outputs for 1, 2 and 64
    segments agree to bf16 rounding."""
    sh = I.AttnShape(1, 8, 2, 1, 2048, 128, "bf16", seed=3)
    q, k, v = I.decode_inputs(sh)
    outs = [_run(rf, q, k, v, sh.scale, s).float() for s in (1, 2, 64)]
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() <= 8e-3


def test_workspace_reuse_gives_identical_results(rf):
    """Nothing carries over between calls through the workspace: calling
    twice with the same workspace (and once with a fresh one) gives the
    same bits."""
    sh = I.AttnShape(4, 32, 8, 1, 3000, 128, "bf16", seed=5)
    q, k, v = (t.cuda() for t in I.decode_inputs(sh))
    nbytes = rf.rf_attn_decode_splitkv_workspace_size(4, 32, 8, 3000, 128, 0)
    ws = torch.full((nbytes,), 0xFF, dtype=torch.uint8, device="cuda")
    outs = []
    for w in (ws, ws, torch.zeros_like(ws)):
        o = torch.full_like(q, float("nan"))
        rf.rf_attn_decode_splitkv(q, k, v, o, sh.scale, w, 0)
        outs.append(o)
    assert rf.rf_get_device_status() == rf.RF_OK
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
