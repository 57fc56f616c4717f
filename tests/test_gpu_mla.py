"""GPU parity: latent-KV (multi-latent attention) decode -- the two-CTA
kernel that exchanges partial scores, and the segment merge -- against the
fp64 oracle, through the C ABI."""
import pytest
import torch

import workloads as I
from oracle import attention as A
from tests.helpers import Guarded, assert_bf16_close, assert_bf16_close_scaled

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rf():
    import cascaded_reductions_loop_gb300 as m
    assert torch.cuda.is_available()
    return m


def _run(rf, q, ckv, scale, num_splits=0, shift=0):
    """One call with guard bytes around the output and the workspace (both
    starting `shift` bytes past a 256-byte boundary)."""
    B, Hq, _ = q.shape
    Lk = ckv.shape[1]
    qd, cd = q.cuda(), ckv.cuda()
    o = Guarded((B, Hq, 512), torch.bfloat16, shift=shift)
    nbytes = rf.rf_mla_decode_workspace_size(B, Hq, Lk, 576, 512, num_splits)
    ws = Guarded((nbytes,), torch.uint8, fill=0xFF, shift=shift) if nbytes else None
    rf.rf_mla_decode(qd, cd, o.t, scale, None if ws is None else ws.t, num_splits)
    assert rf.rf_get_device_status() == rf.RF_OK
    o.check("mla output")
    if ws is not None:
        ws.check("mla workspace")
    return o.t.cpu()


@pytest.mark.parametrize("B,Hq,Lk,splits", [
    (2, 128, 100, 1), (2, 128, 100, 2), (2, 128, 100, 4), (1, 128, 1, 0), (1, 128, 31, 1),
    (1, 128, 32, 1), (1, 128, 33, 2), (3, 16, 257, 0), (2, 1, 64, 1), (1, 100, 1000, 3),
    (1, 128, 2048, 0), (2, 128, 4096, 5), (4, 64, 700, 0), (1, 128, 63, 1), (1, 128, 65, 2),
    (2, 128, 129, 3), (1, 128, 192, 3)])
def test_mla_small(rf, B, Hq, Lk, splits):
    sh = I.MLAShape(B, Hq, Lk, seed=2000 + Lk + splits)
    q, c = I.mla_inputs(sh)
    o = _run(rf, q, c, sh.scale, splits)
    assert_bf16_close(o, A.mla_decode(q, c, sh.scale, 512), f"mla {B},{Hq},{Lk},{splits}")


@pytest.mark.parametrize("rising", [True, False])
def test_mla_reference_maximum_moves(rf, rising):
    """Cache rows scaled by a ramp: with a rising ramp the running maximum
    grows by many times the lazy threshold across the tiles (O and l are
    rescaled in place several times); with a falling one it never moves."""
    sh = I.MLAShape(2, 128, 1024, seed=31)
    q, c = I.mla_inputs(sh)
    ramp = torch.linspace(0.2, 3.0, 1024)
    if not rising:
        ramp = ramp.flip(0)
    c = (c.float() * ramp[None, :, None]).to(torch.bfloat16)
    ref = A.mla_decode(q, c, sh.scale, 512)                  # |O| up to ~3x the unscaled case
    for splits in (1, 3):
        o = _run(rf, q, c, sh.scale, splits)
        assert_bf16_close_scaled(o, ref, f"ramp {rising} {splits}")


def test_mla_one_dominant_row_late(rf):
    """A single cache row far above all others in the last tile: every
    earlier contribution is scaled down to nothing and O is that row."""
    sh = I.MLAShape(1, 128, 300, seed=32)
    q, c = I.mla_inputs(sh)
    c = c.float() * 0.05
    c[0, 290] = q[0, 0].float() * 0.5            # head 0: ~30 (log2) above the rest
    c = c.to(torch.bfloat16)
    o = _run(rf, q, c, sh.scale, 1)
    assert_bf16_close(o, A.mla_decode(q, c, sh.scale, 512), "dominant row")


def test_mla_decode_full(rf):
    """The full workload in the launch configuration the benchmark times
    (automatic segment count): every (batch, head) row."""
    s = I.MLA_DECODE
    q, c = I.mla_inputs(s)
    o = _run(rf, q, c, s.scale)
    assert_bf16_close(o, A.mla_decode(q, c, s.scale, 512), "mla full")


def test_mla_long_context_split(rf):
    """Few batches over a long cache: the automatic choice cuts every batch
    into several segments, merged by the second kernel; every row checked."""
    s = I.MLAShape(B=8, Hq=128, Lk=32768, seed=33)
    assert rf.rf_mla_decode_num_splits(s.B, s.Hq, s.Lk, 576, 512, 0) > 1
    q, c = I.mla_inputs(s)
    o = _run(rf, q, c, s.scale)
    assert_bf16_close(o, A.mla_decode(q, c, s.scale, 512), "mla long")


def test_mla_repeatable(rf):
    """Repeated calls give identical bits (no order-dependent reduction)."""
    sh = I.MLAShape(3, 128, 777, seed=34)
    q, c = I.mla_inputs(sh)
    outs = [_run(rf, q, c, sh.scale, sp) for sp in (2, 2, 2)]
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


@pytest.mark.parametrize("splits", [1, 3])
def test_mla_outputs_16_byte_aligned(rf, splits):
    """O and the workspace 16-byte but not 32-byte aligned (the documented
    minimum alignment): the result is the same as with aligned buffers."""
    sh = I.MLAShape(2, 128, 300, seed=41)
    q, c = I.mla_inputs(sh)
    ref = A.mla_decode(q, c, sh.scale, 512)
    o16 = _run(rf, q, c, sh.scale, splits, shift=16)
    o32 = _run(rf, q, c, sh.scale, splits)
    assert_bf16_close(o16, ref, "mla, 16-byte aligned outputs")
    assert torch.equal(o16, o32)
