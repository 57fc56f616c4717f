"""GPU parity: row absmax -> E4M3 quantisation -> FP8 GEMM -> dequantisation
against the fp64 oracle, through the C ABI.  sx and the E4M3 bytes must
match bit for bit."""
import numpy as np
import pytest
import torch

from cascaded_reductions_loop_gb300 import inputs as I
from oracle import fp8_quant_gemm as F
from tests.helpers import assert_fp8_y_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rf():
    import cascaded_reductions_loop_gb300 as m
    assert torch.cuda.is_available()
    return m


def _run(rf, x, wq, sw, with_outputs=True):
    M, K = x.shape
    N = wq.shape[0]
    y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    sx = torch.full((M,), float("nan"), dtype=torch.float32, device="cuda") if with_outputs else None
    xq = torch.full((M, K), 0x7F, dtype=torch.uint8, device="cuda") if with_outputs else None
    ws = None
    if not with_outputs:
        ws = torch.empty(rf.rf_absmax_fp8_gemm_workspace_size(M, N, K), dtype=torch.uint8,
                         device="cuda")
    rf.rf_absmax_fp8_gemm(x.cuda(), wq.cuda(), sw.cuda(), y, sx_out=sx, xq_out=xq, workspace=ws)
    assert rf.rf_get_device_status() == rf.RF_OK
    return (y.cpu(), None if sx is None else sx.cpu().numpy(),
            None if xq is None else xq.cpu().numpy())


def test_fp8_full_size(rf):
    s = I.FP8_GEMM
    x, wq, sw = I.fp8_inputs(s)
    y, sx, xq = _run(rf, x, wq, sw)
    _, ref_sx = F.row_scale(x)
    np.testing.assert_array_equal(sx.view(np.uint32), ref_sx.view(np.uint32))
    ref_xq = F.quantise(x, ref_sx)
    bad = np.nonzero(xq != ref_xq)
    assert bad[0].size == 0, f"{bad[0].size} E4M3 bytes differ, first at {bad[0][:3]}, {bad[1][:3]}"
    rng = np.random.default_rng(1)
    rows = sorted(set(rng.integers(0, s.M, 40).tolist()) | {0, s.M - 1})
    _, _, ref_y = F.absmax_fp8_gemm(x, wq, sw, rows=rows)
    assert_fp8_y_close(y[rows], ref_y, "FP8 GEMM sampled rows")
    assert torch.isfinite(y.float()).all()


@pytest.mark.parametrize("M,N,K", [(200, 300, 272), (1, 16, 16), (130, 264, 4096),
                                   (257, 512, 384), (64, 1000, 5008)])
def test_fp8_ragged(rf, M, N, K):
    x, wq, sw = I.fp8_inputs(I.FP8Shape(M=M, N=N, K=K, seed=M + N + K))
    y, sx, xq = _run(rf, x, wq, sw)
    ref_sx, ref_xq, ref_y = F.absmax_fp8_gemm(x, wq, sw)
    np.testing.assert_array_equal(sx.view(np.uint32), ref_sx.view(np.uint32))
    np.testing.assert_array_equal(xq, ref_xq)
    assert_fp8_y_close(y, ref_y, f"FP8 {M}x{N}x{K}")


def test_fp8_workspace_path_matches(rf):
    x, wq, sw = I.fp8_inputs(I.FP8Shape(M=256, N=256, K=512, seed=4))
    y1, _, _ = _run(rf, x, wq, sw, with_outputs=True)
    y2, _, _ = _run(rf, x, wq, sw, with_outputs=False)
    assert torch.equal(y1, y2)


def test_fp8_zero_row_and_signed_zero(rf):
    """A zero row gives sx = 0 and codes 0x00; a value that rounds to zero
    keeps its sign (0x80)."""
    x, wq, sw = I.fp8_inputs(I.FP8Shape(M=64, N=32, K=64, seed=5))
    x = x.clone()
    x[3] = 0
    x[5, :] = 0
    x[5, 0] = 448.0
    x[5, 1] = -1e-4          # |x/sx| = 1e-4 < 2^-10: rounds to -0
    x[5, 2] = 1e-4
    y, sx, xq = _run(rf, x, wq, sw)
    assert sx[3] == 0 and (xq[3] == 0).all() and (y[3].float() == 0).all()
    assert xq[5, 1] == 0x80 and xq[5, 2] == 0x00 and xq[5, 0] == 0x7E
    ref_sx, ref_xq, ref_y = F.absmax_fp8_gemm(x, wq, sw)
    np.testing.assert_array_equal(xq, ref_xq)
    assert_fp8_y_close(y, ref_y, "zero rows")


def _domain_rows(a_lo, a_hi):
    """Rows of 4096 bf16 covering every pair (row max a, x) with |x| <= a for
    a's bit pattern in [a_lo, a_hi): element 0 is a, then 2047 magnitudes m
    (both signs) of block b of a's range, zeros where m > a."""
    a_list, b_list = [], []
    for a in range(a_lo, a_hi):
        nb = a // 2047 + 1
        a_list += [a] * nb
        b_list += range(nb)
    a_t = torch.tensor(a_list, dtype=torch.int32, device="cuda")[:, None]
    b_t = torch.tensor(b_list, dtype=torch.int32, device="cuda")[:, None]
    mag = b_t * 2047 + torch.arange(2047, dtype=torch.int32, device="cuda")[None, :]
    valid = mag <= a_t
    pos = torch.where(valid, mag, torch.zeros_like(mag))
    neg = torch.where(valid, mag | 0x8000, torch.zeros_like(mag))
    body = torch.stack([pos, neg], dim=2).reshape(len(a_list), 4094)
    bits = torch.cat([a_t, body, torch.zeros_like(a_t)], dim=1)          # 4096 columns
    return bits.to(torch.int16).view(torch.bfloat16).contiguous()


def test_quantisation_exhaustive_against_ieee_division(rf):
    """Every bf16 x against every positive finite bf16 row max a >= |x|: the
    kernel's codes equal E4M3(fp32(x / sx)) with an IEEE fp32 division (torch's
    CUDA division) and torch's float8_e4m3fn cast; sx = a / 448 likewise."""
    wq = torch.zeros(16, 4096, dtype=torch.uint8, device="cuda")
    sw = torch.ones(16, dtype=torch.float32, device="cuda")
    total = 0
    step = 2048
    for a_lo in range(1, 0x7F80, step):
        x = _domain_rows(a_lo, min(a_lo + step, 0x7F80))
        M = x.shape[0]
        y = torch.empty(M, 16, dtype=torch.bfloat16, device="cuda")
        sx = torch.empty(M, dtype=torch.float32, device="cuda")
        xq = torch.empty(M, 4096, dtype=torch.uint8, device="cuda")
        rf.rf_absmax_fp8_gemm(x, wq, sw, y, sx_out=sx, xq_out=xq)
        assert rf.rf_get_device_status() == rf.RF_OK
        # tensor / tensor: an IEEE division (dividing by a Python scalar would
        # multiply by its reciprocal instead)
        ref_sx = x[:, 0].float() / torch.full((M,), 448.0, device="cuda")
        assert torch.equal(sx.view(torch.int32), ref_sx.view(torch.int32))
        t = x.float() / ref_sx[:, None]
        ref = t.to(torch.float8_e4m3fn).view(torch.uint8)
        bad = (xq != ref).nonzero()
        assert bad.numel() == 0, f"{bad.shape[0]} codes differ, first (row, col) {bad[:3].tolist()}"
        total += M * 4095
    assert total > 1_000_000_000
