"""GPU parity: row absmax -> E4M3 quantisation -> FP8 GEMM -> dequantisation
against the fp64 oracle, through the C ABI.  sx and the E4M3 bytes must
match bit for bit; Y is compared element by element (all of it, at every
size, the full 4096^3 workload included).  The pre-quantised weight is made
by each side with its own quantiser and checked bit for bit too."""
import numpy as np
import pytest
import torch

import workloads as I
from oracle import fp8_quant_gemm as F
from tests.helpers import Guarded, assert_fp8_y_close, fp8_weight_gpu, fp8_weight_oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def rf():
    import cascaded_reductions_loop_gb300 as m
    assert torch.cuda.is_available()
    return m


def _weights(rf, w):
    """(device wq, device sw) from the library and (wq, sw) from the oracle,
    checked equal bit for bit."""
    wq_d, sw_d = fp8_weight_gpu(rf, w)
    wq_o, sw_o = fp8_weight_oracle(w)
    np.testing.assert_array_equal(sw_d.cpu().numpy().view(np.uint32), sw_o.view(np.uint32))
    bad = np.nonzero(wq_d.cpu().numpy() != wq_o)
    assert bad[0].size == 0, f"{bad[0].size} weight codes differ, first at {bad[0][:3]}, {bad[1][:3]}"
    return wq_d, sw_d, wq_o, sw_o


def _run(rf, x, wq, sw, with_outputs=True, y_shift=0):
    """Runs the fused call with guard bytes around every output; returns
    (Y, sx, xq) on the host (sx, xq None when kept in the workspace).  Y
    starts y_shift bytes past a 256-byte boundary."""
    M, K = x.shape
    N = wq.shape[0]
    y = Guarded((M, N), torch.bfloat16, shift=y_shift)
    sx = Guarded((M,), torch.float32) if with_outputs else None
    xq = Guarded((M, K), torch.uint8) if with_outputs else None
    need = rf.rf_absmax_fp8_gemm_workspace_size(M, N, K)
    ws = Guarded((need,), torch.uint8, fill=0x5A)
    rf.rf_absmax_fp8_gemm(x.cuda(), wq, sw, y.t, ws.t, sx_out=None if sx is None else sx.t,
                          xq_out=None if xq is None else xq.t)
    assert rf.rf_get_device_status() == rf.RF_OK
    for g, name in ((y, "Y"), (sx, "sx"), (xq, "xq"), (ws, "workspace")):
        if g is not None:
            g.check(name)
    return (y.t.cpu(), None if sx is None else sx.t.cpu().numpy(),
            None if xq is None else xq.t.cpu().numpy())


def _check_all(x, y, sx, xq, wq_o, sw_o, what):
    ref_sx, ref_xq, ref_y = F.absmax_fp8_gemm(x, wq_o, sw_o)
    np.testing.assert_array_equal(sx.view(np.uint32), ref_sx.view(np.uint32))
    bad = np.nonzero(xq != ref_xq)
    assert bad[0].size == 0, f"{what}: {bad[0].size} E4M3 bytes differ, first at {bad[0][:3]}, {bad[1][:3]}"
    assert_fp8_y_close(y, ref_y, what)


def test_fp8_full_size(rf):
    """The 4096^3 workload: every sx, every code and every element of Y."""
    s = I.FP8_GEMM
    x, w = I.fp8_inputs(s)
    wq_d, sw_d, wq_o, sw_o = _weights(rf, w)
    y, sx, xq = _run(rf, x, wq_d, sw_d)
    _check_all(x, y, sx, xq, wq_o, sw_o, "FP8 4096^3")


@pytest.mark.parametrize("M,N,K", [(200, 300, 272), (1, 16, 16), (130, 264, 4096),
                                   (257, 512, 384), (64, 1000, 5008), (700, 520, 1040),
                                   (4096, 256, 128), (300, 4096, 256),
                                   # 100 pair tiles: whole rounds of full tiles, then halves;
                                   # 64 pair tiles: all full (too many left for halves)
                                   (2560, 2560, 256), (1024, 4096, 384)])
def test_fp8_ragged(rf, M, N, K):
    x, w = I.fp8_inputs(I.FP8Shape(M=M, N=N, K=K, seed=M + N + K))
    wq_d, sw_d, wq_o, sw_o = _weights(rf, w)
    y, sx, xq = _run(rf, x, wq_d, sw_d)
    _check_all(x, y, sx, xq, wq_o, sw_o, f"FP8 {M}x{N}x{K}")


def test_fp8_workspace_path_matches(rf):
    """Codes and scales kept in the workspace give the same Y bits."""
    x, w = I.fp8_inputs(I.FP8Shape(M=600, N=512, K=512, seed=4))
    wq_d, sw_d, _, _ = _weights(rf, w)
    y1, _, _ = _run(rf, x, wq_d, sw_d, with_outputs=True)
    y2, _, _ = _run(rf, x, wq_d, sw_d, with_outputs=False)
    assert torch.equal(y1, y2)


def test_fp8_zero_row_and_signed_zero(rf):
    """A zero row gives sx = 0 and codes 0x00; a value that rounds to zero
    keeps its sign (0x80)."""
    x, w = I.fp8_inputs(I.FP8Shape(M=64, N=32, K=64, seed=5))
    x = x.clone()
    x[3] = 0
    x[5, :] = 0
    x[5, 0] = 448.0
    x[5, 1] = -1e-4          # |x/sx| = 1e-4 < 2^-10: rounds to -0
    x[5, 2] = 1e-4
    wq_d, sw_d, wq_o, sw_o = _weights(rf, w)
    y, sx, xq = _run(rf, x, wq_d, sw_d)
    assert sx[3] == 0 and (xq[3] == 0).all() and (y[3].float() == 0).all()
    assert xq[5, 1] == 0x80 and xq[5, 2] == 0x00 and xq[5, 0] == 0x7E
    _check_all(x, y, sx, xq, wq_o, sw_o, "zero rows")


def test_absmax_quant_standalone_matches_oracle(rf):
    """rf_absmax_quant_fp8 alone (the weight quantiser above) on ragged rows,
    short and longer than 4096 elements, with zero rows."""
    for (M, K) in ((1, 16), (333, 4096), (70, 4112), (5, 10000)):
        x, _ = I.fp8_inputs(I.FP8Shape(M=M, N=16, K=K, seed=M * 7 + K))
        x = x.clone()
        x[M // 2] = 0
        sx = Guarded((M,), torch.float32)
        xq = Guarded((M, K), torch.uint8)
        rf.rf_absmax_quant_fp8(x.cuda(), sx.t, xq.t)
        assert rf.rf_get_device_status() == rf.RF_OK
        sx.check("sx")
        xq.check("xq")
        _, ref_sx = F.row_scale(x)
        np.testing.assert_array_equal(sx.t.cpu().numpy().view(np.uint32), ref_sx.view(np.uint32))
        np.testing.assert_array_equal(xq.t.cpu().numpy(), F.quantise(x, ref_sx))


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


@pytest.mark.parametrize("fused", [False, True])
def test_quantisation_exhaustive_against_ieee_division(rf, fused):
    """Every bf16 x against every positive finite bf16 row max a >= |x|: the
    kernel's codes equal E4M3(fp32(x / sx)) with an IEEE fp32 division (torch's
    CUDA division) and torch's float8_e4m3fn cast; sx = a / 448 likewise.
    Run through the standalone quantiser and through the fused call."""
    wq = torch.zeros(16, 4096, dtype=torch.uint8, device="cuda")
    sw = torch.ones(16, dtype=torch.float32, device="cuda")
    total = 0
    step = 2048
    for a_lo in range(1, 0x7F80, step):
        x = _domain_rows(a_lo, min(a_lo + step, 0x7F80))
        M = x.shape[0]
        sx = torch.empty(M, dtype=torch.float32, device="cuda")
        xq = torch.empty(M, 4096, dtype=torch.uint8, device="cuda")
        if fused:
            y = torch.empty(M, 16, dtype=torch.bfloat16, device="cuda")
            ws = torch.empty(rf.rf_absmax_fp8_gemm_workspace_size(M, 16, 4096), dtype=torch.uint8,
                             device="cuda")
            rf.rf_absmax_fp8_gemm(x, wq, sw, y, ws, sx_out=sx, xq_out=xq)
        else:
            rf.rf_absmax_quant_fp8(x, sx, xq)
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


def test_fp8_y_16_byte_aligned(rf):
    """Y 16-byte but not 32-byte aligned: the epilogue stores 16-byte pieces
    instead of 32-byte ones; the bits are the same."""
    x, w = I.fp8_inputs(I.FP8Shape(M=300, N=512, K=256, seed=42))
    wq_d, sw_d, wq_o, sw_o = _weights(rf, w)
    y16, sx, xq = _run(rf, x, wq_d, sw_d, y_shift=16)
    y32, _, _ = _run(rf, x, wq_d, sw_d)
    _check_all(x, y16, sx, xq, wq_o, sw_o, "FP8 Y at a 16-byte offset")
    assert torch.equal(y16, y32)
