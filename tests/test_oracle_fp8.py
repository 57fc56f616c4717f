"""Pins for the FP8 quantised-GEMM oracle (CPU only): the E4M3 codec against
the format definition, a worked example and torch's float8_e4m3fn cast; the
scale against IEEE fp32 division done by numpy; the GEMM against exact int64
arithmetic."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import fp8_quant_gemm as F

ALL = np.arange(256, dtype=np.uint8)


def _torch_decode(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8).copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_golden_codes(golden_dir):
    d = json.load(open(os.path.join(golden_dir, "e4m3_codes.json")))
    for v, c in d["exact"]:
        assert F.e4m3_encode([v])[0] == c
        assert F.e4m3_decode([c])[0] == v
    for v, c in d["rounded"]:
        assert F.e4m3_encode([v])[0] == c


def test_decode_all_codes_definition_and_library():
    v = F.e4m3_decode(ALL)
    for c in range(256):
        s = -1.0 if c & 0x80 else 1.0
        e, m = (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            assert np.isnan(v[c])
        elif e == 0:
            assert v[c] == s * m * 2.0 ** -9
        else:
            assert v[c] == s * (1 + m / 8) * 2.0 ** (e - 7)
    t = _torch_decode(ALL)
    np.testing.assert_array_equal(np.isnan(v), np.isnan(t))
    ok = ~np.isnan(v)
    np.testing.assert_array_equal(v[ok], t[ok])
    assert np.nanmax(v) == 448.0


def test_roundtrip_all_codes():
    v = F.e4m3_decode(ALL)
    ok = ~np.isnan(v)
    np.testing.assert_array_equal(F.e4m3_encode(v[ok]), ALL[ok])   # includes +0 / -0


def test_midpoints_round_to_even():
    pos = np.array([c for c in range(0, 0x7F)], dtype=np.uint8)       # 0 .. 448, ascending
    v = F.e4m3_decode(pos)
    mids = (v[:-1] + v[1:]) / 2
    got = F.e4m3_encode(mids)
    even = np.where(pos[:-1] % 2 == 0, pos[:-1], pos[1:])
    np.testing.assert_array_equal(got, even)
    np.testing.assert_array_equal(F.e4m3_encode(-mids), even | 0x80)
    # just off the midpoint goes to the nearer code
    np.testing.assert_array_equal(F.e4m3_encode(np.nextafter(mids, 0)), pos[:-1])
    np.testing.assert_array_equal(F.e4m3_encode(np.nextafter(mids, 1e9)), pos[1:])


def test_saturation_and_specials():
    big = np.array([448.0, 449.0, 463.99, 464.0, 480.0, 1e6, np.inf])
    np.testing.assert_array_equal(F.e4m3_encode(big), 0x7E)
    np.testing.assert_array_equal(F.e4m3_encode(-big), 0xFE)
    assert F.e4m3_encode([np.nan])[0] == 0x7F
    assert F.e4m3_encode([-0.0])[0] == 0x80 and F.e4m3_encode([-1e-9])[0] == 0x80


def test_encode_matches_library_cast_in_range():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(200000) * 60,
                        rng.standard_normal(50000) * 0.01,
                        rng.uniform(-448, 448, 50000)]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(F.e4m3_encode(x.astype(np.float64)), ref)


def test_golden_gemm(golden_dir):
    d = json.load(open(os.path.join(golden_dir, "fp8_gemm_2x2.json")))
    sx, xq, Y = F.absmax_fp8_gemm(np.array(d["X"]), np.array(d["Wq"], np.uint8), np.array(d["sw"]))
    np.testing.assert_array_equal(sx, np.array(d["sx"], np.float32))
    np.testing.assert_array_equal(xq, d["xq"])
    np.testing.assert_array_equal(Y, d["Y"])


def _bf16_matrix(seed, M, K):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(M, K, generator=g)
    mask = torch.rand(M, K, generator=g) < 0.01
    return torch.where(mask, 20 * x, x).to(torch.bfloat16)


def test_scale_is_ieee_fp32_division():
    X = _bf16_matrix(1, 300, 257)
    a, sx = F.row_scale(X)
    Xf = X.float().numpy()
    np.testing.assert_array_equal(a, np.abs(Xf).max(axis=1).astype(np.float64))
    ref = np.abs(Xf).max(axis=1) / np.float32(448.0)            # numpy fp32 IEEE division
    assert ref.dtype == np.float32
    np.testing.assert_array_equal(sx, ref)


def test_quantise_matches_fp32_division_then_library_cast():
    X = _bf16_matrix(2, 256, 512)
    _, sx = F.row_scale(X)
    q = F.quantise(X, sx)
    t = X.float().numpy() / sx[:, None]                           # fp32 IEEE division
    # absmax / fp32(absmax / 448) may land a few ulp above 448: still below the
    # 464 midpoint, so the cast (non-saturating) and the oracle agree there
    assert t.dtype == np.float32 and np.abs(t).max() < 464.0
    ref = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(q, ref)
    # the absmax element of every row lands on +-448
    arg = np.abs(X.float().numpy()).argmax(axis=1)
    assert set(q[np.arange(256), arg].tolist()) <= {0x7E, 0xFE}


def test_zero_row():
    X = _bf16_matrix(3, 4, 64)
    X[2] = 0
    wq = torch.randint(0, 0x7E, (8, 64), dtype=torch.uint8)
    sx, xq, Y = F.absmax_fp8_gemm(X, wq, torch.ones(8))
    assert sx[2] == 0 and (xq[2] == 0).all() and (Y[2] == 0).all()


def test_gemm_exact_against_int64():
    rng = np.random.default_rng(3)
    M, N, K = 64, 48, 4096
    xq = rng.integers(0, 256, (M, K), dtype=np.uint8)
    wq = rng.integers(0, 256, (N, K), dtype=np.uint8)
    xq[(xq & 0x7F) == 0x7F] = 0x7E          # no NaN codes
    wq[(wq & 0x7F) == 0x7F] = 0x7E
    sx = np.ones(M, np.float32)
    sw = np.ones(N, np.float32)
    Y = F.gemm_dequant(xq, wq, sx, sw)
    # integer images: dec(c) * 2^9 is an integer for every finite code
    xi = (F.e4m3_decode(xq) * 512).astype(np.int64)
    wi = (F.e4m3_decode(wq) * 512).astype(np.int64)
    exact = xi @ wi.T                         # int64, no rounding
    np.testing.assert_array_equal(Y * 2.0 ** 18, exact.astype(np.float64))
    # a transposed operand would not match
    assert not np.array_equal(F.gemm_dequant(xq, wq[::-1], sx, sw), Y)


def test_scales_multiply_per_row_and_column():
    rng = np.random.default_rng(4)
    xq = rng.integers(0, 0x7E, (5, 32), dtype=np.uint8)
    wq = rng.integers(0, 0x7E, (3, 32), dtype=np.uint8)
    sx = np.array([1, 2, 4, 0.5, 0.25], np.float32)
    sw = np.array([1, 8, 0.125], np.float32)
    base = F.gemm_dequant(xq, wq, np.ones(5, np.float32), np.ones(3, np.float32))
    np.testing.assert_array_equal(F.gemm_dequant(xq, wq, sx, sw), base * sx[:, None] * sw[None, :])
