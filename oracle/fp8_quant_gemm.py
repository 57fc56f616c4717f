"""Oracle: the dynamic FP8 quantised GEMM cascade, pass by pass.

Test infrastructure only (see the package docstring for who may import it).

The cascade ([E] §4.3):

    scale   = max(abs(X)) / quant_max        (a max reduction)
    quant_X = round(X / scale)               (depends on that max)
    Y       = quant_X @ W                    (a sum reduction over K)

Readings where the article is silent or loose:

* the max is taken per row of X (one scale sx[m] per token row) and
  quant_max = 448, the largest finite E4M3 value [OCP];
* sx[m] = fp32(absmax[m] / 448), and the quotient X / sx is the correctly
  rounded fp32 quotient (one IEEE division);
* "round" is round-to-nearest-even onto the E4M3 grid [OCP] with saturation
  to +-448 (values beyond the largest finite code clamp to it); a value
  that rounds to zero keeps its sign (-0 is code 0x80);
* a row whose absmax is 0 gets sx = 0 and all-zero codes (0x00);
* W arrives pre-quantised: Wq [N][K] E4M3 codes with one fp32 scale sw[n]
  per output column, and Y = (Xq @ Wq^T) * sx[m] * sw[n].

Exactness notes.  Every E4M3 value is an integer multiple of 2^-9 with
magnitude <= 448 < 2^9, so each product dec(q) * dec(w) is a multiple of
2^-18 below 2^18 and a sum of K = 4096 of them stays below 2^30: in units of
2^-18 that is below 2^48 < 2^53, so the fp64 GEMM below is exact whatever
order the library sums in.  For the fp32 quotient, a fp64 quotient of two
fp32 numbers rounded once more to fp32 equals the correctly rounded fp32
quotient (53 >= 2*24 + 2).
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0
E4M3_MIN_NORMAL = 2.0 ** -6
E4M3_SUBNORMAL_STEP = 2.0 ** -9


def _f64(t) -> np.ndarray:
    if hasattr(t, "detach"):
        import torch

        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def _u8(t) -> np.ndarray:
    if hasattr(t, "detach"):
        import torch

        return t.detach().to("cpu").view(torch.uint8).numpy()
    return np.asarray(t, dtype=np.uint8)


# ------------------------------------------------------------- E4M3 codec


def e4m3_decode(codes) -> np.ndarray:
    """Value of each E4M3 code [OCP]: sign bit 7, exponent bits 6..3 (bias
    7), mantissa bits 2..0; exponent 0 encodes subnormals m * 2^-9; S.1111.111
    is NaN (the format has no infinities)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * E4M3_SUBNORMAL_STEP,
                   (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


def e4m3_encode(x) -> np.ndarray:
    """Round-to-nearest-even onto the E4M3 grid with saturation to +-448.

    For |x| >= 2^-6 the grid spacing in the binade [2^e, 2^(e+1)) is 2^(e-3)
    (three mantissa bits); below 2^-6 it is the subnormal step 2^-9.  The
    scaled value |x| / spacing is exact (a power-of-two scaling), so rint
    (ties to even) performs the rounding.  NaN maps to 0x7F.
    """
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    neg = np.signbit(x)
    nan = np.isnan(x)
    a = np.where(nan, 0.0, a)
    a = np.minimum(a, 1e30)                     # inf -> large, saturates below
    _, ex = np.frexp(a)                         # a = f * 2^ex, f in [0.5, 1)
    e = ex.astype(np.int64) - 1                 # a in [2^e, 2^(e+1))
    spacing = np.where(a < E4M3_MIN_NORMAL, E4M3_SUBNORMAL_STEP,
                       np.exp2((e - 3).astype(np.float64)))
    r = np.rint(a / spacing) * spacing          # RNE onto the grid
    r = np.minimum(r, E4M3_MAX)                 # satfinite
    # encode the (now representable) magnitude r
    _, er = np.frexp(r)
    er = er.astype(np.int64) - 1
    sub = r < E4M3_MIN_NORMAL
    code_sub = np.rint(r / E4M3_SUBNORMAL_STEP).astype(np.int64)
    mant = np.rint((r / np.exp2(er.astype(np.float64)) - 1.0) * 8.0).astype(np.int64)
    code_norm = ((er + 7) << 3) | mant
    code = np.where(sub, code_sub, code_norm)
    code = np.where(neg, code | 0x80, code)
    code = np.where(nan, 0x7F, code)
    return code.astype(np.uint8)


# ------------------------------------------------------------ the cascade


def row_scale(X) -> tuple[np.ndarray, np.ndarray]:
    """Pass 1: absmax[m] = max_k |X[m,k]| (exact) and
    sx[m] = fp32(absmax[m] / 448).  Returns (absmax fp64, sx fp32)."""
    X = _f64(X)
    a = np.abs(X).max(axis=1)
    sx = (a / E4M3_MAX).astype(np.float32)
    return a, sx


def quantise(X, sx: np.ndarray) -> np.ndarray:
    """Pass 2: q[m,k] = E4M3_RNE_sat(fp32(X[m,k] / sx[m])); rows with
    sx = 0 quantise to 0x00."""
    X = _f64(X)
    s = np.asarray(sx, dtype=np.float32).astype(np.float64)[:, None]
    zero = s == 0.0
    t = np.where(zero, 0.0, X / np.where(zero, 1.0, s)).astype(np.float32)
    q = e4m3_encode(t.astype(np.float64))
    return np.where(zero, np.uint8(0), q).astype(np.uint8)


def gemm_dequant(xq: np.ndarray, wq, sx: np.ndarray, sw) -> np.ndarray:
    """Pass 3: Y[m,n] = (sum_k dec(xq[m,k]) dec(wq[n,k])) * sx[m] * sw[n],
    in fp64 (the sum is exact, see the module docstring)."""
    A = e4m3_decode(xq)
    Bm = e4m3_decode(_u8(wq))
    acc = A @ Bm.T
    return acc * np.asarray(sx, np.float64)[:, None] * _f64(sw)[None, :]


def absmax_fp8_gemm(X, wq, sw, rows=None):
    """Whole cascade.  Returns (sx fp32 [M'], xq uint8 [M',K], Y fp64 [M',N])
    for all rows of X, or for the listed ``rows`` only."""
    Xs = X if rows is None else X[list(rows)]
    _, sx = row_scale(Xs)
    xq = quantise(Xs, sx)
    Y = gemm_dequant(xq, wq, sx, sw)
    return sx, xq, Y
