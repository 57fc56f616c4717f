"""Shared comparison helpers and tolerances for the GPU parity tests.

Tolerances (written here once, used by every parity test):
* bf16 in / fp32 accumulation / bf16 out (prefill, decode): elementwise
  max-abs error <= 2e-2 and relative L2 error <= 5e-3 against the fp64
  oracle.  Sources of error: bf16 P (2^-9 relative per weight), fp32
  accumulation, bf16 output rounding (2^-9 relative).
* bf16 attention outputs that the test's own input construction makes large
  (|O| well above the ~1 of N(0, 1) workloads, e.g. cache rows scaled up):
  the same bounds with the max-abs one scaled, |O - O_ref| <= 2e-2 *
  max(1, |O_ref|), since both bf16 roundings (P and O) are relative.
* fp32 tiny attention: relative L2 <= 1e-5 and
  |O - O_ref| <= 1e-5 * max(1, |O_ref|) elementwise.
* FP8 GEMM output Y (magnitudes up to ~1e3, where one bf16 ulp is 4 or
  more): |Y - Y_ref| <= 2e-2 * max(1, |Y_ref|) elementwise and relative
  L2 <= 5e-3.
* MoE weights: the scores are exact integers, so the weights differ only
  by fp32 exp/divide rounding: |w - w_ref| <= 1e-6.
* Integer and byte outputs (top-k indices, E4M3 codes) and the fp32 row
  scale sx (one IEEE division of exact values): bit-exact.
"""
import numpy as np
import torch

BF16_MAX_ABS = 2e-2
BF16_REL_L2 = 5e-3
F32_REL = 1e-5
FP8_Y_REL = 2e-2
FP8_Y_REL_L2 = 5e-3
MOE_W_ABS = 1e-6


def to64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().to("cpu", torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


def rel_l2(got, ref) -> float:
    got, ref = to64(got), to64(ref)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def assert_bf16_close(got, ref, what=""):
    got, ref = to64(got), to64(ref)
    assert np.isfinite(got).all(), f"{what}: non-finite output (unwritten element?)"
    err = np.abs(got - ref).max()
    r = rel_l2(got, ref)
    assert err <= BF16_MAX_ABS, f"{what}: max-abs {err:.3e} > {BF16_MAX_ABS}"
    assert r <= BF16_REL_L2, f"{what}: rel-L2 {r:.3e} > {BF16_REL_L2}"


def assert_bf16_close_scaled(got, ref, what=""):
    got, ref = to64(got), to64(ref)
    assert np.isfinite(got).all(), f"{what}: non-finite output (unwritten element?)"
    bound = BF16_MAX_ABS * np.maximum(1.0, np.abs(ref))
    bad = np.abs(got - ref) > bound
    assert not bad.any(), f"{what}: {bad.sum()} elements outside 2e-2 * max(1, |ref|)"
    assert rel_l2(got, ref) <= BF16_REL_L2, f"{what}: rel-L2 {rel_l2(got, ref):.3e}"


def assert_f32_close(got, ref, what=""):
    got, ref = to64(got), to64(ref)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    bound = F32_REL * np.maximum(1.0, np.abs(ref))
    bad = np.abs(got - ref) > bound
    assert not bad.any(), f"{what}: {bad.sum()} elements outside 1e-5 (max {np.abs(got - ref).max():.3e})"
    assert rel_l2(got, ref) <= F32_REL, f"{what}: rel-L2 {rel_l2(got, ref):.3e}"


def assert_fp8_y_close(got, ref, what=""):
    got, ref = to64(got), to64(ref)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    bound = FP8_Y_REL * np.maximum(1.0, np.abs(ref))
    bad = np.abs(got - ref) > bound
    assert not bad.any(), f"{what}: {bad.sum()} elements outside tolerance"
    assert rel_l2(got, ref) <= FP8_Y_REL_L2, f"{what}: rel-L2 {rel_l2(got, ref):.3e}"


# ------------------------------------------------------------------ FP8 weight

def fp8_weight_gpu(rf, w):
    """The pre-quantised weight as the CUDA path makes it: the library's own
    per-row absmax quantiser (rf_absmax_quant_fp8) applied to W [N, K].
    Returns device tensors (wq uint8 [N, K], sw fp32 [N])."""
    w = w.cuda()
    N, K = w.shape
    sw = torch.empty(N, dtype=torch.float32, device="cuda")
    wq = torch.empty(N, K, dtype=torch.uint8, device="cuda")
    rf.rf_absmax_quant_fp8(w, sw, wq)
    return wq, sw


def fp8_weight_oracle(w):
    """The same weight as the oracle makes it (row_scale, then quantise):
    (wq uint8 [N, K], sw fp32 [N]) numpy arrays."""
    from oracle import fp8_quant_gemm as F
    _, sw = F.row_scale(w)
    return F.quantise(w, sw), sw


# ------------------------------------------------------------------ guard bytes

GUARD_FRONT = 256      # keeps the tensor 256-byte aligned
GUARD_BACK = 4096
GUARD_BYTE = 0xA5


class Guarded:
    """A device output tensor with guard bytes of a known pattern in front of
    and behind it.  ``check()`` asserts that the kernel wrote nothing outside
    the tensor (the out-of-bounds-write detector of the ragged parity cases)."""

    def __init__(self, shape, dtype, fill=None, shift=0):
        """shift: extra bytes before the tensor (e.g. 16 for a start that is
        16-byte but not 32-byte aligned)."""
        n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.n = n
        self.front = GUARD_FRONT + shift
        self.raw = torch.full((self.front + n + GUARD_BACK,), GUARD_BYTE, dtype=torch.uint8,
                              device="cuda")
        self.t = self.raw[self.front:self.front + n].view(dtype).view(shape)
        if fill is None:
            fill = float("nan") if dtype.is_floating_point else 0x7F
        self.t.fill_(fill)

    def check(self, what=""):
        front = self.raw[:self.front]
        back = self.raw[self.front + self.n:]
        bad_f = int((front != GUARD_BYTE).sum().item())
        bad_b = int((back != GUARD_BYTE).sum().item())
        assert bad_f == 0 and bad_b == 0, \
            f"{what}: {bad_f} guard bytes before and {bad_b} after the output were overwritten"
