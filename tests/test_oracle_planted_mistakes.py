"""The oracle's pins tell plausible mistakes apart (CPU only).

Each test writes a plausible wrong variant of one oracle step here, in the
test (a flipped tie rule, a softmax taken before the selection, a reciprocal
multiply for the division, round-half-up for round-to-nearest-even, a
transposed operand, a sign error, a dropped scale, the wrong value dims),
and shows that the pin guarding that step rejects it while the oracle
itself passes.  The oracle is not changed."""
import json
import os

import numpy as np
import torch

from oracle import attention as A
from oracle import fp8_quant_gemm as F
from oracle import moe_gate as G


def _rand(seed, *shape):
    return np.random.default_rng(seed).standard_normal(shape)


# --------------------------------------------------------------- MoE gate


def _golden_tie(golden_dir):
    d = json.load(open(os.path.join(golden_dir, "moe_gate_tie.json")))
    return d, np.array(d["x"], float), np.array(d["w_gate"], float)


def test_tie_rule_to_the_higher_index_fails_the_worked_example(golden_dir):
    d, x, w = _golden_tie(golden_dir)
    scores = G.gate_scores(x, w)
    E = scores.shape[1]
    # wrong: among equal scores the higher expert index first
    wrong = (E - 1 - np.argsort(-scores[:, ::-1], axis=1, kind="stable"))[:, :d["k"]]
    assert not np.array_equal(wrong, d["idx"])
    np.testing.assert_array_equal(G.topk_select(scores, d["k"]), d["idx"])


def test_softmax_before_the_selection_fails_the_worked_example(golden_dir):
    d, x, w = _golden_tie(golden_dir)
    scores = G.gate_scores(x, w)
    idx = G.topk_select(scores, d["k"]).astype(np.int64)
    # wrong: softmax over all experts, then the selected probabilities
    p = np.exp(scores - scores.max(axis=1, keepdims=True))
    wrong = np.take_along_axis(p / p.sum(axis=1, keepdims=True), idx, axis=1)
    assert np.abs(wrong - np.array(d["weights"])).max() > 1e-2
    sel = np.take_along_axis(scores, idx, axis=1)
    np.testing.assert_allclose(G.softmax_selected(sel), d["weights"], rtol=0, atol=1e-15)


# ------------------------------------------------------------------- FP8


def test_reciprocal_multiply_fails_the_division_pin():
    """fp32(x * fp32(1/s)) differs from the correctly rounded fp32(x / s) in
    the last bit for some x, and where that moves the quotient across an
    E4M3 rounding boundary the code changes."""
    X = torch.from_numpy(_rand(1, 512, 2048)).to(torch.bfloat16)
    _, sx = F.row_scale(X)
    q = F.quantise(X, sx)
    x32 = X.float().numpy()
    inv = (np.float32(1.0) / sx.astype(np.float32))[:, None]
    wrong = F.e4m3_encode((x32 * inv).astype(np.float32).astype(np.float64))
    assert (wrong != q).any()
    # the pin: the fp32 quotient by IEEE division, cast by the library
    ref = torch.from_numpy((x32 / sx[:, None]).astype(np.float32)).to(torch.float8_e4m3fn)
    np.testing.assert_array_equal(q, ref.view(torch.uint8).numpy())


def test_round_half_up_fails_the_midpoint_pin():
    codes = np.arange(0x00, 0x7E, dtype=np.uint8)            # positive finite codes
    v = F.e4m3_decode(codes)
    mids = (v[:-1] + v[1:]) / 2
    # wrong: ties rounded away from zero instead of to the even code
    spacing = np.diff(v)
    wrong = v[:-1] + np.floor((mids - v[:-1]) / spacing + 0.5) * spacing
    right = F.e4m3_decode(F.e4m3_encode(mids))
    even = np.where(codes[:-1] % 2 == 0, v[:-1], v[1:])
    assert (wrong != even).any()
    np.testing.assert_array_equal(right, even)


def test_transposed_weight_fails_the_integer_product_pin():
    rng = np.random.default_rng(3)
    xq = F.e4m3_encode(rng.integers(-8, 9, (16, 16)).astype(float))
    wq = F.e4m3_encode(rng.integers(-8, 9, (16, 16)).astype(float))
    ones = np.ones(16, np.float32)
    exact = (F.e4m3_decode(xq).astype(np.int64) @ F.e4m3_decode(wq).astype(np.int64).T)
    wrong = F.e4m3_decode(xq) @ F.e4m3_decode(wq)            # W read as [K][N]
    assert not np.array_equal(wrong, exact)
    np.testing.assert_array_equal(F.gemm_dequant(xq, wq, ones, ones), exact)


# ------------------------------------------------------------- attention


def _sdpa(q, k, v, scale):
    return torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), scale=scale).numpy()


def test_sign_error_in_the_exponent_fails_the_library_pin():
    q, k, v = _rand(4, 1, 2, 5, 8), _rand(5, 1, 2, 9, 8), _rand(6, 1, 2, 9, 8)
    ref = _sdpa(q, k, v, 0.3)
    s = 0.3 * np.einsum("bhid,bhjd->bhij", q, k)
    m = s.max(axis=-1, keepdims=True)
    p = np.exp(m - s)                                        # wrong sign
    wrong = np.einsum("bhij,bhjd->bhid", p / p.sum(axis=-1, keepdims=True), v)
    assert np.abs(wrong - ref).max() > 1e-2
    np.testing.assert_allclose(A.attention(q, k, v, 0.3), ref, rtol=1e-12, atol=1e-12)


def test_dropped_scale_fails_the_library_pin():
    q, k, v = _rand(7, 1, 1, 4, 16), _rand(8, 1, 1, 6, 16), _rand(9, 1, 1, 6, 16)
    ref = _sdpa(q, k, v, 0.25)
    assert np.abs(A.attention(q, k, v, 1.0) - ref).max() > 1e-2
    np.testing.assert_allclose(A.attention(q, k, v, 0.25), ref, rtol=1e-12, atol=1e-12)


def test_wrong_value_dims_fail_the_latent_decode_pin():
    """Latent decode: values are the first dv dims of each cache row; taking
    the last dv instead is caught by the library routine with v = c[..., :dv]."""
    B, Hq, Lk, dqk, dv = 1, 3, 7, 24, 16
    q, c = _rand(10, B, Hq, dqk), _rand(11, B, Lk, dqk)
    qt = torch.from_numpy(q)[:, :, None]                      # [B, Hq, 1, dqk]
    ct = torch.from_numpy(c)[:, None]                         # [B, 1, Lk, dqk]
    ref = torch.nn.functional.scaled_dot_product_attention(
        qt, ct.expand(B, Hq, Lk, dqk), ct[..., :dv].expand(B, Hq, Lk, dv), scale=0.2)[:, :, 0]
    wrong = torch.nn.functional.scaled_dot_product_attention(
        qt, ct.expand(B, Hq, Lk, dqk), ct[..., dqk - dv:].expand(B, Hq, Lk, dv), scale=0.2)[:, :, 0]
    assert (wrong - ref).abs().max() > 1e-2
    np.testing.assert_allclose(A.mla_decode(q, c, 0.2, dv), ref.numpy(), rtol=1e-12, atol=1e-12)
