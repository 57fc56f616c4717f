"""The seeded input generators: shapes, dtypes, determinism and the value
sets the workloads promise (integers in {-2..2}, ~1% outliers)."""
import torch

import workloads as I


def test_attention_shapes_and_determinism():
    s = I.AttnShape(2, 4, 2, 3, 70, 64, "bf16", seed=9)
    q, k, v = I.attention_inputs(s)
    assert q.shape == (2, 4, 3, 64) and k.shape == (2, 2, 70, 64) and v.dtype == torch.bfloat16
    q2, k2, v2 = I.attention_inputs(s)
    assert torch.equal(q, q2) and torch.equal(k, k2) and torch.equal(v, v2)
    qd, kd, vd = I.decode_inputs(I.AttnShape(2, 4, 2, 1, 70, 128, "bf16", seed=9))
    assert qd.shape == (2, 4, 128)
    assert I.TINY_ATTN.scale == 0.125 and abs(I.DECODE_2K.scale - 128 ** -0.5) < 1e-15


def test_moe_values_are_small_integers():
    x, w = I.moe_inputs(I.MoEShape(T=64, D=128, E=64, k=2, seed=1))
    assert x.shape == (64, 128) and w.shape == (64, 128)
    for t in (x, w):
        assert set(t.float().unique().tolist()) <= {-2.0, -1.0, 0.0, 1.0, 2.0}


def test_fp8_inputs():
    x, w = I.fp8_inputs(I.FP8Shape(M=256, N=64, K=512, seed=2))
    assert x.dtype == torch.bfloat16 and w.dtype == torch.bfloat16
    assert x.shape == (256, 512) and w.shape == (64, 512)
    frac = (x.float().abs() > 6).float().mean().item()      # outliers (|N(0,1)| > 6 is ~2e-9)
    assert 0.004 < frac < 0.012
    assert (w.float().abs() < 7).all()                      # the weight has no outliers
    x2, w2 = I.fp8_inputs(I.FP8Shape(M=256, N=64, K=512, seed=2))
    assert torch.equal(x, x2) and torch.equal(w, w2)
