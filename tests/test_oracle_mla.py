"""Pins for the latent-KV (multi-latent attention) decode oracle (CPU only).

The oracle is tied to a library routine (torch's fp64
scaled_dot_product_attention with one shared key/value head and a value
width below the key width), to closed forms (zero query, one key, one
dominant key) and to the multi-segment identity of the cascade.
"""
import numpy as np
import pytest
import torch

from oracle import attention as A


def _rand(seed, *shape):
    return np.random.default_rng(seed).standard_normal(shape)


@pytest.mark.parametrize("B,Hq,Lk,dqk,dv", [(2, 4, 37, 24, 16), (1, 3, 5, 10, 8), (3, 2, 64, 40, 32)])
def test_matches_library_sdpa(B, Hq, Lk, dqk, dv):
    q, c = _rand(1, B, Hq, dqk), _rand(2, B, Lk, dqk)
    scale = 0.29
    o = A.mla_decode(q, c, scale, dv)
    qt = torch.from_numpy(q)[:, :, None, :]                       # [B, Hq, 1, dqk]
    kt = torch.from_numpy(c)[:, None].expand(B, Hq, Lk, dqk)      # one head, shared
    vt = torch.from_numpy(c[:, :, :dv])[:, None].expand(B, Hq, Lk, dv)
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, scale=scale)
    np.testing.assert_allclose(o, ref[:, :, 0].numpy(), rtol=0, atol=1e-13)


def test_zero_query_is_mean_of_leading_dims():
    B, Hq, Lk, dqk, dv = 2, 3, 11, 12, 8
    c = _rand(3, B, Lk, dqk)
    o = A.mla_decode(np.zeros((B, Hq, dqk)), c, 0.5, dv)
    for b in range(B):
        for h in range(Hq):
            np.testing.assert_allclose(o[b, h], c[b, :, :dv].mean(axis=0), rtol=0, atol=1e-14)


def test_one_key_returns_its_latent_dims():
    q, c = _rand(4, 2, 5, 12), _rand(5, 2, 1, 12)
    o = A.mla_decode(q, c, 0.7, 9)
    for b in range(2):
        for h in range(5):
            np.testing.assert_array_equal(o[b, h], c[b, 0, :9])


def test_dominant_key():
    """A key whose score is 60 above every other one takes all the weight
    (to within e^-60); the positional dims count in the score."""
    B, Hq, Lk, dqk, dv = 1, 2, 20, 12, 8
    c = _rand(6, B, Lk, dqk) * 0.01
    q = np.zeros((B, Hq, dqk))
    q[0, :, dqk - 1] = 1.0                   # only the last positional dim scores
    c[0, 13, dqk - 1] = 60.0
    o = A.mla_decode(q, c, 1.0, dv)
    for h in range(Hq):
        np.testing.assert_allclose(o[0, h], c[0, 13, :dv], rtol=0, atol=1e-15)


def test_rows_match_full():
    q, c = _rand(7, 3, 4, 16), _rand(8, 3, 9, 16)
    full = A.mla_decode(q, c, 0.3, 12)
    rows = [(2, 1), (0, 3), (1, 0), (2, 1)]
    sub = A.mla_decode(q, c, 0.3, 12, rows=rows)
    for i, (b, h) in enumerate(rows):
        np.testing.assert_array_equal(sub[i], full[b, h])


@pytest.mark.parametrize("bounds", [[0, 5, 31], [0, 1, 2, 31], [0, 16, 17, 30, 31]])
def test_segment_merge_equals_single_pass(bounds):
    """Multi-segment identity: partial states of any key split, merged,
    give the single-pass value (values = the leading dims of the keys)."""
    q, c = _rand(9, 1, 2, 20), _rand(10, 1, 31, 20)
    dv, scale = 14, 0.4
    o = A.mla_decode(q, c, scale, dv)
    for h in range(2):
        parts = [A.segment_partial(q[0, h], c[0], c[0, :, :dv], scale, bounds[j], bounds[j + 1])
                 for j in range(len(bounds) - 1)]
        np.testing.assert_allclose(A.merge_partials(parts), o[0, h], rtol=0, atol=1e-13)
