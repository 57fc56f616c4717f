"""Pins for the attention oracle (CPU only).

Each check ties the oracle to something other than itself: a worked example,
a closed form, a library routine (torch's fp64 scaled_dot_product_attention),
or an algebraic identity of the cascade.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import attention as A

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _rand(seed, *shape):
    return np.random.default_rng(seed).standard_normal(shape)


def test_golden_two_keys(golden_dir):
    d = json.load(open(os.path.join(golden_dir, "attn_two_keys.json")))
    q = np.array(d["q"])[None, None, None, :]
    k = np.array(d["k"])[None, None]
    v = np.array(d["v"])[None, None]
    o = A.attention(q, k, v, d["scale"])[0, 0, 0]
    np.testing.assert_allclose(o, d["o"], rtol=0, atol=1e-14)
    P = A.probabilities(q, k, v, d["scale"], 0, 0)[0]
    np.testing.assert_allclose(P, d["weights"], rtol=0, atol=1e-15)


@pytest.mark.parametrize("Hq,Hkv", [(1, 1), (4, 1), (8, 2)])
def test_matches_library_sdpa(Hq, Hkv):
    """torch's fp64 SDPA with explicit scale; GQA by repeating each K/V head
    over its contiguous group of Hq/Hkv query heads."""
    B, Lq, Lk, d, scale = 2, 5, 37, 16, 0.37
    q = torch.from_numpy(_rand(1, B, Hq, Lq, d))
    k = torch.from_numpy(_rand(2, B, Hkv, Lk, d))
    v = torch.from_numpy(_rand(3, B, Hkv, Lk, d))
    rep = Hq // Hkv
    ref = torch.nn.functional.scaled_dot_product_attention(
        q, k.repeat_interleave(rep, dim=1), v.repeat_interleave(rep, dim=1), scale=scale)
    got = A.attention(q, k, v, scale)
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)
    rows = [(1, Hq - 1, 3), (0, 0, 0), (1, 0, Lq - 1)]
    got_rows = A.attention(q, k, v, scale, rows=rows)
    for i, (b, h, iq) in enumerate(rows):
        np.testing.assert_allclose(got_rows[i], ref[b, h, iq].numpy(), rtol=1e-12, atol=1e-12)


def test_probabilities_sum_to_one():
    q, k, v = _rand(4, 1, 2, 7, 8), _rand(5, 1, 2, 50, 8) * 3, _rand(6, 1, 2, 50, 8)
    for h in range(2):
        P = A.probabilities(q, k, v, 0.5, 0, h)
        assert (P >= 0).all()
        np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=0, atol=1e-14)


def test_uniform_scores_give_mean_of_v():
    q = np.zeros((1, 1, 3, 8))
    k, v = _rand(7, 1, 1, 33, 8), _rand(8, 1, 1, 33, 8)
    o = A.attention(q, k, v, 1.0)
    np.testing.assert_allclose(o[0, 0], np.broadcast_to(v[0, 0].mean(axis=0), (3, 8)),
                               rtol=0, atol=1e-14)


def test_dominant_score_returns_that_row():
    Lk, d, j = 40, 8, 17
    k = _rand(9, 1, 1, Lk, d) * 0.01
    q = np.zeros((1, 1, 1, d))
    q[..., 0] = 1.0
    k[0, 0, j, 0] = 60.0          # s_j exceeds every other score by ~60
    v = _rand(10, 1, 1, Lk, d)
    o = A.attention(q, k, v, 1.0)[0, 0, 0]
    np.testing.assert_allclose(o, v[0, 0, j], rtol=0, atol=1e-20 + 50 * math.exp(-59.0))


def test_single_key_returns_v0():
    q, k, v = _rand(11, 1, 1, 4, 8), _rand(12, 1, 1, 1, 8), _rand(13, 1, 1, 1, 8)
    o = A.attention(q, k, v, 0.3)
    np.testing.assert_array_equal(o[0, 0], np.broadcast_to(v[0, 0, 0], (4, 8)))


def test_shift_invariance_and_scale_matters():
    """Adding one constant to every score leaves o unchanged (the reason for
    subtracting m); changing the scale changes o."""
    d = 8
    q = np.zeros((1, 1, 1, d))
    q[..., 0] = 1.0
    k, v = _rand(14, 1, 1, 20, d), _rand(15, 1, 1, 20, d)
    k2 = k.copy()
    k2[..., 0] += 5.0
    o1, o2 = A.attention(q, k, v, 0.7), A.attention(q, k2, v, 0.7)
    np.testing.assert_allclose(o1, o2, rtol=0, atol=1e-13)
    assert np.abs(A.attention(q, k, v, 1.4) - o1).max() > 1e-3


def test_decode_layout_matches_prefill_layout():
    q, k, v = _rand(16, 2, 8, 16), _rand(17, 2, 2, 30, 16), _rand(18, 2, 2, 30, 16)
    o = A.decode_attention(q, k, v, 0.25)
    ref = A.attention(q.reshape(2, 8, 1, 16), k, v, 0.25)[:, :, 0]
    np.testing.assert_array_equal(o, ref)
    rows = [(1, 7), (0, 3)]
    np.testing.assert_array_equal(A.decode_attention(q, k, v, 0.25, rows=rows),
                                  np.stack([ref[1, 7], ref[0, 3]]))


@pytest.mark.parametrize("tile", [1, 3, 8, 64, 100])
def test_incremental_equals_three_pass(tile):
    q, K, V = _rand(19, 16) * 2, _rand(20, 100, 16), _rand(21, 100, 16)
    np.testing.assert_allclose(A.attention_incremental(q, K, V, 0.5, tile),
                               A.three_pass_row(q, K, V, 0.5), rtol=1e-12, atol=1e-13)


def test_every_segment_split_merges_to_three_pass():
    """All 2^(Lk-1) ways of cutting Lk = 9 keys into contiguous segments,
    plus splits with empty segments."""
    Lk = 9
    q, K, V = _rand(22, 4) * 3, _rand(23, Lk, 4), _rand(24, Lk, 4)
    ref = A.three_pass_row(q, K, V, 1.0)
    for r in range(Lk):
        for cuts in itertools.combinations(range(1, Lk), r):
            bounds = [0, *cuts, Lk]
            np.testing.assert_allclose(A.attention_segments(q, K, V, 1.0, bounds), ref,
                                       rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(A.attention_segments(q, K, V, 1.0, [0, 0, 4, 4, 9, 9]), ref,
                               rtol=1e-12, atol=1e-13)


def test_planted_mistakes_are_caught():
    """Sanity of the pins themselves: a merge that forgets to rescale, or an
    incremental loop that forgets to rescale o, disagrees with the library."""
    q, K, V = _rand(25, 8) * 3, _rand(26, 40, 8), _rand(27, 40, 8)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q)[None, None, None], torch.from_numpy(K)[None, None],
        torch.from_numpy(V)[None, None], scale=1.0)[0, 0, 0].numpy()
    parts = [A.segment_partial(q, K, V, 1.0, a, a + 10) for a in range(0, 40, 10)]
    bad = sum(p[2] for p in parts) / sum(p[1] for p in parts)
    assert np.abs(bad - ref).max() > 1e-3
    np.testing.assert_allclose(A.merge_partials(parts), ref, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------- causal mask


@pytest.mark.parametrize("L", [1, 6, 33])
def test_causal_square_matches_library_sdpa(L):
    """Lq = Lk: torch's fp64 SDPA with is_causal=True (lower-triangular
    mask) is the same mask under either alignment convention."""
    q = torch.from_numpy(_rand(40, 2, 3, L, 16))
    k = torch.from_numpy(_rand(41, 2, 3, L, 16))
    v = torch.from_numpy(_rand(42, 2, 3, L, 16))
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=0.4)
    np.testing.assert_allclose(A.attention(q, k, v, 0.4, causal=True), ref.numpy(),
                               rtol=1e-12, atol=1e-12)
    np.testing.assert_array_equal(A.attention(q, k, v, 0.4, causal=True)[:, :, 0],
                                  v[:, :, 0].numpy())      # row 0 reads key 0 only


@pytest.mark.parametrize("Lq,Lk", [(5, 40), (17, 18), (1, 9)])
def test_causal_bottom_right_matches_library_sdpa_with_mask(Lq, Lk):
    """Lq <= Lk: row i reads keys 0 .. i + Lk - Lq, i.e. the boolean mask
    tril(ones(Lq, Lk), diagonal = Lk - Lq) given to torch's SDPA."""
    q = torch.from_numpy(_rand(43, 1, 2, Lq, 8))
    k = torch.from_numpy(_rand(44, 1, 2, Lk, 8))
    v = torch.from_numpy(_rand(45, 1, 2, Lk, 8))
    mask = torch.ones(Lq, Lk, dtype=torch.bool).tril(diagonal=Lk - Lq)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, attn_mask=mask, scale=0.6)
    np.testing.assert_allclose(A.attention(q, k, v, 0.6, causal=True), ref.numpy(),
                               rtol=1e-12, atol=1e-12)
    if Lq == 1:      # one query row sees every key: the causal result is the unmasked one
        np.testing.assert_array_equal(A.attention(q, k, v, 0.6, causal=True),
                                      A.attention(q, k, v, 0.6))


def test_causal_uniform_scores_give_running_mean_of_v():
    """Q = 0: every visible key has the same weight, so row i is the mean of
    the first i + Lk - Lq + 1 rows of V (closed form via a cumulative sum)."""
    Lq, Lk, d = 12, 20, 4
    q = np.zeros((1, 1, Lq, d))
    k, v = _rand(46, 1, 1, Lk, d), _rand(47, 1, 1, Lk, d)
    o = A.attention(q, k, v, 1.0, causal=True)[0, 0]
    csum = np.cumsum(v[0, 0], axis=0)
    n = np.arange(Lq) + (Lk - Lq) + 1
    np.testing.assert_allclose(o, csum[n - 1] / n[:, None], rtol=0, atol=1e-14)


def test_causal_rows_without_keys_are_zero():
    """Lq > Lk: rows i < Lq - Lk read no key and are zero by definition; the
    remaining rows match the square case on the last Lk query rows."""
    Lq, Lk = 10, 4
    q, k, v = _rand(48, 1, 1, Lq, 8), _rand(49, 1, 1, Lk, 8), _rand(50, 1, 1, Lk, 8)
    o = A.attention(q, k, v, 0.5, causal=True)[0, 0]
    np.testing.assert_array_equal(o[:Lq - Lk], 0.0)
    sq = A.attention(q[:, :, Lq - Lk:], k, v, 0.5, causal=True)[0, 0]
    np.testing.assert_array_equal(o[Lq - Lk:], sq)
    rows = [(0, 0, i) for i in range(Lq)]
    np.testing.assert_array_equal(A.attention(q, k, v, 0.5, causal=True, rows=rows), o)


# ------------------------------------------------------ variable lengths


def test_varlen_equal_lengths_match_fixed_layout():
    B, H, L, d = 3, 2, 11, 8
    q, k, v = _rand(60, B, H, L, d), _rand(61, B, H, L, d), _rand(62, B, H, L, d)
    pack = lambda t: t.transpose(0, 2, 1, 3).reshape(B * L, H, d)     # [B,H,L,d] -> [B*L,H,d]
    cu = np.arange(B + 1) * L
    for causal in (False, True):
        got = A.attention_varlen(pack(q), pack(k), pack(v), cu, cu, 0.3, causal=causal)
        np.testing.assert_allclose(got, pack(A.attention(q, k, v, 0.3, causal=causal)),
                                   rtol=1e-13, atol=1e-14)


def test_varlen_sequences_match_library_sdpa():
    """Every sequence of a ragged batch against torch's fp64 SDPA on its own
    tokens (with is_causal for the causal case, square sequences)."""
    lens = [5, 1, 17, 0, 9]
    cu = np.concatenate([[0], np.cumsum(lens)])
    H, d = 3, 8
    q, k, v = (_rand(63 + i, cu[-1], H, d) for i in range(3))
    for causal in (False, True):
        got = A.attention_varlen(q, k, v, cu, cu, 0.45, causal=causal)
        for b, n in enumerate(lens):
            if n == 0:
                continue
            sl = slice(cu[b], cu[b + 1])
            t = lambda x: torch.from_numpy(x[sl].transpose(1, 0, 2)[None].copy())
            ref = torch.nn.functional.scaled_dot_product_attention(
                t(q), t(k), t(v), is_causal=causal, scale=0.45)[0].numpy().transpose(1, 0, 2)
            np.testing.assert_allclose(got[sl], ref, rtol=1e-12, atol=1e-12)


def test_varlen_sequence_without_keys_is_zero():
    cu_q = np.array([0, 3, 7])
    cu_k = np.array([0, 0, 5])          # sequence 0 has no keys
    q, k, v = _rand(70, 7, 2, 4), _rand(71, 5, 2, 4), _rand(72, 5, 2, 4)
    o = A.attention_varlen(q, k, v, cu_q, cu_k, 1.0)
    np.testing.assert_array_equal(o[:3], 0.0)
    assert np.abs(o[3:]).max() > 0
