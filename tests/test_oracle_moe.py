"""Pins for the MoE gate oracle (CPU only): exact integer scores, brute-force
top-k enumeration, the closed form of a two-way softmax, and a worked
example with ties."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import moe_gate as G


def _int_inputs(seed, T, D, E):
    rng = np.random.default_rng(seed)
    return rng.integers(-2, 3, (T, D)), rng.integers(-2, 3, (E, D))


def test_golden_ties(golden_dir):
    d = json.load(open(os.path.join(golden_dir, "moe_gate_tie.json")))
    idx, w, scores = G.moe_gate(np.array(d["x"], float), np.array(d["w_gate"], float), d["k"])
    np.testing.assert_array_equal(scores, d["scores"])
    np.testing.assert_array_equal(idx, d["idx"])
    np.testing.assert_allclose(w, d["weights"], rtol=0, atol=1e-15)


def test_scores_equal_integer_matmul():
    x, w = _int_inputs(1, 64, 512, 64)
    got = G.gate_scores(x.astype(float), w.astype(float))
    exact = x.astype(np.int64) @ w.astype(np.int64).T
    np.testing.assert_array_equal(got, exact.astype(float))


def _brute_top2(s):
    """Enumerate every ordered pair (i, j), i != j; keep the one whose
    (score_i, -i, score_j, -j) is largest subject to i ranking above j."""
    E = len(s)
    best = None
    for i in range(E):
        for j in range(E):
            if i == j or (s[i], -i) < (s[j], -j):
                continue
            key = (s[i], -i, s[j], -j)
            if best is None or key > best[0]:
                best = (key, (i, j))
    return best[1]


def test_top2_equals_brute_force_with_ties():
    # D = 16 keeps scores in a narrow integer range, so ties are frequent
    x, w = _int_inputs(2, 300, 16, 64)
    s = G.gate_scores(x.astype(float), w.astype(float))
    idx = G.topk_select(s, 2)
    n_ties = 0
    for t in range(s.shape[0]):
        assert tuple(idx[t]) == _brute_top2(list(s[t]))
        n_ties += int((s[t] == s[t, idx[t, 1]]).sum() > 1)
    assert n_ties > 30      # the tie-break is really exercised


def test_topk_values_match_library():
    x, w = _int_inputs(3, 200, 256, 64)
    s = G.gate_scores(x.astype(float), w.astype(float))
    for k in (1, 2, 4, 8):
        idx = G.topk_select(s, k)
        vals = np.take_along_axis(s, idx.astype(np.int64), axis=1)
        np.testing.assert_array_equal(vals, torch.topk(torch.from_numpy(s), k).values.numpy())
        # indices are distinct and ordered by (score desc, index asc)
        for t in range(s.shape[0]):
            keys = [(-s[t, e], e) for e in idx[t]]
            assert keys == sorted(keys) and len(set(idx[t])) == k


def test_two_way_softmax_closed_form():
    x, w = _int_inputs(4, 100, 64, 64)
    idx, wts, s = G.moe_gate(x.astype(float), w.astype(float), 2)
    s1 = np.take_along_axis(s, idx[:, :1].astype(np.int64), axis=1)[:, 0]
    s2 = np.take_along_axis(s, idx[:, 1:].astype(np.int64), axis=1)[:, 0]
    w1 = 1.0 / (1.0 + np.exp(s2 - s1))
    np.testing.assert_allclose(wts[:, 0], w1, rtol=1e-15, atol=0)
    np.testing.assert_allclose(wts.sum(axis=1), 1.0, rtol=0, atol=1e-15)
    assert (wts[:, 0] >= wts[:, 1]).all()


def test_rows_subset_matches_full():
    x, w = _int_inputs(5, 50, 128, 64)
    i_full, w_full, _ = G.moe_gate(x.astype(float), w.astype(float), 2)
    rows = [49, 0, 17]
    i_sub, w_sub, _ = G.moe_gate(x.astype(float), w.astype(float), 2, rows=rows)
    np.testing.assert_array_equal(i_sub, i_full[rows])
    np.testing.assert_array_equal(w_sub, w_full[rows])


def test_softmax_after_topk_not_before():
    """Reading of the article's order: softmax runs over the selected scores
    only, so the two weights sum to 1 even when other experts score close."""
    s = np.array([[3.0, 2.0, 2.0, 1.0]])
    idx = G.topk_select(s, 2)
    w = G.softmax_selected(np.take_along_axis(s, idx.astype(np.int64), axis=1))
    assert idx.tolist() == [[0, 1]]
    np.testing.assert_allclose(w[0], [1 / (1 + math.exp(-1)), math.exp(-1) / (1 + math.exp(-1))])


@pytest.mark.parametrize("E,k", [(8, 3), (5, 5), (12, 1)])
def test_topk_equals_brute_force_small_expert_counts(E, k):
    """Every ordered k-tuple of distinct experts is enumerated; the oracle's
    choice must be the tuple whose keys (score, -index) are in strictly
    descending order and that no other such tuple beats lexicographically."""
    x, w = _int_inputs(20 + E + k, 60, 6, E)
    s = G.gate_scores(x.astype(float), w.astype(float))
    idx = G.topk_select(s, k)
    for t in range(s.shape[0]):
        best = None
        for tup in itertools.permutations(range(E), k):
            keys = [(s[t, e], -e) for e in tup]
            if any(keys[i] <= keys[i + 1] for i in range(k - 1)):
                continue
            if best is None or keys > best[0]:
                best = (keys, tup)
        assert tuple(idx[t]) == best[1]


def test_topk_values_match_library_256_experts():
    x, w = _int_inputs(31, 100, 64, 256)
    s = G.gate_scores(x.astype(float), w.astype(float))
    idx = G.topk_select(s, 8)
    vals = np.take_along_axis(s, idx.astype(np.int64), axis=1)
    np.testing.assert_array_equal(vals, torch.topk(torch.from_numpy(s), 8).values.numpy())
    exact = x.astype(np.int64) @ w.astype(np.int64).T
    np.testing.assert_array_equal(s, exact.astype(float))


def test_single_expert_gets_weight_one():
    x, w = _int_inputs(32, 10, 16, 1)
    idx, wts, _ = G.moe_gate(x.astype(float), w.astype(float), 1)
    assert (idx == 0).all() and (wts == 1.0).all()
