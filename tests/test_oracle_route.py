"""Pins for the oracle's estimate (a-3), routing (a-1) and permutation (a-2).

Each check is independent of the oracle's own code: the page's worked
example, brute force over all k-subsets, scipy's softmax/expit, numpy's
bincount and stable argsort, and the invariants the pages state."""
import itertools
import json
import math
import os

import numpy as np
import pytest
from scipy.special import expit, softmax

FLT_MAX = float(np.finfo(np.float32).max)
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_estimate_worked_example(oracle):
    with open(os.path.join(GOLDEN, "estimate_h20.json")) as f:
        g = json.load(f)
    assert g["T"] * g["top_k"] / g["experts"] == pytest.approx(g["rows_per_expert"])
    assert oracle.estimate(g["T"], g["top_k"], g["experts"]) == g["estimate"]


@pytest.mark.parametrize("T,k,E,want", [(1, 8, 128, 1), (0, 8, 128, 1), (16, 2, 8, 4),
                                        (128, 8, 128, 8), (4096, 8, 128, 256), (1, 1, 1, 1),
                                        (3, 2, 4, 2)])
def test_estimate_clamp_and_exact(oracle, T, k, E, want):
    assert oracle.estimate(T, k, E) == want
    assert want == max(1, -(-T * k // E))


def _sanitised(row):
    out = []
    for v in row:
        v = float(v)
        if math.isnan(v):
            out.append(-FLT_MAX)
        elif math.isinf(v):
            out.append(FLT_MAX if v > 0 else -FLT_MAX)
        else:
            out.append(v)
    return out


def _beats(a, b):
    """(value, index) pair a ranks before b: larger value, then lower index."""
    return a[0] > b[0] or (a[0] == b[0] and a[1] < b[1])


def _brute_topk(row, k):
    s = _sanitised(row)
    E = len(s)
    found = []
    for sub in itertools.combinations(range(E), k):
        inside = [(s[i], i) for i in sub]
        outside = [(s[i], i) for i in range(E) if i not in sub]
        if all(_beats(a, b) for a in inside for b in outside):
            found.append(sub)
    assert len(found) == 1
    sub = list(found[0])
    # order inside the set: repeated pairwise max under the same ranking
    ordered = []
    while sub:
        best = sub[0]
        for i in sub[1:]:
            if _beats((s[i], i), (s[best], best)):
                best = i
        ordered.append(best)
        sub.remove(best)
    return ordered


def _rows(rng, n, E):
    rows = []
    for _ in range(n):
        kind = rng.integers(5)
        if kind == 0:
            r = rng.standard_normal(E)
        elif kind == 1:  # many ties
            r = rng.integers(-2, 3, E).astype(float)
        elif kind == 2:  # NaN sprinkled
            r = rng.standard_normal(E)
            r[rng.random(E) < 0.4] = np.nan
        elif kind == 3:  # infinities
            r = rng.standard_normal(E)
            r[rng.integers(E)] = np.inf
            r[rng.integers(E)] = -np.inf
        else:
            r = np.full(E, np.nan)
        rows.append(r.astype(np.float32))
    return np.stack(rows)


@pytest.mark.parametrize("E,k", [(8, 2), (6, 3), (5, 5), (7, 1), (8, 4)])
def test_topk_brute_force(oracle, E, k):
    rng = np.random.default_rng(100 + E * 10 + k)
    logits = _rows(rng, 60, E)
    ids, _ = oracle.route(logits, k)
    for t in range(logits.shape[0]):
        assert list(ids[t]) == _brute_topk(logits[t], k)
        assert len(set(ids[t].tolist())) == k


def test_all_nan_and_all_equal_rows(oracle):
    E, k = 128, 8
    logits = np.full((3, E), np.nan, np.float32)
    logits[1] = 0.25
    logits[2, :] = np.nan
    logits[2, 77] = -3.0  # one finite logit among NaN wins the first slot
    for scoring in (oracle.SOFTMAX, oracle.SIGMOID):
        ids, w = oracle.route(logits, k, scoring=scoring, renorm=True)
        assert list(ids[0]) == list(range(k))
        assert list(ids[1]) == list(range(k))
        assert list(ids[2]) == [77] + list(range(k - 1))
        np.testing.assert_allclose(w[0], 1.0 / k, rtol=0, atol=1e-15)
        np.testing.assert_allclose(w[1], 1.0 / k, rtol=0, atol=1e-15)
        for t in range(3):
            assert len(set(ids[t].tolist())) == k
            assert abs(w[t].sum() - 1.0) < 1e-12


@pytest.mark.parametrize("scoring", [0, 1])
@pytest.mark.parametrize("renorm", [True, False])
def test_weights_closed_form(oracle, scoring, renorm):
    rng = np.random.default_rng(21)
    E, k = 40, 6
    logits = (rng.standard_normal((50, E)) * 2).astype(np.float32)
    logits[3, :5] = np.nan
    ids, w = oracle.route(logits, k, scoring=scoring, renorm=renorm)
    for t in range(logits.shape[0]):
        s = np.array(_sanitised(logits[t]), np.float64)
        if scoring == 0:
            if renorm:
                # renormalised softmax equals the softmax over the k picks
                ref = softmax(s[ids[t]])
            else:
                ref = softmax(s)[ids[t]]
        else:
            sig = expit(s[ids[t]])
            ref = sig / sig.sum() if renorm else sig
        np.testing.assert_allclose(w[t], ref, rtol=1e-12, atol=1e-300)
        if renorm:
            assert abs(w[t].sum() - 1.0) < 1e-12


def test_permutation_against_numpy(oracle):
    rng = np.random.default_rng(8)
    for E, T, k in [(8, 16, 2), (400, 288, 6), (128, 1, 8), (5, 40, 5)]:
        logits = rng.standard_normal((T, E)).astype(np.float32)
        ids, _ = oracle.route(logits, k)
        flat = ids.reshape(-1)
        counts, offsets, src, pos = oracle.permute(flat, E)
        np.testing.assert_array_equal(counts, np.bincount(flat, minlength=E))
        np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
        np.testing.assert_array_equal(src, np.argsort(flat, kind="stable"))
        assert counts.sum() == T * k
        assert counts.max() <= T  # distinct ids per token
        assert np.all(src[pos] == np.arange(T * k))
        assert np.all(pos[src] == np.arange(T * k))
        for e in range(E):
            seg = src[offsets[e]:offsets[e + 1]]
            assert np.all(flat[seg] == e)
            assert np.all(np.diff(seg) > 0)


def test_permutation_concentrated_all_same_experts(oracle):
    # every token on the same k experts (the crash repro shape of PR #39593)
    T, E, k = 64, 16, 4
    logits = np.zeros((T, E), np.float32)
    logits[:, [3, 9, 1, 12]] = [4.0, 3.0, 2.0, 1.0]
    ids, _ = oracle.route(logits, k)
    assert np.all(ids == np.array([3, 9, 1, 12]))
    counts, offsets, src, pos = oracle.permute(ids.reshape(-1), E)
    assert sorted(np.nonzero(counts)[0].tolist()) == [1, 3, 9, 12]
    assert np.all(counts[[1, 3, 9, 12]] == T)


def _brute_grouped(row, k, n_group, topk_group):
    """the unique kept-group set in which every kept group beats every other
    group under (group max, lower group), then brute-force top-k inside"""
    s = _sanitised(row)
    E = len(s)
    gs = E // n_group
    gmax = [max(s[g * gs:(g + 1) * gs]) for g in range(n_group)]
    found = []
    for sub in itertools.combinations(range(n_group), topk_group):
        if all(_beats((gmax[a], a), (gmax[b], b)) for a in sub for b in range(n_group)
               if b not in sub):
            found.append(sub)
    assert len(found) == 1
    cand = [e for e in range(E) if e // gs in found[0]]
    best = None
    for sub in itertools.combinations(cand, k):
        if all(_beats((s[i], i), (s[j], j)) for i in sub for j in cand if j not in sub):
            assert best is None
            best = list(sub)
    ordered = []
    while best:
        b = best[0]
        for i in best[1:]:
            if _beats((s[i], i), (s[b], b)):
                b = i
        ordered.append(b)
        best.remove(b)
    return ordered


@pytest.mark.parametrize("E,k,n_group,topk_group", [(8, 2, 4, 2), (12, 3, 4, 2), (8, 4, 2, 1),
                                                    (6, 2, 3, 3), (8, 1, 8, 1)])
def test_grouped_topk_brute_force(oracle, E, k, n_group, topk_group):
    rng = np.random.default_rng(200 + E * 10 + k + n_group)
    logits = _rows(rng, 60, E)
    ids, w = oracle.route_grouped(logits, k, n_group, topk_group)
    for t in range(logits.shape[0]):
        assert list(ids[t]) == _brute_grouped(logits[t], k, n_group, topk_group)
        assert len(set(ids[t].tolist())) == k
        assert abs(w[t].sum() - 1.0) < 1e-12


def test_grouped_topk_reductions(oracle):
    rng = np.random.default_rng(31)
    logits = _rows(rng, 40, 16)
    # one group, or all groups kept: plain top-k
    for n_group, topk_group in [(1, 1), (4, 4), (16, 16)]:
        ids_g, w_g = oracle.route_grouped(logits, 4, n_group, topk_group)
        ids, w = oracle.route(logits, 4)
        np.testing.assert_array_equal(ids_g, ids)
        np.testing.assert_allclose(w_g, w, rtol=1e-15)
    # all-NaN rows: distinct ids from the lowest groups
    nan = np.full((2, 16), np.nan, np.float32)
    ids, w = oracle.route_grouped(nan, 4, 4, 2)
    assert list(ids[0]) == [0, 1, 2, 3]
    np.testing.assert_allclose(w, 0.25)
