"""Property checks of the oracle's routing and permutation on random small
cases (hypothesis): every id distinct, picks ordered by (sanitised logit,
then lower index), each pick beating every unpicked expert, weights summing
to 1 with renormalisation, grouped picks inside the kept groups, and the
permutation a stable sort by expert."""
import math

import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

FLT_MAX = float(np.finfo(np.float32).max)


def _san(v):
    v = float(v)
    if math.isnan(v):
        return -FLT_MAX
    if math.isinf(v):
        return FLT_MAX if v > 0 else -FLT_MAX
    return v


def _beats(a, b):
    return a[0] > b[0] or (a[0] == b[0] and a[1] < b[1])


logit = st.one_of(st.floats(-8, 8, width=32), st.just(float("nan")), st.just(float("inf")),
                  st.just(float("-inf")), st.sampled_from([0.0, 1.0, -1.0]))


@st.composite
def routing_case(draw):
    E = draw(st.integers(1, 24))
    k = draw(st.integers(1, E))
    T = draw(st.integers(1, 6))
    rows = draw(st.lists(st.lists(logit, min_size=E, max_size=E), min_size=T, max_size=T))
    return np.array(rows, np.float32), k


@settings(max_examples=60, deadline=None)
@given(routing_case(), st.sampled_from([0, 1]), st.booleans())
def test_route_properties(oracle, case, scoring, renorm):
    logits, k = case
    ids, w = oracle.route(logits, k, scoring=scoring, renorm=renorm)
    for t in range(logits.shape[0]):
        s = [_san(v) for v in logits[t]]
        picked = list(ids[t])
        assert len(set(picked)) == k
        for a, b in zip(picked, picked[1:]):
            assert _beats((s[a], a), (s[b], b))
        for e in range(len(s)):
            if e not in picked:
                assert _beats((s[picked[-1]], picked[-1]), (s[e], e))
        assert np.all(w[t] >= 0)
        if renorm:
            assert abs(w[t].sum() - 1.0) < 1e-12


@st.composite
def grouped_case(draw):
    n_group = draw(st.integers(1, 6))
    gs = draw(st.integers(1, 4))
    E = n_group * gs
    topk_group = draw(st.integers(1, n_group))
    k = draw(st.integers(1, topk_group * gs))
    T = draw(st.integers(1, 4))
    rows = draw(st.lists(st.lists(logit, min_size=E, max_size=E), min_size=T, max_size=T))
    return np.array(rows, np.float32), k, n_group, topk_group


@settings(max_examples=60, deadline=None)
@given(grouped_case())
def test_grouped_route_properties(oracle, case):
    logits, k, n_group, topk_group = case
    E = logits.shape[1]
    gs = E // n_group
    ids, w = oracle.route_grouped(logits, k, n_group, topk_group)
    for t in range(logits.shape[0]):
        s = [_san(v) for v in logits[t]]
        gmax = [max(s[g * gs:(g + 1) * gs]) for g in range(n_group)]
        order = sorted(range(n_group), key=lambda g: (-gmax[g], g))
        kept = set(order[:topk_group])
        picked = list(ids[t])
        assert len(set(picked)) == k
        assert all(e // gs in kept for e in picked)
        cand = [e for e in range(E) if e // gs in kept and e not in picked]
        for e in cand:
            assert _beats((s[picked[-1]], picked[-1]), (s[e], e))
        assert abs(w[t].sum() - 1.0) < 1e-12


@settings(max_examples=60, deadline=None)
@given(st.integers(1, 12), st.lists(st.integers(0, 11), min_size=0, max_size=40))
def test_permute_is_stable_sort(oracle, E, raw):
    flat = np.array([r % E for r in raw], np.int32)
    counts, offsets, src, pos = oracle.permute(flat, E)
    assert counts.sum() == flat.size
    np.testing.assert_array_equal(src, np.argsort(flat, kind="stable"))
    if flat.size:
        np.testing.assert_array_equal(pos[src], np.arange(flat.size))
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
