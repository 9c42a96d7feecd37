"""Pins of the router oracle (oracle/router.py) against facts that do not come
from the oracle itself: a worked example, a library softmax + stable sort,
invariants and special cases."""

import os

import numpy as np
import pytest
from scipy.special import softmax

from oracle import router as R

GOLD = os.path.join(os.path.dirname(__file__), "golden", "router_example.txt")


def _golden():
    d = {}
    for ln in open(GOLD):
        if ln.startswith("#") or not ln.strip():
            continue
        k, *v = ln.split()
        d[k] = v
    return d


def test_worked_example():
    g = _golden()
    logits = np.array([[float(x) for x in g["logits"]]])
    k = int(g["top_k"][0])
    ids, w = R.route_topk(logits, k)
    assert ids[0].tolist() == [int(x) for x in g["ids"]]
    np.testing.assert_allclose(w[0], [float(x) for x in g["renorm_weights"]], rtol=1e-15)
    _, wp = R.route_topk(logits, k, renormalize=False)
    np.testing.assert_allclose(wp[0], [float(x) for x in g["plain_weights"]], rtol=1e-15)


@pytest.mark.parametrize("E,k", [(8, 2), (257, 9), (288, 8), (64, 64)])
def test_matches_library_softmax_and_stable_sort(E, k):
    rng = np.random.default_rng(E * 31 + k)
    l = rng.standard_normal((20, E))
    ids, w = R.route_topk(l, k, renormalize=False)
    p = softmax(l, axis=1)
    for t in range(20):
        ref = np.argsort(-l[t], kind="stable")[:k]
        assert ids[t].tolist() == ref.tolist()
        np.testing.assert_allclose(w[t], p[t, ref], rtol=1e-12)
    _, wr = R.route_topk(l, k, renormalize=True)
    sel = np.take_along_axis(p, ids, axis=1)
    np.testing.assert_allclose(wr, sel / sel.sum(axis=1, keepdims=True), rtol=1e-12)


def test_invariants_on_ties_and_scale():
    rng = np.random.default_rng(5)
    l = rng.integers(-3, 4, size=(50, 40)).astype(np.float64)   # many equal logits
    ids, w = R.route_topk(l, 7, routed_scale=2.5)
    for t in range(50):
        s = ids[t]
        assert len(set(s.tolist())) == 7
        chosen = l[t, s]
        others = np.delete(l[t], s)
        assert chosen.min() >= others.max()                     # nothing larger left behind
        # equal logits: ascending index, and no unselected expert with an equal
        # logit and a lower index than a selected one
        for a, b in zip(s[:-1], s[1:]):
            assert l[t, a] > l[t, b] or (l[t, a] == l[t, b] and a < b)
        thr = chosen.min()
        tied = np.nonzero(l[t] == thr)[0]
        assert set(s[chosen == thr].tolist()) == set(tied[: (chosen == thr).sum()].tolist())
        np.testing.assert_allclose(w[t].sum(), 2.5, rtol=1e-12)
        assert np.all(np.diff(w[t]) <= 0)


def test_special_cases():
    # uniform logits: the first k experts, equal weights 1/k
    ids, w = R.route_topk(np.zeros((3, 10)), 4)
    assert ids.tolist() == [[0, 1, 2, 3]] * 3
    np.testing.assert_allclose(w, 0.25)
    # top_k = E: every expert, weights = the full softmax in descending order
    l = np.array([[0.5, -1.0, 2.0]])
    ids, w = R.route_topk(l, 3)
    assert ids.tolist() == [[2, 0, 1]]
    np.testing.assert_allclose(w[0], softmax(l[0])[[2, 0, 1]], rtol=1e-15)
    # top_k = 1 with renormalisation: weight exactly routed_scale
    ids, w = R.route_topk(np.array([[1.0, 7.0, 3.0]]), 1, routed_scale=1.5)
    assert ids.tolist() == [[1]] and w.tolist() == [[1.5]]
    # a large logit spread stays finite (max subtracted)
    ids, w = R.route_topk(np.array([[1000.0, -1000.0, 999.0]]), 2)
    np.testing.assert_allclose(w[0], [1 / (1 + np.exp(-1)), np.exp(-1) / (1 + np.exp(-1))], rtol=1e-15)
    with pytest.raises(ValueError):
        R.route_topk(np.zeros((1, 4)), 5)
