"""Pins for the router oracle: brute-force selection, closed forms of the
softmax, the tie rule, and planted mistakes."""

import math

import numpy as np
import pytest

import oracle.router as R
from oracle.router import router_topk


def brute_topk_ids(row, k):
    """k rounds of 'take the largest remaining logit; on equal logits the lower id'."""
    key = [(-math.inf if math.isnan(v) else float(v)) for v in row]
    taken, out = set(), []
    for _ in range(k):
        best = None
        for e in range(len(key)):          # ascending id: replace only on strictly greater
            if e in taken:
                continue
            if best is None or key[e] > key[best]:
                best = e
        taken.add(best)
        out.append(best)
    return out


@pytest.mark.parametrize("E,k", [(8, 2), (8, 8), (64, 8), (33, 5), (512, 10)])
def test_ids_match_brute_force_with_ties(E, k):
    g = np.random.default_rng(E * 31 + k)
    logits = np.round(g.standard_normal((40, E)), 1).astype(np.float32)   # many exact ties
    ids, _ = router_topk(logits, k)
    for t in range(40):
        assert ids[t].tolist() == brute_topk_ids(logits[t], k)


def test_equal_logits_lower_id_first_and_uniform_weights():
    E, k = 16, 5
    ids, w = router_topk(np.full((3, E), 0.25, dtype=np.float32), k)
    assert (ids == np.arange(k)).all()
    assert np.all(w == 1.0 / E)


def test_two_way_softmax_is_logistic():
    """softmax over two logits (a, b) gives 1 / (1 + exp(b - a)) for a."""
    for a, b in [(0.3, -1.2), (2.0, 1.5), (-4.0, -4.5), (10.0, -10.0)]:
        ids, w = router_topk(np.array([[a, b]], dtype=np.float32), 1)
        fa, fb = float(np.float32(a)), float(np.float32(b))
        assert ids[0, 0] == 0
        assert abs(w[0, 0] - 1.0 / (1.0 + math.exp(fb - fa))) < 1e-15


def test_geometric_logits_closed_form():
    """l_e = -e ln2 -> p_e = 2^-e / (2 - 2^(1-E)); weights halve down the list."""
    E = 12
    logits = (-np.arange(E) * math.log(2.0)).astype(np.float32)[None, :]
    ids, w = router_topk(logits, E)
    assert ids[0].tolist() == list(range(E))
    l64 = logits[0].astype(np.float64)
    z = sum(math.exp(v) for v in l64)
    for e in range(E):
        assert abs(w[0, e] - math.exp(l64[e]) / z) < 1e-15
    assert abs(w[0, 0] - 1.0 / (2.0 - 2.0 ** (1 - E))) < 1e-6      # float32 rounding of ln2 multiples


def test_shift_invariance_and_full_k_sums_to_one():
    g = np.random.default_rng(3)
    l = g.standard_normal((5, 64)).astype(np.float32)
    ids_a, w_a = router_topk(l, 64)
    ids_b, w_b = router_topk(l + np.float32(4.0), 64)
    assert (ids_a == ids_b).all()
    assert np.allclose(w_a, w_b, rtol=1e-5, atol=0)
    assert np.allclose(w_a.sum(axis=1), 1.0, rtol=0, atol=1e-12)


def test_weights_descend_and_renormalize():
    g = np.random.default_rng(4)
    l = g.standard_normal((20, 64)).astype(np.float32)
    ids, w = router_topk(l, 8)
    assert (np.diff(w, axis=1) <= 0).all()
    assert (w.sum(axis=1) < 1.0).all()
    _, wr = router_topk(l, 8, renormalize=True)
    assert np.allclose(wr.sum(axis=1), 1.0, atol=1e-12)
    assert np.allclose(wr, w / w.sum(axis=1, keepdims=True), rtol=1e-14)


def test_nan_ranks_last():
    l = np.array([[np.nan, 1.0, -5.0, np.nan, 0.5]], dtype=np.float32)
    ids, _ = router_topk(l, 4)
    assert ids[0].tolist() == [1, 4, 2, 0]


def test_bad_k_raises():
    with pytest.raises(ValueError):
        router_topk(np.zeros((1, 4), np.float32), 5)


# planted mistakes -------------------------------------------------------------

def test_planted_mistakes_are_caught(monkeypatch):
    l = np.round(np.random.default_rng(9).standard_normal((30, 16)), 1).astype(np.float32)
    good = [brute_topk_ids(r, 4) for r in l]

    # higher id wins ties
    def bad_ties(logits, k, renormalize=False):
        ids, w = router_topk(logits[:, ::-1], k, renormalize)
        return (logits.shape[1] - 1 - ids).astype(np.int32), w
    ids, _ = bad_ties(l, 4)
    assert ids.tolist() != good

    # softmax without max subtraction overflow guard is fine, but a sign slip is not
    monkeypatch.setattr(R, "softmax_f64", lambda x: R.np.exp(-x) / R.np.exp(-x).sum(-1, keepdims=True))
    _, w = R.router_topk(np.array([[0.0, math.log(3.0)]], np.float32), 1)
    assert abs(w[0, 0] - 0.75) > 0.1
