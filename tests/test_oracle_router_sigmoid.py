"""Pins of the oracle's sigmoid-score router (selection on score + expert bias) and of its
backward, against what is fixed independently of the oracle's code: a library logistic
function, brute force over all K-subsets of tiny rows, closed forms of bias steering, exact
ties, invariants, and finite differences of the oracle's own forward."""
import itertools

import numpy as np
import pytest

import oracle as O

scipy_special = pytest.importorskip("scipy.special")

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _ulp_close(a, b, n=1):
    a = np.asarray(a, np.float32)
    b = np.asarray(b, np.float32)
    return np.all(np.abs(a.astype(np.float64) - b) <= n * np.spacing(np.maximum(np.abs(a), np.abs(b))))


def test_scores_are_the_logistic_function():
    """Without renormalisation the probabilities are the scores themselves: the logistic
    function of the logit (scipy's expit in double, rounded to fp32), within one fp32 ulp."""
    rng = np.random.default_rng(0)
    T, E, K = 64, 40, 40                   # K = E: every score comes out
    lg = (rng.standard_normal((T, E)) * 4).astype(np.float32)
    ids, probs = O.route_sigmoid_topk(lg, K)
    ref = scipy_special.expit(np.take_along_axis(lg, ids, 1).astype(np.float64)).astype(np.float32)
    assert _ulp_close(probs, ref)
    # K = E: each row's ids are a permutation
    assert np.array_equal(np.sort(ids, 1), np.tile(np.arange(E), (T, 1)))


def test_zero_bias_selects_what_the_softmax_router_selects():
    """The logistic function is increasing: with no bias and well-separated logits the ids
    (and their order) are the softmax router's."""
    rng = np.random.default_rng(1)
    T, E, K = 50, 64, 6
    lg = np.stack([rng.permutation(E) for _ in range(T)]).astype(np.float32) * (6.0 / E) - 3.0
    ids_s, _ = O.route_sigmoid_topk(lg, K)
    ids_m, _ = O.route_topk(lg, K)
    assert np.array_equal(ids_s, ids_m)


@pytest.mark.parametrize("renorm", [False, True])
def test_brute_force_over_all_subsets(renorm):
    """Tiny rows: the selected set is the K-subset whose every key beats every key outside it
    (keys s + b in fp32, s from scipy's expit; equal keys: lower index wins), listed in the
    order of a library sort on (-key, index)."""
    rng = np.random.default_rng(2)
    for trial in range(300):
        E = int(rng.integers(1, 8))
        K = int(rng.integers(1, E + 1))
        lg = rng.choice(np.float32([-2, -1, -0.5, 0, 0.5, 1, 2]), E).astype(np.float32)
        b = rng.choice(np.float32([-0.25, 0, 0.125, 0.25]), E).astype(np.float32)
        ids, probs = O.route_sigmoid_topk(lg[None], K, bias=b, renorm=renorm)
        s = scipy_special.expit(lg.astype(np.float64)).astype(np.float32)
        key = s + b                                   # fp32 addition
        beats = lambda i, j: key[i] > key[j] or (key[i] == key[j] and i < j)
        winners = [c for c in itertools.combinations(range(E), K)
                   if all(beats(i, j) for i in c for j in range(E) if j not in c)]
        assert len(winners) == 1
        order = sorted(winners[0], key=lambda e: (-float(key[e]), e))
        assert list(ids[0]) == order, (trial, lg, b, ids)
        sel = s[order].astype(np.float64)
        want = sel / sel.sum() if renorm else sel
        assert np.allclose(probs[0], want, rtol=2e-7, atol=0)


def test_bias_steers_the_selection_closed_form():
    """All logits 0 (every score 1/2): the bias alone orders the experts; the probabilities
    are the scores (1/2 each), or 1/K renormalised. A bias above 1 wins over any logit."""
    lg = np.zeros((1, 4), np.float32)
    b = np.float32([0.0, 1.0, 0.0, 2.0])
    ids, probs = O.route_sigmoid_topk(lg, 2, bias=b)
    assert list(ids[0]) == [3, 1] and np.all(probs == 0.5)
    ids, probs = O.route_sigmoid_topk(lg, 2, bias=b, renorm=True)
    assert list(ids[0]) == [3, 1] and np.all(probs == 0.5)
    lg2 = np.float32([[30.0, -30.0, 0.0]])
    ids, probs = O.route_sigmoid_topk(lg2, 1, bias=np.float32([0.0, 1.5, 0.0]))
    assert ids[0, 0] == 1                              # s_1 + 1.5 > 1 > s_0
    assert abs(probs[0, 0] - scipy_special.expit(-30.0)) <= 1e-20


def test_exact_ties_go_to_the_lower_index():
    lg = np.full((3, 9), 0.75, np.float32)
    ids, _ = O.route_sigmoid_topk(lg, 4, bias=np.zeros(9, np.float32))
    assert np.array_equal(ids, np.tile(np.arange(4), (3, 1)))


def test_a_constant_bias_shift_changes_nothing():
    """Adding the same exactly representable constant to every bias keeps the order of the
    keys (and the scores), so ids and probabilities are unchanged."""
    rng = np.random.default_rng(3)
    T, E, K = 20, 32, 5
    lg = rng.standard_normal((T, E)).astype(np.float32)
    b = (rng.integers(-8, 9, E) / 64).astype(np.float32)
    for renorm in (False, True):
        i1, p1 = O.route_sigmoid_topk(lg, K, bias=b, renorm=renorm)
        i2, p2 = O.route_sigmoid_topk(lg, K, bias=b + np.float32(4.0), renorm=renorm)
        assert np.array_equal(i1, i2) and np.array_equal(p1, p2)
        _, p3 = O.route_sigmoid_topk(lg, K, bias=b, renorm=True)
        if renorm:
            assert np.allclose(p3.sum(1), 1.0, atol=1e-6)


@pytest.mark.parametrize("renorm", [False, True])
def test_backward_matches_finite_differences_of_the_forward(renorm):
    """dF/dl for F(l) = sum g[t,k] probs(l)[t,k], selection fixed: central differences of the
    oracle's forward (fp32 logits in, fp32 probabilities out)."""
    rng = np.random.default_rng(4)
    T, E, K = 4, 9, 3
    lg = (rng.permutation(E * T).reshape(T, E) * 0.11 - 2.0).astype(np.float32)
    b = (rng.integers(-4, 5, E) / 16).astype(np.float32)
    ids, _ = O.route_sigmoid_topk(lg, K, bias=b, renorm=renorm)
    g = rng.standard_normal((T, K)).astype(np.float32)
    d = O.route_sigmoid_backward(lg, ids, g, renorm)
    h = 2.0 ** -7

    def F(x):
        i2, p2 = O.route_sigmoid_topk(x, K, bias=b, renorm=renorm)
        assert np.array_equal(i2, ids)
        return float((g.astype(np.float64) * p2).sum())

    fd = np.zeros((T, E))
    for t in range(T):
        for e in range(E):
            up, dn = lg.copy(), lg.copy()
            up[t, e] += h
            dn[t, e] -= h
            fd[t, e] = (F(up) - F(dn)) / (2 * h)
    assert np.abs(fd - d).max() <= 2e-4 * max(1.0, np.abs(d).max())


def test_backward_invariants():
    """Zero off the selection; renormalised rows: the selected gradients sum to zero when every
    score's weight s (1 - s) is equal (all logits equal); invalid routes carry nothing."""
    rng = np.random.default_rng(5)
    T, E, K = 6, 24, 4
    lg = rng.standard_normal((T, E)).astype(np.float32)
    ids, _ = O.route_sigmoid_topk(lg, K)
    g = rng.standard_normal((T, K)).astype(np.float32)
    for renorm in (False, True):
        d = O.route_sigmoid_backward(lg, ids, g, renorm)
        mask = np.zeros((T, E), bool)
        np.put_along_axis(mask, ids, True, axis=1)
        assert np.all(d[~mask] == 0.0)
    flat = np.full((T, E), 0.3, np.float32)
    d = O.route_sigmoid_backward(flat, ids, g, True)
    assert np.abs(d.sum(1)).max() < 1e-12
    ids2 = ids.copy()
    ids2[:, -1] = -1
    g2 = g.copy()
    g2[:, -1] = 1e6
    g3 = g.copy()
    g3[:, -1] = 0.0
    ids3 = ids.copy()
    ids3[:, -1] = -1
    assert np.allclose(O.route_sigmoid_backward(lg, ids2, g2, False), O.route_sigmoid_backward(lg, ids3, g3, False),
                       rtol=0, atol=1e-12)
