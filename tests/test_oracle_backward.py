"""Pins of the oracle's router, combine and permute backward against what is fixed
independently of their formulas: finite differences of the oracle's own forward,
adjoint identities of the forward maps (exact on bf16-representable data), a closed
form and invariants."""
import numpy as np
import pytest

import oracle as O

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _bf(a):
    """float array -> bf16 bits (values chosen exactly representable)."""
    return O.f64_to_bf16(np.asarray(a, np.float64))


def _val(bits):
    return O.bf16_to_f64(bits)


# ------------------------------------------------------------------ router backward
@pytest.mark.parametrize("renorm", [False, True])
def test_route_backward_matches_finite_differences_of_the_forward(renorm):
    """dF/dl for F(l) = sum_{t,k} g[t,k] probs(l)[t,k], selection fixed: central
    differences of the oracle's forward router (fp32 logits in and probs out)."""
    rng = np.random.default_rng(1)
    T, E, K = 4, 9, 3
    # well-separated logits: a step of h never changes the selection
    lg = (rng.permutation(E * T).reshape(T, E) * 0.37 - 6.0).astype(np.float32)
    ids, _ = O.route_topk(lg, K, renorm)
    g = rng.standard_normal((T, K)).astype(np.float32)
    d = O.route_backward(lg, ids, g, renorm)
    h = 2.0 ** -7

    def F(x):
        i2, p2 = O.route_topk(x, K, renorm)
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


def test_route_backward_two_experts_closed_form():
    """E = 2, K = 1: p = sigmoid(l0 - l1) for the winner; dl0 = g p (1 - p), dl1 = -g p (1 - p)."""
    lg = np.array([[0.75, -0.5], [-1.25, 2.0]], np.float32)
    ids, probs = O.route_topk(lg, 1)
    g = np.array([[2.0], [-0.5]], np.float32)
    d = O.route_backward(lg, ids, g)
    for t in range(2):
        w = int(ids[t, 0])
        p = 1.0 / (1.0 + np.exp(-(float(lg[t, w]) - float(lg[t, 1 - w]))))
        assert abs(d[t, w] - g[t, 0] * p * (1 - p)) < 1e-12
        assert abs(d[t, 1 - w] + g[t, 0] * p * (1 - p)) < 1e-12


@pytest.mark.parametrize("renorm", [False, True])
def test_route_backward_invariants(renorm):
    """Rows sum to 0 (softmax is shift-invariant); renormalised: zero off the selection;
    invalid routes (-1) carry no gradient."""
    rng = np.random.default_rng(2)
    T, E, K = 6, 40, 5
    lg = rng.standard_normal((T, E)).astype(np.float32)
    ids, _ = O.route_topk(lg, K, renorm)
    g = rng.standard_normal((T, K)).astype(np.float32)
    d = O.route_backward(lg, ids, g, renorm)
    assert np.abs(d.sum(1)).max() < 1e-12
    if renorm:
        mask = np.zeros((T, E), bool)
        np.put_along_axis(mask, ids, True, axis=1)
        assert np.all(d[~mask] == 0.0)
    ids2 = ids.copy()
    ids2[:, -1] = -1
    g2 = g.copy()
    g2[:, -1] = 1e6                      # ignored: the route is invalid
    d2 = O.route_backward(lg, ids2, g2, False)
    g3 = g.copy()
    g3[:, -1] = 0.0
    d3 = O.route_backward(lg, ids, g3, False)
    assert np.allclose(d2, d3, rtol=0, atol=1e-12)


# ------------------------------------------------------------------ combine / permute backward
def _routes(T, K, E, rng, invalid=0.2):
    ids = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    ids[rng.random((T, K)) < invalid] = -1
    return ids


def test_combine_backward_adjoint_identities():
    """With integer data and power-of-two probabilities every sum below is exact, so
    <dy, combine(y_perm, p)> = <dy_perm, y_perm> = sum p * dprobs hold exactly."""
    rng = np.random.default_rng(3)
    T, K, E, H = 12, 3, 5, 16
    ids = _routes(T, K, E, rng)
    op = O.permute(None, ids, E)
    rm, R = op["row_map"], op["R"]
    yp = _bf(rng.integers(-4, 5, (T * K, H)))
    probs = rng.choice([0.25, 0.5, 1.0], (T, K)).astype(np.float32)
    dy = _bf(rng.integers(-2, 3, (T, H)))
    y = O.combine(yp, rm, probs)
    dyp, dpr = O.combine_backward(dy, yp, rm, probs)
    lhs = float((_val(dy) * _val(y)).sum())
    assert lhs == float((_val(dyp)[:R] * _val(yp)[:R]).sum())
    assert lhs == float((probs.astype(np.float64) * dpr).sum())
    assert np.all(dpr[rm < 0] == 0.0)
    assert np.all(dyp[R:] == 0)


def test_combine_backward_dprobs_is_the_exact_derivative():
    """combine is linear in p: a step of 1/4 in one p[t,k] moves <dy, y> by dprobs[t,k] / 4."""
    rng = np.random.default_rng(4)
    T, K, E, H = 5, 2, 4, 8
    ids = _routes(T, K, E, rng, invalid=0.0)
    rm = O.permute(None, ids, E)["row_map"]
    yp = _bf(rng.integers(-3, 4, (T * K, H)))
    probs = np.full((T, K), 0.5, np.float32)
    dy = _bf(rng.integers(-2, 3, (T, H)))
    _, dpr = O.combine_backward(dy, yp, rm, probs)

    def F(p):
        return float((_val(dy) * _val(O.combine(yp, rm, p))).sum())
    for t in range(T):
        for k in range(K):
            p2 = probs.copy()
            p2[t, k] += 0.25
            assert F(p2) - F(probs) == dpr[t, k] * 0.25


def test_permute_backward_adjoint_and_route_count():
    """<permute_backward(d), x> = <d, permute(x)>, and permute_backward(permute(x)) gives
    x times the number of valid routes of each token (exact on integers)."""
    rng = np.random.default_rng(5)
    T, K, E, H = 10, 4, 6, 24
    ids = _routes(T, K, E, rng)
    x = _bf(rng.integers(-3, 4, (T, H)))
    op = O.permute(x, ids, E)
    d = _bf(rng.integers(-2, 3, (T * K, H)))
    d[op["R"]:] = 0
    dx = O.permute_backward(d, op["row_map"])
    assert float((_val(dx) * _val(x)).sum()) == float((_val(d) * _val(op["x_perm"])).sum())
    back = _val(O.permute_backward(op["x_perm"], op["row_map"]))
    nvalid = (op["row_map"] >= 0).sum(1)[:, None]
    assert np.array_equal(back, _val(x) * nvalid)
