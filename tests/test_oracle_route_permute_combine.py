"""Pins for the oracle's router, permutation and combine.

Independent references: brute-force full stable sort (pure Python) on tiny
inputs, closed forms of the softmax, and the invariants a dropless
permutation must satisfy (every valid route exactly once, round trip, empty
experts). Page values: the route-metadata sizes printed on "Sparser MoE
end-to-end", section "Preserve a compact route" (tests/golden/).
"""
import itertools
import math
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- router
def _brute_topk(row, K):
    order = sorted(range(len(row)), key=lambda e: (-float(row[e]), e))
    return order[:K]


@pytest.mark.parametrize("E", [1, 2, 3, 5, 8, 16])
def test_router_ids_match_brute_force_with_ties(E):
    rng = np.random.default_rng(E)
    T = 64
    pool = np.array([-np.inf, -1.5, -0.0, 0.0, 0.25, 0.25, 1.0, 3.0], np.float32)
    lg = rng.choice(pool, size=(T, E)).astype(np.float32)
    lg[0] = 0.0                                   # whole row tied
    lg[1, ::2] = -0.0                             # +0 / -0 tie
    lg[2] = rng.standard_normal(E).astype(np.float32)
    for K in range(1, E + 1):
        ids, _ = O.route_topk(lg, K)
        for t in range(T):
            assert list(ids[t]) == _brute_topk(lg[t], K), (t, K)


def test_router_full_argsort_when_k_equals_e():
    rng = np.random.default_rng(7)
    lg = rng.standard_normal((32, 12)).astype(np.float32)
    ids, probs = O.route_topk(lg, 12)
    for t in range(32):
        assert sorted(ids[t]) == list(range(12))
        assert np.all(np.diff(lg[t, ids[t]]) <= 0)
    # softmax over all E sums to one
    assert np.allclose(probs.astype(np.float64).sum(1), 1.0, atol=1e-6)


def test_router_probs_closed_forms():
    # equal logits: 1/E each
    _, p = O.route_topk(np.zeros((4, 10), np.float32), 3)
    assert np.allclose(p, 0.1, atol=1e-7)
    # two experts, logit gap d: softmax is the logistic function of d
    d = np.linspace(-8, 8, 33).astype(np.float32)
    lg = np.stack([d, np.zeros_like(d)], 1)
    _, p = O.route_topk(lg, 2)
    top = np.maximum(d, 0)
    want_top = 1.0 / (1.0 + np.exp(-np.abs(d.astype(np.float64))))
    assert np.allclose(p[:, 0], want_top, atol=1e-7)
    assert np.allclose(p[:, 1], 1 - want_top, atol=1e-7)
    del top
    # ratios: p_i / p_j = exp(l_i - l_j)
    rng = np.random.default_rng(8)
    lg = rng.standard_normal((16, 20)).astype(np.float32)
    ids, p = O.route_topk(lg, 5)
    for t in range(16):
        l = lg[t, ids[t]].astype(np.float64)
        assert np.allclose(p[t, 1:] / p[t, 0], np.exp(l[1:] - l[0]), rtol=1e-6)


def test_router_renorm_sums_to_one_and_keeps_ratios():
    rng = np.random.default_rng(9)
    lg = rng.standard_normal((64, 8)).astype(np.float32) * 3
    ids, p = O.route_topk(lg, 2, renorm=True)
    ids0, p0 = O.route_topk(lg, 2, renorm=False)
    assert np.array_equal(ids, ids0)
    assert np.allclose(p.astype(np.float64).sum(1), 1.0, atol=1e-6)
    assert np.allclose(p / p.sum(1, keepdims=True), p0 / p0.sum(1, keepdims=True), atol=1e-6)


def test_router_matches_torch_topk_on_distinct_values():
    g = torch.Generator().manual_seed(11)
    lg = torch.randn(500, 64, generator=g)
    ids, p = O.route_topk(lg.numpy(), 6)
    ref = torch.topk(lg, 6, dim=1, sorted=True)
    assert np.array_equal(ids, ref.indices.numpy())
    sm = torch.softmax(lg.double(), dim=1).gather(1, ref.indices)
    assert np.allclose(p, sm.numpy(), atol=1e-7)


# --------------------------------------------------------------- permute
def _brute_permute(ids, E):
    T, K = ids.shape
    pairs = sorted((int(ids[t, k]), t * K + k) for t in range(T) for k in range(K)
                   if 0 <= ids[t, k] < E)
    row_map = -np.ones((T, K), np.int32)
    perm_src = []
    for r, (e, i) in enumerate(pairs):
        row_map[i // K, i % K] = r
        perm_src.append(i // K)
    sizes = np.bincount([e for e, _ in pairs], minlength=E).astype(np.int32)
    return row_map, np.array(perm_src, np.int32), sizes


@pytest.mark.parametrize("T,K,E", [(1, 1, 1), (7, 2, 4), (33, 3, 8), (64, 8, 32), (10, 4, 300)])
def test_permute_matches_brute_force_sort(T, K, E):
    rng = np.random.default_rng(T * 1000 + E)
    ids = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    ids[rng.random((T, K)) < 0.1] = -1            # invalid routes
    x = rng.integers(0, 65535, size=(T, 16), dtype=np.uint16)
    out = O.permute(x, ids, E)
    rm, ps, sizes = _brute_permute(ids, E)
    R = int((ids >= 0).sum())
    assert out["R"] == R == sizes.sum()
    assert np.array_equal(out["row_map"], rm)
    assert np.array_equal(out["perm_src"][:R], ps)
    assert np.array_equal(out["group_sizes"], sizes)
    assert np.array_equal(out["group_offsets"], np.concatenate([[0], np.cumsum(sizes)]))
    # round trip: each valid route's destination holds its token's row, bit for bit
    for t in range(T):
        for k in range(K):
            if ids[t, k] >= 0:
                assert np.array_equal(out["x_perm"][out["row_map"][t, k]], x[t])


def test_permute_every_valid_route_exactly_once_and_empty_experts():
    rng = np.random.default_rng(12)
    T, K, E = 200, 4, 16
    ids = np.stack([rng.choice([0, 3, 5, 9, 15], size=K, replace=False) for _ in range(T)])
    out = O.permute(None, ids.astype(np.int32), E)
    gs, go = out["group_sizes"], out["group_offsets"]
    assert gs.sum() == T * K
    for e in range(E):
        if e not in (0, 3, 5, 9, 15):
            assert gs[e] == 0 and go[e] == go[e + 1]
    rows = np.sort(out["row_map"].ravel())
    assert np.array_equal(rows, np.arange(T * K))
    # perm_src inverts row_map
    for t in range(T):
        for k in range(K):
            assert out["perm_src"][out["row_map"][t, k]] == t


def test_permute_out_of_range_ids_are_skipped():
    ids = np.array([[0, 5], [-1, 1], [7, -3]], np.int32)     # E = 2: 5, 7, -3 out of range
    out = O.permute(None, ids, 2)
    assert out["R"] == 2
    assert out["row_map"].tolist() == [[0, -1], [-1, 1], [-1, -1]]


def test_route_metadata_sizes_from_page():
    """Page values: T=8192, E=2304, K=36 -> 18.87 MB bool map vs 0.59 MB int16 ids (32x)."""
    vals = {}
    with open(os.path.join(GOLDEN, "route_metadata_sizes.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, v = line.split("=")
                vals[k.strip()] = float(v)
    T, E, K = int(vals["T"]), int(vals["E"]), int(vals["K"])
    bool_map = T * E * 1
    compact = T * K * 2
    assert round(bool_map / 1e6, 2) == vals["bool_map_MB"]
    assert round(compact / 1e6, 2) == vals["int16_ids_MB"]
    assert bool_map // compact == vals["ratio"]
    # the oracle's compact route really is [T, K]
    lg = np.zeros((4, E), np.float32)
    ids, _ = O.route_topk(lg, K)
    assert ids.shape == (4, K)


# --------------------------------------------------------------- combine
def _torch_bf16(x64):
    return torch.from_numpy(np.asarray(x64, np.float64)).to(torch.float32).to(
        torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_combine_identity_experts_equals_weighted_sum_of_token():
    rng = np.random.default_rng(13)
    T, H, E, K = 40, 64, 6, 3
    x = _torch_bf16(rng.standard_normal((T, H)) * 0.5)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    ids, probs = O.route_topk(lg, K)
    ids[5] = -1                                    # token with no valid route
    ids[6, 1] = -1
    perm = O.permute(x, ids, E)
    y = O.combine(perm["x_perm"], perm["row_map"], probs)
    xv = O.bf16_to_f64(x)
    want = np.zeros((T, H))
    for t in range(T):
        for k in range(K):
            if ids[t, k] >= 0:
                want[t] += float(probs[t, k]) * xv[t]
    got = O.bf16_to_f64(y)
    ulp = np.abs(O.bf16_to_f64(_torch_bf16(want))) * 2.0 ** -7 + 1e-30
    assert np.all(np.abs(got - want) <= ulp)
    assert np.all(y[5] == 0)


def test_combine_renorm_all_valid_recovers_token():
    rng = np.random.default_rng(14)
    T, H, E, K = 32, 32, 8, 2
    x = _torch_bf16(rng.standard_normal((T, H)))
    ids, probs = O.route_topk(rng.standard_normal((T, E)).astype(np.float32), K, renorm=True)
    perm = O.permute(x, ids, E)
    y = O.combine(perm["x_perm"], perm["row_map"], probs)
    xv, yv = O.bf16_to_f64(x), O.bf16_to_f64(y)
    assert np.all(np.abs(yv - xv) <= np.abs(xv) * 2.0 ** -7)


def test_combine_respects_k_and_row_map():
    # two tokens, hand-built routes and rows
    yp = _torch_bf16(np.array([[1.0, 2.0], [10.0, 20.0], [100.0, 200.0]]))
    rm = np.array([[2, 0], [-1, 1]], np.int32)
    pr = np.array([[0.5, 0.25], [0.9, 1.0]], np.float32)
    y = O.bf16_to_f64(O.combine(yp, rm, pr))
    assert np.allclose(y, [[50.25, 100.5], [10.0, 20.0]])
