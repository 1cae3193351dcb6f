"""GPU parity of the router backward, the combine backward and the permute backward
with the oracle, through the C ABI. Bars: dlogits within 2e-6 absolute (fp32 softmax
arithmetic against the exact value); dy_perm, dx and dprobs within max|err| / max|ref|
<= 1e-2 (the combine bar; dprobs checked to 1e-3)."""
import numpy as np
import pytest
import torch

import oracle as O
from dropless_moe_expert_router_gb300 import api, workloads as W
from helpers import bf16_bits, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dropless_moe_expert_router_gb300 import build
    build.build()
    api.moe_get_device_errors(clear=True)


def _id_dtype(wl):
    return torch.int16 if wl.id_bits == 16 else torch.int32


def _routes(wl, seed=0):
    lg = W.logits(wl, seed=seed)
    ids, probs = O.route_topk(lg.numpy(), wl.K, wl.renorm)
    bad = W.invalid_mask(wl, seed=seed).numpy()
    ids[bad] = -1
    probs[bad] = 0.0
    return lg, ids, probs


# ------------------------------------------------------------------ router backward
@pytest.mark.parametrize("name", ["tiny", "mixtral", "dsv3", "large_e", "heavy"])
def test_route_backward_matches_oracle(name):
    wl = W.get(name)
    lg, ids, _ = _routes(wl)
    g = W.dprobs(wl)
    d = api.moe_route_topk_backward(lg.cuda(), torch.from_numpy(ids).to(_id_dtype(wl)).cuda(), g.cuda(),
                                    renorm=wl.renorm)
    ref = O.route_backward(lg.numpy(), ids, g.numpy(), wl.renorm)
    assert np.abs(d.cpu().numpy().astype(np.float64) - ref).max() <= 2e-6
    assert api.moe_get_device_errors() == 0


@pytest.mark.parametrize("T,E,K,renorm", [(1, 1, 1, False), (5, 3, 3, True), (33, 64, 7, False),
                                          (17, 300, 36, True), (9, 2304, 128, False), (8, 40, 40, True)])
def test_route_backward_edge_shapes_duplicates_and_invalid(T, E, K, renorm):
    """Random (not top-K) ids with repeats and -1 entries: the oracle's set semantics
    (a repeated expert's gradients summed once, counted once in a renormalised denominator)."""
    rng = np.random.default_rng(T * 31 + E)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    ids = rng.integers(-1, E, (T, K)).astype(np.int32)
    ids[0, :] = ids[0, 0]                       # one row: a single expert repeated
    g = rng.standard_normal((T, K)).astype(np.float32)
    for dt in (torch.int32, torch.int16):
        d = api.moe_route_topk_backward(torch.from_numpy(lg).cuda(), torch.from_numpy(ids).to(dt).cuda(),
                                        torch.from_numpy(g).cuda(), renorm=renorm)
        ref = O.route_backward(lg, ids, g, renorm)
        assert np.abs(d.cpu().numpy().astype(np.float64) - ref).max() <= 2e-6


# ------------------------------------------------------------------ combine / permute backward
@pytest.mark.parametrize("name", ["tiny", "mixtral", "dsv3", "large_e"])
def test_combine_backward_matches_oracle(name):
    wl = W.get(name)
    _, ids, probs = _routes(wl)
    op = O.permute(None, ids, wl.E)
    rm, R = op["row_map"], op["R"]
    yp = W.expert_out(wl)
    dy = W.dy(wl)
    dyp, dpr = api.moe_unpermute_combine_backward(dy.cuda(), yp.cuda(), torch.from_numpy(rm).cuda(),
                                                  torch.from_numpy(probs).cuda())
    ref_dyp, ref_dpr = O.combine_backward(bf16_bits(dy), bf16_bits(yp), rm, probs)
    got = O.bf16_to_f64(bf16_bits(dyp)[:R])
    assert rel_err(got, O.bf16_to_f64(ref_dyp[:R])) <= 1e-2
    assert rel_err(dpr.cpu().numpy().astype(np.float64), ref_dpr) <= 1e-3
    assert np.all(dpr.cpu().numpy()[rm < 0] == 0.0)


@pytest.mark.parametrize("name", ["tiny", "mixtral", "dsv3", "large_e"])
def test_permute_backward_matches_oracle(name):
    wl = W.get(name)
    _, ids, _ = _routes(wl)
    op = O.permute(None, ids, wl.E)
    rm = op["row_map"]
    dxp = W.expert_out(wl, seed=3)
    dx = api.moe_permute_backward(dxp.cuda(), torch.from_numpy(rm).cuda())
    ref = O.permute_backward(bf16_bits(dxp), rm)
    assert rel_err(O.bf16_to_f64(bf16_bits(dx)), O.bf16_to_f64(ref)) <= 1e-2
    if wl.K <= 2:
        # two bf16 values add exactly in fp32: the single rounding matches the oracle's
        assert np.array_equal(bf16_bits(dx), ref)


def test_combine_backward_all_routes_invalid_and_single_token():
    wl = W.get("tiny", T=1, H=64)
    rm = np.full((1, wl.K), -1, np.int32)
    probs = np.zeros((1, wl.K), np.float32)
    yp = W.expert_out(wl)
    dy = W.dy(wl)
    dyp, dpr = api.moe_unpermute_combine_backward(dy.cuda(), yp.cuda(), torch.from_numpy(rm).cuda(),
                                                  torch.from_numpy(probs).cuda())
    assert np.all(dpr.cpu().numpy() == 0.0)
    dx = api.moe_permute_backward(yp.cuda(), torch.from_numpy(rm).cuda())
    assert torch.count_nonzero(dx.float()).item() == 0


@pytest.mark.parametrize("name,over", [("tiny", {}), ("tiny", {"H": 96}), ("tiny", {"H": 2080, "T": 77}),
                                       ("mixtral", {"T": 1024}), ("dsv3", {"T": 512}), ("heavy", {"T": 256})])
def test_combine_backward_fused_mxfp8_matches_oracle(name, over):
    """The combine backward's row-wise MXFP8 codes and scales of dy_perm: with power-of-two
    probabilities p * dy is exact, so dy_perm equals the oracle's bit for bit and its codes
    and scales must equal the oracle's row quantiser of the oracle's dy_perm. H = 96 and
    2080 leave a ragged last slice of the row (not a multiple of 256 columns)."""
    wl = W.get(name, **over)
    _, ids, _ = _routes(wl)
    rng = np.random.default_rng(7)
    probs = np.where(ids >= 0, 2.0 ** -rng.integers(0, 5, ids.shape), 0.0).astype(np.float32)
    op = O.permute(None, ids, wl.E)
    rm, R = op["row_map"], op["R"]
    yp = W.expert_out(wl)
    dy = W.dy(wl)
    R_cap, H = yp.shape
    q = torch.zeros((R_cap, H), dtype=torch.uint8, device="cuda")
    s = torch.zeros((R_cap, H // 32), dtype=torch.uint8, device="cuda")
    dyp, dpr = api.moe_unpermute_combine_backward(dy.cuda(), yp.cuda(), torch.from_numpy(rm).cuda(),
                                                  torch.from_numpy(probs).cuda(), dy_perm_q=q, dy_perm_scales=s)
    ref_dyp, ref_dpr = O.combine_backward(bf16_bits(dy), bf16_bits(yp), rm, probs)
    assert np.array_equal(bf16_bits(dyp)[:R], ref_dyp[:R])
    ref_q, ref_s = O.quant_rows(ref_dyp[:R])
    assert np.array_equal(q.cpu().numpy()[:R], ref_q)
    assert np.array_equal(s.cpu().numpy()[:R], ref_s)
    assert rel_err(dpr.cpu().numpy().astype(np.float64), ref_dpr) <= 1e-3
    assert api.moe_get_device_errors() == 0


def test_combine_backward_fused_mxfp8_argument_errors():
    wl = W.get("tiny", H=72)                    # H % 32 != 0: no 1x32 blocks
    _, ids, probs = _routes(wl)
    rm = O.permute(None, ids, wl.E)["row_map"]
    yp = W.expert_out(wl).cuda()
    q = torch.zeros(yp.shape, dtype=torch.uint8, device="cuda")
    s = torch.zeros((yp.shape[0], 2), dtype=torch.uint8, device="cuda")
    with pytest.raises(Exception):
        api.moe_unpermute_combine_backward(W.dy(wl).cuda(), yp, torch.from_numpy(rm).cuda(),
                                           torch.from_numpy(probs).cuda(), dy_perm_q=q, dy_perm_scales=s)
    with pytest.raises(ValueError):
        api.moe_unpermute_combine_backward(W.dy(wl).cuda(), yp, torch.from_numpy(rm).cuda(),
                                           torch.from_numpy(probs).cuda(), dy_perm_q=q)
