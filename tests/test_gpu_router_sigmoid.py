"""GPU parity of the sigmoid-score router (selection on sigmoid(logit) + expert bias) and of
its backward with the oracle, through the C ABI.

Bars: ids equal to the oracle's in every row (both sides decide on the logistic rounded once to
fp32 from its exact value); probs within 1e-6 absolute; dlogits within 2e-6 absolute."""
import numpy as np
import pytest
import torch

import oracle as O
from dropless_moe_expert_router_gb300 import api, workloads as W
from dropless_moe_expert_router_gb300.api import MoeError

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dropless_moe_expert_router_gb300 import build
    build.build()
    api.moe_get_device_errors(clear=True)


def _inputs(T, E, seed, bias_scale=0.05, logit_scale=1.0):
    rng = np.random.default_rng(seed)
    lg = (rng.standard_normal((T, E)) * logit_scale).astype(np.float32)
    b = None if bias_scale is None else rng.uniform(-bias_scale, bias_scale, E).astype(np.float32)
    return lg, b


def _check(lg, b, K, renorm, ids_gpu, probs_gpu):
    ref_ids, ref_p = O.route_sigmoid_topk(lg, K, bias=b, renorm=renorm)
    assert np.array_equal(ids_gpu.astype(np.int64), ref_ids)
    assert np.abs(probs_gpu - ref_p).max(initial=0.0) <= 1e-6
    return ref_ids


@pytest.mark.parametrize("T,E,K,renorm,bias,i16", [
    (4096, 256, 8, True, 0.05, False),      # DeepSeek-V3 router shape
    (8192, 32, 4, True, 0.05, False),       # the dsv3_sigmoid workload's router
    (1000, 1024, 64, False, 0.02, False),   # largest E and K of this path
    (777, 100, 40, True, 0.1, True),        # K > 32: two output slots per lane; ragged E
    (333, 33, 33, False, None, True),       # K = E, no bias
    (5, 1, 1, True, 0.3, False),            # one expert
])
def test_sigmoid_router_matches_oracle(T, E, K, renorm, bias, i16):
    lg, b = _inputs(T, E, seed=T + E, bias_scale=bias)
    dt = torch.int16 if i16 else torch.int32
    ids, probs = api.moe_route_sigmoid_topk(torch.from_numpy(lg).cuda(), K,
                                            expert_bias=None if b is None else torch.from_numpy(b).cuda(),
                                            id_dtype=dt, renorm=renorm)
    assert ids.dtype == dt
    _check(lg, b, K, renorm, ids.cpu().numpy(), probs.cpu().numpy())
    assert api.moe_get_device_errors() == 0


@pytest.mark.parametrize("T,E,K,spread", [(2048, 256, 8, 1e-6), (1024, 1000, 40, 3e-6), (4096, 32, 4, 2e-7)])
def test_sigmoid_router_near_ties_are_exact(T, E, K, spread):
    """Logits packed into a tiny interval: scores a few fp32 ulp apart, where an fp32 logistic
    alone would order some of them differently from the exactly rounded one."""
    rng = np.random.default_rng(T + E)
    lg = (0.3 + spread * rng.random((T, E))).astype(np.float32)
    b = (rng.integers(-2, 3, E) * 6e-8).astype(np.float32)          # biases of a few ulp
    ids, probs = api.moe_route_sigmoid_topk(torch.from_numpy(lg).cuda(), K, expert_bias=torch.from_numpy(b).cuda())
    _check(lg, b, K, False, ids.cpu().numpy(), probs.cpu().numpy())
    assert api.moe_get_device_errors() == 0


def test_sigmoid_router_ties_and_saturated_scores_are_exact():
    """Equal logits and biases: ties go to the lower index. Logits of +inf and 40 give a score
    of exactly 1 in fp32 on both sides (and -inf exactly 0), so those keys tie as well."""
    T, E, K = 64, 48, 6
    lg = np.full((T, E), 0.25, np.float32)
    lg[1::2, ::3] = np.inf
    lg[2::4, 5::7] = -np.inf
    lg[3::4, 1::5] = 40.0
    lg[3::4, 2::5] = -40.0
    b = np.zeros(E, np.float32)
    b[7] = 2.0                                   # expert 7 always first
    ids, probs = api.moe_route_sigmoid_topk(torch.from_numpy(lg).cuda(), K, expert_bias=torch.from_numpy(b).cuda())
    ref_ids, ref_p = O.route_sigmoid_topk(lg, K, bias=b)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    assert np.abs(probs.cpu().numpy() - ref_p).max() <= 1e-6
    assert np.all(ref_ids[:, 0] == 7)


def test_sigmoid_router_layer_stage_and_bias_statistics():
    """The layer's sigmoid router gives the API's routes, and its expert load (the permute's
    group sizes) is the oracle's count of valid routes per expert."""
    from dropless_moe_expert_router_gb300.layer import MoELayer
    wl = W.get("dsv3_sigmoid", T=512, H=512, F=512, E=16)
    w1, w3, w2 = (t.cuda() for t in W.weights(wl))
    eb = W.expert_bias(wl)
    layer = MoELayer(w1, w3, w2, T=wl.T, K=wl.K, precision=wl.precision, renorm=wl.renorm, score="sigmoid",
                     expert_bias=eb.cuda())
    lg = W.logits(wl)
    x = W.x(wl)
    layer.forward(x.cuda(), lg.cuda())
    torch.cuda.synchronize()
    ref_ids = _check(lg.numpy(), eb.numpy(), wl.K, wl.renorm, layer.ids.cpu().numpy(), layer.probs.cpu().numpy())
    op = O.permute(None, ref_ids, wl.E)
    assert np.array_equal(layer.expert_load.cpu().numpy(), op["group_sizes"])
    with pytest.raises(ValueError):
        MoELayer(w1, w3, w2, T=wl.T, K=wl.K, precision=wl.precision, expert_bias=eb.cuda())


@pytest.mark.parametrize("renorm", [False, True])
@pytest.mark.parametrize("T,E,K", [(4096, 256, 8), (300, 1024, 64), (77, 40, 40)])
def test_sigmoid_router_backward_matches_oracle(T, E, K, renorm):
    lg, b = _inputs(T, E, seed=3 * T + E)
    ids, _ = O.route_sigmoid_topk(lg, K, bias=b, renorm=renorm)
    g = np.random.default_rng(T).standard_normal((T, K)).astype(np.float32)
    d = api.moe_route_sigmoid_topk_backward(torch.from_numpy(lg).cuda(), torch.from_numpy(ids).cuda(),
                                            torch.from_numpy(g).cuda(), renorm=renorm)
    ref = O.route_sigmoid_backward(lg, ids, g, renorm)
    assert np.abs(d.cpu().numpy().astype(np.float64) - ref).max() <= 2e-6


@pytest.mark.parametrize("renorm", [False, True])
def test_sigmoid_router_backward_duplicates_and_invalid(renorm):
    """Random ids with repeats and -1 entries: set semantics (a repeated expert once, its
    gradients summed), invalid routes skipped, int16 and int32 ids."""
    rng = np.random.default_rng(11)
    T, E, K = 65, 70, 37
    lg = rng.standard_normal((T, E)).astype(np.float32)
    ids = rng.integers(-1, E, (T, K)).astype(np.int32)
    ids[0, :] = ids[0, 0]
    ids[1, :] = -1
    g = rng.standard_normal((T, K)).astype(np.float32)
    ref = O.route_sigmoid_backward(lg, ids, g, renorm)
    for dt in (torch.int32, torch.int16):
        d = api.moe_route_sigmoid_topk_backward(torch.from_numpy(lg).cuda(), torch.from_numpy(ids).to(dt).cuda(),
                                                torch.from_numpy(g).cuda(), renorm=renorm)
        assert np.abs(d.cpu().numpy().astype(np.float64) - ref).max() <= 2e-6


def test_sigmoid_router_limits_are_status_codes():
    lg = torch.zeros((4, 1025), device="cuda")
    with pytest.raises(MoeError):
        api.moe_route_sigmoid_topk(lg, 2)                    # E > 1024: unsupported
    with pytest.raises(MoeError):
        api.moe_route_sigmoid_topk(lg[:, :100].contiguous(), 65)   # K > 64: unsupported
    with pytest.raises(MoeError):
        api.moe_route_sigmoid_topk(lg[:, :8].contiguous(), 9)      # K > E
    assert api.moe_get_device_errors() == 0
