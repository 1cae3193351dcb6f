"""The whole layer (forward, and forward + backward) is capturable in one CUDA
graph and its replays follow new routing without re-capture (group sizes stay
on the device); the GEMM's bounded waits give up and report instead of
hanging; bad routes are flagged, not trapped."""
import numpy as np
import pytest
import torch

import oracle as O
from dropless_moe_expert_router_gb300 import api, workloads as W
from dropless_moe_expert_router_gb300.layer import MoELayer
from helpers import bf16_bits, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dropless_moe_expert_router_gb300 import build
    build.build()
    api.moe_get_device_errors(clear=True)


def _layer(wl, training=False):
    w1, w3, w2 = (t.cuda() for t in W.weights(wl))
    return MoELayer(w1, w3, w2, T=wl.T, K=wl.K, precision=wl.precision, renorm=wl.renorm, training=training)


@pytest.mark.parametrize("name,overrides", [("tiny", {}), ("mixtral", dict(T=2048, H=1024, F=2048))])
def test_forward_graph_replays_follow_new_routes(name, overrides):
    wl = W.get(name, **overrides)
    layer = _layer(wl)
    x = W.x(wl).cuda()
    lg_static = W.logits(wl, seed=0).cuda()
    layer.forward(x, lg_static)              # warm-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):                # global capture mode: a host sync would fail it
        y_graph = layer.forward(x, lg_static)
    sizes = set()
    for seed in (1, 2, 3):
        lg = W.logits(wl, seed=seed).cuda()
        lg_static.copy_(lg)
        g.replay()
        torch.cuda.synchronize()
        got = y_graph.clone()
        sizes.add(tuple(layer.perm.group_sizes.cpu().tolist()))
        # eager run on the same inputs gives the same bits (deterministic kernels)
        ref = layer.forward(x, lg).clone()
        torch.cuda.synchronize()
        assert torch.equal(got, ref)
        if name == "tiny":
            # and matches the oracle layer output
            ids, probs = O.route_topk(lg.cpu().numpy(), wl.K, wl.renorm)
            op = O.permute(bf16_bits(x), ids, wl.E)
            Ws = [O.Operand(O.MAT_BF16, bf16_bits(t)) for t in W.weights(wl)]
            R = op["R"]
            out = O.swiglu_rows(O.Operand(O.MAT_BF16, op["x_perm"]), *Ws, op["group_offsets"],
                                np.arange(R, dtype=np.int32), want=("y_bf16",))
            yp = np.zeros((wl.R_cap, wl.H), np.uint16)
            yp[:R] = out["y_bf16"]
            yo = O.combine(yp, op["row_map"], probs)
            assert rel_err(O.bf16_to_f64(bf16_bits(got)), O.bf16_to_f64(yo)) <= 1e-2
    assert len(sizes) == 3, "replays should see different group sizes"
    assert api.moe_get_device_errors() == 0


def test_training_step_graph_matches_eager():
    wl = W.get("tiny", T=512, H=256, F=256)
    layer = _layer(wl, training=True)
    x = W.x(wl).cuda()
    lg = W.logits(wl).cuda()
    dy = W.dy_perm(wl).cuda()

    def step():
        layer.forward(x, lg)
        return layer.backward(x, dy)
    step()
    torch.cuda.synchronize()
    eager = [t.clone() for t in step()]
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        outs = step()
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(outs, eager):
        assert torch.equal(a, b)


@pytest.mark.parametrize("precision", ["bf16", "mxfp8"])
def test_full_layer_backward_graph_matches_eager(precision):
    """Forward + the whole layer's backward (combine, expert MLP, permute and router backward)
    captured in one graph: replays give the eager results bit for bit. MXFP8: the combine
    backward's fused quantisation of dy_perm feeds the dgrad exactly as the separate row
    quantiser would."""
    hf = 512 if precision == "mxfp8" else 256    # MXFP8 GEMMs take H, F in multiples of 512
    wl = W.get("tiny", T=512, H=hf, F=hf, precision=precision)
    layer = _layer(wl, training=True)
    x = W.x(wl).cuda()
    lg = W.logits(wl).cuda()
    dy = W.dy(wl).cuda()

    def step():
        layer.forward(x, lg)
        return layer.backward_full(x, lg, dy)
    step()
    torch.cuda.synchronize()
    eager = [t.clone() for t in step()]
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        outs = step()
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(outs, eager):
        assert torch.equal(a, b)
    # the pieces compose: dx is the permute backward of the expert backward's dx_perm
    assert torch.equal(outs[0], api.moe_permute_backward(layer.dx, layer.perm.row_map))
    if precision == "mxfp8":
        dab = layer.dab.clone()
        q, sc = layer.dy_q.clone(), layer.dy_s.clone()
        layer.stage_dgrad_dh(layer.dy_perm, dy_quantised=False)
        torch.cuda.synchronize()
        R = int(layer.perm.group_offsets[-1].item())
        assert torch.equal(layer.dy_q[:R], q[:R]) and torch.equal(layer.dy_s[:R], sc[:R])
        assert torch.equal(layer.dab, dab)


def test_bounded_wait_gives_up_and_reports():
    api.moe_get_device_errors(clear=True)
    api.moe_debug_bounded_wait_selftest(20000)          # 20 ms on a barrier nothing arrives on
    errs = api.moe_get_device_errors(clear=True)
    assert errs & api.MOE_DEVERR_TIMEOUT
    # the context is still usable afterwards
    lg = torch.randn(64, 8, device="cuda")
    ids, _ = api.moe_route_topk(lg, 2)
    torch.cuda.synchronize()
    assert torch.equal(ids.long().cpu(), torch.topk(lg.cpu(), 2, dim=1).indices)


def test_argument_errors_come_back_as_status_codes():
    x = torch.zeros((8, 30), dtype=torch.bfloat16, device="cuda")      # H % 32 != 0
    ids = torch.zeros((8, 2), dtype=torch.int32, device="cuda")
    with pytest.raises(api.MoeError) as ei:
        api.moe_permute(x, ids, 4)
    assert ei.value.status == 1
    lg = torch.zeros((8, 4), device="cuda")
    with pytest.raises(api.MoeError):
        api.moe_route_topk(lg, 5)                                       # K > E


@pytest.mark.parametrize("precision", ["bf16", "mxfp8", "nvfp4"])
def test_forward_host_transfers_give_the_device_result(precision):
    """forward_host from page-locked host tensors, every transfer: overlapped (two sets of device
    buffers in turn, copies on the layer's own streams), sliced (three token slices, each through
    the whole layer), direct access (the permute reads x and the combine writes y in host memory
    through their device addresses) and plain copies. Each result equals the device forward's bit
    for bit once host_event has completed, also for back-to-back overlapped calls on different
    batches with no synchronisation between them; pageable memory is refused where page-locked
    memory is required."""
    from dropless_moe_expert_router_gb300.layer import MoELayer
    HF = 512 if precision != "bf16" else 256
    wl = W.get("tiny", T=301, H=HF, F=HF, E=8, K=2, precision=precision)
    w1, w3, w2 = (t.cuda() for t in W.weights(wl))
    layer = MoELayer(w1, w3, w2, T=wl.T, K=wl.K, precision=precision)
    xs = [W.x(wl, seed=s) for s in range(3)]
    lgs = [W.logits(wl, seed=s) for s in range(3)]
    refs = [layer.forward(x.cuda(), lg.cuda()).clone().cpu() for x, lg in zip(xs, lgs)]
    x, lg, ref = xs[0], lgs[0], refs[0]
    xh, lh = x.pin_memory(), lg.pin_memory()
    yh = torch.empty((wl.T, wl.H), dtype=torch.bfloat16).pin_memory()
    nv4 = precision == "nvfp4"
    for transfer in ["copy", "auto", "overlapped"] + ([] if nv4 else ["sliced", "sliced", "direct"]):
        yh.fill_(7)
        layer.forward_host(xh, lh, yh, transfer=transfer)
        layer.host_event.synchronize()
        assert torch.equal(yh, ref), transfer
    # back-to-back overlapped calls on three batches, twice round, each into its own output
    xhs = [t.pin_memory() for t in xs]
    lhs = [t.pin_memory() for t in lgs]
    yhs = [torch.full((wl.T, wl.H), 7, dtype=torch.bfloat16).pin_memory() for _ in range(6)]
    for j in range(6):
        layer.forward_host(xhs[j % 3], lhs[j % 3], yhs[j], transfer="overlapped")
    torch.cuda.synchronize()
    for j in range(6):
        assert torch.equal(yhs[j], refs[j % 3]), j
    if nv4:                      # slices would change the amax scaling of x and h: refused
        for transfer in ("sliced", "direct"):
            with pytest.raises(ValueError):
                layer.forward_host(xh, lh, yh, transfer=transfer)
    else:
        sizes = layer._slices()[0]
        assert sum(sizes) == wl.T and len(sizes) == 3
        assert api.moe_host_mapped_pointer(xh) is not None
        assert api.moe_host_mapped_pointer(torch.empty((4, 8), dtype=torch.bfloat16)) is None   # pageable
    for transfer in ("overlapped", "sliced", "direct"):
        with pytest.raises(ValueError):
            layer.forward_host(x, lg, torch.empty_like(x), transfer=transfer)
    yc = torch.empty_like(x)                                    # pageable: "auto" copies
    layer.forward_host(x, lg, yc)
    torch.cuda.synchronize()
    assert torch.equal(yc, ref)
    assert api.moe_get_device_errors() == 0
