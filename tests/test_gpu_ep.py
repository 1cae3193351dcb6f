"""GPU parity of the expert-parallel forward, through the C ABI.

- moe_ep_recv_expert_ids bit-exact against the oracle (ranks x local experts up to the pages'
  72 x 32, empty segments, spare capacity, a capacity that cuts the last segment).
- G ranks emulated in this one process on this one GPU, a thread per rank: the layer's
  all-to-alls move slices by device copies after a host barrier (no kernel waits on another).
  Every rank's output equals the single-GPU layer's on its tokens (each row meets the same
  expert with the same operands), bf16 and MXFP8, and is within the oracle tolerance of the
  oracle's single-process layer on the small shapes.
- One rank over NCCL (the real exchange code path, a world of one) equals the single-GPU layer."""
import os
import socket
import threading

import numpy as np
import pytest
import torch

import oracle as O
from dropless_moe_expert_router_gb300 import api, workloads as W
from dropless_moe_expert_router_gb300.ep import ExpertParallelMoE
from dropless_moe_expert_router_gb300.layer import MoELayer
from helpers import bf16_bits, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dropless_moe_expert_router_gb300 import build
    build.build()
    api.moe_get_device_errors(clear=True)


@pytest.mark.parametrize("G,E_loc,scale,R_extra", [(72, 32, 30, 100), (1, 8, 500, 0), (5, 3, 4, 17), (3, 4, 0, 9)])
def test_recv_expert_ids_match_oracle(G, E_loc, scale, R_extra):
    rng = np.random.default_rng(G * 100 + E_loc)
    counts = rng.integers(0, scale + 1, (G, E_loc)).astype(np.int32)
    counts[rng.random((G, E_loc)) < 0.2] = 0                  # empty segments
    total = int(counts.sum())
    for R_cap in (total + R_extra, max(0, total - 7)):
        got = api.moe_ep_recv_expert_ids(torch.from_numpy(counts).cuda(), R_cap)
        assert np.array_equal(got.cpu().numpy(), O.ep_recv_expert_ids(counts, R_cap))
    assert api.moe_get_device_errors() == 0


class _Shared:
    def __init__(self, G):
        self.G = G
        self.slots = [None] * G
        self.barrier = threading.Barrier(G, timeout=120)


class EmulatedComm:
    """All-to-all among G ranks that are threads of this process on one GPU: each rank posts its
    input once its stream has finished writing it, all meet at a host barrier, each copies its
    slices from every source, and all meet again before any input is reused."""

    def __init__(self, shared, rank):
        self.s, self.rank = shared, rank

    def all_to_all(self, out, inp, out_splits=None, in_splits=None):
        s, G = self.s, self.s.G
        if in_splits is None:
            in_splits = [inp.shape[0] // G] * G
        torch.cuda.current_stream().synchronize()
        s.slots[self.rank] = (inp, list(in_splits))
        s.barrier.wait()
        o = 0
        for src in range(G):
            sinp, sp = s.slots[src]
            start, n = sum(sp[:self.rank]), sp[self.rank]
            out[o:o + n].copy_(sinp[start:start + n])
            o += n
        assert o == out.shape[0]
        torch.cuda.current_stream().synchronize()
        s.barrier.wait()


def _run_emulated(G, wl, precision, w, xs, lgs):
    E_loc = wl.E // G
    shared = _Shared(G)
    layers = [ExpertParallelMoE(*(t[r * E_loc:(r + 1) * E_loc].contiguous().cuda() for t in w), E=wl.E, K=wl.K,
                                rank=r, world=G, precision=precision, renorm=wl.renorm,
                                comm=EmulatedComm(shared, r)) for r in range(G)]
    outs, errs = [None] * G, [None] * G

    def body(r):
        try:
            torch.cuda.set_device(0)
            outs[r] = layers[r].forward(xs[r].cuda(), lgs[r].cuda())
            torch.cuda.current_stream().synchronize()
        except BaseException as e:              # reported by the main thread
            errs[r] = e
            shared.barrier.abort()

    th = [threading.Thread(target=body, args=(r,)) for r in range(G)]
    for t in th:
        t.start()
    for t in th:
        t.join()
    for e in errs:
        if e is not None:
            raise e
    return outs, layers


def _single_gpu(wl, precision, w, x, lg):
    layer = MoELayer(*(t.cuda() for t in w), T=wl.T, K=wl.K, precision=precision, renorm=wl.renorm)
    y = layer.forward(x.cuda(), lg.cuda()).clone()
    torch.cuda.synchronize()
    return y


def _oracle_layer(wl, precision, w, x, lg):
    ids, probs = O.route_topk(lg.numpy(), wl.K, wl.renorm)
    op = O.permute(bf16_bits(x), ids, wl.E)
    R, off = op["R"], op["group_offsets"]
    rows = np.arange(R, dtype=np.int32)
    if precision == "mxfp8":
        def along(t):   # [E, Kc, N] with blocks along Kc
            qs, ss = zip(*(O.quant_rows(np.ascontiguousarray(bf16_bits(t[e]).T)) for e in range(t.shape[0])))
            return O.Operand(O.MAT_MXFP8, np.ascontiguousarray(np.stack(qs).transpose(0, 2, 1)),
                             np.ascontiguousarray(np.stack(ss).transpose(0, 2, 1)))
        xq, xs = O.quant_rows(op["x_perm"])
        ops = [O.Operand(O.MAT_MXFP8, xq, xs)] + [along(t) for t in w]
        hm = O.H_MXFP8
    else:
        ops = [O.Operand(O.MAT_BF16, op["x_perm"])] + [O.Operand(O.MAT_BF16, bf16_bits(t)) for t in w]
        hm = O.H_BF16
    y_perm = np.zeros_like(op["x_perm"])
    y_perm[:R] = O.swiglu_rows(*ops, off, rows, h_mode=hm, want=("y_bf16",))["y_bf16"]
    return O.combine(y_perm, op["row_map"], probs)


@pytest.mark.parametrize("G,precision", [(2, "bf16"), (4, "bf16"), (2, "mxfp8"), (4, "mxfp8")])
def test_ep_emulated_ranks_equal_single_gpu_layer_and_oracle(G, precision):
    HF = 512 if precision == "mxfp8" else 256
    wl = W.get("tiny", T=256, H=HF, F=HF, E=8, K=2, precision=precision, bias="normal", bias_scale=1.0,
               renorm=True)
    w = W.weights(wl)
    xs = [W.x(wl, seed=r) for r in range(G)]
    lgs = [W.logits(wl, seed=r) for r in range(G)]
    outs, layers = _run_emulated(G, wl, precision, w, xs, lgs)
    tol = 3e-2 if precision == "mxfp8" else 1e-2
    for r in range(G):
        assert torch.equal(outs[r], _single_gpu(wl, precision, w, xs[r], lgs[r])), r
        ref = _oracle_layer(wl, precision, w, xs[r], lgs[r])
        assert rel_err(O.bf16_to_f64(bf16_bits(outs[r])), O.bf16_to_f64(ref)) <= tol
    assert sum(l.last["received"] for l in layers) == G * wl.T * wl.K
    assert api.moe_get_device_errors() == 0


def test_ep_emulated_dsv3_shape_mxfp8_four_ranks():
    """The DeepSeek-V3-like slice (T=8192 per rank, H=7168, E=32 -> 8 per rank, top-4, F=2048,
    Zipf-skewed routing with empty experts) over four emulated ranks equals the single-GPU layer."""
    wl = W.get("dsv3")
    G = 4
    w = W.weights(wl)
    xs = [W.x(wl, seed=r) for r in range(G)]
    lgs = [W.logits(wl, seed=r) for r in range(G)]
    outs, layers = _run_emulated(G, wl, "mxfp8", w, xs, lgs)
    for r in range(G):
        assert torch.equal(outs[r], _single_gpu(wl, "mxfp8", w, xs[r], lgs[r])), r
    recv = [l.last["received"] for l in layers]
    assert sum(recv) == G * wl.T * wl.K and recv[0] > recv[-1]      # the skew lands on rank 0's experts
    assert api.moe_get_device_errors() == 0


def test_ep_one_rank_over_nccl_equals_single_gpu_layer():
    import torch.distributed as dist
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1,
                            device_id=torch.device("cuda", 0))
    try:
        wl = W.get("tiny", T=512, H=256, F=512, E=8, K=2)
        w = W.weights(wl)
        layer = ExpertParallelMoE(*(t.cuda() for t in w), E=wl.E, K=wl.K, rank=0, world=1)
        x, lg = W.x(wl), W.logits(wl)
        y = layer.forward(x.cuda(), lg.cuda())
        torch.cuda.synchronize()
        assert torch.equal(y, _single_gpu(wl, "bf16", w, x, lg))
    finally:
        dist.destroy_process_group()
    assert api.moe_get_device_errors() == 0
