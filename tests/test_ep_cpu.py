"""The expert-parallel layer's exchange logic on the CPU: world_size 2 and 3 over gloo, the
library's kernels replaced by CPU stand-ins built from the oracle (same methods, same tensors),
so that the layer's own code -- group-size exchange, row counts, the row all-to-alls, the
receiving side's expert ids and local permute, the way back and the combine -- runs unchanged.
Every rank's output must equal the oracle's single-process layer on its tokens, bit for bit."""
import os
import socket
import types

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle as O


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, np.uint16).view(np.int16)).view(torch.bfloat16)


class OracleKernels:
    """CPU stand-ins for the library entry points, computed by the oracle."""

    def route_topk(self, logits, K, renorm, id_dtype):
        ids, probs = O.route_topk(logits.numpy(), K, renorm)
        return torch.from_numpy(ids).to(id_dtype), torch.from_numpy(probs)

    def permute(self, x, ids, E, fuse_mxfp8):
        assert not fuse_mxfp8
        op = O.permute(_bits(x), ids.to(torch.int32).numpy(), E)
        return types.SimpleNamespace(x_perm=_bf16(op["x_perm"]), x_perm_scales=None,
                                     group_sizes=torch.from_numpy(op["group_sizes"]),
                                     group_offsets=torch.from_numpy(op["group_offsets"]),
                                     row_map=torch.from_numpy(op["row_map"]), perm_src=torch.from_numpy(op["perm_src"]))

    def recv_expert_ids(self, recv_counts, R_cap):
        return torch.from_numpy(O.ep_recv_expert_ids(recv_counts.numpy(), R_cap))

    def prepare_weights(self, w1, w3, w2, precision):
        return tuple(_bits(w) for w in (w1, w3, w2))

    def swiglu_gemm(self, x_perm, x_scales, weights, group_offsets):
        off = group_offsets.numpy()
        out = np.zeros((x_perm.shape[0], weights[0].shape[1]), np.uint16)
        R = int(off[-1])
        if R:
            ops = [O.Operand(O.MAT_BF16, t) for t in (_bits(x_perm),) + weights]
            out[:R] = O.swiglu_rows(*ops, off, np.arange(R, dtype=np.int32), h_mode=O.H_BF16,
                                    want=("y_bf16",))["y_bf16"]
        return _bf16(out)

    def gather_rows(self, y_perm, row_map):
        return _bf16(O.permute_backward(_bits(y_perm), row_map.numpy()))

    def combine(self, y_perm, row_map, probs):
        return _bf16(O.combine(_bits(y_perm), row_map.numpy(), probs.numpy()))


def _problem(E, H, F, T, world, seed=0):
    g = torch.Generator().manual_seed(seed)
    w = [(torch.randn(s, generator=g) * 0.3).to(torch.bfloat16) for s in ((E, H, F), (E, H, F), (E, F, H))]
    xs = [torch.randn((T, H), generator=g).to(torch.bfloat16) for _ in range(world)]
    bias = torch.randn(E, generator=g) * 1.5            # skew: some ranks' experts get more rows
    lgs = [(torch.randn((T, E), generator=g) + bias).contiguous() for _ in range(world)]
    return w, xs, lgs


def _single(x, lg, w, E, K, renorm):
    """The oracle's single-process layer on one batch."""
    ids, probs = O.route_topk(lg.numpy(), K, renorm)
    op = O.permute(_bits(x), ids, E)
    R = op["R"]
    y_perm = np.zeros_like(op["x_perm"])
    if R:
        ops = [O.Operand(O.MAT_BF16, t) for t in (op["x_perm"],) + tuple(_bits(t) for t in w)]
        y_perm[:R] = O.swiglu_rows(*ops, op["group_offsets"], np.arange(R, dtype=np.int32), h_mode=O.H_BF16,
                                   want=("y_bf16",))["y_bf16"]
    return O.combine(y_perm, op["row_map"], probs)


def _rank(rank, world, port, cfg, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from dropless_moe_expert_router_gb300.ep import ExpertParallelMoE
    E, H, F, T, K, renorm = cfg
    w, xs, lgs = _problem(E, H, F, T, world)
    E_loc = E // world
    mine = [t[rank * E_loc:(rank + 1) * E_loc].contiguous() for t in w]
    layer = ExpertParallelMoE(*mine, E=E, K=K, rank=rank, world=world, renorm=renorm, kernels=OracleKernels())
    y = layer.forward(xs[rank], lgs[rank])
    out[rank] = (_bits(y).copy(), layer.last)
    dist.barrier()
    dist.destroy_process_group()


def _port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("world,E,K,renorm", [(2, 4, 2, True), (3, 6, 2, False)])
def test_ep_forward_over_gloo_equals_single_process_oracle(world, E, K, renorm):
    cfg = (E, 32, 32, 48, K, renorm)
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_rank, args=(world, _port(), cfg, out), nprocs=world, join=True)
    w, xs, lgs = _problem(E, 32, 32, 48, world)
    total_recv = 0
    for r in range(world):
        y, last = out[r]
        assert np.array_equal(y, _single(xs[r], lgs[r], w, E, K, renorm)), r
        assert last["routes"] == sum(last["send_splits"]) == 48 * K
        total_recv += last["received"]
    assert total_recv == world * 48 * K                      # every route went to exactly one rank
