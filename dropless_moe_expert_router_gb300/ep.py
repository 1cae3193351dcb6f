"""Expert-parallel forward of the dropless MoE layer: G ranks, one process per GPU, each rank
holding E/G of the experts and its own batch of tokens.

"Dropless MoE acceleration in JAX with NVIDIA Transformer Engine", section "Optimization 2:
Expert parallelism to fuse Dispatch and Combine"; "Sparser MoE end-to-end", section "Remove work
that has no selected route" (only selected routes travel, as a compact [T, K] route list; the
destination works only on its own experts' rows; the source pulls its rows back and reduces
them with its probabilities).

Rank g owns experts g*E_loc .. g*E_loc + E_loc - 1. One forward:

1. route and permute on the source (the library's kernels): the rows of every destination's
   experts are contiguous in the expert-contiguous order;
2. exchange the group sizes (an all-to-all of E int32 per rank) and read the per-rank row
   counts on the host -- the one device-to-host copy of this path (2 E int32), which sizes the
   row exchange;
3. exchange the rows (an all-to-all of bf16 rows, only selected routes);
4. on the destination: the local expert of each received row (moe_ep_recv_expert_ids), then
   moe_permute of the received rows with those ids (K = 1, E_loc experts; fused MXFP8 for the
   MXFP8 layer) gives the local experts' contiguous order; the grouped SwiGLU GEMMs;
5. the received order back (moe_permute_backward with K = 1 gathers each row's result);
6. exchange the rows back (the reverse all-to-all): every source has its rows in its own
   permuted order again;
7. combine on the source with its probabilities (moe_unpermute_combine).

Every arithmetic step runs in the library's kernels; the exchanges are torch.distributed
all-to-alls (NCCL between GPUs). Each row meets the same expert with the same operands as in
the single-GPU layer. Forward only; the row counts read on the host make this path, unlike the
single-GPU layer, not capturable in one CUDA graph.
"""
from __future__ import annotations

from typing import List, Optional

import torch

from . import api


class TorchComm:
    """The exchanges over a torch.distributed process group (NCCL on GPUs, gloo on the CPU)."""

    def __init__(self, group=None):
        self.group = group

    def all_to_all(self, out: torch.Tensor, inp: torch.Tensor, out_splits: Optional[List[int]] = None,
                   in_splits: Optional[List[int]] = None) -> None:
        import torch.distributed as dist
        dist.all_to_all_single(out, inp, out_splits, in_splits, group=self.group)


class LibraryKernels:
    """The library entry points the expert-parallel layer calls (a test may pass CPU stand-ins
    with the same methods to check the exchange logic without a GPU)."""

    def route_topk(self, logits, K, renorm, id_dtype):
        return api.moe_route_topk(logits, K, renorm=renorm, id_dtype=id_dtype)

    def permute(self, x, ids, E, fuse_mxfp8):
        return api.moe_permute(x, ids, E, fuse_mxfp8=fuse_mxfp8)

    def recv_expert_ids(self, recv_counts, R_cap):
        return api.moe_ep_recv_expert_ids(recv_counts, R_cap)

    def prepare_weights(self, w1, w3, w2, precision):
        return api.moe_prepare_weights(w1, w3, w2, precision)

    def swiglu_gemm(self, x_perm, x_scales, weights, group_offsets):
        return api.moe_grouped_swiglu_gemm(x_perm, x_scales, weights, group_offsets)[0]

    def gather_rows(self, y_perm, row_map):
        return api.moe_permute_backward(y_perm, row_map)

    def combine(self, y_perm, row_map, probs):
        return api.moe_unpermute_combine(y_perm, row_map, probs)


class ExpertParallelMoE:
    """This rank's share of an expert-parallel MoE layer.

    w1, w3 [E_loc, H, F] and w2 [E_loc, F, H]: the weights of this rank's experts
    (rank * E_loc ...), E the experts of the whole layer (E % world == 0)."""

    def __init__(self, w1: torch.Tensor, w3: torch.Tensor, w2: torch.Tensor, *, E: int, K: int, rank: int,
                 world: int, precision: str = "bf16", renorm: bool = False, id_dtype=torch.int32,
                 comm=None, kernels=None):
        E_loc, H, F = w1.shape
        if E % world or E // world != E_loc:
            raise ValueError(f"{E} experts over {world} ranks: each rank holds E / world = {E // world}, got {E_loc}")
        if precision not in ("bf16", "mxfp8"):
            raise ValueError("precision must be 'bf16' or 'mxfp8'")
        self.E, self.E_loc, self.H, self.F, self.K = E, E_loc, H, F, K
        self.rank, self.world = rank, world
        self.precision, self.renorm, self.id_dtype = precision, renorm, id_dtype
        self.comm = comm if comm is not None else TorchComm()
        self.k = kernels if kernels is not None else LibraryKernels()
        self.weights = self.k.prepare_weights(w1, w3, w2, precision)
        self.last = {}

    def forward(self, x: torch.Tensor, logits: torch.Tensor) -> torch.Tensor:
        """x [T, H] bf16 and logits [T, E] fp32 of this rank's tokens -> y [T, H] bf16."""
        k, G, E_loc, H = self.k, self.world, self.E_loc, self.H
        T = x.shape[0]
        dev = x.device
        # 1. route and permute on the source (bf16 rows travel)
        ids, probs = k.route_topk(logits, self.K, self.renorm, self.id_dtype)
        p = k.permute(x, ids, self.E, False)
        # 2. group sizes to their experts' ranks; the row counts to the host
        recv_counts = torch.empty((G * E_loc,), dtype=torch.int32, device=dev)
        self.comm.all_to_all(recv_counts, p.group_sizes.contiguous())
        counts = torch.stack([p.group_sizes, recv_counts]).view(2, G, E_loc).sum(dim=2).cpu()
        send_splits = [int(v) for v in counts[0]]
        recv_splits = [int(v) for v in counts[1]]
        R, N = sum(send_splits), sum(recv_splits)
        # 3. the selected routes' rows to their experts' ranks
        recv_x = torch.empty((N, H), dtype=torch.bfloat16, device=dev)
        self.comm.all_to_all(recv_x, p.x_perm[:R], recv_splits, send_splits)
        # 4. local expert order and the local experts' grouped GEMMs
        y_recv = torch.empty((N, H), dtype=torch.bfloat16, device=dev)
        if N > 0:
            lid = k.recv_expert_ids(recv_counts.view(G, E_loc), N)
            loc = k.permute(recv_x, lid.view(N, 1), E_loc, self.precision == "mxfp8")
            y_loc = k.swiglu_gemm(loc.x_perm, loc.x_perm_scales, self.weights, loc.group_offsets)
            # 5. back to the received order
            y_recv = k.gather_rows(y_loc, loc.row_map)
        # 6. the rows back to their sources, in each source's permuted order
        y_back = torch.zeros((T * self.K, H), dtype=torch.bfloat16, device=dev)
        self.comm.all_to_all(y_back[:R], y_recv, send_splits, recv_splits)
        # 7. combine with the source's probabilities
        self.last = dict(send_splits=send_splits, recv_splits=recv_splits, routes=R, received=N)
        return k.combine(y_back, p.row_map, probs)
