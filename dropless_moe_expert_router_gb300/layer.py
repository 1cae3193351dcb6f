"""The dropless MoE layer forward as one object over the C ABI.

``MoELayer`` owns the packed expert weights and every intermediate buffer
(allocated once, with torch, at construction), so ``forward`` enqueues the five
library steps -- router top-K, permute, grouped GEMM up (SwiGLU), grouped GEMM
down, combine -- on the current stream with no allocation, no host sync and no
device-to-host copy. ``forward_host`` is the end-to-end call for inputs and
outputs in (pinned) host memory.
"""
from __future__ import annotations

import ctypes as C
from typing import Optional

import torch

from . import _lib, api


class MoELayer:
    def __init__(self, w1: torch.Tensor, w3: torch.Tensor, w2: torch.Tensor, *, T: int, K: int,
                 precision: str = "bf16", renorm: bool = False, id_dtype=torch.int32, stream=None):
        E, H, F = w1.shape
        self.E, self.H, self.F, self.T, self.K = E, H, F, T, K
        self.precision = precision
        self.renorm = renorm
        self.fp8 = precision == "mxfp8"
        dev = w1.device
        self.weights = api.moe_prepare_weights(w1, w3, w2, precision, stream=stream)
        R_cap = T * K
        self.R_cap = R_cap
        self.ids = torch.empty((T, K), dtype=id_dtype, device=dev)
        self.probs = torch.empty((T, K), dtype=torch.float32, device=dev)
        self.perm = api.permute_buffers(T, H, K, E, dev, fuse_mxfp8=self.fp8)
        self.workspace = torch.empty(api.moe_permute_workspace_size(T, K, E), dtype=torch.uint8, device=dev)
        self.h = torch.empty((R_cap, F), dtype=torch.uint8 if self.fp8 else torch.bfloat16, device=dev)
        self.h_scales = torch.empty((R_cap, F // 32), dtype=torch.uint8, device=dev) if self.fp8 else None
        self.y_perm = torch.empty((R_cap, H), dtype=torch.bfloat16, device=dev)
        self.y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        self.x_dev = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        self.logits_dev = torch.empty((T, E), dtype=torch.float32, device=dev)
        self._lib = _lib.load()

    # number of library kernel launches one forward enqueues
    LAUNCHES_PER_FORWARD = 7   # router 1, permute 3 (rank, scan, scatter), GEMM 2, combine 1

    def stage_route(self, logits, stream=None):
        api.moe_route_topk(logits, self.K, renorm=self.renorm, ids=self.ids, probs=self.probs, stream=stream)

    def stage_permute(self, x, stream=None):
        api.moe_permute(x, self.ids, self.E, fuse_mxfp8=self.fp8, out=self.perm, workspace=self.workspace,
                        stream=stream)

    def stage_gemm_up(self, stream=None):
        w = self.weights
        st = self._lib.moe_grouped_gemm_up(
            api._ptr(self.perm.x_perm), api._ptr(self.perm.x_perm_scales), api._ptr(w.w13),
            api._ptr(w.w13_scales), api._dt_code(w.precision), api._ptr(self.perm.group_offsets), w.E, w.H,
            w.F, self.R_cap, api._ptr(self.h), api._ptr(self.h_scales), None, None, api._stream(stream))
        api._check("moe_grouped_gemm_up", st)

    def stage_gemm_down(self, stream=None):
        w = self.weights
        st = self._lib.moe_grouped_gemm_down(
            api._ptr(self.h), api._ptr(self.h_scales), api._ptr(w.w2), api._ptr(w.w2_scales),
            api._dt_code(w.precision), api._ptr(self.perm.group_offsets), w.E, w.H, w.F, self.R_cap,
            api._ptr(self.y_perm), api._stream(stream))
        api._check("moe_grouped_gemm_down", st)

    def stage_combine(self, stream=None):
        api.moe_unpermute_combine(self.y_perm, self.perm.row_map, self.probs, y=self.y, stream=stream)

    def forward(self, x: torch.Tensor, logits: torch.Tensor, stream=None) -> torch.Tensor:
        """x [T, H] bf16 and logits [T, E] fp32 on the device -> y [T, H] bf16 (a layer-owned buffer)."""
        self.stage_route(logits, stream)
        self.stage_permute(x, stream)
        self.stage_gemm_up(stream)
        self.stage_gemm_down(stream)
        self.stage_combine(stream)
        return self.y

    def forward_host(self, x_host: torch.Tensor, logits_host: torch.Tensor, y_host: torch.Tensor,
                     stream=None) -> torch.Tensor:
        """End to end from host memory: copy x and logits in, run the layer, copy y out
        (all enqueued on the stream; pinned host tensors make the copies asynchronous)."""
        s = stream if stream is not None else torch.cuda.current_stream()
        with torch.cuda.stream(s):
            self.x_dev.copy_(x_host, non_blocking=True)
            self.logits_dev.copy_(logits_host, non_blocking=True)
            self.forward(self.x_dev, self.logits_dev, s)
            y_host.copy_(self.y, non_blocking=True)
        return y_host
