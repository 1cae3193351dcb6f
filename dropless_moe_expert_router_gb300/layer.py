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
                 precision: str = "bf16", renorm: bool = False, id_dtype=torch.int32, training: bool = False,
                 score: str = "softmax", expert_bias: Optional[torch.Tensor] = None, stream=None,
                 packed_weights=None):
        E, H, F = w1.shape
        # (packed_weights: the packed forward weights of another layer with the same experts,
        # shared instead of packed again)
        self._args = dict(K=K, precision=precision, renorm=renorm, id_dtype=id_dtype, score=score,
                          expert_bias=expert_bias)
        self._w = (w1, w3, w2)
        self._slice_layers = None
        self._slots = None
        self.host_event = None      # set by forward_host: y_host holds the result once it completes
        self.E, self.H, self.F, self.T, self.K = E, H, F, T, K
        self.precision = precision
        self.renorm = renorm
        if score not in ("softmax", "sigmoid"):
            raise ValueError("score must be 'softmax' or 'sigmoid'")
        if expert_bias is not None and score != "sigmoid":
            raise ValueError("an expert bias steers only the sigmoid router's selection")
        self.score = score
        self.expert_bias = expert_bias      # [E] fp32 on the device; the caller may update it in place
        if precision not in ("bf16", "mxfp8", "nvfp4"):
            raise ValueError("precision must be 'bf16', 'mxfp8' or 'nvfp4'")
        self.fp8 = precision == "mxfp8"
        self.nv4 = precision == "nvfp4"
        if self.nv4 and training:
            raise ValueError("the NVFP4 layer is forward-only")
        self.training = training
        dev = w1.device
        if packed_weights is not None:
            self.weights = packed_weights
        elif self.nv4:
            self.weights = api.moe_prepare_weights_nvfp4(w1, w3, w2, stream=stream)
        else:
            self.weights = api.moe_prepare_weights(w1, w3, w2, precision, stream=stream)
        self.bwd_weights = api.moe_prepare_weights_bwd(w1, w3, w2, precision, stream=stream) if training else None
        R_cap = T * K
        self.R_cap = R_cap
        self.ids = torch.empty((T, K), dtype=id_dtype, device=dev)
        self.probs = torch.empty((T, K), dtype=torch.float32, device=dev)
        self.perm = api.permute_buffers(T, H, K, E, dev, fuse_mxfp8=self.fp8, nvfp4=self.nv4)
        self.workspace = torch.empty(api.moe_permute_workspace_size(T, K, E), dtype=torch.uint8, device=dev)
        self.h = torch.empty((R_cap, F), dtype=torch.uint8 if self.fp8 else torch.bfloat16, device=dev)
        self.h_scales = torch.empty((R_cap, F // 32), dtype=torch.uint8, device=dev) if self.fp8 else None
        if self.nv4:
            # NVFP4 operands of the two GEMMs: x_perm (written by the permute) and h quantised
            # with their tensors' amax
            u8, f32 = torch.uint8, torch.float32
            self.x_amax = torch.empty((1,), dtype=f32, device=dev)
            self.h_amax = torch.empty((1,), dtype=f32, device=dev)
            self.h_q = torch.empty((R_cap, F // 2), dtype=u8, device=dev)
            self.h_s = torch.empty((R_cap, F // 16), dtype=u8, device=dev)
        self.y_perm = torch.empty((R_cap, H), dtype=torch.bfloat16, device=dev)
        self.y = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        self.x_dev = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
        self.logits_dev = torch.empty((T, E), dtype=torch.float32, device=dev)
        self._lib = _lib.load()
        if training:
            bf = torch.bfloat16
            kpad = api.moe_grouped_transpose_kpad(R_cap, E)
            self.ab = torch.empty((R_cap, 2 * F), dtype=bf, device=dev)
            self.h_bf16 = torch.empty((R_cap, F), dtype=bf, device=dev) if self.fp8 else None
            self.dab = torch.empty((R_cap, 2 * F), dtype=bf, device=dev)
            self.dx = torch.empty((R_cap, H), dtype=bf, device=dev)
            # full-layer backward: gradients of y_perm, probs, the tokens and the logits
            self.dy_perm = torch.empty((R_cap, H), dtype=bf, device=dev)
            self.dprobs = torch.empty((T, K), dtype=torch.float32, device=dev)
            self.dx_tokens = torch.empty((T, H), dtype=bf, device=dev)
            self.dlogits = torch.empty((T, E), dtype=torch.float32, device=dev)
            u8 = torch.uint8
            self.dy_q = torch.empty((R_cap, H), dtype=u8, device=dev) if self.fp8 else None
            self.dy_s = torch.empty((R_cap, H // 32), dtype=u8, device=dev) if self.fp8 else None
            self.dab_q = torch.empty((R_cap, 2 * F), dtype=u8, device=dev) if self.fp8 else None
            self.dab_s = torch.empty((R_cap, 2 * F // 32), dtype=u8, device=dev) if self.fp8 else None
            tdt = u8 if self.fp8 else bf

            def tbuf(C):
                return (torch.empty((C, kpad), dtype=tdt, device=dev),
                        torch.empty((C, kpad // 32), dtype=u8, device=dev) if self.fp8 else None)
            self.hT, self.dyT, self.xT, self.dabT = tbuf(F), tbuf(H), tbuf(H), tbuf(2 * F)
            self.dW1 = torch.empty((E, H, F), dtype=bf, device=dev)
            self.dW3 = torch.empty((E, H, F), dtype=bf, device=dev)
            self.dW2 = torch.empty((E, F, H), dtype=bf, device=dev)

    # number of library kernel launches one forward enqueues: router 1, permute 2 or 3
    # (rank, [scan,] scatter), GEMM 2, combine 1
    @property
    def launches_per_forward(self) -> int:
        # (NVFP4 adds the routed tokens' amax and the quantisation of h)
        return 4 + api.moe_permute_kernel_launches(self.T, self.K, self.E) + (2 if self.nv4 else 0)

    def stage_route(self, logits, stream=None):
        if self.score == "sigmoid":
            api.moe_route_sigmoid_topk(logits, self.K, expert_bias=self.expert_bias, renorm=self.renorm, ids=self.ids,
                                       probs=self.probs, stream=stream)
        else:
            api.moe_route_topk(logits, self.K, renorm=self.renorm, ids=self.ids, probs=self.probs, stream=stream)

    @property
    def expert_load(self) -> torch.Tensor:
        """Valid routes per expert of the last forward ([E] int32 on the device): the statistics
        a bias-balancing update of the sigmoid router reads (the permute's group sizes)."""
        return self.perm.group_sizes

    def stage_permute(self, x, stream=None):
        if self.nv4:
            api.moe_permute_nvfp4(x, self.ids, self.E, amax=self.x_amax, out=self.perm, workspace=self.workspace,
                                  stream=stream)
            return
        api.moe_permute(x, self.ids, self.E, fuse_mxfp8=self.fp8, out=self.perm, workspace=self.workspace,
                        stream=stream)

    def stage_quant_h(self, stream=None):
        """NVFP4 only: h quantised with the amax the up projection gathered."""
        if not self.nv4:
            return
        api.moe_quant_nvfp4(self.h, self.h_amax, valid_rows=self.perm.group_offsets[self.E:], q=self.h_q,
                            scales=self.h_s, stream=stream)

    def stage_gemm_up(self, stream=None):
        w = self.weights
        if self.nv4:
            # h (bf16) and its amax from the NVFP4 operands
            api.moe_grouped_gemm_up_nvfp4(self.perm.x_perm, self.perm.x_perm_scales, self.x_amax, w, self.perm.group_offsets, h=self.h,
                                          h_amax=self.h_amax, stream=stream)
            return
        ab = self.ab if self.training else None
        hb = self.h_bf16 if self.training else None
        st = self._lib.moe_grouped_gemm_up(
            api._ptr(self.perm.x_perm), api._ptr(self.perm.x_perm_scales), api._ptr(w.w13),
            api._ptr(w.w13_scales), api._dt_code(w.precision), api._ptr(self.perm.group_offsets), w.E, w.H,
            w.F, self.R_cap, api._ptr(self.h), api._ptr(self.h_scales), api._ptr(ab), api._ptr(hb),
            api._stream(stream))
        api._check("moe_grouped_gemm_up", st)

    def stage_gemm_down(self, stream=None):
        w = self.weights
        if self.nv4:
            api.moe_grouped_gemm_down_nvfp4(self.h_q, self.h_s, self.h_amax, w, self.perm.group_offsets,
                                            y_perm=self.y_perm, stream=stream)
            return
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
        self.stage_quant_h(stream)
        self.stage_gemm_down(stream)
        self.stage_combine(stream)
        return self.y

    # ------------------------------------------------------------ backward
    # library launches of the expert-MLP backward: dgrad 1, dx 1, transposes 4, wgrad 2 (+ dy's
    # quantisation for MXFP8; dab's comes out of the dgrad epilogue); the full layer backward adds
    # combine, permute and router backward (and for MXFP8 the combine backward quantises dy_perm)
    @property
    def launches_per_backward(self) -> int:
        return 8 + (1 if self.fp8 else 0)

    @property
    def launches_per_backward_full(self) -> int:
        return 8 + 3

    def stage_combine_backward(self, dy: torch.Tensor, stream=None):
        """dy [T, H] bf16 (gradient of the layer output) -> dy_perm [R_cap, H], dprobs [T, K]
        (MXFP8: and dy_perm's row-wise codes and scales, the down-projection dgrad's operand)."""
        api.moe_unpermute_combine_backward(dy, self.y_perm, self.perm.row_map, self.probs, dy_perm=self.dy_perm,
                                           dprobs=self.dprobs, dy_perm_q=self.dy_q, dy_perm_scales=self.dy_s,
                                           stream=stream)

    def stage_permute_backward(self, stream=None):
        """dx_perm (the expert backward's) -> dx [T, H]: each token's rows summed."""
        api.moe_permute_backward(self.dx, self.perm.row_map, dx=self.dx_tokens, stream=stream)

    def stage_route_backward(self, logits: torch.Tensor, stream=None):
        """dprobs -> dlogits [T, E] through the router's score function (selection fixed)."""
        if self.score == "sigmoid":
            api.moe_route_sigmoid_topk_backward(logits, self.ids, self.dprobs, renorm=self.renorm,
                                                dlogits=self.dlogits, stream=stream)
            return
        api.moe_route_topk_backward(logits, self.ids, self.dprobs, renorm=self.renorm, dlogits=self.dlogits,
                                    stream=stream)

    def stage_dgrad_dh(self, dy_perm: torch.Tensor, stream=None, dy_quantised: bool = False):
        """dy_perm [R_cap, H] bf16 -> dab = SwiGLU backward of dh = dy W2^T (bf16). dy_quantised:
        (MXFP8) dy_perm's codes and scales are already in dy_q / dy_s (the combine backward's)."""
        goff = self.perm.group_offsets
        bw = self.bwd_weights
        if self.fp8:
            if not dy_quantised:
                api.moe_quant_mxfp8_grouped(dy_perm, goff, q=self.dy_q, scales=self.dy_s, stream=stream)
            api.moe_grouped_swiglu_dgrad(self.dy_q, self.dy_s, bw, self.ab, goff, dab=self.dab, dab_q=self.dab_q,
                                         dab_scales=self.dab_s, stream=stream)
        else:
            api.moe_grouped_swiglu_dgrad(dy_perm, None, bw, self.ab, goff, dab=self.dab, stream=stream)

    def stage_dgrad_dx(self, stream=None):
        """dab -> dx = da W1^T + db W3^T [R_cap, H] bf16 (MXFP8: from the codes and scales of dab
        that the dgrad epilogue wrote)."""
        goff = self.perm.group_offsets
        bw = self.bwd_weights
        if self.fp8:
            api.moe_grouped_gemm_dx(self.dab_q, self.dab_s, bw, goff, dx=self.dx, stream=stream)
        else:
            api.moe_grouped_gemm_dx(self.dab, None, bw, goff, dx=self.dx, stream=stream)
        return self.dx

    def stage_transposes(self, x: torch.Tensor, dy_perm: torch.Tensor, stream=None):
        """Group-padded transposed (and, for MXFP8, column-quantised) weight-gradient operands."""
        goff = self.perm.group_offsets
        prec = self.precision
        h_src = self.h_bf16 if self.fp8 else self.h
        api.moe_grouped_transpose(h_src, goff, prec, xT=self.hT[0], xT_scales=self.hT[1], stream=stream)
        api.moe_grouped_transpose(dy_perm, goff, prec, xT=self.dyT[0], xT_scales=self.dyT[1], stream=stream)
        api.moe_grouped_transpose(x, goff, prec, R_cap=self.R_cap, src_rows=self.perm.perm_src, xT=self.xT[0],
                                  xT_scales=self.xT[1], stream=stream)
        api.moe_grouped_transpose(self.dab, goff, prec, xT=self.dabT[0], xT_scales=self.dabT[1], stream=stream)

    def stage_wgrad_gemm(self, stream=None):
        """dW2 = h^T dy, dW1 = x^T da, dW3 = x^T db per expert."""
        goff = self.perm.group_offsets
        prec = self.precision
        api.moe_grouped_gemm_wgrad(self.hT[0], self.hT[1], self.dyT[0], self.dyT[1], prec, goff, self.R_cap,
                                   dw=self.dW2, stream=stream)
        api.moe_grouped_gemm_wgrad(self.xT[0], self.xT[1], self.dabT[0], self.dabT[1], prec, goff, self.R_cap,
                                   split=True, dw=self.dW1, dw2=self.dW3, stream=stream)
        return self.dW1, self.dW3, self.dW2

    def backward(self, x: torch.Tensor, dy_perm: torch.Tensor, stream=None, dy_quantised: bool = False):
        """Grouped backward of the expert MLP after a training forward (x: the forward's tokens,
        dy_perm: gradient of y_perm) -> (dx_perm, dW1, dW3, dW2)."""
        self.stage_dgrad_dh(dy_perm, stream, dy_quantised)
        dx = self.stage_dgrad_dx(stream)
        self.stage_transposes(x, dy_perm, stream)
        return (dx,) + tuple(self.stage_wgrad_gemm(stream))

    def backward_full(self, x: torch.Tensor, logits: torch.Tensor, dy: torch.Tensor, stream=None):
        """Backward of the whole layer after a training forward (x, logits: the forward's inputs;
        dy [T, H]: gradient of its output) -> (dx [T, H], dlogits [T, E], dW1, dW3, dW2)."""
        self.stage_combine_backward(dy, stream)
        _, dw1, dw3, dw2 = self.backward(x, self.dy_perm, stream, dy_quantised=self.fp8)
        self.stage_permute_backward(stream)
        self.stage_route_backward(logits, stream)
        return self.dx_tokens, self.dlogits, dw1, dw3, dw2

    def _slices(self):
        """Layers over consecutive slices of the tokens (an eighth, three quarters, an eighth),
        sharing the packed weights, and the two copy streams of the sliced transfer."""
        if self._slice_layers is None:
            t0 = max(1, self.T // 8)
            sizes = [t for t in (t0, self.T - 2 * t0, t0) if t > 0] if self.T >= 3 else [self.T]
            layers = [MoELayer(*self._w, T=t, packed_weights=self.weights, **self._args) for t in sizes]
            dev = self.weights.w13.device
            self._slice_layers = (sizes, layers, torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev))
        return self._slice_layers

    def _forward_mapped(self, xd: int, logits_host: torch.Tensor, yd: int, s) -> None:
        """The forward with x read from, and y written to, host memory at device addresses xd, yd
        (enqueued on stream s; the logits are copied in)."""
        with torch.cuda.stream(s):
            self.logits_dev.copy_(logits_host, non_blocking=True)
            self.stage_route(self.logits_dev, s)
            self._permute_mapped(xd, s)
            self.stage_gemm_up(s)
            self.stage_gemm_down(s)
            self._combine_mapped(yd, s)

    def _permute_mapped(self, xd: int, s) -> None:
        p = self.perm
        st = self._lib.moe_permute(
            xd, self.T, self.H, api._ptr(self.ids), api._id_code(self.ids.dtype), self.K, self.E,
            api._ptr(p.x_perm), api._ptr(p.x_perm_scales), api._ptr(p.group_sizes), api._ptr(p.group_offsets),
            api._ptr(p.row_map), api._ptr(p.perm_src), api.MOE_PERMUTE_FUSE_MXFP8 if self.fp8 else 0,
            api._ptr(self.workspace), self.workspace.numel(), api._stream(s))
        api._check("moe_permute", st)

    def _combine_mapped(self, yd: int, s) -> None:
        st = self._lib.moe_unpermute_combine(api._ptr(self.y_perm), api._ptr(self.perm.row_map), api._ptr(self.probs),
                                             self.T, self.K, self.H, yd, api._stream(s))
        api._check("moe_unpermute_combine", st)

    def forward_host(self, x_host: torch.Tensor, logits_host: torch.Tensor, y_host: torch.Tensor,
                     stream=None, transfer: str = "auto") -> torch.Tensor:
        """End to end from host memory: x [T, H] bf16 and logits [T, E] fp32 in, y [T, H] bf16 out.
        The compute is enqueued on the stream; y_host holds the result once the event
        self.host_event has completed (or after torch.cuda.synchronize()). transfer:

        - "overlapped": the layer's own copy streams move x and logits in and y out through two
          sets of device buffers used in turn, so that consecutive calls overlap. This call's
          input copy waits only until the previous call's permute has read the other set, so it
          runs while that call computes; its output copy runs while the next call computes. x_host
          and logits_host must hold the inputs when the call is made: they are read in the copy
          stream's order, not the stream's. Wants page-locked host tensors (torch's pin_memory).
        - "sliced": the tokens go through in three consecutive slices (an eighth, three
          quarters, an eighth). Each slice has its own route, permute, GEMMs and combine; rows are
          independent, so the result is the whole batch's. A slice's copies overlap the other
          slices' compute within one call, at the price of a partly filled GEMM tile per expert
          and slice. Wants page-locked host tensors.
        - "direct": the permute reads x and the combine writes y in page-locked host memory
          through their device addresses; only the logits are copied in.
        - "copy": x and logits copied in, the whole forward, y copied out, all on the stream.
        - "auto": "overlapped" when the three host tensors are page-locked, else "copy".

        A training layer always copies: its backward reads the device copy of x. The NVFP4 layer
        neither slices (x and h are scaled by their whole tensors' amax) nor reads x directly."""
        if transfer not in ("auto", "overlapped", "sliced", "direct", "copy"):
            raise ValueError("transfer must be 'auto', 'overlapped', 'sliced', 'direct' or 'copy'")
        for t, shape, dt in ((x_host, (self.T, self.H), torch.bfloat16), (y_host, (self.T, self.H), torch.bfloat16),
                             (logits_host, (self.T, self.E), torch.float32)):
            if tuple(t.shape) != shape or t.dtype != dt:
                raise ValueError(f"host tensor must be {shape} {dt}")
        s = stream if stream is not None else torch.cuda.current_stream()
        pinned = x_host.is_pinned() and y_host.is_pinned() and logits_host.is_pinned()
        if transfer == "auto":
            transfer = "overlapped" if pinned and not self.training else "copy"
        if transfer != "copy" and self.training:
            raise ValueError("a training layer copies x in: its backward reads the device copy")
        if transfer in ("sliced", "direct") and self.nv4:
            raise ValueError("the NVFP4 layer copies x in whole: it scales x by the whole tensor's amax")
        if transfer in ("overlapped", "sliced") and not pinned:
            raise ValueError(f"the {transfer} transfer wants page-locked host tensors")
        if transfer == "overlapped":
            self._forward_overlapped(x_host, logits_host, y_host, s)
            return y_host
        if transfer == "sliced":
            self._forward_sliced(x_host, logits_host, y_host, s)
        elif transfer == "direct":
            xd = api.moe_host_mapped_pointer(x_host)
            yd = api.moe_host_mapped_pointer(y_host)
            if xd is None or yd is None:
                raise ValueError("x_host and y_host must be page-locked memory the device can address")
            self._forward_mapped(xd, logits_host, yd, s)
        else:
            with torch.cuda.stream(s):
                self.x_dev.copy_(x_host, non_blocking=True)
                self.logits_dev.copy_(logits_host, non_blocking=True)
                self.forward(self.x_dev, self.logits_dev, s)
                y_host.copy_(self.y, non_blocking=True)
        self.host_event = torch.cuda.Event()
        self.host_event.record(s)
        return y_host

    def _forward_overlapped(self, x_host, logits_host, y_host, s) -> None:
        if self._slots is None:
            dev = self.x_dev.device
            # (buffers of their own: forward's y and the copy transfer's x, logits stay untouched)
            bufs = [(torch.empty_like(self.x_dev), torch.empty_like(self.logits_dev), torch.empty_like(self.y))
                    for _ in range(2)]
            self._slots = dict(bufs=bufs, next=0,
                               cin=torch.cuda.Stream(device=dev), cout=torch.cuda.Stream(device=dev),
                               read=[None, None], sent=[None, None])
        sl = self._slots
        i = sl["next"]
        sl["next"] = i ^ 1
        xs, ls, ys = sl["bufs"][i]
        cin, cout = sl["cin"], sl["cout"]
        if sl["read"][i] is not None:
            cin.wait_event(sl["read"][i])          # this set's previous permute has read it
        with torch.cuda.stream(cin):
            xs.copy_(x_host, non_blocking=True)
            ls.copy_(logits_host, non_blocking=True)
            arrived = torch.cuda.Event()
            arrived.record(cin)
        s.wait_event(arrived)
        if sl["sent"][i] is not None:
            s.wait_event(sl["sent"][i])            # this set's previous y has reached the host
        with torch.cuda.stream(s):
            self.stage_route(ls, s)
            self.stage_permute(xs, s)
            read = torch.cuda.Event()
            read.record(s)
            self.stage_gemm_up(s)
            self.stage_quant_h(s)
            self.stage_gemm_down(s)
            api.moe_unpermute_combine(self.y_perm, self.perm.row_map, self.probs, y=ys, stream=s)
            done = torch.cuda.Event()
            done.record(s)
        sl["read"][i] = read
        cout.wait_event(done)
        with torch.cuda.stream(cout):
            y_host.copy_(ys, non_blocking=True)
            sent = torch.cuda.Event()
            sent.record(cout)
        sl["sent"][i] = sent
        self.host_event = sent

    def _forward_sliced(self, x_host, logits_host, y_host, s) -> None:
        sizes, parts, cin, cout = self._slices()
        start = torch.cuda.Event()
        start.record(s)
        cin.wait_event(start)
        cout.wait_event(start)
        arrived, off = [], 0
        with torch.cuda.stream(cin):
            for t, L in zip(sizes, parts):
                L.x_dev.copy_(x_host[off:off + t], non_blocking=True)
                L.logits_dev.copy_(logits_host[off:off + t], non_blocking=True)
                e = torch.cuda.Event()
                e.record(cin)
                arrived.append(e)
                off += t
        off = 0
        for t, L, e in zip(sizes, parts, arrived):
            s.wait_event(e)
            with torch.cuda.stream(s):
                L.forward(L.x_dev, L.logits_dev, s)
            done = torch.cuda.Event()
            done.record(s)
            cout.wait_event(done)
            with torch.cuda.stream(cout):
                y_host[off:off + t].copy_(L.y, non_blocking=True)
            off += t
        out = torch.cuda.Event()
        out.record(cout)
        s.wait_event(out)
