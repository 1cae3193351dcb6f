"""Thin Python binding of the C ABI (include/moe_gb300.h).

Each function has the name of its C entry point and only marshals arguments:
it checks devices and dtypes, allocates outputs with torch when the caller did
not pass them, and hands raw pointers, sizes and the current CUDA stream to
the library. Every step of the computation runs in the library's kernels.
"""
from __future__ import annotations

import ctypes as C
from typing import NamedTuple, Optional

import torch

from . import _lib

MOE_I16, MOE_I32, MOE_BF16, MOE_MXFP8 = 0, 1, 2, 3
MOE_ROUTE_RENORM = 1
MOE_PERMUTE_FUSE_MXFP8 = 2
MOE_QUANT_COLWISE = 4
MOE_DEVERR_BAD_ID = 1
MOE_DEVERR_TIMEOUT = 2


class MoeError(RuntimeError):
    def __init__(self, fn: str, status: int):
        name = _lib.load().moe_status_string(status).decode()
        super().__init__(f"{fn} failed: {name} ({status})")
        self.status = status


def _check(fn: str, status: int) -> None:
    if status != 0:
        raise MoeError(fn, status)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def _want(t: torch.Tensor, name: str, dtype=None, ndim=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims")


def _id_code(dtype: torch.dtype) -> int:
    if dtype == torch.int16:
        return MOE_I16
    if dtype == torch.int32:
        return MOE_I32
    raise ValueError("ids must be int16 or int32")


# --------------------------------------------------------------------- router
def moe_route_topk(logits: torch.Tensor, K: int, *, id_dtype=torch.int32, renorm: bool = False,
                   ids: Optional[torch.Tensor] = None, probs: Optional[torch.Tensor] = None,
                   stream=None):
    """logits [T, E] fp32 -> (ids [T, K] int16/int32, probs [T, K] fp32)."""
    _want(logits, "logits", torch.float32, 2)
    T, E = logits.shape
    if ids is None:
        ids = torch.empty((T, K), dtype=id_dtype, device=logits.device)
    if probs is None:
        probs = torch.empty((T, K), dtype=torch.float32, device=logits.device)
    _want(ids, "ids", None, 2)
    _want(probs, "probs", torch.float32, 2)
    st = _lib.load().moe_route_topk(_ptr(logits), T, E, K, _ptr(ids), _id_code(ids.dtype), _ptr(probs),
                                    MOE_ROUTE_RENORM if renorm else 0, _stream(stream))
    _check("moe_route_topk", st)
    return ids, probs


def moe_route_sigmoid_topk(logits: torch.Tensor, K: int, *, expert_bias: Optional[torch.Tensor] = None,
                           id_dtype=torch.int32, renorm: bool = False, ids: Optional[torch.Tensor] = None,
                           probs: Optional[torch.Tensor] = None, stream=None):
    """logits [T, E] fp32 (+ expert_bias [E] fp32) -> (ids [T, K], probs [T, K] fp32): selection on
    sigmoid(logit) + bias, probs the sigmoid scores (renormalised over the K selected with renorm)."""
    _want(logits, "logits", torch.float32, 2)
    T, E = logits.shape
    if expert_bias is not None:
        _want(expert_bias, "expert_bias", torch.float32, 1)
        if expert_bias.numel() != E:
            raise ValueError("expert_bias must have E entries")
    if ids is None:
        ids = torch.empty((T, K), dtype=id_dtype, device=logits.device)
    if probs is None:
        probs = torch.empty((T, K), dtype=torch.float32, device=logits.device)
    _want(ids, "ids", None, 2)
    _want(probs, "probs", torch.float32, 2)
    st = _lib.load().moe_route_sigmoid_topk(_ptr(logits), _ptr(expert_bias), T, E, K, _ptr(ids),
                                            _id_code(ids.dtype), _ptr(probs), MOE_ROUTE_RENORM if renorm else 0,
                                            _stream(stream))
    _check("moe_route_sigmoid_topk", st)
    return ids, probs


def moe_route_sigmoid_topk_backward(logits: torch.Tensor, ids: torch.Tensor, dprobs: torch.Tensor, *,
                                    renorm: bool = False, dlogits: Optional[torch.Tensor] = None,
                                    stream=None) -> torch.Tensor:
    """logits [T, E], ids [T, K], dprobs [T, K] -> dlogits [T, E] fp32 of the sigmoid router."""
    _want(logits, "logits", torch.float32, 2)
    _want(ids, "ids", None, 2)
    _want(dprobs, "dprobs", torch.float32, 2)
    T, E = logits.shape
    K = ids.shape[1]
    if dlogits is None:
        dlogits = torch.empty((T, E), dtype=torch.float32, device=logits.device)
    _want(dlogits, "dlogits", torch.float32, 2)
    st = _lib.load().moe_route_sigmoid_topk_backward(_ptr(logits), _ptr(ids), _id_code(ids.dtype), _ptr(dprobs),
                                                     T, E, K, MOE_ROUTE_RENORM if renorm else 0, _ptr(dlogits),
                                                     _stream(stream))
    _check("moe_route_sigmoid_topk_backward", st)
    return dlogits


# -------------------------------------------------------------------- permute
class Permuted(NamedTuple):
    x_perm: torch.Tensor          # [T*K, H] bf16, or uint8 E4M3 payloads when fused
    x_perm_scales: Optional[torch.Tensor]  # [T*K, H/32] uint8 E8M0 (fused MXFP8 only)
    group_sizes: torch.Tensor     # [E] int32
    group_offsets: torch.Tensor   # [E+1] int32
    row_map: torch.Tensor         # [T, K] int32
    perm_src: torch.Tensor        # [T*K] int32


def moe_permute_workspace_size(T: int, K: int, E: int) -> int:
    return int(_lib.load().moe_permute_workspace_size(T, K, E))


def moe_permute_kernel_launches(T: int, K: int, E: int) -> int:
    return int(_lib.load().moe_permute_kernel_launches(T, K, E))


def permute_buffers(T: int, H: int, K: int, E: int, device, fuse_mxfp8: bool = False,
                    nvfp4: bool = False) -> Permuted:
    R_cap = T * K
    dev = torch.device(device)
    if nvfp4:
        xp = torch.empty((R_cap, H // 2), dtype=torch.uint8, device=dev)
        xs = torch.empty((R_cap, H // 16), dtype=torch.uint8, device=dev)
    elif fuse_mxfp8:
        xp = torch.empty((R_cap, H), dtype=torch.uint8, device=dev)
        xs = torch.empty((R_cap, H // 32), dtype=torch.uint8, device=dev)
    else:
        xp = torch.empty((R_cap, H), dtype=torch.bfloat16, device=dev)
        xs = None
    return Permuted(xp, xs, torch.empty(E, dtype=torch.int32, device=dev),
                    torch.empty(E + 1, dtype=torch.int32, device=dev),
                    torch.empty((T, K), dtype=torch.int32, device=dev),
                    torch.empty(R_cap, dtype=torch.int32, device=dev))


def moe_permute(x: torch.Tensor, ids: torch.Tensor, E: int, *, fuse_mxfp8: bool = False,
                out: Optional[Permuted] = None, workspace: Optional[torch.Tensor] = None,
                stream=None) -> Permuted:
    """x [T, H] bf16, ids [T, K] -> Permuted (see the C header for each field)."""
    _want(x, "x", torch.bfloat16, 2)
    _want(ids, "ids", None, 2)
    T, H = x.shape
    K = ids.shape[1]
    if out is None:
        out = permute_buffers(T, H, K, E, x.device, fuse_mxfp8)
    ws_bytes = moe_permute_workspace_size(T, K, E)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=x.device)
    st = _lib.load().moe_permute(
        _ptr(x), T, H, _ptr(ids), _id_code(ids.dtype), K, E, _ptr(out.x_perm), _ptr(out.x_perm_scales),
        _ptr(out.group_sizes), _ptr(out.group_offsets), _ptr(out.row_map), _ptr(out.perm_src),
        MOE_PERMUTE_FUSE_MXFP8 if fuse_mxfp8 else 0, _ptr(workspace), workspace.numel(), _stream(stream))
    _check("moe_permute", st)
    return out


def moe_permute_nvfp4(x: torch.Tensor, ids: torch.Tensor, E: int, *, amax: Optional[torch.Tensor] = None,
                      out: Optional[Permuted] = None, workspace: Optional[torch.Tensor] = None,
                      stream=None):
    """moe_permute writing NVFP4 rows: the routed tokens' amax first (-> amax [1] fp32), then the
    scatter quantises each row as it copies it (x_perm [R_cap, H/2] packed E2M1, x_perm_scales
    [R_cap, H/16] E4M3). Returns (Permuted, amax)."""
    _want(x, "x", torch.bfloat16, 2)
    _want(ids, "ids", None, 2)
    T, H = x.shape
    K = ids.shape[1]
    if out is None:
        out = permute_buffers(T, H, K, E, x.device, nvfp4=True)
    if amax is None:
        amax = torch.empty((1,), dtype=torch.float32, device=x.device)
    ws_bytes = moe_permute_workspace_size(T, K, E)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=x.device)
    st = _lib.load().moe_permute_nvfp4(
        _ptr(x), T, H, _ptr(ids), _id_code(ids.dtype), K, E, _ptr(amax), _ptr(out.x_perm), _ptr(out.x_perm_scales),
        _ptr(out.group_sizes), _ptr(out.group_offsets), _ptr(out.row_map), _ptr(out.perm_src), _ptr(workspace),
        workspace.numel(), _stream(stream))
    _check("moe_permute_nvfp4", st)
    return out, amax


def moe_permute_noalloc(x: torch.Tensor, ids: torch.Tensor, E: int, *, fuse_mxfp8: bool = False,
                        out: Optional[Permuted] = None, stream=None) -> Permuted:
    """moe_permute for callers that may not allocate device memory: the library's
    static scratch array replaces the workspace (outputs are still the caller's)."""
    _want(x, "x", torch.bfloat16, 2)
    _want(ids, "ids", None, 2)
    T, H = x.shape
    K = ids.shape[1]
    if out is None:
        out = permute_buffers(T, H, K, E, x.device, fuse_mxfp8)
    st = _lib.load().moe_permute_noalloc(
        _ptr(x), T, H, _ptr(ids), _id_code(ids.dtype), K, E, _ptr(out.x_perm), _ptr(out.x_perm_scales),
        _ptr(out.group_sizes), _ptr(out.group_offsets), _ptr(out.row_map), _ptr(out.perm_src),
        MOE_PERMUTE_FUSE_MXFP8 if fuse_mxfp8 else 0, _stream(stream))
    _check("moe_permute_noalloc", st)
    return out


def moe_permute_noalloc_max_scratch() -> int:
    return int(_lib.load().moe_permute_noalloc_max_scratch())


# ---------------------------------------------------------------- quantiser
def colwise_scale_rows(R_cap: int, E: int) -> int:
    return E + R_cap // 32 + 1


def moe_quant_mxfp8_grouped(x: torch.Tensor, group_offsets: torch.Tensor, *, colwise: bool = False,
                            q: Optional[torch.Tensor] = None, scales: Optional[torch.Tensor] = None,
                            stream=None):
    """x [R_cap, H] bf16 -> (q [R_cap, H] uint8, scales) row-wise or group-aware column-wise."""
    _want(x, "x", torch.bfloat16, 2)
    _want(group_offsets, "group_offsets", torch.int32, 1)
    R_cap, H = x.shape
    E = group_offsets.numel() - 1
    if q is None:
        q = torch.empty((R_cap, H), dtype=torch.uint8, device=x.device)
    if scales is None:
        shape = (colwise_scale_rows(R_cap, E), H) if colwise else (R_cap, H // 32)
        scales = torch.empty(shape, dtype=torch.uint8, device=x.device)
    st = _lib.load().moe_quant_mxfp8_grouped(_ptr(x), R_cap, H, _ptr(group_offsets), E, _ptr(q),
                                             _ptr(scales), MOE_QUANT_COLWISE if colwise else 0,
                                             _stream(stream))
    _check("moe_quant_mxfp8_grouped", st)
    return q, scales


# ------------------------------------------------------------------- combine
def moe_unpermute_combine(y_perm: torch.Tensor, row_map: torch.Tensor, probs: torch.Tensor, *,
                          y: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """y_perm [R_cap, H] bf16, row_map [T, K], probs [T, K] -> y [T, H] bf16."""
    _want(y_perm, "y_perm", torch.bfloat16, 2)
    _want(row_map, "row_map", torch.int32, 2)
    _want(probs, "probs", torch.float32, 2)
    T, K = row_map.shape
    H = y_perm.shape[1]
    if y is None:
        y = torch.empty((T, H), dtype=torch.bfloat16, device=y_perm.device)
    st = _lib.load().moe_unpermute_combine(_ptr(y_perm), _ptr(row_map), _ptr(probs), T, K, H, _ptr(y),
                                           _stream(stream))
    _check("moe_unpermute_combine", st)
    return y


# -------------------------------------------------------------------- backward of route / permute / combine
def moe_route_topk_backward(logits: torch.Tensor, ids: torch.Tensor, dprobs: torch.Tensor, *,
                            renorm: bool = False, dlogits: Optional[torch.Tensor] = None,
                            stream=None) -> torch.Tensor:
    """logits [T, E] fp32, ids [T, K], dprobs [T, K] fp32 -> dlogits [T, E] fp32."""
    _want(logits, "logits", torch.float32, 2)
    _want(ids, "ids", None, 2)
    _want(dprobs, "dprobs", torch.float32, 2)
    T, E = logits.shape
    K = ids.shape[1]
    if dlogits is None:
        dlogits = torch.empty((T, E), dtype=torch.float32, device=logits.device)
    _want(dlogits, "dlogits", torch.float32, 2)
    st = _lib.load().moe_route_topk_backward(_ptr(logits), _ptr(ids), _id_code(ids.dtype), _ptr(dprobs), T, E, K,
                                             MOE_ROUTE_RENORM if renorm else 0, _ptr(dlogits), _stream(stream))
    _check("moe_route_topk_backward", st)
    return dlogits


def moe_unpermute_combine_backward(dy: torch.Tensor, y_perm: torch.Tensor, row_map: torch.Tensor,
                                   probs: torch.Tensor, *, dy_perm: Optional[torch.Tensor] = None,
                                   dprobs: Optional[torch.Tensor] = None, dy_perm_q: Optional[torch.Tensor] = None,
                                   dy_perm_scales: Optional[torch.Tensor] = None, stream=None):
    """dy [T, H] bf16, y_perm [R_cap, H] bf16, row_map [T, K], probs [T, K] ->
    (dy_perm [R_cap, H] bf16, dprobs [T, K] fp32). With dy_perm_q [R_cap, H] uint8 and
    dy_perm_scales [R_cap, H/32] uint8 given, the kernel also writes the row-wise MXFP8
    codes and scales of dy_perm into them."""
    _want(dy, "dy", torch.bfloat16, 2)
    _want(y_perm, "y_perm", torch.bfloat16, 2)
    _want(row_map, "row_map", torch.int32, 2)
    _want(probs, "probs", torch.float32, 2)
    T, K = row_map.shape
    H = y_perm.shape[1]
    if dy_perm is None:
        dy_perm = torch.empty_like(y_perm)    # rows no route maps to are not written
    if dprobs is None:
        dprobs = torch.empty((T, K), dtype=torch.float32, device=dy.device)
    _want(dy_perm, "dy_perm", torch.bfloat16, 2)
    _want(dprobs, "dprobs", torch.float32, 2)
    if (dy_perm_q is None) != (dy_perm_scales is None):
        raise ValueError("dy_perm_q and dy_perm_scales go together")
    if dy_perm_q is not None:
        _want(dy_perm_q, "dy_perm_q", torch.uint8, 2)
        _want(dy_perm_scales, "dy_perm_scales", torch.uint8, 2)
        if tuple(dy_perm_q.shape) != tuple(y_perm.shape) or tuple(dy_perm_scales.shape) != (y_perm.shape[0], H // 32):
            raise ValueError("dy_perm_q must be [R_cap, H] and dy_perm_scales [R_cap, H/32]")
    st = _lib.load().moe_unpermute_combine_backward(_ptr(dy), _ptr(y_perm), _ptr(row_map), _ptr(probs), T, K, H,
                                                    _ptr(dy_perm), _ptr(dprobs),
                                                    _ptr(dy_perm_q), _ptr(dy_perm_scales), _stream(stream))
    _check("moe_unpermute_combine_backward", st)
    return dy_perm, dprobs


def moe_permute_backward(dx_perm: torch.Tensor, row_map: torch.Tensor, *, dx: Optional[torch.Tensor] = None,
                         stream=None) -> torch.Tensor:
    """dx_perm [R_cap, H] bf16, row_map [T, K] -> dx [T, H] bf16 (each token's rows summed)."""
    _want(dx_perm, "dx_perm", torch.bfloat16, 2)
    _want(row_map, "row_map", torch.int32, 2)
    T, K = row_map.shape
    H = dx_perm.shape[1]
    if dx is None:
        dx = torch.empty((T, H), dtype=torch.bfloat16, device=dx_perm.device)
    _want(dx, "dx", torch.bfloat16, 2)
    st = _lib.load().moe_permute_backward(_ptr(dx_perm), _ptr(row_map), T, K, H, _ptr(dx), _stream(stream))
    _check("moe_permute_backward", st)
    return dx


# -------------------------------------------------------------------- expert parallelism
def moe_ep_recv_expert_ids(recv_counts: torch.Tensor, R_cap: int, *, ids: Optional[torch.Tensor] = None,
                           stream=None) -> torch.Tensor:
    """recv_counts [G, E_loc] int32 (rows received from each source for each local expert, on the
    device) -> ids [R_cap] int32: the local expert of each received row, -1 past them."""
    _want(recv_counts, "recv_counts", torch.int32, 2)
    G, E_loc = recv_counts.shape
    if ids is None:
        ids = torch.empty((R_cap,), dtype=torch.int32, device=recv_counts.device)
    _want(ids, "ids", torch.int32, 1)
    st = _lib.load().moe_ep_recv_expert_ids(_ptr(recv_counts), G, E_loc, R_cap, _ptr(ids), _stream(stream))
    _check("moe_ep_recv_expert_ids", st)
    return ids


# -------------------------------------------------------------------- errors
def moe_get_device_errors(clear: bool = True) -> int:
    v = C.c_uint32(0)
    st = _lib.load().moe_get_device_errors(C.byref(v), 1 if clear else 0)
    if st not in (0, 6):
        _check("moe_get_device_errors", st)
    return int(v.value)


def moe_debug_bounded_wait_selftest(limit_us: int, stream=None) -> None:
    """Enqueue the bounded-wait self-test (sets MOE_DEVERR_TIMEOUT after limit_us)."""
    _check("moe_debug_bounded_wait_selftest",
           _lib.load().moe_debug_bounded_wait_selftest(int(limit_us), _stream(stream)))


def moe_route_ids_bytes(T: int, K: int, id_dtype=torch.int16) -> int:
    return int(_lib.load().moe_route_ids_bytes(T, K, _id_code(id_dtype)))


def moe_route_probs_bytes(T: int, K: int) -> int:
    return int(_lib.load().moe_route_probs_bytes(T, K))


def moe_host_mapped_pointer(t: torch.Tensor) -> Optional[int]:
    """Device address of a page-locked host tensor's data (the kernels can read and write it
    directly), or None when the tensor is not in page-locked memory the device can address."""
    if t.is_cuda or not t.is_contiguous() or t.numel() == 0:
        return None
    out = C.c_void_p()
    st = _lib.load().moe_host_mapped_pointer(C.c_void_p(t.data_ptr()), C.byref(out))
    return int(out.value) if st == 0 and out.value else None


# ------------------------------------------------------------- expert GEMMs
def _dt_code(precision: str) -> int:
    if precision == "bf16":
        return MOE_BF16
    if precision == "mxfp8":
        return MOE_MXFP8
    raise ValueError("precision must be 'bf16' or 'mxfp8'")


class PackedWeights(NamedTuple):
    precision: str
    E: int
    H: int
    F: int
    w13: torch.Tensor                 # [E, 2F, H] bf16 or uint8 (E4M3)
    w13_scales: Optional[torch.Tensor]  # [E, 2F, H/32] uint8 (MXFP8)
    w2: torch.Tensor                  # [E, H, F] bf16 or uint8
    w2_scales: Optional[torch.Tensor]   # [E, H, F/32] uint8 (MXFP8)


def moe_prepare_weights(w1: torch.Tensor, w3: torch.Tensor, w2: torch.Tensor, precision: str = "bf16",
                        stream=None) -> PackedWeights:
    """Pack logical W1, W3 [E, H, F] and W2 [E, F, H] (bf16) for the grouped GEMMs (one-time)."""
    for t, n in ((w1, "w1"), (w3, "w3"), (w2, "w2")):
        _want(t, n, torch.bfloat16, 3)
    E, H, F = w1.shape
    dev = w1.device
    fp8 = precision == "mxfp8"
    pdt = torch.uint8 if fp8 else torch.bfloat16
    w13 = torch.empty((E, 2 * F, H), dtype=pdt, device=dev)
    w2p = torch.empty((E, H, F), dtype=pdt, device=dev)
    s13 = torch.empty((E, 2 * F, H // 32), dtype=torch.uint8, device=dev) if fp8 else None
    s2 = torch.empty((E, H, F // 32), dtype=torch.uint8, device=dev) if fp8 else None
    st = _lib.load().moe_prepare_weights(_ptr(w1), _ptr(w3), _ptr(w2), E, H, F, _dt_code(precision),
                                         _ptr(w13), _ptr(s13), _ptr(w2p), _ptr(s2), _stream(stream))
    _check("moe_prepare_weights", st)
    return PackedWeights(precision, E, H, F, w13, s13, w2p, s2)


def moe_grouped_swiglu_gemm(x_perm: torch.Tensor, x_scales: Optional[torch.Tensor], w: PackedWeights,
                            group_offsets: torch.Tensor, *, h: Optional[torch.Tensor] = None,
                            h_scales: Optional[torch.Tensor] = None, y_perm: Optional[torch.Tensor] = None,
                            stream=None):
    """Grouped SwiGLU MLP on permuted rows -> (y_perm [R_cap, H] bf16, h, h_scales)."""
    fp8 = w.precision == "mxfp8"
    _want(x_perm, "x_perm", torch.uint8 if fp8 else torch.bfloat16, 2)
    _want(group_offsets, "group_offsets", torch.int32, 1)
    R_cap = x_perm.shape[0]
    dev = x_perm.device
    if h is None:
        h = torch.empty((R_cap, w.F), dtype=torch.uint8 if fp8 else torch.bfloat16, device=dev)
    if fp8 and h_scales is None:
        h_scales = torch.empty((R_cap, w.F // 32), dtype=torch.uint8, device=dev)
    if y_perm is None:
        y_perm = torch.empty((R_cap, w.H), dtype=torch.bfloat16, device=dev)
    st = _lib.load().moe_grouped_swiglu_gemm(
        _ptr(x_perm), _ptr(x_scales), _ptr(w.w13), _ptr(w.w13_scales), _ptr(w.w2), _ptr(w.w2_scales),
        _dt_code(w.precision), _ptr(group_offsets), w.E, w.H, w.F, R_cap, _ptr(h), _ptr(h_scales),
        _ptr(y_perm), _stream(stream))
    _check("moe_grouped_swiglu_gemm", st)
    return y_perm, h, h_scales


def moe_grouped_gemm_up(x_perm: torch.Tensor, x_scales: Optional[torch.Tensor], w: PackedWeights,
                        group_offsets: torch.Tensor, *, h: Optional[torch.Tensor] = None,
                        h_scales: Optional[torch.Tensor] = None, ab: Optional[torch.Tensor] = None,
                        h_bf16: Optional[torch.Tensor] = None, stream=None):
    """Up projection + SwiGLU; optionally saves ab [R_cap, 2F] bf16 and (MXFP8) h_bf16 [R_cap, F]."""
    fp8 = w.precision == "mxfp8"
    R_cap = x_perm.shape[0]
    dev = x_perm.device
    if h is None:
        h = torch.empty((R_cap, w.F), dtype=torch.uint8 if fp8 else torch.bfloat16, device=dev)
    if fp8 and h_scales is None:
        h_scales = torch.empty((R_cap, w.F // 32), dtype=torch.uint8, device=dev)
    st = _lib.load().moe_grouped_gemm_up(
        _ptr(x_perm), _ptr(x_scales), _ptr(w.w13), _ptr(w.w13_scales), _dt_code(w.precision),
        _ptr(group_offsets), w.E, w.H, w.F, R_cap, _ptr(h), _ptr(h_scales), _ptr(ab), _ptr(h_bf16),
        _stream(stream))
    _check("moe_grouped_gemm_up", st)
    return h, h_scales


def moe_grouped_gemm_down(h: torch.Tensor, h_scales: Optional[torch.Tensor], w: PackedWeights,
                          group_offsets: torch.Tensor, *, y_perm: Optional[torch.Tensor] = None,
                          stream=None) -> torch.Tensor:
    """Down projection y_perm = h W2[e] per group -> y_perm [R_cap, H] bf16."""
    fp8 = w.precision == "mxfp8"
    _want(h, "h", torch.uint8 if fp8 else torch.bfloat16, 2)
    _want(group_offsets, "group_offsets", torch.int32, 1)
    R_cap = h.shape[0]
    if y_perm is None:
        y_perm = torch.empty((R_cap, w.H), dtype=torch.bfloat16, device=h.device)
    st = _lib.load().moe_grouped_gemm_down(
        _ptr(h), _ptr(h_scales), _ptr(w.w2), _ptr(w.w2_scales), _dt_code(w.precision), _ptr(group_offsets),
        w.E, w.H, w.F, R_cap, _ptr(y_perm), _stream(stream))
    _check("moe_grouped_gemm_down", st)
    return y_perm


# ---------------------------------------------------------------------- NVFP4
def moe_amax_bf16(x: torch.Tensor, *, valid_rows: Optional[torch.Tensor] = None, amax: Optional[torch.Tensor] = None,
                  stream=None) -> torch.Tensor:
    """max |x| over the rows of a bf16 matrix (over the first *valid_rows rows when that device int
    is given) -> amax [1] fp32 on the device."""
    _want(x, "x", torch.bfloat16, None)
    x2 = x.reshape(-1, x.shape[-1])
    if amax is None:
        amax = torch.empty((1,), dtype=torch.float32, device=x.device)
    st = _lib.load().moe_amax_bf16(_ptr(x2), x2.shape[0], x2.shape[1], _ptr(valid_rows), _ptr(amax), _stream(stream))
    _check("moe_amax_bf16", st)
    return amax


def moe_quant_nvfp4(x: torch.Tensor, amax: torch.Tensor, *, valid_rows: Optional[torch.Tensor] = None,
                    q: Optional[torch.Tensor] = None, scales: Optional[torch.Tensor] = None, stream=None):
    """Row-wise NVFP4 of a bf16 matrix [..., C] with the tensor encode scale of the device amax ->
    (q [..., C/2] uint8 packed E2M1, scales [..., C/16] uint8 E4M3)."""
    _want(x, "x", torch.bfloat16, None)
    C_ = x.shape[-1]
    if q is None:
        q = torch.empty(x.shape[:-1] + (C_ // 2,), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty(x.shape[:-1] + (C_ // 16,), dtype=torch.uint8, device=x.device)
    rows = x.numel() // C_
    st = _lib.load().moe_quant_nvfp4(_ptr(x), rows, C_, _ptr(valid_rows), _ptr(amax), _ptr(q), _ptr(scales),
                                     _stream(stream))
    _check("moe_quant_nvfp4", st)
    return q, scales


class Nvfp4Weights(NamedTuple):
    E: int
    H: int
    F: int
    w13: torch.Tensor          # [E, 2F, H/2] packed E2M1 (the layout of PackedWeights.w13)
    w13_scales: torch.Tensor   # [E, 2F, H/16] E4M3
    w13_amax: torch.Tensor     # [1] fp32
    w2: torch.Tensor           # [E, H, F/2]
    w2_scales: torch.Tensor    # [E, H, F/16]
    w2_amax: torch.Tensor      # [1] fp32


def moe_prepare_weights_nvfp4(w1: torch.Tensor, w3: torch.Tensor, w2: torch.Tensor, stream=None) -> Nvfp4Weights:
    """One-time: pack the logical weights (bf16) into the grouped GEMMs' layouts and quantise each
    stacked tensor row-wise to NVFP4 along its contraction dimension, with its own amax."""
    pw = moe_prepare_weights(w1, w3, w2, "bf16", stream=stream)
    a13 = moe_amax_bf16(pw.w13, stream=stream)
    q13, s13 = moe_quant_nvfp4(pw.w13, a13, stream=stream)
    a2 = moe_amax_bf16(pw.w2, stream=stream)
    q2, s2 = moe_quant_nvfp4(pw.w2, a2, stream=stream)
    return Nvfp4Weights(pw.E, pw.H, pw.F, q13, s13, a13, q2, s2, a2)


def moe_grouped_gemm_up_nvfp4(x_q: torch.Tensor, x_scales: torch.Tensor, x_amax: torch.Tensor, w: Nvfp4Weights,
                              group_offsets: torch.Tensor, *, h: Optional[torch.Tensor] = None,
                              h_amax: Optional[torch.Tensor] = None, ab: Optional[torch.Tensor] = None,
                              stream=None):
    """NVFP4 x [R_cap, H/2] -> (h [R_cap, F] bf16 = silu(x W1) * (x W3), h_amax [1] fp32)."""
    R_cap = x_q.shape[0]
    if h is None:
        h = torch.empty((R_cap, w.F), dtype=torch.bfloat16, device=x_q.device)
    if h_amax is None:
        h_amax = torch.empty((1,), dtype=torch.float32, device=x_q.device)
    st = _lib.load().moe_grouped_gemm_up_nvfp4(
        _ptr(x_q), _ptr(x_scales), _ptr(x_amax), _ptr(w.w13), _ptr(w.w13_scales), _ptr(w.w13_amax),
        _ptr(group_offsets), w.E, w.H, w.F, R_cap, _ptr(h), _ptr(h_amax), _ptr(ab), _stream(stream))
    _check("moe_grouped_gemm_up_nvfp4", st)
    return h, h_amax


def moe_grouped_gemm_down_nvfp4(h_q: torch.Tensor, h_scales: torch.Tensor, h_amax: torch.Tensor, w: Nvfp4Weights,
                                group_offsets: torch.Tensor, *, y_perm: Optional[torch.Tensor] = None,
                                stream=None) -> torch.Tensor:
    """NVFP4 h [R_cap, F/2] -> y_perm [R_cap, H] bf16 = h W2."""
    R_cap = h_q.shape[0]
    if y_perm is None:
        y_perm = torch.empty((R_cap, w.H), dtype=torch.bfloat16, device=h_q.device)
    st = _lib.load().moe_grouped_gemm_down_nvfp4(
        _ptr(h_q), _ptr(h_scales), _ptr(h_amax), _ptr(w.w2), _ptr(w.w2_scales), _ptr(w.w2_amax),
        _ptr(group_offsets), w.E, w.H, w.F, R_cap, _ptr(y_perm), _stream(stream))
    _check("moe_grouped_gemm_down_nvfp4", st)
    return y_perm


class BwdWeights(NamedTuple):
    precision: str
    E: int
    H: int
    F: int
    w2b: torch.Tensor                   # [E, F, H] bf16 or uint8
    w2b_scales: Optional[torch.Tensor]  # [E, F, H/32]
    w13t: torch.Tensor                  # [E, H, 2F]
    w13t_scales: Optional[torch.Tensor]  # [E, H, 2F/32]


def moe_prepare_weights_bwd(w1: torch.Tensor, w3: torch.Tensor, w2: torch.Tensor, precision: str = "bf16",
                            stream=None) -> BwdWeights:
    """Pack logical W1, W3 [E, H, F] and W2 [E, F, H] for the backward GEMMs (one-time)."""
    for t, n in ((w1, "w1"), (w3, "w3"), (w2, "w2")):
        _want(t, n, torch.bfloat16, 3)
    E, H, F = w1.shape
    dev = w1.device
    fp8 = precision == "mxfp8"
    pdt = torch.uint8 if fp8 else torch.bfloat16
    w2b = torch.empty((E, F, H), dtype=pdt, device=dev)
    w13t = torch.empty((E, H, 2 * F), dtype=pdt, device=dev)
    s2 = torch.empty((E, F, H // 32), dtype=torch.uint8, device=dev) if fp8 else None
    s13 = torch.empty((E, H, 2 * F // 32), dtype=torch.uint8, device=dev) if fp8 else None
    st = _lib.load().moe_prepare_weights_bwd(_ptr(w1), _ptr(w3), _ptr(w2), E, H, F, _dt_code(precision),
                                             _ptr(w2b), _ptr(s2), _ptr(w13t), _ptr(s13), _stream(stream))
    _check("moe_prepare_weights_bwd", st)
    return BwdWeights(precision, E, H, F, w2b, s2, w13t, s13)


def moe_grouped_swiglu_dgrad(dy: torch.Tensor, dy_scales: Optional[torch.Tensor], bw: BwdWeights,
                             ab: torch.Tensor, group_offsets: torch.Tensor, *, dab: Optional[torch.Tensor] = None,
                             dab_q: Optional[torch.Tensor] = None, dab_scales: Optional[torch.Tensor] = None,
                             stream=None) -> torch.Tensor:
    """dy [R_cap, H] (bf16 or MXFP8 codes) -> dab [R_cap, 2F] bf16 (da | db interleaved per 128).
    With dab_q [R_cap, 2F] uint8 and dab_scales [R_cap, 2F/32] uint8 given, the epilogue also
    writes the row-wise MXFP8 codes and scales of dab into them."""
    R_cap = dy.shape[0]
    if dab is None:
        dab = torch.empty((R_cap, 2 * bw.F), dtype=torch.bfloat16, device=dy.device)
    if (dab_q is None) != (dab_scales is None):
        raise ValueError("dab_q and dab_scales go together")
    if dab_q is not None:
        _want(dab_q, "dab_q", torch.uint8, 2)
        _want(dab_scales, "dab_scales", torch.uint8, 2)
        if tuple(dab_q.shape) != (R_cap, 2 * bw.F) or tuple(dab_scales.shape) != (R_cap, 2 * bw.F // 32):
            raise ValueError("dab_q must be [R_cap, 2F] and dab_scales [R_cap, 2F/32]")
    st = _lib.load().moe_grouped_swiglu_dgrad(
        _ptr(dy), _ptr(dy_scales), _ptr(bw.w2b), _ptr(bw.w2b_scales), _ptr(ab), _dt_code(bw.precision),
        _ptr(group_offsets), bw.E, bw.H, bw.F, R_cap, _ptr(dab), _ptr(dab_q), _ptr(dab_scales), _stream(stream))
    _check("moe_grouped_swiglu_dgrad", st)
    return dab


def moe_grouped_gemm_dx(dab: torch.Tensor, dab_scales: Optional[torch.Tensor], bw: BwdWeights,
                        group_offsets: torch.Tensor, *, dx: Optional[torch.Tensor] = None,
                        stream=None) -> torch.Tensor:
    """dab [R_cap, 2F] (bf16 or MXFP8 codes) -> dx [R_cap, H] bf16."""
    R_cap = dab.shape[0]
    if dx is None:
        dx = torch.empty((R_cap, bw.H), dtype=torch.bfloat16, device=dab.device)
    st = _lib.load().moe_grouped_gemm_dx(
        _ptr(dab), _ptr(dab_scales), _ptr(bw.w13t), _ptr(bw.w13t_scales), _dt_code(bw.precision),
        _ptr(group_offsets), bw.E, bw.H, bw.F, R_cap, _ptr(dx), _stream(stream))
    _check("moe_grouped_gemm_dx", st)
    return dx


def moe_grouped_transpose_kpad(R_cap: int, E: int) -> int:
    return int(_lib.load().moe_grouped_transpose_kpad(R_cap, E))


def moe_grouped_transpose(x: torch.Tensor, group_offsets: torch.Tensor, precision: str = "bf16", *,
                          R_cap: Optional[int] = None, src_rows: Optional[torch.Tensor] = None,
                          xT: Optional[torch.Tensor] = None, xT_scales: Optional[torch.Tensor] = None,
                          stream=None):
    """Group-padded transposed weight-gradient operand [C, Kpad] (bf16, or MXFP8 + scales)."""
    _want(x, "x", torch.bfloat16, 2)
    C = x.shape[1]
    if R_cap is None:
        R_cap = x.shape[0]
    E = group_offsets.numel() - 1
    kpad = moe_grouped_transpose_kpad(R_cap, E)
    fp8 = precision == "mxfp8"
    if xT is None:
        xT = torch.empty((C, kpad), dtype=torch.uint8 if fp8 else torch.bfloat16, device=x.device)
    if fp8 and xT_scales is None:
        xT_scales = torch.empty((C, kpad // 32), dtype=torch.uint8, device=x.device)
    st = _lib.load().moe_grouped_transpose(_ptr(x), _ptr(src_rows), R_cap, C, _ptr(group_offsets), E,
                                           _dt_code(precision), _ptr(xT), _ptr(xT_scales), _stream(stream))
    _check("moe_grouped_transpose", st)
    return xT, xT_scales


def moe_grouped_gemm_wgrad(aT: torch.Tensor, aT_scales: Optional[torch.Tensor], bT: torch.Tensor,
                           bT_scales: Optional[torch.Tensor], precision: str, group_offsets: torch.Tensor,
                           R_cap: int, *, split: bool = False, dw: Optional[torch.Tensor] = None,
                           dw2: Optional[torch.Tensor] = None, stream=None):
    """dW[e] = sum over group e's rows of a^T b, from transposed operands [M, Kpad], [N, Kpad]."""
    M, N = aT.shape[0], bT.shape[0]
    E = group_offsets.numel() - 1
    dev = aT.device
    if split:
        if dw is None:
            dw = torch.empty((E, M, N // 2), dtype=torch.bfloat16, device=dev)
        if dw2 is None:
            dw2 = torch.empty((E, M, N // 2), dtype=torch.bfloat16, device=dev)
    elif dw is None:
        dw = torch.empty((E, M, N), dtype=torch.bfloat16, device=dev)
    st = _lib.load().moe_grouped_gemm_wgrad(
        _ptr(aT), _ptr(aT_scales), _ptr(bT), _ptr(bT_scales), _dt_code(precision), _ptr(group_offsets), E, M, N,
        R_cap, _ptr(dw), _ptr(dw2 if split else None), _stream(stream))
    _check("moe_grouped_gemm_wgrad", st)
    return (dw, dw2) if split else dw
