"""CPU oracle for the dropless MoE layer hot path (Python access layer).

TEST INFRASTRUCTURE: only the test suite, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package. The library
(``dropless_moe_expert_router_gb300``) never imports it, and this package never
imports the library: the oracle and the CUDA path share no code.

The arithmetic lives in ``moe_oracle.c`` (plain single-threaded C, double
precision); this module compiles it with gcc on first use (or through
``build()``) and wraps each function with numpy marshalling only.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libmoe_oracle.so")
_lock = threading.Lock()
_lib = None

MAT_BF16, MAT_F64, MAT_MXFP8 = 0, 1, 2
H_NONE, H_BF16, H_MXFP8 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the oracle into oracle/_build/libmoe_oracle.so (gcc, -O2, IEEE)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + ".%d.tmp" % os.getpid()
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
             "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            P = C.c_void_p
            i32, i64, dbl = C.c_int, C.c_long, C.c_double
            L.oracle_bf16_to_double.restype = dbl
            L.oracle_bf16_to_double.argtypes = [C.c_uint16]
            L.oracle_double_to_bf16.restype = C.c_uint16
            L.oracle_double_to_bf16.argtypes = [dbl]
            L.oracle_e4m3_decode.restype = dbl
            L.oracle_e4m3_decode.argtypes = [C.c_uint8]
            L.oracle_e4m3_encode.restype = C.c_uint8
            L.oracle_e4m3_encode.argtypes = [dbl]
            L.oracle_e8m0_scale_byte.restype = i32
            L.oracle_e8m0_scale_byte.argtypes = [dbl]
            L.oracle_quant_rows_bf16.restype = None
            L.oracle_quant_rows_bf16.argtypes = [P, i64, i64, P, P]
            L.oracle_quant_cols_grouped_bf16.restype = None
            L.oracle_quant_cols_grouped_bf16.argtypes = [P, i64, P, i32, P, P]
            L.oracle_route_topk.restype = None
            L.oracle_route_topk.argtypes = [P, i32, i32, i32, i32, P, P]
            L.oracle_permute.restype = i64
            L.oracle_permute.argtypes = [P, i32, i32, P, i32, i32, P, P, P, P, P]
            L.oracle_combine.restype = None
            L.oracle_combine.argtypes = [P, P, P, i32, i32, i32, P]
            L.oracle_route_backward.restype = None
            L.oracle_route_backward.argtypes = [P, P, P, i32, i32, i32, i32, P]
            L.oracle_combine_backward.restype = None
            L.oracle_combine_backward.argtypes = [P, P, P, P, i32, i32, i32, P, P]
            L.oracle_permute_backward.restype = None
            L.oracle_permute_backward.argtypes = [P, P, i32, i32, i32, P]
            L.oracle_swiglu_rows.restype = None
            L.oracle_swiglu_rows.argtypes = [i32, P, P, i32, P, P, P, P, P, P, P, i32, i32, i32,
                                             i64, P, i64, i32, P, P, P, P, P, P, P, P]
            L.oracle_swiglu_dgrad_rows.restype = None
            L.oracle_swiglu_dgrad_rows.argtypes = [i32, P, P, i32, P, P, i32, i32, P, P, P, P, P,
                                                   P, P, i32, i32, i32, i64, P, i64, i32, P, P, P, P]
            L.oracle_wgrad_expert.restype = None
            L.oracle_wgrad_expert.argtypes = [i32, P, P, i64, i32, P, P, i64, P, i32, i32, i64,
                                              P, i64, P]
            L.oracle_expert_of_row.restype = i32
            L.oracle_expert_of_row.argtypes = [P, i32, i64]
            L.oracle_route_sigmoid_topk.restype = None
            L.oracle_route_sigmoid_topk.argtypes = [P, P, i32, i32, i32, i32, P, P]
            L.oracle_route_sigmoid_backward.restype = None
            L.oracle_route_sigmoid_backward.argtypes = [P, P, P, i32, i32, i32, i32, P]
            f32 = C.c_float
            L.oracle_e2m1_decode.restype = dbl
            L.oracle_e2m1_decode.argtypes = [C.c_uint8]
            L.oracle_e2m1_encode.restype = C.c_uint8
            L.oracle_e2m1_encode.argtypes = [dbl]
            L.oracle_nvfp4_encode_scale.restype = f32
            L.oracle_nvfp4_encode_scale.argtypes = [f32]
            L.oracle_quant_rows_nvfp4.restype = None
            L.oracle_quant_rows_nvfp4.argtypes = [P, i64, i64, f32, P, P]
            L.oracle_nvfp4_decode.restype = None
            L.oracle_nvfp4_decode.argtypes = [P, P, i64, i64, f32, P]
            L.oracle_double_to_bf16_n.restype = None
            L.oracle_double_to_bf16_n.argtypes = [P, i64, P]
            L.oracle_swiglu_n.restype = None
            L.oracle_swiglu_n.argtypes = [P, P, i64, P]
            L.oracle_swiglu_grad_n.restype = None
            L.oracle_swiglu_grad_n.argtypes = [P, P, P, i64, P, P]
            L.oracle_quant_rows_f64.restype = None
            L.oracle_quant_rows_f64.argtypes = [P, i64, i64, P, P]
            L.oracle_ep_recv_expert_ids.restype = None
            L.oracle_ep_recv_expert_ids.argtypes = [P, i32, i32, i64, P]
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


# ----------------------------------------------------------------- formats
def bf16_to_f64(bits) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f64_to_bf16(v) -> np.ndarray:
    """bf16 bits of float64 values (round to nearest even), element by element in C."""
    flat = np.ascontiguousarray(np.asarray(v, dtype=np.float64).ravel())
    out = np.empty(flat.size, np.uint16)
    lib().oracle_double_to_bf16_n(_p(flat), flat.size, _p(out))
    return out.reshape(np.shape(v))


def e4m3_decode(codes) -> np.ndarray:
    L = lib()
    c = np.asarray(codes, dtype=np.uint8).ravel()
    return np.array([L.oracle_e4m3_decode(int(x)) for x in c]).reshape(np.shape(codes))


def e4m3_encode(v) -> np.ndarray:
    L = lib()
    flat = np.asarray(v, dtype=np.float64).ravel()
    return np.array([L.oracle_e4m3_encode(float(x)) for x in flat],
                    dtype=np.uint8).reshape(np.shape(v))


_E4M3_TABLE = None


def e4m3_table() -> np.ndarray:
    """The 256 E4M3 code values (oracle_e4m3_decode of every code), float64."""
    global _E4M3_TABLE
    if _E4M3_TABLE is None:
        L = lib()
        _E4M3_TABLE = np.array([L.oracle_e4m3_decode(c) for c in range(256)], np.float64)
    return _E4M3_TABLE


def mx_decode_rows(q, s) -> np.ndarray:
    """Values (float64) of row-wise MXFP8 [rows, cols] codes with [rows, cols/32] scales:
    code value times 2^(scale byte - 127) (exact in float64)."""
    q = np.asarray(q, np.uint8)
    sc = np.ldexp(1.0, np.asarray(s, np.int64) - 127)
    return e4m3_table()[q] * np.repeat(sc, 32, axis=-1)


def mx_decode_cols(q, s) -> np.ndarray:
    """Values (float64) of column-wise MXFP8 codes of one group [rows, cols] starting at
    row 0, scales [rows/32 (rounded up), cols]: block b covers rows 32b .. 32b + 31."""
    q = np.asarray(q, np.uint8)
    sc = np.ldexp(1.0, np.asarray(s, np.int64) - 127)
    return e4m3_table()[q] * np.repeat(sc, 32, axis=0)[: q.shape[0]]


def e8m0_scale_byte(amax: float) -> int:
    return lib().oracle_e8m0_scale_byte(float(amax))


def quant_rows_f64(x):
    """Row-wise 1x32 MXFP8 of a float64 matrix (unrounded values) -> (q, s)."""
    xv = _c(x, np.float64)
    rows, cols = xv.shape
    q = np.zeros((rows, cols), np.uint8)
    s = np.zeros((rows, cols // 32), np.uint8)
    lib().oracle_quant_rows_f64(_p(xv), rows, cols, _p(q), _p(s))
    return q, s


def quant_rows(x_bf16):
    """Row-wise 1x32 MXFP8 of a bf16 matrix -> (q [rows, cols] u8, s [rows, cols/32] u8)."""
    x = _c(x_bf16, np.uint16)
    rows, cols = x.shape
    q = np.zeros((rows, cols), np.uint8)
    s = np.zeros((rows, cols // 32), np.uint8)
    lib().oracle_quant_rows_bf16(_p(x), rows, cols, _p(q), _p(s))
    return q, s


def e2m1_decode(code: int) -> float:
    return lib().oracle_e2m1_decode(int(code))


def e2m1_encode(v: float) -> int:
    return int(lib().oracle_e2m1_encode(float(v)))


def nvfp4_encode_scale(amax: float) -> float:
    """The fp32 tensor encode scale 448 * 6 / amax (1 for an all-zero tensor)."""
    return float(lib().oracle_nvfp4_encode_scale(float(np.float32(amax))))


def bf16_amax(x_bf16) -> float:
    """max |x| of a bf16 matrix (exact)."""
    return float(np.abs(bf16_to_f64(x_bf16)).max(initial=0.0))


def quant_rows_nvfp4(x_bf16, S=None):
    """Row-wise NVFP4 of a bf16 matrix -> (q [rows, cols/2] packed E2M1, s [rows, cols/16] E4M3,
    S the fp32 encode scale used: that of x's own amax unless given)."""
    x = _c(x_bf16, np.uint16)
    rows, cols = x.shape
    if S is None:
        S = nvfp4_encode_scale(bf16_amax(x))
    q = np.zeros((rows, cols // 2), np.uint8)
    s = np.zeros((rows, cols // 16), np.uint8)
    lib().oracle_quant_rows_nvfp4(_p(x), rows, cols, float(S), _p(q), _p(s))
    return q, s, float(S)


def nvfp4_decode(q, s, S):
    """Values (float64) of an NVFP4 matrix."""
    qv = _c(q, np.uint8)
    sv = _c(s, np.uint8)
    rows, half = qv.shape
    out = np.zeros((rows, 2 * half))
    lib().oracle_nvfp4_decode(_p(qv), _p(sv), rows, 2 * half, float(S), _p(out))
    return out


def grouped_matmul(a, b, group_offsets):
    """out[r] = a[r] @ b[e].T for the rows r of each group e (a [R, K], b [E, N, K], float64;
    a library matmul per group). Rows past the last group stay 0."""
    off = np.asarray(group_offsets, np.int64)
    out = np.zeros((a.shape[0], b.shape[1]))
    for e in range(off.size - 1):
        if off[e + 1] > off[e]:
            out[off[e]:off[e + 1]] = a[off[e]:off[e + 1]] @ b[e].T
    return out


def colwise_scale_rows(R_cap: int, E: int) -> int:
    """Rows of the padded group-aware column-wise scale layout."""
    return E + R_cap // 32 + 1


def quant_cols_grouped(x_bf16, group_offsets, fill_q=0, fill_s=0):
    """Group-aware column-wise (32x1) MXFP8 of a bf16 matrix [R_cap, cols]."""
    x = _c(x_bf16, np.uint16)
    off = _c(group_offsets, np.int32)
    R_cap, cols = x.shape
    E = off.size - 1
    q = np.full((R_cap, cols), fill_q, np.uint8)
    s = np.full((colwise_scale_rows(R_cap, E), cols), fill_s, np.uint8)
    lib().oracle_quant_cols_grouped_bf16(_p(x), cols, _p(off), E, _p(q), _p(s))
    return q, s


# ------------------------------------------------------------------ router
def route_topk(logits, K: int, renorm: bool = False):
    lg = _c(logits, np.float32)
    T, E = lg.shape
    ids = np.zeros((T, K), np.int32)
    probs = np.zeros((T, K), np.float32)
    lib().oracle_route_topk(_p(lg), T, E, K, int(bool(renorm)), _p(ids), _p(probs))
    return ids, probs


def route_sigmoid_topk(logits, K: int, bias=None, renorm: bool = False):
    """Sigmoid scores, selection on score + bias -> (ids [T, K] int32, probs [T, K] fp32)."""
    lg = _c(logits, np.float32)
    T, E = lg.shape
    b = None if bias is None else _c(bias, np.float32)
    ids = np.zeros((T, K), np.int32)
    probs = np.zeros((T, K), np.float32)
    lib().oracle_route_sigmoid_topk(_p(lg), _p(b), T, E, K, int(bool(renorm)), _p(ids), _p(probs))
    return ids, probs


def route_sigmoid_backward(logits, ids, dprobs, renorm: bool = False):
    """dlogits [T, E] (float64) of route_sigmoid_topk's probabilities, selection held fixed."""
    lg = _c(logits, np.float32)
    T, E = lg.shape
    idv = _c(ids, np.int32)
    K = idv.shape[1]
    dp = _c(dprobs, np.float32)
    out = np.zeros((T, E), np.float64)
    lib().oracle_route_sigmoid_backward(_p(lg), _p(idv), _p(dp), T, E, K, int(bool(renorm)), _p(out))
    return out


# ----------------------------------------------------------------- permute
def permute(x_bf16, ids, E: int):
    """Returns dict(x_perm [T*K, H] (rows >= R zero), group_sizes, group_offsets,
    row_map [T,K], perm_src [T*K] (entries >= R are -1), R)."""
    idv = _c(ids, np.int32)
    T, K = idv.shape
    if x_bf16 is None:
        x, H = None, 0
    else:
        x = _c(x_bf16, np.uint16)
        H = x.shape[1]
    xp = None if x is None else np.zeros((T * K, H), np.uint16)
    gs = np.zeros(E, np.int32)
    go = np.zeros(E + 1, np.int32)
    rm = np.zeros((T, K), np.int32)
    ps = np.full(T * K, -1, np.int32)
    R = lib().oracle_permute(_p(x), T, H, _p(idv), K, E, _p(xp), _p(gs), _p(go), _p(rm), _p(ps))
    return dict(x_perm=xp, group_sizes=gs, group_offsets=go, row_map=rm, perm_src=ps, R=int(R))


# ----------------------------------------------------------------- combine
def combine(y_perm_bf16, row_map, probs):
    yp = _c(y_perm_bf16, np.uint16)
    rm = _c(row_map, np.int32)
    pr = _c(probs, np.float32)
    T, K = rm.shape
    H = yp.shape[1]
    y = np.zeros((T, H), np.uint16)
    lib().oracle_combine(_p(yp), _p(rm), _p(pr), T, K, H, _p(y))
    return y


# ---------------------------------------------------------------- backward
def route_backward(logits, ids, dprobs, renorm: bool = False):
    """dlogits [T, E] (float64) of the router's probabilities, selection held fixed."""
    lg = _c(logits, np.float32)
    T, E = lg.shape
    idv = _c(ids, np.int32)
    K = idv.shape[1]
    dp = _c(dprobs, np.float32)
    out = np.zeros((T, E), np.float64)
    lib().oracle_route_backward(_p(lg), _p(idv), _p(dp), T, E, K, int(bool(renorm)), _p(out))
    return out


def combine_backward(dy_bf16, y_perm_bf16, row_map, probs, dy_perm_init=None):
    """(dy_perm [rows of y_perm, H] bf16 bits -- rows no route maps to keep dy_perm_init
    (zeros by default) --, dprobs [T, K] float64)."""
    dy = _c(dy_bf16, np.uint16)
    yp = _c(y_perm_bf16, np.uint16)
    rm = _c(row_map, np.int32)
    pr = _c(probs, np.float32)
    T, K = rm.shape
    H = yp.shape[1]
    dyp = np.zeros(yp.shape, np.uint16) if dy_perm_init is None else np.array(dy_perm_init, np.uint16)
    dp = np.zeros((T, K), np.float64)
    lib().oracle_combine_backward(_p(dy), _p(yp), _p(rm), _p(pr), T, K, H, _p(dyp), _p(dp))
    return dyp, dp


def permute_backward(dx_perm_bf16, row_map):
    """dx [T, H] bf16 bits: the sum over each token's valid routes of its dx_perm rows."""
    dxp = _c(dx_perm_bf16, np.uint16)
    rm = _c(row_map, np.int32)
    T, K = rm.shape
    H = dxp.shape[1]
    dx = np.zeros((T, H), np.uint16)
    lib().oracle_permute_backward(_p(dxp), _p(rm), T, K, H, _p(dx))
    return dx


# ------------------------------------------------------------ grouped MLP
class Operand:
    """An oracle operand: kind MAT_BF16 (uint16 bits), MAT_F64 or MAT_MXFP8 (codes + scales)."""

    def __init__(self, kind, v, s=None):
        self.kind = kind
        dt = {MAT_BF16: np.uint16, MAT_F64: np.float64, MAT_MXFP8: np.uint8}[kind]
        self.v = np.ascontiguousarray(v, dtype=dt)
        self.s = None if s is None else np.ascontiguousarray(s, dtype=np.uint8)


def swiglu_rows(x: Operand, w1: Operand, w3: Operand, w2: Operand, group_offsets, rows,
                h_mode=H_BF16, want=("y_bf16",)):
    """Grouped SwiGLU MLP for the listed permuted rows. `want` picks outputs among
    y_bf16, y_f64, h_bf16, h_q, h_s, h_f64, a_f64, b_f64."""
    off = _c(group_offsets, np.int32)
    E = off.size - 1
    R_cap, H = x.v.shape
    F = w1.v.shape[-1]
    rw = _c(rows, np.int32)
    n = rw.size
    outs = {
        "y_bf16": np.zeros((n, H), np.uint16) if "y_bf16" in want else None,
        "y_f64": np.zeros((n, H)) if "y_f64" in want else None,
        "h_bf16": np.zeros((n, F), np.uint16) if "h_bf16" in want else None,
        "h_q": np.zeros((n, F), np.uint8) if "h_q" in want else None,
        "h_s": np.zeros((n, F // 32), np.uint8) if "h_s" in want else None,
        "h_f64": np.zeros((n, F)) if "h_f64" in want else None,
        "a_f64": np.zeros((n, F)) if "a_f64" in want else None,
        "b_f64": np.zeros((n, F)) if "b_f64" in want else None,
    }
    lib().oracle_swiglu_rows(
        x.kind, _p(x.v), _p(x.s), w1.kind, _p(w1.v), _p(w1.s), _p(w3.v), _p(w3.s),
        _p(w2.v), _p(w2.s), _p(off), E, H, F, R_cap, _p(rw), n, h_mode,
        _p(outs["y_bf16"]), _p(outs["y_f64"]), _p(outs["h_bf16"]), _p(outs["h_q"]),
        _p(outs["h_s"]), _p(outs["h_f64"]), _p(outs["a_f64"]), _p(outs["b_f64"]))
    return {k: v for k, v in outs.items() if v is not None}


DAB_NONE, DAB_BF16, DAB_MXFP8 = 0, 1, 2


def swiglu_dgrad_rows(dy: Operand, a: Operand, b: Operand, w1: Operand, w3: Operand,
                      w2: Operand, group_offsets, rows, w_blk_rows=0, dab_mode=DAB_NONE,
                      want=("dx_bf16",)):
    off = _c(group_offsets, np.int32)
    E = off.size - 1
    R_cap, H = dy.v.shape
    F = w1.v.shape[-1]
    rw = _c(rows, np.int32)
    n = rw.size
    outs = {
        "dx_bf16": np.zeros((n, H), np.uint16) if "dx_bf16" in want else None,
        "dx_f64": np.zeros((n, H)) if "dx_f64" in want else None,
        "da_f64": np.zeros((n, F)) if "da_f64" in want else None,
        "db_f64": np.zeros((n, F)) if "db_f64" in want else None,
    }
    assert a.kind == b.kind
    lib().oracle_swiglu_dgrad_rows(
        dy.kind, _p(dy.v), _p(dy.s), a.kind, _p(a.v), _p(b.v), w1.kind, int(w_blk_rows),
        _p(w1.v), _p(w1.s), _p(w3.v), _p(w3.s), _p(w2.v), _p(w2.s), _p(off), E, H, F, R_cap,
        _p(rw), n, int(dab_mode), _p(outs["dx_bf16"]), _p(outs["dx_f64"]), _p(outs["da_f64"]),
        _p(outs["db_f64"]))
    return {k: v for k, v in outs.items() if v is not None}


def wgrad_expert(A: Operand, B: Operand, group_offsets, e: int, cols=None):
    """dW[c1, c2] = sum over group e's rows of A[r, c1] * B[r, c2], for c2 in cols."""
    off = _c(group_offsets, np.int32)
    E = off.size - 1
    R_cap, n1 = A.v.shape
    n2 = B.v.shape[1]
    cl = np.arange(n2, dtype=np.int32) if cols is None else _c(cols, np.int32)
    out = np.zeros((n1, cl.size))
    lib().oracle_wgrad_expert(A.kind, _p(A.v), _p(A.s), n1, B.kind, _p(B.v), _p(B.s), n2,
                              _p(off), E, int(e), R_cap, _p(cl), cl.size, _p(out))
    return out


def expert_of_row(group_offsets, r: int) -> int:
    off = _c(group_offsets, np.int32)
    return lib().oracle_expert_of_row(_p(off), off.size - 1, int(r))


# ------------------------------------------------- whole-expert blocks of rows
def swiglu(a, b) -> np.ndarray:
    """h = silu(a) * b element by element (the SwiGLU step, in C)."""
    av, bv = _c(a, np.float64), _c(b, np.float64)
    h = np.empty(av.shape)
    lib().oracle_swiglu_n(_p(av), _p(bv), av.size, _p(h))
    return h


def swiglu_grad(dh, a, b):
    """(da, db) of the SwiGLU step at (a, b) applied to dh (in C)."""
    dv, av, bv = _c(dh, np.float64), _c(a, np.float64), _c(b, np.float64)
    da, db = np.empty(av.shape), np.empty(av.shape)
    lib().oracle_swiglu_grad_n(_p(dv), _p(av), _p(bv), av.size, _p(da), _p(db))
    return da, db


def expert_swiglu_block(xv, w1v, w3v, w2v=None, h_mode=H_BF16):
    """One expert's grouped SwiGLU MLP on a block of its rows, from operand VALUES (decoded
    bf16 / MXFP8 / NVFP4, float64), as oracle_swiglu_rows defines it for each row:
      a = x W1, b = x W3 (a library matmul per product, float64),
      h = silu(a) * b; with w2v: y = round_h(h) W2.
    xv [n, H]; w1v, w3v [H, F'] -- any F' columns of the expert's F (every output column is
    independent of the others); w2v [F, H] (all F columns needed). round_h is bf16 (H_BF16),
    MXFP8 1x32 along F from the unrounded h (H_MXFP8), or none (H_NONE).
    Returns dict(a, b, h (unrounded), h_bf16 (bits, H_BF16), h_q / h_s (H_MXFP8),
    y (float64, unrounded; with w2v))."""
    a = np.asarray(xv) @ np.asarray(w1v)
    b = np.asarray(xv) @ np.asarray(w3v)
    h = swiglu(a, b)
    out = dict(a=a, b=b, h=h)
    if h_mode == H_BF16:
        out["h_bf16"] = f64_to_bf16(h)
        hr = bf16_to_f64(out["h_bf16"])
    elif h_mode == H_MXFP8:
        out["h_q"], out["h_s"] = quant_rows_f64(h)
        hr = mx_decode_rows(out["h_q"], out["h_s"])
    else:
        hr = h
    if w2v is not None:
        out["y"] = hr @ np.asarray(w2v)
    return out


def expert_swiglu_dgrad_block(dyv, w2v_rows, a_bf16, b_bf16):
    """One expert's SwiGLU backward on a block of its rows at F' columns, as
    oracle_swiglu_dgrad_rows defines it per row:
      dh = dy W2^T at those columns (a library matmul, float64), then (da, db) from dh and
      the saved bf16 pre-activations a, b.
    dyv [n, H] values; w2v_rows [F', H]: the rows of the expert's W2 [F, H] at the F'
    columns (values as the backward contracts them); a_bf16, b_bf16 [n, F'] bits.
    Returns (da, db) unrounded, float64."""
    dh = np.asarray(dyv) @ np.asarray(w2v_rows).T
    return swiglu_grad(dh, bf16_to_f64(a_bf16), bf16_to_f64(b_bf16))


# ------------------------------------------------------ expert parallelism
def ep_recv_expert_ids(counts, R_cap: int):
    """Local expert (int32) of each row a rank receives in the expert-parallel dispatch:
    counts [G, E_loc] = rows from source s for local expert j, received source by source and
    expert by expert; rows past them -> -1."""
    c = _c(counts, np.int32)
    G, E_loc = c.shape
    ids = np.empty(int(R_cap), np.int32)
    lib().oracle_ep_recv_expert_ids(_p(c), G, E_loc, int(R_cap), _p(ids))
    return ids
