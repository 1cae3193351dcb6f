"""GPU parity of the weight packing and the grouped SwiGLU GEMMs (BF16 and
MXFP8) against the CPU oracle, through the C ABI.

Bar: packed weights (a transposition, plus MXFP8 codes and scales) bit-exact;
h and y_perm within max|err| / max|ref| <= 1e-2 (BF16) or 3e-2 (MXFP8). Large
workloads compare a seeded sample of rows (rows are independent, so a sampled
row is exact parity for that row): the first and last row of every group plus
random rows."""
import numpy as np
import pytest
import torch

import oracle as O
from dropless_moe_expert_router_gb300 import api, workloads as W
from helpers import bf16_bits, rel_err, u8

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dropless_moe_expert_router_gb300 import build
    build.build()
    api.moe_get_device_errors(clear=True)


def _w13_row(f, half):
    return (f // 128) * 256 + half * 128 + (f % 128)


def _oracle_weight_quant(w):
    """Oracle MXFP8 of logical weights [E, Kc, N] along their contraction dim Kc
    -> (q [E, Kc, N], s [E, Kc/32, N]) in the oracle's view layout (experts quantised on a
    thread pool: the C oracle is reentrant and releases the interpreter while it runs)."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    with ThreadPoolExecutor(max_workers=max(1, os.cpu_count() or 1)) as pool:
        parts = list(pool.map(lambda e: O.quant_rows(np.ascontiguousarray(bf16_bits(w[e]).T)), range(w.shape[0])))
    return (np.ascontiguousarray(np.stack([q.T for q, _ in parts])),
            np.ascontiguousarray(np.stack([s.T for _, s in parts])))


def _sample_rows(off, n_random, seed=0, tile_rows=None):
    """The first and last row of every group, n_random random rows, and with tile_rows one
    random row in every tile_rows-row tile of every group (tiles start at each group's first
    row, as the GEMM's row tiles do)."""
    off = np.asarray(off)
    R = int(off[-1])
    rows = set()
    g = np.random.default_rng(seed)
    for e in range(off.size - 1):
        if off[e + 1] > off[e]:
            rows.add(int(off[e]))
            rows.add(int(off[e + 1]) - 1)
            if tile_rows:
                for t0 in range(int(off[e]), int(off[e + 1]), tile_rows):
                    rows.add(int(g.integers(t0, min(t0 + tile_rows, int(off[e + 1])))))
    if R > 0:
        rows.update(int(r) for r in g.choice(R, size=min(n_random, R), replace=False))
    return np.array(sorted(rows), np.int32)


def _run(wl, precision, n_random=None, sizes=None, seed=0, tile_rows=None):
    """GPU: route -> permute -> packed weights -> grouped SwiGLU GEMM.
    Oracle: its own route -> permute -> quantisation -> grouped MLP on sampled rows."""
    fp8 = precision == "mxfp8"
    x = W.x(wl, seed)
    w1, w3, w2 = W.weights(wl, seed)
    if sizes is None:
        lg = W.logits(wl, seed)
        ids, _ = O.route_topk(lg.numpy(), wl.K, wl.renorm)
    else:  # hand-made group sizes: token t routes to expert e(t) in slot 0, invalid elsewhere
        ids = -np.ones((wl.T, wl.K), np.int32)
        col = np.repeat(np.arange(len(sizes)), sizes)[: wl.T]
        ids[: col.size, 0] = col
    op = O.permute(None, ids, wl.E)
    off = op["group_offsets"]
    # GPU path
    dev = torch.device("cuda")
    p = api.moe_permute(x.to(dev), torch.from_numpy(ids).to(dev), wl.E, fuse_mxfp8=fp8)
    pw = api.moe_prepare_weights(w1.to(dev), w3.to(dev), w2.to(dev), precision)
    y_perm, h, hs = api.moe_grouped_swiglu_gemm(p.x_perm, p.x_perm_scales, pw, p.group_offsets)
    torch.cuda.synchronize()
    assert api.moe_get_device_errors() == 0
    rows = np.arange(op["R"], dtype=np.int32) if n_random is None else _sample_rows(off, n_random, seed, tile_rows)
    # oracle operands
    if fp8:
        xq, xs = O.quant_rows(bf16_bits(x))
        src = op["perm_src"][: wl.R_cap].copy()
        src[src < 0] = 0
        X = O.Operand(O.MAT_MXFP8, xq[src], xs[src])
        wq = [_oracle_weight_quant(w) for w in (w1, w3, w2)]
        Ws = [O.Operand(O.MAT_MXFP8, q, s) for q, s in wq]
        out = O.swiglu_rows(X, *Ws, off, rows, h_mode=O.H_MXFP8, want=("y_bf16", "h_q", "h_s", "h_f64"))
    elif rows.size > 64:
        # many sampled rows of a wide layer: the oracle's expert-block forward, one expert at a time
        xb = bf16_bits(x)
        src = op["perm_src"]
        out = dict(y_bf16=np.zeros((rows.size, wl.H), np.uint16), h_bf16=np.zeros((rows.size, wl.F), np.uint16))
        ex = np.array([O.expert_of_row(off, int(r)) for r in rows])
        for e in np.unique(ex):
            sel = np.nonzero(ex == e)[0]
            wv = [O.bf16_to_f64(bf16_bits(w[e])) for w in (w1, w3, w2)]
            blk = O.expert_swiglu_block(O.bf16_to_f64(xb[src[rows[sel]]]), *wv, h_mode=O.H_BF16)
            out["h_bf16"][sel] = blk["h_bf16"]
            out["y_bf16"][sel] = O.f64_to_bf16(blk["y"])
        wq = None
    else:
        xp = np.zeros((wl.R_cap, wl.H), np.uint16)
        xb = bf16_bits(x)
        src = op["perm_src"]
        xp[: op["R"]] = xb[src[: op["R"]]]
        X = O.Operand(O.MAT_BF16, xp)
        Ws = [O.Operand(O.MAT_BF16, bf16_bits(w)) for w in (w1, w3, w2)]
        out = O.swiglu_rows(X, *Ws, off, rows, h_mode=O.H_BF16, want=("y_bf16", "h_bf16"))
        wq = None
    ridx = torch.from_numpy(rows).long().to(dev)
    res = dict(rows=rows, off=off, out=out, y=bf16_bits(y_perm.index_select(0, ridx)),
               h=h.index_select(0, ridx), hs=None if hs is None else hs.index_select(0, ridx),
               pw=pw, wq=wq, w=(w1, w3, w2))
    return res


def _check_bf16(res):
    h_ref = O.bf16_to_f64(res["out"]["h_bf16"])
    h_got = O.bf16_to_f64(bf16_bits(res["h"]))
    assert rel_err(h_got, h_ref) <= 1e-2
    y_ref = O.bf16_to_f64(res["out"]["y_bf16"])
    y_got = O.bf16_to_f64(res["y"])
    e = rel_err(y_got, y_ref)
    assert e <= 1e-2, e
    return e


def _mx_decode(q, s):
    v = torch.from_numpy(np.ascontiguousarray(q)).view(torch.float8_e4m3fn).double().numpy()
    return v * np.exp2(np.repeat(s.astype(np.float64), 32, axis=-1) - 127)


def _check_mxfp8(res):
    h_ref = _mx_decode(res["out"]["h_q"], res["out"]["h_s"])
    h_got = _mx_decode(u8(res["h"]), u8(res["hs"]))
    assert rel_err(h_got, h_ref) <= 3e-2
    y_ref = O.bf16_to_f64(res["out"]["y_bf16"])
    y_got = O.bf16_to_f64(res["y"])
    e = rel_err(y_got, y_ref)
    assert e <= 3e-2, e
    return e


# --------------------------------------------------------------- packing
@pytest.mark.parametrize("precision", ["bf16", "mxfp8"])
def test_weight_packing_matches_layout_and_oracle_quantisation(precision):
    wl = W.get("tiny", E=3, H=256, F=384)
    w1, w3, w2 = W.weights(wl)
    pw = api.moe_prepare_weights(w1.cuda(), w3.cuda(), w2.cuda(), precision)
    torch.cuda.synchronize()
    F = wl.F
    perm1 = np.array([_w13_row(f, 0) for f in range(F)])
    perm3 = np.array([_w13_row(f, 1) for f in range(F)])
    if precision == "bf16":
        w13 = bf16_bits(pw.w13)
        assert np.array_equal(w13[:, perm1, :], bf16_bits(w1).transpose(0, 2, 1))
        assert np.array_equal(w13[:, perm3, :], bf16_bits(w3).transpose(0, 2, 1))
        assert np.array_equal(bf16_bits(pw.w2), bf16_bits(w2).transpose(0, 2, 1))
    else:
        q13, s13, q2, s2 = u8(pw.w13), u8(pw.w13_scales), u8(pw.w2), u8(pw.w2_scales)
        for w, perm in ((w1, perm1), (w3, perm3)):
            oq, os_ = _oracle_weight_quant(w)     # [E, H, F], [E, H/32, F]
            assert np.array_equal(q13[:, perm, :], oq.transpose(0, 2, 1))
            assert np.array_equal(s13[:, perm, :], os_.transpose(0, 2, 1))
        oq, os_ = _oracle_weight_quant(w2)        # [E, F, H], [E, F/32, H]
        assert np.array_equal(q2, oq.transpose(0, 2, 1))
        assert np.array_equal(s2, os_.transpose(0, 2, 1))


# ------------------------------------------------------------------ BF16
def test_gemm_bf16_tiny_all_rows():
    _check_bf16(_run(W.get("tiny"), "bf16"))


@pytest.mark.parametrize("sizes", [(0, 1, 127, 129, 300, 0, 3), (600,), (1, 1, 1, 1), (0, 0, 0, 256)])
def test_gemm_bf16_ragged_groups(sizes):
    T = int(sum(sizes)) + 5
    wl = W.get("tiny", T=T, E=len(sizes), K=1, H=256, F=256)
    _check_bf16(_run(wl, "bf16", sizes=list(sizes)))


def test_gemm_bf16_pair_tiles_ragged():
    """Enough rows per expert for 256-row CTA-pair tiles: empty, 1-row and ragged groups,
    pair tiles whose second CTA has no valid row."""
    sizes = (0, 700, 1, 513, 0, 1024)
    wl = W.get("tiny", T=3200, E=len(sizes), K=1, H=256, F=256)
    _check_bf16(_run(wl, "bf16", sizes=list(sizes)))


def test_gemm_bf16_mixtral_sampled():
    """Full Mixtral-like shape: one random row in every 256-row CTA-pair tile of every expert
    (72 tiles), the first and last row of every group and 16 random rows."""
    res = _run(W.get("mixtral"), "bf16", n_random=16, tile_rows=256)
    off = np.asarray(res["off"])
    tiles = sum(-(-int(off[e + 1] - off[e]) // 256) for e in range(off.size - 1))
    covered = {(O.expert_of_row(off, int(r)), (int(r) - int(off[O.expert_of_row(off, int(r))])) // 256)
               for r in res["rows"]}
    assert len(covered) == tiles
    _check_bf16(res)


def test_gemm_bf16_large_e_sampled():
    _check_bf16(_run(W.get("large_e"), "bf16", n_random=1500))


# ----------------------------------------------------------------- MXFP8
def test_gemm_mxfp8_tiny_all_rows():
    _check_mxfp8(_run(W.get("tiny", precision="mxfp8", H=512, F=512), "mxfp8"))


@pytest.mark.parametrize("sizes", [(0, 1, 127, 129, 300, 0, 3), (1, 1, 1, 1)])
def test_gemm_mxfp8_ragged_groups(sizes):
    T = int(sum(sizes)) + 5
    wl = W.get("tiny", T=T, E=len(sizes), K=1, H=512, F=512, precision="mxfp8")
    _check_mxfp8(_run(wl, "mxfp8", sizes=list(sizes)))


def test_gemm_mxfp8_wide_h_ragged():
    """A wider MXFP8 layer (H = 3584, seven scale boxes per row; 14 output tiles of the
    down projection), every row of ragged groups checked."""
    sizes = (0, 1, 127, 129, 300, 0, 3)
    T = int(sum(sizes)) + 5
    wl = W.get("tiny", T=T, E=len(sizes), K=1, H=3584, F=512, precision="mxfp8")
    _check_mxfp8(_run(wl, "mxfp8", sizes=list(sizes)))


def test_gemm_mxfp8_dsv3_sampled():
    _check_mxfp8(_run(W.get("dsv3"), "mxfp8", n_random=64))
