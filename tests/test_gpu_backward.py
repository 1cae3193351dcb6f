"""GPU parity of the grouped backward (dgrad, weight packing for it, group-padded
transposition, wgrad) against the CPU oracle, through the C ABI.

Bar: transposed operands (a data movement, plus MXFP8 codes and scales)
bit-exact; saved pre-activations, dab, dx and dW within max|err| / max|ref|
<= 1e-2 (bf16) or 3e-2 (MXFP8). At the full heavy-skew shape the oracle makes
every operand itself: sampled rows of the forward and of dab / dx, and whole
experts (every row) at sampled columns of F for a|b, h, dab and the three weight
gradients."""
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


def _interleave(a, b):
    """[R, F] + [R, F] -> [R, 2F] with 128-column blocks a | b (the packed layout)."""
    R, F = a.shape
    out = np.empty((R, 2 * F), a.dtype)
    for j in range(F // 128):
        out[:, 256 * j:256 * j + 128] = a[:, 128 * j:128 * j + 128]
        out[:, 256 * j + 128:256 * j + 256] = b[:, 128 * j:128 * j + 128]
    return out


def _quant_along_rows_of(w):
    """Oracle MXFP8 of [E, rows, cols] weights with blocks along cols -> (q, s [E, rows, cols/32])."""
    qs, ss = zip(*(O.quant_rows(bf16_bits(w[e])) for e in range(w.shape[0])))
    return np.stack(qs), np.stack(ss)


def _quant_along_cols_of(w):
    """... with blocks along rows (contraction over rows) -> (q [E, rows, cols], s [E, rows/32, cols])."""
    qs, ss = [], []
    for e in range(w.shape[0]):
        q, s = O.quant_rows(np.ascontiguousarray(bf16_bits(w[e]).T))
        qs.append(q.T)
        ss.append(s.T)
    return np.ascontiguousarray(np.stack(qs)), np.ascontiguousarray(np.stack(ss))


def _padded_cols(off):
    """Padded contraction column of every permuted row r < R: P_e + (r - off[e])."""
    off = np.asarray(off)
    cols = np.empty(int(off[-1]), np.int64)
    for e in range(off.size - 1):
        P = 128 * (e + off[e] // 128)
        cols[off[e]:off[e + 1]] = P + np.arange(off[e + 1] - off[e])
    return cols


def _gpu_backward(wl, ids, precision, seed=0):
    fp8 = precision == "mxfp8"
    dev = torch.device("cuda")
    x = W.x(wl, seed)
    w1, w3, w2 = W.weights(wl, seed)
    dy = W.dy_perm(wl, seed)
    p = api.moe_permute(x.to(dev), torch.from_numpy(ids).to(dev), wl.E, fuse_mxfp8=fp8)
    goff = p.group_offsets
    pw = api.moe_prepare_weights(w1.to(dev), w3.to(dev), w2.to(dev), precision)
    bw = api.moe_prepare_weights_bwd(w1.to(dev), w3.to(dev), w2.to(dev), precision)
    R_cap = wl.R_cap
    ab = torch.empty((R_cap, 2 * wl.F), dtype=torch.bfloat16, device=dev)
    h_bf16 = torch.empty((R_cap, wl.F), dtype=torch.bfloat16, device=dev) if fp8 else None
    h, hs = api.moe_grouped_gemm_up(p.x_perm, p.x_perm_scales, pw, goff, ab=ab, h_bf16=h_bf16)
    y = api.moe_grouped_gemm_down(h, hs, pw, goff)
    dyd = dy.to(dev)
    if fp8:
        dyq, dys = api.moe_quant_mxfp8_grouped(dyd, goff)
        dabq = torch.zeros((R_cap, 2 * wl.F), dtype=torch.uint8, device=dev)
        dabs = torch.zeros((R_cap, 2 * wl.F // 32), dtype=torch.uint8, device=dev)
        dab = api.moe_grouped_swiglu_dgrad(dyq, dys, bw, ab, goff, dab_q=dabq, dab_scales=dabs)
        # the epilogue's codes and scales of dab are the row quantiser's (pinned to the oracle's)
        sq, ss = api.moe_quant_mxfp8_grouped(dab, goff)
        R = int(goff[-1].item())
        assert torch.equal(dabq[:R], sq[:R]) and torch.equal(dabs[:R], ss[:R])
        dx = api.moe_grouped_gemm_dx(dabq, dabs, bw, goff)
    else:
        dab = api.moe_grouped_swiglu_dgrad(dyd, None, bw, ab, goff)
        dx = api.moe_grouped_gemm_dx(dab, None, bw, goff)
    hT, hTs = api.moe_grouped_transpose(h_bf16 if fp8 else h, goff, precision)
    dyT, dyTs = api.moe_grouped_transpose(dyd, goff, precision)
    xT, xTs = api.moe_grouped_transpose(x.to(dev), goff, precision, R_cap=R_cap, src_rows=p.perm_src)
    dabT, dabTs = api.moe_grouped_transpose(dab, goff, precision)
    dW2 = api.moe_grouped_gemm_wgrad(hT, hTs, dyT, dyTs, precision, goff, R_cap)
    dW1, dW3 = api.moe_grouped_gemm_wgrad(xT, xTs, dabT, dabTs, precision, goff, R_cap, split=True)
    torch.cuda.synchronize()
    assert api.moe_get_device_errors() == 0
    return dict(x=x, w=(w1, w3, w2), dy=dy, ab=ab, h_bf16=h_bf16, h=h, hs=hs, y=y, dab=dab, dx=dx, dW1=dW1, dW3=dW3,
                dW2=dW2, T=dict(hT=(hT, hTs), dyT=(dyT, dyTs), xT=(xT, xTs), dabT=(dabT, dabTs)))


def _oracle_operands(wl, ids, x, w, dy, precision):
    fp8 = precision == "mxfp8"
    op = O.permute(bf16_bits(x), ids, wl.E)
    off = op["group_offsets"]
    w1, w3, w2 = w
    if fp8:
        xq, xs = O.quant_rows(bf16_bits(x))
        src = op["perm_src"].copy()
        src[src < 0] = 0
        X = O.Operand(O.MAT_MXFP8, xq[src], xs[src])
        Wf = [O.Operand(O.MAT_MXFP8, *_quant_along_cols_of(t)) for t in (w1, w3, w2)]
        Wb = [O.Operand(O.MAT_MXFP8, *_quant_along_rows_of(t)) for t in (w1, w3, w2)]
        DY = O.Operand(O.MAT_MXFP8, *O.quant_rows(bf16_bits(dy)))
    else:
        X = O.Operand(O.MAT_BF16, op["x_perm"])
        Wf = [O.Operand(O.MAT_BF16, bf16_bits(t)) for t in (w1, w3, w2)]
        Wb = Wf
        DY = O.Operand(O.MAT_BF16, bf16_bits(dy))
    return op, off, X, Wf, Wb, DY


def _mx_decode_T(q, s):
    v = torch.from_numpy(np.ascontiguousarray(q)).view(torch.float8_e4m3fn).double().numpy()
    return v * np.exp2(np.repeat(s.astype(np.float64), 32, axis=-1) - 127)


def _check_small(wl, ids, precision):
    tol = 3e-2 if precision == "mxfp8" else 1e-2
    g = _gpu_backward(wl, ids, precision)
    op, off, X, Wf, Wb, DY = _oracle_operands(wl, ids, g["x"], g["w"], g["dy"], precision)
    R = op["R"]
    rows = np.arange(R, dtype=np.int32)
    hmode = O.H_MXFP8 if precision == "mxfp8" else O.H_BF16
    fw = O.swiglu_rows(X, *Wf, off, rows, h_mode=hmode, want=("a_f64", "b_f64", "h_f64"))
    a16, b16 = O.f64_to_bf16(fw["a_f64"]), O.f64_to_bf16(fw["b_f64"])
    # saved pre-activations
    got_ab = O.bf16_to_f64(bf16_bits(g["ab"][:R]))
    assert rel_err(got_ab, O.bf16_to_f64(_interleave(a16, b16))) <= tol
    # dgrad: SwiGLU backward from the bf16 (a, b), dx from bf16 (then MXFP8) da, db
    pad = lambda v: np.concatenate([v, np.zeros((wl.R_cap - R, v.shape[1]), v.dtype)])
    A16, B16 = O.Operand(O.MAT_BF16, pad(a16)), O.Operand(O.MAT_BF16, pad(b16))
    dab_mode = O.DAB_MXFP8 if precision == "mxfp8" else O.DAB_BF16
    bw = O.swiglu_dgrad_rows(DY, A16, B16, *Wb, off, rows, w_blk_rows=0, dab_mode=dab_mode,
                             want=("dx_bf16", "da_f64", "db_f64"))
    da16, db16 = O.f64_to_bf16(bw["da_f64"]), O.f64_to_bf16(bw["db_f64"])
    got_dab = O.bf16_to_f64(bf16_bits(g["dab"][:R]))
    assert rel_err(got_dab, O.bf16_to_f64(_interleave(da16, db16))) <= tol
    assert rel_err(O.bf16_to_f64(bf16_bits(g["dx"][:R])), O.bf16_to_f64(bw["dx_bf16"])) <= tol
    # wgrad operands (oracle's own roundings) and transposed layouts
    h16 = O.f64_to_bf16(fw["h_f64"])
    xp = pad(op["x_perm"][:R])
    ops = dict(h=pad(h16), dy=bf16_bits(g["dy"]), x=xp, da=pad(da16), db=pad(db16))
    cols = _padded_cols(off)
    if precision == "mxfp8":
        views = {k: O.Operand(O.MAT_MXFP8, *O.quant_cols_grouped(v, off)) for k, v in ops.items()}
        # transposed MXFP8 layouts: payload at [c][P_e + i], scale at [c][P_e/32 + b]
        for key, src in (("xT", "x"), ("dyT", "dy")):
            qT, sT = (u8(t) for t in g["T"][key])
            oq, os_ = O.quant_cols_grouped(ops[src], off)
            assert np.array_equal(qT[:, cols], oq[:R].T)
            for e in range(wl.E):
                for b in range((int(off[e + 1] - off[e]) + 31) // 32):
                    P = 128 * (e + off[e] // 128)
                    assert np.array_equal(sT[:, P // 32 + b], os_[e + off[e] // 32 + b])
    else:
        views = {k: O.Operand(O.MAT_BF16, v) for k, v in ops.items()}
        xT = bf16_bits(g["T"]["xT"][0])
        assert np.array_equal(xT[:, cols], op["x_perm"][:R].T)
        dyT = bf16_bits(g["T"]["dyT"][0])
        assert np.array_equal(dyT[:, cols], bf16_bits(g["dy"])[:R].T)
    for e in range(wl.E):
        ref2 = O.wgrad_expert(views["h"], views["dy"], off, e)
        ref1 = O.wgrad_expert(views["x"], views["da"], off, e)
        ref3 = O.wgrad_expert(views["x"], views["db"], off, e)
        for got, ref in ((g["dW2"][e], ref2), (g["dW1"][e], ref1), (g["dW3"][e], ref3)):
            gv = O.bf16_to_f64(bf16_bits(got))
            if off[e + 1] == off[e]:
                assert np.all(gv == 0)
            else:
                assert rel_err(gv, ref) <= tol, (e, rel_err(gv, ref))


def _ids_from_sizes(T, K, sizes):
    ids = -np.ones((T, K), np.int32)
    col = np.repeat(np.arange(len(sizes)), sizes)[:T]
    ids[: col.size, 0] = col
    return ids


@pytest.mark.parametrize("precision", ["bf16", "mxfp8"])
def test_backward_small_ragged(precision):
    sizes = (0, 37, 130, 200, 1)
    T = sum(sizes) + 3
    HF = 512 if precision == "mxfp8" else 256   # MXFP8 contractions are whole 512-element scale boxes
    wl = W.get("tiny", T=T, E=len(sizes), K=1, H=HF, F=HF, precision=precision, act_std=0.3)
    _check_small(wl, _ids_from_sizes(T, 1, sizes), precision)


def test_backward_mxfp8_wide_h_ragged():
    """MXFP8 backward on a wider layer (H = 3584: 14 output tiles of the dx product)."""
    sizes = (0, 37, 100, 1)
    T = sum(sizes) + 3
    wl = W.get("tiny", T=T, E=len(sizes), K=1, H=3584, F=512, precision="mxfp8", act_std=0.3)
    _check_small(wl, _ids_from_sizes(T, 1, sizes), "mxfp8")


def test_backward_bf16_pair_tiles_ragged():
    """bf16 backward with groups large enough for 256-row CTA-pair tiles (dgrad, dx, wgrad)."""
    sizes = (300, 0, 1100, 513)
    T = 2100
    wl = W.get("tiny", T=T, E=len(sizes), K=1, H=256, F=256, act_std=0.3)
    _check_small(wl, _ids_from_sizes(T, 1, sizes), "bf16")


@pytest.mark.parametrize("precision", ["bf16", "mxfp8"])
def test_backward_small_routed(precision):
    wl = W.get("tiny", T=384, E=6, K=2, H=512, F=512, precision=precision, act_std=0.1)
    ids, _ = O.route_topk(W.logits(wl).numpy(), wl.K)
    _check_small(wl, ids, precision)


def _w13_col(f, half):
    """Packed column of pre-activation column f: a (half 0) or b (half 1), 128-column blocks."""
    return (f // 128) * 256 + half * 128 + (f % 128)


def _chunks(n, size=4096):
    for i in range(0, n, size):
        yield i, min(n, i + size)


def test_backward_heavy_full_size():
    """Full heavy-skew training shape (T=32768, H=7168, E=32, top-8, F=2048, MXFP8). Every
    operand on the oracle side is made by the oracle from the workload's x, W and dy.
    Sampled rows (16 random plus the first and last row of three experts): the forward's MXFP8
    h (decoded), its bf16 copy, y_perm and the saved a|b; dab and dx.
    Whole experts (the smallest, the median and the largest, 350 / 2,897 / 32,708 rows) at 32
    sampled columns of F: a|b, bf16 h and dab on every row of the expert; dW2 at those rows of
    dW2 (256 sampled columns of H) and dW1, dW3 at those columns (256 sampled rows of H), the
    wgrad operands being the oracle's own h, dab, x and dy in group-aware column-wise MXFP8."""
    wl = W.get("heavy")
    lg = W.logits(wl)
    ids, _ = O.route_topk(lg.numpy(), wl.K)
    g = _gpu_backward(wl, ids, "mxfp8")
    x, (w1, w3, w2), dy = g["x"], g["w"], g["dy"]
    op = O.permute(None, ids, wl.E)
    off, src = op["group_offsets"], op["perm_src"]
    sizes = np.diff(off)
    nz = np.nonzero(sizes)[0]
    by_size = nz[np.argsort(sizes[nz], kind="stable")]
    experts = sorted({int(by_size[0]), int(by_size[len(by_size) // 2]), int(by_size[-1])})
    rng = np.random.default_rng(0)
    xb = bf16_bits(x)
    xq, xs = O.quant_rows(xb)                         # MXFP8 x of every token (the permute's rows)
    f64 = lambda bits: O.bf16_to_f64(bits)

    # ---- sampled rows: the oracle's row functions
    rows = set(int(r) for r in rng.choice(int(off[-1]), 16, replace=False))
    for e in experts:
        rows.update((int(off[e]), int(off[e + 1]) - 1))
    rows = np.array(sorted(rows), np.int32)
    need = sorted({O.expert_of_row(off, int(r)) for r in rows})

    def stack(w, fn):  # oracle quantisation of the experts that sampled rows use; zeros elsewhere
        q = s = None
        for e in need:
            qe, se = fn(w[e:e + 1])
            if q is None:
                q = np.zeros((wl.E,) + qe.shape[1:], np.uint8)
                s = np.zeros((wl.E,) + se.shape[1:], np.uint8)
            q[e], s[e] = qe[0], se[0]
        return O.Operand(O.MAT_MXFP8, q, s)
    Wf = [stack(t, _quant_along_cols_of) for t in (w1, w3, w2)]
    Wb = [stack(t, _quant_along_rows_of) for t in (w1, w3, w2)]
    dyq, dys = O.quant_rows(bf16_bits(dy[torch.from_numpy(rows).long()]))
    X = O.Operand(O.MAT_MXFP8, _scatter_rows(xq[src[rows]], rows, wl.R_cap),
                  _scatter_rows(xs[src[rows]], rows, wl.R_cap))
    DY = O.Operand(O.MAT_MXFP8, _scatter_rows(dyq, rows, wl.R_cap), _scatter_rows(dys, rows, wl.R_cap))
    fw = O.swiglu_rows(X, *Wf, off, rows, h_mode=O.H_MXFP8,
                       want=("a_f64", "b_f64", "h_f64", "h_q", "h_s", "y_bf16"))
    ridx = torch.from_numpy(rows).long().cuda()
    assert rel_err(O.mx_decode_rows(u8(g["h"].index_select(0, ridx)), u8(g["hs"].index_select(0, ridx))),
                   O.mx_decode_rows(fw["h_q"], fw["h_s"])) <= 3e-2
    assert rel_err(f64(bf16_bits(g["h_bf16"].index_select(0, ridx))), f64(O.f64_to_bf16(fw["h_f64"]))) <= 3e-2
    assert rel_err(f64(bf16_bits(g["y"].index_select(0, ridx))), f64(fw["y_bf16"])) <= 3e-2
    a16, b16 = O.f64_to_bf16(fw["a_f64"]), O.f64_to_bf16(fw["b_f64"])
    full = lambda v: _scatter_rows(v, rows, wl.R_cap)
    bw = O.swiglu_dgrad_rows(DY, O.Operand(O.MAT_BF16, full(a16)), O.Operand(O.MAT_BF16, full(b16)), *Wb, off,
                             rows, w_blk_rows=0, dab_mode=O.DAB_MXFP8, want=("dx_bf16", "da_f64", "db_f64"))
    assert rel_err(f64(bf16_bits(g["ab"].index_select(0, ridx))), f64(_interleave(a16, b16))) <= 3e-2
    got_dab = f64(bf16_bits(g["dab"].index_select(0, ridx)))
    ref_dab = f64(_interleave(O.f64_to_bf16(bw["da_f64"]), O.f64_to_bf16(bw["db_f64"])))
    assert rel_err(got_dab, ref_dab) <= 3e-2
    assert rel_err(f64(bf16_bits(g["dx"].index_select(0, ridx))), f64(bw["dx_bf16"])) <= 3e-2

    # ---- whole experts at sampled columns: the oracle's expert-block functions
    fs = np.sort(rng.choice(wl.F, 32, replace=False))
    js = np.sort(rng.choice(wl.H, 256, replace=False))     # columns of dW2 [F, H]
    hr = np.sort(rng.choice(wl.H, 256, replace=False))     # rows of dW1, dW3 [H, F]
    fs_t, js_t, hr_t = (torch.from_numpy(v).long() for v in (fs, js, hr))
    ab_cols = torch.tensor([_w13_col(int(f), 0) for f in fs] + [_w13_col(int(f), 1) for f in fs]).cuda()
    dec = lambda qs: O.mx_decode_rows(*qs)
    for e in experts:
        r0, r1 = int(off[e]), int(off[e + 1])
        m = r1 - r0
        tok = src[r0:r1]
        w1c = dec(O.quant_rows(np.ascontiguousarray(bf16_bits(w1[e][:, fs_t]).T))).T    # [H, 32], blocks along H
        w3c = dec(O.quant_rows(np.ascontiguousarray(bf16_bits(w3[e][:, fs_t]).T))).T
        w2r = dec(O.quant_rows(bf16_bits(w2[e][fs_t])))                                 # [32, H], blocks along H
        dyb = bf16_bits(dy[r0:r1])
        a16, b16, h16, da16, db16 = (np.empty((m, fs.size), np.uint16) for _ in range(5))
        for c0, c1 in _chunks(m):
            blk = O.expert_swiglu_block(O.mx_decode_rows(xq[tok[c0:c1]], xs[tok[c0:c1]]), w1c, w3c, h_mode=O.H_BF16)
            a16[c0:c1], b16[c0:c1], h16[c0:c1] = O.f64_to_bf16(blk["a"]), O.f64_to_bf16(blk["b"]), blk["h_bf16"]
            da, db = O.expert_swiglu_dgrad_block(dec(O.quant_rows(dyb[c0:c1])), w2r, a16[c0:c1], b16[c0:c1])
            da16[c0:c1], db16[c0:c1] = O.f64_to_bf16(da), O.f64_to_bf16(db)
        rr = torch.arange(r0, r1, device="cuda")
        got_ab = f64(bf16_bits(g["ab"].index_select(0, rr).index_select(1, ab_cols)))
        assert rel_err(got_ab, f64(np.concatenate([a16, b16], axis=1))) <= 3e-2, e
        got_h = f64(bf16_bits(g["h_bf16"].index_select(0, rr).index_select(1, fs_t.cuda())))
        assert rel_err(got_h, f64(h16)) <= 3e-2, e
        got_dab = f64(bf16_bits(g["dab"].index_select(0, rr).index_select(1, ab_cols)))
        assert rel_err(got_dab, f64(np.concatenate([da16, db16], axis=1))) <= 3e-2, e
        one = np.array([0, m], np.int32)
        col = lambda v: O.Operand(O.MAT_MXFP8, *O.quant_cols_grouped(np.ascontiguousarray(v), one))
        ref2 = O.wgrad_expert(col(h16), col(dyb[:, js]), one, 0)                           # [32, 256]
        got2 = f64(bf16_bits(g["dW2"][e].index_select(0, fs_t.cuda()).index_select(1, js_t.cuda())))
        assert rel_err(got2, ref2) <= 3e-2, (e, rel_err(got2, ref2))
        xc = col(xb[:, hr][tok])
        for dW, d16 in ((g["dW1"], da16), (g["dW3"], db16)):
            ref = O.wgrad_expert(xc, col(d16), one, 0)                                      # [256, 32]
            got = f64(bf16_bits(dW[e].index_select(0, hr_t.cuda()).index_select(1, fs_t.cuda())))
            assert rel_err(got, ref) <= 3e-2, (e, rel_err(got, ref))
    assert api.moe_get_device_errors() == 0


def _scatter_rows(v, rows, R_cap):
    out = np.zeros((R_cap, v.shape[1]), v.dtype)
    out[rows] = v
    return out
