"""Pins for the oracle's grouped SwiGLU MLP (forward, dgrad, wgrad).

Independent references: numpy float64 matmuls per expert on the logical
layouts (a library routine), hand-built weights with known results, torch's
float8 decode for MXFP8 operands, and central finite differences for the
backward formulas.
"""
import numpy as np
import pytest
import torch

import oracle as O


def _bf16(x):
    t = torch.from_numpy(np.asarray(x, np.float64)).to(torch.float32).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _f(bits):
    return O.bf16_to_f64(bits)


def _problem(seed, E=4, H=64, F=96, sizes=(5, 0, 17, 9), R_extra=6, std=0.3):
    rng = np.random.default_rng(seed)
    sizes = np.array(sizes, np.int32)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    R_cap = int(off[-1]) + R_extra
    x = _bf16(rng.standard_normal((R_cap, H)) * std)
    w1 = _bf16(rng.standard_normal((E, H, F)) * std)
    w3 = _bf16(rng.standard_normal((E, H, F)) * std)
    w2 = _bf16(rng.standard_normal((E, F, H)) * std)
    return x, w1, w3, w2, off


def _silu(a):
    return a / (1 + np.exp(-a))


def _np_forward(xv, w1v, w3v, w2v, off, round_h=None):
    E = off.size - 1
    y = np.zeros((int(off[-1]), xv.shape[1]))
    for e in range(E):
        r0, r1 = off[e], off[e + 1]
        a = xv[r0:r1] @ w1v[e]
        b = xv[r0:r1] @ w3v[e]
        h = _silu(a) * b
        if round_h is not None:
            h = round_h(h)
        y[r0:r1] = h @ w2v[e]
    return y


def test_forward_f64_matches_numpy_per_expert():
    x, w1, w3, w2, off = _problem(1)
    R = int(off[-1])
    rows = np.arange(R, dtype=np.int32)
    out = O.swiglu_rows(O.Operand(O.MAT_BF16, x), O.Operand(O.MAT_BF16, w1),
                        O.Operand(O.MAT_BF16, w3), O.Operand(O.MAT_BF16, w2), off, rows,
                        h_mode=O.H_NONE, want=("y_f64", "h_f64"))
    want = _np_forward(_f(x), _f(w1), _f(w3), _f(w2), off)
    assert np.allclose(out["y_f64"], want, rtol=1e-12, atol=1e-12)


def test_forward_bf16_h_rounding_and_output():
    x, w1, w3, w2, off = _problem(2)
    R = int(off[-1])
    rows = np.arange(R, dtype=np.int32)[::-1].copy()          # any row order
    out = O.swiglu_rows(O.Operand(O.MAT_BF16, x), O.Operand(O.MAT_BF16, w1),
                        O.Operand(O.MAT_BF16, w3), O.Operand(O.MAT_BF16, w2), off, rows,
                        h_mode=O.H_BF16, want=("y_bf16", "h_bf16", "h_f64"))
    assert np.array_equal(out["h_bf16"], _bf16(out["h_f64"]))
    want = _np_forward(_f(x), _f(w1), _f(w3), _f(w2), off, round_h=lambda h: _f(_bf16(h)))
    got = _f(out["y_bf16"])
    assert np.all(np.abs(got - want[rows]) <= np.abs(want[rows]) * 2.0 ** -8 + 1e-30)


def test_forward_hand_cases():
    E, H, F = 2, 32, 32
    off = np.array([0, 3, 5], np.int32)
    x = _bf16(np.random.default_rng(3).standard_normal((5, H)))
    z = np.zeros((E, H, F), np.uint16)
    w2 = _bf16(np.ones((E, F, H)))
    rows = np.arange(5, dtype=np.int32)
    out = O.swiglu_rows(O.Operand(O.MAT_BF16, x), O.Operand(O.MAT_BF16, z),
                        O.Operand(O.MAT_BF16, z), O.Operand(O.MAT_BF16, w2), off, rows,
                        want=("y_f64",))
    assert np.all(out["y_f64"] == 0)
    # one-hot: W1[e][h, f] = [h == f] * 8 (large a -> silu(a) ~ a), W3 = [h == f],
    # W2[e] = I * (e + 1): y[r, j] = (e+1) * silu(8 x_j) * x_j
    w1 = np.zeros((E, H, F))
    w3 = np.zeros((E, H, F))
    w2 = np.zeros((E, F, H))
    for e in range(E):
        w1[e] = np.eye(H) * 8
        w3[e] = np.eye(H)
        w2[e] = np.eye(H) * (e + 1)
    out = O.swiglu_rows(O.Operand(O.MAT_BF16, x), O.Operand(O.MAT_BF16, _bf16(w1)),
                        O.Operand(O.MAT_BF16, _bf16(w3)), O.Operand(O.MAT_BF16, _bf16(w2)),
                        off, rows, h_mode=O.H_NONE, want=("y_f64",))
    xv = _f(x)
    scale = np.array([1, 1, 1, 2, 2])[:, None]
    assert np.allclose(out["y_f64"], scale * _silu(8 * xv) * xv, rtol=1e-12)


def _mx_decode(q, s, blk_rows):
    v = torch.from_numpy(q).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    if blk_rows:
        sc = np.repeat(s.astype(np.float64), 32, axis=-2)
    else:
        sc = np.repeat(s.astype(np.float64), 32, axis=-1)
    return v * np.exp2(sc - 127)


def test_forward_mxfp8_operands_match_numpy_on_decoded_values():
    x, w1, w3, w2, off = _problem(4, H=64, F=64)
    E = off.size - 1
    xq, xs = O.quant_rows(x)
    # weights quantised along their contraction dimension (rows of [H,F] / [F,H])
    def qcols(w):
        qs, ss = [], []
        for e in range(E):
            q, s = O.quant_rows(np.ascontiguousarray(w[e].T))
            qs.append(q.T)
            ss.append(s.T)
        return np.ascontiguousarray(np.stack(qs)), np.ascontiguousarray(np.stack(ss))
    w1q, w1s = qcols(w1)
    w3q, w3s = qcols(w3)
    w2q, w2s = qcols(w2)
    R = int(off[-1])
    rows = np.arange(R, dtype=np.int32)
    out = O.swiglu_rows(O.Operand(O.MAT_MXFP8, xq, xs), O.Operand(O.MAT_MXFP8, w1q, w1s),
                        O.Operand(O.MAT_MXFP8, w3q, w3s), O.Operand(O.MAT_MXFP8, w2q, w2s),
                        off, rows, h_mode=O.H_MXFP8, want=("y_f64", "h_q", "h_s", "h_f64"))
    xd = _mx_decode(xq, xs, False)
    w1d, w3d, w2d = (_mx_decode(q, s, True) for q, s in ((w1q, w1s), (w3q, w3s), (w2q, w2s)))
    # h is quantised row-wise along F, straight from the unrounded value
    hq, hs = out["h_q"], out["h_s"]
    hd = _mx_decode(hq, hs, False)
    want_h = np.concatenate([_silu(xd[off[e]:off[e + 1]] @ w1d[e]) * (xd[off[e]:off[e + 1]] @ w3d[e])
                             for e in range(E)])
    assert np.allclose(out["h_f64"], want_h, rtol=1e-12, atol=1e-14)
    err = np.abs(hd - want_h)
    unit = np.exp2(np.repeat(hs - 127.0, 32, 1))
    sat = np.abs(want_h) / unit > 448          # above E4M3's range at this block scale
    assert np.all(err[~sat] <= (np.abs(want_h) * 2.0 ** -4 + unit * 2 ** -10)[~sat])
    assert np.all(np.abs(hd[sat]) == 448 * unit[sat])
    want_y = np.concatenate([hd[off[e]:off[e + 1]] @ w2d[e] for e in range(E)])
    assert np.allclose(out["y_f64"], want_y, rtol=1e-12, atol=1e-14)


def test_dgrad_matches_finite_differences():
    E, H, F = 2, 8, 8
    rng = np.random.default_rng(5)
    off = np.array([0, 2, 5], np.int32)
    x = rng.standard_normal((5, H))
    w1, w3 = rng.standard_normal((E, H, F)), rng.standard_normal((E, H, F))
    w2 = rng.standard_normal((E, F, H))
    dy = rng.standard_normal((5, H))
    rows = np.arange(5, dtype=np.int32)
    W = lambda a: O.Operand(O.MAT_F64, a)

    def loss(xx, ww1, ww3):
        y = O.swiglu_rows(W(xx), W(ww1), W(ww3), W(w2), off, rows, h_mode=O.H_NONE,
                          want=("y_f64",))["y_f64"]
        return float((y * dy).sum())

    fw = O.swiglu_rows(W(x), W(w1), W(w3), W(w2), off, rows, h_mode=O.H_NONE,
                       want=("a_f64", "b_f64"))
    bw = O.swiglu_dgrad_rows(W(dy), W(fw["a_f64"]), W(fw["b_f64"]), W(w1), W(w3), W(w2),
                             off, rows, want=("dx_f64", "da_f64", "db_f64"))
    eps = 1e-6
    for r in range(5):
        for h in range(H):
            xp, xm = x.copy(), x.copy()
            xp[r, h] += eps
            xm[r, h] -= eps
            fd = (loss(xp, w1, w3) - loss(xm, w1, w3)) / (2 * eps)
            assert abs(fd - bw["dx_f64"][r, h]) <= 1e-6 * (1 + abs(fd))
    # wgrad of W1 / W3 from da / db: dW1[e] = x_e^T da_e
    for e in range(E):
        dW1 = O.wgrad_expert(W(x), W(bw["da_f64"]), off, e)
        dW3 = O.wgrad_expert(W(x), W(bw["db_f64"]), off, e)
        for (h, f) in [(0, 0), (3, 5), (7, 7), (2, 6)]:
            for ww, dW in ((0, dW1), (1, dW3)):
                wp = [w1.copy(), w3.copy()]
                wm = [w1.copy(), w3.copy()]
                wp[ww][e, h, f] += eps
                wm[ww][e, h, f] -= eps
                fd = (loss(x, *wp) - loss(x, *wm)) / (2 * eps)
                assert abs(fd - dW[h, f]) <= 1e-6 * (1 + abs(fd))


def test_wgrad_dw2_matches_finite_differences_and_numpy():
    E, H, F = 3, 8, 16
    rng = np.random.default_rng(6)
    off = np.array([0, 4, 4, 7], np.int32)          # expert 1 is empty
    x = rng.standard_normal((9, H))
    w1, w3 = rng.standard_normal((E, H, F)), rng.standard_normal((E, H, F))
    w2 = rng.standard_normal((E, F, H))
    dy = rng.standard_normal((9, H))
    rows = np.arange(7, dtype=np.int32)
    W = lambda a: O.Operand(O.MAT_F64, a)
    fw = O.swiglu_rows(W(x), W(w1), W(w3), W(w2), off, rows, h_mode=O.H_NONE, want=("h_f64",))
    h = np.zeros((9, F))
    h[:7] = fw["h_f64"]
    for e in range(E):
        dW2 = O.wgrad_expert(W(h), W(dy), off, e)
        r0, r1 = off[e], off[e + 1]
        assert np.allclose(dW2, h[r0:r1].T @ dy[r0:r1], rtol=1e-13, atol=1e-13)
        cols = np.array([H - 1, 0, 3], np.int32)
        sub = O.wgrad_expert(W(h), W(dy), off, e, cols=cols)
        assert np.allclose(sub, dW2[:, cols])
    e, f, j = 2, 5, 3
    eps = 1e-6

    def loss(ww2):
        y = O.swiglu_rows(W(x), W(w1), W(w3), W(ww2), off, rows, h_mode=O.H_NONE,
                          want=("y_f64",))["y_f64"]
        return float((y * dy[:7]).sum())
    wp, wm = w2.copy(), w2.copy()
    wp[e, f, j] += eps
    wm[e, f, j] -= eps
    fd = (loss(wp) - loss(wm)) / (2 * eps)
    assert abs(fd - O.wgrad_expert(W(h), W(dy), off, e)[f, j]) <= 1e-6 * (1 + abs(fd))


def test_wgrad_mxfp8_colwise_operands_decode_like_torch():
    rng = np.random.default_rng(7)
    sizes = np.array([40, 0, 33], np.int32)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    R_cap = int(off[-1]) + 5
    a = _bf16(rng.standard_normal((R_cap, 32)))
    b = _bf16(rng.standard_normal((R_cap, 64)))
    aq, as_ = O.quant_cols_grouped(a, off)
    bq, bs = O.quant_cols_grouped(b, off)
    for e in (0, 2):
        got = O.wgrad_expert(O.Operand(O.MAT_MXFP8, aq, as_), O.Operand(O.MAT_MXFP8, bq, bs),
                             off, e)
        r0, r1 = off[e], off[e + 1]
        ad = torch.from_numpy(aq[r0:r1]).view(torch.float8_e4m3fn).double().numpy()
        bd = torch.from_numpy(bq[r0:r1]).view(torch.float8_e4m3fn).double().numpy()
        srows = e + r0 // 32 + np.arange(r1 - r0) // 32
        ad = ad * np.exp2(as_[srows].astype(np.float64) - 127)
        bd = bd * np.exp2(bs[srows].astype(np.float64) - 127)
        assert np.allclose(got, ad.T @ bd, rtol=1e-12, atol=1e-12)
        # and the decoded operands approximate the bf16 ones
        assert np.allclose(ad, _f(a[r0:r1]), rtol=2 ** -3, atol=1e-3)   # saturation: <= 1/8


def test_dgrad_dab_rounding_modes_follow_their_operands():
    """dab_mode 1 / 2: dx equals the plain product of the bf16 (then MXFP8) da, db with
    W1, W3, computed here with numpy on operands rounded by torch."""
    E, H, F = 2, 32, 64
    rng = np.random.default_rng(8)
    off = np.array([0, 3, 7], np.int32)
    W = lambda a: O.Operand(O.MAT_F64, a)
    x = rng.standard_normal((7, H))
    w1, w3 = rng.standard_normal((E, H, F)) * 0.2, rng.standard_normal((E, H, F)) * 0.2
    w2 = rng.standard_normal((E, F, H)) * 0.2
    dy = rng.standard_normal((7, H))
    rows = np.arange(7, dtype=np.int32)
    fw = O.swiglu_rows(W(x), W(w1), W(w3), W(w2), off, rows, h_mode=O.H_NONE, want=("a_f64", "b_f64"))
    base = O.swiglu_dgrad_rows(W(dy), W(fw["a_f64"]), W(fw["b_f64"]), W(w1), W(w3), W(w2), off, rows,
                               want=("dx_f64", "da_f64", "db_f64"))
    tb = lambda a: torch.from_numpy(a).to(torch.float32).to(torch.bfloat16).double().numpy()

    def mx(a):
        out = np.empty_like(a)
        for r in range(a.shape[0]):
            for blk in range(a.shape[1] // 32):
                v = a[r, 32 * blk:32 * blk + 32]
                amax = np.abs(v).max()
                e = O.e8m0_scale_byte(amax) - 127
                q = torch.from_numpy(np.clip(v / 2.0 ** e, -448, 448)).to(torch.float32).to(
                    torch.float8_e4m3fn).double().numpy()
                out[r, 32 * blk:32 * blk + 32] = q * 2.0 ** e
        return out
    for mode, rnd in ((O.DAB_BF16, tb), (O.DAB_MXFP8, lambda a: mx(tb(a)))):
        got = O.swiglu_dgrad_rows(W(dy), W(fw["a_f64"]), W(fw["b_f64"]), W(w1), W(w3), W(w2), off,
                                  rows, dab_mode=mode, want=("dx_f64", "da_f64"))
        assert np.array_equal(got["da_f64"], base["da_f64"])      # unrounded outputs unchanged
        da, db = rnd(base["da_f64"]), rnd(base["db_f64"])
        want = np.concatenate([da[off[e]:off[e + 1]] @ w1[e].T + db[off[e]:off[e + 1]] @ w3[e].T
                               for e in range(E)])
        assert np.allclose(got["dx_f64"], want, rtol=1e-12, atol=1e-12)


# ------------------------------------------------ whole-expert blocks of rows
def test_mx_decode_matches_torch_float8():
    """Row-wise and column-wise MXFP8 decoding against torch's float8_e4m3fn values (a library
    conversion) times the power-of-two scales."""
    rng = np.random.default_rng(7)
    x = _bf16(rng.standard_normal((70, 96)) * np.exp(rng.uniform(-6, 6, (70, 1))))
    q, s = O.quant_rows(x)
    tv = torch.from_numpy(q).view(torch.float8_e4m3fn).double().numpy()
    assert np.array_equal(O.mx_decode_rows(q, s), tv * np.repeat(np.exp2(s.astype(np.float64) - 127), 32, axis=1))
    off = np.array([0, 70], np.int32)
    qc, sc = O.quant_cols_grouped(x, off)
    tv = torch.from_numpy(qc).view(torch.float8_e4m3fn).double().numpy()
    want = tv * np.exp2(np.repeat(sc[:3].astype(np.float64), 32, axis=0)[:70] - 127)
    assert np.array_equal(O.mx_decode_cols(qc, sc[:3]), want)


def test_quant_rows_f64_equals_bf16_quantiser_on_bf16_values():
    rng = np.random.default_rng(8)
    x = _bf16(rng.standard_normal((9, 128)) * 3)
    assert all(np.array_equal(a, b) for a, b in zip(O.quant_rows_f64(_f(x)), O.quant_rows(x)))


@pytest.mark.parametrize("kind", ["bf16", "mxfp8"])
def test_expert_block_forward_matches_row_oracle(kind):
    """The expert-block forward (a library matmul per product) reproduces oracle_swiglu_rows:
    pre-activations and h to 1e-12, bf16 h bit for bit, MXFP8 h codes and scales bit for bit
    where the two float64 h agree, y to 1e-12; a subset of F columns gives those columns."""
    x, w1, w3, w2, off = _problem(11, H=64, F=96)
    if kind == "mxfp8":
        x, w1, w3, w2, off = _problem(11, H=64, F=64)        # MXFP8: whole 32-blocks along H and F
        xq, xs = O.quant_rows(x)
        w1q, w1s = zip(*(O.quant_rows(np.ascontiguousarray(w1[e].T)) for e in range(w1.shape[0])))
        w3q, w3s = zip(*(O.quant_rows(np.ascontiguousarray(w3[e].T)) for e in range(w3.shape[0])))
        w2q, w2s = zip(*(O.quant_rows(np.ascontiguousarray(w2[e].T)) for e in range(w2.shape[0])))
        ops = [O.Operand(O.MAT_MXFP8, xq, xs)] + [
            O.Operand(O.MAT_MXFP8, np.ascontiguousarray(np.stack(q).transpose(0, 2, 1)),
                      np.ascontiguousarray(np.stack(s).transpose(0, 2, 1)))
            for q, s in ((w1q, w1s), (w3q, w3s), (w2q, w2s))]
        xv = O.mx_decode_rows(xq, xs)
        wv = [np.stack([O.mx_decode_rows(q[e], s[e]).T for e in range(len(q))])
              for q, s in ((w1q, w1s), (w3q, w3s), (w2q, w2s))]
        hm = O.H_MXFP8
    else:
        ops = [O.Operand(O.MAT_BF16, t) for t in (x, w1, w3, w2)]
        xv, wv, hm = _f(x), [_f(w1), _f(w3), _f(w2)], O.H_BF16
    rows = np.arange(int(off[-1]), dtype=np.int32)
    ref = O.swiglu_rows(*ops, off, rows, h_mode=hm,
                        want=("a_f64", "b_f64", "h_f64", "y_f64", "h_bf16", "h_q", "h_s"))
    for e in range(off.size - 1):
        r0, r1 = off[e], off[e + 1]
        if r1 == r0:
            continue
        blk = O.expert_swiglu_block(xv[r0:r1], wv[0][e], wv[1][e], wv[2][e], h_mode=hm)
        for k in ("a", "b", "h", "y"):
            assert np.allclose(blk[k], ref[k + "_f64"][r0:r1], rtol=1e-12, atol=1e-15), k
        if hm == O.H_BF16:
            assert np.array_equal(blk["h_bf16"], ref["h_bf16"][r0:r1])
        else:
            assert np.array_equal(blk["h_q"], ref["h_q"][r0:r1]) and np.array_equal(blk["h_s"], ref["h_s"][r0:r1])
        cols = np.array([3, 17, 40], np.int64)
        sub = O.expert_swiglu_block(xv[r0:r1], wv[0][e][:, cols], wv[1][e][:, cols], h_mode=O.H_NONE)
        assert np.allclose(sub["h"], ref["h_f64"][r0:r1][:, cols], rtol=1e-12, atol=1e-15)


def test_expert_block_dgrad_matches_row_oracle():
    """The expert-block SwiGLU backward at a subset of F columns reproduces
    oracle_swiglu_dgrad_rows' da, db (from the same bf16 pre-activations)."""
    x, w1, w3, w2, off = _problem(12, H=64, F=96)
    rng = np.random.default_rng(12)
    R_cap = x.shape[0]
    dy = _bf16(rng.standard_normal((R_cap, 64)) * 0.3)
    a16 = _bf16(rng.standard_normal((R_cap, 96)))
    b16 = _bf16(rng.standard_normal((R_cap, 96)))
    rows = np.arange(int(off[-1]), dtype=np.int32)
    Wo = [O.Operand(O.MAT_BF16, t) for t in (w1, w3, w2)]
    ref = O.swiglu_dgrad_rows(O.Operand(O.MAT_BF16, dy), O.Operand(O.MAT_BF16, a16), O.Operand(O.MAT_BF16, b16),
                              *Wo, off, rows, want=("da_f64", "db_f64"))
    cols = np.array([0, 5, 31, 95], np.int64)
    for e in range(off.size - 1):
        r0, r1 = off[e], off[e + 1]
        if r1 == r0:
            continue
        da, db = O.expert_swiglu_dgrad_block(_f(dy[r0:r1]), _f(w2[e][cols]), a16[r0:r1][:, cols], b16[r0:r1][:, cols])
        assert np.allclose(da, ref["da_f64"][r0:r1][:, cols], rtol=1e-12, atol=1e-15)
        assert np.allclose(db, ref["db_f64"][r0:r1][:, cols], rtol=1e-12, atol=1e-15)


def test_swiglu_steps_match_finite_differences_and_closed_forms():
    """h = silu(a) b: silu(0) = 0, silu(a) -> a for large a, h linear in b; its gradient matches
    central differences of the forward step."""
    a = np.array([0.0, 30.0, -30.0, 1.5, -0.7, 2.0])
    b = np.array([2.0, 1.0, 1.0, -0.3, 0.9, 0.0])
    h = O.swiglu(a, b)
    assert h[0] == 0.0 and abs(h[1] - 30.0) < 1e-9 and abs(h[2]) < 1e-9 and h[5] == 0.0
    assert np.allclose(O.swiglu(a, 2 * b), 2 * h, rtol=0, atol=0)
    dh = np.array([1.0, -2.0, 0.5, 1.25, -1.0, 3.0])
    da, db = O.swiglu_grad(dh, a, b)
    eps = 1e-6
    fda = dh * (O.swiglu(a + eps, b) - O.swiglu(a - eps, b)) / (2 * eps)
    fdb = dh * (O.swiglu(a, b + eps) - O.swiglu(a, b - eps)) / (2 * eps)
    assert np.allclose(da, fda, rtol=1e-6, atol=1e-8) and np.allclose(db, fdb, rtol=1e-6, atol=1e-8)
