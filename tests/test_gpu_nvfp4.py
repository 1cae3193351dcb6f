"""GPU parity of the NVFP4 path with the oracle, through the C ABI: the tensor amax and the
row-wise quantiser bit for bit (codes, E4M3 scales, amax); the grouped GEMMs (tcgen05 kind
mxf4nvf4) against the oracle's products of the decoded operands -- h within max|err|/max|ref|
<= 1e-2 (the same decoded operands on both sides), y_perm within 3e-2 (the oracle quantises its
own h, whose codes may differ from the GPU's where the two h differ by a rounding); and the
layer's NVFP4 forward replayed from a CUDA graph."""
import numpy as np
import pytest
import torch

import oracle as O
from dropless_moe_expert_router_gb300 import api, workloads as W
from dropless_moe_expert_router_gb300.api import MoeError
from helpers import bf16_bits, rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dropless_moe_expert_router_gb300 import build
    build.build()
    api.moe_get_device_errors(clear=True)


def _bf16(a):
    return torch.from_numpy(O.f64_to_bf16(np.asarray(a, np.float64)).view(np.int16)).view(torch.bfloat16)


@pytest.mark.parametrize("rows,cols,valid,spread", [(64, 256, None, 4.0), (300, 512, 257, 20.0),
                                                   (7, 16, 7, 0.0), (1, 7168, None, 8.0)])
def test_amax_and_quant_match_oracle(rows, cols, valid, spread):
    rng = np.random.default_rng(rows + cols)
    x = rng.standard_normal((rows, cols)) * np.exp(rng.uniform(-spread, spread, (rows, 1)))
    xb = _bf16(x)
    vr = None if valid is None else torch.tensor([valid], dtype=torch.int32, device="cuda")
    n = rows if valid is None else valid
    amax = api.moe_amax_bf16(xb.cuda(), valid_rows=vr)
    q = torch.zeros((rows, cols // 2), dtype=torch.uint8, device="cuda")
    s = torch.zeros((rows, cols // 16), dtype=torch.uint8, device="cuda")
    api.moe_quant_nvfp4(xb.cuda(), amax, valid_rows=vr, q=q, scales=s)
    ref_amax = O.bf16_amax(bf16_bits(xb)[:n])
    assert float(amax.item()) == ref_amax
    rq, rs, _ = O.quant_rows_nvfp4(bf16_bits(xb)[:n], S=O.nvfp4_encode_scale(ref_amax))
    assert np.array_equal(q.cpu().numpy()[:n], rq)
    assert np.array_equal(s.cpu().numpy()[:n], rs)
    assert not q.cpu().numpy()[n:].any() and not s.cpu().numpy()[n:].any()     # rows past n untouched
    assert api.moe_get_device_errors() == 0


def test_quant_ties_and_zero_tensor():
    """S = 1 (the tensor amax is 2688) and block scales of exactly 1 (block amax 6): the scaled
    values are the inputs themselves, so every E2M1 midpoint is hit exactly."""
    g = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    mids = [(g[i] + g[i + 1]) / 2 for i in range(7)]
    row = np.zeros((2, 64))
    row[0, 0] = 2688.0
    blk = [6.0] + mids + [-m for m in mids] + [-0.0]
    row[1, :16] = blk
    row[1, 16:32] = [-b for b in blk]
    xb = _bf16(row)
    amax = api.moe_amax_bf16(xb.cuda())
    q, s = api.moe_quant_nvfp4(xb.cuda(), amax)
    rq, rs, S = O.quant_rows_nvfp4(bf16_bits(xb))
    assert S == 1.0 and rs[1, 0] == 0x38                        # E4M3 1.0
    assert np.array_equal(q.cpu().numpy(), rq) and np.array_equal(s.cpu().numpy(), rs)
    z = torch.zeros((4, 32), dtype=torch.bfloat16, device="cuda")
    a0 = api.moe_amax_bf16(z)
    qz, sz = api.moe_quant_nvfp4(z, a0)
    assert a0.item() == 0.0 and not qz.any() and not sz.any()


@pytest.mark.parametrize("T,H,E,K,i16,invalid", [(300, 512, 8, 2, False, 0.1), (129, 7168, 32, 4, True, 0.0),
                                                 (64, 256, 2304, 36, True, 0.05), (1, 32, 1, 1, False, 0.0)])
def test_permute_nvfp4_matches_oracle(T, H, E, K, i16, invalid):
    """The fused permute's NVFP4 rows are the oracle's permuted rows quantised with the amax of
    the routed rows: a token whose routes are all invalid (and whose row holds the largest value)
    takes no part in it. Routing outputs as moe_permute's."""
    rng = np.random.default_rng(T * 7 + E)
    x = rng.standard_normal((T, H)) * np.exp(rng.uniform(-3, 3, (T, 1)))
    ids = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
    ids[rng.random((T, K)) < invalid] = -1
    if T > 1:
        ids[T // 2, :] = -1
        x[T // 2, 5] = 1e4
    xb = _bf16(x)
    dt = torch.int16 if i16 else torch.int32
    p, amax = api.moe_permute_nvfp4(xb.cuda(), torch.from_numpy(ids).to(dt).cuda(), E)
    torch.cuda.synchronize()
    op = O.permute(bf16_bits(xb), ids, E)
    R = op["R"]
    assert np.array_equal(p.group_sizes.cpu().numpy(), op["group_sizes"])
    assert np.array_equal(p.group_offsets.cpu().numpy(), op["group_offsets"])
    assert np.array_equal(p.row_map.cpu().numpy(), op["row_map"])
    assert np.array_equal(p.perm_src.cpu().numpy()[:R], op["perm_src"][:R])
    ref_amax = O.bf16_amax(op["x_perm"][:R])
    assert float(amax.item()) == ref_amax
    rq, rs, _ = O.quant_rows_nvfp4(op["x_perm"][:R], S=O.nvfp4_encode_scale(ref_amax))
    assert np.array_equal(p.x_perm.cpu().numpy()[:R], rq)
    assert np.array_equal(p.x_perm_scales.cpu().numpy()[:R], rs)
    assert api.moe_get_device_errors() == 0


def _oracle_weights_nvfp4(w1, w3, w2):
    """Decoded weights (float64, logical layouts) as the GPU packs and quantises them: W1, W3 along
    H with one amax over both, W2 along F with its own amax."""
    b1, b3, b2 = bf16_bits(w1), bf16_bits(w3), bf16_bits(w2)
    S13 = O.nvfp4_encode_scale(max(O.bf16_amax(b1), O.bf16_amax(b3)))
    S2 = O.nvfp4_encode_scale(O.bf16_amax(b2))

    def dec_t(wb, S):   # quantise each expert's W^T rows (the contraction along the last axis)
        out = []
        for e in range(wb.shape[0]):
            q, s, _ = O.quant_rows_nvfp4(np.ascontiguousarray(wb[e].T), S=S)
            out.append(O.nvfp4_decode(q, s, S).T)
        return np.stack(out)
    return dec_t(b1, S13), dec_t(b3, S13), dec_t(b2, S2)


@pytest.mark.parametrize("T,H,F,E,K", [(200, 512, 512, 4, 2), (96, 256, 768, 4, 3)])
def test_nvfp4_grouped_gemms_match_oracle(T, H, F, E, K):
    rng = np.random.default_rng(T + H)
    wl = W.get("tiny", T=T, H=H, F=F, E=E, K=K)
    w1, w3, w2 = W.weights(wl)
    x = W.x(wl)
    # distinct experts per token among the first E - 1: the last expert stays empty
    ids = np.stack([rng.choice(E - 1, K, replace=False) for _ in range(T)]).astype(np.int32)
    op = O.permute(bf16_bits(x), ids, E)
    R, off = op["R"], op["group_offsets"]
    xp = torch.from_numpy(op["x_perm"].view(np.int16)).view(torch.bfloat16).cuda()
    goff = torch.from_numpy(off).cuda()
    nw = api.moe_prepare_weights_nvfp4(w1.cuda(), w3.cuda(), w2.cuda())
    xa = api.moe_amax_bf16(xp, valid_rows=goff[E:])
    xq, xs = api.moe_quant_nvfp4(xp, xa, valid_rows=goff[E:])
    h, ha = api.moe_grouped_gemm_up_nvfp4(xq, xs, xa, nw, goff)
    hq, hs = api.moe_quant_nvfp4(h, ha, valid_rows=goff[E:])
    y = api.moe_grouped_gemm_down_nvfp4(hq, hs, ha, nw, goff)
    torch.cuda.synchronize()
    assert api.moe_get_device_errors() == 0
    # oracle: the same decoded operands
    Sx = O.nvfp4_encode_scale(O.bf16_amax(op["x_perm"][:R]))
    rq, rs, _ = O.quant_rows_nvfp4(op["x_perm"][:R], S=Sx)
    assert np.array_equal(xq.cpu().numpy()[:R], rq) and np.array_equal(xs.cpu().numpy()[:R], rs)
    X = np.zeros((T * K, H))
    X[:R] = O.nvfp4_decode(rq, rs, Sx)
    W1d, W3d, W2d = _oracle_weights_nvfp4(w1, w3, w2)
    rows = np.arange(R, dtype=np.int32)
    fw = O.swiglu_rows(O.Operand(O.MAT_F64, X), O.Operand(O.MAT_F64, W1d), O.Operand(O.MAT_F64, W3d),
                       O.Operand(O.MAT_F64, W2d), off, rows, h_mode=O.H_BF16, want=("h_bf16",))
    h_ref = fw["h_bf16"]
    assert rel_err(O.bf16_to_f64(bf16_bits(h)[:R]), O.bf16_to_f64(h_ref)) <= 1e-2
    assert abs(float(ha.item()) - O.bf16_amax(h_ref)) <= 1e-2 * O.bf16_amax(h_ref)
    Sh = O.nvfp4_encode_scale(O.bf16_amax(h_ref))
    hq_r, hs_r, _ = O.quant_rows_nvfp4(h_ref, S=Sh)
    Hd = np.zeros((T * K, F))
    Hd[:R] = O.nvfp4_decode(hq_r, hs_r, Sh)
    y_ref = O.grouped_matmul(Hd, np.ascontiguousarray(W2d.transpose(0, 2, 1)), off)
    assert rel_err(O.bf16_to_f64(bf16_bits(y)[:R]), y_ref[:R]) <= 3e-2


def test_nvfp4_grouped_gemms_full_dsv3_shape_sampled():
    """The DeepSeek-V3-like NVFP4 layer at full size (T=8192, H=7168, E=32, top-4, F=2048, six
    empty experts): the permute's amax, codes and scales on sampled rows; h on sampled rows (the
    first and last row of every non-empty group plus 24 random rows); h's amax against the
    oracle's over every row (the oracle computes h for all rows, one expert at a time); y_perm on
    the sampled rows from the oracle's own NVFP4 h."""
    import os
    from concurrent.futures import ThreadPoolExecutor
    wl = W.get("dsv3_nvfp4")
    x = W.x(wl)
    w1, w3, w2 = W.weights(wl)
    ids, _ = O.route_topk(W.logits(wl).numpy(), wl.K, wl.renorm)
    op = O.permute(bf16_bits(x), ids, wl.E)
    R, off = op["R"], op["group_offsets"]
    dev = torch.device("cuda")
    nw = api.moe_prepare_weights_nvfp4(w1.to(dev), w3.to(dev), w2.to(dev))
    p, xa = api.moe_permute_nvfp4(x.to(dev), torch.from_numpy(ids).to(dev), wl.E)
    goff = p.group_offsets
    h, ha = api.moe_grouped_gemm_up_nvfp4(p.x_perm, p.x_perm_scales, xa, nw, goff)
    hq, hs = api.moe_quant_nvfp4(h, ha, valid_rows=goff[wl.E:])
    y = api.moe_grouped_gemm_down_nvfp4(hq, hs, ha, nw, goff)
    torch.cuda.synchronize()
    assert api.moe_get_device_errors() == 0
    rng = np.random.default_rng(5)
    rows = set(int(r) for r in rng.choice(R, 24, replace=False))
    for e in range(wl.E):
        if off[e + 1] > off[e]:
            rows.update((int(off[e]), int(off[e + 1]) - 1))
    rows = np.array(sorted(rows), np.int64)
    ridx = torch.from_numpy(rows).cuda()
    # x: amax of the routed rows, NVFP4 codes and scales of the sampled rows
    Sx = O.nvfp4_encode_scale(O.bf16_amax(op["x_perm"][:R]))
    assert float(xa.item()) == O.bf16_amax(op["x_perm"][:R])
    rq, rs, _ = O.quant_rows_nvfp4(op["x_perm"][rows], S=Sx)
    assert np.array_equal(p.x_perm.index_select(0, ridx).cpu().numpy(), rq)
    assert np.array_equal(p.x_perm_scales.index_select(0, ridx).cpu().numpy(), rs)
    # weights: one encode scale per stacked tensor, blocks along the contraction dimension
    b1, b3, b2 = bf16_bits(w1), bf16_bits(w3), bf16_bits(w2)
    S13 = O.nvfp4_encode_scale(max(O.bf16_amax(b1), O.bf16_amax(b3)))
    S2 = O.nvfp4_encode_scale(O.bf16_amax(b2))
    live = [e for e in range(wl.E) if off[e + 1] > off[e]]
    with ThreadPoolExecutor(max_workers=max(1, os.cpu_count() or 1)) as pool:   # the C oracle is reentrant
        quant = lambda wb, S: pool.submit(O.quant_rows_nvfp4, np.ascontiguousarray(wb.T), S)
        w13f = {e: (quant(b1[e], S13), quant(b3[e], S13)) for e in live}
        ex_rows = {e: rows[(rows >= off[e]) & (rows < off[e + 1])] for e in live}
        w2f = {e: quant(b2[e], S2) for e in live if ex_rows[e].size}
        xf = {e: pool.submit(O.quant_rows_nvfp4, op["x_perm"][off[e]:off[e + 1]], Sx) for e in live}
        dec = lambda fut: O.nvfp4_decode(*fut.result()).T
        h_amax, h_rows, y_rows = 0.0, {}, {}
        for e in live:
            r0, r1 = int(off[e]), int(off[e + 1])
            xv = O.nvfp4_decode(*xf.pop(e).result())
            blk = O.expert_swiglu_block(xv, dec(w13f[e][0]), dec(w13f[e][1]), h_mode=O.H_BF16)
            h_amax = max(h_amax, O.bf16_amax(blk["h_bf16"]))
            if ex_rows[e].size:
                h_rows[e] = blk["h_bf16"][ex_rows[e] - r0]
                y_rows[e] = dec(w2f[e])                          # W2[e] values [F, H]
    # h on the sampled rows, and its amax over every row
    h_ref = np.concatenate([h_rows[e] for e in live if e in h_rows])
    assert rel_err(O.bf16_to_f64(bf16_bits(h.index_select(0, ridx))), O.bf16_to_f64(h_ref)) <= 1e-2
    assert abs(float(ha.item()) - h_amax) <= 1e-2 * h_amax
    # y_perm on the sampled rows: the oracle's NVFP4 of its own h (encode scale of its amax)
    Sh = O.nvfp4_encode_scale(h_amax)
    y_ref = np.concatenate([O.nvfp4_decode(*O.quant_rows_nvfp4(h_rows[e], S=Sh)) @ y_rows[e]
                            for e in live if e in h_rows])
    assert rel_err(O.bf16_to_f64(bf16_bits(y.index_select(0, ridx))), y_ref) <= 3e-2


def test_nvfp4_layer_graph_replay_matches_eager():
    from dropless_moe_expert_router_gb300.layer import MoELayer
    wl = W.get("dsv3_nvfp4", T=256, H=512, F=512, E=8)
    w1, w3, w2 = (t.cuda() for t in W.weights(wl))
    layer = MoELayer(w1, w3, w2, T=wl.T, K=wl.K, precision="nvfp4")
    x, lg = W.x(wl).cuda(), W.logits(wl).cuda()
    eager = layer.forward(x, lg).clone()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        out = layer.forward(x, lg)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    assert torch.isfinite(out.float()).all() and out.float().abs().max() > 0
    assert layer.launches_per_forward == 6 + api.moe_permute_kernel_launches(wl.T, wl.K, wl.E)
    with pytest.raises(ValueError):
        MoELayer(w1, w3, w2, T=wl.T, K=wl.K, precision="nvfp4", training=True)


def test_nvfp4_gemm_shape_limits_are_status_codes():
    E, H, F, R_cap = 2, 384, 512, 64                      # H % 256 != 0: not whole 256-element k-blocks
    u8 = dict(dtype=torch.uint8, device="cuda")
    a = torch.ones((1,), dtype=torch.float32, device="cuda")
    nw = api.Nvfp4Weights(E, H, F, torch.zeros((E, 2 * F, H // 2), **u8), torch.zeros((E, 2 * F, H // 16), **u8), a,
                          torch.zeros((E, H, F // 2), **u8), torch.zeros((E, H, F // 16), **u8), a)
    xq = torch.zeros((R_cap, H // 2), **u8)
    xs = torch.zeros((R_cap, H // 16), **u8)
    goff = torch.zeros((E + 1,), dtype=torch.int32, device="cuda")
    with pytest.raises(MoeError):
        api.moe_grouped_gemm_up_nvfp4(xq, xs, a, nw, goff)
    with pytest.raises(MoeError):
        api.moe_grouped_gemm_down_nvfp4(torch.zeros((R_cap, F // 2), **u8), torch.zeros((R_cap, F // 16), **u8), a,
                                        nw, goff)
    assert api.moe_get_device_errors() == 0
