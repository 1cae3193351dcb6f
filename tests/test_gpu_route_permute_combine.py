"""GPU parity of the router, permute (plain and fused MXFP8), standalone MXFP8
quantiser and combine against the CPU oracle, through the C ABI.

Bar: ids, group sizes/offsets, row_map, perm_src, permuted rows, E4M3 payloads
and E8M0 scales bit-exact; probs within 1e-6 absolute; combine within
max|err| / max|ref| <= 1e-2 (bf16 inputs, fp32 accumulation)."""
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


def _id_dtype(wl):
    return torch.int16 if wl.id_bits == 16 else torch.int32


def _routes(wl, seed=0):
    """Oracle routes with the workload's invalid-route mask applied."""
    lg = W.logits(wl, seed)
    ids, probs = O.route_topk(lg.numpy(), wl.K, wl.renorm)
    bad = W.invalid_mask(wl, seed).numpy()
    ids = ids.copy()
    probs = probs.copy()
    ids[bad] = -1
    probs[bad] = 0.0
    return lg, ids, probs


# ------------------------------------------------------------------ router
@pytest.mark.parametrize("name", ["tiny", "mixtral", "dsv3", "large_e", "heavy"])
def test_router_matches_oracle(name):
    wl = W.get(name)
    lg = W.logits(wl)
    ids, probs = api.moe_route_topk(lg.cuda(), wl.K, id_dtype=_id_dtype(wl), renorm=wl.renorm)
    oids, oprobs = O.route_topk(lg.numpy(), wl.K, wl.renorm)
    assert np.array_equal(ids.cpu().numpy().astype(np.int32), oids)
    assert np.abs(probs.cpu().numpy() - oprobs).max() <= 1e-6


@pytest.mark.parametrize("T,E,K,renorm", [(1, 1, 1, False), (3, 2, 2, True), (37, 5, 5, False),
                                          (100, 32, 1, False), (64, 64, 16, True), (50, 200, 7, False),
                                          (50, 256, 32, False), (33, 300, 36, True), (20, 1000, 128, False),
                                          (10, 2304, 36, False), (9, 4096, 100, True),
                                          (16, 512, 64, True), (12, 2304, 128, False), (40, 2300, 36, True),
                                          (24, 2302, 36, False), (20, 1028, 65, False)])
def test_router_edge_shapes_and_ties(T, E, K, renorm):
    g = torch.Generator().manual_seed(T * 7919 + E)
    # a coarse value pool forces many exact ties, plus +-0 and -inf
    pool = torch.tensor([-float("inf"), -2.0, -0.0, 0.0, 0.5, 1.0, 1.0, 3.0])
    lg = pool[torch.randint(0, pool.numel(), (T, E), generator=g)]
    lg[0, : E // 2] = 1.0
    if T > 1:
        lg[1] = torch.randn(E, generator=g)
    for dt in (torch.int32, torch.int16):
        ids, probs = api.moe_route_topk(lg.cuda(), K, id_dtype=dt, renorm=renorm)
        oids, oprobs = O.route_topk(lg.numpy(), K, renorm)
        assert np.array_equal(ids.cpu().numpy().astype(np.int32), oids)
        assert np.abs(probs.cpu().numpy() - oprobs).max() <= 1e-6


# ----------------------------------------------------------------- permute
def _check_permute_meta(p, op, R):
    assert np.array_equal(p.group_sizes.cpu().numpy(), op["group_sizes"])
    assert np.array_equal(p.group_offsets.cpu().numpy(), op["group_offsets"])
    assert np.array_equal(p.row_map.cpu().numpy(), op["row_map"])
    assert np.array_equal(p.perm_src[:R].cpu().numpy(), op["perm_src"][:R])


@pytest.mark.parametrize("name", ["tiny", "mixtral", "large_e"])
def test_permute_bf16_matches_oracle(name):
    wl = W.get(name)
    _, ids, _ = _routes(wl)
    x = W.x(wl)
    p = api.moe_permute(x.cuda(), torch.from_numpy(ids).to(_id_dtype(wl)).cuda(), wl.E)
    op = O.permute(bf16_bits(x), ids, wl.E)
    R = op["R"]
    assert R == int((ids >= 0).sum())
    _check_permute_meta(p, op, R)
    assert np.array_equal(bf16_bits(p.x_perm[:R]), op["x_perm"][:R])
    assert api.moe_get_device_errors() == 0


def _sample_tokens(T, n, seed=0):
    g = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, T - 1], g.choice(T, size=min(n, T), replace=False)]))


@pytest.mark.parametrize("name", ["tiny", "dsv3", "heavy"])
def test_permute_fused_mxfp8_matches_oracle(name):
    wl = W.get(name)
    _, ids, _ = _routes(wl)
    x = W.x(wl)
    p = api.moe_permute(x.cuda(), torch.from_numpy(ids).to(_id_dtype(wl)).cuda(), wl.E, fuse_mxfp8=True)
    op = O.permute(None, ids, wl.E)
    R = op["R"]
    _check_permute_meta(p, op, R)
    # fused quantisation: each destination row holds the MXFP8 code of its token row
    toks = np.arange(wl.T) if wl.T <= 4096 else _sample_tokens(wl.T, 1024)
    xq, xs = O.quant_rows(bf16_bits(x[torch.from_numpy(toks)]))
    rm = op["row_map"][toks]
    for k in range(wl.K):
        ok = rm[:, k] >= 0
        rows = torch.from_numpy(rm[ok, k]).long().cuda()
        assert np.array_equal(u8(p.x_perm.index_select(0, rows)), xq[ok])
        assert np.array_equal(u8(p.x_perm_scales.index_select(0, rows)), xs[ok])


@pytest.mark.parametrize("case", ["one_token", "all_invalid", "one_expert", "k_equals_e", "e1",
                                  "bad_ids", "int16_many_experts", "dup_ids", "dup_ids_many_experts",
                                  "k128_many_experts", "k1_many_experts", "many_experts_invalid"])
def test_permute_edge_cases(case):
    """Edge shapes of the counting sort, bit for bit against the oracle. Above 64 experts the
    count kernel ranks from per-expert token masks; a token that lists an expert twice (ids
    no router here produces, but legal input) sends its tile down the flattened-order path."""
    g = torch.Generator().manual_seed(sum(map(ord, case)))
    T, H, E, K = 300, 64, 8, 2
    if case == "one_token":
        T = 1
    if case == "k_equals_e":
        K = E = 6
    if case == "e1":
        E, K = 1, 1
    if case == "int16_many_experts":
        T, E, K = 200, 3000, 36
    if case == "dup_ids":
        K = 4
    if case in ("dup_ids_many_experts", "many_experts_invalid"):
        T, E, K = 300, 300, 8
    if case == "k128_many_experts":
        T, E, K = 130, 256, 128
    if case == "k1_many_experts":
        T, E, K = 1000, 100, 1
    lg = torch.randn((T, E), generator=g)
    if case == "one_expert":
        lg[:, 3] += 100.0
    ids, _ = O.route_topk(lg.numpy(), K)
    ids = ids.copy()
    if case == "all_invalid":
        ids[:] = -1
    if case == "bad_ids":
        ids[5, 0] = E + 3
        ids[7, 1] = -9
    if case in ("dup_ids", "dup_ids_many_experts"):
        # tokens in the first, a middle and the last tile list an expert two or three times
        for t in (0, 5, 63, 64, 150, 299):
            ids[t, K - 1] = ids[t, 0]
        ids[150, K - 2] = ids[150, 0]
    if case == "many_experts_invalid":
        ids[torch.rand((T, K), generator=g).numpy() < 0.3] = -1
    x = (torch.randn((T, H), generator=g) * 0.1).to(torch.bfloat16)
    dt = torch.int16 if case == "int16_many_experts" else torch.int32
    api.moe_get_device_errors(clear=True)
    p = api.moe_permute(x.cuda(), torch.from_numpy(ids).to(dt).cuda(), E)
    op = O.permute(bf16_bits(x), ids, E)
    R = op["R"]
    _check_permute_meta(p, op, R)
    assert np.array_equal(bf16_bits(p.x_perm[:R]), op["x_perm"][:R])
    errs = api.moe_get_device_errors(clear=True)
    assert errs == (api.MOE_DEVERR_BAD_ID if case == "bad_ids" else 0)


def test_permute_then_combine_with_identity_experts_round_trip():
    wl = W.get("tiny", T=512)
    lg, ids, probs = _routes(wl)
    x = W.x(wl).cuda()
    idt = torch.from_numpy(ids).cuda()
    p = api.moe_permute(x, idt, wl.E)
    # unit probs and one route per token: combine undoes the permutation exactly
    ones = torch.zeros((wl.T, wl.K), dtype=torch.float32, device="cuda")
    ones[:, 0] = 1.0
    y = api.moe_unpermute_combine(p.x_perm, p.row_map, ones)
    assert torch.equal(y, x)


# ----------------------------------------------------------- quantiser
@pytest.mark.parametrize("name", ["tiny", "dsv3"])
def test_quant_rowwise_matches_oracle(name):
    wl = W.get(name) if name == "tiny" else W.get(name, T=2048)
    _, ids, _ = _routes(wl)
    x = W.x(wl)
    p = api.moe_permute(x.cuda(), torch.from_numpy(ids).cuda(), wl.E)
    R = int(p.group_offsets[-1])
    q, s = api.moe_quant_mxfp8_grouped(p.x_perm, p.group_offsets)
    oq, os_ = O.quant_rows(bf16_bits(p.x_perm[:R]))
    assert np.array_equal(u8(q[:R]), oq)
    assert np.array_equal(u8(s[:R]), os_)


@pytest.mark.parametrize("sizes", [(64, 32, 96), (0, 40, 1, 0, 70, 5, 33), (3000,), (0, 0, 17)])
def test_quant_colwise_grouped_matches_oracle(sizes):
    sizes = np.array(sizes, np.int32)
    off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    R_cap, H = int(off[-1]) + 7, 320
    g = torch.Generator().manual_seed(int(sizes.sum()))
    x = (torch.randn((R_cap, H), generator=g) * 0.05)
    for e in range(sizes.size):
        x[off[e]:off[e + 1]] *= 2.0 ** (3 * e - 6)
    x = x.to(torch.bfloat16)
    E = sizes.size
    fill = 0xAB
    q = torch.full((R_cap, H), fill, dtype=torch.uint8, device="cuda")
    s = torch.full((api.colwise_scale_rows(R_cap, E), H), fill, dtype=torch.uint8, device="cuda")
    api.moe_quant_mxfp8_grouped(x.cuda(), torch.from_numpy(off).cuda(), colwise=True, q=q, scales=s)
    oq, os_ = O.quant_cols_grouped(bf16_bits(x), off, fill_q=fill, fill_s=fill)
    assert np.array_equal(u8(q), oq)
    assert np.array_equal(u8(s), os_)


# ------------------------------------------------------------------ combine
@pytest.mark.parametrize("name", ["tiny", "mixtral", "large_e", "dsv3"])
def test_combine_matches_oracle(name):
    wl = W.get(name)
    _, ids, probs = _routes(wl)
    op = O.permute(None, ids, wl.E)
    yp = W.expert_out(wl)
    y = api.moe_unpermute_combine(yp.cuda(), torch.from_numpy(op["row_map"]).cuda(),
                                  torch.from_numpy(probs).cuda())
    oy = O.combine(bf16_bits(yp), op["row_map"], probs)
    got, ref = O.bf16_to_f64(bf16_bits(y)), O.bf16_to_f64(oy)
    assert rel_err(got, ref) <= 1e-2
    # fp32 accumulation in k order vs double: one bf16 rounding step apart, plus the
    # fp32 rounding of terms that cancel (bounded relative to the row's magnitude)
    row = np.abs(ref).max(axis=1, keepdims=True)
    assert np.all(np.abs(got - ref) <= np.abs(ref) * 2.0 ** -7 + row * 2.0 ** -16)
    # tokens whose routes are all invalid come back as zeros
    dead = np.all(op["row_map"] < 0, axis=1)
    assert np.all(got[dead] == 0)
