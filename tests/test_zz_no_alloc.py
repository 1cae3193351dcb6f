"""moe_permute_noalloc: the permute entry point for callers that cannot allocate
device memory (a server that reserved all GPU memory up front, a plug-in whose
host owns the allocator, code that must not risk cudaMalloc's implicit sync).
It must give exactly what moe_permute gives with a caller workspace, call after
call, although every call reuses one static scratch array.

This file is collected last on purpose, so that a run stopping at its first
failure has already run every other test."""
import numpy as np
import pytest
import torch

from dropless_moe_expert_router_gb300 import api

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    from dropless_moe_expert_router_gb300 import build
    build.build()


def _case(T, H, E, K, seed, id_dtype):
    g = torch.Generator().manual_seed(seed)
    lg = torch.randn((T, E), generator=g)
    ids = torch.topk(lg, K, dim=1).indices.to(id_dtype)
    ids[torch.rand((T, K), generator=g) < 0.05] = -1            # some invalid routes
    x = (torch.randn((T, H), generator=g) * 0.02).to(torch.bfloat16)
    return x.cuda(), ids.cuda()


def _same(a: api.Permuted, b: api.Permuted):
    R = int(a.group_offsets[-1])
    assert torch.equal(a.group_sizes, b.group_sizes)
    assert torch.equal(a.group_offsets, b.group_offsets)
    assert torch.equal(a.row_map, b.row_map)
    assert torch.equal(a.perm_src[:R], b.perm_src[:R])
    assert torch.equal(a.x_perm[:R], b.x_perm[:R])
    if a.x_perm_scales is not None:
        assert torch.equal(a.x_perm_scales[:R], b.x_perm_scales[:R])


def test_noalloc_permute_matches_workspace_permute_on_consecutive_calls():
    # a large-expert call fills much of the static scratch, then a small one must
    # not be affected by what the first left behind; then the first shape again
    cases = [(2048, 512, 2304, 36, 1, torch.int16, False),
             (1000, 256, 8, 2, 2, torch.int32, True),
             (2048, 512, 2304, 36, 3, torch.int16, False)]
    for T, H, E, K, seed, dt, fuse in cases:
        x, ids = _case(T, H, E, K, seed, dt)
        ref = api.moe_permute(x, ids, E, fuse_mxfp8=fuse)
        got = api.moe_permute_noalloc(x, ids, E, fuse_mxfp8=fuse)
        torch.cuda.synchronize()
        _same(got, ref)
    assert api.moe_get_device_errors() == 0


def test_noalloc_permute_rejects_problems_beyond_its_scratch():
    """A problem whose count table exceeds the static scratch gets MOE_ERR_WORKSPACE before
    anything is enqueued (the small buffers passed are never touched); argument errors are
    reported first, as moe_permute reports them."""
    cap = api.moe_permute_noalloc_max_scratch()
    T, H, K, E = 1 << 20, 64, 2, 8192                   # needs E * T/64 * 4 bytes of table
    assert api.moe_permute_workspace_size(T, K, E) > cap
    from dropless_moe_expert_router_gb300 import _lib
    buf = torch.zeros(4096, dtype=torch.uint8, device="cuda")       # stands for every buffer
    ints = torch.zeros(E + 1, dtype=torch.int32, device="cuda")
    p = buf.data_ptr()
    L = _lib.load()
    st = L.moe_permute_noalloc(p, T, H, p, 1, K, E, p, None, ints.data_ptr(), ints.data_ptr(), p, p, 0, None)
    assert st == 3   # MOE_ERR_WORKSPACE, nothing enqueued
    st = L.moe_permute_noalloc(p, T, H, p, 1, K, E, None, None, ints.data_ptr(), ints.data_ptr(), p, p, 0, None)
    assert st == 1   # MOE_ERR_INVALID_ARG: the null x_perm is reported before the size
    torch.cuda.synchronize()
    assert not buf.any() and not ints.any()
