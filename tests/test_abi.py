"""The C-ABI library loads and exports every entry point include/*.h declares;
host-side helpers (no GPU needed)."""
import glob
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def lib():
    from dropless_moe_expert_router_gb300 import _lib, build
    build.build()
    return _lib.load()


def _declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        for m in re.finditer(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(moe_[a-z0-9_]+)\s*\(",
                             src, flags=re.M):
            names.append(m.group(1))
    return sorted(set(names))


def test_header_declares_the_hot_path():
    names = _declared_functions()
    for required in ("moe_route_topk", "moe_permute", "moe_quant_mxfp8_grouped",
                     "moe_unpermute_combine", "moe_get_device_errors"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    from dropless_moe_expert_router_gb300 import _lib
    for name in _declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"{name} has no ctypes signature"


def test_status_strings(lib):
    assert lib.moe_status_string(0) == b"MOE_OK"
    assert lib.moe_status_string(1) == b"MOE_ERR_INVALID_ARG"
    assert lib.moe_status_string(99) == b"MOE_ERR_UNKNOWN"


def test_argument_errors_need_no_gpu(lib):
    # bad shapes are rejected synchronously, before any CUDA call
    assert lib.moe_route_topk(None, 4, 8, 9, None, 1, None, 0, None) == 1   # K > E
    assert lib.moe_route_topk(None, 4, 40000, 2, None, 0, None, 0, None) == 1  # int16 ids, E too big
    assert lib.moe_route_topk(None, 0, 8, 2, None, 1, None, 0, None) == 0   # T = 0 is a no-op
    assert lib.moe_permute(None, 4, 30, None, 1, 2, 8, None, None, None, None, None, None,
                           0, None, 0, None) == 1                            # H % 32 != 0
    assert lib.moe_unpermute_combine(None, None, None, 4, 2, 12, None, None) == 1  # H % 8 != 0
    assert lib.moe_quant_mxfp8_grouped(None, 4, 64, None, 2, None, None, 8, None) == 1  # bad flag


def test_argument_errors_of_the_later_entry_points_need_no_gpu(lib):
    """Sigmoid router, NVFP4 and backward entry points reject bad shapes before any CUDA call
    (1 = MOE_ERR_INVALID_ARG, 2 = MOE_ERR_UNSUPPORTED)."""
    # sigmoid router: K > E; E past the register-resident limit; K past 64; T = 0 is a no-op
    assert lib.moe_route_sigmoid_topk(None, None, 4, 8, 9, None, 1, None, 0, None) == 1
    assert lib.moe_route_sigmoid_topk(None, None, 4, 1025, 2, None, 1, None, 0, None) == 2
    assert lib.moe_route_sigmoid_topk(None, None, 4, 100, 65, None, 1, None, 0, None) == 2
    assert lib.moe_route_sigmoid_topk(None, None, 0, 8, 2, None, 1, None, 0, None) == 0
    assert lib.moe_route_sigmoid_topk(None, None, 4, 8, 2, None, 1, None, 4, None) == 1     # unknown flag
    assert lib.moe_route_sigmoid_topk_backward(None, None, 1, None, 4, 8, 9, 0, None, None) == 1
    # NVFP4: cols not whole 16-element blocks; the GEMMs' 256-element k-blocks
    assert lib.moe_quant_nvfp4(None, 4, 24, None, None, None, None, None) == 1
    assert lib.moe_amax_bf16(None, 4, 12, None, None, None) == 1
    import ctypes
    goff = ctypes.c_void_p(256)     # non-null placeholder: the shape check returns before any use
    assert lib.moe_grouped_gemm_up_nvfp4(None, None, None, None, None, None, goff, 2, 384, 512, 64,
                                         None, None, None, None) == 2
    assert lib.moe_grouped_gemm_down_nvfp4(None, None, None, None, None, None, goff, 2, 512, 640, 64,
                                           None, None) == 2
    assert lib.moe_grouped_gemm_up_nvfp4(None, None, None, None, None, None, None, 2, 512, 512, 64,
                                         None, None, None, None) == 1                      # no offsets
    assert lib.moe_permute_nvfp4(None, 4, 48, None, 1, 2, 8, None, None, None, None, None, None, None,
                                 None, 0, None) == 1                                           # H % 32 != 0
    # combine backward: the fused MXFP8 outputs go together and need whole 32-element blocks
    assert lib.moe_unpermute_combine_backward(None, None, None, None, 4, 2, 72, None, None, None, None,
                                              None) == 1


def test_workspace_size_covers_the_tile_table(lib):
    # one int32 per (expert, token tile) plus a 16-byte counter
    assert lib.moe_permute_workspace_size(8192, 2, 8) >= 8 * (8192 // 128) * 4 + 16
    assert lib.moe_permute_workspace_size(8192, 36, 2304) >= 2304 * (8192 // 64) * 4 + 16   # 64-token tiles above 64 experts
    assert lib.moe_permute_workspace_size(-1, 2, 8) == 0


def test_permute_expert_limit_needs_no_gpu(lib):
    """Above 64 experts the count kernel holds a 64-bit token mask and a count per expert in
    shared memory (12 bytes each, within 227 KB): E = 19370 passes the argument checks (and then
    stops at the missing workspace), E = 19371 is unsupported. No pointer is dereferenced."""
    import ctypes
    g = ctypes.c_void_p(16)       # stands for the group buffers (never touched on these paths)
    args = lambda E: (None, 0, 64, None, 1, 2, E, None, None, g, g, None, None, 0, None, 0, None)
    assert lib.moe_permute(*args(19370)) == 3       # MOE_ERR_WORKSPACE
    assert lib.moe_permute(*args(19371)) == 2       # MOE_ERR_UNSUPPORTED
    assert lib.moe_permute(*args(64)) == 3


def test_permute_launch_count(lib):
    # the count table is scanned inside the scatter kernel when it is small (<= 2048 entries)
    assert lib.moe_permute_kernel_launches(8192, 2, 8) == 2          # 8 experts x 64 tiles
    assert lib.moe_permute_kernel_launches(8192, 4, 32) == 2         # 32 x 64
    assert lib.moe_permute_kernel_launches(32768, 8, 32) == 3        # 32 x 256: separate scan
    assert lib.moe_permute_kernel_launches(8192, 36, 2304) == 3      # 2304 x 256: separate scan
    assert lib.moe_permute_kernel_launches(32, 2, 8192) == 3         # table + offsets past 48 KB
    assert lib.moe_permute_kernel_launches(0, 2, 8) == 0
    assert lib.moe_permute_kernel_launches(-1, 2, 8) == -1


def test_compact_route_sizes_match_page(lib):
    """Page values ("Sparser MoE end-to-end", "Preserve a compact route" and
    "Remove work that has no selected route"): 18.87 MB -> 0.59 MB (32x), and a
    9,216-byte FP32 prob row vs a 128-byte 32-expert slice."""
    vals = {}
    for line in open(os.path.join(GOLDEN, "route_metadata_sizes.txt")):
        line = line.split("#", 1)[0].strip()
        if line:
            k, v = line.split("=")
            vals[k.strip()] = float(v)
    T, E, K = int(vals["T"]), int(vals["E"]), int(vals["K"])
    ids_bytes = lib.moe_route_ids_bytes(T, K, 0)
    assert round(ids_bytes / 1e6, 2) == vals["int16_ids_MB"]
    assert round(T * E / 1e6, 2) == vals["bool_map_MB"]
    assert (T * E) // ids_bytes == vals["ratio"]
    assert lib.moe_route_probs_bytes(1, E) == vals["prob_row_bytes"]
    assert lib.moe_route_probs_bytes(1, int(vals["local_experts"])) == vals["prob_slice_bytes"]
