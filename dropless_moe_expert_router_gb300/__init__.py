"""GB300-native dropless Mixture-of-Experts layer hot path.

router top-K -> permute (dispatch, optional fused MXFP8) -> grouped SwiGLU
GEMMs -> probability-weighted combine, as hand-written sm_103a CUDA kernels
behind the C ABI in include/moe_gb300.h. This package is the thin Python
binding (``api``), the in-tree build (``build``) and the named synthetic
workloads (``workloads``).
"""
from .api import (MoeError, Permuted, moe_get_device_errors, moe_permute,  # noqa: F401
                  moe_permute_workspace_size, moe_quant_mxfp8_grouped, moe_route_ids_bytes,
                  moe_route_probs_bytes, moe_route_topk, moe_unpermute_combine, permute_buffers,
                  PackedWeights, moe_prepare_weights, moe_grouped_swiglu_gemm)
