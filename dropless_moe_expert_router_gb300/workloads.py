"""Named workloads and seeded synthetic inputs for the dropless MoE layer.

This module only draws random numbers and states shapes: it holds none of the
layer's arithmetic, so both the CUDA path and the CPU oracle can be fed from it.
Every tensor is drawn on the CPU from its own seeded ``torch.Generator``
(seed = 1000 * base_seed + tensor id), so inputs are reproducible and do not
depend on the device.

Workloads (shapes of the models the pages discuss; weights are random, there is
no trained model or dataset behind them):

* ``tiny``        T=256, H=256, E=8, K=2, F=512, bf16; logits N(0,1).
* ``mixtral``     T=8192, H=4096, E=8, K=2, F=14336, bf16; logits N(0,1) plus a
                  per-expert bias N(0, 0.5) (mild skew); probs renormalised over
                  the K selected experts.
* ``dsv3``        T=8192, H=7168, E=32, K=4, F=2048, MXFP8; logits N(0,1) plus
                  gamma * ln p_e with p_e ~ (e+1)^-1.1 (Zipf), gamma chosen so that
                  about five experts receive no token.
* ``large_e``     T=8192, H=F=512, E=2304, K=36, bf16, int16 ids; logits N(0,1);
                  about 2 % of the (t,k) routes are marked invalid (-1).
* ``heavy``       T=32768, H=7168, E=32, K=8, F=2048, MXFP8, forward plus backward;
                  logits N(0,1) plus ln p_e with p_e ~ (e+1)^-1.5.
* ``dsv3_nvfp4``  the ``dsv3`` layer and routing with NVFP4 GEMM operands (forward).
* ``dsv3_sigmoid`` the ``dsv3`` layer and logits with the sigmoid-score router: selection
                  on sigmoid(logit) plus a per-expert bias U(-0.05, 0.05) (a balancing
                  correction), probs renormalised over the K selected scores.
"""
from __future__ import annotations

import dataclasses
import math

import torch

# tensor ids of the per-tensor generators
_X, _LOGITS, _BIAS, _W1, _W3, _W2, _INVALID, _DY = 1, 2, 3, 4, 5, 6, 7, 8
_EXPERT_BIAS = 12


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    E: int
    K: int
    F: int
    precision: str = "bf16"        # "bf16", "mxfp8" or "nvfp4" (operands of the expert GEMMs)
    bias: str = "none"             # "none", "normal", "zipf"
    bias_scale: float = 0.0        # std of the normal bias, or gamma of the Zipf bias
    zipf_s: float = 0.0
    renorm: bool = False
    id_bits: int = 32              # 16 or 32
    invalid_frac: float = 0.0
    backward: bool = False
    act_std: float = 0.02          # std of x, weights and dy
    score: str = "softmax"         # router score function: "softmax" or "sigmoid"
    expert_bias_scale: float = 0.0 # sigmoid router: selection bias ~ U(-scale, scale) per expert

    @property
    def R_cap(self) -> int:
        return self.T * self.K


WORKLOADS = {
    "tiny": Workload("tiny", T=256, H=256, E=8, K=2, F=512),
    "mixtral": Workload("mixtral", T=8192, H=4096, E=8, K=2, F=14336, bias="normal",
                        bias_scale=0.5, renorm=True),
    "dsv3": Workload("dsv3", T=8192, H=7168, E=32, K=4, F=2048, precision="mxfp8",
                     bias="zipf", bias_scale=2.0, zipf_s=1.1),
    "large_e": Workload("large_e", T=8192, H=512, E=2304, K=36, F=512, id_bits=16,
                        invalid_frac=0.02),
    "heavy": Workload("heavy", T=32768, H=7168, E=32, K=8, F=2048, precision="mxfp8",
                      bias="zipf", bias_scale=1.0, zipf_s=1.5, backward=True),
    "dsv3_nvfp4": Workload("dsv3_nvfp4", T=8192, H=7168, E=32, K=4, F=2048, precision="nvfp4",
                           bias="zipf", bias_scale=2.0, zipf_s=1.1),
    "dsv3_sigmoid": Workload("dsv3_sigmoid", T=8192, H=7168, E=32, K=4, F=2048, precision="mxfp8",
                             bias="zipf", bias_scale=2.0, zipf_s=1.1, score="sigmoid",
                             expert_bias_scale=0.05, renorm=True),
    # reduced Mixtral-like shape for profiler captures (same tile shapes and K loop,
    # a quarter of F and half of T: about 1.5 GB on the device)
    "mixtral_prof": Workload("mixtral_prof", T=4096, H=4096, E=8, K=2, F=3584, bias="normal",
                             bias_scale=0.5, renorm=True),
    # the 2,304-expert routing with narrow rows for profiler captures of the router and the
    # permute's count and scan kernels (the same ids and tiles; about 0.5 GB on the device)
    "large_e_prof": Workload("large_e_prof", T=8192, H=256, E=2304, K=36, F=128, id_bits=16,
                             invalid_frac=0.02),
    # reduced MXFP8 training shape for profiler captures (H, F of the DeepSeek-V3-like
    # slice, 8 experts, about 2 GB on the device)
    "dsv3_prof": Workload("dsv3_prof", T=4096, H=7168, E=8, K=2, F=2048, precision="mxfp8",
                          backward=True),
}


def get(name: str, **overrides) -> Workload:
    """A named workload, optionally with fields replaced (e.g. a smaller T)."""
    wl = WORKLOADS[name]
    return dataclasses.replace(wl, **overrides) if overrides else wl


def _gen(seed: int, tid: int) -> torch.Generator:
    return torch.Generator().manual_seed(1000 * seed + tid)


def _normal(shape, std, seed, tid, dtype=torch.bfloat16):
    g = _gen(seed, tid)
    out = torch.empty(shape, dtype=dtype)
    # draw in slabs along dim 0 to bound the fp32 temporary
    n0 = shape[0]
    per = max(1, (1 << 26) // max(1, math.prod(shape[1:])))
    for i in range(0, n0, per):
        j = min(n0, i + per)
        out[i:j] = (torch.randn((j - i,) + tuple(shape[1:]), generator=g) * std).to(dtype)
    return out


def logits(wl: Workload, seed: int = 0) -> torch.Tensor:
    """Router logits [T, E] fp32: N(0,1) plus the workload's per-expert bias."""
    lg = torch.randn((wl.T, wl.E), generator=_gen(seed, _LOGITS))
    if wl.bias == "normal":
        lg += torch.randn((wl.E,), generator=_gen(seed, _BIAS)) * wl.bias_scale
    elif wl.bias == "zipf":
        ranks = torch.arange(1, wl.E + 1, dtype=torch.float64)
        lnp = -wl.zipf_s * torch.log(ranks)
        lnp -= torch.logsumexp(lnp, 0)          # ln of the normalised Zipf pmf
        lg += (wl.bias_scale * lnp).to(torch.float32)
    return lg.contiguous()


def expert_bias(wl: Workload, seed: int = 0):
    """The sigmoid router's per-expert selection bias [E] fp32 ~ U(-s, s), or None."""
    if wl.score != "sigmoid" or wl.expert_bias_scale <= 0:
        return None
    u = torch.rand((wl.E,), generator=_gen(seed, _EXPERT_BIAS), dtype=torch.float64)
    return ((2 * u - 1) * wl.expert_bias_scale).to(torch.float32)


def x(wl: Workload, seed: int = 0) -> torch.Tensor:
    """Token activations [T, H] bf16 ~ N(0, 0.02)."""
    return _normal((wl.T, wl.H), wl.act_std, seed, _X)


def weights(wl: Workload, seed: int = 0):
    """Expert weights in their logical layouts: W1, W3 [E, H, F] and W2 [E, F, H], bf16."""
    w1 = _normal((wl.E, wl.H, wl.F), wl.act_std, seed, _W1)
    w3 = _normal((wl.E, wl.H, wl.F), wl.act_std, seed, _W3)
    w2 = _normal((wl.E, wl.F, wl.H), wl.act_std, seed, _W2)
    return w1, w3, w2


def invalid_mask(wl: Workload, seed: int = 0) -> torch.Tensor:
    """Bernoulli(invalid_frac) mask [T, K] of routes to mark invalid (-1) after routing."""
    if wl.invalid_frac <= 0:
        return torch.zeros((wl.T, wl.K), dtype=torch.bool)
    u = torch.rand((wl.T, wl.K), generator=_gen(seed, _INVALID))
    return u < wl.invalid_frac


def dy_perm(wl: Workload, seed: int = 0) -> torch.Tensor:
    """Upstream gradient of the permuted expert outputs [T*K, H] bf16 ~ N(0, 0.02)."""
    return _normal((wl.R_cap, wl.H), wl.act_std, seed, _DY)


_YPERM = 9


def expert_out(wl: Workload, seed: int = 0) -> torch.Tensor:
    """Synthetic expert outputs in permuted order [T*K, H] bf16 ~ N(0, 0.02) (to test combine alone)."""
    return _normal((wl.R_cap, wl.H), wl.act_std, seed, _YPERM)


_DYOUT, _DPROBS = 10, 11


def dy(wl: Workload, seed: int = 0) -> torch.Tensor:
    """Upstream gradient of the layer output [T, H] bf16 ~ N(0, 0.02)."""
    return _normal((wl.T, wl.H), wl.act_std, seed, _DYOUT)


def dprobs(wl: Workload, seed: int = 0) -> torch.Tensor:
    """Upstream gradient of the router probabilities [T, K] fp32 ~ N(0, 1)."""
    return torch.randn((wl.T, wl.K), generator=_gen(seed, _DPROBS)).contiguous()
