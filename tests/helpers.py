"""Small marshalling helpers shared by the tests (no arithmetic of the method)."""
import numpy as np
import torch


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> numpy uint16 payloads."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().numpy().view(np.uint8)


def rel_err(got: np.ndarray, ref: np.ndarray) -> float:
    """max |got - ref| / max |ref| (the parity measure for floating-point outputs)."""
    den = float(np.abs(ref).max())
    return float(np.abs(got - ref).max()) / (den if den > 0 else 1.0)
