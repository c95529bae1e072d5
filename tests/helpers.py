"""Small helpers shared by the GPU tests: device/host conversion of bf16
tensors and the rounding-error bound used for fp32 reductions."""
import numpy as np
import torch

U32 = 2.0 ** -23   # fp32 spacing at 1; covers truncating accumulators too


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (on the host)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(
        np.uint16)


def f32bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy().view(np.uint32)


def from_bits(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(
        torch.bfloat16).to(device)


def gamma(n, u=U32):
    return n * u / (1 - n * u)


def sum_bound(orc, x_bits, w_bits):
    """sum_k |x_mk| |w_nk| in float64 for the rounding bound."""
    xf = np.abs(orc.bf16_value(x_bits).astype(np.float64))
    wf = np.abs(orc.bf16_value(w_bits).astype(np.float64))
    return xf @ wf.T


def norm_rel_err(a, b):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-30))
