"""Helpers shared by the GPU parity tests (conversion between device tensors
and the numpy arrays the oracle takes)."""
import numpy as np
import torch

BF16_TOL = 2e-2  # max-abs, bf16 inputs / fp32 accumulation
F32_TOL = 1e-4   # max-abs, fp32


def tol_for(dtype):
    return F32_TOL if dtype == torch.float32 else BF16_TOL


def f32_np(t: torch.Tensor) -> np.ndarray:
    """Exact fp32 values of a (bf16 or fp32) tensor as a numpy array."""
    return t.detach().float().cpu().contiguous().numpy()


def bytes_np(t: torch.Tensor) -> np.ndarray:
    """Raw bytes of a tensor, shape [..., last_dim * element_size]."""
    t = t.detach().contiguous().cpu()
    return t.view(torch.uint8).numpy().reshape(*t.shape[:-1], -1)


def random_bytes(shape, dtype, gen, device="cuda"):
    """A tensor of the given element dtype holding uniformly random bytes
    (any bit pattern, NaN payloads included: copies must preserve them)."""
    elt = torch.empty((), dtype=dtype).element_size()
    raw = torch.randint(0, 256, (*shape[:-1], shape[-1] * elt), dtype=torch.uint8, generator=gen)
    return raw.view(dtype).reshape(shape).to(device)


def max_abs(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.size == 0:
        return 0.0
    return float(np.abs(a - b).max())
