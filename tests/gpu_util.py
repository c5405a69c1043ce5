"""Helpers of the GPU parity tests: device transfer and error measures."""
import numpy as np
import torch

import spectral_corrected_optimizer_gb300 as so
from spectral_corrected_optimizer_gb300 import build as sob

_built = False


def ensure_lib():
    global _built
    if not _built:
        sob.build()
        so.lib()
        _built = True


def dev(a: np.ndarray) -> torch.Tensor:
    """Host numpy -> CUDA tensor with the same bytes (uint16 arrays become bfloat16)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(a).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def rel(a, b) -> float:
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    return float(np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300))
