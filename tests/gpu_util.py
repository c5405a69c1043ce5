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


GUARD_BYTES = 4096
GUARD_FILL = 0xA5


class Guarded:
    """A device output buffer with GUARD_BYTES of a known byte pattern on each
    side (stand-in for a memory checker: a kernel that writes past either end
    of its output changes the pattern).  `t` is the buffer itself (16-byte
    aligned); `intact()` tells whether both guards still hold the pattern."""

    def __init__(self, shape, dtype=torch.float32, fill=None):
        shape = tuple(shape)
        esize = torch.empty((), dtype=dtype).element_size()
        self.n = int(np.prod(shape, dtype=np.int64)) * esize
        self.raw = torch.full((2 * GUARD_BYTES + self.n,), GUARD_FILL, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD_BYTES:GUARD_BYTES + self.n].view(dtype).view(shape)
        if fill is not None:
            self.t.fill_(fill)

    def intact(self) -> bool:
        head = self.raw[:GUARD_BYTES]
        tail = self.raw[GUARD_BYTES + self.n:]
        return bool((head == GUARD_FILL).all().item() and (tail == GUARD_FILL).all().item())

