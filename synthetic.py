"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module only draws random numbers and shapes them; it holds none of the
method's arithmetic (no EMA, no SVD, no filter, no mask function, no K rule).
Both the CUDA path and the oracle receive the arrays made here.

Readings of the workload text (stated once, used everywhere):
  * ``N(0, x)``: x is the standard deviation (weights "~N(0,0.02)" is the usual
    init std).
  * Anchor-gradient signal: ``scale * A @ B.T`` with A (m x rank), B (n x rank),
    both ~N(0,1)/sqrt(m), scale 1e-2.
  * Anchor gradient = signal + N(0,1e-4) noise; masked gradient = anchor
    gradient + N(0,1e-2) noise, fresh noise for every steady step.
  * Activations / activation gradients for the mask: ~N(0,1), rounded to bf16
    (round to nearest even) where the workload says bf16.
  * Data-parallel outer synchronisation: the starting PowerSGD Q ~N(0,1) (the
    same on every worker); a worker's weights after one outer period are the
    outer weights minus a drift ~N(0, 1e-3), fresh per worker and period.

Every stream is keyed by ``numpy.random.SeedSequence([seed, tag, index])`` so
that any single tensor can be regenerated on its own.
"""
from __future__ import annotations

import numpy as np

# tags that separate independent random streams
_TAG_W, _TAG_SIG_A, _TAG_SIG_B, _TAG_ANC_NOISE, _TAG_MASK_NOISE = 1, 2, 3, 4, 5
_TAG_H, _TAG_GRAD = 6, 7
_TAG_DP_Q, _TAG_DP_DRIFT = 8, 9

# shapes (out_features m, in_features n) of one Llama-3.2-1B decoder layer
LLAMA_1B_LAYER = {
    "q": (2048, 2048), "k": (512, 2048), "v": (512, 2048), "o": (2048, 2048),
    "gate": (8192, 2048), "up": (8192, 2048), "down": (2048, 8192),
}
# shapes of one 7B-class decoder layer (hidden 4096, intermediate 14336, kv 1024)
LLAMA_7B_LAYER = {
    "q": (4096, 4096), "k": (1024, 4096), "v": (1024, 4096), "o": (4096, 4096),
    "gate": (14336, 4096), "up": (14336, 4096), "down": (4096, 14336),
}
# full Llama-3.2-1B: 16 layers of the 7 matrices, plus these AdamW-only tensors
LLAMA_1B_LAYERS = 16
LLAMA_1B_EMBED = (128256, 2048)
LLAMA_1B_NORMS = 2 * LLAMA_1B_LAYERS + 1   # two RMSNorm vectors per layer + final


def _rng(seed: int, tag: int, index: int = 0) -> np.random.Generator:
    return np.random.default_rng(np.random.SeedSequence([int(seed), int(tag), int(index)]))


def normal_f32(seed: int, tag: int, index: int, shape, std: float) -> np.ndarray:
    """float32 array ~N(0, std) from an independent keyed stream."""
    x = _rng(seed, tag, index).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounding = ((u >> 16) & 1) + np.uint32(0x7FFF)
    out = ((u + rounding) >> 16).astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = np.uint16(0x7FC0)
    return out


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


class MatrixInputs:
    """Inputs of the spectral-corrected step for one weight matrix (m x n, row-major)."""

    def __init__(self, m: int, n: int, seed: int = 0, rank: int = 8, signal_scale: float = 1e-2,
                 anchor_noise: float = 1e-4, mask_noise: float = 1e-2, w_std: float = 0.02,
                 factor_norm: int | None = None):
        self.m, self.n, self.seed, self.rank = m, n, seed, rank
        self.signal_scale, self.anchor_noise, self.mask_noise, self.w_std = (
            signal_scale, anchor_noise, mask_noise, w_std)
        self.factor_norm = m if factor_norm is None else factor_norm
        self._signal = None

    def weights(self) -> np.ndarray:
        return normal_f32(self.seed, _TAG_W, 0, (self.m, self.n), self.w_std)

    def signal(self) -> np.ndarray:
        if self._signal is None:
            inv = np.float32(1.0 / np.sqrt(self.factor_norm))
            a = normal_f32(self.seed, _TAG_SIG_A, 0, (self.m, self.rank), 1.0) * inv
            b = normal_f32(self.seed, _TAG_SIG_B, 0, (self.n, self.rank), 1.0) * inv
            self._signal = (np.float32(self.signal_scale) * (a @ b.T)).astype(np.float32)
        return self._signal

    def anchor_grad(self, index: int = 0) -> np.ndarray:
        """Anchor gradient number ``index``: fixed low-rank signal + fresh noise."""
        g = self.signal() + normal_f32(self.seed, _TAG_ANC_NOISE, index, (self.m, self.n),
                                       self.anchor_noise)
        return g.astype(np.float32)

    def masked_grad(self, step: int, anchor_index: int = 0) -> np.ndarray:
        """Masked gradient of steady step ``step``: anchor gradient + fresh N(0, mask_noise)."""
        g = self.anchor_grad(anchor_index) + normal_f32(self.seed, _TAG_MASK_NOISE, step,
                                                        (self.m, self.n), self.mask_noise)
        return g.astype(np.float32)


def toy_matrix_inputs(seed: int = 0) -> MatrixInputs:
    """Toy case: W 256x128, rank-8 anchor signal with factors ~N(0,1)/sqrt(256)."""
    return MatrixInputs(256, 128, seed=seed, rank=8, factor_norm=256)


def layer_inputs(shapes: dict, seed: int = 0, rank: int = 32) -> dict:
    """One MatrixInputs per named matrix; each matrix gets its own seed offset."""
    return {name: MatrixInputs(m, n, seed=seed * 1000 + i, rank=rank)
            for i, (name, (m, n)) in enumerate(shapes.items())}


def activations_bf16(rows: int, H: int, seed: int = 0, index: int = 0) -> np.ndarray:
    """bf16 activations ~N(0,1) as uint16 bit patterns, shape (rows, H)."""
    return f32_to_bf16_bits(normal_f32(seed, _TAG_H, index, (rows, H), 1.0))


def act_grads_f32(rows: int, H: int, seed: int = 0, index: int = 0) -> np.ndarray:
    return normal_f32(seed, _TAG_GRAD, index, (rows, H), 1.0)


def act_grads_bf16(rows: int, H: int, seed: int = 0, index: int = 0) -> np.ndarray:
    return f32_to_bf16_bits(act_grads_f32(rows, H, seed, index))


def dp_q0(n: int, k: int, seed: int = 0, index: int = 0) -> np.ndarray:
    """Starting Q (n x k) of the PowerSGD power step, ~N(0, 1)."""
    return normal_f32(seed, _TAG_DP_Q, index, (n, k), 1.0)


def dp_drift(m: int, n: int, seed: int = 0, worker: int = 0, period: int = 0,
             scale: float = 1e-3) -> np.ndarray:
    """Change of one worker's weights over one outer period, ~N(0, scale)."""
    return normal_f32(seed, _TAG_DP_DRIFT, worker * 1_000_003 + period, (m, n), scale)
