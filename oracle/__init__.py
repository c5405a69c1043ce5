"""Test infrastructure: the CPU oracle of the spectral-corrected optimizer step
and of the in-graph activation mask.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never calls it, and it calls nothing of the product path.

Everything floating point is float64.  Each function cites the passage of
"Communication-Efficient LLM Adaptation over Decentralized GPU Meshes"
(papernotes.org notes, NeurIPS 2026, arXiv 2609.14339) that it follows; the
steps are written in the pages' order and notation with no blocking, fusion
or reordering.  Library primitives used as single steps: numpy matmul.  The
SVD and the mask function are this package's own code (``oracle_c.c``).

Readings of places where the pages are silent (each one also listed in the
design notes):
  * anchor EMA starts from M = 0 and has no bias correction (none printed);
  * the SVD is the full thin SVD, r = min(m, n) (the pages reject hard
    truncation, every direction gets a soft weight d_i);
  * tau_p is an absolute threshold on the raw singular values;
  * d_i = 0 when s_i = 0 and tau_p = 0;
  * AdamW is the decoupled-weight-decay form with bias correction and eps
    outside the square root (the PyTorch ``AdamW`` definition);
  * the mask keeps a uniform pseudo-random K-subset of each row, selected by
    the keyed permutation in ``oracle_c.c``; no 1/(1-p) rescale;
  * K = floor((1-p) H + 1/2) evaluated in double;
  * key design 4 (data-parallel side): the outer synchronisation is DiLoCo's
    outer SGD with Nesterov momentum on the pseudo-gradient theta - W_local,
    compressed by one warm-started PowerSGD power step with error feedback;
    the rank k of each matrix gives mn / ((m + n) k) = 64; the orthonormal
    basis is Gram-Schmidt with dependent columns set to zero; workers' P and Q
    are summed and the decompressed update scaled by 1 / workers;
  * the mask fused with the layer boundary (key design 1 with the decoder
    layer around it): a bf16 sum is the float32 sum rounded to bf16 (nearest
    even); RMSNorm (Llama form, x = h / sqrt(mean(h^2) + eps) * gamma) is
    computed in float64 and rounded once.

Parity pins: every function here is checked in ``tests/test_oracle_*.py``
against closed forms, brute force, published test vectors or independent
library routines (LAPACK through numpy, torch.optim.AdamW, torch.optim.SGD,
torch autograd).
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_c.c")
_LIB_DIR = os.path.join(_HERE, "_build")
_LIB = os.path.join(_LIB_DIR, "liboracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile oracle_c.c with gcc into oracle/_build/liboracle.so (plain C11, -O2)."""
    os.makedirs(_LIB_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u32, u64, i32, i64, vp = (ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int32,
                                  ctypes.c_int64, ctypes.c_void_p)
        lib.oracle_sm64.restype = u64
        lib.oracle_sm64.argtypes = [u64]
        lib.oracle_fmix32.restype = u32
        lib.oracle_fmix32.argtypes = [u32]
        lib.oracle_mask_seed.restype = u64
        lib.oracle_mask_seed.argtypes = [u32, u64, u64]
        lib.oracle_mask_row_keys.restype = None
        lib.oracle_mask_row_keys.argtypes = [u64, u64, vp]
        lib.oracle_mask_perm.restype = u32
        lib.oracle_mask_perm.argtypes = [vp, u32, u32]
        lib.oracle_mask_indices.restype = ctypes.c_int
        lib.oracle_mask_indices.argtypes = [vp, i64, i32, i32, u32, u64, u64]
        for f in (lib.oracle_mask_pack, lib.oracle_mask_unpack):
            f.restype = ctypes.c_int
            f.argtypes = [vp, vp, i64, i32, i32, i32, u32, u64, u64]
        lib.oracle_thin_svd.restype = ctypes.c_int
        lib.oracle_thin_svd.argtypes = [vp, i64, i64, vp, vp, vp, i32, ctypes.c_double, vp]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


# ---------------------------------------------------------------------------
# key design 1: in-graph activation mask  h~ = h (.) m,  K = round((1-p)H),
# m = g(layer, step, B, S, H); backward dL/dh = (dL/dh~) (.) m
# ---------------------------------------------------------------------------

def mask_K(p: float, H: int) -> int:
    """K = round((1-p) H) kept dims per token (key design 1, mask equation).
    Rounding reading: floor(x + 1/2) in double."""
    return int(np.floor((1.0 - float(p)) * float(H) + 0.5))


def sm64(z: int) -> int:
    return int(_load().oracle_sm64(z & (2**64 - 1)))


def fmix32(x: int) -> int:
    return int(_load().oracle_fmix32(x & 0xFFFFFFFF))


def mask_seed(layer: int, step: int, batch_id: int) -> int:
    """Shared pseudo-random seed from (layer, step, batch metadata) (key design 1)."""
    return int(_load().oracle_mask_seed(layer, step, batch_id))


def mask_row_keys(seed: int, row: int) -> np.ndarray:
    keys = np.zeros(4, dtype=np.uint32)
    _load().oracle_mask_row_keys(seed, row, _ptr(keys))
    return keys


def mask_perm(keys: np.ndarray, H: int, k: int) -> int:
    keys = np.ascontiguousarray(keys, dtype=np.uint32)
    return int(_load().oracle_mask_perm(_ptr(keys), H, k))


def mask_indices(rows: int, H: int, K: int, layer: int, step: int, batch_id: int = 0) -> np.ndarray:
    """int32 [rows, K]: the kept dims of each row in packed (k) order."""
    out = np.zeros((rows, K), dtype=np.int32)
    rc = _load().oracle_mask_indices(_ptr(out), rows, H, K, layer, step, batch_id)
    if rc != 0:
        raise ValueError("oracle_mask_indices: bad arguments")
    return out


def mask_matrix(rows: int, H: int, K: int, layer: int, step: int, batch_id: int = 0) -> np.ndarray:
    """The mask m in {0,1}^{rows x H} as a bool array (never sent on the wire)."""
    m = np.zeros((rows, H), dtype=bool)
    idx = mask_indices(rows, H, K, layer, step, batch_id)
    np.put_along_axis(m, idx.astype(np.int64), True, axis=1)
    return m


def mask_pack(dense: np.ndarray, K: int, layer: int, step: int, batch_id: int = 0) -> np.ndarray:
    """Forward pack: packed[r, k] = h[r, pi_r(k)] -- only K values per token travel."""
    dense = np.ascontiguousarray(dense)
    rows, H = dense.shape
    out = np.zeros((rows, K), dtype=dense.dtype)
    rc = _load().oracle_mask_pack(_ptr(dense), _ptr(out), rows, H, K, dense.itemsize,
                                  layer, step, batch_id)
    if rc != 0:
        raise ValueError("oracle_mask_pack: bad arguments")
    return out


def mask_unpack(packed: np.ndarray, H: int, layer: int, step: int, batch_id: int = 0) -> np.ndarray:
    """Receiver unpack: h~[r, pi_r(k)] = packed[r, k], every other entry +0."""
    packed = np.ascontiguousarray(packed)
    rows, K = packed.shape
    out = np.empty((rows, H), dtype=packed.dtype)
    rc = _load().oracle_mask_unpack(_ptr(packed), _ptr(out), rows, H, K, packed.itemsize,
                                    layer, step, batch_id)
    if rc != 0:
        raise ValueError("oracle_mask_unpack: bad arguments")
    return out


# ---------------------------------------------------------------------------
# key design 2: anchor EMA  M_t = beta_anc M_{t-} + (1 - beta_anc) G_tau^anc
# ---------------------------------------------------------------------------

def anchor_ema(M: np.ndarray, G_anc: np.ndarray, beta_anc: float) -> np.ndarray:
    """Anchor momentum update (key design 2, EMA equation); float64."""
    return beta_anc * np.asarray(M, dtype=np.float64) + (1.0 - beta_anc) * np.asarray(G_anc, np.float64)


# ---------------------------------------------------------------------------
# key design 3: spectral correction
#   M = U S V^T;  d_i = s_i / (s_i + tau_p);
#   X = U^T G V;  X_filt = diag(d) X diag(d);  G_filt = U X_filt V^T;
#   G_proj = alpha G + (1 - alpha) G_filt  -> AdamW
# ---------------------------------------------------------------------------

def thin_svd(M: np.ndarray, max_sweeps: int = 80, tol: float | None = None):
    """Thin SVD M = U diag(s) V^T, r = min(m, n), s descending (key design 3).

    One-sided Jacobi in float64 (oracle_c.c).  Returns (U, s, V, sweeps)."""
    M = np.ascontiguousarray(M, dtype=np.float64)
    m, n = M.shape
    r = min(m, n)
    if tol is None:
        tol = 4e-16 * max(1.0, np.sqrt(max(m, n)))
    U = np.zeros((m, r))
    s = np.zeros(r)
    V = np.zeros((n, r))
    sweeps = np.zeros(1, dtype=np.int32)
    rc = _load().oracle_thin_svd(_ptr(M), m, n, _ptr(U), _ptr(s), _ptr(V), max_sweeps, tol,
                                 _ptr(sweeps))
    if rc == 4:
        raise RuntimeError("oracle_thin_svd did not converge in %d sweeps" % max_sweeps)
    if rc != 0:
        raise RuntimeError("oracle_thin_svd failed with status %d" % rc)
    return U, s, V, int(sweeps[0])


def filter_coeffs(s: np.ndarray, tau_p: float) -> np.ndarray:
    """Tikhonov soft filter d_i = s_i / (s_i + tau_p) (key design 3); 0 where s_i + tau_p = 0."""
    s = np.asarray(s, dtype=np.float64)
    den = s + tau_p
    return np.where(den > 0, s / np.where(den > 0, den, 1.0), 0.0)


def project(U: np.ndarray, V: np.ndarray, d: np.ndarray, G: np.ndarray):
    """Two-sided projection (key design 3): returns (X, X_filt, G_filt)."""
    U, V, d, G = (np.asarray(a, dtype=np.float64) for a in (U, V, d, G))
    X = U.T @ G @ V
    X_filt = np.diag(d) @ X @ np.diag(d)
    G_filt = U @ X_filt @ V.T
    return X, X_filt, G_filt


def blend(G_mask: np.ndarray, G_filt: np.ndarray, alpha: float) -> np.ndarray:
    """Convex combination G_proj = alpha G_mask + (1 - alpha) G_filt (key design 3)."""
    return alpha * np.asarray(G_mask, np.float64) + (1.0 - alpha) * np.asarray(G_filt, np.float64)


def adamw(W, m, v, g, t: int, lr: float, beta1: float, beta2: float, eps: float, wd: float):
    """One AdamW update at step t (t already incremented), decoupled weight decay.
    Returns (W_new, m_new, v_new), all float64."""
    W, m, v, g = (np.asarray(a, dtype=np.float64) for a in (W, m, v, g))
    W = W * (1.0 - lr * wd)
    m = beta1 * m + (1.0 - beta1) * g
    v = beta2 * v + (1.0 - beta2) * g * g
    m_hat = m / (1.0 - beta1 ** t)
    v_hat = v / (1.0 - beta2 ** t)
    W = W - lr * m_hat / (np.sqrt(v_hat) + eps)
    return W, m, v


class SpectralOptimizer:
    """The whole spectral-corrected optimizer for one weight matrix, float64.

    State: anchor momentum M (starts at 0, separate from AdamW's moments),
    thin SVD factors U, s, V and filter d (all zero before the first refresh,
    so the filtered gradient is 0 and G_proj = alpha G_mask until then),
    AdamW moments m, v and step counter t."""

    def __init__(self, m: int, n: int, beta_anc=0.9, tau_p=1e-3, alpha=0.3, beta1=0.9,
                 beta2=0.999, eps=1e-8, weight_decay=0.01):
        self.shape = (m, n)
        r = min(m, n)
        self.beta_anc, self.tau_p, self.alpha = beta_anc, tau_p, alpha
        self.beta1, self.beta2, self.eps, self.wd = beta1, beta2, eps, weight_decay
        self.M = np.zeros((m, n))
        self.U, self.s, self.V, self.d = np.zeros((m, r)), np.zeros(r), np.zeros((n, r)), np.zeros(r)
        self.exp_avg, self.exp_avg_sq, self.t = np.zeros((m, n)), np.zeros((m, n)), 0

    def anchor_update(self, G_anc):
        self.M = anchor_ema(self.M, G_anc, self.beta_anc)

    def svd_refresh(self):
        self.U, self.s, self.V, _ = thin_svd(self.M)
        self.d = filter_coeffs(self.s, self.tau_p)

    def step(self, W, G_mask, lr: float):
        """Returns (W_new, G_filt, G_proj)."""
        _, _, G_filt = project(self.U, self.V, self.d, G_mask)
        G_proj = blend(G_mask, G_filt, self.alpha)
        self.t += 1
        W_new, self.exp_avg, self.exp_avg_sq = adamw(W, self.exp_avg, self.exp_avg_sq, G_proj,
                                                     self.t, lr, self.beta1, self.beta2, self.eps,
                                                     self.wd)
        return W_new, G_filt, G_proj


# ---------------------------------------------------------------------------
# key design 4: dual compression on the data-parallel side -- the outer
# (Streaming DiLoCo) synchronisation of each weight matrix, its traffic cut
# 64x by PowerSGD low-rank compression.  The pages name the two methods and
# the ratio only; the steps below are the plainest reading of the two
# methods' own publications (PowerSGD: Vogels, Karimireddy and Jaggi,
# NeurIPS 2019, rank-k power step with error feedback and a warm-started Q;
# DiLoCo: Douillard et al. 2023, outer SGD with Nesterov momentum on the
# pseudo-gradient theta_outer - theta_local).
#
# Per matrix and worker, in order:
#   M     = E + (X - Y)                    (error feedback; Y optional)
#   P     = M Q                            -> summed over workers
#   P^    = orthonormal basis of P         (Gram-Schmidt, columns in order)
#   Q     = M^T P^                         -> summed over workers
#   D     = s P^ Q^T                       (s = 1 / number of workers)
#   E     = M - D                          (what the compression left out)
# then either the decompressed gradient D is handed on, or the outer step
#   b        = mu b + D
#   theta    = theta - eta (D + mu b)      (Nesterov, dampening 0)
#   W_local  = (1 - mix) theta + mix W_local
# ---------------------------------------------------------------------------

GS_DROP = 1e-10  # a column whose residual norm^2 is <= GS_DROP * its norm^2 is dependent


def dpsync_rank(m: int, n: int, ratio: float = 64.0) -> int:
    """Rank k of the low-rank factors that sends ratio-times fewer values than the
    m x n matrix: mn / ((m + n) k) = ratio, rounded half up, clamped to [1, min(m, n)]."""
    k = int(np.floor(m * n / (ratio * (m + n)) + 0.5))
    return max(1, min(min(m, n), k))


def dpsync_compress_p(X, Y, E, Q, error_feedback: bool = True):
    """First half of the power step: M = E + X - Y (Y may be None; E is ignored
    without error feedback) and P = M Q.  Returns (M, P) in float64."""
    M = np.asarray(X, dtype=np.float64).copy()
    if Y is not None:
        M = M - np.asarray(Y, dtype=np.float64)
    if error_feedback:
        M = np.asarray(E, dtype=np.float64) + M
    return M, M @ np.asarray(Q, dtype=np.float64)


def orthogonalize(P, drop: float = GS_DROP):
    """Orthonormal basis of the columns of P by Gram-Schmidt, column by column,
    each column projected twice against the accepted ones ("twice is enough").
    A column whose residual has norm^2 <= drop * (its own norm^2) is dependent
    and becomes a zero column; so does an all-zero column.  On full-rank P
    this is the Q factor of the thin QR with a positive diagonal of R."""
    P = np.asarray(P, dtype=np.float64)
    m, k = P.shape
    out = np.zeros((m, k))
    for c in range(k):
        v = P[:, c].copy()
        norm2 = float(v @ v)
        for _ in range(2):
            for j in range(c):
                v -= (out[:, j] @ v) * out[:, j]
        res2 = float(v @ v)
        if norm2 > 0.0 and res2 > drop * norm2:
            out[:, c] = v / np.sqrt(res2)
    return out


def dpsync_compress_q(M, P_hat):
    """Second half of the power step: Q = M^T P^ (float64)."""
    return np.asarray(M, dtype=np.float64).T @ np.asarray(P_hat, dtype=np.float64)


def dpsync_decompress(M, P_hat, Q_sum, q_scale: float = 1.0, error_feedback: bool = True):
    """D = q_scale P^ Q_sum^T (Q_sum is the sum over workers, q_scale = 1/workers)
    and the new error E = M - D (zero without error feedback).  Returns (D, E)."""
    D = q_scale * (np.asarray(P_hat, dtype=np.float64) @ np.asarray(Q_sum, dtype=np.float64).T)
    E = np.asarray(M, dtype=np.float64) - D if error_feedback else np.zeros_like(D)
    return D, E


def outer_nesterov(theta, mom, D, lr: float, momentum: float, W_local=None, mix: float = 0.0):
    """Outer optimizer step on the decompressed pseudo-gradient D: SGD with
    Nesterov momentum (dampening 0), then the worker's weights restart from the
    new outer weights, optionally mixed with its own (mix = 0: replaced).
    Returns (theta, mom, W_local) in float64."""
    theta, mom, D = (np.asarray(a, dtype=np.float64) for a in (theta, mom, D))
    mom = momentum * mom + D
    theta = theta - lr * (D + momentum * mom)
    if W_local is None or mix == 0.0:
        W_new = theta.copy()
    else:
        W_new = (1.0 - mix) * theta + mix * np.asarray(W_local, dtype=np.float64)
    return theta, mom, W_new


class DPSync:
    """The whole data-parallel synchronisation of one weight matrix on one
    worker, float64.  `allreduce(a)` returns the sum of `a` over the workers
    (identity for one worker); `workers` is their number.

    State: error E (starts at 0), the warm-started Q (given, n x k), and in
    outer mode the outer weights theta (set by `set_outer`) and momentum."""

    def __init__(self, m: int, n: int, Q0, rank: int = 0, ratio: float = 64.0,
                 error_feedback: bool = True, outer_lr: float = 0.7, outer_momentum: float = 0.9,
                 mix: float = 0.0):
        self.k = rank if rank > 0 else dpsync_rank(m, n, ratio)
        self.Q = np.asarray(Q0, dtype=np.float64).reshape(n, self.k).copy()
        self.E = np.zeros((m, n))
        self.error_feedback = error_feedback
        self.outer_lr, self.outer_momentum, self.mix = outer_lr, outer_momentum, mix
        self.theta = None
        self.mom = np.zeros((m, n))

    def set_outer(self, W):
        self.theta = np.asarray(W, dtype=np.float64).copy()
        self.mom = np.zeros_like(self.theta)

    def _power(self, X, Y, allreduce, workers):
        M, P = dpsync_compress_p(X, Y, self.E, self.Q, self.error_feedback)
        P_hat = orthogonalize(allreduce(P))
        self.Q = allreduce(dpsync_compress_q(M, P_hat))
        D, E = dpsync_decompress(M, P_hat, self.Q, 1.0 / workers, self.error_feedback)
        if self.error_feedback:
            self.E = E
        return D, P_hat

    def sync_grad(self, G, allreduce=lambda a: a, workers: int = 1):
        """Returns the decompressed mean gradient D."""
        return self._power(G, None, allreduce, workers)[0]

    def outer_sync(self, W_local, allreduce=lambda a: a, workers: int = 1):
        """Returns the worker's new weights; theta and the momentum advance."""
        D, _ = self._power(self.theta, W_local, allreduce, workers)
        self.theta, self.mom, W_new = outer_nesterov(self.theta, self.mom, D, self.outer_lr,
                                                     self.outer_momentum, W_local, self.mix)
        return W_new


# ---------------------------------------------------------------------------
# key design 1 at the layer boundary: the mask folded into the ops next to it.
# The page sends only the K kept values of the boundary activation and of its
# gradient; on the sender the boundary value is the decoder layer's residual
# sum h = a + b, on the receiver the next layer starts with RMSNorm of h~
# (Llama: x = h / sqrt(mean(h^2) + eps) * gamma) and keeps h~ for its residual
# branch.  All tensors bf16 (uint16 bit patterns here).  Readings: a bf16 sum
# is the float32 sum rounded to bf16 (nearest even); RMSNorm is computed in
# float64 here and rounded once to bf16 at the end.
# ---------------------------------------------------------------------------

def bf16_bits(x) -> np.ndarray:
    """Round to bfloat16, nearest with ties to even (via float32), as uint16 bits."""
    x = np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float32))
    u = x.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    return np.where(np.isnan(x), np.uint16(0x7FC0), r)


def bf16_value(bits) -> np.ndarray:
    """float64 value of bf16 bit patterns."""
    b = np.ascontiguousarray(np.asarray(bits, dtype=np.uint16)).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def mask_pack_add(a, b, K: int, layer: int, step: int, batch_id: int = 0) -> np.ndarray:
    """Sender: packed[r, k] = bf16(a + b)[r, pi_r(k)] (the residual sum is formed at
    the kept dims only)."""
    s = (bf16_value(a).astype(np.float32) + bf16_value(b).astype(np.float32))
    return mask_pack(bf16_bits(s), K, layer, step, batch_id)


def mask_unpack_rmsnorm(packed, gamma, eps: float, H: int, layer: int, step: int, batch_id: int = 0):
    """Receiver: h~ = unpack(packed) and x = RMSNorm(h~) * gamma.  Returns
    (h~ bits, x bits, x in float64 before rounding)."""
    h = mask_unpack(np.ascontiguousarray(packed, dtype=np.uint16), H, layer, step, batch_id)
    hv = bf16_value(h)
    r = 1.0 / np.sqrt(np.mean(hv * hv, axis=1, keepdims=True) + eps)
    x = hv * r * bf16_value(gamma)[None, :]
    return h, bf16_bits(x), x


def mask_rmsnorm_backward_pack(packed_h, gamma, eps: float, dx, g_res, layer: int, step: int,
                               batch_id: int = 0):
    """Receiver backward: dL/dh~ = g_res + RMSNorm backward of the upstream gradient
    dx, sent at the kept dims only:
      dL/dh~_j = g_res_j + gamma_j dx_j / r - h~_j (sum_i gamma_i dx_i h~_i) / (H r^3),
    r = sqrt(mean(h~^2) + eps).  Returns (packed bits, float64 values)."""
    packed_h = np.ascontiguousarray(packed_h, dtype=np.uint16)
    rows, K = packed_h.shape
    H = np.asarray(gamma).shape[0]
    h = bf16_value(mask_unpack(packed_h, H, layer, step, batch_id))
    g = bf16_value(gamma)[None, :]
    dxv = bf16_value(dx)
    rr = np.sqrt(np.mean(h * h, axis=1, keepdims=True) + eps)
    s = np.sum(g * dxv * h, axis=1, keepdims=True)
    dh = g * dxv / rr - h * s / (H * rr ** 3)
    if g_res is not None:
        dh = dh + bf16_value(g_res)
    idx = mask_indices(rows, H, K, layer, step, batch_id).astype(np.int64)
    vals = np.take_along_axis(dh, idx, axis=1)
    return bf16_bits(vals), vals


def mask_unpack_add(packed, g, layer: int, step: int, batch_id: int = 0) -> np.ndarray:
    """Sender backward: g[r, pi_r(k)] <- bf16(g + packed[r, k]); every other entry of g
    unchanged (the returned array is a new one)."""
    g = np.array(g, dtype=np.uint16, copy=True)
    packed = np.ascontiguousarray(packed, dtype=np.uint16)
    rows, K = packed.shape
    idx = mask_indices(rows, g.shape[1], K, layer, step, batch_id).astype(np.int64)
    cur = np.take_along_axis(g, idx, axis=1)
    s = bf16_value(cur).astype(np.float32) + bf16_value(packed).astype(np.float32)
    np.put_along_axis(g, idx, bf16_bits(s), axis=1)
    return g
