"""Python binding of libspecoptim.so (argument marshalling only).

Every operation runs in the library's CUDA kernels; this module only checks
shapes and dtypes of torch tensors, passes their device pointers and the
current CUDA stream through the C-ABI declared in include/specoptim.h, and
turns status codes into exceptions.  There is no CPU path: without the built
library every call raises.

Method: "Communication-Efficient LLM Adaptation over Decentralized GPU Meshes"
(arXiv 2609.14339), key designs 1 (activation mask), 2 (anchor EMA) and 3
(spectral-correction optimizer); key design 4 (PowerSGD-compressed outer
synchronisation) is bound in the ``dpsync`` submodule.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

LIB_PATH = _build.LIB

OK, ERR_INVALID_ARG, ERR_MISALIGNED, ERR_CUDA, ERR_NOT_CONVERGED, ERR_NOT_IMPLEMENTED, ERR_TIMEOUT, ERR_BOUNDS = range(8)
PREC_TF32, PREC_FP32 = 0, 1

_STATUS = {1: "invalid argument", 2: "misaligned pointer", 3: "CUDA error", 4: "SVD not converged",
           5: "not implemented", 6: "device-side wait timed out", 7: "index check failed (checked build)"}


class SpecOptimError(RuntimeError):
    def __init__(self, code: int, what: str, msg: str):
        super().__init__("%s failed: %s (%d): %s" % (what, _STATUS.get(code, "error"), code, msg))
        self.code = code


class Config(ctypes.Structure):
    _fields_ = [("m", ctypes.c_int32), ("n", ctypes.c_int32), ("beta_anc", ctypes.c_float),
                ("tau_p", ctypes.c_float), ("alpha", ctypes.c_float), ("beta1", ctypes.c_float),
                ("beta2", ctypes.c_float), ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float),
                ("precision", ctypes.c_int32), ("svd_max_sweeps", ctypes.c_int32),
                ("svd_tol", ctypes.c_float), ("svd_inner_sweeps", ctypes.c_int32)]


class DPConfig(ctypes.Structure):
    """dpsync_config of include/dpsync.h."""
    _fields_ = [("m", ctypes.c_int32), ("n", ctypes.c_int32), ("rank", ctypes.c_int32),
                ("ratio", ctypes.c_float), ("error_feedback", ctypes.c_int32),
                ("outer_lr", ctypes.c_float), ("outer_momentum", ctypes.c_float),
                ("mix", ctypes.c_float)]


# (name, restype, argtypes) of every exported entry point of include/specoptim.h,
# include/mask_fused.h and include/dpsync.h
_vp, _i32, _i64, _u32, _u64, _f32, _f64 = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                                           ctypes.c_uint32, ctypes.c_uint64, ctypes.c_float,
                                           ctypes.c_double)
_int = ctypes.c_int
SIGNATURES = [
    ("specoptim_config_default", _int, [ctypes.POINTER(Config), _i32, _i32]),
    ("specoptim_create", _int, [ctypes.POINTER(_vp), ctypes.POINTER(Config), _vp]),
    ("specoptim_destroy", _int, [_vp]),
    ("specoptim_anchor_update", _int, [_vp, _vp, _vp]),
    ("specoptim_svd_refresh", _int, [_vp, _vp, ctypes.POINTER(_i32)]),
    ("specoptim_svd_refresh_many", _int, [ctypes.POINTER(_vp), _i32, _vp, ctypes.POINTER(_i32)]),
    ("specoptim_svd_refresh_begin", _int, [ctypes.POINTER(_vp), _i32, _vp]),
    ("specoptim_svd_refresh_end", _int, [ctypes.POINTER(_vp), _i32, _vp, ctypes.POINTER(_i32)]),
    ("specoptim_step", _int, [_vp, _vp, _vp, _f32, _vp, _vp, _vp]),
    ("specoptim_step_many", _int, [ctypes.POINTER(_vp), _i32, ctypes.POINTER(_vp), ctypes.POINTER(_vp), _f32, _vp]),
    ("specoptim_get_factors", _int, [_vp, _vp, _vp, _vp, _vp, _vp]),
    ("specoptim_get_state", _int, [_vp, _vp, _vp, _vp, ctypes.POINTER(_i64), _vp]),
    ("specoptim_set_state", _int, [_vp, _vp, _vp, _vp, _i64, _vp]),
    ("specoptim_adamw", _int, [_vp, _vp, _vp, _vp, _i64, _i64, _f32, _f32, _f32, _f32, _f32, _vp]),
    ("specoptim_gemm_nt", _int, [_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _i32, _vp]),
    ("specoptim_filter_noalloc", _int, [_vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _vp]),
    ("specoptim_selftest_wait_timeout", _int, [_u32, _vp]),
    ("specoptim_check_device", _int, [_vp]),
    ("specoptim_trace_enable", _int, [_i32]),
    ("specoptim_launch_count", _i64, []),
    ("specoptim_trace_reset", _int, []),
    ("specoptim_trace_report", _int, [ctypes.c_char_p, _i64]),
    ("specoptim_last_error", ctypes.c_char_p, []),
    ("mask_keep_count", _i32, [_f64, _i32]),
    ("mask_pack", _int, [_vp, _vp, _i64, _i32, _i32, _i32, _u32, _u64, _u64, _vp]),
    ("mask_unpack", _int, [_vp, _vp, _i64, _i32, _i32, _i32, _u32, _u64, _u64, _vp]),
    ("mask_indices", _int, [_vp, _i64, _i32, _i32, _u32, _u64, _u64, _vp]),
    ("mask_pack_add", _int, [_vp, _vp, _vp, _i64, _i32, _i32, _u32, _u64, _u64, _vp]),
    ("mask_unpack_rmsnorm", _int, [_vp, _vp, _f32, _vp, _vp, _i64, _i32, _i32, _u32, _u64, _u64, _vp]),
    ("mask_rmsnorm_backward_pack", _int, [_vp, _vp, _f32, _vp, _vp, _vp, _i64, _i32, _i32, _u32, _u64, _u64, _vp]),
    ("mask_unpack_add", _int, [_vp, _vp, _i64, _i32, _i32, _u32, _u64, _u64, _vp]),
    ("dpsync_rank", _i32, [_i32, _i32, _f32]),
    ("dpsync_config_default", _int, [ctypes.POINTER(DPConfig), _i32, _i32]),
    ("dpsync_create", _int, [ctypes.POINTER(_vp), ctypes.POINTER(DPConfig), _vp, _vp, _vp]),
    ("dpsync_handle_rank", _i32, [_vp]),
    ("dpsync_destroy", _int, [_vp]),
    ("dpsync_set_outer", _int, [_vp, _vp, _vp]),
    ("dpsync_compress_p_many", _int, [ctypes.POINTER(_vp), _i32, ctypes.POINTER(_vp), ctypes.POINTER(_vp), _vp]),
    ("dpsync_orthogonalize_many", _int, [ctypes.POINTER(_vp), _i32, _vp]),
    ("dpsync_compress_q_many", _int, [ctypes.POINTER(_vp), _i32, _vp]),
    ("dpsync_decompress_many", _int, [ctypes.POINTER(_vp), _i32, ctypes.POINTER(_vp), _f32, _vp]),
    ("dpsync_outer_step_many", _int, [ctypes.POINTER(_vp), _i32, ctypes.POINTER(_vp), _f32, _vp]),
    ("dpsync_get_state", _int, [_vp, _vp, _vp, _vp, _vp, _vp]),
]

_lib = None


def load(path: str):
    """Loads a build of the library from `path` with the C-ABI's signatures set
    (lib() uses it for the library itself; tests use it for the checked build)."""
    if not os.path.exists(path):
        raise ImportError("libspecoptim.so is not built (%s); run "
                          "spectral_corrected_optimizer_gb300.build.build()" % path)
    handle = ctypes.CDLL(path)
    for name, res, args in SIGNATURES:
        f = getattr(handle, name)
        f.restype = res
        f.argtypes = args
    return handle


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        _lib = load(LIB_PATH)
    return _lib


def _check(rc: int, what: str):
    if rc != OK:
        raise SpecOptimError(rc, what, lib().specoptim_last_error().decode(errors="replace"))


def _torch():
    import torch
    return torch


def _stream(stream=None) -> int:
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _f32_2d(t, shape, name):
    torch = _torch()
    if t.dtype != torch.float32 or tuple(t.shape) != tuple(shape):
        raise ValueError("%s must be float32 of shape %s, got %s %s" % (name, shape, t.dtype, tuple(t.shape)))
    return _ptr(t)


def config_default(m: int, n: int, **overrides) -> Config:
    cfg = Config()
    _check(lib().specoptim_config_default(ctypes.byref(cfg), m, n), "specoptim_config_default")
    for k, v in overrides.items():
        if not hasattr(cfg, k):
            raise KeyError(k)
        setattr(cfg, k, v)
    return cfg


class SpectralOptimizer:
    """Spectral-corrected optimizer state of one m x n weight (key designs 2-3)."""

    def __init__(self, m: int, n: int, stream=None, **overrides):
        self.m, self.n, self.r = m, n, min(m, n)
        self.cfg = config_default(m, n, **overrides)
        h = ctypes.c_void_p()
        _check(lib().specoptim_create(ctypes.byref(h), ctypes.byref(self.cfg), _stream(stream)),
               "specoptim_create")
        self._h = h

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            lib().specoptim_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def anchor_update(self, G_anc, stream=None):
        _check(lib().specoptim_anchor_update(self._h, _f32_2d(G_anc, (self.m, self.n), "G_anc"),
                                             _stream(stream)), "specoptim_anchor_update")

    def svd_refresh(self, stream=None) -> int:
        sweeps = ctypes.c_int32(0)
        _check(lib().specoptim_svd_refresh(self._h, _stream(stream), ctypes.byref(sweeps)),
               "specoptim_svd_refresh")
        return sweeps.value

    def step(self, W, G_mask, lr: float, G_filt_out=None, G_proj_out=None, stream=None):
        shape = (self.m, self.n)
        _check(lib().specoptim_step(self._h, _f32_2d(W, shape, "W"), _f32_2d(G_mask, shape, "G_mask"),
                                    float(lr), _stream(stream),
                                    None if G_filt_out is None else _f32_2d(G_filt_out, shape, "G_filt_out"),
                                    None if G_proj_out is None else _f32_2d(G_proj_out, shape, "G_proj_out")),
               "specoptim_step")

    def get_factors(self, stream=None):
        torch = _torch()
        dev = torch.device("cuda", torch.cuda.current_device())
        U = torch.empty((self.m, self.r), device=dev)
        s = torch.empty((self.r,), device=dev)
        V = torch.empty((self.n, self.r), device=dev)
        d = torch.empty((self.r,), device=dev)
        _check(lib().specoptim_get_factors(self._h, _ptr(U), _ptr(s), _ptr(V), _ptr(d), _stream(stream)),
               "specoptim_get_factors")
        return U, s, V, d

    def get_state(self, stream=None):
        torch = _torch()
        dev = torch.device("cuda", torch.cuda.current_device())
        M, m1, m2 = (torch.empty((self.m, self.n), device=dev) for _ in range(3))
        t = ctypes.c_int64(0)
        _check(lib().specoptim_get_state(self._h, _ptr(M), _ptr(m1), _ptr(m2), ctypes.byref(t),
                                         _stream(stream)), "specoptim_get_state")
        return M, m1, m2, t.value

    def set_state(self, M, exp_avg, exp_avg_sq, t: int, stream=None):
        shape = (self.m, self.n)
        _check(lib().specoptim_set_state(self._h, _f32_2d(M, shape, "M"), _f32_2d(exp_avg, shape, "exp_avg"),
                                         _f32_2d(exp_avg_sq, shape, "exp_avg_sq"), int(t), _stream(stream)),
               "specoptim_set_state")


def svd_refresh_many(optimizers, stream=None):
    """One batched SVD refresh of several SpectralOptimizer handles (at most 16)."""
    n = len(optimizers)
    arr = (ctypes.c_void_p * n)(*[o._h.value for o in optimizers])
    sweeps = (ctypes.c_int32 * n)()
    _check(lib().specoptim_svd_refresh_many(arr, n, _stream(stream), sweeps), "specoptim_svd_refresh_many")
    return list(sweeps)


def svd_refresh_begin(optimizers, stream=None):
    """Starts a batched SVD refresh that runs beside later work (returns at once);
    steps enqueued before svd_refresh_end use the previous factors."""
    n = len(optimizers)
    arr = (ctypes.c_void_p * n)(*[o._h.value for o in optimizers])
    _check(lib().specoptim_svd_refresh_begin(arr, n, _stream(stream)), "specoptim_svd_refresh_begin")


def svd_refresh_end(optimizers, stream=None):
    """Completes the refresh begun on the same optimizers (same order); returns the sweeps."""
    n = len(optimizers)
    arr = (ctypes.c_void_p * n)(*[o._h.value for o in optimizers])
    sweeps = (ctypes.c_int32 * n)()
    _check(lib().specoptim_svd_refresh_end(arr, n, _stream(stream), sweeps), "specoptim_svd_refresh_end")
    return list(sweeps)


def step_many(optimizers, Ws, Gs, lr: float, stream=None):
    """One spectral-corrected step of several handles (at most 16) in shared launches."""
    n = len(optimizers)
    if len(Ws) != n or len(Gs) != n:
        raise ValueError("step_many: one W and one G_mask per optimizer")
    hs = (ctypes.c_void_p * n)(*[o._h.value for o in optimizers])
    wp = (ctypes.c_void_p * n)(*[_f32_2d(w, (o.m, o.n), "W") for o, w in zip(optimizers, Ws)])
    gp = (ctypes.c_void_p * n)(*[_f32_2d(g, (o.m, o.n), "G_mask") for o, g in zip(optimizers, Gs)])
    _check(lib().specoptim_step_many(hs, n, wp, gp, float(lr), _stream(stream)), "specoptim_step_many")


def adamw(W, g, exp_avg, exp_avg_sq, t: int, lr: float, beta1=0.9, beta2=0.999, eps=1e-8,
          weight_decay=0.01, stream=None):
    """Plain AdamW in place on fp32 CUDA tensors of equal size."""
    n = W.numel()
    for x, name in ((g, "g"), (exp_avg, "exp_avg"), (exp_avg_sq, "exp_avg_sq")):
        if x.numel() != n:
            raise ValueError("%s has %d elements, W has %d" % (name, x.numel(), n))
    _check(lib().specoptim_adamw(_ptr(W), _ptr(g), _ptr(exp_avg), _ptr(exp_avg_sq), n, int(t), lr,
                                 beta1, beta2, eps, weight_decay, _stream(stream)), "specoptim_adamw")


def gemm_nt(A, B, precision: int = PREC_TF32, out=None, stream=None):
    """C = A @ B.T for fp32 CUDA matrices A (M x K), B (N x K)."""
    torch = _torch()
    M, K = A.shape
    N, K2 = B.shape
    if K != K2 or A.dtype != torch.float32 or B.dtype != torch.float32:
        raise ValueError("gemm_nt: A (M x K) and B (N x K) must be float32 with equal K")
    if out is None:
        out = torch.empty((M, N), device=A.device)
    _check(lib().specoptim_gemm_nt(M, N, K, _ptr(A), K, _ptr(B), K, _ptr(out), N, precision,
                                   _stream(stream)), "specoptim_gemm_nt")
    return out


def check_device(stream=None):
    """Synchronise the stream; raise if a bounded device-side wait of the library gave up."""
    _check(lib().specoptim_check_device(_stream(stream)), "specoptim_check_device")


def trace_enable(on: bool = True):
    _check(lib().specoptim_trace_enable(1 if on else 0), "specoptim_trace_enable")


def launch_count() -> int:
    return int(lib().specoptim_launch_count())


def trace_reset():
    _check(lib().specoptim_trace_reset(), "specoptim_trace_reset")


def trace_report() -> dict:
    """{kernel name: (launches, total device ms)} of the traced launches."""
    buf = ctypes.create_string_buffer(1 << 16)
    _check(lib().specoptim_trace_report(buf, len(buf)), "specoptim_trace_report")
    out = {}
    for line in buf.value.decode().splitlines():
        name, n, ms = line.split()
        out[name] = (int(n), float(ms))
    return out


# ---------------------------------------------------------------- activation mask

def mask_keep_count(p: float, H: int) -> int:
    return int(lib().mask_keep_count(float(p), int(H)))


def _elem_bytes(t) -> int:
    if t.element_size() not in (2, 4):
        raise ValueError("mask tensors must have 2- or 4-byte elements, got %s" % t.dtype)
    return t.element_size()


def mask_pack(dense, K: int, layer: int, step: int, batch_id: int = 0, out=None, stream=None):
    """packed[r, k] = dense[r, pi_r(k)] for a CUDA tensor dense [rows, H]."""
    torch = _torch()
    rows, H = dense.shape
    if out is None:
        out = torch.empty((rows, K), dtype=dense.dtype, device=dense.device)
    elif tuple(out.shape) != (rows, K) or out.dtype != dense.dtype:
        raise ValueError("out must be %s of shape (%d, %d)" % (dense.dtype, rows, K))
    _check(lib().mask_pack(_ptr(dense), _ptr(out), rows, H, K, _elem_bytes(dense), layer, step, batch_id,
                           _stream(stream)), "mask_pack")
    return out


def mask_unpack(packed, H: int, layer: int, step: int, batch_id: int = 0, out=None, stream=None):
    """dense[r, pi_r(k)] = packed[r, k], +0 elsewhere, for a CUDA tensor packed [rows, K]."""
    torch = _torch()
    rows, K = packed.shape
    if out is None:
        out = torch.empty((rows, H), dtype=packed.dtype, device=packed.device)
    elif tuple(out.shape) != (rows, H) or out.dtype != packed.dtype:
        raise ValueError("out must be %s of shape (%d, %d)" % (packed.dtype, rows, H))
    _check(lib().mask_unpack(_ptr(packed), _ptr(out), rows, H, K, _elem_bytes(packed), layer, step,
                             batch_id, _stream(stream)), "mask_unpack")
    return out


def mask_indices(rows: int, H: int, K: int, layer: int, step: int, batch_id: int = 0, device=None,
                 stream=None):
    torch = _torch()
    out = torch.empty((rows, K), dtype=torch.int32, device=device or "cuda")
    _check(lib().mask_indices(_ptr(out), rows, H, K, layer, step, batch_id, _stream(stream)),
           "mask_indices")
    return out


# ---------------------------------------------------------------- mask fused with the layer boundary

def _bf16(t, shape, name):
    torch = _torch()
    if t.dtype != torch.bfloat16 or tuple(t.shape) != tuple(shape):
        raise ValueError("%s must be bfloat16 of shape %s, got %s %s" % (name, shape, t.dtype, tuple(t.shape)))
    return _ptr(t)


def mask_pack_add(a, b, K: int, layer: int, step: int, batch_id: int = 0, out=None, stream=None):
    """packed = pack(a + b) for bf16 CUDA tensors a, b [rows, H] (the sum is formed at the kept dims only)."""
    torch = _torch()
    rows, H = a.shape
    if out is None:
        out = torch.empty((rows, K), dtype=torch.bfloat16, device=a.device)
    _check(lib().mask_pack_add(_bf16(a, (rows, H), "a"), _bf16(b, (rows, H), "b"), _bf16(out, (rows, K), "out"),
                               rows, H, K, layer, step, batch_id, _stream(stream)), "mask_pack_add")
    return out


def mask_unpack_rmsnorm(packed, gamma, eps: float, H: int, layer: int, step: int, batch_id: int = 0,
                        h_out=None, x_out=None, stream=None):
    """(h~, x): h~ = unpack(packed), x = RMSNorm(h~) * gamma, bf16 [rows, H] each."""
    torch = _torch()
    rows, K = packed.shape
    if h_out is None:
        h_out = torch.empty((rows, H), dtype=torch.bfloat16, device=packed.device)
    if x_out is None:
        x_out = torch.empty((rows, H), dtype=torch.bfloat16, device=packed.device)
    _check(lib().mask_unpack_rmsnorm(_bf16(packed, (rows, K), "packed"), _bf16(gamma, (H,), "gamma"), float(eps),
                                     _bf16(h_out, (rows, H), "h_out"), _bf16(x_out, (rows, H), "x_out"), rows, H, K,
                                     layer, step, batch_id, _stream(stream)), "mask_unpack_rmsnorm")
    return h_out, x_out


def mask_rmsnorm_backward_pack(packed_h, gamma, eps: float, dx, g_res, layer: int, step: int, batch_id: int = 0,
                               out=None, stream=None):
    """Packed dL/dh~ (bf16 [rows, K]) from the packed h~, gamma, dx [rows, H] and g_res [rows, H] or None."""
    torch = _torch()
    rows, K = packed_h.shape
    H = gamma.shape[0]
    if out is None:
        out = torch.empty((rows, K), dtype=torch.bfloat16, device=packed_h.device)
    _check(lib().mask_rmsnorm_backward_pack(_bf16(packed_h, (rows, K), "packed_h"), _bf16(gamma, (H,), "gamma"),
                                            float(eps), _bf16(dx, (rows, H), "dx"),
                                            None if g_res is None else _bf16(g_res, (rows, H), "g_res"),
                                            _bf16(out, (rows, K), "out"), rows, H, K, layer, step, batch_id,
                                            _stream(stream)), "mask_rmsnorm_backward_pack")
    return out


def mask_unpack_add(packed, g, layer: int, step: int, batch_id: int = 0, stream=None):
    """g[r, pi_r(k)] += packed[r, k] in place (bf16), other entries unchanged."""
    rows, K = packed.shape
    H = g.shape[1]
    _check(lib().mask_unpack_add(_bf16(packed, (rows, K), "packed"), _bf16(g, (rows, H), "g"), rows, H, K,
                                 layer, step, batch_id, _stream(stream)), "mask_unpack_add")
    return g
