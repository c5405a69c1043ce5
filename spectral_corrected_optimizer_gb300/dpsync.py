"""Binding of include/dpsync.h (argument marshalling only): the data-parallel
outer synchronisation of key design 4 of "Communication-Efficient LLM
Adaptation over Decentralized GPU Meshes" -- Streaming DiLoCo's outer step
travelling PowerSGD-compressed (one warm-started rank-k power step with
error feedback, k chosen for a 64x smaller message).

Every operation runs in the library's CUDA kernels.  What stays on the host is
the order of the calls and the two sums over workers (all-reduces of the
low-rank factors P and Q), which go through torch.distributed when a process
group with more than one rank is initialised.
"""
from __future__ import annotations

import ctypes

from . import DPConfig, _check, _f32_2d, _ptr, _stream, _torch, lib

MAX_BATCH = 16


def rank_for(m: int, n: int, ratio: float = 64.0) -> int:
    """k = floor(mn / (ratio (m + n)) + 1/2), clamped to [1, min(m, n)]."""
    return int(lib().dpsync_rank(int(m), int(n), float(ratio)))


def config_default(m: int, n: int, **overrides) -> DPConfig:
    cfg = DPConfig()
    _check(lib().dpsync_config_default(ctypes.byref(cfg), m, n), "dpsync_config_default")
    for k, v in overrides.items():
        if not hasattr(cfg, k):
            raise KeyError(k)
        setattr(cfg, k, v)
    return cfg


def default_allreduce(group=None):
    """Sum over the workers of `group` in place (nothing for one worker)."""
    torch = _torch()
    dist = torch.distributed
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size(group) == 1:
        return lambda t: None
    return lambda t: dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)


def sync_protocol(ops, allreduce, workers: int, X, Y, finish, outer: bool):
    """The order of one synchronisation: compress_p, sum P over the workers,
    orthogonalize, compress_q, sum Q over the workers, then decompress (or the
    outer step) with q_scale = 1 / workers.  `ops` provides the five calls and
    the flat P and Q buffers (P_flat, Q_flat)."""
    ops.compress_p(X, Y)
    allreduce(ops.P_flat)
    ops.orthogonalize()
    ops.compress_q()
    allreduce(ops.Q_flat)
    if outer:
        ops.outer_step(finish, 1.0 / workers)
    else:
        ops.decompress(finish, 1.0 / workers)


class DPSyncGroup:
    """Synchronisation state of several weight matrices (e.g. one decoder
    layer).  P and Q of all matrices live in two flat fp32 buffers, so each sum
    over workers is one all-reduce; the kernels run once per call for up to 16
    matrices.

    shapes: list of (m, n).  ranks: optional list of k per matrix (0 or absent:
    the 64x rule).  Q0: optional list of starting Q (n x k) tensors, the same on
    every worker; by default N(0, 1) values from a CPU generator seeded with
    `seed`.  Other keyword arguments set dpsync_config fields of every matrix."""

    def __init__(self, shapes, Q0=None, seed: int = 0, stream=None, ranks=None, **overrides):
        torch = _torch()
        self.shapes = [(int(m), int(n)) for m, n in shapes]
        self.cfgs = [config_default(m, n, **overrides) for m, n in self.shapes]
        for cfg, k in zip(self.cfgs, ranks or []):
            cfg.rank = int(k)
        self.ranks = [c.rank if c.rank > 0 else rank_for(c.m, c.n, c.ratio) for c in self.cfgs]
        dev = torch.device("cuda", torch.cuda.current_device())
        self.P_flat = torch.zeros(sum(m * k for (m, _), k in zip(self.shapes, self.ranks)), device=dev)
        self.Q_flat = torch.zeros(sum(n * k for (_, n), k in zip(self.shapes, self.ranks)), device=dev)
        self.P, self.Q = [], []
        po = qo = 0
        for (m, n), k in zip(self.shapes, self.ranks):
            self.P.append(self.P_flat[po:po + m * k].view(m, k))
            self.Q.append(self.Q_flat[qo:qo + n * k].view(n, k))
            po += m * k
            qo += n * k
        gen = torch.Generator().manual_seed(seed)
        for i, ((m, n), k) in enumerate(zip(self.shapes, self.ranks)):
            q = Q0[i] if Q0 is not None else torch.randn(n, k, generator=gen, dtype=torch.float32)
            self.Q[i].copy_(q.reshape(n, k))
        self._h = []
        for cfg, P, Q in zip(self.cfgs, self.P, self.Q):
            h = ctypes.c_void_p()
            _check(lib().dpsync_create(ctypes.byref(h), ctypes.byref(cfg), _ptr(P), _ptr(Q),
                                       _stream(stream)), "dpsync_create")
            self._h.append(h)

    def close(self):
        for h in getattr(self, "_h", []):
            if h is not None and h.value:
                lib().dpsync_destroy(h)
        self._h = []

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __len__(self):
        return len(self.shapes)

    # -- the five calls, chunked by 16 matrices --------------------------------
    def _chunks(self):
        for s in range(0, len(self._h), MAX_BATCH):
            idx = list(range(s, min(len(self._h), s + MAX_BATCH)))
            yield idx, (ctypes.c_void_p * len(idx))(*[self._h[i].value for i in idx])

    def _mats(self, idx, ts, name, allow_none):
        if ts is None:
            if not allow_none:
                raise ValueError("%s: one tensor per matrix is required" % name)
            return None
        return (ctypes.c_void_p * len(idx))(*[
            None if ts[i] is None else _f32_2d(ts[i], self.shapes[i], name) for i in idx])

    def set_outer(self, Ws, stream=None):
        """theta <- W and outer momentum <- 0 for every matrix."""
        for i, W in enumerate(Ws):
            _check(lib().dpsync_set_outer(self._h[i], _f32_2d(W, self.shapes[i], "W"), _stream(stream)),
                   "dpsync_set_outer")
        self._outer = True

    def compress_p(self, X=None, Y=None, stream=None):
        """M = E + X - Y (X None: the outer weights theta); P = M Q."""
        for idx, hs in self._chunks():
            _check(lib().dpsync_compress_p_many(hs, len(idx), self._mats(idx, X, "X", True),
                                                self._mats(idx, Y, "Y", True), _stream(stream)),
                   "dpsync_compress_p_many")

    def orthogonalize(self, stream=None):
        for idx, hs in self._chunks():
            _check(lib().dpsync_orthogonalize_many(hs, len(idx), _stream(stream)), "dpsync_orthogonalize_many")

    def compress_q(self, stream=None):
        for idx, hs in self._chunks():
            _check(lib().dpsync_compress_q_many(hs, len(idx), _stream(stream)), "dpsync_compress_q_many")

    def decompress(self, outs=None, q_scale: float = 1.0, stream=None):
        """D = q_scale P^ Q^T into outs (list of m x n tensors or None); E <- M - D."""
        for idx, hs in self._chunks():
            _check(lib().dpsync_decompress_many(hs, len(idx), self._mats(idx, outs, "out", True),
                                                float(q_scale), _stream(stream)), "dpsync_decompress_many")

    def outer_step(self, W_locals, q_scale: float = 1.0, stream=None):
        """D as in decompress, the outer Nesterov step and the restart of W_local."""
        for idx, hs in self._chunks():
            _check(lib().dpsync_outer_step_many(hs, len(idx), self._mats(idx, W_locals, "W_local", False),
                                                float(q_scale), _stream(stream)), "dpsync_outer_step_many")

    # -- whole synchronisations -------------------------------------------------
    def sync_grad(self, Gs, outs, allreduce=None, workers: int | None = None):
        """PowerSGD on gradients: outs <- the decompressed mean of the workers' Gs."""
        ar, w = self._group(allreduce, workers)
        sync_protocol(self, ar, w, Gs, None, outs, outer=False)

    def outer_sync(self, W_locals, allreduce=None, workers: int | None = None):
        """One outer synchronisation: pseudo-gradient theta - W_local, compressed,
        summed, outer Nesterov step; W_locals restart from the new theta."""
        ar, w = self._group(allreduce, workers)
        sync_protocol(self, ar, w, None, W_locals, W_locals, outer=True)

    @staticmethod
    def _group(allreduce, workers):
        torch = _torch()
        dist = torch.distributed
        if workers is None:
            workers = dist.get_world_size() if dist.is_available() and dist.is_initialized() else 1
        return (allreduce if allreduce is not None else default_allreduce()), workers

    def get_state(self, i: int, stream=None):
        """(E, theta or None, momentum or None, P^) of matrix i as new tensors."""
        torch = _torch()
        m, n = self.shapes[i]
        dev = self.P_flat.device
        E = torch.empty((m, n), device=dev)
        Ph = torch.empty((m, self.ranks[i]), device=dev)
        outer = getattr(self, "_outer", False)
        th = torch.empty((m, n), device=dev) if outer else None
        mo = torch.empty((m, n), device=dev) if outer else None
        _check(lib().dpsync_get_state(self._h[i], _ptr(E), _ptr(th), _ptr(mo), _ptr(Ph), _stream(stream)),
               "dpsync_get_state")
        return E, th, mo, Ph
