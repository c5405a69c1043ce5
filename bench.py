"""Benchmark of the spectral-corrected optimizer + activation-mask hot path.

Method: "Communication-Efficient LLM Adaptation over Decentralized GPU Meshes"
(arXiv 2609.14339): key design 1 (in-graph activation mask, pack / unpack at
pipeline-stage boundaries, backward with the same indices), key design 2
(anchor EMA) and key design 3 (SVD of the anchor momentum, Tikhonov filter,
two-sided projection, blend, AdamW).

Workload (one bench "step" = one pass of the whole hot path):
  * one Llama-3.2-1B decoder layer, 7 fp32 weights (q, o 2048x2048; k, v
    512x2048; gate, up 8192x2048; down 2048x8192), rank-32 anchor signal +
    N(0,1e-4) noise, masked gradients with fresh N(0,1e-2) noise;
  * every step: the spectral-corrected step of all 7 matrices, and the
    stage-boundary mask round trip of a bf16 [32*2048, 2048] activation at
    p = 0.95 (forward pack, receiver unpack, backward pack of the bf16
    activation gradient, sender unpack);
  * every 20th step (the anchor delay of the pages): anchor EMA + SVD refresh
    of the 7 matrices.
value = steps/s of the whole job.  Separate timed loops give the steady step
(no refresh), the refresh, and the activation-mask sweep (15 boundaries x
{pack, unpack, backward pack, backward unpack} at p = 0.90 and 0.95) in GB/s.

With torchrun (N > 1) every rank runs its own replica of the layer (the
optimizer state of different matrices is independent; no data-path
collective): weak scaling, time = max over ranks.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "Llama-3.2-1B-shaped spectral-corrected steps/s; mask pack/unpack HBM GB/s"
REFRESH_EVERY = 20
# Overlapped schedule (measured in the breakdown): steps between an anchor's
# arrival (its EMA and the start of its SVD refresh, which then runs beside the
# steps on the library's own streams) and the first step that filters with its
# factors (the end of the refresh).  The headline runs the refresh in one call
# at the anchor's arrival (use_after = 0), which measured faster on one GPU: the
# persistent step GEMMs and the Jacobi kernels each fill every SM, so running
# them side by side gains nothing and costs the interleaving.
REFRESH_USE_AFTER = 10
MASK_ROWS, MASK_H, MASK_P = 32 * 2048, 2048, 0.95
MASK_BOUNDARIES = 15
POOL = 4               # distinct masked-gradient sets kept resident in HBM

WORKLOAD = ("llama-3.2-1b decoder layer (q,o 2048x2048; k,v 512x2048; gate,up 8192x2048; "
            "down 2048x8192), rank-32 anchor signal, SVD refresh every 20 steps, "
            "mask round trip bf16 [65536,2048] p=0.95 per step")


def env_int(name, default):
    try:
        return int(os.environ.get(name, default))
    except ValueError:
        return default


def strip_comments(text: str) -> str:
    """C/C++/CUDA source without its comments (string and character literals kept)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c in "\"'":
            j = i + 1
            while j < n and text[j] != c:
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return "".join(out)


def code_digest(sources) -> str:
    """First 16 hex digits of the sha256 of the kernel sources' code: comments and
    runs of blank space removed, so that a comment edit keeps a profile valid."""
    import hashlib
    csrc = os.path.join(ROOT, "spectral_corrected_optimizer_gb300", "csrc")
    h = hashlib.sha256()
    for name in sources:
        with open(os.path.join(csrc, name)) as f:
            h.update(" ".join(strip_comments(f.read()).split()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(profile: str, sources, key: str = ""):
    """DRAM bytes per launch from a committed ncu summary under profiles/, or None
    when the code of one of the kernel's sources changed since the counters were
    taken (`key`: the kernel name in front of the figure, for summaries of several
    kernels)."""
    import re
    try:
        with open(os.path.join(ROOT, "profiles", profile)) as f:
            text = f.read()
    except OSError:
        return None
    m = re.search((re.escape(key) + " " if key else "") +
                  r"traffic_bytes_per_launch=([0-9.e+]+) code_sha256_16=([0-9a-f]+)", text)
    if not m or m.group(2) != code_digest(sources):
        return None
    return float(m.group(1))


GEMM_PROFILE = ("gemm_tf32_layer_step.md", ("gemm_tc.cu", "gemm.cuh", "tc.cuh", "specoptim.cu"))
ROTATE_PROFILE = ("jacobi_rotate_layer_refresh.md", ("jacobi_tc.cu", "jacobi.cuh", "tc.cuh"))
APPLY_PROFILE = ("jacobi_apply_layer_refresh.md", ("jacobi_apply_tc.cu", "jacobi.cuh", "tc.cuh"))
DPSYNC_PROFILE = ("dpsync_layer_outer_sync.md", ("dpsync.cu", "tc.cuh", "common.cuh"))
ELEMENTWISE_PROFILE = ("elementwise_ema_adamw.md", ("elementwise.cu", "elementwise.cuh", "common.cuh"))
# values per launch of the profiled elementwise case (bench.py --profile elementwise)
ELEMENTWISE_PROFILE_VALUES = {"ema": 8192 * 2048, "adamw": 32768 * 2048}


def padded_order(r: int) -> int:
    return (r + 127) // 128 * 128


def rotate_bytes(Np: int) -> float:
    """Algorithmic bytes of Q <- Q R for one matrix and round: Q (Np x Np fp32)
    read and written once, and its Np/64 rotations (R^T hi and lo) read once."""
    return 8.0 * Np * Np + 512.0 * Np


def apply_bytes(Np: int) -> float:
    """Algorithmic bytes of A <- R^T A R for one matrix and round: the upper
    128 x 128 super-tiles of A read once, all of A written once, the rotations
    read once."""
    ns = Np // 128
    return ns * (ns + 1) / 2 * 128 * 128 * 4 + 4.0 * Np * Np + 512.0 * Np


def read_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def measure_tf32_peak(torch) -> dict:
    """The TF32 tensor-core peak measured the way the HBM and bf16 peaks of
    MEASURED_PEAKS.json are: torch.matmul (cuBLAS) fp32 8192^3 with TF32
    allowed, 2 N^3 flops; best of 10 (burst) and back to back for about 3 s
    (sustained, under the power cap)."""
    n = 8192
    prev = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = True
    try:
        g = torch.Generator(device="cuda").manual_seed(0)
        a = torch.randn(n, n, device="cuda", generator=g)
        b = torch.randn(n, n, device="cuda", generator=g)
        c = torch.empty(n, n, device="cuda")
        for _ in range(3):
            torch.matmul(a, b, out=c)
        best = min(timed(torch, lambda: torch.matmul(a, b, out=c), False) for _ in range(10))
        reps = max(10, int(3000.0 / best))
        sus = timed(torch, lambda: [torch.matmul(a, b, out=c) for _ in range(reps)], False) / reps
        del a, b, c
    finally:
        torch.backends.cuda.matmul.allow_tf32 = prev
    f = 2.0 * n ** 3
    return {"tf32_tflops": f / (best * 1e-3) / 1e12, "tf32_tflops_sustained": f / (sus * 1e-3) / 1e12,
            "how": "torch.matmul fp32 8192^3 with allow_tf32 (cuBLAS), 2 N^3 flops: best of 10 (burst) and "
                   "%d back to back (sustained), CUDA events" % reps}


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------ the layer on the GPU

def gemm_flops(m: int, n: int) -> float:
    """Algorithmic flops of one matrix's step in the executed association
    (2 sum(M N K) of its GEMMs): P_R G^T and P_L T for m = n; U^T G, P_R T1^T D,
    U T2 for m > n; V^T G^T, P_L T1 D, T2 V^T for m < n."""
    if m == n:
        return 4.0 * n ** 3
    if m > n:
        return 4.0 * m * n * n + 2.0 * n ** 3
    return 4.0 * m * m * n + 2.0 * m ** 3


def step_bytes(m: int, n: int) -> float:
    """Algorithmic HBM bytes of one matrix's step in the executed association:
    the fused epilogue's G read and W, m, v read + write (28 B per element), every
    GEMM operand read once, every intermediate written and read once, and G^T
    written and read for m > n."""
    mn = m * n
    if m == n:
        return 28.0 * mn + 4.0 * (m * m + n * n) + 4.0 * mn + 8.0 * mn
    if m > n:
        r = n
        return 28.0 * mn + 8.0 * mn + 4.0 * mn + 8.0 * m * r + 4.0 * n * n + 16.0 * n * r
    r = m
    return 28.0 * mn + 4.0 * mn + 8.0 * n * r + 4.0 * m * m + 16.0 * m * r


class Layer:
    def __init__(self, seed: int):
        import numpy as np
        import torch
        import spectral_corrected_optimizer_gb300 as so
        import synthetic

        self.so, self.torch = so, torch
        self.names = list(synthetic.LLAMA_1B_LAYER)
        self.inputs = synthetic.layer_inputs(synthetic.LLAMA_1B_LAYER, seed=seed, rank=32)
        self.opt, self.W, self.Ganc, self.Gpool = {}, {}, {}, {}
        for name, inp in self.inputs.items():
            self.opt[name] = so.SpectralOptimizer(inp.m, inp.n)
            self.W[name] = torch.from_numpy(inp.weights()).cuda()
            self.Ganc[name] = [torch.from_numpy(inp.anchor_grad(i)).cuda() for i in range(2)]
            self.Gpool[name] = [torch.from_numpy(inp.masked_grad(t)).cuda() for t in range(POOL)]
        self.K = so.mask_keep_count(MASK_P, MASK_H)
        self.h = torch.from_numpy(synthetic.activations_bf16(MASK_ROWS, MASK_H, seed=seed).view(np.int16)).view(
            torch.bfloat16).cuda()
        self.g = torch.from_numpy(synthetic.act_grads_bf16(MASK_ROWS, MASK_H, seed=seed).view(np.int16)).view(
            torch.bfloat16).cuda()
        self.hp = torch.empty(MASK_ROWS, self.K, dtype=torch.bfloat16, device="cuda")
        self.gp = torch.empty_like(self.hp)
        self.hd = torch.empty_like(self.h)
        self.gd = torch.empty_like(self.g)
        self.lr = 2e-5
        self.last_sweeps = None
        self.pending = False
        self.use_after = 0
        self.flops = sum(gemm_flops(i.m, i.n) for i in self.inputs.values())
        self.bytes = sum(step_bytes(i.m, i.n) for i in self.inputs.values())
        self.params = sum(i.m * i.n for i in self.inputs.values())

    def reset_state(self):
        """Fresh optimizer state and the initial weights: a loop run after this
        one replays the same refresh history (the Jacobi sweep count of a warm-
        started refresh depends on how many refreshes came before it)."""
        self.refresh_end()
        for name, inp in self.inputs.items():
            self.opt[name].close()
            self.opt[name] = self.so.SpectralOptimizer(inp.m, inp.n)
            self.W[name].copy_(self.torch.from_numpy(inp.weights()))

    def refresh(self, idx: int, G=None):
        """Anchor EMA + batched SVD refresh of the 7 matrices in one call; returns
        the Jacobi sweeps each one took."""
        for name in self.names:
            self.opt[name].anchor_update(G[name] if G else self.Ganc[name][idx % 2])
        self.last_sweeps = self.so.svd_refresh_many([self.opt[name] for name in self.names])
        return self.last_sweeps

    def refresh_begin(self, idx: int, G=None):
        """Anchor EMA, then the start of the batched SVD refresh: its Jacobi
        sweeps run beside the following steps, which keep the previous factors."""
        for name in self.names:
            self.opt[name].anchor_update(G[name] if G else self.Ganc[name][idx % 2])
        self.so.svd_refresh_begin([self.opt[name] for name in self.names])
        self.pending = True

    def refresh_end(self):
        """The refresh's factors take effect for the steps enqueued from here on."""
        if self.pending:
            self.last_sweeps = self.so.svd_refresh_end([self.opt[name] for name in self.names])
            self.pending = False

    def schedule(self, i: int, t0: int):
        """What step i does about the anchor, for a run whose timed steps start at
        t0: before t0 (warm-up) a one-call refresh every REFRESH_EVERY steps;
        from t0 on an anchor arrives every REFRESH_EVERY steps (the first at t0)
        and is refreshed in one call (use_after = 0) or begun there and ended
        use_after steps later."""
        if i < t0:
            return "refresh" if i % REFRESH_EVERY == 0 else None
        k = (i - t0) % REFRESH_EVERY
        if self.use_after == 0:
            return "refresh" if k == 0 else None
        return "begin" if k == 0 else ("end" if k == self.use_after else None)

    def spectral(self, i: int, G=None):
        self.so.step_many([self.opt[n] for n in self.names], [self.W[n] for n in self.names],
                          [G[n] if G else self.Gpool[n][i % POOL] for n in self.names], self.lr)

    def mask_round_trip(self, i: int, hp_out=None, gp_out=None, hp_in=None, gp_in=None):
        """Pack the boundary activation and its gradient, and unpack the packed
        values of the neighbouring stages.  On one device the unpack reads the
        values this step packed; a loop that exchanges them over a link passes
        the received ones (hp_in, gp_in) and its own send buffers."""
        so, layer = self.so, i % MASK_BOUNDARIES
        hp = self.hp if hp_out is None else hp_out
        gp = self.gp if gp_out is None else gp_out
        so.mask_pack(self.h, self.K, layer, i, 0, out=hp)
        so.mask_unpack(hp if hp_in is None else hp_in, MASK_H, layer, i, 0, out=self.hd)
        so.mask_pack(self.g, self.K, layer, i, 0, out=gp)
        so.mask_unpack(gp if gp_in is None else gp_in, MASK_H, layer, i, 0, out=self.gd)

    @staticmethod
    def anchor_index(i: int, t0: int) -> int:
        """Which anchor gradient arrives at step i (two alternate)."""
        return (i // REFRESH_EVERY) if i < t0 else (i - t0) // REFRESH_EVERY + 1

    def step(self, i: int, t0: int = 0):
        what = self.schedule(i, t0)
        if what == "refresh":
            self.refresh(self.anchor_index(i, t0))
        elif what == "begin":
            self.refresh_end()
            self.refresh_begin(self.anchor_index(i, t0))
        elif what == "end":
            self.refresh_end()
        self.spectral(i)
        self.mask_round_trip(i)


class ModelWorkload:
    """`n_layers` decoder layers of the given shapes, each with its own optimizer
    state, fed with one layer's synthetic inputs (the values do not change the
    work; generating 16 distinct layers would take minutes of host time), plus
    plain-AdamW tensors (the full model's embedding and norm vectors)."""

    def __init__(self, shapes: dict, n_layers: int, seed: int, plain=(), tau_p: float = 1e-3):
        import numpy as np
        import torch

        import spectral_corrected_optimizer_gb300 as so
        import synthetic

        self.so, self.torch = so, torch
        self.names = list(shapes)
        inputs = synthetic.layer_inputs(shapes, seed=seed, rank=32)
        self.Ganc = {n: [torch.from_numpy(inputs[n].anchor_grad(i)).cuda() for i in range(2)] for n in self.names}
        self.Gm = {n: [torch.from_numpy(inputs[n].masked_grad(t)).cuda() for t in range(2)] for n in self.names}
        W0 = {n: torch.from_numpy(inputs[n].weights()).cuda() for n in self.names}
        self.layers = [{n: so.SpectralOptimizer(*shapes[n], tau_p=tau_p) for n in self.names}
                       for _ in range(n_layers)]
        self.W = [{n: W0[n].clone() for n in self.names} for _ in range(n_layers)]
        self.plain = []
        for i, (rows, cols) in enumerate(plain):
            w = torch.from_numpy(synthetic.normal_f32(seed, 90, i, (rows, cols), 0.02)).cuda()
            g = torch.from_numpy(synthetic.normal_f32(seed, 91, i, (rows, cols), 1e-2)).cuda()
            self.plain.append((w, g, torch.zeros_like(w), torch.zeros_like(w)))
        self.t = 0
        self.flops = n_layers * sum(gemm_flops(*shapes[n]) for n in self.names)
        self.bytes = n_layers * sum(step_bytes(*shapes[n]) for n in self.names) + 28.0 * sum(r * c for r, c in plain)
        self.params = n_layers * sum(m * n for m, n in shapes.values()) + sum(r * c for r, c in plain)

    def refresh(self, idx: int):
        handles = []
        for layer in self.layers:
            for n in self.names:
                layer[n].anchor_update(self.Ganc[n][idx % 2])
                handles.append(layer[n])
        sweeps = []
        for i in range(0, len(handles), 14):  # two layers per batched refresh
            sweeps += self.so.svd_refresh_many(handles[i:i + 14])
        return sweeps

    def step(self, i: int):
        if i % REFRESH_EVERY == 0:
            self.refresh(i // REFRESH_EVERY)
        self.steady(i)

    def steady(self, i: int):
        """One step without the refresh: the spectral step of every matrix and
        the plain AdamW of the other tensors."""
        for layer, W in zip(self.layers, self.W):
            self.so.step_many([layer[n] for n in self.names], [W[n] for n in self.names],
                              [self.Gm[n][i % 2] for n in self.names], 2e-5)
        self.t += 1
        for w, g, m, v in self.plain:
            self.so.adamw(w, g, m, v, self.t, 2e-5)


def run_config(name: str, workload, K: int, W: int, mask_shape=None, peaks=None):
    """Whole-path steps/s of another configuration: W warm-up steps (the first holds
    the first refresh), then K timed steps holding one refresh; the steady step
    alone (no refresh) against its roofline max(F / P_tf32, B / BW) with F and B
    the executed association's flops and bytes; the refresh alone; and, where the
    configuration has one, its mask round trip."""
    torch = workload.torch
    for i in range(W):
        workload.step(i)
    torch.cuda.synchronize()
    ms = timed(torch, lambda: [workload.step(W + i) for i in range(K)], False)
    steady_n = 10
    steady_ms = timed(torch, lambda: [workload.steady(1000 + i) for i in range(steady_n)], False) / steady_n
    sweeps = []
    refresh_ms = timed(torch, lambda: sweeps.append(workload.refresh(7)), False)
    out = {"workload": name, "steps_per_s": K / (ms * 1e-3), "ms_per_step": ms / K, "steps": K, "warmup": W,
           "refreshes_in_timed_steps": sum(1 for i in range(W, W + K) if i % REFRESH_EVERY == 0),
           "refresh_ms": refresh_ms, "refresh_sweeps_max": max(sweeps[0]),
           "steady_step_ms": steady_ms, "steady_steps_per_s": 1e3 / steady_ms,
           "params": workload.params, "gemm_tflop_per_step": workload.flops / 1e12,
           "hbm_gb_per_step": workload.bytes / 1e9}
    if peaks is not None:
        bound = 1e3 * max(workload.flops / (peaks["tf32_tflops"] * 1e12), workload.bytes / (peaks["hbm_gbs"] * 1e9))
        out.update({"step_roofline_ms": bound, "step_frac": bound / steady_ms,
                    "step_roofline_peaks": "%.0f TFLOP/s tf32 (%s), %.0f GB/s HBM" % (
                        peaks["tf32_tflops"], peaks["tf32_source"], peaks["hbm_gbs"])})
    if mask_shape is not None:
        so = workload.so
        rows, H, p = mask_shape
        Kk = so.mask_keep_count(p, H)
        h = torch.randn(rows, H, device="cuda").to(torch.bfloat16)
        hp = torch.empty(rows, Kk, dtype=torch.bfloat16, device="cuda")
        hd = torch.empty_like(h)
        for _ in range(3):
            so.mask_pack(h, Kk, 0, 0, 0, out=hp)
            so.mask_unpack(hp, H, 0, 0, 0, out=hd)
        reps = 20
        t = timed(torch, lambda: [(so.mask_pack(h, Kk, b, 0, 0, out=hp), so.mask_unpack(hp, H, b, 0, 0, out=hd))
                                  for b in range(reps)], False)
        op_bytes = rows * (H + Kk) * 2
        out["mask"] = {"rows": rows, "H": H, "p": p, "K": Kk, "pack_unpack_GBps": 2 * reps * op_bytes / (t * 1e-3) / 1e9,
                       "timing": "eager, %d pack + unpack pairs" % reps}
    return out


def timed(torch, fn, dist_ok):
    """Device time of fn() with a barrier and a synchronize on both sides (ms)."""
    torch.cuda.synchronize()
    if dist_ok:
        import torch.distributed as dist
        dist.barrier()
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    fn()
    stop.record()
    torch.cuda.synchronize()
    if dist_ok:
        import torch.distributed as dist
        dist.barrier()
    return start.elapsed_time(stop)


def max_over_ranks(x: float, dist_ok: bool) -> float:
    if not dist_ok:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def mask_sweep(layer: Layer, p: float):
    """15 boundaries x {fwd pack, unpack, bwd pack, bwd unpack}; returns GB/s figures.

    The sweep is launch-bound from Python (60 launches of ~50 us), so it is timed
    as a CUDA-graph replay (headline) and eagerly (for reference), both without
    tracing; a separate traced eager pass gives the per-kernel averages."""
    so, torch = layer.so, layer.torch
    K = so.mask_keep_count(p, MASK_H)
    hp = torch.empty(MASK_ROWS, K, dtype=torch.bfloat16, device="cuda")
    gp = torch.empty_like(hp)

    def sweep():
        for b in range(MASK_BOUNDARIES):
            so.mask_pack(layer.h, K, b, 0, 0, out=hp)
            so.mask_unpack(hp, MASK_H, b, 0, 0, out=layer.hd)
            so.mask_pack(layer.g, K, b, 0, 0, out=gp)
            so.mask_unpack(gp, MASK_H, b, 0, 0, out=layer.gd)

    e = 2  # bf16
    dense, packed = MASK_ROWS * MASK_H * e, MASK_ROWS * K * e
    op_bytes = dense + packed  # pack: dense read + packed write; unpack: packed read + dense write
    sweep_bytes = 4 * MASK_BOUNDARIES * op_bytes
    sweep()  # warm-up
    eager_ms = timed(torch, sweep, False)
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        sweep()
        with torch.cuda.graph(graph, stream=side):
            sweep()
    torch.cuda.current_stream().wait_stream(side)
    graph.replay()
    graph_ms = timed(torch, graph.replay, False)
    so.trace_enable(True)
    sweep()
    rep = so.trace_report()
    so.trace_enable(False)
    out = {"K": K, "sweep_ms": graph_ms, "ops": 4 * MASK_BOUNDARIES,
           "effective_GBps": sweep_bytes / (graph_ms * 1e-3) / 1e9,
           "eager_sweep_ms": eager_ms, "eager_effective_GBps": sweep_bytes / (eager_ms * 1e-3) / 1e9,
           "timing": "CUDA-graph replay of the 60-launch sweep; eager figure without tracing beside it"}
    for kind in ("mask_pack_bulk", "mask_unpack_bulk"):
        if kind in rep:
            n, t = rep[kind]
            out[kind] = {"launches": n, "avg_us_traced": 1e3 * t / n, "GBps": n * op_bytes / (t * 1e-3) / 1e9}
    return out


def sector_coverage(H: int, K: int, elems: int = 16) -> float:
    """Expected fraction of a row's `elems`-element blocks (16 bf16 = one 32-byte
    sector, 64 bf16 = one 128-byte line) that hold at least one of K kept dims drawn
    without replacement from H."""
    miss = 1.0
    for i in range(elems):
        miss *= max(0.0, (H - K - i) / (H - i))
    return 1.0 - miss


def mask_fused_bench(peaks: dict, peak_src: str, p: float = 0.95, reps: int = 20) -> dict:
    """The mask ops fused with the layer boundary on the workload's bf16 [65536, 2048]
    boundary tensor: each op timed alone (CUDA events, `reps` launches, inputs larger
    than L2), its algorithmic bytes (sector coverage for the gathers at kept dims) and
    the unfused chain it replaces (plain mask ops + torch elementwise) for context."""
    import torch

    import spectral_corrected_optimizer_gb300 as so

    rows, H = MASK_ROWS, MASK_H
    K = so.mask_keep_count(p, H)
    g = torch.Generator(device="cuda").manual_seed(3)
    a = torch.randn(rows, H, device="cuda", generator=g).to(torch.bfloat16)
    b = torch.randn(rows, H, device="cuda", generator=g).to(torch.bfloat16)
    gamma = torch.randn(H, device="cuda", generator=g).to(torch.bfloat16)
    packed = so.mask_pack_add(a, b, K, 1, 0)
    h_out, x_out = torch.empty_like(a), torch.empty_like(a)
    pg = torch.empty_like(packed)
    gg = b.clone()
    # reads at the kept dims come from DRAM in whole 128-byte lines (ncu: the gathers'
    # DRAM reads equal the line coverage), writes of single elements in 32-byte sectors
    cov = sector_coverage(H, K, 64)
    wcov = sector_coverage(H, K, 16)
    dense, pk = rows * H * 2.0, rows * K * 2.0

    def t_ms(fn):
        fn()
        torch.cuda.synchronize()
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        for _ in range(reps):
            fn()
        e.record()
        torch.cuda.synchronize()
        return s.elapsed_time(e) / reps

    ops = {
        "pack_add": (lambda: so.mask_pack_add(a, b, K, 1, 0, out=packed), 2 * cov * dense + pk,
                     lambda: so.mask_pack(a + b, K, 1, 0, 0, out=packed)),
        "unpack_rmsnorm": (lambda: so.mask_unpack_rmsnorm(packed, gamma, 1e-5, H, 1, 0, h_out=h_out, x_out=x_out),
                           pk + 2 * dense,
                           lambda: torch.nn.functional.rms_norm(so.mask_unpack(packed, H, 1, 0, 0, out=h_out),
                                                                (H,), gamma, 1e-5)),
        "rmsnorm_backward_pack": (lambda: so.mask_rmsnorm_backward_pack(packed, gamma, 1e-5, a, b, 1, 0, out=pg),
                                  2 * cov * dense + 2 * pk, None),
        "unpack_add": (lambda: so.mask_unpack_add(packed, gg, 1, 0), pk + (cov + wcov) * dense,
                       lambda: gg.add_(so.mask_unpack(packed, H, 1, 0, 0, out=h_out))),
    }
    out = {"rows": rows, "H": H, "p": p, "K": K, "line_coverage": cov, "sector_coverage": wcov, "ops": {}}
    for name, (fn, byts, unfused) in ops.items():
        ms = t_ms(fn)
        ach = byts / (ms * 1e-3) / 1e9
        rec = {"ms": ms, "algorithmic_bytes": byts, "achieved_GBps": ach, "frac_of_hbm": ach / peaks["hbm_gbs"]}
        if unfused is not None:
            rec["unfused_ms"] = t_ms(unfused)
        out["ops"][name] = rec
    out["peak_source"] = "%s HBM copy bandwidth" % peak_src
    return out


def dp_sync_bytes(m: int, n: int, k: int) -> dict:
    """Algorithmic HBM bytes of one outer synchronisation of an m x n matrix at
    rank k, per kernel: compress_p reads theta, W_local and E and writes E
    (16 B per element) with P written and Q read once; compress_q reads M once
    and P^ once and writes Q; the outer step reads and writes E, theta and the
    momentum and writes W_local (28 B per element) with P^ and Q read once; the
    orthogonalisation reads P three times and writes P^."""
    lo = 4.0 * (m + n) * k
    return {"compress_p": 16.0 * m * n + lo, "compress_q": 4.0 * m * n + lo,
            "outer_step": 28.0 * m * n + lo, "orth": 16.0 * m * k}


def run_dp_sync(shapes, K: int, W: int, peaks: dict, peak_src: str, seed: int = 0) -> dict:
    """PowerSGD-compressed outer synchronisation (key design 4) of the matrices
    `shapes` on this GPU: W warm-up and K timed syncs, then one traced sync for
    the per-kernel split.  One worker per GPU (replicas: the sums over workers
    are the identity), 64x rank rule."""
    import torch

    import spectral_corrected_optimizer_gb300 as so
    import spectral_corrected_optimizer_gb300.dpsync as dp
    import synthetic

    Q0 = [torch.from_numpy(synthetic.dp_q0(n, dp.rank_for(m, n), seed=seed, index=i))
          for i, (m, n) in enumerate(shapes)]
    g = dp.DPSyncGroup(shapes, Q0=Q0)
    theta = [torch.from_numpy(synthetic.normal_f32(seed, 1, i, (m, n), 0.02)).cuda() for i, (m, n) in enumerate(shapes)]
    g.set_outer(theta)
    drift = [torch.from_numpy(synthetic.dp_drift(m, n, seed=seed, worker=0, period=i)).cuda()
             for i, (m, n) in enumerate(shapes)]
    W_local = [t - d for t, d in zip(theta, drift)]

    for _ in range(W):
        g.outer_sync(W_local)
    torch.cuda.synchronize()
    so.trace_reset()
    ms = timed(torch, lambda: [g.outer_sync(W_local) for _ in range(K)], False)
    launches = so.launch_count()
    so.trace_enable(True)
    traced_ms = timed(torch, lambda: g.outer_sync(W_local), False)
    rep = so.trace_report()
    so.trace_enable(False)
    byts = {key: sum(dp_sync_bytes(m, n, k)[key] for (m, n), k in zip(shapes, g.ranks))
            for key in ("compress_p", "compress_q", "outer_step", "orth")}
    hbm = peaks["hbm_gbs"]

    def roof(kernel, trace_name, b):
        n_l, t = rep.get(trace_name, (0, 0.0))
        ach = b / (t * 1e-3) / 1e9 if t > 0 else None
        return {"kernel": kernel, "bound": "hbm", "achieved": ach, "peak": hbm, "unit": "GB/s",
                "frac": ach / hbm if ach else None, "avg_launch_ms": t / max(n_l, 1),
                "algorithmic_bytes_per_launch": b,
                "traffic": profiled_traffic(*DPSYNC_PROFILE, key=kernel.split()[0]),
                "traffic_source": "profiles/" + DPSYNC_PROFILE[0]}

    total_bytes = sum(byts.values())
    values = sum(m * n for m, n in shapes)
    sent = sum((m + n) * k for (m, n), k in zip(shapes, g.ranks))
    out = {"syncs_per_s": K / (ms * 1e-3), "ms_per_sync": ms / K, "gpu_launches_per_sync": launches / K,
           "ranks": g.ranks, "compression": values / sent,
           "hbm_bound_ms": 1e3 * total_bytes / (hbm * 1e9), "frac_of_hbm_bound": 1e3 * total_bytes / (hbm * 1e9) / (ms / K),
           "rooflines": [roof("dp_compress_p", "dp_compress_p", byts["compress_p"]),
                         roof("dp_compress_q", "dp_compress_q", byts["compress_q"]),
                         roof("dp_update (outer step)", "dp_outer_step", byts["outer_step"])],
           "kernels_traced_ms": {k: round(v[1], 4) for k, v in rep.items()}, "traced_sync_ms": traced_ms,
           "peak_source": "%s HBM copy bandwidth" % peak_src,
           "note": "one worker per GPU: the all-reduces of P and Q are the identity; the outer step "
                   "(Nesterov, lr 0.7, momentum 0.9) and error feedback run every sync"}
    g.close()
    return out


def run_ours(args, rank, world, local_rank, dist_ok):
    import torch

    import spectral_corrected_optimizer_gb300 as so
    from spectral_corrected_optimizer_gb300 import build as sob

    if not os.path.exists(sob.LIB) or sob.needs_build():
        if rank == 0:
            sob.build()
        if dist_ok:
            import torch.distributed as dist
            dist.barrier()
    torch.cuda.set_device(local_rank)
    peaks, peak_src = read_peaks()
    layer = Layer(seed=rank)
    K, W = args.steps, args.warmup

    # warm-up (step 0 carries the first anchor update + SVD refresh)
    for i in range(W):
        layer.step(i, t0=W)
    torch.cuda.synchronize()

    # ---- the timed region: K whole-hot-path steps; a refresh begins with the
    # first of them and every REFRESH_EVERY steps, and ends REFRESH_USE_AFTER
    # steps later (one still open after the last step ends inside the region)
    so.trace_reset()
    layer.last_sweeps = None
    with ClockSampler(local_rank) as clocks:
        ms = timed(torch, lambda: ([layer.step(W + i, t0=W) for i in range(K)], layer.refresh_end()), dist_ok)
    launches = so.launch_count()
    timed_sweeps = layer.last_sweeps
    ms_max = max_over_ranks(ms, dist_ok)
    value = world * K / (ms_max * 1e-3)

    # ---- breakdown: steady spectral step (traced), refresh, mask sweep
    steady_n = max(3, min(K, 10))
    so.trace_enable(True)
    steady_ms = timed(torch, lambda: [layer.spectral(1000 + i) for i in range(steady_n)], False) / steady_n
    rep = so.trace_report()
    so.trace_enable(False)
    so.trace_enable(True)
    sweeps = []
    refresh_ms = timed(torch, lambda: sweeps.append(layer.refresh(7)), False)
    refresh_rep = so.trace_report()
    so.trace_enable(False)
    # the overlapped schedule (the refresh begun at the anchor's arrival, running
    # beside the next REFRESH_USE_AFTER steps), for comparison with the headline's
    layer.use_after = REFRESH_USE_AFTER
    layer.reset_state()
    for i in range(W):
        layer.step(i, t0=W)
    torch.cuda.synchronize()
    ov_ms = timed(torch, lambda: ([layer.step(W + i, t0=W) for i in range(K)], layer.refresh_end()), False)
    overlap = {"steps_per_s": K / (ov_ms * 1e-3), "ms_per_step": ov_ms / K, "use_after": REFRESH_USE_AFTER,
               "refresh_sweeps": layer.last_sweeps,
               "schedule": "refresh begun at the anchor's arrival on the library's streams (specoptim_svd_refresh_"
                           "begin), ended %d steps later; the steps in between use the previous factors" %
                           REFRESH_USE_AFTER}
    layer.use_after = 0
    tf32 = measure_tf32_peak(torch)
    tf32_peak = tf32["tf32_tflops_sustained"]
    cfg_peaks = {"tf32_tflops": tf32_peak, "tf32_source": "measured cuBLAS sustained",
                 "hbm_gbs": peaks["hbm_gbs"]}
    elementwise = elementwise_bench(layer, peaks, peak_src)
    mask = {("p%.2f" % p): mask_sweep(layer, p) for p in (0.95, 0.90)}
    mask_fused = mask_fused_bench(peaks, peak_src)
    import synthetic as _syn
    dp_sync = run_dp_sync(list(_syn.LLAMA_1B_LAYER.values()), max(5, min(K, 20)), 3, peaks, peak_src, seed=rank)
    others = {}
    if not args.no_configs:
        import synthetic
        full = ModelWorkload(synthetic.LLAMA_1B_LAYER, synthetic.LLAMA_1B_LAYERS, seed=rank,
                             plain=[synthetic.LLAMA_1B_EMBED] + [(1, 2048)] * synthetic.LLAMA_1B_NORMS)
        others["full_1b"] = run_config("llama-3.2-1b full model: 16 layers x 7 matrices spectral-corrected, "
                                       "embedding 128256x2048 + 33 norm vectors plain AdamW", full, 20, 3,
                                       peaks=cfg_peaks)
        del full
        torch.cuda.empty_cache()
        sweep = {}
        for tau in (1e-4, 1e-3, 1e-2):  # the workload's tau_p values; tau changes d, not the work
            l7 = ModelWorkload(synthetic.LLAMA_7B_LAYER, 1, seed=rank, tau_p=tau)
            res7 = run_config("7B-shaped layer: q,o 4096x4096; k,v 1024x4096; gate,up 14336x4096; "
                              "down 4096x14336", l7, 20, 3,
                              mask_shape=(8 * 4096, 4096, 0.95) if tau == 1e-3 else None, peaks=cfg_peaks)
            sweep["%g" % tau] = {"steps_per_s": res7["steps_per_s"], "refresh_ms": res7["refresh_ms"],
                                 "refresh_sweeps_max": res7["refresh_sweeps_max"],
                                 "steady_step_ms": res7["steady_step_ms"], "step_frac": res7["step_frac"]}
            if tau == 1e-3:
                others["layer_7b"] = res7
            del l7
            torch.cuda.empty_cache()
        others["layer_7b"]["tau_p_sweep"] = sweep
    mask_frac = mask["p0.95"]["effective_GBps"] / peaks["hbm_gbs"]

    # rooflines of the two heaviest kernels: the tensor-core GEMM of the steady
    # step (its three epilogue variants are one kernel) and the Jacobi rotation
    # of the refresh; the primary one is the kernel with more device time per
    # refresh period (REFRESH_EVERY steady steps + one refresh)
    fam = {}
    for k, (n, t) in rep.items():
        key = "gemm_tf32" if k.startswith("gemm_tf32") else k
        a = fam.setdefault(key, [0, 0.0])
        a[0] += n
        a[1] += t
    total_ms = sum(v[1] for v in rep.values())
    g_launch, g_ms = fam.get("gemm_tf32", [0, 0.0])
    g_ach = layer.flops * steady_n / (g_ms * 1e-3) / 1e12 if g_ms > 0 else None
    roof_steady = {"kernel": "gemm_tf32", "bound": "tensor", "achieved": g_ach, "peak": tf32_peak,
                   "unit": "TFLOP/s", "frac": g_ach / tf32_peak if g_ach else None,
                   "peak_source": "measured in this run: cuBLAS tf32 sustained (peaks.tf32)",
                   "launches_per_step": g_launch / steady_n, "avg_launch_ms": g_ms / max(g_launch, 1),
                   "share_of_step": g_ms / total_ms, "traffic": profiled_traffic(*GEMM_PROFILE),
                   "traffic_source": "profiles/gemm_tf32_layer_step.md (ncu DRAM bytes per grouped launch; "
                                     "tensor-pipe activity of each launch in the same file)"}
    # the refresh's two tensor-core rotation kernels, both HBM-bound: A <- R^T A R
    # (jacobi_apply, on the critical chain) and Q <- Q R (jacobi_rotate, on a
    # second stream beside the solves, so its traced time includes sharing the SMs)
    nps = [padded_order(min(i.m, i.n)) for i in layer.inputs.values()]
    rounds = max(n // 32 for n in nps) - 1
    period_ms = REFRESH_EVERY * ms_max / K  # measured: the refresh overlaps the steps

    def hbm_roof(kernel, trace_name, per_matrix, profile):
        launches, ms = refresh_rep.get(trace_name, (0, 0.0))
        total = sum(sw * rounds * per_matrix(n) for sw, n in zip(sweeps[0], nps))
        ach = total / (ms * 1e-3) / 1e9 if ms > 0 else None
        return {"kernel": kernel, "bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": ach / peaks["hbm_gbs"] if ach else None,
                "peak_source": "%s HBM copy bandwidth" % peak_src,
                "launches_per_refresh": launches, "avg_launch_ms": ms / max(launches, 1),
                "algorithmic_bytes_per_refresh": total,
                "algorithmic_bytes_per_launch_all_active": sum(per_matrix(n) for n in nps),
                "traffic": profiled_traffic(*profile),
                "traffic_note": "ncu DRAM bytes per launch with all 7 matrices active "
                                "(compare with algorithmic_bytes_per_launch_all_active)",
                "traffic_source": "profiles/" + profile[0], "share_of_period": ms / period_ms}

    roof_apply = hbm_roof("jacobi_apply", "svd_jacobi_apply", apply_bytes, APPLY_PROFILE)
    roof_rotate = hbm_roof("jacobi_rotate", "svd_jacobi_rotate", rotate_bytes, ROTATE_PROFILE)
    roof_rotate["note"] = "runs beside the solves on a second stream; traced time includes that sharing"
    roof_steady["share_of_period"] = REFRESH_EVERY * g_ms / steady_n / period_ms
    # primary: the heaviest kernel of the critical chain (the Q update overlaps the solves)
    roof = max([roof_steady, roof_apply], key=lambda r: r["share_of_period"])
    step_bound_ms = 1e3 * max(layer.flops / (tf32_peak * 1e12), layer.bytes / (peaks["hbm_gbs"] * 1e9))

    result = {
        "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world, "steps": K, "warmup": W,
        "ms_per_step": ms_max / K, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32 (tf32 tensor-core products, fp32 accumulate; bf16 mask copies)",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": world, "parallelism": "replicas (one layer per GPU)",
                   "l2": "inputs larger than L2: each step streams 0.97 GB of distinct gradients and "
                         "optimizer state and 1 GB of activations",
                   "timed_refresh_sweeps": timed_sweeps,
                   "refresh_schedule": "every %d steps the anchor EMA and a batched SVD refresh of the 7 "
                                       "matrices in one call, before that step's spectral step" % REFRESH_EVERY},
        "gpu_launches": launches,
        "clocks": clocks.summary(),
        "roofline": roof,
        "breakdown": {"roofline_steady_gemm": roof_steady, "roofline_refresh_apply": roof_apply,
                      "roofline_refresh_q_rotate": roof_rotate,"steady_step_ms": steady_ms, "steady_steps_per_s": 1e3 / steady_ms,
                      "step_roofline_ms": step_bound_ms, "step_frac": step_bound_ms / steady_ms,
                      "refresh_ms": refresh_ms, "refresh_sweeps": sweeps[0],
                      "overlapped_refresh_schedule": overlap,
                      "refresh_note": "traced; one more refresh of the same layer (the Jacobi sweep count "
                                      "falls as the anchor EMA settles; the timed steps hold the second refresh)",
                      "kernels": {k: {"launches": v[0], "ms": v[1]} for k, v in rep.items()},
                      "refresh_kernels": {k: {"launches": v[0], "ms": round(v[1], 3)} for k, v in refresh_rep.items()}},
        "mask": dict(mask, frac_of_hbm=mask_frac, hbm_peak_GBps=peaks["hbm_gbs"]),
        "mask_fused": dict(mask_fused, workload="mask fused with the layer boundary: bf16 [65536, 2048], p = 0.95"),
        "dp_outer_sync": dict(dp_sync, workload="PowerSGD-compressed Streaming DiLoCo outer sync of the "
                                                "llama-3.2-1b decoder layer (7 matrices, rank for 64x)"),
        "other_configs": others,
        "elementwise": elementwise,
        "peaks": {"source": peak_src, "hbm_gbs": peaks["hbm_gbs"], "tf32_tflops": tf32_peak,
                  "tf32": tf32, "tf32_used": "sustained (the steady step and its GEMMs run in a loop)"},
    }
    if not args.no_e2e:
        result["e2e"] = run_e2e(layer, K, W, dist_ok, world)
    return result


def elementwise_bench(layer: Layer, peaks: dict, peak_src: str, reps: int = 10) -> dict:
    """HBM throughput of the two elementwise kernels: the anchor EMA of the 7
    matrices of the layer (12 B per element: M and G_anc read, M written) and
    the plain AdamW of the full model's embedding, 128256 x 2048 (28 B per
    element: W, g, m, v read, W, m, v written)."""
    torch, so = layer.torch, layer.so
    names = layer.names
    for n in names:
        layer.opt[n].anchor_update(layer.Ganc[n][0])
    ema_ms = timed(torch, lambda: [layer.opt[n].anchor_update(layer.Ganc[n][i % 2])
                                   for i in range(reps) for n in names], False) / reps
    ema_bytes = 12.0 * layer.params
    rows, cols = 128256, 2048
    g = torch.Generator(device="cuda").manual_seed(1)
    W = torch.randn(rows, cols, device="cuda", generator=g) * 0.02
    G = torch.randn(rows, cols, device="cuda", generator=g) * 1e-2
    m, v = torch.zeros_like(W), torch.zeros_like(W)
    so.adamw(W, G, m, v, 1, 2e-5)
    ad_ms = timed(torch, lambda: [so.adamw(W, G, m, v, 2 + i, 2e-5) for i in range(reps)], False) / reps
    ad_bytes = 28.0 * rows * cols
    del W, G, m, v
    torch.cuda.empty_cache()
    hbm = peaks["hbm_gbs"]

    def per_value(key):  # ncu DRAM bytes per value of the profiled case (grows in proportion)
        t = profiled_traffic(*ELEMENTWISE_PROFILE, key=key)
        return None if t is None else t / ELEMENTWISE_PROFILE_VALUES[key]

    return {"ema": {"kernel": "ema", "bound": "hbm", "ms": ema_ms, "GBps": ema_bytes / (ema_ms * 1e-3) / 1e9,
                    "frac": ema_bytes / (ema_ms * 1e-3) / 1e9 / hbm, "bytes": ema_bytes,
                    "traffic_bytes_per_value": per_value("ema"), "algorithmic_bytes_per_value": 12,
                    "workload": "anchor EMA of the 7 matrices of the llama-3.2-1b layer (7 launches)"},
            "adamw": {"kernel": "adamw", "bound": "hbm", "ms": ad_ms, "GBps": ad_bytes / (ad_ms * 1e-3) / 1e9,
                      "frac": ad_bytes / (ad_ms * 1e-3) / 1e9 / hbm, "bytes": ad_bytes,
                      "traffic_bytes_per_value": per_value("adamw"), "algorithmic_bytes_per_value": 28,
                      "workload": "plain AdamW of the 128256 x 2048 embedding"},
            "peak_source": "%s HBM copy bandwidth" % peak_src,
            "traffic_source": "profiles/" + ELEMENTWISE_PROFILE[0]}


E2E_REPEATS = 3


def run_e2e(layer: Layer, K: int, W: int, dist_ok: bool, world: int):
    """Same steps with host buffers, as a pipeline stage's training loop would
    drive them.  What crosses the host link each step is what the method sends:
    host -> device, the step's masked gradients (every 20th step also the anchor
    gradients) and the packed boundary values received from the neighbouring
    stages (the activation from the previous stage, the gradient from the next);
    device -> host, the packed values this stage sends, and once per anchor
    period (at each anchor's arrival) the updated weights: the parameter
    snapshot that the anchor circuit pulls periodically for its next unmasked
    pass.  The dense boundary
    activation and its gradient are produced and consumed on the device by the
    model's own layers, so they stay resident, as in training.  The copies run on
    two more streams (one per direction), double-buffered: step i+1's inputs
    travel while step i computes, and step i's outputs leave from device-side
    buffers while step i+1 computes.  All of it is inside the timed region."""
    torch = layer.torch
    names = layer.names
    hostG = {n: [g.cpu().pin_memory() for g in layer.Gpool[n][:2]] for n in names}
    hostA = {n: [g.cpu().pin_memory() for g in layer.Ganc[n]] for n in names}
    hostW = {n: torch.empty(layer.W[n].shape, dtype=torch.float32).pin_memory() for n in names}
    # received packed values: one boundary's pack of the synthetic activations
    host_hp = layer.so.mask_pack(layer.h, layer.K, 0, 0, 0).cpu().pin_memory()
    host_gp = layer.so.mask_pack(layer.g, layer.K, 0, 0, 0).cpu().pin_memory()
    sent_hp = [torch.empty_like(host_hp).pin_memory() for _ in range(2)]
    sent_gp = [torch.empty_like(host_gp).pin_memory() for _ in range(2)]
    devG = [{n: torch.empty_like(layer.Gpool[n][0]) for n in names} for _ in range(2)]
    devA = [{n: torch.empty_like(layer.Ganc[n][0]) for n in names} for _ in range(2)]
    in_hp = [torch.empty_like(layer.hp) for _ in range(2)]
    in_gp = [torch.empty_like(layer.gp) for _ in range(2)]
    out_hp = [torch.empty_like(layer.hp) for _ in range(2)]
    out_gp = [torch.empty_like(layer.gp) for _ in range(2)]
    snapW = {n: torch.empty_like(layer.W[n]) for n in names}
    compute, copy, back = torch.cuda.current_stream(), torch.cuda.Stream(), torch.cuda.Stream()
    stats = {"h2d": 0, "d2h": 0}
    freed = [torch.cuda.Event(), torch.cuda.Event()]  # compute done with input buffer b
    loaded = [torch.cuda.Event(), torch.cuda.Event()]  # inputs of buffer b landed
    out_free = [torch.cuda.Event(), torch.cuda.Event()]  # packed send buffer b has left
    snapped, sent = torch.cuda.Event(), torch.cuda.Event()
    for e in freed + out_free + [sent]:
        e.record(compute)

    t0 = W  # the timed steps start here (the refresh schedule of Layer.schedule)

    def load(i):  # on the copy stream: step i's inputs into buffer i % 2
        b = i % 2
        with torch.cuda.stream(copy):
            copy.wait_event(freed[b])
            if layer.schedule(i, t0) in ("refresh", "begin"):
                for n in names:
                    devA[b][n].copy_(hostA[n][layer.anchor_index(i, t0) % 2], non_blocking=True)
                    stats["h2d"] += devA[b][n].numel() * 4
            for n in names:
                devG[b][n].copy_(hostG[n][i % 2], non_blocking=True)
                stats["h2d"] += devG[b][n].numel() * 4
            in_hp[b].copy_(host_hp, non_blocking=True)
            in_gp[b].copy_(host_gp, non_blocking=True)
            stats["h2d"] += (in_hp[b].numel() + in_gp[b].numel()) * 2
            loaded[b].record(copy)

    def one(i, last):
        b = i % 2
        if not last:
            load(i + 1)
        compute.wait_event(loaded[b])
        what = layer.schedule(i, t0)
        if what == "refresh":
            t = time.perf_counter()
            layer.refresh(0, G=devA[b])
            refresh_host.append((time.perf_counter() - t) * 1e3)
        elif what == "begin":
            layer.refresh_end()
            layer.refresh_begin(0, G=devA[b])
        elif what == "end":
            layer.refresh_end()
        layer.spectral(i, G=devG[b])
        compute.wait_event(out_free[b])  # step i-2's packed values have left
        layer.mask_round_trip(i, hp_out=out_hp[b], gp_out=out_gp[b], hp_in=in_hp[b], gp_in=in_gp[b])
        freed[b].record(compute)
        # the anchor circuit pulls a parameter snapshot once per anchor period
        snap = what in ("refresh", "begin")
        if snap:
            compute.wait_event(sent)  # the previous weight snapshot has left
            for n in names:
                snapW[n].copy_(layer.W[n], non_blocking=True)
        snapped.record(compute)
        with torch.cuda.stream(back):
            back.wait_event(snapped)
            sent_hp[b].copy_(out_hp[b], non_blocking=True)
            sent_gp[b].copy_(out_gp[b], non_blocking=True)
            stats["d2h"] += (out_hp[b].numel() + out_gp[b].numel()) * 2
            out_free[b].record(back)
            if snap:
                for n in names:
                    hostW[n].copy_(snapW[n], non_blocking=True)
                    stats["d2h"] += snapW[n].numel() * 4
                sent.record(back)

    def run(first, count):
        load(first)
        for k in range(count):
            one(first + k, k == count - 1)
        compute.wait_stream(copy)
        compute.wait_stream(back)

    samples = []
    refresh_host = []
    with ClockSampler(torch.cuda.current_device()) as clocks:
        for _ in range(E2E_REPEATS):
            layer.reset_state()  # the same steps as the device-resident timed region, same refresh history
            run(0, W)
            stats["h2d"] = stats["d2h"] = 0
            layer.last_sweeps = None
            host = []
            refresh_host.clear()

            def enqueue():
                t = time.perf_counter()
                run(W, K)
                layer.refresh_end()
                host.append((time.perf_counter() - t) * 1e3)

            ms = max_over_ranks(timed(torch, enqueue, dist_ok), dist_ok)
            samples.append((ms, host[0], dict(stats), layer.last_sweeps, list(refresh_host)))
    ms, host_ms, st, sweeps, rh = sorted(samples, key=lambda x: x[0])[len(samples) // 2]
    return {"value": world * K / (ms * 1e-3), "unit": "steps/s", "host_enqueue_ms": host_ms, "device_ms": ms,
            "refresh_call_ms": rh, "clocks": clocks.summary(),
            "h2d_bytes_per_step": st["h2d"] // K, "d2h_bytes_per_step": st["d2h"] // K,
            "timed_refresh_sweeps": sweeps,
            "samples_steps_per_s": [world * K / (x[0] * 1e-3) for x in samples],
            "timing": "median of %d timed regions of the same %d steps, each from a fresh optimizer state after "
                      "the same warm-up (a transient slowdown of the shared host link hits one region, not the "
                      "median)" % (E2E_REPEATS, K),
            "pipeline": "copies on two more streams (one per direction), double-buffered inputs and packed "
                        "sends, weights read back from a device-side snapshot; every copy inside the timed region",
            "link_traffic": "every step: masked gradients in, packed boundary values (K of H per row) both ways; "
                            "every %d steps: anchor gradients in and a weight snapshot out (the anchor circuit's "
                            "periodic parameter pull); the dense boundary tensors stay on the device" % REFRESH_EVERY,
            "link": link_bandwidth(torch)}


def link_bandwidth(torch):
    """Pinned host <-> device copy bandwidth (GB/s) for 512 MB, each direction alone."""
    n = 128 << 20
    h = torch.empty(n, dtype=torch.float32).pin_memory()
    d = torch.empty(n, dtype=torch.float32, device="cuda")
    d.copy_(h, non_blocking=True)
    h2d = timed(torch, lambda: d.copy_(h, non_blocking=True), False)
    d2h = timed(torch, lambda: h.copy_(d, non_blocking=True), False)
    return {"h2d_GBps": 4 * n / (h2d * 1e-3) / 1e9, "d2h_GBps": 4 * n / (d2h * 1e-3) / 1e9}


# ------------------------------------------------------------------ the oracle on the host

class OracleSample:
    """The oracle as it stands, on a bounded sample of the workload: one steady
    spectral step of the 7-matrix layer (projection, blend, AdamW in float64)
    plus one stage-boundary mask round trip.  The SVD factors are random
    matrices of the right shapes (the step's cost does not depend on their
    values); the oracle's SVD refresh is not in the sample."""

    def __init__(self, seed=0):
        import numpy as np

        import oracle
        import synthetic

        self.np, self.oracle = np, oracle
        rng = np.random.default_rng(seed)
        self.mats = []
        for name, inp in synthetic.layer_inputs(synthetic.LLAMA_1B_LAYER, seed=seed, rank=32).items():
            opt = oracle.SpectralOptimizer(inp.m, inp.n)
            r = min(inp.m, inp.n)
            opt.U = rng.standard_normal((inp.m, r)) / np.sqrt(inp.m)
            opt.V = rng.standard_normal((inp.n, r)) / np.sqrt(inp.n)
            opt.d = rng.uniform(0.0, 1.0, r)
            self.mats.append((opt, inp.weights().astype(np.float64), inp.masked_grad(0)))
        self.K = oracle.mask_K(MASK_P, MASK_H)
        self.h = synthetic.activations_bf16(MASK_ROWS, MASK_H, seed=seed)
        self.g = synthetic.act_grads_bf16(MASK_ROWS, MASK_H, seed=seed)

    def step(self, i: int):
        oracle = self.oracle
        for opt, W, G in self.mats:
            opt.step(W, G, 2e-5)
        b = i % MASK_BOUNDARIES
        hp = oracle.mask_pack(self.h, self.K, b, i)
        oracle.mask_unpack(hp, MASK_H, b, i)
        gp = oracle.mask_pack(self.g, self.K, b, i)
        oracle.mask_unpack(gp, MASK_H, b, i)

    def describe(self):
        return ("one steady step of the 7-matrix Llama-3.2-1B layer (float64 projection, blend, "
                "AdamW with random factors of the right shapes; SVD refresh excluded) + one bf16 [65536,2048] "
                "p=0.95 mask round trip; steps/s = 1 / seconds per sample")


def oracle_toy_seconds():
    """The oracle's whole path on the toy workload (256 x 128: anchor EMA, its own
    Jacobi SVD, filter, step; a 64 x 256 bf16 mask round trip), seconds."""
    import oracle
    import synthetic
    inp = synthetic.toy_matrix_inputs()
    t = time.perf_counter()
    opt = oracle.SpectralOptimizer(inp.m, inp.n)
    opt.anchor_update(inp.anchor_grad(0))
    opt.svd_refresh()
    opt.step(inp.weights().astype("float64"), inp.masked_grad(0), 2e-5)
    h = synthetic.activations_bf16(64, 256)
    K = oracle.mask_K(0.95, 256)
    oracle.mask_unpack(oracle.mask_pack(h, K, 3, 7), 256, 3, 7)
    return time.perf_counter() - t


SINGLE_THREAD_SAMPLE = r"""
import json, os, sys, time
sys.path.insert(0, %(root)r)
import numpy as np
import oracle, synthetic, bench
out = {"toy_whole_path_seconds": bench.oracle_toy_seconds()}
inp = synthetic.MatrixInputs(512, 2048, seed=0, rank=32)
opt = oracle.SpectralOptimizer(512, 2048)
rng = np.random.default_rng(0)
opt.U = rng.standard_normal((512, 512)) / np.sqrt(512)
opt.V = rng.standard_normal((2048, 512)) / np.sqrt(2048)
opt.d = rng.uniform(0.0, 1.0, 512)
W, G = inp.weights().astype(np.float64), inp.masked_grad(0)
t = time.perf_counter()
opt.step(W, G, 2e-5)
out["kv_step_seconds"] = time.perf_counter() - t
print(json.dumps(out))
"""


def single_thread_oracle():
    """The oracle on one host thread (BLAS limited to one thread in a child
    process): the toy whole path and one steady step of a 512 x 2048 (k / v)
    matrix."""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        env.pop(k, None)
    try:
        res = subprocess.run([sys.executable, "-c", SINGLE_THREAD_SAMPLE % {"root": ROOT}], env=env,
                             capture_output=True, text=True, timeout=300)
        return json.loads(res.stdout.strip().splitlines()[-1])
    except Exception as e:  # reported, not a failure of the bench
        return {"error": str(e)[:200]}


def cpu_baseline():
    s = OracleSample()
    t = time.perf_counter()
    s.step(0)
    dt = time.perf_counter() - t
    return {"value": 1.0 / dt, "unit": "steps/s", "cores": os.cpu_count(), "kind": "oracle",
            "threads": "numpy's BLAS at its default thread count (one per host core); the C mask oracle "
                       "on one thread",
            "sample": s.describe(), "seconds": dt, "toy_whole_path_seconds": oracle_toy_seconds(),
            "single_thread": single_thread_oracle()}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    s = OracleSample()
    for i in range(args.warmup):
        s.step(i)
    t = time.perf_counter()
    for i in range(args.steps):
        s.step(args.warmup + i)
    dt = time.perf_counter() - t
    value = args.steps / dt
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": "steps/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": WORKLOAD, "global_batch": 1,
                                            "parallelism": "host cores, rank 0 only"},
            "cpu_baseline": {"value": value, "unit": "steps/s", "cores": os.cpu_count(), "kind": "oracle",
                             "sample": s.describe()},
            "e2e": {"value": value, "unit": "steps/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def run_profile_case(args):
    """Small cases for ncu captures (a few hundred MB on the device):
    'gate': steady spectral steps of one 8192x2048 matrix (transpose + 4 GEMMs per step);
    'mask': pack / unpack of one bf16 [65536, 2048] boundary at p = 0.95;
    'refresh': anchor EMA + SVD refresh of one 2048x2048 matrix, twice (the second warm);
    'layer': batched refresh, then grouped steady steps of the 7-matrix 1B layer;
    'dpsync': PowerSGD-compressed outer syncs of the 7-matrix 1B layer;
    'maskfused': the four mask ops fused with the layer boundary on bf16 [65536, 2048];
    'elementwise': per iteration the anchor EMA of one 8192 x 2048 matrix and a plain AdamW
    of 32768 x 2048 values (a quarter of the embedding)."""
    import numpy as np
    import torch

    import spectral_corrected_optimizer_gb300 as so
    import synthetic

    torch.cuda.set_device(env_int("LOCAL_RANK", 0))
    n_iter = args.warmup + args.steps
    if args.profile == "gate":
        inp = synthetic.MatrixInputs(8192, 2048, seed=0, rank=32)
        opt = so.SpectralOptimizer(8192, 2048)
        opt.anchor_update(torch.from_numpy(inp.anchor_grad(0)).cuda())
        W = torch.from_numpy(inp.weights()).cuda()
        G = [torch.from_numpy(inp.masked_grad(t)).cuda() for t in range(2)]
        for i in range(n_iter):
            opt.step(W, G[i % 2], 2e-5)
    elif args.profile == "layer":
        layer = Layer(seed=0)
        layer.refresh(0)
        for i in range(n_iter):
            layer.spectral(i)
    elif args.profile == "maskfused":
        K = so.mask_keep_count(MASK_P, MASK_H)
        gen = torch.Generator(device="cuda").manual_seed(3)
        a = torch.randn(MASK_ROWS, MASK_H, device="cuda", generator=gen).to(torch.bfloat16)
        b = torch.randn(MASK_ROWS, MASK_H, device="cuda", generator=gen).to(torch.bfloat16)
        gamma = torch.randn(MASK_H, device="cuda", generator=gen).to(torch.bfloat16)
        for i in range(n_iter):
            packed = so.mask_pack_add(a, b, K, i, 0)
            so.mask_unpack_rmsnorm(packed, gamma, 1e-5, MASK_H, i, 0)
            so.mask_rmsnorm_backward_pack(packed, gamma, 1e-5, a, b, i, 0)
            so.mask_unpack_add(packed, b, i, 0)
    elif args.profile == "dpsync":
        import spectral_corrected_optimizer_gb300.dpsync as dp
        shapes = list(synthetic.LLAMA_1B_LAYER.values())
        g = dp.DPSyncGroup(shapes, seed=0)
        theta = [torch.from_numpy(synthetic.normal_f32(0, 1, i, (m, n), 0.02)).cuda() for i, (m, n) in enumerate(shapes)]
        g.set_outer(theta)
        W_local = [t - torch.from_numpy(synthetic.dp_drift(m, n, period=i)).cuda()
                   for i, (t, (m, n)) in enumerate(zip(theta, shapes))]
        for i in range(n_iter):
            g.outer_sync(W_local)
    elif args.profile == "elementwise":
        inp = synthetic.MatrixInputs(8192, 2048, seed=0, rank=32)
        opt = so.SpectralOptimizer(8192, 2048)
        Ga = [torch.from_numpy(inp.anchor_grad(i)).cuda() for i in range(2)]
        g = torch.Generator(device="cuda").manual_seed(1)
        W = torch.randn(32768, 2048, device="cuda", generator=g) * 0.02
        G = torch.randn(32768, 2048, device="cuda", generator=g) * 1e-2
        m, v = torch.zeros_like(W), torch.zeros_like(W)
        for i in range(n_iter):
            opt.anchor_update(Ga[i % 2])
            so.adamw(W, G, m, v, i + 1, 2e-5)
    elif args.profile == "refresh":
        inp = synthetic.MatrixInputs(2048, 2048, seed=0, rank=32)
        opt = so.SpectralOptimizer(2048, 2048)
        for i in range(2):
            opt.anchor_update(torch.from_numpy(inp.anchor_grad(i)).cuda())
            opt.svd_refresh()
    else:
        K = so.mask_keep_count(MASK_P, MASK_H)
        h = torch.from_numpy(synthetic.activations_bf16(MASK_ROWS, MASK_H).view(np.int16)).view(
            torch.bfloat16).cuda()
        hp = torch.empty(MASK_ROWS, K, dtype=torch.bfloat16, device="cuda")
        hd = torch.empty_like(h)
        for i in range(n_iter):
            so.mask_pack(h, K, i % MASK_BOUNDARIES, 0, 0, out=hp)
            so.mask_unpack(hp, MASK_H, i % MASK_BOUNDARIES, 0, 0, out=hd)
    torch.cuda.synchronize()
    return {"profile": args.profile, "iterations": n_iter, "launches": so.launch_count()}


def free_port() -> int:
    import socket
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def launch_replicas(n: int) -> int:
    """`bench.py --gpus N` started as one process: start N ranks of this script
    (RANK / LOCAL_RANK / WORLD_SIZE / MASTER_ADDR / MASTER_PORT set as torchrun
    would set them, one GPU each), pass rank 0's output through, and return the
    worst exit status.  The ranks meet over a gloo group: barriers around the
    timed region and the max over ranks of its duration."""
    port = str(free_port())
    procs = []
    for rank in range(n):
        env = dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(n),
                   LOCAL_WORLD_SIZE=str(n), MASTER_ADDR="127.0.0.1", MASTER_PORT=port)
        procs.append(subprocess.Popen([sys.executable, os.path.abspath(__file__)] + sys.argv[1:], env=env,
                                      stdout=None if rank == 0 else subprocess.DEVNULL))
    rcs = [p.wait() for p in procs]
    return max(rcs, key=abs)


def run_dry(args, rank, world, dist_ok):
    """Host-only stand-in for the GPU work (for checking the launcher and the
    max-over-ranks timing without a GPU): rank r "works" for 20 + 10 r ms
    between the two barriers."""
    if dist_ok:
        import torch.distributed as dist
        dist.barrier()
    t = time.perf_counter()
    time.sleep((20 + 10 * rank) * 1e-3)
    ms = (time.perf_counter() - t) * 1e3
    if dist_ok:
        dist.barrier()
    ms_max = max_over_ranks(ms, dist_ok)
    return {"metric": METRIC, "value": world * args.steps / (ms_max * 1e-3), "unit": "steps/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max / args.steps,
            "dry_run": True, "rank_ms": ms, "scaling": "weak"}


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the full-1B and 7B-layer measurements reported beside the headline")
    ap.add_argument("--profile", choices=["gate", "mask", "refresh", "layer", "dpsync", "maskfused", "elementwise"],
                    default=None,
                    help="run a small case for ncu captures instead of the benchmark")
    ap.add_argument("--dry-run", action="store_true",
                    help="host-only stand-in for the GPU work (checks the launcher and the rank timing)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        sys.exit(launch_replicas(args.gpus))

    world = env_int("WORLD_SIZE", 1)
    rank = env_int("RANK", 0)
    local_rank = env_int("LOCAL_RANK", 0)
    dist_ok = False
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        dist_ok = True

    if args.profile:
        print(json.dumps(run_profile_case(args)), flush=True)
        return
    if args.dry_run:
        res = run_dry(args, rank, world, dist_ok)
    elif args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world, local_rank, dist_ok)
        if rank == 0 and world == 1 and not args.no_cpu_baseline:
            res["cpu_baseline"] = cpu_baseline()
    if dist_ok:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)


if __name__ == "__main__":
    main()
