"""The host side of the data-parallel synchronisation with two gloo ranks on
CPU: `sync_protocol` (the order of the calls and the two all-reduces of P and
Q, summed, with q_scale = 1/workers) driven by `default_allreduce`.  The five
compute calls are stood in for by the float64 oracle on each rank, so the
check is that the protocol reproduces the lock-step result of both workers."""
import json
import os
import socket
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

WORKER = r"""
import json, sys
sys.path.insert(0, %(root)r)
import numpy as np
import torch
import torch.distributed as dist
import oracle
import synthetic
from spectral_corrected_optimizer_gb300.dpsync import default_allreduce, sync_protocol

dist.init_process_group("gloo")
rank, world = dist.get_rank(), dist.get_world_size()
m, n, k = 40, 24, 3


class OracleOps:
    # the five calls of one matrix on the float64 oracle; P and Q in torch CPU buffers
    def __init__(self, Q0, theta):
        self.Q_flat = torch.from_numpy(Q0.reshape(-1).copy())
        self.P_flat = torch.zeros(m * k, dtype=torch.float64)
        self.E = np.zeros((m, n))
        self.theta, self.mom = theta.copy(), np.zeros((m, n))

    def compress_p(self, X, Y):
        X = self.theta if X is None else X
        self.M, P = oracle.dpsync_compress_p(X, Y, self.E, self.Q_flat.numpy().reshape(n, k))
        self.P_flat.copy_(torch.from_numpy(P.reshape(-1)))

    def orthogonalize(self):
        self.Ph = oracle.orthogonalize(self.P_flat.numpy().reshape(m, k))

    def compress_q(self):
        self.Q_flat.copy_(torch.from_numpy(oracle.dpsync_compress_q(self.M, self.Ph).reshape(-1)))

    def decompress(self, out, q_scale):
        D, self.E = oracle.dpsync_decompress(self.M, self.Ph, self.Q_flat.numpy().reshape(n, k), q_scale)
        out[...] = D

    def outer_step(self, W, q_scale):
        D, self.E = oracle.dpsync_decompress(self.M, self.Ph, self.Q_flat.numpy().reshape(n, k), q_scale)
        self.theta, self.mom, W[...] = oracle.outer_nesterov(self.theta, self.mom, D, 0.7, 0.9)


Q0 = synthetic.dp_q0(n, k, seed=4).astype(np.float64)
theta0 = synthetic.normal_f32(6, 0, 0, (m, n), 0.02).astype(np.float64)
ops = OracleOps(Q0, theta0)
G = synthetic.normal_f32(5, rank, 0, (m, n), 1.0).astype(np.float64)
out = np.zeros((m, n))
sync_protocol(ops, default_allreduce(), world, G, None, out, outer=False)
W = theta0 - synthetic.dp_drift(m, n, seed=8, worker=rank).astype(np.float64)
sync_protocol(ops, default_allreduce(), world, None, W, W, outer=True)
print(json.dumps({"rank": rank, "D": out.tolist(), "W": W.tolist(), "theta": ops.theta.tolist()}),
      flush=True)
dist.destroy_process_group()
"""


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def lockstep(G_list, W_list):
    import oracle
    import synthetic
    m, n, k = 40, 24, 3
    Q0 = synthetic.dp_q0(n, k, seed=4).astype(np.float64)
    theta = synthetic.normal_f32(6, 0, 0, (m, n), 0.02).astype(np.float64)
    w = len(G_list)
    Es = [np.zeros((m, n)) for _ in range(w)]
    Q = Q0
    outs = []
    for X_list, Y_list in ((G_list, [None] * w), ([theta] * w, W_list)):
        Ms, Ps = zip(*(oracle.dpsync_compress_p(X_list[i], Y_list[i], Es[i], Q) for i in range(w)))
        Ph = oracle.orthogonalize(sum(Ps))
        Q = sum(oracle.dpsync_compress_q(M, Ph) for M in Ms)
        res = [oracle.dpsync_decompress(M, Ph, Q, 1.0 / w) for M in Ms]
        Es = [E for _, E in res]
        outs.append(res[0][0])
    theta_new, _, W_new = oracle.outer_nesterov(theta, np.zeros((m, n)), outs[1], 0.7, 0.9)
    return outs[0], W_new, theta_new


def test_sync_protocol_with_two_gloo_ranks(tmp_path):
    import synthetic
    script = tmp_path / "worker.py"
    script.write_text(WORKER % {"root": ROOT})
    port = free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        procs.append(subprocess.Popen([sys.executable, str(script)], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=180) for p in procs]
    for p, (out, err) in zip(procs, outs):
        assert p.returncode == 0, err
    res = [json.loads(o.strip().splitlines()[-1]) for o, _ in outs]
    m, n = 40, 24
    G = [synthetic.normal_f32(5, r, 0, (m, n), 1.0).astype(np.float64) for r in range(2)]
    theta0 = synthetic.normal_f32(6, 0, 0, (m, n), 0.02).astype(np.float64)
    W = [theta0 - synthetic.dp_drift(m, n, seed=8, worker=r).astype(np.float64) for r in range(2)]
    D_ref, W_ref, theta_ref = lockstep(G, W)
    for r in res:
        assert np.abs(np.array(r["D"]) - D_ref).max() < 1e-12
        assert np.abs(np.array(r["W"]) - W_ref).max() < 1e-12
        assert np.abs(np.array(r["theta"]) - theta_ref).max() < 1e-12
    # and the two workers hold the same decompressed mean and the same outer weights
    assert res[0]["D"] == res[1]["D"] and res[0]["theta"] == res[1]["theta"]
