"""GPU parity of the data-parallel outer synchronisation against the float64
oracle (key design 4 of "Communication-Efficient LLM Adaptation over
Decentralized GPU Meshes": Streaming DiLoCo outer step, PowerSGD-compressed).

Each CUDA call is compared with the oracle function of the same step on the
GPU's own inputs (so that a mismatch names the step), then whole chains of
synchronisations are compared end to end.  Tolerance: relative Frobenius error
<= 1e-4.  The kernels compute in fp32 from fp32 inputs; the sums they form have
at most n or m terms, whose rounding is about sqrt(n) 2^-24 ~ 1e-6 relative,
and the two Cholesky-QR passes return an orthonormal basis to fp32 rounding for
the condition numbers of these inputs (random Q), so 1e-4 keeps a margin of
more than 10x and is tighter than the 2e-3 the optimizer path is held to.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from gpu_util import Guarded, dev, ensure_lib, host, rel

pytestmark = pytest.mark.gpu
TOL = 1e-4

# (m, n, k): every padded rank (8, 16, 32, 64), ragged rows and columns, m below
# and above one compress_q row range (512)
SHAPES = [(300, 516, 5), (1100, 260, 13), (600, 1028, 26), (200, 388, 50), (1030, 132, 64)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def dp():
    import spectral_corrected_optimizer_gb300.dpsync as m
    return m


def make_group(shapes, seed=0, **kw):
    Q0 = [torch.from_numpy(synthetic.dp_q0(n, k, seed=seed, index=i)) for i, (m, n, k) in enumerate(shapes)]
    g = dp().DPSyncGroup([(m, n) for m, n, _ in shapes], Q0=Q0, ranks=[k for _, _, k in shapes], **kw)
    return g, [q.numpy().astype(np.float64) for q in Q0]


def state(g, i, outer=False):
    E, th, mo, Ph = g.get_state(i)
    torch.cuda.synchronize()
    return host(E), (host(th) if th is not None else None), (host(mo) if mo is not None else None), host(Ph)


def test_each_call_matches_the_oracle_on_the_gpu_inputs():
    g, _ = make_group(SHAPES, seed=3)
    for sync in range(2):
        Xs = [synthetic.normal_f32(11, sync, i, (m, n), 1e-2) for i, (m, n, _) in enumerate(SHAPES)]
        Ys = [synthetic.normal_f32(12, sync, i, (m, n), 1e-2) for i, (m, n, _) in enumerate(SHAPES)]
        E_prev = [state(g, i)[0] for i in range(len(SHAPES))]
        Q_prev = [host(q).astype(np.float64) for q in g.Q]
        g.compress_p([dev(x) for x in Xs], [dev(y) for y in Ys])
        torch.cuda.synchronize()
        Ms = []
        for i in range(len(SHAPES)):
            M_ref, P_ref = oracle.dpsync_compress_p(Xs[i], Ys[i], E_prev[i], Q_prev[i])
            M = state(g, i)[0]
            assert rel(M, M_ref) < 1e-6, (sync, i)
            assert rel(host(g.P[i]), P_ref) < TOL, (sync, i)
            Ms.append(M)
        g.orthogonalize()
        Phs = []
        for i, (m, n, k) in enumerate(SHAPES):
            Ph = state(g, i)[3].astype(np.float64)
            assert rel(Ph, oracle.orthogonalize(host(g.P[i]))) < TOL, (sync, i)
            assert np.abs(Ph.T @ Ph - np.eye(k)).max() < 1e-5
            Phs.append(Ph)
        g.compress_q()
        torch.cuda.synchronize()
        for i in range(len(SHAPES)):
            assert rel(host(g.Q[i]), oracle.dpsync_compress_q(Ms[i], Phs[i])) < TOL, (sync, i)
        guarded = [Guarded((m, n)) for m, n, _ in SHAPES]
        outs = [x.t for x in guarded]
        g.decompress(outs, q_scale=0.5)
        torch.cuda.synchronize()
        assert all(x.intact() for x in guarded)
        for i in range(len(SHAPES)):
            D_ref, E_ref = oracle.dpsync_decompress(Ms[i], Phs[i], host(g.Q[i]), 0.5)
            assert rel(host(outs[i]), D_ref) < TOL, (sync, i)
            assert rel(state(g, i)[0], E_ref) < TOL, (sync, i)
    g.close()


@pytest.mark.parametrize("mix", [0.0, 0.25])
def test_outer_sync_chain_matches_the_oracle(mix):
    shapes = SHAPES[:3]
    g, Q0 = make_group(shapes, seed=5, outer_lr=0.7, outer_momentum=0.9, mix=mix)
    refs = []
    thetas = []
    for i, (m, n, k) in enumerate(shapes):
        th = synthetic.normal_f32(21, 0, i, (m, n), 0.02)
        thetas.append(th)
        r = oracle.DPSync(m, n, Q0[i], rank=k, outer_lr=0.7, outer_momentum=0.9, mix=mix)
        r.set_outer(th)
        refs.append(r)
    g.set_outer([dev(t) for t in thetas])
    for period in range(3):
        locals_ = [thetas[i] - synthetic.dp_drift(m, n, seed=2, worker=0, period=period)
                   for i, (m, n, _) in enumerate(shapes)]
        guarded = [Guarded(w.shape) for w in locals_]
        W = [x.t for x in guarded]
        for w, x in zip(locals_, W):
            x.copy_(dev(w))
        g.outer_sync(W)
        torch.cuda.synchronize()
        assert all(x.intact() for x in guarded)
        for i, (m, n, k) in enumerate(shapes):
            th_before = refs[i].theta.copy()
            W_ref = refs[i].outer_sync(locals_[i])
            E, th, mo, _ = state(g, i)
            assert rel(th - th_before, refs[i].theta - th_before) < TOL, (period, i)
            assert rel(mo, refs[i].mom) < TOL, (period, i)
            assert rel(E, refs[i].E) < TOL, (period, i)
            assert rel(host(W[i]) - locals_[i], W_ref - locals_[i]) < TOL, (period, i)
            thetas[i] = th.copy()   # next period drifts from the GPU's outer weights
            refs[i].theta = th.astype(np.float64)


@pytest.mark.parametrize("r,k", [(3, 3), (3, 5), (1, 8)])
def test_low_rank_gradient_is_reproduced_and_dependent_columns_vanish(r, k):
    m, n = 400, 264
    A = synthetic.normal_f32(31, r, 0, (m, r), 1.0)
    B = synthetic.normal_f32(31, r, 1, (n, r), 1.0)
    G = (A @ B.T).astype(np.float32)
    g, _ = make_group([(m, n, k)], seed=7)
    out = torch.empty(m, n, device="cuda")
    g.sync_grad([dev(G)], [out])
    torch.cuda.synchronize()
    assert rel(host(out), G) < 1e-5
    E, _, _, Ph = state(g, 0)
    assert np.linalg.norm(E) < 1e-5 * np.linalg.norm(G)
    norms = np.linalg.norm(Ph, axis=0)
    assert np.allclose(norms[:r], 1.0, atol=1e-5)
    assert not Ph[:, r:].any()       # dependent columns are exactly zero


def test_two_workers_in_lock_step():
    shapes = [(600, 1028, 26), (300, 516, 5)]
    ga, Q0 = make_group(shapes, seed=9)
    gb, _ = make_group(shapes, seed=9)
    Gs = [[synthetic.normal_f32(41, w, i, (m, n), 1e-2) for i, (m, n, _) in enumerate(shapes)] for w in range(2)]
    outs = [[torch.empty(m, n, device="cuda") for m, n, _ in shapes] for _ in range(2)]
    groups = (ga, gb)
    for w in range(2):
        groups[w].compress_p([dev(x) for x in Gs[w]])
    Psum = ga.P_flat + gb.P_flat
    ga.P_flat.copy_(Psum)
    gb.P_flat.copy_(Psum)
    for w in range(2):
        groups[w].orthogonalize()
        groups[w].compress_q()
    Qsum = ga.Q_flat + gb.Q_flat
    ga.Q_flat.copy_(Qsum)
    gb.Q_flat.copy_(Qsum)
    for w in range(2):
        groups[w].decompress(outs[w], q_scale=0.5)
    torch.cuda.synchronize()
    for i, (m, n, k) in enumerate(shapes):
        Ms, Ps = zip(*(oracle.dpsync_compress_p(Gs[w][i], None, np.zeros((m, n)), Q0[i]) for w in range(2)))
        Ph = oracle.orthogonalize(sum(Ps))
        Qs = sum(oracle.dpsync_compress_q(M, Ph) for M in Ms)
        D = oracle.dpsync_decompress(Ms[0], Ph, Qs, 0.5)[0]
        for w in range(2):
            assert rel(host(outs[w][i]), D) < TOL, (w, i)
        assert np.array_equal(host(outs[0][i]), host(outs[1][i]))


@pytest.mark.parametrize("m,n,k", [(1, 4, 1), (5, 8, 1), (17, 4, 4), (64, 256, 8), (8, 12, 8)])
def test_small_and_degenerate_shapes(m, n, k):
    G = synthetic.normal_f32(51, m, n, (m, n), 1.0)
    g, Q0 = make_group([(m, n, k)], seed=11)
    out = torch.empty(m, n, device="cuda")
    g.sync_grad([dev(G)], [out])
    torch.cuda.synchronize()
    ref = oracle.DPSync(m, n, Q0[0], rank=k)
    D = ref.sync_grad(G)
    assert rel(host(out), D) < TOL
    # E is measured against the input: with k = min(m, n) the error is pure rounding
    assert np.linalg.norm(state(g, 0)[0] - ref.E) < TOL * np.linalg.norm(G)


def test_zero_input_gives_zero():
    g, _ = make_group([(128, 256, 16)], seed=13)
    out = torch.full((128, 256), 7.0, device="cuda")
    g.sync_grad([torch.zeros(128, 256, device="cuda")], [out])
    torch.cuda.synchronize()
    assert not host(out).any()
    assert not state(g, 0)[3].any()


def test_host_argument_checks():
    g, _ = make_group([(64, 128, 8)], seed=1)
    with pytest.raises(Exception):
        g.outer_step([torch.zeros(64, 128, device="cuda")])      # no set_outer yet
    with pytest.raises(Exception):
        g.compress_p(None, None)                                  # X = theta needs set_outer
    with pytest.raises(Exception):
        dp().DPSyncGroup([(64, 130)], ranks=[4])                  # n not a multiple of 4
    with pytest.raises(Exception):
        dp().DPSyncGroup([(640, 1280)], ranks=[65])               # rank above 64


def test_full_layer_sync_sampled():
    """The bench's workload: one outer sync of the 7 matrices of a Llama-3.2-1B
    layer (64x rank rule) in one batch, each call checked on sampled rows and
    columns that the oracle computes one by one."""
    shapes = list(synthetic.LLAMA_1B_LAYER.values())
    ranks = [oracle.dpsync_rank(m, n) for m, n in shapes]
    Q0 = [synthetic.dp_q0(n, k, seed=2, index=i) for i, ((m, n), k) in enumerate(zip(shapes, ranks))]
    g = dp().DPSyncGroup(shapes, Q0=[torch.from_numpy(q) for q in Q0])
    assert g.ranks == ranks
    theta = [synthetic.normal_f32(3, 1, i, (m, n), 0.02) for i, (m, n) in enumerate(shapes)]
    W = [theta[i] - synthetic.dp_drift(m, n, seed=3, period=i) for i, (m, n) in enumerate(shapes)]
    g.set_outer([dev(t) for t in theta])
    Wd = [dev(w) for w in W]
    g.compress_p(None, Wd)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    Ms, Ps = [], []
    for i, ((m, n), k) in enumerate(zip(shapes, ranks)):
        M = state(g, i)[0]
        rows = rng.choice(m, 16, replace=False)
        M_ref = theta[i][rows].astype(np.float64) - W[i][rows]
        assert rel(M[rows], M_ref) < 1e-6
        assert rel(host(g.P[i])[rows], M_ref @ Q0[i].astype(np.float64)) < TOL
        Ms.append(M)
        Ps.append(host(g.P[i]).astype(np.float64))
    g.orthogonalize()
    Phs = []
    for i, ((m, n), k) in enumerate(zip(shapes, ranks)):
        Ph = state(g, i)[3].astype(np.float64)
        assert np.abs(Ph.T @ Ph - np.eye(k)).max() < 1e-5
        assert rel(Ph, oracle.orthogonalize(Ps[i])) < TOL
        Phs.append(Ph)
    g.compress_q()
    torch.cuda.synchronize()
    Qs = []
    for i, ((m, n), k) in enumerate(zip(shapes, ranks)):
        cols = rng.choice(n, 16, replace=False)
        Q = host(g.Q[i]).astype(np.float64)
        assert rel(Q[cols], Ms[i][:, cols].astype(np.float64).T @ Phs[i]) < TOL
        Qs.append(Q)
    g.outer_step(Wd, 1.0)
    torch.cuda.synchronize()
    for i, ((m, n), k) in enumerate(zip(shapes, ranks)):
        E, th, mo, _ = state(g, i)
        rows = rng.choice(m, 8, replace=False)
        D = Phs[i][rows] @ Qs[i].T
        assert rel(E[rows], Ms[i][rows] - D) < TOL
        th_ref, mo_ref, W_ref = oracle.outer_nesterov(theta[i][rows], np.zeros((8, n)), D, 0.7, 0.9)
        assert rel(mo[rows], mo_ref) < TOL
        assert rel(th[rows] - theta[i][rows], th_ref - theta[i][rows]) < TOL
        assert np.array_equal(host(Wd[i])[rows], th[rows])
    g.close()
