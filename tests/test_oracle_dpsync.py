"""Pins of the oracle's data-parallel synchronisation (CPU only).

Pages: "Communication-Efficient LLM Adaptation over Decentralized GPU Meshes",
key design 4 (dual compression: Streaming DiLoCo outer synchronisation with
PowerSGD 64x low-rank compression).  The pages print only the ratio, so the
oracle's power step, orthogonalisation, error feedback and outer Nesterov step
are pinned by their mathematical properties and by independent library
routines (LAPACK QR and SVD through numpy, torch.optim.SGD); the "mutant" tests
plant a plausible mistake in a copy of an oracle function and check that a pin
catches it.
"""
import os

import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(4321)
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


def low_rank(m, n, r, rng=RNG):
    return rng.standard_normal((m, r)) @ rng.standard_normal((r, n))


# ------------------------------------------------------------------ rank rule

def test_rank_rule_gives_the_stated_ratio():
    with open(os.path.join(GOLDEN, "dpsync_ratio.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    assert len(rows) == 2
    for name, ratio, tol, *shapes in rows:
        sent = total = 0
        for s in shapes:
            m, n = map(int, s.split("x"))
            k = oracle.dpsync_rank(m, n, float(ratio))
            assert 1 <= k <= min(m, n)
            sent += (m + n) * k
            total += m * n
        assert abs(total / sent - float(ratio)) <= float(tol), name


def test_rank_rule_edges():
    assert oracle.dpsync_rank(2048, 2048) == 16          # 2048^2 / (64 * 4096) = 16 exactly
    assert oracle.dpsync_rank(256, 128) == 1             # 1.33 rounds down
    assert oracle.dpsync_rank(4, 4) == 1                 # below 1 clamps up
    assert oracle.dpsync_rank(100, 3, 0.5) == 3          # clamps to min(m, n)
    assert oracle.dpsync_rank(24, 8, 0.25) == 8          # 24 * 8 / (0.25 * 32) = 24 -> min(m,n)


# ------------------------------------------------------------------ orthogonalisation

@pytest.mark.parametrize("m,k", [(50, 6), (300, 26), (64, 64), (9, 1)])
def test_orthogonalize_matches_lapack_qr(m, k):
    P = RNG.standard_normal((m, k))
    Qr, R = np.linalg.qr(P)                      # Householder QR (LAPACK)
    Qr = Qr * np.sign(np.diag(R))                # positive diagonal convention
    assert np.abs(oracle.orthogonalize(P) - Qr).max() < 1e-12


def test_orthogonalize_is_a_qr_factor_with_positive_diagonal():
    P = ill_conditioned(80, 10, 1e4)
    Ph = oracle.orthogonalize(P)
    assert np.abs(Ph.T @ Ph - np.eye(10)).max() < 1e-12
    R = Ph.T @ P
    assert np.abs(np.tril(R, -1)).max() < 1e-12 * np.abs(R).max()
    assert (np.diag(R) > 0).all()
    assert rel(Ph @ R, P) < 1e-13


def test_orthogonalize_dependent_and_zero_columns_become_zero():
    a, b, c = (RNG.standard_normal(40) for _ in range(3))
    P = np.stack([a, b, 2 * a - 3 * b, np.zeros(40), c, b], axis=1)
    Ph = oracle.orthogonalize(P)
    for j in (2, 3, 5):
        assert not Ph[:, j].any()
    keep = Ph[:, [0, 1, 4]]
    assert np.abs(keep.T @ keep - np.eye(3)).max() < 1e-12
    # the accepted columns span the columns of P
    assert rel(keep @ (keep.T @ P), P) < 1e-13
    assert not oracle.orthogonalize(np.zeros((7, 3))).any()


def test_orthogonalize_drops_columns_below_the_threshold():
    U, _ = np.linalg.qr(RNG.standard_normal((60, 3)))
    eps = np.sqrt(oracle.GS_DROP)
    P = np.stack([U[:, 0], U[:, 0] + 0.3 * eps * U[:, 1], U[:, 0] + 3 * eps * U[:, 2]], axis=1)
    Ph = oracle.orthogonalize(P)
    assert not Ph[:, 1].any()                               # residual 0.3 x threshold: dropped
    assert abs(abs(Ph[:, 2] @ U[:, 2]) - 1) < 1e-9          # residual 3 x threshold: kept


# ------------------------------------------------------------------ power step

@pytest.mark.parametrize("m,n,r,k", [(60, 40, 3, 3), (40, 60, 2, 5), (33, 17, 1, 4), (24, 24, 6, 6)])
def test_one_sync_is_exact_up_to_rank_k(m, n, r, k):
    G = low_rank(m, n, r)
    s = oracle.DPSync(m, n, RNG.standard_normal((n, k)), rank=k)
    D = s.sync_grad(G)
    assert rel(D, G) < 1e-12
    assert np.abs(s.E).max() < 1e-12 * np.abs(G).max()


def test_power_iteration_converges_to_the_truncated_svd():
    m, n, k = 70, 50, 4
    U, _ = np.linalg.qr(RNG.standard_normal((m, n)))
    V, _ = np.linalg.qr(RNG.standard_normal((n, n)))
    s = np.concatenate([[10.0, 7.0, 5.0, 4.0], np.linspace(1.0, 0.1, n - 4)])
    G = U @ np.diag(s) @ V.T
    u, sv, vt = np.linalg.svd(G, full_matrices=False)
    Gk = u[:, :k] @ np.diag(sv[:k]) @ vt[:k]
    sync = oracle.DPSync(m, n, RNG.standard_normal((n, k)), rank=k, error_feedback=False)
    for _ in range(60):          # warm-started Q: subspace iteration, rate (1/4)^2 per sync
        D = sync.sync_grad(G)
    assert rel(D, Gk) < 1e-12


def test_error_feedback_telescopes():
    m, n, k, T = 30, 20, 2, 9
    sync = oracle.DPSync(m, n, RNG.standard_normal((n, k)), rank=k)
    sum_G = np.zeros((m, n))
    sum_D = np.zeros((m, n))
    for _ in range(T):
        G = RNG.standard_normal((m, n))
        sum_G += G
        sum_D += sync.sync_grad(G)
    # every value the compression left out is still in E
    assert rel(sum_D + sync.E, sum_G) < 1e-13
    assert np.abs(sync.E).max() > 0.1


def test_workers_sum_then_scale_equals_one_worker_on_the_mean():
    m, n, k, W = 40, 24, 3, 3
    Q0 = RNG.standard_normal((n, k))
    Gs = [RNG.standard_normal((m, n)) for _ in range(W)]
    # lock-step workers: the all-reduce sums over them, q_scale = 1/W
    Ms, Ps = zip(*(oracle.dpsync_compress_p(G, None, np.zeros((m, n)), Q0) for G in Gs))
    P_hat = oracle.orthogonalize(sum(Ps))
    Q_sum = sum(oracle.dpsync_compress_q(M, P_hat) for M in Ms)
    Ds = [oracle.dpsync_decompress(M, P_hat, Q_sum, 1.0 / W)[0] for M in Ms]
    single = oracle.DPSync(m, n, Q0, rank=k, error_feedback=False).sync_grad(sum(Gs) / W)
    for D in Ds:
        assert rel(D, single) < 1e-13
    # D is the projection of the mean onto span(P^)
    assert rel(Ds[0], P_hat @ (P_hat.T @ (sum(Gs) / W))) < 1e-13


# ------------------------------------------------------------------ outer step

@pytest.mark.parametrize("momentum,lr", [(0.9, 0.7), (0.0, 1.0), (0.5, 0.3)])
def test_outer_nesterov_matches_torch_sgd(momentum, lr):
    theta0 = RNG.standard_normal((6, 5))
    p = torch.nn.Parameter(torch.from_numpy(theta0.copy()))
    opt = torch.optim.SGD([p], lr=lr, momentum=momentum, nesterov=momentum > 0, dampening=0.0)
    theta, mom = theta0.copy(), np.zeros_like(theta0)
    for _ in range(5):
        D = RNG.standard_normal(theta0.shape)
        p.grad = torch.from_numpy(D.copy())
        opt.step()
        theta, mom, W = oracle.outer_nesterov(theta, mom, D, lr, momentum)
        assert np.abs(theta - p.detach().numpy()).max() < 1e-14
        assert np.array_equal(W, theta)


def test_outer_mix():
    theta, mom, W = oracle.outer_nesterov(np.ones((2, 2)), np.zeros((2, 2)), np.zeros((2, 2)),
                                          0.7, 0.9, W_local=np.full((2, 2), 3.0), mix=0.25)
    assert np.allclose(W, 0.75 * 1.0 + 0.25 * 3.0, rtol=0, atol=1e-15)


def test_full_rank_outer_sync_with_unit_lr_is_parameter_averaging():
    m, n, W = 12, 8, 2
    theta0 = RNG.standard_normal((m, n))
    locals_ = [theta0 + 0.1 * RNG.standard_normal((m, n)) for _ in range(W)]
    Q0 = RNG.standard_normal((n, n))
    syncs = [oracle.DPSync(m, n, Q0, rank=n, outer_lr=1.0, outer_momentum=0.0) for _ in range(W)]
    for s in syncs:
        s.set_outer(theta0)
    Ms, Ps = zip(*(oracle.dpsync_compress_p(s.theta, Wl, s.E, s.Q) for s, Wl in zip(syncs, locals_)))
    P_hat = oracle.orthogonalize(sum(Ps))
    Q_sum = sum(oracle.dpsync_compress_q(M, P_hat) for M in Ms)
    D = oracle.dpsync_decompress(Ms[0], P_hat, Q_sum, 1.0 / W)[0]
    theta, _, W_new = oracle.outer_nesterov(theta0, np.zeros((m, n)), D, 1.0, 0.0)
    assert rel(W_new, sum(locals_) / W) < 1e-13


def test_outer_sync_class_runs_the_pieces_in_order():
    m, n, k = 20, 16, 3
    Q0 = RNG.standard_normal((n, k))
    s = oracle.DPSync(m, n, Q0, rank=k)
    theta0 = RNG.standard_normal((m, n))
    s.set_outer(theta0)
    W_local = theta0 - 0.01 * RNG.standard_normal((m, n))
    W_new = s.outer_sync(W_local)
    M, P = oracle.dpsync_compress_p(theta0, W_local, np.zeros((m, n)), Q0)
    Ph = oracle.orthogonalize(P)
    Q = oracle.dpsync_compress_q(M, Ph)
    D, E = oracle.dpsync_decompress(M, Ph, Q)
    theta, mom, W = oracle.outer_nesterov(theta0, np.zeros((m, n)), D, 0.7, 0.9)
    assert np.array_equal(W_new, W) and np.array_equal(s.E, E) and np.array_equal(s.Q, Q)
    assert np.array_equal(s.mom, mom)


# ------------------------------------------------------------------ mutants

def _gs_single_pass(P):
    P = np.asarray(P, np.float64)
    out = np.zeros_like(P)
    for c in range(P.shape[1]):
        v = P[:, c].copy()
        for j in range(c):
            v -= (out[:, j] @ P[:, c]) * out[:, j]      # classical, once
        nv = np.linalg.norm(v)
        if nv > 0:
            out[:, c] = v / nv
    return out


def ill_conditioned(m, k, kappa):
    U, _ = np.linalg.qr(RNG.standard_normal((m, k)))
    V, _ = np.linalg.qr(RNG.standard_normal((k, k)))
    return U @ np.diag(np.logspace(0, -np.log10(kappa), k)) @ V.T


def test_mutant_single_classical_pass_is_caught():
    P = ill_conditioned(80, 10, 1e4)       # every residual above the drop threshold
    Po = oracle.orthogonalize(P)
    assert np.abs(Po.T @ Po - np.eye(10)).max() < 1e-12
    Ph = _gs_single_pass(P)
    assert np.abs(Ph.T @ Ph - np.eye(10)).max() > 1e-11    # fails the orthonormality pin


def test_mutant_transposed_q_and_missing_error_are_caught():
    m, n, k = 30, 20, 2
    G = low_rank(m, n, 2)
    Q0 = RNG.standard_normal((n, k))
    M, P = oracle.dpsync_compress_p(G, None, np.zeros((m, n)), Q0)
    Ph = oracle.orthogonalize(P)
    Q = oracle.dpsync_compress_q(M, Ph)
    assert rel(Ph @ Q.T, G) < 1e-12
    # a plausible slip, Q = M P^ on a square matrix, breaks exactness
    Gs = low_rank(20, 20, 2)
    Ms, Ps = oracle.dpsync_compress_p(Gs, None, np.zeros((20, 20)), RNG.standard_normal((20, 2)))
    Phs = oracle.orthogonalize(Ps)
    assert rel(Phs @ (Ms @ Phs).T, Gs) > 1e-3
    # without the error term the telescoping pin fails
    sync = oracle.DPSync(m, n, Q0, rank=k, error_feedback=False)
    tot_G = tot_D = 0
    for _ in range(4):
        G = RNG.standard_normal((m, n))
        tot_G = tot_G + G
        tot_D = tot_D + sync.sync_grad(G)
    assert rel(tot_D + sync.E, tot_G) > 1e-2
