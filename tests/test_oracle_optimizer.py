"""Pins of the oracle's spectral-corrected optimizer (CPU only).

Pages: "Communication-Efficient LLM Adaptation over Decentralized GPU Meshes",
key design 2 (anchor EMA) and key design 3 (SVD, Tikhonov filter
d_i = s_i/(s_i+tau_p), two-sided projection, convex blend, AdamW).  The pages
print no worked numbers, so every oracle function is pinned by closed forms,
special cases, brute force and independent library routines (LAPACK through
numpy, torch.optim.AdamW).  The "mutant" tests plant a plausible mistake in a
copy of an oracle function and check that some pin catches it.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic

RNG = np.random.default_rng(1234)


def rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return np.linalg.norm(a - b) / max(np.linalg.norm(b), 1e-300)


# ------------------------------------------------------------------ anchor EMA

def test_ema_closed_form_after_k_updates():
    G = RNG.standard_normal((7, 5))
    M = np.zeros_like(G)
    for k in range(1, 12):
        M = oracle.anchor_ema(M, G, 0.9)
        assert np.allclose(M, (1 - 0.9 ** k) * G, rtol=1e-14, atol=0)
    # first update from zero: M = 0.1 G exactly as printed (no bias correction)
    assert np.array_equal(oracle.anchor_ema(np.zeros(3), np.ones(3), 0.9), (1 - 0.9) * np.ones(3))


def test_ema_is_separate_from_the_adam_moments():
    opt = oracle.SpectralOptimizer(6, 4)
    opt.anchor_update(np.ones((6, 4)))
    W = np.zeros((6, 4))
    opt.step(W, np.ones((6, 4)), 1e-3)
    assert np.allclose(opt.M, 0.1)          # untouched by the step
    # m is fed by G_proj only: before the refresh G_filt = 0, so G_proj = 0.3 G
    assert np.allclose(opt.exp_avg, 0.1 * 0.3)


# ------------------------------------------------------------------ thin SVD

def svd_2x2(M):
    a, b, c, d = M.ravel()
    s1 = a * a + b * b + c * c + d * d
    det = a * d - b * c
    root = np.sqrt(max(s1 * s1 - 4 * det * det, 0.0))
    return np.sqrt([(s1 + root) / 2, max((s1 - root) / 2, 0.0)])


def eig_sym_3x3(A):
    """Eigenvalues of a symmetric 3x3 matrix by the trigonometric cubic formula (Smith 1961)."""
    q = np.trace(A) / 3
    p1 = A[0, 1] ** 2 + A[0, 2] ** 2 + A[1, 2] ** 2
    p2 = (A[0, 0] - q) ** 2 + (A[1, 1] - q) ** 2 + (A[2, 2] - q) ** 2 + 2 * p1
    p = np.sqrt(p2 / 6)
    B = (A - q * np.eye(3)) / p
    r = np.clip(np.linalg.det(B) / 2, -1, 1)
    phi = np.arccos(r) / 3
    e1 = q + 2 * p * np.cos(phi)
    e3 = q + 2 * p * np.cos(phi + 2 * np.pi / 3)
    return np.array([e1, 3 * q - e1 - e3, e3])


@pytest.mark.parametrize("shape", [(256, 128), (64, 48), (48, 64), (5, 3), (3, 5), (1, 1), (1, 7), (9, 1)])
def test_svd_reconstructs_and_is_orthonormal(shape):
    M = RNG.standard_normal(shape)
    U, s, V, _ = oracle.thin_svd(M)
    r = min(shape)
    assert U.shape == (shape[0], r) and V.shape == (shape[1], r) and s.shape == (r,)
    assert rel(U @ np.diag(s) @ V.T, M) <= 1e-12
    assert np.abs(U.T @ U - np.eye(r)).max() <= 1e-12
    assert np.abs(V.T @ V - np.eye(r)).max() <= 1e-12
    assert (np.diff(s) <= 0).all() and (s >= 0).all()


@pytest.mark.parametrize("shape", [(256, 128), (64, 48), (48, 64), (30, 30)])
def test_svd_values_match_lapack(shape):
    M = RNG.standard_normal(shape) * np.logspace(0, -6, shape[1])[None, :]
    s = oracle.thin_svd(M)[1]
    ref = np.linalg.svd(M, compute_uv=False)
    assert np.abs(s - ref).max() <= 1e-12 * ref[0]


def test_svd_2x2_and_3x3_closed_forms():
    for _ in range(20):
        M = RNG.standard_normal((2, 2))
        assert np.allclose(oracle.thin_svd(M)[1], svd_2x2(M), rtol=1e-13, atol=1e-15)
        M = RNG.standard_normal((3, 3))
        ev = np.sqrt(np.clip(eig_sym_3x3(M.T @ M), 0, None))
        assert np.allclose(oracle.thin_svd(M)[1], ev, rtol=1e-10, atol=1e-12)


def test_svd_of_diagonal_and_of_constructed_factors():
    diag = np.array([3.0, 0.5, 2.0, 1e-4])
    U, s, V, _ = oracle.thin_svd(np.diag(diag))
    assert np.allclose(s, np.sort(diag)[::-1], rtol=1e-15)
    assert np.allclose(np.abs(U), np.abs(V)) and np.allclose(np.abs(U).sum(0), 1)
    Q1 = np.linalg.qr(RNG.standard_normal((40, 12)))[0]
    Q2 = np.linalg.qr(RNG.standard_normal((25, 12)))[0]
    sv = np.linspace(5, 0.1, 12)
    U, s, V, _ = oracle.thin_svd(Q1 @ np.diag(sv) @ Q2.T)
    assert np.allclose(s[:12], sv, rtol=1e-12)
    # factors are unique up to sign for distinct values: compare sign-free products
    assert np.allclose(U[:, :12] * (U[:, :12] * Q1).sum(0), Q1, atol=1e-10)
    assert np.allclose(V[:, :12] * (V[:, :12] * Q2).sum(0), Q2, atol=1e-10)


def test_svd_rank_deficient_and_zero():
    M = RNG.standard_normal((10, 3)) @ RNG.standard_normal((3, 8))
    U, s, V, _ = oracle.thin_svd(M)
    assert np.all(s[3:] <= 1e-13 * s[0])
    assert np.abs(U.T @ U - np.eye(8)).max() <= 1e-10
    U, s, V, _ = oracle.thin_svd(np.zeros((6, 4)))
    assert np.all(s == 0) and np.abs(U.T @ U - np.eye(4)).max() == 0


# ------------------------------------------------------------------ filter

def test_filter_bounded_monotone_and_limits():
    s = np.concatenate([[0.0], np.logspace(-9, 2, 200)])
    for tau in (1e-5, 1e-3, 1e-1):
        d = oracle.filter_coeffs(s, tau)
        assert (d >= 0).all() and (d <= 1).all()
        assert (np.diff(d) >= 0).all()
        assert d[0] == 0.0
        assert d[-1] > 1 - tau / 100 * 1.01         # s >> tau passes
        assert d[1] < 1e-9 / tau * 1.01             # s << tau attenuated to ~s/tau
        assert np.allclose(d, s / (s + tau))
    assert np.all(oracle.filter_coeffs(s, 1e30) < 1e-27)
    assert oracle.filter_coeffs(np.array([0.0]), 0.0)[0] == 0.0


# ------------------------------------------------------------------ projection

def spectral_fn(A, tau):
    """f(A) = sum_i sqrt(l_i)/(sqrt(l_i)+tau) q_i q_i^T for symmetric PSD A (LAPACK eigh)."""
    lam, Q = np.linalg.eigh(A)
    # eigh returns the exact zero eigenvalues of a rank-deficient Gram matrix as
    # +-1e-16 * lam_max; those are zeros
    lam = np.where(lam > 1e-13 * lam.max(), lam, 0.0)
    sq = np.sqrt(lam)
    return (Q * (sq / (sq + tau))) @ Q.T


def gfilt_independent(M, G, tau):
    """G_filt = (U D U^T) G (V D V^T) with both projectors from eigh of M M^T and M^T M."""
    return spectral_fn(M @ M.T, tau) @ G @ spectral_fn(M.T @ M, tau)


def oracle_gfilt(M, G, tau):
    U, s, V, _ = oracle.thin_svd(M)
    return oracle.project(U, V, oracle.filter_coeffs(s, tau), G)[2]


@pytest.mark.parametrize("shape", [(40, 40), (64, 24), (24, 64), (256, 128)])
@pytest.mark.parametrize("tau", [1e-2, 1.0, 30.0])
def test_projection_matches_spectral_projectors(shape, tau):
    M = RNG.standard_normal(shape)
    G = RNG.standard_normal(shape)
    assert rel(oracle_gfilt(M, G, tau), gfilt_independent(M, G, tau)) <= 1e-9


def test_projection_returns_its_intermediates():
    M, G = RNG.standard_normal((12, 9)), RNG.standard_normal((12, 9))
    U, s, V, _ = oracle.thin_svd(M)
    d = oracle.filter_coeffs(s, 0.5)
    X, Xf, Gf = oracle.project(U, V, d, G)
    assert np.allclose(X, U.T @ G @ V) and np.allclose(Xf, d[:, None] * X * d[None, :])
    assert np.allclose(Gf, U @ Xf @ V.T)


def test_projection_limits():
    G = RNG.standard_normal((30, 30))
    M = RNG.standard_normal((30, 30))
    # tau -> inf: everything filtered out
    assert np.linalg.norm(oracle_gfilt(M, G, 1e14)) <= 1e-12 * np.linalg.norm(G)
    # tau -> 0, square full rank: G_filt -> G
    assert rel(oracle_gfilt(M, G, 1e-14), G) <= 1e-10
    # tall full column rank: V is square, G_filt -> U U^T G = projection on col(M)
    Mt, Gt = RNG.standard_normal((50, 20)), RNG.standard_normal((50, 20))
    Q = np.linalg.qr(Mt)[0]
    assert rel(oracle_gfilt(Mt, Gt, 1e-14), Q @ Q.T @ Gt) <= 1e-10
    # wide full row rank: U is square, G_filt -> G V V^T = projection on row(M)
    Mw, Gw = RNG.standard_normal((20, 50)), RNG.standard_normal((20, 50))
    Q = np.linalg.qr(Mw.T)[0]
    assert rel(oracle_gfilt(Mw, Gw, 1e-14), Gw @ Q @ Q.T) <= 1e-10


def test_projection_diagonal_and_rank_one_closed_forms():
    sd = np.array([2.0, 0.3, 1.1, 0.05, 0.7])
    G = RNG.standard_normal((5, 5))
    tau = 0.2
    d = sd / (sd + tau)
    assert np.allclose(oracle_gfilt(np.diag(sd), G, tau), d[:, None] * G * d[None, :], atol=1e-13)
    u, v = RNG.standard_normal(9), RNG.standard_normal(6)
    sigma = np.linalg.norm(u) * np.linalg.norm(v)
    un, vn = u / np.linalg.norm(u), v / np.linalg.norm(v)
    G = RNG.standard_normal((9, 6))
    d1 = sigma / (sigma + tau)
    want = d1 * d1 * np.outer(un, un) @ G @ np.outer(vn, vn)
    assert rel(oracle_gfilt(np.outer(u, v), G, tau), want) <= 1e-12


# ------------------------------------------------------------------ blend

def test_blend_endpoints():
    G, Gf = RNG.standard_normal((8, 3)), RNG.standard_normal((8, 3))
    assert np.array_equal(oracle.blend(G, Gf, 1.0), G)
    assert np.array_equal(oracle.blend(G, Gf, 0.0), Gf)
    assert np.allclose(oracle.blend(G, Gf, 0.3), 0.3 * G + 0.7 * Gf)


# ------------------------------------------------------------------ AdamW

def test_adamw_matches_torch_reference():
    shape = (7, 5)
    W0 = RNG.standard_normal(shape) * 0.02
    p = torch.nn.Parameter(torch.from_numpy(W0.copy()))
    opt = torch.optim.AdamW([p], lr=2e-5, betas=(0.9, 0.999), eps=1e-8, weight_decay=0.01)
    W, m, v = W0.copy(), np.zeros(shape), np.zeros(shape)
    for t in range(1, 8):
        g = RNG.standard_normal(shape) * 10.0 ** RNG.integers(-6, 1)
        p.grad = torch.from_numpy(g.copy())
        opt.step()
        W, m, v = oracle.adamw(W, m, v, g, t, 2e-5, 0.9, 0.999, 1e-8, 0.01)
        st = opt.state[p]
        assert rel(W - W0, p.detach().numpy() - W0) <= 1e-12
        assert rel(m, st["exp_avg"].numpy()) <= 1e-14
        assert rel(v, st["exp_avg_sq"].numpy()) <= 1e-14


# ------------------------------------------------------------------ whole step

def test_step_before_first_anchor_is_scaled_adamw():
    inp = synthetic.toy_matrix_inputs()
    opt = oracle.SpectralOptimizer(inp.m, inp.n)
    W, G = inp.weights(), inp.masked_grad(0)
    W1, Gf, Gp = opt.step(W, G, 2e-5)
    assert np.all(Gf == 0) and np.allclose(Gp, 0.3 * G.astype(np.float64))


def test_toy_step_matches_independent_pieces():
    inp = synthetic.toy_matrix_inputs()
    opt = oracle.SpectralOptimizer(inp.m, inp.n)
    G_anc = inp.anchor_grad(0)
    opt.anchor_update(G_anc)
    opt.svd_refresh()
    assert opt.s.shape == (128,) and (opt.d >= 0).all() and (opt.d <= 1).all()
    W, G = inp.weights(), inp.masked_grad(0)
    W1, Gf, Gp = opt.step(W, G, 2e-5)
    M = 0.1 * G_anc.astype(np.float64)
    assert rel(Gf, gfilt_independent(M, G.astype(np.float64), 1e-3)) <= 1e-8
    assert rel(Gp, 0.3 * G.astype(np.float64) + 0.7 * Gf) <= 1e-15


# ------------------------------------------------------------------ mutants

def _mutant_projections():
    def transposed_sides(U, V, d, G):
        # U and V swapped in role (only shape-compatible when square)
        X = V.T @ G @ U
        return None, None, V @ (d[:, None] * X * d[None, :]) @ U.T

    def one_sided_filter(U, V, d, G):
        X = U.T @ G @ V
        return None, None, U @ (d[:, None] * X) @ V.T

    def sqrt_filter(U, V, d, G):
        X = U.T @ G @ V
        return None, None, U @ (np.sqrt(d)[:, None] * X * np.sqrt(d)[None, :]) @ V.T

    def dropped_transpose(U, V, d, G):
        X = U.T @ G @ V
        return None, None, U @ (d[:, None] * X * d[None, :]).T @ V.T

    return [transposed_sides, one_sided_filter, sqrt_filter, dropped_transpose]


@pytest.mark.parametrize("mutant", _mutant_projections(), ids=lambda f: f.__name__)
def test_projection_pins_catch_planted_mistakes(mutant, monkeypatch):
    monkeypatch.setattr(oracle, "project", mutant)
    M, G = RNG.standard_normal((30, 30)), RNG.standard_normal((30, 30))
    caught = rel(oracle_gfilt(M, G, 1.0), gfilt_independent(M, G, 1.0)) > 1e-6
    sd = np.array([2.0, 0.3, 1.1, 0.05, 0.7])
    G5 = RNG.standard_normal((5, 5))
    d = sd / (sd + 0.2)
    caught |= not np.allclose(oracle_gfilt(np.diag(sd), G5, 0.2), d[:, None] * G5 * d[None, :], atol=1e-12)
    assert caught


def test_adamw_pin_catches_a_missing_bias_correction(monkeypatch):
    def no_bias(W, m, v, g, t, lr, b1, b2, eps, wd):
        W = W * (1 - lr * wd)
        m = b1 * m + (1 - b1) * g
        v = b2 * v + (1 - b2) * g * g
        return W - lr * m / (np.sqrt(v) + eps), m, v

    monkeypatch.setattr(oracle, "adamw", no_bias)
    with pytest.raises(AssertionError):
        test_adamw_matches_torch_reference()
