"""GPU parity of the mask ops fused with the layer boundary against the oracle
(key design 1 of "Communication-Efficient LLM Adaptation over Decentralized GPU
Meshes", with the decoder layer's residual sum on the sender and RMSNorm on the
receiver).

pack_add, unpack_add and the unpacked h~ are bit-exact (both sides form the
float32 sum of two bf16 values and round it to bf16, nearest even).  The
RMSNorm outputs are fp32 arithmetic rounded once to bf16 against the oracle's
float64: x may differ by one bf16 ulp; the backward value is a sum of three
terms, each carrying at most one fp32-rounding-level error before the final
rounding, so it is held to 2^-8 of the sum of the terms' magnitudes.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from gpu_util import Guarded, dev, ensure_lib, host

pytestmark = pytest.mark.gpu

CASES = [(64, 256, 13, 3, 7), (1000, 2048, 102, 0, 1), (600, 2048, 205, 14, 0), (37, 3000, 150, 2, 5),
         (24, 4096, 205, 1, 3), (16, 256, 0, 0, 0), (16, 256, 256, 0, 0)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


def so():
    import spectral_corrected_optimizer_gb300 as m
    return m


def bf(rows, H, seed, idx, scale=1.0):
    return synthetic.f32_to_bf16_bits(synthetic.normal_f32(seed, 20 + idx, rows, (rows, H), scale))


def ulp_diff(a_bits, b_bits):
    a = a_bits.astype(np.int32)
    b = b_bits.astype(np.int32)
    # same sign: distance in representation; zeros compare exactly
    return np.where((a ^ b) & 0x8000, np.abs(a & 0x7FFF) + np.abs(b & 0x7FFF), np.abs(a - b))


@pytest.mark.parametrize("rows,H,K,layer,step", CASES)
def test_pack_add_bit_exact(rows, H, K, layer, step):
    a, b = bf(rows, H, 1, 0), bf(rows, H, 1, 1, 0.3)
    out = Guarded((rows, K), torch.bfloat16)
    got = so().mask_pack_add(dev(a), dev(b), K, layer, step, out=out.t)
    torch.cuda.synchronize()
    assert np.array_equal(host(got), oracle.mask_pack_add(a, b, K, layer, step))
    assert out.intact()


@pytest.mark.parametrize("rows,H,K,layer,step", CASES)
def test_unpack_rmsnorm(rows, H, K, layer, step):
    packed = bf(rows, K, 2, 0) if K else np.zeros((rows, 0), np.uint16)
    gamma = bf(1, H, 2, 1, 0.5)[0]
    eps = 1e-5
    hg, xg = Guarded((rows, H), torch.bfloat16), Guarded((rows, H), torch.bfloat16)
    h, x = so().mask_unpack_rmsnorm(dev(packed), dev(gamma), eps, H, layer, step, h_out=hg.t, x_out=xg.t)
    torch.cuda.synchronize()
    assert hg.intact() and xg.intact()
    h_ref, x_ref_bits, _ = oracle.mask_unpack_rmsnorm(packed, gamma, eps, H, layer, step)
    assert np.array_equal(host(h), h_ref)
    assert ulp_diff(host(x), x_ref_bits).max() <= 1


@pytest.mark.parametrize("with_res", [True, False])
@pytest.mark.parametrize("rows,H,K,layer,step", CASES[:5])
def test_rmsnorm_backward_pack(rows, H, K, layer, step, with_res):
    packed = bf(rows, K, 3, 0)
    gamma = bf(1, H, 3, 1, 0.7)[0]
    dx = bf(rows, H, 3, 2)
    g_res = bf(rows, H, 3, 3, 0.2) if with_res else None
    eps = 1e-6
    out = Guarded((rows, K), torch.bfloat16)
    got = so().mask_rmsnorm_backward_pack(dev(packed), dev(gamma), eps, dev(dx),
                                          None if g_res is None else dev(g_res), layer, step, out=out.t)
    torch.cuda.synchronize()
    assert out.intact()
    _, ref = oracle.mask_rmsnorm_backward_pack(packed, gamma, eps, dx, g_res, layer, step)
    # magnitude of the terms at each kept dim
    h = oracle.bf16_value(oracle.mask_unpack(packed, H, layer, step))
    idx = oracle.mask_indices(rows, H, K, layer, step).astype(np.int64)
    rr = np.sqrt(np.mean(h * h, axis=1, keepdims=True) + eps)
    gdx = np.abs(oracle.bf16_value(gamma)[None, :] * oracle.bf16_value(dx))
    s = np.abs(np.sum(oracle.bf16_value(gamma)[None, :] * oracle.bf16_value(dx) * h, axis=1, keepdims=True))
    mag = np.take_along_axis(gdx / rr + np.abs(h) * s / (H * rr ** 3), idx, axis=1)
    if g_res is not None:
        mag = mag + np.abs(np.take_along_axis(oracle.bf16_value(g_res), idx, axis=1))
    err = np.abs(oracle.bf16_value(host(got)) - ref)
    assert (err <= 2.0 ** -8 * mag + 1e-30).all()


@pytest.mark.parametrize("rows,H,K,layer,step", CASES)
def test_unpack_add_bit_exact(rows, H, K, layer, step):
    packed = bf(rows, K, 4, 0) if K else np.zeros((rows, 0), np.uint16)
    g = bf(rows, H, 4, 1)
    gg = Guarded((rows, H), torch.bfloat16)
    gd = gg.t
    gd.copy_(dev(g))
    so().mask_unpack_add(dev(packed), gd, layer, step)
    torch.cuda.synchronize()
    assert np.array_equal(host(gd), oracle.mask_unpack_add(packed, g, layer, step))
    assert gg.intact()


def test_full_boundary_sampled_rows():
    """The workload's boundary tensor bf16 [65536, 2048], p = 0.95 (K = 102): every
    fused op on the whole tensor, rows sampled for the oracle."""
    rows, H, K, layer, step = 65536, 2048, so().mask_keep_count(0.95, 2048), 5, 0
    a, b = bf(rows, H, 6, 0), bf(rows, H, 6, 1, 0.3)
    gamma = bf(1, H, 6, 2, 0.5)[0]
    da, db = dev(a), dev(b)
    packed = so().mask_pack_add(da, db, K, layer, step)
    h, x = so().mask_unpack_rmsnorm(packed, dev(gamma), 1e-5, H, layer, step)
    g = db.clone()
    so().mask_unpack_add(packed, g, layer, step)
    torch.cuda.synchronize()
    sample = np.random.default_rng(0).choice(rows, 64, replace=False)
    idx_all = oracle.mask_indices(rows, H, K, layer, step)
    hp, hh, xh, gh = host(packed), host(h), host(x), host(g)
    for r in sample:
        idx = idx_all[r]
        assert np.array_equal(hp[r], oracle.bf16_bits(oracle.bf16_value(a[r, idx]).astype(np.float32)
                                                      + oracle.bf16_value(b[r, idx]).astype(np.float32)))
        dense = np.zeros(H, np.uint16)
        dense[idx] = hp[r]
        assert np.array_equal(hh[r], dense)
        v = oracle.bf16_value(dense)
        xr = oracle.bf16_bits(v / np.sqrt(np.mean(v * v) + 1e-5) * oracle.bf16_value(gamma))
        assert ulp_diff(xh[r], xr).max() <= 1
        gr = b[r].copy()
        gr[idx] = oracle.bf16_bits(oracle.bf16_value(b[r, idx]).astype(np.float32)
                                   + oracle.bf16_value(hp[r]).astype(np.float32))
        assert np.array_equal(gh[r], gr)
