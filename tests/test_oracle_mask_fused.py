"""Pins of the oracle's mask ops fused with the layer boundary (CPU only).

Pages: "Communication-Efficient LLM Adaptation over Decentralized GPU Meshes",
key design 1 (only the K kept values of the boundary activation and of its
gradient travel; the backward uses the same indices).  The fused ops put the
mask next to the ops that produce and consume the boundary tensor: the
decoder layer's residual sum on the sender, RMSNorm on the receiver.  Pinned
against torch CPU routines (bfloat16 conversion and addition, rms_norm and its
autograd in float64) combined with the already pinned pack / unpack.
"""
import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(77)
H, ROWS, LAYER, STEP = 256, 48, 3, 7


def bf16_rand(shape, scale=1.0):
    x = torch.from_numpy((RNG.standard_normal(shape) * scale).astype(np.float32)).to(torch.bfloat16)
    return x.view(torch.int16).numpy().view(np.uint16)


def to_torch(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)


def test_bf16_rounding_matches_torch():
    x = np.concatenate([RNG.standard_normal(4000).astype(np.float32) * 10 ** RNG.uniform(-30, 30, 4000).astype(np.float32),
                        np.array([0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -(1.0 + 2 ** -8), 3.3e38, -3.3e38,
                                  np.inf, -np.inf, 1e-40], dtype=np.float32)])
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(oracle.bf16_bits(x), ref)
    assert np.array_equal(oracle.bf16_value(ref), torch.from_numpy(ref.view(np.int16)).view(torch.bfloat16).double().numpy())


@pytest.mark.parametrize("K", [0, 1, 13, 102, 256])
def test_pack_add_is_pack_of_the_bf16_sum(K):
    a, b = bf16_rand((ROWS, H)), bf16_rand((ROWS, H), 0.3)
    s = (to_torch(a) + to_torch(b)).view(torch.int16).numpy().view(np.uint16)   # torch bf16 add
    assert np.array_equal(oracle.mask_pack_add(a, b, K, LAYER, STEP), oracle.mask_pack(s, K, LAYER, STEP))


@pytest.mark.parametrize("K", [0, 13, 102])
def test_unpack_rmsnorm_matches_torch(K):
    packed = bf16_rand((ROWS, K))
    gamma = bf16_rand((H,), 0.5)
    eps = 1e-5
    h, x_bits, x = oracle.mask_unpack_rmsnorm(packed, gamma, eps, H, LAYER, STEP)
    assert np.array_equal(h, oracle.mask_unpack(packed, H, LAYER, STEP))
    ref = torch.nn.functional.rms_norm(to_torch(h).double(), (H,), to_torch(gamma).double(), eps)
    assert np.abs(x - ref.numpy()).max() <= 1e-12 * max(1.0, np.abs(ref.numpy()).max())
    assert np.array_equal(x_bits, oracle.bf16_bits(ref.numpy()))
    # off-mask dims stay exactly zero, kept dims carry the scaled values
    m = oracle.mask_matrix(ROWS, H, K, LAYER, STEP)
    assert not oracle.bf16_value(x_bits)[~m].any()


@pytest.mark.parametrize("with_res", [True, False])
def test_rmsnorm_backward_pack_matches_autograd(with_res):
    K, eps = 40, 1e-6
    packed = bf16_rand((ROWS, K))
    gamma, dx = bf16_rand((H,), 0.7), bf16_rand((ROWS, H))
    g_res = bf16_rand((ROWS, H), 0.2) if with_res else None
    h = torch.tensor(oracle.bf16_value(oracle.mask_unpack(packed, H, LAYER, STEP)), requires_grad=True)
    y = torch.nn.functional.rms_norm(h, (H,), torch.tensor(oracle.bf16_value(gamma)), eps)
    y.backward(torch.tensor(oracle.bf16_value(dx)))
    full = h.grad.numpy() + (oracle.bf16_value(g_res) if with_res else 0.0)
    idx = oracle.mask_indices(ROWS, H, K, LAYER, STEP).astype(np.int64)
    want = np.take_along_axis(full, idx, axis=1)
    bits, vals = oracle.mask_rmsnorm_backward_pack(packed, gamma, eps, dx, g_res, LAYER, STEP)
    assert np.abs(vals - want).max() <= 1e-12 * max(1.0, np.abs(want).max())
    assert np.array_equal(bits, oracle.bf16_bits(want))


def test_unpack_add_is_unpack_then_bf16_add():
    K = 102
    packed, g = bf16_rand((ROWS, K)), bf16_rand((ROWS, H))
    dense = oracle.mask_unpack(packed, H, LAYER, STEP)
    want = (to_torch(g) + to_torch(dense)).view(torch.int16).numpy().view(np.uint16)
    got = oracle.mask_unpack_add(packed, g, LAYER, STEP)
    # off-mask entries: g + (+0) is g itself (bit for bit, including -0)
    assert np.array_equal(got, want)


def test_mutant_backward_without_the_projection_term_is_caught():
    K, eps = 40, 1e-6
    packed, gamma, dx = bf16_rand((ROWS, K)), bf16_rand((H,)), bf16_rand((ROWS, H))
    h = oracle.bf16_value(oracle.mask_unpack(packed, H, LAYER, STEP))
    rr = np.sqrt(np.mean(h * h, axis=1, keepdims=True) + eps)
    wrong = oracle.bf16_value(gamma)[None, :] * oracle.bf16_value(dx) / rr     # drops -h s / (H r^3)
    idx = oracle.mask_indices(ROWS, H, K, LAYER, STEP).astype(np.int64)
    _, vals = oracle.mask_rmsnorm_backward_pack(packed, gamma, eps, dx, None, LAYER, STEP)
    assert np.abs(np.take_along_axis(wrong, idx, axis=1) - vals).max() > 1e-3
