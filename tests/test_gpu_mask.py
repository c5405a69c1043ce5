"""GPU parity of the activation mask against the oracle: bit-exact indices and
bytes (key design 1 of "Communication-Efficient LLM Adaptation over
Decentralized GPU Meshes": h~ = h (.) m, K kept dims per token, backward
reuses the same indices, off-mask gradient exactly zero)."""
import numpy as np
import pytest
import torch

import oracle
import spectral_corrected_optimizer_gb300 as so
import synthetic
from gpu_util import Guarded, dev, ensure_lib, host

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    ensure_lib()


CASES = [  # rows, H, K, layer, step, batch_id
    (64, 256, 13, 3, 7, 0),          # toy case
    (37, 2048, 102, 0, 0, 0),        # ragged rows at the 1B width, p = 0.95
    (131, 2048, 205, 14, 3, 2),      # p = 0.90
    (19, 4096, 205, 1, 9, 5),        # 7B width
    (45, 3000, 150, 2, 2, 2),        # H not a power of two (cycle walking)
    (9, 7, 7, 0, 1, 0),              # K = H, rows of 14 bytes
    (17, 96, 1, 5, 5, 5),            # K = 1
    (5, 64, 0, 0, 0, 0),             # K = 0
]


@pytest.mark.parametrize("rows,H,K,layer,step,batch", CASES)
def test_indices_bit_exact(rows, H, K, layer, step, batch):
    got = host(so.mask_indices(rows, H, K, layer, step, batch))
    assert np.array_equal(got, oracle.mask_indices(rows, H, K, layer, step, batch))
    out = Guarded((rows, K), torch.int32)
    lib = so.lib()
    assert lib.mask_indices(out.t.data_ptr(), rows, H, K, layer, step, batch,
                            torch.cuda.current_stream().cuda_stream) == so.OK
    assert np.array_equal(host(out.t), got) and out.intact()


@pytest.mark.parametrize("rows,H,K,layer,step,batch", CASES)
@pytest.mark.parametrize("kind", ["bf16", "f32"])
def test_pack_and_unpack_bit_exact(rows, H, K, layer, step, batch, kind):
    if kind == "bf16":
        h = synthetic.activations_bf16(rows, H, seed=rows)
        h[0, :] = 0x8000  # -0.0
        if rows > 2:
            h[1, :] = 0x7FC0  # NaN
            h[2, :] = 0xFF80  # -inf
    else:
        h = synthetic.act_grads_f32(rows, H, seed=rows)
        h[0, :] = -0.0
        if rows > 1:
            h[1, :] = np.nan
    dt = torch.bfloat16 if kind == "bf16" else torch.float32
    want_p = oracle.mask_pack(h, K, layer, step, batch)
    out_p = Guarded((rows, K), dt)
    so.mask_pack(dev(h), K, layer, step, batch, out=out_p.t)
    assert np.array_equal(host(out_p.t).view(np.uint8), want_p.view(np.uint8))
    assert out_p.intact()
    want_u = oracle.mask_unpack(want_p, H, layer, step, batch)
    out_u = Guarded((rows, H), dt)
    so.mask_unpack(dev(want_p), H, layer, step, batch, out=out_u.t)
    assert np.array_equal(host(out_u.t).view(np.uint8), want_u.view(np.uint8))
    assert out_u.intact()


def test_unaligned_buffers_take_the_row_path():
    rows, H, K = 24, 2048, 102
    h = synthetic.activations_bf16(rows, H, seed=5)
    big = torch.zeros(rows * H + 3, dtype=torch.bfloat16, device="cuda")
    view = big[1:1 + rows * H].view(rows, H)  # 2-byte offset: not 16-byte aligned
    view.copy_(dev(h))
    outbig = torch.zeros(rows * K + 5, dtype=torch.bfloat16, device="cuda")
    out = outbig[3:3 + rows * K].view(rows, K)
    so.mask_pack(view, K, 4, 4, 4, out=out)
    assert np.array_equal(host(out), oracle.mask_pack(h, K, 4, 4, 4))
    back = big[1:1 + rows * H].view(rows, H)
    so.mask_unpack(out, H, 4, 4, 4, out=back)
    assert np.array_equal(host(back), oracle.mask_unpack(oracle.mask_pack(h, K, 4, 4, 4), H, 4, 4, 4))


def test_backward_gradient_uses_the_forward_indices():
    rows, H, K, layer, step = 64, 256, 13, 3, 7
    g_up = synthetic.act_grads_f32(rows, H, seed=4)
    g_dev = so.mask_unpack(so.mask_pack(dev(g_up), K, layer, step), H, layer, step)
    m = oracle.mask_matrix(rows, H, K, layer, step)
    # torch autograd of h~ = h * m on the GPU gives the same gradient
    hh = torch.zeros(rows, H, device="cuda", requires_grad=True)
    (hh * torch.from_numpy(m.astype(np.float32)).cuda()).backward(dev(g_up))
    assert torch.equal(hh.grad, g_dev)
    assert (host(g_dev)[~m] == 0).all()


@pytest.mark.parametrize("p", [0.90, 0.95])
def test_full_stage_boundary_activation_bit_exact(p):
    # the mask sweep's boundary tensor: bf16 [32 * 2048, 2048]
    rows, H = 32 * 2048, 2048
    K = so.mask_keep_count(p, H)
    h = synthetic.activations_bf16(rows, H, seed=11)
    hd = dev(h)
    packed = so.mask_pack(hd, K, 7, 0, 0)
    want = oracle.mask_pack(h, K, 7, 0, 0)
    assert np.array_equal(host(packed), want)
    dense = so.mask_unpack(packed, H, 7, 0, 0)
    m = oracle.mask_matrix(rows, H, K, 7, 0, 0)
    got = host(dense)
    assert np.array_equal(got[m], h[m]) and not got[~m].any()
    assert packed.numel() * 2 * H / K == hd.numel() * 2 and (rows * H) / (rows * K) == H / K


def test_7b_width_activation_bit_exact():
    rows, H, K = 8 * 4096, 4096, 205
    h = synthetic.activations_bf16(rows, H, seed=12)
    packed = so.mask_pack(dev(h), K, 3, 1, 0)
    assert np.array_equal(host(packed), oracle.mask_pack(h, K, 3, 1, 0))
    got = host(so.mask_unpack(packed, H, 3, 1, 0))
    assert np.array_equal(got, oracle.mask_unpack(oracle.mask_pack(h, K, 3, 1, 0), H, 3, 1, 0))


def test_sender_and_receiver_calls_agree_across_streams():
    rows, H, K = 256, 2048, 102
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    with torch.cuda.stream(s1):
        a = so.mask_indices(rows, H, K, 5, 1234, 9)
    with torch.cuda.stream(s2):
        b = so.mask_indices(rows, H, K, 5, 1234, 9)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
