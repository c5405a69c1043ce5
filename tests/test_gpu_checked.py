"""The checked build (-DSPECOPTIM_CHECK) on the small mask cases.

In the checked build every mask kernel (pack, unpack, indices and the four ops
fused with the layer boundary) verifies that each kept index it computes lies
below H -- the invariant the keyed permutation and its cycle walking guarantee
(key design 1: exactly K dims of [0, H) per token) -- before it reads or
writes with it; a failure skips the access and surfaces as
SPECOPTIM_ERR_BOUNDS from specoptim_check_device.  These tests run the checked
library on the small and ragged cases (H = 3000 walks cycles; K = 0, 1, H)
and require both the oracle's exact bytes and a clean check, with the output
buffers between guard bytes.
"""
import numpy as np
import pytest
import torch

import oracle
import spectral_corrected_optimizer_gb300 as so
import synthetic
from gpu_util import Guarded, dev, host

pytestmark = pytest.mark.gpu

CASES = [(64, 256, 13, 3, 7), (37, 2048, 102, 0, 0), (45, 3000, 150, 2, 2), (19, 4096, 205, 1, 9),
         (9, 7, 7, 0, 1), (17, 96, 1, 5, 5), (5, 64, 0, 0, 0)]


@pytest.fixture(scope="module")
def chk():
    from spectral_corrected_optimizer_gb300 import build as sob
    return so.load(sob.build(check=True))


def stream():
    return torch.cuda.current_stream().cuda_stream


def clean(lib):
    rc = lib.specoptim_check_device(stream())
    assert rc == so.OK, lib.specoptim_last_error()


@pytest.mark.parametrize("rows,H,K,layer,step", CASES)
def test_checked_mask_ops(chk, rows, H, K, layer, step):
    h = synthetic.activations_bf16(rows, H, seed=rows)
    hd = dev(h)
    idx = Guarded((rows, K), torch.int32)
    assert chk.mask_indices(idx.t.data_ptr(), rows, H, K, layer, step, 0, stream()) == so.OK
    packed = Guarded((rows, K), torch.bfloat16)
    assert chk.mask_pack(hd.data_ptr(), packed.t.data_ptr(), rows, H, K, 2, layer, step, 0, stream()) == so.OK
    dense = Guarded((rows, H), torch.bfloat16)
    assert chk.mask_unpack(packed.t.data_ptr(), dense.t.data_ptr(), rows, H, K, 2, layer, step, 0,
                           stream()) == so.OK
    clean(chk)
    assert np.array_equal(host(idx.t), oracle.mask_indices(rows, H, K, layer, step))
    want = oracle.mask_pack(h, K, layer, step)
    assert np.array_equal(host(packed.t), want)
    assert np.array_equal(host(dense.t), oracle.mask_unpack(want, H, layer, step))
    assert idx.intact() and packed.intact() and dense.intact()


@pytest.mark.parametrize("rows,H,K,layer,step", [c for c in CASES if c[2] > 0])
def test_checked_fused_mask_ops(chk, rows, H, K, layer, step):
    a = synthetic.activations_bf16(rows, H, seed=1, index=rows)
    b = synthetic.activations_bf16(rows, H, seed=2, index=rows)
    gamma = synthetic.activations_bf16(1, H, seed=3)[0]
    da, db, dg = dev(a), dev(b), dev(gamma)
    packed = Guarded((rows, K), torch.bfloat16)
    assert chk.mask_pack_add(da.data_ptr(), db.data_ptr(), packed.t.data_ptr(), rows, H, K, layer, step, 0,
                             stream()) == so.OK
    h_out, x_out = Guarded((rows, H), torch.bfloat16), Guarded((rows, H), torch.bfloat16)
    assert chk.mask_unpack_rmsnorm(packed.t.data_ptr(), dg.data_ptr(), 1e-5, h_out.t.data_ptr(),
                                   x_out.t.data_ptr(), rows, H, K, layer, step, 0, stream()) == so.OK
    grad = Guarded((rows, K), torch.bfloat16)
    assert chk.mask_rmsnorm_backward_pack(packed.t.data_ptr(), dg.data_ptr(), 1e-5, da.data_ptr(),
                                          db.data_ptr(), grad.t.data_ptr(), rows, H, K, layer, step, 0,
                                          stream()) == so.OK
    g = Guarded((rows, H), torch.bfloat16)
    g.t.copy_(db)
    assert chk.mask_unpack_add(packed.t.data_ptr(), g.t.data_ptr(), rows, H, K, layer, step, 0,
                               stream()) == so.OK
    clean(chk)
    want = oracle.mask_pack_add(a, b, K, layer, step)
    assert np.array_equal(host(packed.t), want)
    h_ref, _, _ = oracle.mask_unpack_rmsnorm(want, gamma, 1e-5, H, layer, step)
    assert np.array_equal(host(h_out.t), h_ref)
    assert np.array_equal(host(g.t), oracle.mask_unpack_add(want, b, layer, step))
    assert all(x.intact() for x in (packed, h_out, x_out, grad, g))
