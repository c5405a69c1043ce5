"""The no-allocation entry point, specoptim_filter_noalloc.

It serves callers that cannot call cudaMalloc (code inside a framework that
owns all device memory through its own pool, or on a latency-critical path
that cannot take the device synchronisation of an allocation): its
intermediates live in a 16 MiB static device array instead of memory the
library allocates.

The tests call it through the C-ABI with the factors of a real refresh,
copied out, and check its filtered gradient, on two calls in a row, against
the filtered gradient the allocating entry point (specoptim_step with a
G_filt output) gives for the same factors and gradient, within the parity
tests' TF32 bar (relative Frobenius error 2e-3), and against the oracle's
projection (key design 3, projection equation, float64) of the same factors
and gradient: 2e-3 for TF32, 1e-4 for fp32.  Both precisions; wide, tall,
square and ragged shapes (r = 66 is not a multiple of 4, so the tensor-core
path hands those products to the SIMT kernel).  They also check that a call
allocates no device memory and that a shape whose intermediates do not fit
in the array is rejected with a clear error.

This file is collected last so that a failure here, in a run that stops at the
first failure, comes after every other test has run.
"""
import numpy as np
import pytest
import torch

import oracle
import spectral_corrected_optimizer_gb300 as so
import synthetic
from gpu_util import dev, ensure_lib, host, rel

pytestmark = pytest.mark.gpu

TOL = {so.PREC_TF32: 2e-3, so.PREC_FP32: 1e-4}


def noalloc(U, V, d, G, out, m, n, prec):
    lib = so.lib()
    rc = lib.specoptim_filter_noalloc(U.data_ptr(), V.data_ptr(), d.data_ptr(), G.data_ptr(),
                                      out.data_ptr(), m, n, prec, torch.cuda.current_stream().cuda_stream)
    assert rc == so.OK, lib.specoptim_last_error()


@pytest.mark.parametrize("prec", [so.PREC_TF32, so.PREC_FP32])
@pytest.mark.parametrize("shape", [(512, 2048), (2048, 512), (256, 128), (256, 256), (130, 66)])
def test_noalloc_filter_matches_the_oracle(shape, prec):
    ensure_lib()
    m, n = shape
    inp = synthetic.MatrixInputs(m, n, seed=21, rank=8)
    opt = so.SpectralOptimizer(m, n)
    opt.anchor_update(dev(inp.anchor_grad(0)))
    opt.svd_refresh()
    U, s, V, d = opt.get_factors()
    Uh, Vh, dh = (host(x).astype(np.float64) for x in (U, V, d))
    for call in range(2):
        Gh = inp.masked_grad(call)
        G = dev(Gh)
        ref = torch.empty(m, n, device="cuda")
        opt.step(dev(inp.weights()), G, 2e-5, G_filt_out=ref)  # the allocating entry point
        out = torch.full((m, n), float("nan"), device="cuda")
        noalloc(U, V, d, G, out, m, n, prec)
        torch.cuda.synchronize()
        got = host(out)
        assert np.isfinite(got).all()
        assert rel(got, host(ref)) <= TOL[so.PREC_TF32], (call, rel(got, host(ref)))
        want = oracle.project(Uh, Vh, dh, Gh.astype(np.float64))[2]
        assert rel(got, want) <= TOL[prec], (call, rel(got, want))
    opt.close()


def test_noalloc_call_allocates_no_device_memory():
    ensure_lib()
    m, n = 512, 2048
    inp = synthetic.MatrixInputs(m, n, seed=22, rank=8)
    rng = np.random.default_rng(5)
    U = dev(np.linalg.qr(rng.standard_normal((m, m)))[0].astype(np.float32))  # m x m orthonormal
    V = dev(np.linalg.qr(rng.standard_normal((n, m)))[0].astype(np.float32))  # n x m orthonormal
    d = torch.rand(m, device="cuda")
    G = dev(inp.masked_grad(0))
    out = torch.empty(m, n, device="cuda")
    noalloc(U, V, d, G, out, m, n, so.PREC_TF32)  # first call on the device: symbol lookup
    first = out.clone()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(2):
        noalloc(U, V, d, G, out, m, n, so.PREC_TF32)
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert free1 == free0
    assert torch.equal(out, first)  # the shared array keeps nothing a later call depends on


def test_noalloc_rejects_shapes_beyond_the_scratch():
    ensure_lib()
    lib = so.lib()
    m = n = 2048
    t = torch.zeros(m * n, device="cuda")
    v = torch.zeros(m, device="cuda")
    rc = lib.specoptim_filter_noalloc(t.data_ptr(), t.data_ptr(), v.data_ptr(), t.data_ptr(),
                                      t.data_ptr(), m, n, so.PREC_TF32, None)
    assert rc == so.ERR_INVALID_ARG
    assert b"scratch" in lib.specoptim_last_error()
