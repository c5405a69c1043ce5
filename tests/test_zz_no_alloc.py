"""The no-allocation entry point, specoptim_filter_noalloc.

It serves callers that cannot call cudaMalloc (code inside a framework that
owns all device memory through its own pool, or on a latency-critical path
that cannot take the device synchronisation of an allocation): its
intermediates live in a 16 MiB static device array instead of memory the
library allocates.  The test calls it through the C-ABI and checks its
filtered gradient against the one the allocating entry point
(specoptim_step with a G_filt output) produces for the same factors and
gradient, on two calls in a row, within the TF32 tolerance of the parity tests
(relative Frobenius error 2e-3).  It also checks that a shape whose
intermediates do not fit in the array is rejected with a clear error.

This file is collected last so that a failure here, in a run that stops at the
first failure, comes after every other test has run.
"""
import numpy as np
import pytest
import torch

import spectral_corrected_optimizer_gb300 as so
import synthetic
from gpu_util import dev, ensure_lib, host, rel

pytestmark = pytest.mark.gpu

TOL = 2e-3


@pytest.mark.parametrize("shape", [(512, 2048), (256, 128)])
def test_noalloc_filter_matches_the_step(shape):
    ensure_lib()
    lib = so.lib()
    m, n = shape
    inp = synthetic.MatrixInputs(m, n, seed=21, rank=8)
    opt = so.SpectralOptimizer(m, n)
    opt.anchor_update(dev(inp.anchor_grad(0)))
    opt.svd_refresh()
    U, s, V, d = opt.get_factors()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        G = dev(inp.masked_grad(call))
        ref = torch.empty(m, n, device="cuda")
        opt.step(dev(inp.weights()), G, 2e-5, G_filt_out=ref)
        out = torch.full((m, n), float("nan"), device="cuda")
        rc = lib.specoptim_filter_noalloc(U.data_ptr(), V.data_ptr(), d.data_ptr(), G.data_ptr(),
                                          out.data_ptr(), m, n, so.PREC_TF32, stream)
        assert rc == so.OK, lib.specoptim_last_error()
        torch.cuda.synchronize()
        assert np.isfinite(host(out)).all()
        assert rel(host(out), host(ref)) <= TOL


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
