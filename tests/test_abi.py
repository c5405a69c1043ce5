"""The C-ABI library builds for sm_103a, loads without a GPU, exports every
entry point that include/*.h declares, and validates arguments on the host
(no compute call here: these run on machines without a GPU)."""
import ctypes
import glob
import os
import re

import pytest

import oracle
import spectral_corrected_optimizer_gb300 as so
from spectral_corrected_optimizer_gb300 import build as sob

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    sob.build()
    return so.lib()


def declared_functions():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\**\s*([A-Za-z_]\w*)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 15
    for name in names:
        assert hasattr(lib, name), name
    # and the binding declares a signature for each of them
    assert {s[0] for s in so.SIGNATURES} == set(names)


def test_keep_count_matches_oracle(lib):
    for p in (0.0, 0.5, 0.9, 0.95, 0.99, 1.0):
        for H in (1, 2, 7, 256, 2048, 3000, 4096):
            assert so.mask_keep_count(p, H) == oracle.mask_K(p, H)
    assert so.mask_keep_count(-0.1, 10) == -1 and so.mask_keep_count(0.5, 0) == -1


def test_mask_argument_errors_are_reported_without_a_gpu(lib):
    vp = ctypes.c_void_p(16)
    assert lib.mask_pack(vp, vp, 4, 8, 9, 2, 0, 0, 0, None) == so.ERR_INVALID_ARG   # K > H
    assert b"K outside" in lib.specoptim_last_error()
    assert lib.mask_pack(vp, vp, 4, 8, 2, 3, 0, 0, 0, None) == so.ERR_INVALID_ARG   # elem_bytes
    assert lib.mask_unpack(vp, vp, -1, 8, 2, 2, 0, 0, 0, None) == so.ERR_INVALID_ARG
    assert lib.mask_indices(None, 4, 8, 2, 0, 0, 0, None) == so.ERR_INVALID_ARG
    # empty work is a no-op success
    assert lib.mask_pack(None, None, 0, 8, 2, 2, 0, 0, 0, None) == so.OK


def test_config_defaults_are_the_pages_recipe(lib):
    cfg = so.config_default(256, 128)
    assert (cfg.m, cfg.n) == (256, 128)
    assert cfg.tau_p == pytest.approx(1e-3) and cfg.alpha == pytest.approx(0.3)
    assert cfg.beta_anc == pytest.approx(0.9)
    assert cfg.precision == so.PREC_TF32


@pytest.mark.parametrize("field,value", [("m", 0), ("tau_p", 0.0), ("alpha", 1.5), ("beta2", 1.0),
                                         ("precision", 7), ("svd_max_sweeps", 0)])
def test_create_rejects_bad_config_before_touching_the_gpu(lib, field, value):
    cfg = so.config_default(16, 8)
    setattr(cfg, field, value)
    h = ctypes.c_void_p()
    assert lib.specoptim_create(ctypes.byref(h), ctypes.byref(cfg), None) == so.ERR_INVALID_ARG
    assert h.value is None


def test_null_handles_are_rejected(lib):
    assert lib.specoptim_step(None, None, None, 1e-3, None, None, None) == so.ERR_INVALID_ARG
    assert lib.specoptim_svd_refresh(None, None, None) == so.ERR_INVALID_ARG
    assert lib.specoptim_destroy(None) == so.OK


def test_dpsync_rank_matches_the_oracle(lib):
    for m, n in [(2048, 2048), (512, 2048), (8192, 2048), (2048, 8192), (14336, 4096), (256, 128),
                 (4, 4), (1, 7), (100, 3)]:
        assert lib.dpsync_rank(m, n, 64.0) == oracle.dpsync_rank(m, n, 64.0)
    assert lib.dpsync_rank(0, 4, 64.0) == -1 and lib.dpsync_rank(4, 4, 0.0) == -1


@pytest.mark.parametrize("field,value", [("m", 0), ("n", 6), ("rank", 65), ("rank", -1), ("mix", 1.5)])
def test_dpsync_create_rejects_bad_config_before_touching_the_gpu(lib, field, value):
    cfg = so.DPConfig()
    assert lib.dpsync_config_default(ctypes.byref(cfg), 256, 128) == so.OK
    assert (cfg.ratio, cfg.error_feedback, cfg.mix) == (64.0, 1, 0.0)
    setattr(cfg, field, value)
    h = ctypes.c_void_p()
    dummy = ctypes.c_void_p(1 << 20)
    assert lib.dpsync_create(ctypes.byref(h), ctypes.byref(cfg), dummy, dummy, None) == so.ERR_INVALID_ARG
    assert h.value is None
    assert lib.dpsync_compress_p_many(None, 1, None, None, None) == so.ERR_INVALID_ARG


def test_binding_refuses_tensors_it_cannot_pass_as_device_pointers(lib):
    # the binding checks device, dtype, shape and element size before any
    # pointer reaches the library (a host tensor would otherwise be read by a kernel)
    torch = pytest.importorskip("torch")
    h = torch.zeros(4, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        so.mask_pack(h, 2, 0, 0)
    with pytest.raises(ValueError, match="CUDA"):
        so.mask_unpack(torch.zeros(4, 2, dtype=torch.bfloat16), 8, 0, 0)
    with pytest.raises(ValueError, match="shape"):
        so.mask_pack(h, 2, 0, 0, out=torch.zeros(4, 3, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="2- or 4-byte"):
        so._elem_bytes(torch.zeros(4, 8, dtype=torch.float64))
    with pytest.raises(ValueError, match="float32"):
        so._f32_2d(torch.zeros(2, 3, dtype=torch.float64), (2, 3), "W")
    with pytest.raises(ValueError, match="float32"):
        so._f32_2d(torch.zeros(3, 2), (2, 3), "W")
    with pytest.raises(ValueError, match="CUDA"):
        so._f32_2d(torch.zeros(2, 3), (2, 3), "W")


def test_refresh_begin_end_argument_errors_without_a_gpu(lib):
    null = (ctypes.c_void_p * 1)(None)
    assert lib.specoptim_svd_refresh_begin(None, 1, None) == so.ERR_INVALID_ARG
    assert lib.specoptim_svd_refresh_begin(null, 1, None) == so.ERR_INVALID_ARG
    assert lib.specoptim_svd_refresh_begin(null, 0, None) == so.ERR_INVALID_ARG
    assert lib.specoptim_svd_refresh_end(None, 1, None, None) == so.ERR_INVALID_ARG
    assert lib.specoptim_svd_refresh_end(null, 17, None, None) == so.ERR_INVALID_ARG
    assert b"handle" in lib.specoptim_last_error()
