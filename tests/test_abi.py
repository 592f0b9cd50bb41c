"""The C-ABI library loads on any host and exports every symbol nnt.h declares;
argument validation runs before any device work (no GPU needed)."""
import ctypes as C

import pytest

from tile_task_transformer_gb300 import nnt


@pytest.fixture(scope="module")
def L():
    from tile_task_transformer_gb300 import build
    build.build()
    return nnt.lib()


def test_exports_every_declared_symbol(L):
    syms = nnt.header_symbols()
    assert "nnt_create_model" in syms and "nnt_forward" in syms and "nnt_adamw_step" in syms
    for s in syms:
        assert hasattr(L, s), s
    # and the binding declares a signature for each of them
    assert set(syms) == set(nnt._SIGS)


def _create(cfg, tiles=None):
    h = C.c_void_p()
    t = tiles or nnt.Tiles()
    st = nnt.lib().nnt_create_model(C.byref(cfg), C.byref(t), C.byref(nnt.Options()), C.byref(h))
    return st, h


@pytest.mark.parametrize("cfg,tiles,why", [
    (nnt.Config(2, 64, 4, 256, 256, 32, 2, 0, 1e-5), nnt.Tiles(0, 12, 0, 0, 0, 0), "seq_tile"),
    (nnt.Config(2, 64, 4, 256, 256, 32, 2, 0, 1e-5), nnt.Tiles(0, 0, 0, 0, 3, 0), "head_tile"),
    (nnt.Config(2, 64, 4, 256, 256, 32, 2, 0, 1e-5), nnt.Tiles(3, 0, 0, 0, 0, 0), "batch_tile"),
    (nnt.Config(2, 64, 5, 256, 256, 32, 2, 0, 1e-5), None, "d_model % n_head"),
    (nnt.Config(2, 64, 4, 256, 70000, 32, 2, 0, 1e-5), None, "vocab"),
    (nnt.Config(2, 64, 4, 256, 256, 32, 2, 7, 1e-5), None, "dtype"),
    (nnt.Config(2, 68, 4, 256, 256, 32, 2, 0, 1e-5), None, "multiple of 8"),
    (nnt.Config(2, 64, 4, 256, 256, 8192, 4, 0, 1e-5), None, "batch*n_ctx"),
])
def test_invalid_shapes_rejected_before_device_work(L, cfg, tiles, why):
    st, h = _create(cfg, tiles)
    assert st == nnt.ERR_INVALID_ARG, why
    assert h.value is None
    assert L.nnt_last_error(None)


def test_null_safety(L):
    L.nnt_destroy(None)
    assert L.nnt_num_params(None) == -1
    assert L.nnt_backward(None) == nnt.ERR_INVALID_ARG
    st = L.nnt_create_model(None, None, None, None)
    assert st == nnt.ERR_INVALID_ARG
