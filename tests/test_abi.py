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
    (nnt.Config(2, 64, 4, 256, 256, 8192, 129, 0, 1e-5), None, "batch*n_ctx"),  # > 2^20 tokens
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


# Stand-alone tile tasks: invalid arguments are rejected before any device work,
# so these run without a GPU (the pointers are never dereferenced).
P = 4096  # a non-NULL stand-in address


@pytest.mark.parametrize("call,why", [
    (lambda: nnt.op_flash_attention_fwd(P, P, P, P, P, 2, 128, 32), "head size 32 has no fused kernel"),
    (lambda: nnt.op_flash_attention_fwd(P, None, P, P, P, 2, 128, 64), "NULL k"),
    (lambda: nnt.op_flash_attention_bwd(P, P, P, P, P, P, P, P, P, 0, 128, 64), "Z = 0"),
    (lambda: nnt.op_cross_entropy(P, 0, 100, 100, P, 1, P, 100, P, P, nnt.F32), "no rows"),
    (lambda: nnt.op_cross_entropy(P, 4, 0, 4, P, 1, P, 4, P, P, nnt.F32), "no columns"),
    (lambda: nnt.op_cross_entropy(P, 4, 100, 100, P, 1, P, 100, P, P, 5), "dtype"),
    (lambda: nnt.op_gemm(P, 8, 0, P, 8, 1, P, 16, nnt.F32, 16, 16, 16), "lda < K"),
    (lambda: nnt.op_gemm(P, 16, 0, P, 16, 1, P, 16, nnt.F32, 16, 16, 16, beta=0.5), "beta 0.5"),
    (lambda: nnt.op_gemm(P, 16, 0, P, 16, 1, P, 16, nnt.BF16, 16, 16, 16, beta=1.0), "beta 1 with bf16 C"),
    (lambda: nnt.op_adamw(P, P, P, P, None, 10, 3e-4, 0.9, 0.999, 0.0, 0.1, 0.1, 0.001), "eps 0"),
    (lambda: nnt.op_adamw(P, P, P, P, None, 10, 3e-4, 0.9, 0.999, 1e-8, 0.1, 0.0, 0.001), "bc1 0"),
    (lambda: nnt.op_embedding_fwd(P, 32, P, P, P, 2, 32, 64, 70000), "vocab over uint16"),
    (lambda: nnt.op_embedding_fwd(P, 16, P, P, P, 2, 32, 64, 256), "ids stride < seq"),
    (lambda: nnt.op_layernorm_fwd(P, P, P, P, P, P, 4, 40000, 1e-5, nnt.F32), "cols > 32768"),
    (lambda: nnt.op_gelu_fwd(P, P, 10, 9), "dtype"),
])
def test_op_arguments_rejected_before_device_work(L, call, why):
    with pytest.raises(nnt.NNTError) as e:
        call()
    assert e.value.status == nnt.ERR_INVALID_ARG, why
    assert L.nnt_last_error(None)


def test_fault_injection_arguments_checked_on_host(L):
    assert L.nnt_set_fault_injection(4, 1) == nnt.ERR_INVALID_ARG
    assert L.nnt_set_fault_injection(-1, 1) == nnt.ERR_INVALID_ARG
    assert L.nnt_set_fault_injection(nnt.FAULT_COPY, -2) == nnt.ERR_INVALID_ARG
    for k in range(4):  # arm and disarm: host-only, no device call
        assert L.nnt_set_fault_injection(k, 3) == nnt.OK
        assert L.nnt_set_fault_injection(k, 0) == nnt.OK


def test_wait_selftest_limit_checked_before_device_work(L):
    assert L.nnt_op_wait_selftest(999, 0, None) == nnt.ERR_INVALID_ARG
    assert L.nnt_op_wait_selftest(1_000_000_001, 0, None) == nnt.ERR_INVALID_ARG
