"""The allocation plan nnt_create_model checks before allocating (CPU).

nnt_plan_memory runs the model's allocation plan without allocating; with a
device budget given it needs no GPU. These tests pin its byte counts to the
closed forms of the parameter state and of the host offload of AdamW moments.
"""
import pytest

from tile_task_transformer_gb300 import nnt, synth

GIB = 1 << 30


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from tile_task_transformer_gb300 import build
    build.build()
    nnt.lib()


def n_params(L, d, f, V, S):
    return sum(int(__import__("numpy").prod(sh)) for _, sh in synth.param_names_shapes(L, d, f, V, S))


def test_resident_plan_holds_the_parameter_state_on_the_device():
    # fp32 master, gradient, m, v and the bf16 copy: 18 bytes per parameter
    # (each tensor padded to 64 elements), plus activations
    L, d, H, f, V, S, B = 12, 768, 12, 3072, 50257, 1024, 4
    dev, host = nnt.plan_memory(L, d, H, f, V, S, B, hbm_budget_bytes=200 * GIB)
    n = n_params(L, d, f, V, S)
    assert host == 64  # the pinned loss word only
    assert 18 * n <= dev <= 18 * n + 8 * GIB


def test_offload_plan_moves_moments_to_pinned_host_memory():
    # wide-8: 26.6B parameters, fp32 state 426 GB: with offload the moments
    # that do not fit the device budget go to pinned host memory
    L, d, H, f, V, S, B = 8, 16384, 128, 65536, 50257, 1024, 4
    n = n_params(L, d, f, V, S)
    budget = 280 * GIB
    dev, host = nnt.plan_memory(L, d, H, f, V, S, B, allow_host_offload=True, hbm_budget_bytes=budget)
    assert dev <= budget
    assert host > 0 and host <= 8 * n + 64
    # every moment lives either on the device or on the host
    dev_all, _ = nnt.plan_memory(L, d, H, f, V, S, B, allow_host_offload=True, hbm_budget_bytes=1)
    _, host_all = nnt.plan_memory(L, d, H, f, V, S, B, allow_host_offload=True, hbm_budget_bytes=1)
    assert host_all >= 8 * n and host_all <= 8 * n + 8 * 64 * 4 * L * 12 + 64 + 8 * GIB // 1024
    assert abs((dev + host) - (dev_all + host_all)) <= 1024  # two minimum-size moment buffers
    # without offload everything stays on the device, whatever the budget
    dev_res, host_res = nnt.plan_memory(L, d, H, f, V, S, B, hbm_budget_bytes=budget)
    assert host_res == 64 and dev_res > 18 * n


def test_plan_rejects_invalid_shapes():
    with pytest.raises(nnt.NNTError) as e:
        nnt.plan_memory(2, 64, 5, 256, 256, 32, 2, hbm_budget_bytes=GIB)
    assert e.value.status == nnt.ERR_INVALID_ARG
