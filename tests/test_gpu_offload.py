"""Fused backward + AdamW and host offload of AdamW moments (GPU).

nnt_backward_adamw applies each chunk's AdamW update as soon as its gradient is
final. It runs the same kernels on the same values as nnt_backward followed by
nnt_adamw_step, so the weights and moments must agree bit for bit, also when a
small device budget forces part of the moments into pinned host memory and the
layer-matrix gradients through the ring.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from tile_task_transformer_gb300 import nnt, synth  # noqa: E402

pytestmark = pytest.mark.gpu

TINY = dict(n_layer=2, d_model=64, n_head=4, d_ff=256, vocab=256, n_ctx=32, batch=2)
TINY_TILES = {"seq_tile": 16, "embd_tile": 32}
SMALL = dict(n_layer=12, d_model=768, n_head=12, d_ff=3072, vocab=50257, n_ctx=1024, batch=4)
SMALL_TILES = {"seq_tile": 1024, "embd_tile": 768, "inner_tile": 3072, "head_tile": 12, "batch_tile": 4}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nnt.lib()


def make(cfg, tiles, dtype, **kw):
    return nnt.Model(cfg["n_layer"], cfg["d_model"], cfg["n_head"], cfg["d_ff"], cfg["vocab"],
                     cfg["n_ctx"], cfg["batch"], dtype=dtype, tiles=tiles, seed=11, **kw)


def state(m):
    return ({n: m.get_param(i) for i, n in enumerate(m.names)},
            {n: m.get_adam_state(i, 0) for i, n in enumerate(m.names)},
            {n: m.get_adam_state(i, 1) for i, n in enumerate(m.names)})


def run(m, wins, fused):
    losses = []
    for w in wins:
        losses.append(m.forward(w))
        if fused:
            m.backward_adamw()
        else:
            m.backward()
            m.adamw_step()
    return losses, state(m)


def compare(a, b):
    la, (pa, ma, va) = a
    lb, (pb, mb, vb) = b
    assert la == lb
    for n in pa:
        np.testing.assert_array_equal(pa[n], pb[n], err_msg=n)
        np.testing.assert_array_equal(ma[n], mb[n], err_msg=n)
        np.testing.assert_array_equal(va[n], vb[n], err_msg=n)


def offload_budget(cfg, tiles, dtype, **kw):
    """A device budget that holds everything except about half of the moments."""
    m = make(cfg, tiles, dtype, **kw)
    st = m.stats()
    m.close()
    n_flat_bytes = sum(int(np.prod(s)) for s in m.shapes) * 4
    return st["device_bytes"] - n_flat_bytes


@pytest.mark.parametrize("dtype", [nnt.F32, nnt.BF16])
def test_tiny_fused_equals_separate(dtype):
    wins = [synth.token_windows(s, TINY["batch"], TINY["n_ctx"], TINY["vocab"]) for s in (1, 2)]
    a = run(make(TINY, TINY_TILES, dtype), wins, fused=False)
    b = run(make(TINY, TINY_TILES, dtype), wins, fused=True)
    compare(a, b)


@pytest.mark.parametrize("dtype,graph", [(nnt.F32, False), (nnt.BF16, True)])
def test_tiny_offloaded_moments_equal_device_moments(dtype, graph):
    wins = [synth.token_windows(s, TINY["batch"], TINY["n_ctx"], TINY["vocab"]) for s in (3, 4, 5)]
    budget = offload_budget(TINY, TINY_TILES, dtype)
    ref = run(make(TINY, TINY_TILES, dtype, use_cuda_graph=graph), wins, fused=False)
    m = make(TINY, TINY_TILES, dtype, allow_host_offload=True, hbm_budget_bytes=budget,
             use_cuda_graph=graph)
    st = m.stats()
    assert st["offload_active"] == 1 and st["host_pinned_bytes"] > 0
    # whole gradients are not kept in this mode
    m.forward(wins[0])
    with pytest.raises(nnt.NNTError) as e:
        m.backward()
    assert e.value.status == nnt.ERR_STATE
    m.close()
    m = make(TINY, TINY_TILES, dtype, allow_host_offload=True, hbm_budget_bytes=budget,
             use_cuda_graph=graph)
    got = run(m, wins, fused=True)
    assert m.stats()["h2d_bytes"] > 0  # moments read over the host link
    with pytest.raises(nnt.NNTError) as e:
        m.get_grad(m.names.index("h0.fc.w"))
    assert e.value.status == nnt.ERR_STATE
    m.close()
    compare(ref, got)


def test_gpt2_small_offloaded_fused_step_equals_separate():
    wins = [synth.token_windows(s, SMALL["batch"], SMALL["n_ctx"], SMALL["vocab"]) for s in (6, 7)]
    kw = dict(use_cuda_graph=True, n_streams=2)
    ref = run(make(SMALL, SMALL_TILES, nnt.BF16, **kw), wins, fused=False)
    budget = offload_budget(SMALL, SMALL_TILES, nnt.BF16, **kw)
    m = make(SMALL, SMALL_TILES, nnt.BF16, allow_host_offload=True, hbm_budget_bytes=budget, **kw)
    assert m.stats()["offload_active"] == 1
    got = run(m, wins, fused=True)
    m.close()
    compare(ref, got)
