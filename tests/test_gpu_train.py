"""Minibatch gradient accumulation, learning-rate warm-up and multi-step
training through the C ABI (GPU).

README "Minimal working GPT example": --batch sequences per optimizer step,
processed --minibatch at a time, the step taken once the whole batch's
gradients are collected; --start-lr / --full-lr-iter ramp the rate up over the
first AdamW iterations. The oracle's batch_gradient / train_batch / train are
the plain definitions (mean of the minibatch gradients; straight-line warm-up).

Tolerances as for the single step: loss within 1e-3 absolute, gradients and
weights 2e-2 normwise (fp32 path: 1e-4, the fp32 rounding scale of the tiny
model).
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import gpt2 as O  # noqa: E402
from tile_task_transformer_gb300 import nnt, synth  # noqa: E402

pytestmark = pytest.mark.gpu

TINY = O.GPT2Config(n_layer=2, d_model=64, n_head=4, d_ff=256, vocab=256, seq=32, batch=2)
TINY_TILES = {"seq_tile": 16, "embd_tile": 32}
SMALL_TILES = {"seq_tile": 1024, "embd_tile": 768, "inner_tile": 3072, "head_tile": 12}
HP = dict(lr=1e-3, start_lr=1e-4, full_lr_iter=3)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nnt.lib()


def relerr(a, r):
    r = np.asarray(r, np.float64)
    return float(np.abs(np.asarray(a, np.float64) - r).max() / max(np.abs(r).max(), 1e-30))


def make(cfg, dtype, tiles, **kw):
    return nnt.Model(cfg.n_layer, cfg.d_model, cfg.n_head, cfg.d_ff, cfg.vocab, cfg.seq, cfg.batch,
                     dtype=dtype, tiles=tiles, **kw)


def minibatches(seed, k, cfg):
    return [synth.token_windows(seed * 100 + i, cfg.batch, cfg.seq, cfg.vocab) for i in range(k)]


def gpu_batch(m, mbs, **hp):
    """One optimizer step over the minibatches; returns (mean loss, mean gradient)."""
    losses = []
    for w in mbs:
        losses.append(m.forward(w))
        m.backward(accumulate=True)
    grads = {n: g / len(mbs) for n, g in m.grads().items()}  # the stored sum / k
    m.adamw_step(**hp)
    return sum(losses) / len(mbs), grads


@pytest.mark.parametrize("dtype,graph", [(nnt.F32, False), (nnt.F32, True), (nnt.BF16, True)])
def test_tiny_accumulated_batch_matches_oracle(dtype, graph):
    tol = 1e-4 if dtype == nnt.F32 else 2e-2
    params = synth.gpt2_params(5, TINY.n_layer, TINY.d_model, TINY.d_ff, TINY.vocab, TINY.seq)
    batches = [minibatches(s, 3, TINY) for s in (1, 2)]
    hp = O.AdamWHyper(**HP)
    m = make(TINY, dtype, TINY_TILES, use_cuda_graph=graph)
    m.set_params(params)
    p, mom1, mom2 = params, None, None
    moved = 0.0  # sum of the rates so far: the most one element can drift from a sign flip
    for step, mbs in enumerate(batches, start=1):
        moved += 2 * O.scheduled_lr(hp, step)
        loss, grads = gpu_batch(m, mbs, **HP)
        rloss, rgrads, p, mom1, mom2 = O.train_batch(TINY, p, mbs, hp, mom1, mom2, step)
        assert abs(loss - rloss) < (1e-5 if dtype == nnt.F32 else 1e-3), (step, loss, rloss)
        for n in rgrads:
            assert relerr(grads[n], rgrads[n]) < tol, (step, n, relerr(grads[n], rgrads[n]))
        got = m.params()
        for n in p:
            # weights after the step: normwise, plus the sign-flip allowance of
            # an unresolved near-zero gradient (each element moves ~lr per step)
            assert np.abs(got[n] - p[n]).max() <= moved * (1 + tol) + tol * np.abs(p[n]).max(), (step, n)
            m1 = m.get_adam_state(m.names.index(n), 0)
            assert relerr(m1, mom1[n]) < tol, (step, n)
    m.close()


def test_accumulating_one_minibatch_equals_plain_backward():
    """k = 1: nnt_backward_accumulate after an update is nnt_backward, bit for bit."""
    params = synth.gpt2_params(6, TINY.n_layer, TINY.d_model, TINY.d_ff, TINY.vocab, TINY.seq)
    win = synth.token_windows(6, TINY.batch, TINY.seq, TINY.vocab)
    out = []
    for acc in (False, True):
        m = make(TINY, nnt.BF16, TINY_TILES, use_cuda_graph=True)
        m.set_params(params)
        m.forward(win)
        m.backward(accumulate=acc)
        g = m.grads()
        m.adamw_step()
        out.append((g, m.params()))
        m.close()
    for n in out[0][0]:
        np.testing.assert_array_equal(out[0][0][n], out[1][0][n], err_msg=n)
        np.testing.assert_array_equal(out[0][1][n], out[1][1][n], err_msg=n)


def test_zero_start_rate_keeps_weights_and_call_order():
    """Warm-up from start_lr = 0: the first update leaves every weight
    bit-identical (lr multiplies both the decay and the Adam term) while the
    moments take the gradient; the second moves them. Call-order rules:
    nnt_backward_adamw refuses to run over pending accumulated gradients."""
    params = synth.gpt2_params(7, TINY.n_layer, TINY.d_model, TINY.d_ff, TINY.vocab, TINY.seq)
    m = make(TINY, nnt.F32, TINY_TILES)
    m.set_params(params)
    wins = minibatches(7, 2, TINY)
    m.forward(wins[0])
    m.backward(accumulate=True)
    m.forward(wins[1])
    with pytest.raises(nnt.NNTError) as e:
        m.backward_adamw()
    assert e.value.status == nnt.ERR_STATE
    m.backward(accumulate=True)
    g = m.grads()
    m.adamw_step(lr=3e-4, start_lr=0.0, full_lr_iter=4)
    new = m.params()
    for i, n in enumerate(m.names):
        np.testing.assert_array_equal(new[n], params[n], err_msg=n)
        # m = (1 - beta1) * mean gradient
        np.testing.assert_allclose(m.get_adam_state(i, 0), 0.1 * g[n] / 2, rtol=1e-6, atol=1e-30)
    with pytest.raises(nnt.NNTError) as e:
        m.adamw_step()  # gradients were consumed by the update
    assert e.value.status == nnt.ERR_STATE
    m.forward(wins[0])
    m.backward()
    m.adamw_step(lr=3e-4, start_lr=0.0, full_lr_iter=4)
    assert any(np.abs(m.get_param(i) - params[n]).max() > 0 for i, n in enumerate(m.names))
    m.close()


def test_tiny_training_run_loss_curve_matches_oracle():
    """Eight optimizer steps of two minibatches each, with warm-up, on a fixed
    synthetic stream: the GPU's per-step batch losses follow the oracle's."""
    params = synth.gpt2_params(8, TINY.n_layer, TINY.d_model, TINY.d_ff, TINY.vocab, TINY.seq)
    batches = [minibatches(20 + s, 2, TINY) for s in range(8)]
    hp = O.AdamWHyper(lr=2e-3, start_lr=0.0, full_lr_iter=3)
    rlosses, rfinal, _, _ = O.train(TINY, params, batches, hp)
    m = make(TINY, nnt.F32, TINY_TILES, use_cuda_graph=True)
    m.set_params(params)
    losses = [gpu_batch(m, mbs, lr=2e-3, start_lr=0.0, full_lr_iter=3)[0] for mbs in batches]
    final = m.params()
    m.close()
    print("loss curve gpu", np.round(losses, 5), "oracle", np.round(rlosses, 5))
    np.testing.assert_allclose(losses, rlosses, atol=1e-4)
    worst = max(rfinal, key=lambda n: relerr(final[n], rfinal[n]))
    print("largest normwise weight deviation after 8 steps", worst, relerr(final[worst], rfinal[worst]))
    for n in rfinal:
        assert relerr(final[n], rfinal[n]) < 1e-3, (n, relerr(final[n], rfinal[n]))


def test_gpt2_small_accumulated_minibatches_equal_one_big_batch():
    """GPT2-small shape, bf16: the mean of two 4-sequence minibatch gradients
    equals the gradient of the 8 sequences in one pass (the mean loss is linear
    in the per-token terms; the power-of-two normaliser keeps bf16 rounding
    alike), up to fp32 summation order."""
    cfg4 = O.GPT2Config(n_layer=12, d_model=768, n_head=12, d_ff=3072, vocab=50257, seq=1024, batch=4)
    cfg8 = O.GPT2Config(n_layer=12, d_model=768, n_head=12, d_ff=3072, vocab=50257, seq=1024, batch=8)
    w8 = synth.token_windows(9, 8, 1024, 50257)
    a = make(cfg4, nnt.BF16, SMALL_TILES, use_cuda_graph=True, n_streams=2, seed=3)
    l1 = a.forward(np.ascontiguousarray(w8[:4]))
    a.backward(accumulate=True)
    l2 = a.forward(np.ascontiguousarray(w8[4:]))
    a.backward(accumulate=True)
    ga = {n: g / 2 for n, g in a.grads().items()}
    a.close()
    b = make(cfg8, nnt.BF16, SMALL_TILES, use_cuda_graph=True, n_streams=2, seed=3)
    lb = b.forward(w8)
    b.backward()
    gb = b.grads()
    b.close()
    assert abs((l1 + l2) / 2 - lb) < 1e-4, ((l1 + l2) / 2, lb)
    worst = max(relerr(ga[n], gb[n]) for n in gb)
    print("worst normwise difference", worst)
    assert worst < 5e-3
