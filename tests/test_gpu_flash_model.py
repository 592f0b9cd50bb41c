"""The training step with fused attention tile tasks (README --flashattention)
against the oracle, and against the step with materialised scores (GPU).

Configurations with head size 64 (and 128) in bf16 use the fused tasks by
default; the sequence length 320 leaves a ragged 64-row tail in the last
128-query block. Tolerances are the step's: loss within 1e-3, gradients and
updated weights 2e-2 normwise.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import gpt2 as O  # noqa: E402
from tile_task_transformer_gb300 import nnt, synth  # noqa: E402

pytestmark = pytest.mark.gpu

MID = O.GPT2Config(n_layer=2, d_model=256, n_head=4, d_ff=1024, vocab=512, seq=320, batch=2)
MID128 = O.GPT2Config(n_layer=1, d_model=256, n_head=2, d_ff=512, vocab=384, seq=192, batch=2)
TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nnt.lib()


def relerr(a, r):
    r = np.asarray(r, np.float64)
    return float(np.abs(np.asarray(a, np.float64) - r).max() / max(np.abs(r).max(), 1e-30))


def make(cfg, tiles=None, **kw):
    return nnt.Model(cfg.n_layer, cfg.d_model, cfg.n_head, cfg.d_ff, cfg.vocab, cfg.seq, cfg.batch,
                     dtype=nnt.BF16, tiles=tiles or {}, **kw)


def gpu_step(cfg, params, win, tiles=None, **kw):
    m = make(cfg, tiles, **kw)
    m.set_params(params)
    flash = m.stats()["flash_attention"]
    loss = m.forward(win)
    m.backward()
    grads = m.grads()
    m.adamw_step()
    new = m.params()
    m.close()
    return flash, loss, grads, new


@pytest.mark.parametrize("cfg,tiles", [
    (MID, {}),
    (MID, {"seq_tile": 160, "head_tile": 2, "batch_tile": 1}),
    (MID128, {"seq_tile": 64}),
])
def test_flash_step_matches_oracle(cfg, tiles):
    params = synth.gpt2_params(21, cfg.n_layer, cfg.d_model, cfg.d_ff, cfg.vocab, cfg.seq)
    win = synth.token_windows(21, cfg.batch, cfg.seq, cfg.vocab)
    flash, loss, grads, new = gpu_step(cfg, params, win, tiles, use_cuda_graph=True)
    assert flash == 1
    rloss, rgrads, rnew, _, _ = O.train_step(cfg, params, win)
    assert abs(loss - rloss) < 1e-3, (loss, rloss)
    worst = 0.0
    for n in rgrads:
        e = relerr(grads[n], rgrads[n])
        worst = max(worst, e)
        assert e < TOL, (n, e)
        bound = 2 * 3e-4 * (1 + TOL) + TOL * np.abs(rnew[n]).max()
        assert np.abs(new[n] - rnew[n]).max() <= bound, n
    print("worst normwise gradient error", worst)


def test_flash_and_materialised_attention_agree():
    cfg = MID
    params = synth.gpt2_params(22, cfg.n_layer, cfg.d_model, cfg.d_ff, cfg.vocab, cfg.seq)
    win = synth.token_windows(22, cfg.batch, cfg.seq, cfg.vocab)
    fa, la, ga, _ = gpu_step(cfg, params, win, flash_attention=1)
    fb, lb, gb, _ = gpu_step(cfg, params, win, flash_attention=-1)
    assert (fa, fb) == (1, 0)
    assert abs(la - lb) < 1e-3
    for n in ga:
        assert relerr(ga[n], gb[n]) < TOL, n


def test_flash_required_but_unusable_is_rejected():
    tiny = O.GPT2Config(n_layer=1, d_model=64, n_head=4, d_ff=128, vocab=64, seq=32, batch=1)
    with pytest.raises(nnt.NNTError) as e:
        make(tiny, flash_attention=1)  # head size 16
    assert e.value.status == nnt.ERR_INVALID_ARG
    m = make(tiny)  # auto: falls back to materialised scores
    assert m.stats()["flash_attention"] == 0
    m.close()


def test_flash_saves_the_score_buffers():
    cfg = MID
    a = make(cfg, flash_attention=1)
    b = make(cfg, flash_attention=-1)
    saved = b.stats()["device_bytes"] - a.stats()["device_bytes"]
    a.close()
    b.close()
    B, H, S, L = cfg.batch, cfg.n_head, cfg.seq, cfg.n_layer
    # P per layer (bf16) and one fp32 score buffer, less the per-layer lse, D and
    # the one bf16 dS^T buffer of the fused backward
    expect = L * B * H * S * S * 2 + B * H * S * S * 4 - (L + 1) * B * H * S * 4 - B * H * S * S * 2
    assert abs(saved - expect) <= 4096 * (L + 2), (saved, expect)
