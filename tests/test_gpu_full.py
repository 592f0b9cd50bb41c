"""Parity at the benchmark sizes, in the benchmark's launch configuration (GPU).

* GPT2-small shape (12 x 768, vocab 50257, 4 x 1024 tokens, tiles of the
  NNTile README example): the whole step against the fp64 oracle.
* wide-4 (4 x 8192, 64 heads, d_ff 32768, 8 x 1024 tokens, 3.6B parameters):
  the batch holds two distinct sequences four times each, so the loss, the
  gradients and the AdamW update equal those of the two sequences alone, which
  the oracle computes; with wte = 0 every logit is 0 and the loss is ln V
  exactly.
"""
import json
import math
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import gpt2 as O  # noqa: E402
from tile_task_transformer_gb300 import nnt, synth  # noqa: E402

pytestmark = pytest.mark.gpu

SMALL = O.GPT2Config(n_layer=12, d_model=768, n_head=12, d_ff=3072, vocab=50257, seq=1024, batch=4)
SMALL_TILES = {"seq_tile": 1024, "embd_tile": 768, "inner_tile": 3072, "head_tile": 12, "batch_tile": 4}
WIDE4 = O.GPT2Config(n_layer=4, d_model=8192, n_head=64, d_ff=32768, vocab=50257, seq=1024, batch=8)
WIDE4_TILES = {"seq_tile": 1024, "embd_tile": 2048, "inner_tile": 4096, "head_tile": 16}
TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nnt.lib()


def relerr(a, r):
    """Normwise relative error in the max norm: max|a - r| / max|r|."""
    r = np.asarray(r, np.float64)
    return float(np.abs(np.asarray(a, np.float64) - r).max() / max(np.abs(r).max(), 1e-30))


def relerr2(a, r):
    """Normwise relative error in the 2-norm: ||a - r|| / ||r||."""
    r = np.asarray(r, np.float64)
    return float(np.linalg.norm(np.asarray(a, np.float64) - r) / max(np.linalg.norm(r), 1e-30))


def make(cfg, tiles, **kw):
    return nnt.Model(cfg.n_layer, cfg.d_model, cfg.n_head, cfg.d_ff, cfg.vocab, cfg.seq, cfg.batch,
                     dtype=nnt.BF16, tiles=tiles, use_cuda_graph=True, n_streams=2, **kw)


def test_gpt2_small_full_step_matches_oracle():
    cfg = SMALL
    params = synth.gpt2_params(1, cfg.n_layer, cfg.d_model, cfg.d_ff, cfg.vocab, cfg.seq)
    win = synth.token_windows(1, cfg.batch, cfg.seq, cfg.vocab)
    m = make(cfg, SMALL_TILES)
    m.set_params(params)
    loss = m.forward(win)
    m.backward()
    grads = m.grads()
    m.adamw_step()
    new = m.params()
    mom1 = {n: m.get_adam_state(i, 0) for i, n in enumerate(m.names)}
    m.close()
    rloss, rgrads, rnew, rm, _ = O.train_step(cfg, params, win)
    assert abs(loss - rloss) < 1e-3, (loss, rloss)
    worst = _step_checks(grads, new, mom1, params, rgrads, rnew, rm)
    print("worst normwise grad error", max(worst.values()))


def test_wide4_zero_embedding_loss_is_log_vocab():
    cfg = WIDE4
    m = make(cfg, WIDE4_TILES, seed=7)
    m.set_param(0, np.zeros((cfg.vocab, cfg.d_model), np.float32))
    loss = m.forward(synth.token_windows(7, cfg.batch, cfg.seq, cfg.vocab))
    m.close()
    assert abs(loss - math.log(cfg.vocab)) < 1e-4


def _step_checks(grads, new, mom1, params, rgrads, rnew, rm, norm=relerr, spread=None):
    """Normwise gradient, first-moment and updated-weight errors of one step
    (gradients and moments in the given norm, updated weights in the max norm).
    With ``spread`` (per tensor: how far the oracle's own result moves between
    fp32 and fp64 accumulation), a gradient or moment may be off by twice its
    spread where that exceeds the tolerance."""
    worst = {}
    for n in rgrads:
        tol = max(TOL, 2 * spread[n]) if spread else TOL
        e = norm(grads[n], rgrads[n])
        worst[n] = e
        assert e < tol, (n, e, tol)
        assert norm(mom1[n], rm[n]) < tol, n
        w0 = params[n].astype(np.float64)
        if np.abs(w0).max() > 0:
            assert relerr(new[n], rnew[n]) < TOL, n
        # at t = 1 the update is -lr (wd w + g/(|g| + eps)): a gradient that is
        # ~0 in both may flip sign, which moves the weight by 2 lr
        bound = 2 * 3e-4 * (1 + TOL) + TOL * np.abs(rnew[n]).max()
        assert np.abs(new[n] - rnew[n]).max() <= bound, n
        sel = np.abs(rgrads[n]) > 0.2 * np.abs(rgrads[n]).max()
        assert relerr((new[n] - w0)[sel], (rnew[n] - w0)[sel]) < TOL, n
    return worst


def test_wide4_step_matches_bf16_operand_oracle():
    """The whole wide-4 step (forward, backward, AdamW at t = 1) on a batch of
    two distinct sequences, each repeated 4 times: the mean over the 8 windows
    equals the mean over the two, which the oracle computes.

    The reference is the oracle with every matrix-product operand rounded to
    bf16 (the stated precision: bf16 GEMM operands, fp32 accumulation and fp32
    everything else): loss within 1e-3 of it and updated weights within 2e-2
    in the max norm. At d_model 8192 a gradient is not fully determined by that
    precision: the oracle's own bf16-operand step evaluated with fp32 and with
    fp64 accumulation differs by up to 1.7% per tensor (relative 2-norm;
    tests/golden/wide4_accumulation_spread.json, written by the oracle alone),
    and two evaluations that differ only in fp32 summation order are expected
    about sqrt(2) times that apart. Gradients and first moments are therefore
    checked in the relative 2-norm within 2e-2, or twice their spread where
    that is larger, and, as a check of their structure, within twice the
    spread plus 2e-3. Max-norm errors and the departures from the unrounded
    oracle are printed (the logits are asserted in the max norm)."""
    cfg = WIDE4
    two = O.GPT2Config(n_layer=cfg.n_layer, d_model=cfg.d_model, n_head=cfg.n_head, d_ff=cfg.d_ff,
                       vocab=cfg.vocab, seq=cfg.seq, batch=2)
    params = synth.gpt2_params(3, cfg.n_layer, cfg.d_model, cfg.d_ff, cfg.vocab, cfg.seq)
    seqs = np.concatenate([synth.token_windows(3, 1, cfg.seq, cfg.vocab),
                           synth.token_windows(4, 1, cfg.seq, cfg.vocab)])
    win = np.ascontiguousarray(np.tile(seqs, (cfg.batch // 2, 1)))  # s0, s1, s0, s1, ...
    m = make(cfg, WIDE4_TILES)
    m.set_params(params)
    loss = m.forward(win)
    logits = m.logits()[: 2 * cfg.seq]  # windows 0 and 1: rows b * S + s
    m.backward()
    grads = m.grads()
    m.adamw_step()
    new = m.params()
    mom1 = {n: m.get_adam_state(i, 0) for i, n in enumerate(m.names)}
    m.close()

    bloss, bcache = O.forward(two, params, seqs, dtype=np.float32, gemm_operands="bf16")
    bgrads = O.backward_bf16_operands(two, params, bcache, dtype=np.float32)
    del bcache
    bnew, bm, _ = O.adamw_step(params, bgrads, None, None, 1, O.AdamWHyper(), np.float32)
    assert abs(loss - bloss) < 1e-3, (loss, bloss)
    with open(os.path.join(os.path.dirname(__file__), "golden", "wide4_accumulation_spread.json")) as fh:
        spread = {n: v["two_norm"] for n, v in json.load(fh)["tensors"].items()}
    worst = _step_checks(grads, new, mom1, params, bgrads, bnew, bm, norm=relerr2, spread=spread)
    for n, e in worst.items():
        assert e <= 2 * spread[n] + 2e-3, (n, e, spread[n])
    worst_max = {n: relerr(grads[n], bgrads[n]) for n in bgrads}
    del bnew, bm

    rloss, cache = O.forward(two, params, seqs, dtype=np.float32)
    assert relerr(logits, cache["z"]) < TOL
    rgrads = O.backward(two, params, cache, dtype=np.float32)
    del cache
    print(f"loss: gpu {loss:.6f} bf16-operand oracle {bloss:.6f} unrounded oracle {rloss:.6f}")
    for n in rgrads:
        print(f"{n}: gpu-vs-bf16 2-norm {worst[n]:.4f} (oracle fp32/fp64 spread {spread[n]:.4f}) "
              f"max-norm {worst_max[n]:.4f}; "
              f"gpu-vs-unrounded max-norm {relerr(grads[n], rgrads[n]):.4f}; "
              f"bf16-vs-unrounded max-norm {relerr(bgrads[n], rgrads[n]):.4f}")
