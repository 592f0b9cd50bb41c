"""Pins for the CPU oracle: checks against things other than the oracle itself.

The NNTile pages print no worked example, loss value or gradient, so the pins
are closed forms, invariants, brute-force scalar loops on tiny inputs and
central finite differences (all CPU-only).
"""
import json
import math
import os

import numpy as np
import pytest

from oracle import gpt2 as O
from tile_task_transformer_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_params(cfg, seed, std=0.3):
    rng = np.random.default_rng(seed)
    p = {}
    for name, shape in O.param_order(cfg):
        if name.endswith(".g"):
            p[name] = 1.0 + 0.2 * rng.standard_normal(shape)
        else:
            p[name] = std * rng.standard_normal(shape)
    return p


def _windows(cfg, seed):
    rng = np.random.default_rng(seed)
    return rng.integers(0, cfg.vocab, size=(cfg.batch, cfg.seq + 1)).astype(np.uint16)


# ---------------------------------------------------------------- brute force

def _bf_layernorm(row, g, b, eps):
    n = len(row)
    mu = sum(row) / n
    var = sum((r - mu) ** 2 for r in row) / n
    return [g[j] * (row[j] - mu) / math.sqrt(var + eps) + b[j] for j in range(n)]


def _bf_gelu(u):
    return 0.5 * u * (1.0 + math.erf(u / math.sqrt(2.0)))


def _bf_attention(qkv, H):
    """Scalar-loop causal attention, one query at a time."""
    B, S, d3 = qkv.shape
    d = d3 // 3
    hd = d // H
    out = np.zeros((B, S, d))
    for b in range(B):
        for h in range(H):
            for i in range(S):
                sc = []
                for j in range(i + 1):
                    dot = 0.0
                    for c in range(hd):
                        dot += qkv[b, i, h * hd + c] * qkv[b, j, d + h * hd + c]
                    sc.append(dot / math.sqrt(hd))
                mx = max(sc)
                ex = [math.exp(s - mx) for s in sc]
                tot = sum(ex)
                for c in range(hd):
                    out[b, i, h * hd + c] = sum(ex[j] / tot * qkv[b, j, 2 * d + h * hd + c]
                                                for j in range(i + 1))
    return out


def _bf_full_forward(cfg, p, win):
    """The whole forward pass with scalar loops (no numpy linear algebra)."""
    B, S, d, f, V = cfg.batch, cfg.seq, cfg.d_model, cfg.d_ff, cfg.vocab
    x = np.zeros((B, S, d))
    for b in range(B):
        for s in range(S):
            for j in range(d):
                x[b, s, j] = p["wte"][win[b, s], j] + p["wpe"][s, j]

    def lin(a, w, bias):
        n_out, n_in = w.shape
        y = np.zeros(a.shape[:-1] + (n_out,))
        for idx in np.ndindex(a.shape[:-1]):
            for o in range(n_out):
                acc = 0.0 if bias is None else bias[o]
                for i in range(n_in):
                    acc += a[idx + (i,)] * w[o, i]
                y[idx + (o,)] = acc
        return y

    def ln(a, g, bb):
        y = np.zeros_like(a)
        for idx in np.ndindex(a.shape[:-1]):
            y[idx] = _bf_layernorm(list(a[idx]), g, bb, cfg.ln_eps)
        return y

    for l in range(cfg.n_layer):
        q = f"h{l}."
        h = ln(x, p[q + "ln1.g"], p[q + "ln1.b"])
        qkv = lin(h, p[q + "qkv.w"], p[q + "qkv.b"])
        x = x + lin(_bf_attention(qkv, cfg.n_head), p[q + "o.w"], p[q + "o.b"])
        h = ln(x, p[q + "ln2.g"], p[q + "ln2.b"])
        u = lin(h, p[q + "fc.w"], p[q + "fc.b"])
        gl = np.vectorize(lambda t: 0.5 * t * (1 + math.tanh(math.sqrt(2 / math.pi)
                                                            * (t + 0.044715 * t ** 3))))(u)
        x = x + lin(gl, p[q + "proj.w"], p[q + "proj.b"])
    y = ln(x, p["ln_f.g"], p["ln_f.b"])
    z = lin(y, p["wte"], None)
    tot = 0.0
    for b in range(B):
        for s in range(S):
            row = z[b, s]
            mx = max(row)
            lse = mx + math.log(sum(math.exp(r - mx) for r in row))
            tot += lse - row[win[b, s + 1]]
    return tot / (B * S)


MICRO = O.GPT2Config(n_layer=2, d_model=8, n_head=2, d_ff=16, vocab=11, seq=5, batch=2)


def test_forward_matches_scalar_loops():
    p = _rand_params(MICRO, 1)
    win = _windows(MICRO, 2)
    loss, _ = O.forward(MICRO, p, win)
    assert abs(loss - _bf_full_forward(MICRO, p, win)) < 1e-12


def test_attention_matches_scalar_loops():
    rng = np.random.default_rng(3)
    qkv = rng.standard_normal((2, 6, 3 * 8))
    out, P = O.attention_forward(qkv, 2)
    np.testing.assert_allclose(out, _bf_attention(qkv, 2), rtol=0, atol=1e-13)


def test_zero_layers_is_softmax_regression():
    """L = 0: embedding -> LN -> tied logits -> CE, on V=8, d=4 by scalar loops."""
    cfg = O.GPT2Config(n_layer=0, d_model=4, n_head=1, d_ff=4, vocab=8, seq=3, batch=2)
    p = _rand_params(cfg, 4, std=0.7)
    win = _windows(cfg, 5)
    loss, _ = O.forward(cfg, p, win)
    assert abs(loss - _bf_full_forward(cfg, p, win)) < 1e-13


# ------------------------------------------------------------ closed forms

@pytest.mark.parametrize("V", [256, 50257])
def test_zero_embedding_gives_log_vocab(V):
    """wte = 0 makes every logit 0: loss = ln V and dz = (1/V - onehot)/T."""
    cfg = O.GPT2Config(n_layer=1, d_model=8, n_head=2, d_ff=16, vocab=V, seq=4, batch=2)
    p = _rand_params(cfg, 6)
    p["wte"] = np.zeros_like(p["wte"])
    win = _windows(cfg, 7)
    loss, cache = O.forward(cfg, p, win)
    assert abs(loss - math.log(V)) < 1e-12
    T = cfg.batch * cfg.seq
    expect = np.full((T, V), 1.0 / V / T)
    expect[np.arange(T), win[:, 1:].reshape(-1).astype(np.int64)] -= 1.0 / T
    np.testing.assert_allclose(cache["dz"], expect, rtol=0, atol=1e-16)


def test_cross_entropy_against_loops_and_grad_rows_sum_to_zero():
    rng = np.random.default_rng(8)
    z = 3.0 * rng.standard_normal((7, 13))
    t = rng.integers(0, 13, size=7)
    loss, dz = O.cross_entropy_forward_backward(z, t)
    ref = sum(math.log(sum(math.exp(v) for v in z[i])) - z[i, t[i]] for i in range(7)) / 7
    assert abs(loss - ref) < 1e-13
    np.testing.assert_allclose(dz.sum(axis=1), 0.0, atol=1e-16)


def test_softmax_rows_sum_to_one_and_mask_is_exact_zero():
    rng = np.random.default_rng(9)
    s = 4.0 * rng.standard_normal((3, 9, 9))
    P = O.causal_softmax_forward(s)
    np.testing.assert_allclose(P.sum(axis=-1), 1.0, atol=1e-15)
    assert np.all(P[:, np.triu_indices(9, 1)[0], np.triu_indices(9, 1)[1]] == 0.0)
    # brute force row 5 of matrix 1
    ex = [math.exp(v) for v in s[1, 5, :6]]
    np.testing.assert_allclose(P[1, 5, :6], np.array(ex) / sum(ex), rtol=1e-14)
    # backward: rows of dS sum to zero, masked entries zero
    dP = rng.standard_normal(P.shape)
    dS = O.causal_softmax_backward(dP, P)
    np.testing.assert_allclose(dS.sum(axis=-1), 0.0, atol=1e-14)
    assert np.all(dS[:, 0, 1:] == 0.0)


def test_single_position_attention_returns_values():
    """S = 1: the only key is the query itself, so the output equals v."""
    rng = np.random.default_rng(10)
    qkv = rng.standard_normal((3, 1, 3 * 12))
    out, _ = O.attention_forward(qkv, 3)
    np.testing.assert_array_equal(out, qkv[..., 24:])


def test_layernorm_invariants():
    rng = np.random.default_rng(11)
    x = 2.0 + 3.0 * rng.standard_normal((5, 33))
    eps = 1e-5
    y, mu, rstd = O.layernorm_forward(x, np.ones(33), np.zeros(33), eps)
    np.testing.assert_allclose(y.mean(axis=-1), 0.0, atol=1e-14)
    var = x.var(axis=-1)
    np.testing.assert_allclose(y.var(axis=-1), var / (var + eps), rtol=1e-13)
    np.testing.assert_allclose(y[2], _bf_layernorm(list(x[2]), [1.0] * 33, [0.0] * 33, eps),
                               rtol=1e-13)
    dy = rng.standard_normal(x.shape)
    dx, dg, db = O.layernorm_backward(dy, x, mu, rstd, np.ones(33))
    xhat = (x - mu[:, None]) * rstd[:, None]
    np.testing.assert_allclose(dx.sum(axis=-1), 0.0, atol=1e-13)
    # sum_j dx_j xhat_j = rstd * sum_j (dy_j xhat_j) * eps / (var + eps): zero only for eps = 0
    np.testing.assert_allclose((dx * xhat).sum(axis=-1),
                               rstd * (dy * xhat).sum(axis=-1) * eps / (var + eps), rtol=1e-6, atol=1e-15)
    np.testing.assert_allclose(db, dy.sum(axis=0), rtol=1e-14)


def test_gelu_against_erf_form_and_odd_identity():
    x = np.linspace(-8.0, 8.0, 4001)
    g = O.gelu_forward(x)
    exact = np.array([_bf_gelu(v) for v in x])
    # the tanh form is within 5e-4 of the exact erf GELU everywhere
    assert np.abs(g - exact).max() < 5e-4
    # gelu(x) - gelu(-x) = x holds exactly for the tanh form
    np.testing.assert_allclose(g - O.gelu_forward(-x), x, atol=1e-14)
    assert O.gelu_forward(np.array([0.0]))[0] == 0.0
    # derivative against central differences
    h = 1e-6
    fd = (O.gelu_forward(x + h) - O.gelu_forward(x - h)) / (2 * h)
    np.testing.assert_allclose(O.gelu_backward(np.ones_like(x), x), fd, atol=1e-8)


def test_linear_matches_triple_loop():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((4, 3, 5))
    w = rng.standard_normal((6, 5))
    b = rng.standard_normal(6)
    y = O.linear_forward(x, w, b)
    for i in range(4):
        for j in range(3):
            for o in range(6):
                assert abs(y[i, j, o] - (b[o] + sum(x[i, j, k] * w[o, k] for k in range(5)))) < 1e-13


def test_embedding_float32_scatter_order():
    """float32 scatter-add matches a scalar loop in token order, bit for bit."""
    rng = np.random.default_rng(13)
    B, S, d, V = 3, 7, 5, 4
    ids = rng.integers(0, V, size=(B, S))
    dx = rng.standard_normal((B, S, d)).astype(np.float32)
    w0 = rng.standard_normal((V, d)).astype(np.float32)
    p0 = rng.standard_normal((S, d)).astype(np.float32)
    dwte, dwpe = O.embedding_backward(dx, ids, w0, p0)
    ref = w0.copy()
    for b in range(B):
        for s in range(S):
            for j in range(d):
                ref[ids[b, s], j] = np.float32(ref[ids[b, s], j] + dx[b, s, j])
    np.testing.assert_array_equal(dwte, ref)
    refp = p0.copy()
    for b in range(B):
        for s in range(S):
            for j in range(d):
                refp[s, j] = np.float32(refp[s, j] + dx[b, s, j])
    np.testing.assert_array_equal(dwpe, refp)
    x = O.embedding_forward(ids, w0, p0)
    assert x.dtype == np.float32
    np.testing.assert_array_equal(x[1, 2], w0[ids[1, 2]] + p0[2])


def test_adamw_first_step_closed_form():
    """At t = 1: mhat = g, sqrt(vhat) = |g|, so w1 = w0 (1 - lr wd) - lr g/(|g| + eps)."""
    with open(os.path.join(GOLDEN, "readme_hyperparams.json")) as fh:
        hpj = json.load(fh)
    hp = O.AdamWHyper(lr=hpj["lr"], eps=hpj["optimizer_eps"], weight_decay=hpj["weight_decay"])
    rng = np.random.default_rng(14)
    w = rng.standard_normal(1000)
    g = rng.standard_normal(1000)
    g[:10] = 0.0
    w1, m1, v1 = O.adamw_update(w, g, np.zeros_like(w), np.zeros_like(w), 1, hp)
    expect = w * (1 - hp.lr * hp.weight_decay) - hp.lr * g / (np.abs(g) + hp.eps)
    np.testing.assert_allclose(w1, expect, rtol=1e-12, atol=1e-18)
    np.testing.assert_array_equal(w1[:10], w[:10] - hp.lr * hp.weight_decay * w[:10])
    np.testing.assert_allclose(m1, 0.1 * g, rtol=1e-14)
    np.testing.assert_allclose(v1, 0.001 * g * g, rtol=1e-12)
    # second step against the definition unrolled by hand
    g2 = rng.standard_normal(1000)
    w2, _, _ = O.adamw_update(w1, g2, m1, v1, 2, hp)
    m2 = 0.9 * 0.1 * g + 0.1 * g2
    v2 = 0.999 * 0.001 * g * g + 0.001 * g2 * g2
    e2 = w1 - hp.lr * hp.weight_decay * w1 - hp.lr * (m2 / 0.19) / (np.sqrt(v2 / (1 - 0.999 ** 2)) + hp.eps)
    np.testing.assert_allclose(w2, e2, rtol=1e-12)


def test_readme_hyperparams_are_oracle_defaults():
    with open(os.path.join(GOLDEN, "readme_hyperparams.json")) as fh:
        hpj = json.load(fh)
    hp = O.AdamWHyper()
    assert hp.lr == hpj["lr"] and hp.eps == hpj["optimizer_eps"]
    assert hp.weight_decay == hpj["weight_decay"]


# -------------------------------------------------------- finite differences

def _fd_check(cfg, seed, n_probe=16):
    p = _rand_params(cfg, seed)
    win = _windows(cfg, seed + 100)
    loss, cache = O.forward(cfg, p, win)
    grads = O.backward(cfg, p, cache)
    rng = np.random.default_rng(seed + 200)
    h = 1e-5
    for name, shape in O.param_order(cfg):
        flat = p[name].reshape(-1)
        idx = rng.choice(flat.size, size=min(n_probe, flat.size), replace=False)
        scale = max(np.abs(grads[name]).max(), 1e-6)
        for i in idx:
            old = flat[i]
            flat[i] = old + h
            lp, _ = O.forward(cfg, p, win, keep=False)
            flat[i] = old - h
            lm, _ = O.forward(cfg, p, win, keep=False)
            flat[i] = old
            fd = (lp - lm) / (2 * h)
            an = grads[name].reshape(-1)[i]
            assert abs(fd - an) <= 1e-6 * scale + 1e-10, (name, i, fd, an)


@pytest.mark.parametrize("n_layer", [0, 1, 2])
def test_gradients_match_central_differences(n_layer):
    cfg = O.GPT2Config(n_layer=n_layer, d_model=8, n_head=2, d_ff=16, vocab=11, seq=5, batch=2)
    _fd_check(cfg, 20 + n_layer)


def test_causality_of_logits():
    cfg = O.GPT2Config(n_layer=2, d_model=8, n_head=2, d_ff=16, vocab=11, seq=6, batch=1)
    p = _rand_params(cfg, 30)
    win = _windows(cfg, 31)
    _, c1 = O.forward(cfg, p, win)
    win2 = win.copy()
    win2[0, 4] = (int(win2[0, 4]) + 3) % cfg.vocab
    _, c2 = O.forward(cfg, p, win2)
    np.testing.assert_allclose(c1["z"][:4], c2["z"][:4], rtol=0, atol=1e-14)
    assert np.abs(c1["z"][4] - c2["z"][4]).max() > 1e-6


def test_float32_and_float64_oracles_agree_on_tiny_config():
    cfg = O.GPT2Config(n_layer=2, d_model=64, n_head=4, d_ff=256, vocab=256, seq=32, batch=2)
    p = synth.gpt2_params(0, 2, 64, 256, 256, 32)
    win = synth.token_windows(0, 2, 32, 256)
    l64, g64, _, _, _ = O.train_step(cfg, p, win, dtype=np.float64)
    l32, g32, _, _, _ = O.train_step(cfg, p, win, dtype=np.float32)
    assert abs(l64 - l32) < 1e-4
    for k in g64:
        err = np.abs(g64[k] - g32[k]).max() / max(np.abs(g64[k]).max(), 1e-12)
        assert err < 1e-4, k


def test_step_flops_counts_by_hand():
    cfg = O.GPT2Config(n_layer=1, d_model=2, n_head=1, d_ff=4, vocab=3, seq=2, batch=1)
    # dense per token: 2*(2*6 + 2*2 + 2*2*4) = 64 ; lm head 2*2*3 = 12 ; T = 2
    # attention: 2 products * 2*hd*S(S+1)/2 = 2*2*2*3 = 24
    assert O.step_flops(cfg) == 3.0 * (2 * (64 + 12) + 24)


def test_round_bf16_exact_cases_and_library_agreement():
    one = 1.0
    cases = {
        one: one,
        one + 2.0 ** -8: one,                          # tie, even neighbour is 1
        one + 2.0 ** -7 + 2.0 ** -8: one + 2.0 ** -6,  # tie, rounds up to the even neighbour
        one + 2.0 ** -9: one,                           # below half an ulp
        one + 2.0 ** -8 + 2.0 ** -12: one + 2.0 ** -7,  # above half an ulp
        -3.0: -3.0,
        0.0: 0.0,
    }
    for a, want in cases.items():
        assert O.round_bf16(np.array([a]))[0] == np.float32(want), a
    torch = pytest.importorskip("torch")
    x = np.random.default_rng(15).standard_normal(100000).astype(np.float32) * 10.0 ** \
        np.random.default_rng(16).integers(-20, 20, 100000)
    lib = torch.from_numpy(x).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(O.round_bf16(x), lib)


def test_bf16_operand_model_reduces_to_forward_without_rounding_when_exact():
    """With all GEMM operands already bf16-representable the precision model
    changes nothing but the rounding of activations between products; on a
    tiny model the two forwards agree to the bf16 scale."""
    cfg = O.GPT2Config(n_layer=1, d_model=8, n_head=2, d_ff=16, vocab=11, seq=5, batch=2)
    p = {k: O.round_bf16(v) for k, v in _rand_params(cfg, 40).items()}
    win = _windows(cfg, 41)
    l_ref, _ = O.forward(cfg, p, win)
    l_bf, _ = O.forward(cfg, p, win, gemm_operands="bf16")
    assert abs(l_ref - l_bf) < 2e-2 and l_ref != l_bf


def test_bf16_precision_model_reduces_to_exact_step_with_identity_rounding():
    """With the rounding replaced by the identity, the precision-model forward
    and backward are term for term the plain ones."""
    cfg = O.GPT2Config(n_layer=2, d_model=8, n_head=2, d_ff=16, vocab=11, seq=5, batch=2)
    p = _rand_params(cfg, 42)
    win = _windows(cfg, 43)
    ident = lambda a: np.asarray(a, dtype=np.float64)  # noqa: E731
    l0, c0 = O.forward(cfg, p, win)
    g0 = O.backward(cfg, p, c0)
    l1, c1 = O._forward_bf16_operands(cfg, p, win, np.float64, r=ident)
    g1 = O.backward_bf16_operands(cfg, p, c1, np.float64, r=ident)
    assert abs(l0 - l1) < 1e-13
    for k in g0:
        np.testing.assert_allclose(g1[k], g0[k], rtol=1e-10, atol=1e-14, err_msg=k)
    # and with bfloat16 rounding the gradients stay close to the exact ones
    lb, cb = O.forward(cfg, p, win, gemm_operands="bf16")
    gb = O.backward_bf16_operands(cfg, p, cb)
    for k in g0:
        assert np.abs(gb[k] - g0[k]).max() <= 3e-2 * np.abs(g0[k]).max() + 1e-12, k


def test_streamed_bf16_step_matches_whole_model():
    """The layer-streamed bf16-operand step (one layer's parameters at a time,
    bf16 values cached as bit patterns, attention one sequence at a time) gives
    the whole-model precision model's loss, logits and gradients."""
    cfg = O.GPT2Config(n_layer=3, d_model=32, n_head=2, d_ff=64, vocab=37, seq=12, batch=3)
    p = {k: v.astype(np.float32) for k, v in _rand_params(cfg, 46).items()}
    win = _windows(cfg, 47)
    head = {k: p[k] for k in ("wte", "wpe", "ln_f.g", "ln_f.b")}
    layer = lambda l: {k[len(f"h{l}."):]: v for k, v in p.items() if k.startswith(f"h{l}.")}  # noqa: E731
    l0, c0 = O.forward(cfg, p, win, dtype=np.float32, gemm_operands="bf16")
    g0 = O.backward_bf16_operands(cfg, p, c0, dtype=np.float32)
    l1, c1 = O.forward_bf16_streamed(cfg, layer, head, win)
    assert abs(l1 - l0) < 1e-6
    np.testing.assert_allclose(c1["z"], c0["z"], rtol=1e-5, atol=1e-6)
    g1 = O.backward_bf16_streamed(cfg, layer, head, c1)
    assert set(g1) == set(g0)
    for k in g0:
        scale = np.abs(g0[k]).max()
        assert np.abs(g1[k] - g0[k]).max() <= 1e-4 * scale + 1e-9, k
    # only the requested layers' parameter gradients (plus wte, wpe, ln_f)
    g2 = O.backward_bf16_streamed(cfg, layer, head, c1, want={0, 2})
    assert set(g2) == {k for k in g0 if not k.startswith("h1.")}
    for k in g2:
        np.testing.assert_array_equal(g2[k], g1[k])
    # the same in fp64 arithmetic (used to measure what fp32 accumulation leaves open)
    l64, c64 = O.forward(cfg, p, win, dtype=np.float64, gemm_operands="bf16")
    g64 = O.backward_bf16_operands(cfg, p, c64, dtype=np.float64)
    l3, c3 = O.forward_bf16_streamed(cfg, layer, head, win, dtype=np.float64)
    assert abs(l3 - l64) < 1e-12
    g3 = O.backward_bf16_streamed(cfg, layer, head, c3, dtype=np.float64)
    for k in g64:
        assert np.abs(g3[k] - g64[k]).max() <= 1e-10 * np.abs(g64[k]).max() + 1e-15, k
    # bf16 bit patterns round-trip
    x = np.random.default_rng(0).standard_normal(1000).astype(np.float32)
    np.testing.assert_array_equal(O.from_bf16_bits(O.bf16_bits(x)), O.round_bf16(x))


# ------------------------------------- gradient accumulation and lr warm-up

def test_warmup_schedule_end_points_from_readme():
    """README flags: --start-lr is the rate of the first batch, --full-lr-iter the
    iteration that first uses --lr, and 1 means the full rate throughout."""
    with open(os.path.join(GOLDEN, "readme_hyperparams.json")) as fh:
        hpj = json.load(fh)
    hp = O.AdamWHyper(lr=hpj["lr"], start_lr=hpj["start_lr"], full_lr_iter=hpj["full_lr_iter"])
    assert O.scheduled_lr(hp, 1) == hpj["start_lr"]
    assert O.scheduled_lr(hp, hpj["full_lr_iter"]) == hpj["lr"]
    assert O.scheduled_lr(hp, hpj["full_lr_iter"] + 5) == hpj["lr"]
    rates = [O.scheduled_lr(hp, t) for t in range(1, hpj["full_lr_iter"] + 1)]
    assert all(a < b for a, b in zip(rates, rates[1:]))  # strictly rising to the full rate
    for t in (1, 2, 7, 100):
        assert O.scheduled_lr(O.AdamWHyper(lr=hpj["lr"], start_lr=0.0, full_lr_iter=1), t) == hpj["lr"]
    # the constant-rate default
    assert O.scheduled_lr(O.AdamWHyper(), 1) == O.AdamWHyper().lr


def test_zero_start_rate_leaves_weights_unchanged_on_first_step():
    """lr = 0 multiplies both the decay and the Adam term: w stays bit-identical,
    while the moments still take the first gradient."""
    cfg = O.GPT2Config(n_layer=1, d_model=8, n_head=2, d_ff=16, vocab=11, seq=4, batch=2)
    p = _rand_params(cfg, 31)
    hp = O.AdamWHyper(start_lr=0.0, full_lr_iter=4)
    loss, grads, new, m, v = O.train_step(cfg, p, _windows(cfg, 32), hp)
    for n in p:
        np.testing.assert_array_equal(new[n], p[n])
        np.testing.assert_allclose(m[n], 0.1 * grads[n], rtol=1e-14)


def test_minibatch_accumulation_equals_whole_batch_gradient():
    """The mean loss over a batch is the mean of its equal-sized minibatches'
    mean losses, so accumulated minibatch gradients / k must equal the gradient
    of the batch processed at once (batch linearity, computed another way)."""
    big = O.GPT2Config(n_layer=2, d_model=8, n_head=2, d_ff=16, vocab=13, seq=5, batch=4)
    small = O.GPT2Config(n_layer=2, d_model=8, n_head=2, d_ff=16, vocab=13, seq=5, batch=2)
    p = _rand_params(big, 33)
    win = _windows(big, 34)
    loss_all, cache = O.forward(big, p, win)
    g_all = O.backward(big, p, cache)
    loss_acc, g_acc = O.batch_gradient(small, p, [win[:2], win[2:]])
    assert abs(loss_acc - loss_all) < 1e-13
    for n in g_all:
        np.testing.assert_allclose(g_acc[n], g_all[n], rtol=1e-10, atol=1e-14)
    # a wrong normaliser (sum instead of mean) is caught
    assert not np.allclose(2 * g_acc["wte"], g_all["wte"])


def test_training_on_one_batch_lowers_the_loss():
    """Several AdamW steps on a repeated batch must lower its loss (descent on a
    smooth objective with a small rate); the warm-up schedule's first step at
    rate 0 leaves the loss of step 2 equal to that of step 1."""
    cfg = O.GPT2Config(n_layer=1, d_model=16, n_head=2, d_ff=32, vocab=17, seq=6, batch=2)
    p = _rand_params(cfg, 35, std=0.1)
    mbs = [_windows(cfg, 36), _windows(cfg, 37)]
    hp = O.AdamWHyper(lr=1e-2, start_lr=0.0, full_lr_iter=3)
    losses, final, _, _ = O.train(cfg, p, [mbs] * 6, hp)
    assert losses[1] == losses[0]
    assert all(b < a for a, b in zip(losses[1:], losses[2:])), losses


def test_causal_logsumexp_normalises_the_causal_softmax():
    """exp(scores - lse) must reproduce the (separately pinned) causal softmax on
    the causal entries, and lse of a single-entry row is that entry."""
    rng = np.random.default_rng(41)
    sc = 4.0 * rng.standard_normal((3, 7, 7))
    lse = O.causal_logsumexp(sc)
    P = O.causal_softmax_forward(sc)
    tri = np.tril(np.ones((7, 7), dtype=bool))
    np.testing.assert_allclose(np.exp(sc - lse[..., None])[:, tri], P[:, tri], rtol=1e-12)
    np.testing.assert_array_equal(lse[:, 0], sc[:, 0, 0])
    # a brute-force row
    q = 5
    ref = math.log(sum(math.exp(sc[1, q, k]) for k in range(q + 1)))
    assert abs(lse[1, q] - ref) < 1e-12
