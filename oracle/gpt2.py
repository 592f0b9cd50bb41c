"""Plain CPU oracle of one GPT2 training step: forward, backward, AdamW.

TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's CPU
baseline leg use this module; the library never calls it, and it shares no
code with the CUDA path (it imports numpy only).

What it computes is the untiled definition of the step the NNTile pages
describe: the tile-wise task graph only reorders this arithmetic
("NNTile: a machine learning framework ..." review page, section "What carries
the argument": every tensor split into tiles, every layer -- embedding, linear,
layer norm, softmax, attention, cross-entropy, Adam -- written as tasks on
tiles). The model is GPT2 (title of the first page) with pre-LN blocks (its
reference "On Layer Normalization in the Transformer Architecture"), Layer
Normalization (reference "Layer Normalization"), scaled dot-product causal
attention (reference "Attention Is All You Need"), mean cross-entropy over all
tokens (README "Minimal working GPT example", flag --loss-reduction=mean) and
decoupled weight decay AdamW (reference "Decoupled Weight Decay
Regularization"; README flags --optimizer=fusedadamw, --optimizer-eps=1e-8,
--weight-decay=0.1, --lr=3e-4).

Readings where the pages are silent (each also listed in the design notes):
  * LayerNorm eps 1e-5, biased variance.
  * GELU: the tanh approximation used by GPT2.
  * attention scale 1/sqrt(head_dim); causal mask = probability exactly 0.
  * no dropout, no gradient clipping, AdamW betas (0.9, 0.999).
  * learning-rate warm-up (README flags --start-lr, --full-lr-iter): the pages
    give the rate of the first iteration and the iteration from which the full
    rate applies; in between the rate is read as the straight line joining
    them. With full_lr_iter <= 1 (the default here) the rate is constant.
  * gradient accumulation (README flags --batch, --minibatch): the optimizer
    step uses the gradient of the mean loss over the whole batch, i.e. the
    mean of the minibatch gradients when every minibatch holds the same
    number of tokens.
  * weight decay applied to every parameter (one --weight-decay flag, no
    exclusion list on the pages).
  * tied LM head (wte used as the output projection, no LM bias); the two
    gradient contributions to wte are summed.
  * targets are the next token: window ``[B, S+1]``, inputs ``[:, :S]``,
    targets ``[:, 1:]``.

Arithmetic runs in ``dtype`` (float64 by default). Weight matrices are stored
``[out, in]``; a linear layer is ``y = x W^T + b``.

Precision model (optional): ``forward(..., gemm_operands="bf16")`` rounds both
operands of every matrix product to bfloat16 (round to nearest, ties to even)
before multiplying in ``dtype`` -- the "bf16 in, fp32 accumulate" precision of
the tensor-core path -- so that the effect of that rounding on the loss can be
told apart from arithmetic errors.
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class GPT2Config:
    n_layer: int
    d_model: int
    n_head: int
    d_ff: int
    vocab: int
    seq: int
    batch: int
    ln_eps: float = 1e-5

    @property
    def head_dim(self) -> int:
        return self.d_model // self.n_head


@dataclass(frozen=True)
class AdamWHyper:
    lr: float = 3e-4
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.1
    start_lr: float = 0.0  # rate of iteration 1 when full_lr_iter > 1
    full_lr_iter: int = 0  # first iteration at the full rate (<= 1: always)


def param_order(cfg: GPT2Config):
    """Names and shapes in the fixed parameter order (weights ``[out, in]``)."""
    d, f = cfg.d_model, cfg.d_ff
    out = [("wte", (cfg.vocab, d)), ("wpe", (cfg.seq, d))]
    for l in range(cfg.n_layer):
        p = f"h{l}."
        out += [(p + "ln1.g", (d,)), (p + "ln1.b", (d,)),
                (p + "qkv.w", (3 * d, d)), (p + "qkv.b", (3 * d,)),
                (p + "o.w", (d, d)), (p + "o.b", (d,)),
                (p + "ln2.g", (d,)), (p + "ln2.b", (d,)),
                (p + "fc.w", (f, d)), (p + "fc.b", (f,)),
                (p + "proj.w", (d, f)), (p + "proj.b", (d,))]
    out += [("ln_f.g", (d,)), ("ln_f.b", (d,))]
    return out


# --------------------------------------------------------------------------
# single operations
# --------------------------------------------------------------------------

def round_bf16(a):
    """Round to the nearest bfloat16 (ties to even), returned as float32.

    bfloat16 keeps the top 16 bits of an IEEE float32: add 0x7FFF plus the
    lowest kept bit, then clear the low 16 bits. NaN stays NaN.
    """
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    out = r.astype(np.uint32).view(np.float32)
    return np.where(np.isnan(f), f, out)


def embedding_forward(ids, wte, wpe):
    """x[b, s, :] = wte[ids[b, s], :] + wpe[s, :] (one add, in the arrays' dtype)."""
    S = ids.shape[1]
    return wte[ids.astype(np.int64)] + wpe[:S][None, :, :]


def embedding_backward(dx, ids, dwte, dwpe):
    """Scatter-add of the embedding gradient, returning updated copies.

    ``dwte[ids[t]] += dx[t]`` for flat token index t = b*S + s taken in
    increasing order, and ``dwpe[s] += dx[b, s]`` for b in increasing order.
    The additions happen one at a time in the arrays' dtype, so a float32 call
    fixes the exact rounding sequence.
    """
    B, S, d = dx.shape
    dwte = dwte.copy()
    dwpe = dwpe.copy()
    flat_ids = ids.reshape(-1).astype(np.int64)
    flat_dx = dx.reshape(B * S, d)
    for t in range(B * S):
        v = flat_ids[t]
        dwte[v] = dwte[v] + flat_dx[t]
    for b in range(B):
        dwpe[:S] = dwpe[:S] + dx[b]
    return dwte, dwpe


def layernorm_forward(x, gamma, beta, eps):
    """Layer normalisation over the last axis (biased variance).

    Returns ``y = gamma * xhat + beta``, the mean and ``rstd = 1/sqrt(var + eps)``.
    """
    mu = x.mean(axis=-1, keepdims=True)
    var = ((x - mu) ** 2).mean(axis=-1, keepdims=True)
    rstd = 1.0 / np.sqrt(var + eps)
    xhat = (x - mu) * rstd
    return gamma * xhat + beta, mu[..., 0], rstd[..., 0]


def layernorm_backward(dy, x, mu, rstd, gamma):
    """Gradients of :func:`layernorm_forward`.

    With ``g = gamma * dy``: ``dx = rstd * (g - mean(g) - xhat * mean(g * xhat))``;
    ``dgamma = sum over rows of dy * xhat``; ``dbeta = sum over rows of dy``.
    """
    xhat = (x - mu[..., None]) * rstd[..., None]
    g = gamma * dy
    dx = rstd[..., None] * (g - g.mean(axis=-1, keepdims=True)
                            - xhat * (g * xhat).mean(axis=-1, keepdims=True))
    rows = tuple(range(dy.ndim - 1))
    return dx, (dy * xhat).sum(axis=rows), dy.sum(axis=rows)


GELU_C = math.sqrt(2.0 / math.pi)
GELU_A = 0.044715


def gelu_forward(u):
    """tanh-form GELU: 0.5 u (1 + tanh(sqrt(2/pi) (u + 0.044715 u^3)))."""
    return 0.5 * u * (1.0 + np.tanh(GELU_C * (u + GELU_A * u ** 3)))


def gelu_backward(dg, u):
    """dL/du for :func:`gelu_forward`, by the product and chain rules."""
    t = np.tanh(GELU_C * (u + GELU_A * u ** 3))
    dt_du = (1.0 - t * t) * GELU_C * (1.0 + 3.0 * GELU_A * u * u)
    return dg * (0.5 * (1.0 + t) + 0.5 * u * dt_du)


def causal_softmax_forward(scores):
    """Row softmax over the last axis with key index > query index masked out.

    ``scores[..., q, k]``; masked entries get probability exactly 0.
    """
    S_q, S_k = scores.shape[-2:]
    mask = np.triu(np.ones((S_q, S_k), dtype=bool), k=1)
    s = np.where(mask, -np.inf, scores)
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    return e / e.sum(axis=-1, keepdims=True)


def causal_logsumexp(scores):
    """Natural log of each row's softmax normaliser over the causal entries:
    lse[q] = log sum_{k <= q} exp(scores[q, k]), so that the causal softmax is
    exp(scores - lse) on those entries. (A fused attention keeps this per row
    instead of the probabilities.)"""
    S_q, S_k = scores.shape[-2:]
    mask = np.triu(np.ones((S_q, S_k), dtype=bool), k=1)
    s = np.where(mask, -np.inf, scores)
    m = s.max(axis=-1)
    return m + np.log(np.exp(s - m[..., None]).sum(axis=-1))


def causal_softmax_backward(dP, P):
    """dS = P * (dP - rowsum(dP * P)); masked entries (P = 0) give 0."""
    return P * (dP - (dP * P).sum(axis=-1, keepdims=True))


def split_heads(t, n_head):
    B, S, d = t.shape
    return t.reshape(B, S, n_head, d // n_head).transpose(0, 2, 1, 3)


def merge_heads(t):
    B, H, S, hd = t.shape
    return t.transpose(0, 2, 1, 3).reshape(B, S, H * hd)


def attention_forward(qkv, n_head):
    """Causal multi-head attention on the fused ``[B, S, 3d]`` projection.

    Columns ``[0, d)`` are queries, ``[d, 2d)`` keys, ``[2d, 3d)`` values; head h
    owns columns ``h*hd .. h*hd+hd-1`` of each part.
    Returns the merged output ``[B, S, d]`` and the probabilities ``[B, H, S, S]``.
    """
    d = qkv.shape[-1] // 3
    q = split_heads(qkv[..., :d], n_head)
    k = split_heads(qkv[..., d:2 * d], n_head)
    v = split_heads(qkv[..., 2 * d:], n_head)
    scale = 1.0 / math.sqrt(d // n_head)
    P = causal_softmax_forward((q @ k.transpose(0, 1, 3, 2)) * scale)
    return merge_heads(P @ v), P


def attention_backward(do, qkv, P, n_head):
    """Gradient of :func:`attention_forward` w.r.t. the fused projection."""
    d = qkv.shape[-1] // 3
    q = split_heads(qkv[..., :d], n_head)
    k = split_heads(qkv[..., d:2 * d], n_head)
    v = split_heads(qkv[..., 2 * d:], n_head)
    scale = 1.0 / math.sqrt(d // n_head)
    dO = split_heads(do, n_head)
    dv = P.transpose(0, 1, 3, 2) @ dO
    dP = dO @ v.transpose(0, 1, 3, 2)
    dS = causal_softmax_backward(dP, P) * scale
    dq = dS @ k
    dk = dS.transpose(0, 1, 3, 2) @ q
    return np.concatenate([merge_heads(dq), merge_heads(dk), merge_heads(dv)], axis=-1)


def linear_forward(x, w, b=None):
    """y = x W^T (+ b), W stored ``[out, in]``."""
    y = x @ w.T
    return y if b is None else y + b


def cross_entropy_forward_backward(z, targets):
    """Mean next-token cross-entropy and its gradient w.r.t. the logits.

    ``loss = (1/T) sum_t [logsumexp(z_t) - z_t[y_t]]`` over all T tokens;
    ``dz = (softmax(z) - onehot(y)) / T``.
    """
    T = z.shape[0]
    m = z.max(axis=-1, keepdims=True)
    e = np.exp(z - m)
    ssum = e.sum(axis=-1, keepdims=True)
    lse = (m + np.log(ssum))[:, 0]
    rows = np.arange(T)
    loss = (lse - z[rows, targets]).sum() / T
    dz = e / ssum
    dz[rows, targets] -= 1.0
    return loss, dz / T


def adamw_update(w, g, m, v, step, hp: AdamWHyper):
    """One decoupled-weight-decay Adam update (PyTorch AdamW order).

    m = b1 m + (1-b1) g; v = b2 v + (1-b2) g^2; mhat = m/(1-b1^t);
    vhat = v/(1-b2^t); w <- w - lr*wd*w - lr*mhat/(sqrt(vhat)+eps), both terms
    using the pre-update w.
    """
    m = hp.beta1 * m + (1.0 - hp.beta1) * g
    v = hp.beta2 * v + (1.0 - hp.beta2) * g * g
    mhat = m / (1.0 - hp.beta1 ** step)
    vhat = v / (1.0 - hp.beta2 ** step)
    w = w - hp.lr * hp.weight_decay * w - hp.lr * mhat / (np.sqrt(vhat) + hp.eps)
    return w, m, v


# --------------------------------------------------------------------------
# whole step
# --------------------------------------------------------------------------

def _cast(params, dtype):
    return {k: np.asarray(v, dtype=dtype) for k, v in params.items()}


def forward(cfg: GPT2Config, params, windows, dtype=np.float64, keep=True, gemm_operands=None):
    """Forward pass; returns ``(loss, cache)``. ``windows`` is ``[B, S+1]``.

    ``gemm_operands="bf16"`` applies the bfloat16 precision model (module doc)
    to every matrix product; the cache is then meant for the loss only.
    """
    if gemm_operands == "bf16":
        return _forward_bf16_operands(cfg, params, windows, dtype)
    p = _cast(params, dtype)
    ids = windows[:, :cfg.seq].astype(np.int64)
    tgt = windows[:, 1:cfg.seq + 1].astype(np.int64)
    B, S, d = cfg.batch, cfg.seq, cfg.d_model
    cache = {"ids": ids, "layers": []}
    x = embedding_forward(ids, p["wte"], p["wpe"])
    for l in range(cfg.n_layer):
        q = f"h{l}."
        c = {"x_in": x}
        h1, c["mu1"], c["r1"] = layernorm_forward(x, p[q + "ln1.g"], p[q + "ln1.b"], cfg.ln_eps)
        qkv = linear_forward(h1, p[q + "qkv.w"], p[q + "qkv.b"])
        o, P = attention_forward(qkv, cfg.n_head)
        x = x + linear_forward(o, p[q + "o.w"], p[q + "o.b"])
        c["x_mid"] = x
        h2, c["mu2"], c["r2"] = layernorm_forward(x, p[q + "ln2.g"], p[q + "ln2.b"], cfg.ln_eps)
        u = linear_forward(h2, p[q + "fc.w"], p[q + "fc.b"])
        g = gelu_forward(u)
        x = x + linear_forward(g, p[q + "proj.w"], p[q + "proj.b"])
        if keep:
            c.update(h1=h1, qkv=qkv, o=o, P=P, h2=h2, u=u, g=g)
            cache["layers"].append(c)
    cache["x_L"] = x
    y, cache["muf"], cache["rf"] = layernorm_forward(x, p["ln_f.g"], p["ln_f.b"], cfg.ln_eps)
    cache["y"] = y
    z = linear_forward(y.reshape(B * S, d), p["wte"])
    loss, dz = cross_entropy_forward_backward(z, tgt.reshape(-1))
    cache["z"] = z
    cache["dz"] = dz
    return loss, cache


def _forward_bf16_operands(cfg: GPT2Config, params, windows, dtype, r=None):
    """The forward of :func:`forward` with both operands of each matrix product
    (activations and weights, including Q, K, V and the probabilities) rounded
    by ``r`` (bfloat16 by default) first; everything else as in
    :func:`forward`. The cache feeds :func:`backward_bf16_operands`."""
    p = _cast(params, dtype)
    if r is None:
        r = lambda a: round_bf16(a).astype(dtype)  # noqa: E731
    ids = windows[:, :cfg.seq].astype(np.int64)
    tgt = windows[:, 1:cfg.seq + 1].astype(np.int64)
    B, S, d, H = cfg.batch, cfg.seq, cfg.d_model, cfg.n_head
    c = {"ids": ids, "layers": []}
    x = embedding_forward(ids, p["wte"], p["wpe"])
    for l in range(cfg.n_layer):
        q = f"h{l}."
        L = {"x_in": x}
        h1, L["mu1"], L["r1"] = layernorm_forward(x, p[q + "ln1.g"], p[q + "ln1.b"], cfg.ln_eps)
        L["h1"] = r(h1)
        qkv = linear_forward(L["h1"], r(p[q + "qkv.w"]), p[q + "qkv.b"])
        L["q"] = split_heads(r(qkv[..., :d]), H)
        L["k"] = split_heads(r(qkv[..., d:2 * d]), H)
        L["v"] = split_heads(r(qkv[..., 2 * d:]), H)
        P = causal_softmax_forward((L["q"] @ L["k"].transpose(0, 1, 3, 2)) * (1.0 / math.sqrt(d // H)))
        L["P"] = r(P)
        L["o"] = r(merge_heads(L["P"] @ L["v"]))
        x = x + linear_forward(L["o"], r(p[q + "o.w"]), p[q + "o.b"])
        L["x_mid"] = x
        h2, L["mu2"], L["r2"] = layernorm_forward(x, p[q + "ln2.g"], p[q + "ln2.b"], cfg.ln_eps)
        L["h2"] = r(h2)
        L["u"] = linear_forward(L["h2"], r(p[q + "fc.w"]), p[q + "fc.b"])
        L["g"] = r(gelu_forward(L["u"]))
        x = x + linear_forward(L["g"], r(p[q + "proj.w"]), p[q + "proj.b"])
        c["layers"].append(L)
    c["x_L"] = x
    y, c["muf"], c["rf"] = layernorm_forward(x, p["ln_f.g"], p["ln_f.b"], cfg.ln_eps)
    c["y"] = r(y)
    z = linear_forward(c["y"].reshape(B * S, d), r(p["wte"]))
    loss, dz = cross_entropy_forward_backward(z, tgt.reshape(-1))
    c["z"] = z
    c["dz"] = dz
    return loss, c


def backward_bf16_operands(cfg: GPT2Config, params, cache, dtype=np.float64, r=None):
    """Gradients under the bfloat16 precision model: the backward of
    :func:`backward` with every operand of every matrix product rounded by
    ``r`` (bfloat16 by default) -- weights, activations and the gradients that
    enter products (logits, GELU-input, attention-score, head-output and fused
    projection gradients) -- and nothing else: the softmax backward takes the
    unrounded probabilities (recomputed from the rounded q and k, as the
    forward formed them) and the bias gradients sum unrounded values. Needs
    the cache of ``forward(..., gemm_operands="bf16")``."""
    p = _cast(params, dtype)
    if r is None:
        r = lambda a: round_bf16(a).astype(dtype)  # noqa: E731
    B, S, d, H = cfg.batch, cfg.seq, cfg.d_model, cfg.n_head
    scale = 1.0 / math.sqrt(d // H)
    grads = {}
    dz = r(cache["dz"])
    dwte = dz.T @ cache["y"].reshape(B * S, d)
    dy = (dz @ r(p["wte"])).reshape(B, S, d)
    dx, grads["ln_f.g"], grads["ln_f.b"] = layernorm_backward(
        dy, cache["x_L"], cache["muf"], cache["rf"], p["ln_f.g"])
    for l in reversed(range(cfg.n_layer)):
        q = f"h{l}."
        c = cache["layers"][l]
        dxa = r(dx)
        grads[q + "proj.w"] = dxa.reshape(B * S, d).T @ c["g"].reshape(B * S, -1)
        grads[q + "proj.b"] = dx.sum(axis=(0, 1))
        du_f = gelu_backward(dxa @ r(p[q + "proj.w"]), c["u"])
        du = r(du_f)
        grads[q + "fc.w"] = du.reshape(B * S, -1).T @ c["h2"].reshape(B * S, d)
        grads[q + "fc.b"] = du_f.sum(axis=(0, 1))
        dh2 = du @ r(p[q + "fc.w"])
        dln, grads[q + "ln2.g"], grads[q + "ln2.b"] = layernorm_backward(
            dh2, c["x_mid"], c["mu2"], c["r2"], p[q + "ln2.g"])
        dx = dx + dln
        dxa = r(dx)
        grads[q + "o.w"] = dxa.reshape(B * S, d).T @ c["o"].reshape(B * S, d)
        grads[q + "o.b"] = dx.sum(axis=(0, 1))
        dO = split_heads(r(dxa @ r(p[q + "o.w"])), H)
        P = causal_softmax_forward((c["q"] @ c["k"].transpose(0, 1, 3, 2)) * scale)
        dv = r(P).transpose(0, 1, 3, 2) @ dO
        dP = dO @ c["v"].transpose(0, 1, 3, 2)
        dS = r(causal_softmax_backward(dP, P) * scale)
        dqkv_f = np.concatenate([merge_heads(dS @ c["k"]), merge_heads(dS.transpose(0, 1, 3, 2) @ c["q"]),
                                 merge_heads(dv)], axis=-1)
        dqkv = r(dqkv_f)
        grads[q + "qkv.w"] = dqkv.reshape(B * S, -1).T @ c["h1"].reshape(B * S, d)
        grads[q + "qkv.b"] = dqkv_f.sum(axis=(0, 1))
        dh1 = dqkv @ r(p[q + "qkv.w"])
        dln, grads[q + "ln1.g"], grads[q + "ln1.b"] = layernorm_backward(
            dh1, c["x_in"], c["mu1"], c["r1"], p[q + "ln1.g"])
        dx = dx + dln
    dwpe = np.zeros_like(p["wpe"])
    grads["wte"], grads["wpe"] = embedding_backward(dx, cache["ids"], dwte, dwpe)
    return grads


def backward(cfg: GPT2Config, params, cache, dtype=np.float64):
    """Reverse-mode gradients of the mean loss w.r.t. every parameter."""
    p = _cast(params, dtype)
    B, S, d = cfg.batch, cfg.seq, cfg.d_model
    grads = {}
    dz = cache["dz"]
    y = cache["y"].reshape(B * S, d)
    dwte = dz.T @ y
    dy = (dz @ p["wte"]).reshape(B, S, d)
    dx, grads["ln_f.g"], grads["ln_f.b"] = layernorm_backward(
        dy, cache["x_L"], cache["muf"], cache["rf"], p["ln_f.g"])
    for l in reversed(range(cfg.n_layer)):
        q = f"h{l}."
        c = cache["layers"][l]
        dg = dx @ p[q + "proj.w"]
        grads[q + "proj.w"] = dx.reshape(B * S, d).T @ c["g"].reshape(B * S, -1)
        grads[q + "proj.b"] = dx.sum(axis=(0, 1))
        du = gelu_backward(dg, c["u"])
        grads[q + "fc.w"] = du.reshape(B * S, -1).T @ c["h2"].reshape(B * S, d)
        grads[q + "fc.b"] = du.sum(axis=(0, 1))
        dh2 = du @ p[q + "fc.w"]
        dln, grads[q + "ln2.g"], grads[q + "ln2.b"] = layernorm_backward(
            dh2, c["x_mid"], c["mu2"], c["r2"], p[q + "ln2.g"])
        dx = dx + dln
        do = dx @ p[q + "o.w"]
        grads[q + "o.w"] = dx.reshape(B * S, d).T @ c["o"].reshape(B * S, d)
        grads[q + "o.b"] = dx.sum(axis=(0, 1))
        dqkv = attention_backward(do, c["qkv"], c["P"], cfg.n_head)
        grads[q + "qkv.w"] = dqkv.reshape(B * S, -1).T @ c["h1"].reshape(B * S, d)
        grads[q + "qkv.b"] = dqkv.sum(axis=(0, 1))
        dh1 = dqkv @ p[q + "qkv.w"]
        dln, grads[q + "ln1.g"], grads[q + "ln1.b"] = layernorm_backward(
            dh1, c["x_in"], c["mu1"], c["r1"], p[q + "ln1.g"])
        dx = dx + dln
    dwpe = np.zeros_like(p["wpe"])
    grads["wte"], grads["wpe"] = embedding_backward(dx, cache["ids"], dwte, dwpe)
    return grads


def scheduled_lr(hp: AdamWHyper, step: int) -> float:
    """Rate of AdamW iteration ``step`` (1-based) under the warm-up flags.

    README "Minimal working GPT example": --start-lr is the rate used for the
    first batch and --full-lr-iter the AdamW iteration that first uses the full
    --lr (1 = full rate from the start). Between the two the rate rises along a
    straight line (a reading: the pages name only the end points).
    """
    if hp.full_lr_iter <= 1 or step >= hp.full_lr_iter:
        return hp.lr
    return hp.start_lr + (hp.lr - hp.start_lr) * (step - 1) / (hp.full_lr_iter - 1)


def adamw_step(params, grads, m, v, step, hp: AdamWHyper, dtype=np.float64):
    """AdamW over every parameter; returns new (params, m, v) dictionaries.

    The rate is that of iteration ``step`` under the warm-up schedule.
    """
    hp = AdamWHyper(lr=scheduled_lr(hp, step), beta1=hp.beta1, beta2=hp.beta2, eps=hp.eps,
                    weight_decay=hp.weight_decay)
    new_p, new_m, new_v = {}, {}, {}
    for k in params:
        w = np.asarray(params[k], dtype=dtype)
        mk = np.zeros_like(w) if m is None else np.asarray(m[k], dtype=dtype)
        vk = np.zeros_like(w) if v is None else np.asarray(v[k], dtype=dtype)
        new_p[k], new_m[k], new_v[k] = adamw_update(w, np.asarray(grads[k], dtype=dtype),
                                                    mk, vk, step, hp)
    return new_p, new_m, new_v


def train_step(cfg: GPT2Config, params, windows, hp: AdamWHyper = AdamWHyper(),
               m=None, v=None, step=1, dtype=np.float64):
    """forward + backward + AdamW; returns (loss, grads, new_params, new_m, new_v)."""
    loss, cache = forward(cfg, params, windows, dtype)
    grads = backward(cfg, params, cache, dtype)
    new_p, new_m, new_v = adamw_step(params, grads, m, v, step, hp, dtype)
    return loss, grads, new_p, new_m, new_v


def batch_gradient(cfg: GPT2Config, params, minibatches, dtype=np.float64):
    """Loss and gradient of one optimizer batch given as a list of minibatches.

    README "Minimal working GPT example": --batch sequences form the batch, the
    optimizer step happens after the gradients of the whole batch are
    collected, and --minibatch sequences are processed at a time; the loss is
    the mean over all tokens (--loss-reduction=mean). Every minibatch here has
    the same shape, so the batch loss and its gradient are the means of the
    minibatch losses and gradients.
    """
    losses, total = [], None
    for windows in minibatches:
        loss, cache = forward(cfg, params, windows, dtype)
        grads = backward(cfg, params, cache, dtype)
        del cache
        losses.append(loss)
        total = grads if total is None else {n: total[n] + grads[n] for n in total}
    k = len(minibatches)
    return sum(losses) / k, {n: g / k for n, g in total.items()}


def train_batch(cfg: GPT2Config, params, minibatches, hp: AdamWHyper = AdamWHyper(),
                m=None, v=None, step=1, dtype=np.float64):
    """One optimizer step over a batch of minibatches; same returns as train_step."""
    loss, grads = batch_gradient(cfg, params, minibatches, dtype)
    new_p, new_m, new_v = adamw_step(params, grads, m, v, step, hp, dtype)
    return loss, grads, new_p, new_m, new_v


def train(cfg: GPT2Config, params, batches, hp: AdamWHyper = AdamWHyper(), dtype=np.float64):
    """Several optimizer steps; ``batches[i]`` is the list of minibatch windows of
    step i + 1. Returns (per-step batch losses, final params, m, v)."""
    m = v = None
    losses = []
    for i, mbs in enumerate(batches):
        loss, _, params, m, v = train_batch(cfg, params, mbs, hp, m, v, i + 1, dtype)
        losses.append(loss)
    return losses, params, m, v


def step_flops(cfg: GPT2Config) -> float:
    """Algorithmic FLOPs of one step: 3x the forward matmuls plus causal attention.

    Forward matmuls per token: 2*(d*3d + d*d + 2*d*f) per layer plus 2*d*V for
    the LM head; attention QK^T and PV count only the causal half
    (S(S+1)/2 key positions per query row, 2*hd flops each, two products).
    Backward is twice the forward. Elementwise work is not counted.
    """
    d, f, V, S, B, L = cfg.d_model, cfg.d_ff, cfg.vocab, cfg.seq, cfg.batch, cfg.n_layer
    T = B * S
    dense = 2.0 * T * (L * (3 * d * d + d * d + 2 * d * f) + d * V)
    attn = L * B * cfg.n_head * 2 * (2.0 * cfg.head_dim * S * (S + 1) / 2)
    return 3.0 * (dense + attn)


# --------------------------------------------------------------------------
# Layer-streamed bf16-operand step, for models whose parameters and gradients
# do not fit in host memory at once (the 8-layer, 26.6B-parameter wide GPT2 of
# the review page's "Core claim"). Same arithmetic as forward(...,
# gemm_operands="bf16") and backward_bf16_operands in float32; only one
# layer's parameters are held at a time, values the precision model rounds to
# bf16 are cached as bf16 bit patterns, and attention runs one sequence at a
# time.

def bf16_bits(a):
    """bfloat16 bit patterns (uint16) of :func:`round_bf16` of ``a``."""
    return (round_bf16(a).view(np.uint32) >> 16).astype(np.uint16)


def from_bf16_bits(b):
    """float32 values of bfloat16 bit patterns."""
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def forward_bf16_streamed(cfg: GPT2Config, layer_params, head_params, windows, dtype=np.float32):
    """Loss and cache of the bf16-operand forward, one layer in memory at a time.

    ``layer_params(l)`` returns layer l's tensors keyed without the ``h{l}.``
    prefix (weights may already be bf16-rounded: rounding is idempotent);
    ``head_params`` holds ``wte``, ``wpe``, ``ln_f.g``, ``ln_f.b``. ``dtype``
    is the arithmetic (float32, or float64 to measure what fp32 accumulation
    leaves undetermined)."""
    f32 = dtype
    r = lambda a: round_bf16(a).astype(f32)  # noqa: E731
    ids = windows[:, :cfg.seq].astype(np.int64)
    tgt = windows[:, 1:cfg.seq + 1].astype(np.int64)
    B, S, d, H = cfg.batch, cfg.seq, cfg.d_model, cfg.n_head
    scale = 1.0 / math.sqrt(d // H)
    wte = np.asarray(head_params["wte"], f32)
    c = {"ids": ids, "layers": []}
    x = embedding_forward(ids, wte, np.asarray(head_params["wpe"], f32))
    for l in range(cfg.n_layer):
        p = {k: np.asarray(v, f32) for k, v in layer_params(l).items()}
        L = {"x_in": x}
        h1, L["mu1"], L["r1"] = layernorm_forward(x, p["ln1.g"], p["ln1.b"], cfg.ln_eps)
        h1 = r(h1)
        L["h1"] = bf16_bits(h1)
        qkv = linear_forward(h1, r(p["qkv.w"]), p["qkv.b"])
        del h1
        q = split_heads(r(qkv[..., :d]), H)
        k = split_heads(r(qkv[..., d:2 * d]), H)
        v = split_heads(r(qkv[..., 2 * d:]), H)
        del qkv
        o = np.empty((B, H, S, d // H), f32)
        for b in range(B):
            P = r(causal_softmax_forward((q[b:b + 1] @ k[b:b + 1].transpose(0, 1, 3, 2)) * scale))
            o[b:b + 1] = P @ v[b:b + 1]
            del P
        L["q"], L["k"], L["v"] = bf16_bits(q), bf16_bits(k), bf16_bits(v)
        del q, k, v
        o = r(merge_heads(o))
        L["o"] = bf16_bits(o)
        x = x + linear_forward(o, r(p["o.w"]), p["o.b"])
        del o
        L["x_mid"] = x
        h2, L["mu2"], L["r2"] = layernorm_forward(x, p["ln2.g"], p["ln2.b"], cfg.ln_eps)
        h2 = r(h2)
        L["h2"] = bf16_bits(h2)
        L["u"] = linear_forward(h2, r(p["fc.w"]), p["fc.b"])
        del h2
        g = r(gelu_forward(L["u"]))
        L["g"] = bf16_bits(g)
        x = x + linear_forward(g, r(p["proj.w"]), p["proj.b"])
        del g, p
        c["layers"].append(L)
    c["x_L"] = x
    y, c["muf"], c["rf"] = layernorm_forward(x, np.asarray(head_params["ln_f.g"], f32),
                                              np.asarray(head_params["ln_f.b"], f32), cfg.ln_eps)
    y = r(y)
    c["y"] = bf16_bits(y)
    z = linear_forward(y.reshape(B * S, d), r(wte))
    loss, dz = cross_entropy_forward_backward(z, tgt.reshape(-1))
    c["z"] = z
    c["dz"] = dz
    return loss, c


def backward_bf16_streamed(cfg: GPT2Config, layer_params, head_params, cache, want=None,
                           dtype=np.float32, grad_dtype=None):
    """Gradients of the bf16-operand step (as :func:`backward_bf16_operands`),
    one layer in memory at a time, from the cache of
    :func:`forward_bf16_streamed`.

    ``want``: layer indices whose parameter gradients are returned (default:
    all). Other layers skip their weight- and bias-gradient sums, which feed
    nothing else; the gradients of wte, wpe and ln_f are always returned.
    ``dtype`` as in :func:`forward_bf16_streamed`; ``grad_dtype`` (default
    ``dtype``) is the type the returned gradients are stored in as soon as each
    is formed (float32 keeps an fp64 run's memory down)."""
    f32 = dtype
    r = lambda a: round_bf16(a).astype(f32)  # noqa: E731
    unpack = lambda b: from_bf16_bits(b).astype(f32)  # noqa: E731
    B, S, d, H = cfg.batch, cfg.seq, cfg.d_model, cfg.n_head
    T = B * S
    scale = 1.0 / math.sqrt(d // H)
    gdt = grad_dtype or dtype

    class _Grads(dict):
        def __setitem__(self, k, v):
            super().__setitem__(k, np.asarray(v).astype(gdt, copy=False))

    grads = _Grads()
    wte = np.asarray(head_params["wte"], f32)
    dz = r(cache["dz"])
    dwte = dz.T @ unpack(cache["y"]).reshape(T, d)
    dy = (dz @ r(wte)).reshape(B, S, d)
    del dz
    dx, grads["ln_f.g"], grads["ln_f.b"] = layernorm_backward(
        dy, cache["x_L"], cache["muf"], cache["rf"], np.asarray(head_params["ln_f.g"], f32))
    del dy
    for l in reversed(range(cfg.n_layer)):
        q = f"h{l}."
        c = cache["layers"][l]
        p = {k: np.asarray(v, f32) for k, v in layer_params(l).items()}
        keep = want is None or l in want
        dxa = r(dx)
        if keep:
            grads[q + "proj.w"] = dxa.reshape(T, d).T @ unpack(c["g"]).reshape(T, -1)
            grads[q + "proj.b"] = dx.sum(axis=(0, 1))
        du_f = gelu_backward(dxa @ r(p["proj.w"]), c["u"])
        du = r(du_f)
        if keep:
            grads[q + "fc.w"] = du.reshape(T, -1).T @ unpack(c["h2"]).reshape(T, d)
            grads[q + "fc.b"] = du_f.sum(axis=(0, 1))
        del du_f
        dh2 = du @ r(p["fc.w"])
        del du
        dln, g2, b2 = layernorm_backward(dh2, c["x_mid"], c["mu2"], c["r2"], p["ln2.g"])
        del dh2
        if keep:
            grads[q + "ln2.g"], grads[q + "ln2.b"] = g2, b2
        dx = dx + dln
        dxa = r(dx)
        if keep:
            grads[q + "o.w"] = dxa.reshape(T, d).T @ unpack(c["o"]).reshape(T, d)
            grads[q + "o.b"] = dx.sum(axis=(0, 1))
        dO = split_heads(r(dxa @ r(p["o.w"])), H)
        del dxa
        qh, kh, vh = unpack(c["q"]), unpack(c["k"]), unpack(c["v"])
        dqkv_f = np.empty((B, S, 3 * d), f32)
        for b in range(B):
            sl = slice(b, b + 1)
            P = causal_softmax_forward((qh[sl] @ kh[sl].transpose(0, 1, 3, 2)) * scale)
            dv = r(P).transpose(0, 1, 3, 2) @ dO[sl]
            dS = r(causal_softmax_backward(dO[sl] @ vh[sl].transpose(0, 1, 3, 2), P) * scale)
            del P
            dqkv_f[sl] = np.concatenate([merge_heads(dS @ kh[sl]),
                                         merge_heads(dS.transpose(0, 1, 3, 2) @ qh[sl]),
                                         merge_heads(dv)], axis=-1)
            del dS, dv
        del dO, qh, kh, vh
        dqkv = r(dqkv_f)
        if keep:
            grads[q + "qkv.w"] = dqkv.reshape(T, -1).T @ unpack(c["h1"]).reshape(T, d)
            grads[q + "qkv.b"] = dqkv_f.sum(axis=(0, 1))
        del dqkv_f
        dh1 = dqkv @ r(p["qkv.w"])
        del dqkv
        dln, g1, b1 = layernorm_backward(dh1, c["x_in"], c["mu1"], c["r1"], p["ln1.g"])
        del dh1, p
        if keep:
            grads[q + "ln1.g"], grads[q + "ln1.b"] = g1, b1
        dx = dx + dln
    grads["wte"], grads["wpe"] = embedding_backward(
        dx, cache["ids"], dwte, np.zeros_like(np.asarray(head_params["wpe"], f32)))
    return dict(grads)
