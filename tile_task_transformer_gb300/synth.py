"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

This module holds no arithmetic of the training step itself: only a counter-based
random generator and the recipes that turn it into GPT2 weights and token windows.

Generator (both sides implement it from its published definitions):
  * splitmix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
    generators", OOPSLA 2014): z += 0x9E3779B97F4A7C15; two xor-shift-multiply
    rounds; final xor-shift.
  * a stream is keyed by ``key = splitmix64(splitmix64(seed) ^ stream)``; its
    element ``i`` is ``splitmix64(key + i)`` (mod 2**64).
  * uniform double in (0, 1): ``((bits >> 11) + 0.5) * 2**-53``.
  * normal: Box and Muller (1958) on the pair of uniforms (2j, 2j+1); element
    2j takes the cosine branch, 2j+1 the sine branch; the double is scaled by
    ``std`` and rounded once to fp32.

Token ids stand in for the nanoGPT-style uint16 ``train.bin`` stream the NNTile
README's GPT example reads ("Minimal working GPT example"): ``id = bits % vocab``.
The library's device-side initialiser (``nnt_create_model`` with a seed)
implements the same generator, so large models need no host-side generation.
"""
from __future__ import annotations

import numpy as np

_GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# stream ids: parameter tensor i uses stream i; tokens use TOKEN_STREAM
TOKEN_STREAM = 0xF00D


def splitmix64(x):
    """splitmix64 finaliser applied elementwise to uint64 values (wrapping)."""
    x = np.asarray(x, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = x + _GOLDEN
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        return z ^ (z >> np.uint64(31))


def stream_key(seed: int, stream: int) -> np.uint64:
    return splitmix64(splitmix64(np.uint64(seed & 0xFFFFFFFFFFFFFFFF)) ^ np.uint64(stream))


def bits(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    """``count`` 64-bit outputs of the stream, elements ``start .. start+count-1``."""
    key = stream_key(seed, stream)
    idx = np.arange(start, start + count, dtype=np.uint64)
    with np.errstate(over="ignore"):
        return splitmix64(key + idx)


def uniform01(seed: int, stream: int, start: int, count: int) -> np.ndarray:
    b = bits(seed, stream, start, count)
    return ((b >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def _normal_pairs(seed, stream, p0, n, count, std, out):
    u = uniform01(seed, stream, 2 * p0, 2 * n).reshape(n, 2)
    r = np.sqrt(-2.0 * np.log(u[:, 0]))
    t = 2.0 * np.pi * u[:, 1]
    z = np.empty((n, 2), dtype=np.float64)
    z[:, 0] = r * np.cos(t)
    z[:, 1] = r * np.sin(t)
    z = z.reshape(-1)
    e = min(2 * (p0 + n), count)
    out[2 * p0:e] = (z[: e - 2 * p0] * std).astype(np.float32)


def normal_f32(seed: int, stream: int, count: int, std: float) -> np.ndarray:
    """``count`` N(0, std^2) values rounded to fp32 (Box-Muller, see module doc).

    Large requests are generated in chunks on a thread pool (numpy releases the
    interpreter lock in its element-wise loops); the values do not depend on it.
    """
    out = np.empty(count, dtype=np.float32)
    chunk = 1 << 22  # pairs per chunk, to bound temporary memory
    npairs = (count + 1) // 2
    starts = list(range(0, npairs, chunk))
    if len(starts) <= 1:
        for p0 in starts:
            _normal_pairs(seed, stream, p0, min(chunk, npairs - p0), count, std, out)
        return out
    import concurrent.futures as cf
    import os
    with cf.ThreadPoolExecutor(max_workers=min(len(starts), os.cpu_count() or 4)) as ex:
        list(ex.map(lambda p0: _normal_pairs(seed, stream, p0, min(chunk, npairs - p0), count, std, out),
                    starts))
    return out


def token_windows(seed: int, batch: int, seq: int, vocab: int) -> np.ndarray:
    """``[batch, seq+1]`` uint16 windows; inputs are ``[:, :seq]``, targets ``[:, 1:]``."""
    n = batch * (seq + 1)
    b = bits(seed, TOKEN_STREAM, 0, n)
    return (b % np.uint64(vocab)).astype(np.uint16).reshape(batch, seq + 1)


def param_names_shapes(n_layer: int, d_model: int, d_ff: int, vocab: int, n_ctx: int):
    """Parameter tensors in their fixed order, weights as ``[out, in]``.

    Order: wte, wpe, per layer (ln1.g, ln1.b, qkv.w, qkv.b, o.w, o.b, ln2.g,
    ln2.b, fc.w, fc.b, proj.w, proj.b), then ln_f.g, ln_f.b.
    """
    d, f = d_model, d_ff
    out = [("wte", (vocab, d)), ("wpe", (n_ctx, d))]
    for l in range(n_layer):
        p = f"h{l}."
        out += [
            (p + "ln1.g", (d,)), (p + "ln1.b", (d,)),
            (p + "qkv.w", (3 * d, d)), (p + "qkv.b", (3 * d,)),
            (p + "o.w", (d, d)), (p + "o.b", (d,)),
            (p + "ln2.g", (d,)), (p + "ln2.b", (d,)),
            (p + "fc.w", (f, d)), (p + "fc.b", (f,)),
            (p + "proj.w", (d, f)), (p + "proj.b", (d,)),
        ]
    out += [("ln_f.g", (d,)), ("ln_f.b", (d,))]
    return out


def gpt2_tensor(seed: int, index: int, name: str, shape, std: float = 0.02,
                zero_bias: bool = False) -> np.ndarray:
    """Parameter tensor ``index`` (named ``name``) of :func:`param_names_shapes`:
    LayerNorm gains 1 and shifts 0, other tensors N(0, std) from stream ``index``
    (biases 0 with ``zero_bias``)."""
    n = int(np.prod(shape))
    if name.endswith(".g") and ("ln" in name):
        a = np.ones(n, dtype=np.float32)
    elif name.endswith(".b") and ("ln" in name):
        a = np.zeros(n, dtype=np.float32)
    elif zero_bias and name.endswith(".b"):
        a = np.zeros(n, dtype=np.float32)
    else:
        a = normal_f32(seed, index, n, std)
    return a.reshape(shape)


def gpt2_params(seed: int, n_layer: int, d_model: int, d_ff: int, vocab: int, n_ctx: int,
                std: float = 0.02, zero_bias: bool = False) -> dict:
    """Seeded fp32 GPT2 parameters: N(0, std) weights and biases, LayerNorm g=1, b=0.

    Tensor ``i`` of :func:`param_names_shapes` draws from stream ``i``.
    """
    return {name: gpt2_tensor(seed, i, name, shape, std, zero_bias)
            for i, (name, shape) in enumerate(param_names_shapes(n_layer, d_model, d_ff, vocab, n_ctx))}


def normal_matrix(seed: int, stream: int, shape, std: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    return normal_f32(seed, stream, n, std).reshape(shape)
