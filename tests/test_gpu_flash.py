"""Fused causal attention (flash) tile task through the C ABI against the oracle (GPU).

The oracle is the plain definition (scores, causal softmax, P V and their
gradients in fp64) on the same bf16-valued q, k, v, dO. The fused kernels
multiply bf16 operands (P and dS rounded to bf16) with fp32 accumulation and
write bf16 outputs, so outputs and gradients are compared normwise
(max|gpu - ref| / max|ref|) within 2e-2, the step's bf16 tolerance; the
log-sum-exp within 2e-3 absolute (fp32 sums).
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import gpt2 as O  # noqa: E402
from tile_task_transformer_gb300 import nnt  # noqa: E402

pytestmark = pytest.mark.gpu

TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nnt.lib()


def relerr(a, r):
    return float(np.abs(np.asarray(a, np.float64) - r).max() / max(np.abs(r).max(), 1e-30))


def bf16_tensor(x):
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).cuda()


def as_np(t):
    return t.float().cpu().numpy().astype(np.float64)


def oracle(q, k, v, do):
    """Per (sequence, head) item: O, lse (base 2), dq, dk, dv in fp64."""
    Z, S, hd = q.shape
    qkv = np.concatenate([q, k, v], axis=-1)  # [Z, S, 3 hd]: one head per item
    out, P = O.attention_forward(qkv, 1)
    sc = (q @ k.transpose(0, 2, 1)) / math.sqrt(hd)
    lse2 = O.causal_logsumexp(sc) / math.log(2.0)
    d = O.attention_backward(do, qkv, P, 1)
    return out, lse2, d[..., :hd], d[..., hd:2 * hd], d[..., 2 * hd:]


def run(q, k, v, do, Z, S, hd):
    tq, tk, tv, tdo = (bf16_tensor(x) for x in (q, k, v, do))
    to = torch.empty_like(tq)
    lse = torch.empty((Z, S), dtype=torch.float32, device="cuda")
    nnt.op_flash_attention_fwd(tq, tk, tv, to, lse, Z, S, hd)
    dq, dk, dv = (torch.empty_like(tq) for _ in range(3))
    nnt.op_flash_attention_bwd(tq, tk, tv, to, tdo, lse, dq, dk, dv, Z, S, hd)
    torch.cuda.synchronize()
    code = nnt.read_device_error()
    assert code == 0, code
    return as_np(to), lse.cpu().numpy().astype(np.float64), as_np(dq), as_np(dk), as_np(dv)


def inputs(seed, Z, S, hd, qscale=1.0):
    rng = np.random.default_rng(seed)
    r = lambda s=1.0: as_np(bf16_tensor(s * rng.standard_normal((Z, S, hd))))  # noqa: E731
    return r(qscale), r(), r(), r()


@pytest.mark.parametrize("Z,S,hd", [
    (3, 128, 64),     # one block
    (2, 200, 64),     # ragged tail inside the second block
    (4, 513, 64),     # five blocks, one-row tail
    (3, 1024, 64),    # eight blocks: every operand stage and buffer of the pipelined
                      # dK/dV kernel is reused (S a multiple of 8: dS^T stored, dQ by GEMM)
    (2, 384, 128),    # head size 128, three blocks
    (2, 257, 128),    # head size 128, ragged
    (1, 1, 64),       # a single position: O = v, all gradients but dv zero
])
def test_flash_attention_matches_oracle(Z, S, hd):
    q, k, v, do = inputs(Z * 1000 + S + hd, Z, S, hd)
    got = run(q, k, v, do, Z, S, hd)
    ref = oracle(q, k, v, do)
    names = ["o", "lse", "dq", "dk", "dv"]
    errs = {}
    for n, g, r in zip(names, got, ref):
        if n == "lse":
            errs[n] = float(np.abs(g - r).max())
            assert errs[n] < 2e-3, (n, errs[n])
        elif np.abs(r).max() == 0:
            assert np.abs(g).max() == 0, n
        else:
            errs[n] = relerr(g, r)
            assert errs[n] < TOL, (n, errs[n])
    print("normwise errors", {n: f"{e:.2e}" for n, e in errs.items()})


def test_flash_attention_large_scores_force_rescaling():
    """Scores of spread ~30 with the row maximum moving late in the row make the
    running maximum grow by more than 2^8 between key blocks, exercising the
    rescale of O and of the row sums."""
    Z, S, hd = 2, 640, 64
    rng = np.random.default_rng(5)
    q = rng.standard_normal((Z, S, hd))
    k = rng.standard_normal((Z, S, hd)) * np.linspace(0.2, 3.0, S)[None, :, None]
    q, k = as_np(bf16_tensor(3.0 * q)), as_np(bf16_tensor(k))
    v = as_np(bf16_tensor(rng.standard_normal((Z, S, hd))))
    do = as_np(bf16_tensor(rng.standard_normal((Z, S, hd))))
    got = run(q, k, v, do, Z, S, hd)
    ref = oracle(q, k, v, do)
    assert np.abs(got[1] - ref[1]).max() < 2e-3 * max(1.0, np.abs(ref[1]).max())
    for i in (0, 2, 3, 4):
        assert relerr(got[i], ref[i]) < TOL, i


def test_flash_attention_backward_is_deterministic():
    Z, S, hd = 3, 300, 64
    q, k, v, do = inputs(77, Z, S, hd)
    a = run(q, k, v, do, Z, S, hd)
    b = run(q, k, v, do, Z, S, hd)
    for x, y in zip(a, b):
        np.testing.assert_array_equal(x, y)


def test_flash_attention_rejects_unsupported_head_size():
    t = torch.zeros((1, 16, 32), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((1, 16), dtype=torch.float32, device="cuda")
    with pytest.raises(nnt.NNTError) as e:
        nnt.op_flash_attention_fwd(t, t, t, t, lse, 1, 16, 32)
    assert e.value.status == nnt.ERR_INVALID_ARG
