"""Tile kernels through the C ABI against the CPU oracle (GPU).

Tolerances (fp32 kernels): elementwise |gpu - ref| <= 1e-5 max(|ref|,
1e-6 max|ref|), i.e. 1e-5 relative with a floor a million times below the
tensor's largest value. Outputs that are sums whose terms cancel (LayerNorm
output gamma*xhat + beta, the LayerNorm and softmax gradients, GELU's
1 + tanh, column sums of random-sign values, the AdamW first moment and update)
carry the fp32 rounding of their terms, not of their value: for those the
reference magnitude is the magnitude of the terms (``terms=``), computed from
the same formula with absolute values. bf16 outputs: one bf16 rounding of the
fp32 value (2^-8 relative) on top. Embedding gather/scatter: bit-exact.
"""
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import gpt2 as O  # noqa: E402
from tile_task_transformer_gb300 import nnt, synth  # noqa: E402

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nnt.lib()


def close32(a, r, rtol=1e-5, terms=None):
    """|a - r| <= rtol * max(|r|, 1e-6 max|r|) elementwise; with ``terms`` (the
    magnitude of the terms whose sum r is, same shape) the larger of |r| and
    ``terms`` is the reference magnitude."""
    a = np.asarray(a, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    mag = np.abs(r)
    if terms is not None:
        mag = np.maximum(mag, np.asarray(terms, dtype=np.float64))
    floor = 1e-6 * max(np.abs(r).max(), 1e-30)
    err = np.abs(a - r) - rtol * np.maximum(mag, floor)
    assert err.max() <= 0, f"max excess {err.max():.3e} (largest |ref| {np.abs(r).max():.3e})"


def close_bf16(a, r):
    a = np.asarray(a, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    scale = max(np.abs(r).max(), 1e-30)
    assert (np.abs(a - r) <= 2.0 ** -8 * np.abs(r) + 1e-5 * scale).all()


def t(a, dtype=torch.float32):
    return torch.as_tensor(np.ascontiguousarray(a)).to(DEV, dtype)


def n(x):
    return x.float().cpu().numpy()


ACT = {nnt.F32: torch.float32, nnt.BF16: torch.bfloat16}


@pytest.mark.parametrize("rows,cols", [(7, 64), (33, 768), (64, 3072), (5, 8192), (3, 16384), (2, 32768)])
@pytest.mark.parametrize("dtype", [nnt.F32, nnt.BF16])
def test_layernorm_fwd(rows, cols, dtype):
    x = synth.normal_matrix(4, 1, (rows, cols), 1.0) + 0.5
    g = synth.normal_matrix(4, 2, (cols,), 1.0)
    b = synth.normal_matrix(4, 3, (cols,), 1.0)
    y = torch.empty(rows, cols, dtype=ACT[dtype], device=DEV)
    mu = torch.empty(rows, device=DEV)
    rs = torch.empty(rows, device=DEV)
    nnt.op_layernorm_fwd(t(x), t(g), t(b), y, mu, rs, rows, cols, 1e-5, dtype)
    torch.cuda.synchronize()
    ry, rmu, rrs = O.layernorm_forward(x.astype(np.float64), g, b, 1e-5)
    close32(n(mu), rmu, terms=np.abs(x).mean(axis=1))
    close32(n(rs), rrs)
    if dtype == nnt.F32:
        # y = g (x - mu) rstd + b: x - mu and the final sum both cancel
        xmag = (np.abs(x) + np.abs(rmu)[:, None]) * rrs[:, None]
        close32(n(y), ry, terms=np.abs(g) * xmag + np.abs(b))
    else:
        close_bf16(n(y), ry)


@pytest.mark.parametrize("rows,cols", [(9, 64), (130, 768), (300, 1024), (17, 8192)])
@pytest.mark.parametrize("resid", [False, True])
def test_layernorm_bwd(rows, cols, resid):
    x = synth.normal_matrix(5, 1, (rows, cols), 1.0)
    g = synth.normal_matrix(5, 2, (cols,), 1.0)
    dy = synth.normal_matrix(5, 3, (rows, cols), 1.0)
    r = synth.normal_matrix(5, 4, (rows, cols), 1.0)
    _, mu, rs = O.layernorm_forward(x.astype(np.float64), g, np.zeros(cols), 1e-5)
    mu32, rs32 = mu.astype(np.float32), rs.astype(np.float32)
    dx = torch.empty(rows, cols, device=DEV)
    dxa = torch.empty(rows, cols, dtype=torch.bfloat16, device=DEV)
    dg = torch.empty(cols, device=DEV)
    db = torch.empty(cols, device=DEV)
    rdev = t(r) if resid else None
    nnt.op_layernorm_bwd(t(dy), t(x), t(mu32), t(rs32), t(g), rdev, dx, dxa, dg, db, rows, cols, nnt.BF16)
    torch.cuda.synchronize()
    rdx, rdg, rdb = O.layernorm_backward(dy.astype(np.float64), x.astype(np.float64),
                                         mu32.astype(np.float64), rs32.astype(np.float64), g)
    # magnitudes of the cancelling terms: dx = rstd (gdy - mean(gdy) -
    # xhat mean(gdy xhat)) (+ resid), dgamma = sum dy xhat, dbeta = sum dy
    x64, dy64 = x.astype(np.float64), dy.astype(np.float64)
    xhat = (x64 - mu32[:, None]) * rs32[:, None]
    xmag = (np.abs(x64) + np.abs(mu32)[:, None]) * rs32[:, None]  # x - mu cancels too
    gdy = np.abs(g * dy64)
    dx_terms = rs32[:, None] * (gdy + gdy.mean(axis=1, keepdims=True)
                                + xmag * (gdy * xmag).mean(axis=1, keepdims=True))
    if resid:
        rdx = rdx + r
        dx_terms = dx_terms + np.abs(r)
    close32(n(dx), rdx, terms=dx_terms)
    close_bf16(n(dxa), n(dx))
    close32(n(dg), rdg, terms=np.abs(dy64 * xmag).sum(axis=0))
    close32(n(db), rdb, terms=np.abs(dy64).sum(axis=0))


@pytest.mark.parametrize("nmat,seq", [(3, 32), (2, 256), (4, 1024), (1, 2048)])
@pytest.mark.parametrize("dtype", [nnt.F32, nnt.BF16])
def test_softmax_causal(nmat, seq, dtype):
    s = synth.normal_matrix(6, 1, (nmat, seq, seq), 3.0)
    p = torch.full((nmat, seq, seq), float("nan"), dtype=ACT[dtype], device=DEV)
    nnt.op_softmax_causal_fwd(t(s), p, nmat, seq, dtype)
    torch.cuda.synchronize()
    rp = O.causal_softmax_forward(s.astype(np.float64))
    P = n(p)
    q = np.arange(seq)[:, None]
    k = np.arange(seq)[None, :]
    wend = np.minimum(seq, (q + 1 + 127) // 128 * 128)
    written = k < wend
    assert np.isfinite(P[:, written]).all()
    assert (P[:, written & (k > q)] == 0).all()
    chk = close32 if dtype == nnt.F32 else close_bf16
    chk(P[:, k <= q], rp[:, k <= q])
    if dtype == nnt.F32:  # rows sum to 1 within fp32 rounding
        assert np.abs(np.where(k <= q, P, 0.0).sum(axis=2) - 1).max() < 1e-5
    # backward on the forward's output
    dP = synth.normal_matrix(6, 2, (nmat, seq, seq), 1.0)
    ds = torch.full((nmat, seq, seq), float("nan"), dtype=ACT[dtype], device=DEV)
    scale = 1.0 / math.sqrt(64)
    nnt.op_softmax_causal_bwd(p, t(dP), ds, nmat, seq, scale, dtype)
    torch.cuda.synchronize()
    Pin = np.where(k <= q, P, 0.0).astype(np.float64)  # the kernel's P (unwritten tail excluded)
    rds = O.causal_softmax_backward(dP.astype(np.float64), Pin) * scale
    DS = n(ds)
    assert np.isfinite(DS[:, written]).all()
    assert (DS[:, written & (k > q)] == 0).all()
    if dtype == nnt.F32:
        # dS = scale P (dP - sum_k P dP): magnitude of the cancelling terms
        dPc = np.where(k <= q, dP.astype(np.float64), 0.0)
        ds_terms = scale * Pin * (np.abs(dPc) + (Pin * np.abs(dPc)).sum(axis=2, keepdims=True))
        close32(DS[:, k <= q], rds[:, k <= q], terms=ds_terms[:, k <= q])
    else:
        chk(DS[:, k <= q], rds[:, k <= q])


@pytest.mark.parametrize("dtype", [nnt.F32, nnt.BF16])
def test_gelu(dtype):
    N = 4 * 12345
    u = synth.normal_matrix(7, 1, (N,), 2.0)
    g = torch.empty(N, dtype=ACT[dtype], device=DEV)
    nnt.op_gelu_fwd(t(u), g, N, dtype)
    dg = synth.normal_matrix(7, 2, (N,), 1.0)
    du = torch.empty(N, dtype=ACT[dtype], device=DEV)
    dgt = t(dg, ACT[dtype])
    nnt.op_gelu_bwd(dgt, t(u), du, N, dtype)
    torch.cuda.synchronize()
    u64 = u.astype(np.float64)
    rg = O.gelu_forward(u64)
    rdu = O.gelu_backward(n(dgt).astype(np.float64), u64)
    if dtype == nnt.F32:
        # gelu(u) = u (1 + tanh(a))/2 and gelu'(u) = (1 + tanh(a))/2 + u (1 - tanh(a)^2) a'/2
        # cancel in 1 + tanh(a) for negative u: magnitudes of their terms
        c, k3 = math.sqrt(2 / math.pi), 0.044715
        th = np.tanh(c * (u64 + k3 * u64 ** 3))
        close32(n(g), rg, terms=0.5 * np.abs(u64) * (1 + np.abs(th)))
        dterm = 0.5 * (1 + np.abs(th)) + 0.5 * np.abs(u64) * (1 + th * th) * c * (1 + 3 * k3 * u64 ** 2)
        close32(n(du), rdu, terms=np.abs(n(dgt)) * dterm)
    else:
        close_bf16(n(g), rg)
        close_bf16(n(du), rdu)


# Both kernels on every shape. The cluster-pair kernel holds rows of up to 55296
# logits in shared memory, half a row per CTA: more rows than clusters in the
# 300-row case, padding past the columns, a second half that is empty (3
# columns) or holds only the tail (5); 60000 logits always take the two-pass
# kernel.
@pytest.mark.parametrize("rows,cols,pad", [(5, 256, 0), (64, 50257, 0), (3, 1000, 0),
                                           (300, 50257, 0), (7, 1000, 4000), (9, 3, 0),
                                           (2, 5, 0), (3, 60000, 0)])
@pytest.mark.parametrize("dtype", [nnt.F32, nnt.BF16])
@pytest.mark.parametrize("kernel", ["pair", "twopass"])
def test_cross_entropy(rows, cols, pad, dtype, kernel, monkeypatch):
    monkeypatch.setenv("NNT_CE_KERNEL", kernel)
    ldz = (cols + 3) // 4 * 4 + pad
    lddz = (cols + 7) // 8 * 8
    z = np.zeros((rows, ldz), np.float32)
    z[:, :cols] = synth.normal_matrix(8, 1, (rows, cols), 3.0)
    tgt = (synth.bits(8, 2, 0, rows) % np.uint64(cols)).astype(np.uint16)
    dz = torch.full((rows, lddz), float("nan"), dtype=ACT[dtype], device=DEV)
    rl = torch.empty(rows, device=DEV)
    loss = torch.empty(1, device=DEV)
    tg = torch.as_tensor(tgt.view(np.int16)).to(DEV)
    nnt.op_cross_entropy(t(z), rows, cols, ldz, tg, 1, dz, lddz, rl, loss, dtype)
    torch.cuda.synchronize()
    rloss, rdz = O.cross_entropy_forward_backward(z[:, :cols].astype(np.float64), tgt.astype(np.int64))
    assert abs(loss.item() - rloss) <= 1e-5 * abs(rloss)
    D = n(dz)
    assert (D[:, cols:] == 0).all()
    (close32 if dtype == nnt.F32 else close_bf16)(D[:, :cols], rdz)


def test_cross_entropy_uniform_logits_is_log_vocab():
    rows, cols = 16, 50257
    ldz = 50260
    z = torch.zeros(rows, ldz, device=DEV)
    tg = torch.arange(rows, dtype=torch.int16, device=DEV)
    dz = torch.empty(rows, ldz, device=DEV)
    rl = torch.empty(rows, device=DEV)
    loss = torch.empty(1, device=DEV)
    nnt.op_cross_entropy(z, rows, cols, ldz, tg, 1, dz, ldz, rl, loss, nnt.F32)
    torch.cuda.synchronize()
    assert abs(loss.item() - math.log(cols)) < 1e-5


def test_adamw():
    N = 1_000_003
    w = synth.normal_matrix(9, 1, (N,), 0.02)
    g = synth.normal_matrix(9, 2, (N,), 1e-3)
    m0 = synth.normal_matrix(9, 3, (N,), 1e-4)
    v0 = np.abs(synth.normal_matrix(9, 4, (N,), 1e-6))
    # the oracle gets the hyper-parameters as the kernel receives them (fp32):
    # 1 - beta2 of the fp32 0.999 is 1.3e-5 away from 1 - 0.999
    f32 = lambda v: float(np.float32(v))  # noqa: E731
    h0 = O.AdamWHyper()
    hp = O.AdamWHyper(lr=f32(h0.lr), beta1=f32(h0.beta1), beta2=f32(h0.beta2), eps=f32(h0.eps),
                      weight_decay=f32(h0.weight_decay))
    step = 7
    bc1, bc2 = f32(1 - hp.beta1 ** step), f32(1 - hp.beta2 ** step)
    W, G, M, V = t(w), t(g), t(m0), t(v0)
    Wb = torch.empty(N, dtype=torch.bfloat16, device=DEV)
    nnt.op_adamw(W, G, M, V, Wb, N, hp.lr, hp.beta1, hp.beta2, hp.eps, hp.weight_decay, bc1, bc2)
    torch.cuda.synchronize()
    rw, rm, rv = O.adamw_update(w.astype(np.float64), g.astype(np.float64), m0.astype(np.float64),
                                v0.astype(np.float64), step, hp)
    w64, g64, m64, v64 = (a.astype(np.float64) for a in (w, g, m0, v0))
    # m = b1 m0 + (1 - b1) g can cancel; v = b2 v0 + (1 - b2) g^2 cannot
    close32(n(M), rm, terms=hp.beta1 * np.abs(m64) + (1 - hp.beta1) * np.abs(g64))
    close32(n(V), rv)
    # w_new = w - lr wd w - lr mhat / (sqrt(vhat) + eps): the terms can cancel
    upd_terms = hp.lr * (hp.weight_decay * np.abs(w64) + np.abs(rm / bc1) / (np.sqrt(rv / bc2) + hp.eps))
    close32(n(W), rw, terms=np.abs(w64) + upd_terms)
    # the update w_new - w itself to 1e-4 of its terms; the fp32 roundings of
    # w - lr wd w and of w_new (half an ulp each) are part of the difference
    close32(n(W) - w64, rw - w64, rtol=1e-4, terms=upd_terms + 2.0 ** -23 * (np.abs(w64) + np.abs(rw)) / 1e-4)
    assert torch.equal(Wb, W.to(torch.bfloat16))


@pytest.mark.parametrize("B,S,d,V", [(2, 32, 64, 256), (4, 1024, 768, 50257), (3, 100, 16, 7)])
def test_embedding_bit_exact(B, S, d, V):
    ids = (synth.bits(10, 1, 0, B * (S + 1)) % np.uint64(V)).astype(np.uint16).reshape(B, S + 1)
    wte = synth.normal_matrix(10, 2, (V, d), 0.02)
    wpe = synth.normal_matrix(10, 3, (S, d), 0.02)
    x = torch.empty(B, S, d, device=DEV)
    idt = torch.as_tensor(ids.view(np.int16)).to(DEV)
    nnt.op_embedding_fwd(idt, S + 1, t(wte), t(wpe), x, B, S, d, V)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(n(x), O.embedding_forward(ids[:, :S], wte, wpe))
    dx = synth.normal_matrix(10, 4, (B, S, d), 1.0)
    dwte0 = synth.normal_matrix(10, 5, (V, d), 1.0)
    dwpe0 = synth.normal_matrix(10, 6, (S, d), 1.0)
    DW, DP = t(dwte0), t(dwpe0)
    nnt.op_embedding_bwd(idt, S + 1, t(dx), DW, DP, B, S, d, V)
    torch.cuda.synchronize()
    rw, rp = O.embedding_backward(dx, ids[:, :S], dwte0, dwpe0)
    np.testing.assert_array_equal(n(DW), rw)
    np.testing.assert_array_equal(n(DP), rp)


def test_token_out_of_range_sets_error_word():
    B, S, d, V = 1, 8, 16, 10
    ids = np.arange(S + 1, dtype=np.uint16).reshape(1, S + 1) * 2  # ids up to 16 >= V
    wte = np.zeros((V, d), np.float32)
    wpe = np.zeros((S, d), np.float32)
    x = torch.empty(B, S, d, device=DEV)
    nnt.read_device_error()
    nnt.op_embedding_fwd(torch.as_tensor(ids.view(np.int16)).to(DEV), S + 1, t(wte), t(wpe), x, B, S, d, V)
    assert nnt.read_device_error() & 1
    assert nnt.read_device_error() == 0


@pytest.mark.parametrize("M,N,K", [(64, 64, 64), (100, 70, 33), (256, 512, 768), (129, 257, 1000)])
@pytest.mark.parametrize("at,bt", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_gemm_cuda_cores_fp32(M, N, K, at, bt):
    A = synth.normal_matrix(11, 1, (K, M) if at else (M, K), 1.0)
    Bm = synth.normal_matrix(11, 2, (K, N) if bt else (N, K), 1.0)
    C = torch.empty(M, N, device=DEV)
    nnt.op_gemm(t(A), M if at else K, at, t(Bm), N if bt else K, bt, C, N, nnt.F32, M, N, K,
                dtype=nnt.F32, backend=1)
    torch.cuda.synchronize()
    a = A.T if at else A
    b = Bm if bt else Bm.T
    ref = a.astype(np.float64) @ b.astype(np.float64)
    err = np.abs(n(C) - ref).max() / np.abs(ref).max()
    assert err < 1e-5


def _bf16_round(a):
    return torch.as_tensor(a).to(torch.bfloat16).float().numpy().astype(np.float64)


@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 512, 768), (300, 200, 1000), (64, 64, 16),
                                   (1024, 2304, 768), (4096, 768, 3072), (200, 50257, 64)])
@pytest.mark.parametrize("at,bt", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_gemm_tensor_cores_bf16(M, N, K, at, bt):
    """tcgen05 GEMM vs fp64 products of the same bf16 inputs."""
    if (at and M % 8) or (bt and N % 8) or (not at and K % 8) or (not bt and K % 8):
        pytest.skip("leading dimension must be a multiple of 8 for TMA")
    A = synth.normal_matrix(12, 1, (K, M) if at else (M, K), 1.0)
    Bm = synth.normal_matrix(12, 2, (K, N) if bt else (N, K), 1.0)
    At, Bt = t(A, torch.bfloat16), t(Bm, torch.bfloat16)
    ldc = (N + 3) // 4 * 4
    C = torch.full((M, ldc), float("nan"), device=DEV)
    nnt.op_gemm(At, M if at else K, at, Bt, N if bt else K, bt, C, ldc, nnt.F32, M, N, K,
                dtype=nnt.BF16, backend=0)
    torch.cuda.synchronize()
    assert nnt.read_device_error() == 0
    a = _bf16_round(A)
    b = _bf16_round(Bm)
    ref = (a.T if at else a) @ (b if bt else b.T)
    err = np.abs(n(C)[:, :N] - ref).max() / np.abs(ref).max()
    assert err < 1e-5, err


def test_gemm_tensor_cores_bf16_out_and_accumulate():
    M, N, K = 256, 384, 512
    A = synth.normal_matrix(13, 1, (M, K), 1.0)
    Bm = synth.normal_matrix(13, 2, (N, K), 1.0)
    C0 = synth.normal_matrix(13, 3, (M, N), 1.0)
    C = t(C0)
    nnt.op_gemm(t(A, torch.bfloat16), K, 0, t(Bm, torch.bfloat16), K, 0, C, N, nnt.F32, M, N, K,
                alpha=0.5, beta=1.0, dtype=nnt.BF16, backend=0)
    Cb = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    nnt.op_gemm(t(A, torch.bfloat16), K, 0, t(Bm, torch.bfloat16), K, 0, Cb, N, nnt.BF16, M, N, K,
                dtype=nnt.BF16, backend=0)
    torch.cuda.synchronize()
    ref = _bf16_round(A) @ _bf16_round(Bm).T
    assert np.abs(n(C) - (C0 + 0.5 * ref)).max() / np.abs(ref).max() < 1e-5
    close_bf16(n(Cb), ref)


@pytest.mark.parametrize("B,S,d,V", [(32, 1024, 768, 50257), (17, 1000, 64, 300)])
def test_embedding_scatter_beyond_one_sort_block(B, S, d, V):
    """More tokens than one CTA of the token sort holds (16384): the blocks are
    sorted separately and each id's runs are added block by block, still in
    token order, so the result stays bit-exact."""
    ids = (synth.bits(14, 1, 0, B * (S + 1)) % np.uint64(V)).astype(np.uint16).reshape(B, S + 1)
    dx = synth.normal_matrix(14, 2, (B, S, d), 1.0)
    dwte0 = synth.normal_matrix(14, 3, (V, d), 1.0)
    dwpe0 = synth.normal_matrix(14, 4, (S, d), 1.0)
    DW, DP = t(dwte0), t(dwpe0)
    nnt.op_embedding_bwd(torch.as_tensor(ids.view(np.int16)).to(DEV), S + 1, t(dx), DW, DP, B, S, d, V)
    torch.cuda.synchronize()
    rw, rp = O.embedding_backward(dx, ids[:, :S], dwte0, dwpe0)
    np.testing.assert_array_equal(n(DW), rw)
    np.testing.assert_array_equal(n(DP), rp)
