"""ctypes binding of libnnt.so (C ABI declared in include/nnt.h).

Argument marshalling only: every step of the training step runs in the
library's CUDA kernels. Device buffers are passed as raw pointers (e.g. a torch
tensor's ``data_ptr()``), streams as ``cudaStream_t`` handles (``stream.cuda_stream``).
If the library has not been built, :func:`lib` raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os
import re

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libnnt.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "nnt.h")

OK, ERR_INVALID_ARG, ERR_OOM, ERR_CUDA, ERR_TIMEOUT, ERR_STATE, ERR_INTERNAL = range(7)
F32, BF16 = 0, 1
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "OOM", 3: "CUDA", 4: "TIMEOUT", 5: "STATE",
                6: "INTERNAL"}


class NNTError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"nnt error {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


class Config(C.Structure):
    _fields_ = [("n_layer", C.c_int32), ("d_model", C.c_int32), ("n_head", C.c_int32),
                ("d_ff", C.c_int32), ("vocab", C.c_int32), ("n_ctx", C.c_int32),
                ("batch", C.c_int32), ("dtype", C.c_int32), ("ln_eps", C.c_float)]


class Tiles(C.Structure):
    _fields_ = [("batch_tile", C.c_int32), ("seq_tile", C.c_int32), ("embd_tile", C.c_int32),
                ("inner_tile", C.c_int32), ("head_tile", C.c_int32), ("vocab_tile", C.c_int32)]


class Options(C.Structure):
    _fields_ = [("stream", C.c_void_p), ("hbm_budget_bytes", C.c_uint64),
                ("allow_host_offload", C.c_int32), ("init_seed", C.c_uint64),
                ("init_std", C.c_float), ("init_zero_bias", C.c_int32), ("n_streams", C.c_int32),
                ("use_cuda_graph", C.c_int32), ("timeout_ms", C.c_uint32),
                ("gemm_backend", C.c_int32), ("trace", C.c_int32),
                ("gemm_min_task_cols", C.c_int32), ("flash_attention", C.c_int32),
                ("host_budget_bytes", C.c_uint64)]


class AdamW(C.Structure):
    _fields_ = [("lr", C.c_float), ("beta1", C.c_float), ("beta2", C.c_float), ("eps", C.c_float),
                ("weight_decay", C.c_float), ("start_lr", C.c_float), ("full_lr_iter", C.c_int32)]


class Stats(C.Structure):
    _fields_ = [("last_forward_ms", C.c_double), ("last_backward_ms", C.c_double),
                ("last_adamw_ms", C.c_double), ("device_bytes", C.c_uint64),
                ("host_pinned_bytes", C.c_uint64), ("h2d_bytes", C.c_uint64),
                ("d2h_bytes", C.c_uint64), ("n_tasks_forward", C.c_int64),
                ("n_tasks_backward", C.c_int64), ("n_tasks_adamw", C.c_int64),
                ("n_tiles", C.c_int64), ("n_params", C.c_int64), ("n_streams", C.c_int32),
                ("offload_active", C.c_int32), ("kernels_forward", C.c_int64),
                ("kernels_backward", C.c_int64), ("kernels_adamw", C.c_int64),
                ("flash_attention", C.c_int32)]


_P = C.c_void_p
_I64 = C.c_int64
_I32 = C.c_int32
_F = C.c_float
_SIGS = {
    "nnt_create_model": (C.c_int, [C.POINTER(Config), C.POINTER(Tiles), C.POINTER(Options), C.POINTER(_P)]),
    "nnt_plan_memory": (C.c_int, [C.POINTER(Config), C.POINTER(Tiles), C.POINTER(Options),
                                  C.POINTER(C.c_uint64), C.POINTER(C.c_uint64)]),
    "nnt_forward": (C.c_int, [_P, _P, _I32, C.POINTER(_F)]),
    "nnt_backward": (C.c_int, [_P]),
    "nnt_backward_accumulate": (C.c_int, [_P]),
    "nnt_adamw_step": (C.c_int, [_P, C.POINTER(AdamW)]),
    "nnt_backward_adamw": (C.c_int, [_P, C.POINTER(AdamW)]),
    "nnt_destroy": (None, [_P]),
    "nnt_num_params": (_I32, [_P]),
    "nnt_param_info": (C.c_int, [_P, _I32, C.POINTER(C.c_char_p), C.POINTER(_I64)]),
    "nnt_get_param": (C.c_int, [_P, _I32, _P]),
    "nnt_set_param": (C.c_int, [_P, _I32, _P]),
    "nnt_get_grad": (C.c_int, [_P, _I32, _P]),
    "nnt_get_adam_state": (C.c_int, [_P, _I32, _I32, _P]),
    "nnt_get_logits": (C.c_int, [_P, _P]),
    "nnt_get_stats": (C.c_int, [_P, C.POINTER(Stats)]),
    "nnt_get_task_times": (_I32, [_P, _I32, C.POINTER(C.c_char_p), C.POINTER(_I64),
                                  C.POINTER(C.c_double), C.POINTER(C.c_double), C.POINTER(C.c_double)]),
    "nnt_last_error": (C.c_char_p, [_P]),
    "nnt_set_trace": (C.c_int, [_P, _I32]),
    "nnt_op_layernorm_fwd": (C.c_int, [_P, _P, _P, _P, _P, _P, _I64, _I64, _F, _I32, _P]),
    "nnt_op_layernorm_bwd": (C.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I32, _P]),
    "nnt_op_softmax_causal_fwd": (C.c_int, [_P, _P, _I64, _I64, _I32, _P]),
    "nnt_op_softmax_causal_bwd": (C.c_int, [_P, _P, _P, _I64, _I64, _F, _I32, _P]),
    "nnt_op_flash_attention_fwd": (C.c_int, [_P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "nnt_op_flash_attention_bwd": (C.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "nnt_op_gelu_fwd": (C.c_int, [_P, _P, _I64, _I32, _P]),
    "nnt_op_gelu_bwd": (C.c_int, [_P, _P, _P, _I64, _I32, _P]),
    "nnt_op_cross_entropy": (C.c_int, [_P, _I64, _I64, _I64, _P, _I64, _P, _I64, _P, _P, _I32, _P]),
    "nnt_op_adamw": (C.c_int, [_P, _P, _P, _P, _P, _I64, _F, _F, _F, _F, _F, _F, _F, _P]),
    "nnt_op_embedding_fwd": (C.c_int, [_P, _I64, _P, _P, _P, _I64, _I64, _I64, _I64, _P]),
    "nnt_op_embedding_bwd": (C.c_int, [_P, _I64, _P, _P, _P, _I64, _I64, _I64, _I64, _P]),
    "nnt_op_embedding_bwd_noalloc": (C.c_int, [_P, _I64, _P, _P, _P, _I64, _I64, _I64, _I64, _P]),
    "nnt_op_gemm": (C.c_int, [_P, _I64, _I32, _P, _I64, _I32, _P, _I64, _I32, _I64, _I64, _I64, _F,
                              _F, _I32, _I32, _P]),
    "nnt_op_read_error": (C.c_int, [C.POINTER(C.c_uint32), _P]),
    "nnt_set_fault_injection": (C.c_int, [_I32, _I64]),
    "nnt_op_wait_selftest": (C.c_int, [_I64, _I32, _P]),
    "nnt_plan_schedule": (C.c_int, [_I32, _P, _P, _P, _P, _P, _I32, _P, _P, _P, _I64, _P, _P, _I64]),
}

_lib = None


def lib():
    """Load libnnt.so (built by ``tile_task_transformer_gb300.build``); raises if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build the CUDA library first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def header_symbols():
    """Names of the functions include/nnt.h declares."""
    with open(HEADER) as fh:
        text = fh.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nnt_[a-z0-9_]+)\s*\(", text)))


def check(status: int, model=None):
    if status != OK:
        msg = lib().nnt_last_error(model)
        raise NNTError(status, msg.decode() if msg else "")


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    raise TypeError(f"cannot pass {type(x)} as a pointer")


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


class Model:
    """One GPT2 training step on tiled tensors (nnt_create_model ... nnt_destroy)."""

    def __init__(self, n_layer, d_model, n_head, d_ff, vocab, n_ctx, batch, dtype=BF16,
                 ln_eps=1e-5, tiles=None, seed=0, init_std=0.0, zero_bias=False, stream=None,
                 n_streams=2, use_cuda_graph=False, timeout_ms=0, gemm_backend=0, trace=False,
                 allow_host_offload=False, hbm_budget_bytes=0, gemm_min_task_cols=0,
                 flash_attention=0, host_budget_bytes=0):
        self.cfg = Config(n_layer, d_model, n_head, d_ff, vocab, n_ctx, batch, dtype, ln_eps)
        t = tiles or {}
        self.tiles = Tiles(t.get("batch_tile", 0), t.get("seq_tile", 0), t.get("embd_tile", 0),
                           t.get("inner_tile", 0), t.get("head_tile", 0), t.get("vocab_tile", 0))
        self.opts = Options(_stream(stream), hbm_budget_bytes, int(allow_host_offload), seed,
                            init_std, int(zero_bias), n_streams, int(use_cuda_graph), timeout_ms,
                            gemm_backend, int(trace), gemm_min_task_cols, flash_attention,
                            host_budget_bytes)
        h = C.c_void_p()
        check(lib().nnt_create_model(C.byref(self.cfg), C.byref(self.tiles), C.byref(self.opts),
                                     C.byref(h)))
        self.h = h
        self.names = []
        self.shapes = []
        for i in range(lib().nnt_num_params(h)):
            nm = C.c_char_p()
            sh = (C.c_int64 * 2)()
            check(lib().nnt_param_info(h, i, C.byref(nm), sh), h)
            self.names.append(nm.value.decode())
            self.shapes.append((sh[0],) if sh[1] == 0 else (sh[0], sh[1]))

    def close(self):
        if getattr(self, "h", None):
            lib().nnt_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ---- step
    def forward(self, tokens, want_loss=True):
        """tokens: numpy uint16 [B, S+1] (host) or a torch uint16/int16 CUDA tensor."""
        loss = C.c_float(float("nan"))
        on_dev = 0
        if isinstance(tokens, np.ndarray):
            assert tokens.dtype == np.uint16 and tokens.flags.c_contiguous
            ptr = tokens.ctypes.data
        else:
            on_dev = 1 if tokens.is_cuda else 0
            ptr = tokens.data_ptr()
        check(lib().nnt_forward(self.h, ptr, on_dev, C.byref(loss) if want_loss else None), self.h)
        return loss.value if want_loss else None

    def backward(self, accumulate=False):
        """Gradients of the last forward; accumulate=True adds them to the ones
        summed since the last update (nnt_backward_accumulate)."""
        fn = lib().nnt_backward_accumulate if accumulate else lib().nnt_backward
        check(fn(self.h), self.h)

    def adamw_step(self, lr=3e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1,
                   start_lr=0.0, full_lr_iter=0):
        hp = AdamW(lr, beta1, beta2, eps, weight_decay, start_lr, full_lr_iter)
        check(lib().nnt_adamw_step(self.h, C.byref(hp)), self.h)

    def backward_adamw(self, lr=3e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1,
                       start_lr=0.0, full_lr_iter=0):
        """Backward with each chunk's AdamW update fused in (nnt_backward_adamw)."""
        hp = AdamW(lr, beta1, beta2, eps, weight_decay, start_lr, full_lr_iter)
        check(lib().nnt_backward_adamw(self.h, C.byref(hp)), self.h)

    # ---- parity surface
    def _get(self, fn, i, *extra):
        out = np.empty(self.shapes[i], dtype=np.float32)
        check(fn(self.h, i, *extra, out.ctypes.data), self.h)
        return out

    def get_param(self, i):
        return self._get(lib().nnt_get_param, i)

    def get_grad(self, i):
        return self._get(lib().nnt_get_grad, i)

    def get_adam_state(self, i, which):
        return self._get(lib().nnt_get_adam_state, i, which)

    def set_param(self, i, arr):
        a = np.ascontiguousarray(arr, dtype=np.float32).reshape(self.shapes[i])
        check(lib().nnt_set_param(self.h, i, a.ctypes.data), self.h)

    def set_params(self, params: dict):
        for i, n in enumerate(self.names):
            self.set_param(i, params[n])

    def params(self):
        return {n: self.get_param(i) for i, n in enumerate(self.names)}

    def grads(self):
        return {n: self.get_grad(i) for i, n in enumerate(self.names)}

    def logits(self):
        T = self.cfg.batch * self.cfg.n_ctx
        out = np.empty((T, self.cfg.vocab), dtype=np.float32)
        check(lib().nnt_get_logits(self.h, out.ctypes.data), self.h)
        return out

    def stats(self):
        s = Stats()
        check(lib().nnt_get_stats(self.h, C.byref(s)), self.h)
        return {k: getattr(s, k) for k, _ in Stats._fields_}

    def set_trace(self, on: bool):
        check(lib().nnt_set_trace(self.h, int(on)), self.h)

    def task_times(self):
        n = 64
        names = (C.c_char_p * n)()
        launches = (C.c_int64 * n)()
        ms = (C.c_double * n)()
        fl = (C.c_double * n)()
        by = (C.c_double * n)()
        k = lib().nnt_get_task_times(self.h, n, names, launches, ms, fl, by)
        return {names[i].decode(): {"launches": launches[i], "ms": ms[i], "flops": fl[i],
                                    "bytes": by[i]} for i in range(min(k, n))}


# ---- single tile tasks (device pointers; see include/nnt.h)
def op_layernorm_fwd(x, g, b, y, mean, rstd, rows, cols, eps, dtype, stream=None):
    check(lib().nnt_op_layernorm_fwd(_ptr(x), _ptr(g), _ptr(b), _ptr(y), _ptr(mean), _ptr(rstd),
                                     rows, cols, eps, dtype, _stream(stream)))


def op_layernorm_bwd(dy, x, mean, rstd, g, resid, dx, dx_act, dg, db, rows, cols, dtype, stream=None):
    check(lib().nnt_op_layernorm_bwd(_ptr(dy), _ptr(x), _ptr(mean), _ptr(rstd), _ptr(g), _ptr(resid),
                                     _ptr(dx), _ptr(dx_act), _ptr(dg), _ptr(db), rows, cols, dtype,
                                     _stream(stream)))


def op_softmax_causal_fwd(s, p, nmat, seq, dtype, stream=None):
    check(lib().nnt_op_softmax_causal_fwd(_ptr(s), _ptr(p), nmat, seq, dtype, _stream(stream)))


def op_softmax_causal_bwd(p, dp, ds, nmat, seq, scale, dtype, stream=None):
    check(lib().nnt_op_softmax_causal_bwd(_ptr(p), _ptr(dp), _ptr(ds), nmat, seq, scale, dtype,
                                          _stream(stream)))


def op_flash_attention_fwd(q, k, v, o, lse, Z, S, hd, stream=None):
    """Fused causal attention forward on bf16 [Z][S][hd] buffers (lse fp32 [Z][S])."""
    check(lib().nnt_op_flash_attention_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), Z, S, hd,
                                           _stream(stream)))


def op_flash_attention_bwd(q, k, v, o, do, lse, dq, dk, dv, Z, S, hd, stream=None):
    check(lib().nnt_op_flash_attention_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse),
                                           _ptr(dq), _ptr(dk), _ptr(dv), Z, S, hd, _stream(stream)))


def op_gelu_fwd(u, g, n, dtype, stream=None):
    check(lib().nnt_op_gelu_fwd(_ptr(u), _ptr(g), n, dtype, _stream(stream)))


def op_gelu_bwd(dg, u, du, n, dtype, stream=None):
    check(lib().nnt_op_gelu_bwd(_ptr(dg), _ptr(u), _ptr(du), n, dtype, _stream(stream)))


def op_cross_entropy(z, rows, cols, ldz, tgt, tgt_stride, dz, lddz, row_loss, loss, dtype, stream=None):
    check(lib().nnt_op_cross_entropy(_ptr(z), rows, cols, ldz, _ptr(tgt), tgt_stride, _ptr(dz), lddz,
                                     _ptr(row_loss), _ptr(loss), dtype, _stream(stream)))


def op_adamw(w, g, m, v, w_bf16, n, lr, beta1, beta2, eps, wd, bc1, bc2, stream=None):
    check(lib().nnt_op_adamw(_ptr(w), _ptr(g), _ptr(m), _ptr(v), _ptr(w_bf16), n, lr, beta1, beta2,
                             eps, wd, bc1, bc2, _stream(stream)))


def op_embedding_fwd(ids, ids_stride, wte, wpe, x, batch, seq, d, vocab, stream=None):
    check(lib().nnt_op_embedding_fwd(_ptr(ids), ids_stride, _ptr(wte), _ptr(wpe), _ptr(x), batch, seq,
                                     d, vocab, _stream(stream)))


def op_embedding_bwd(ids, ids_stride, dx, dwte, dwpe, batch, seq, d, vocab, stream=None):
    check(lib().nnt_op_embedding_bwd(_ptr(ids), ids_stride, _ptr(dx), _ptr(dwte), _ptr(dwpe), batch,
                                     seq, d, vocab, _stream(stream)))


def op_embedding_bwd_noalloc(ids, ids_stride, dx, dwte, dwpe, batch, seq, d, vocab, stream=None):
    """nnt_op_embedding_bwd without any device allocation (fixed scratch of 16384 tokens)."""
    check(lib().nnt_op_embedding_bwd_noalloc(_ptr(ids), ids_stride, _ptr(dx), _ptr(dwte), _ptr(dwpe),
                                             batch, seq, d, vocab, _stream(stream)))


def op_gemm(a, lda, a_trans, b, ldb, b_trans, c, ldc, c_dtype, M, N, K, alpha=1.0, beta=0.0,
            dtype=BF16, backend=0, stream=None):
    check(lib().nnt_op_gemm(_ptr(a), lda, a_trans, _ptr(b), ldb, b_trans, _ptr(c), ldc, c_dtype, M,
                            N, K, alpha, beta, dtype, backend, _stream(stream)))


def plan_memory(n_layer, d_model, n_head, d_ff, vocab, n_ctx, batch, dtype=BF16, ln_eps=1e-5,
                tiles=None, allow_host_offload=False, hbm_budget_bytes=0, flash_attention=0):
    """(device bytes, pinned host bytes) nnt_create_model would allocate (nnt_plan_memory)."""
    cfg = Config(n_layer, d_model, n_head, d_ff, vocab, n_ctx, batch, dtype, ln_eps)
    t = tiles or {}
    tl = Tiles(t.get("batch_tile", 0), t.get("seq_tile", 0), t.get("embd_tile", 0),
               t.get("inner_tile", 0), t.get("head_tile", 0), t.get("vocab_tile", 0))
    opts = Options()
    opts.allow_host_offload = int(allow_host_offload)
    opts.hbm_budget_bytes = hbm_budget_bytes
    opts.flash_attention = flash_attention
    dev, host = C.c_uint64(0), C.c_uint64(0)
    check(lib().nnt_plan_memory(C.byref(cfg), C.byref(tl), C.byref(opts), C.byref(dev), C.byref(host)))
    return dev.value, host.value


FAULT_DEVICE_ALLOC, FAULT_HOST_ALLOC, FAULT_COPY, FAULT_EVENT_WAIT = 0, 1, 2, 3


def set_fault_injection(kind: int, nth: int):
    """Make the nth call of ``kind`` from now on fail (host side; 0 disarms)."""
    check(lib().nnt_set_fault_injection(kind, nth))


def op_wait_selftest(limit_ns: int, arrive: bool, stream=None):
    """One bounded mbarrier wait on the device (nnt_op_wait_selftest)."""
    check(lib().nnt_op_wait_selftest(limit_ns, int(arrive), _stream(stream)))


def read_device_error(stream=None) -> int:
    code = C.c_uint32(0)
    check(lib().nnt_op_read_error(C.byref(code), _stream(stream)))
    return code.value


def plan_schedule(uses, n_streams, copy=None, hints=None):
    """The executor's plan for tasks given by their tile accesses (host only).

    ``uses[i]`` lists task i's ``(tile, mode)`` pairs (mode 1 read, 2 write,
    3 both); ``copy`` and ``hints`` are optional per-task lists (copy-stream
    task; pinned compute stream or -1). Returns ``(streams, deps, waits)``:
    each task's stream, its direct dependencies and its cross-stream waits."""
    n = len(uses)
    off = np.zeros(n + 1, np.int64)
    off[1:] = np.cumsum([len(u) for u in uses])
    tiles = np.array([t for u in uses for t, _ in u], np.int64)
    modes = np.array([m for u in uses for _, m in u], np.int32)
    cp = None if copy is None else np.ascontiguousarray(copy, np.int32)
    hi = None if hints is None else np.ascontiguousarray(hints, np.int32)
    streams = np.zeros(n, np.int32)
    dep_off = np.zeros(n + 1, np.int64)
    wait_off = np.zeros(n + 1, np.int64)
    cap_d = cap_w = 0
    dep = wait = np.zeros(0, np.int32)
    for _ in range(2):  # the first call sizes the outputs
        st = lib().nnt_plan_schedule(n, _ptr(off), _ptr(tiles) if tiles.size else None,
                                     _ptr(modes) if modes.size else None, _ptr(cp), _ptr(hi),
                                     n_streams, _ptr(streams), _ptr(dep_off),
                                     _ptr(dep) if dep.size else None, cap_d, _ptr(wait_off),
                                     _ptr(wait) if wait.size else None, cap_w)
        if st == OK:
            break
        if dep_off[n] <= cap_d and wait_off[n] <= cap_w:
            check(st)
        cap_d, cap_w = int(dep_off[n]), int(wait_off[n])
        dep = np.zeros(max(cap_d, 1), np.int32)
        wait = np.zeros(max(cap_w, 1), np.int32)
    else:
        check(st)
    deps = [dep[dep_off[i]:dep_off[i + 1]].tolist() for i in range(n)]
    waits = [wait[wait_off[i]:wait_off[i + 1]].tolist() for i in range(n)]
    return streams.tolist(), deps, waits
