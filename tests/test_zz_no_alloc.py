"""The allocation-free embedding scatter-add against the regular one (GPU).

nnt_op_embedding_bwd_noalloc serves callers that cannot allocate device memory
while they run: hosts that own all device memory through their own allocator
or a fixed budget, and loops that cannot afford an allocation's implicit
device synchronisation. It must give the same bits as nnt_op_embedding_bwd,
call after call, although every call reuses the same fixed scratch array, and
it must leave the device's free memory unchanged.

The file is collected last (``zz``) so that a run stopping at the first
failure has run every other test first; the tests themselves need no state
from earlier tests and also pass alone in a fresh process.
"""
import numpy as np
import pytest

from tile_task_transformer_gb300 import nnt, synth

pytestmark = pytest.mark.gpu


def _case(seed, B, S, d, V):
    ids = (synth.bits(seed, 1, 0, B * (S + 1)) % np.uint64(V)).astype(np.uint16).reshape(B, S + 1)
    dx = synth.normal_matrix(seed, 2, (B, S, d), 1.0)
    w0 = synth.normal_matrix(seed, 3, (V, d), 1.0)
    p0 = synth.normal_matrix(seed, 4, (S, d), 1.0)
    return ids, dx, w0, p0


def _torch():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch


def test_noalloc_allocates_nothing():
    """Free device memory is the same before and after calls (the fixed
    scratch is part of the library's image). One call first: with lazy module
    loading, the kernels' code is loaded onto the device at their first launch."""
    torch = _torch()
    B, S, d, V = 2, 512, 64, 1000
    ids, dx, w0, p0 = _case(20, B, S, d, V)
    idt = torch.as_tensor(ids.view(np.int16)).cuda()
    dxt, wt, pt = torch.as_tensor(dx).cuda(), torch.as_tensor(w0).cuda(), torch.as_tensor(p0).cuda()
    nnt.op_embedding_bwd_noalloc(idt, S + 1, dxt, wt, pt, B, S, d, V)
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(2):
        nnt.op_embedding_bwd_noalloc(idt, S + 1, dxt, wt, pt, B, S, d, V)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0


def test_noalloc_matches_regular_call_twice():
    torch = _torch()
    for seed, (B, S, d, V) in [(21, (4, 1024, 768, 50257)), (22, (16, 1024, 64, 1000))]:
        ids, dx, w0, p0 = _case(seed, B, S, d, V)
        idt = torch.as_tensor(ids.view(np.int16)).cuda()
        dxt = torch.as_tensor(dx).cuda()
        ref_w, ref_p = torch.as_tensor(w0).cuda(), torch.as_tensor(p0).cuda()
        got_w, got_p = ref_w.clone(), ref_p.clone()
        nnt.op_embedding_bwd(idt, S + 1, dxt, ref_w, ref_p, B, S, d, V)
        nnt.op_embedding_bwd_noalloc(idt, S + 1, dxt, got_w, got_p, B, S, d, V)
        torch.cuda.synchronize()
        assert torch.equal(got_w, ref_w)
        assert torch.equal(got_p, ref_p)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    torch = _torch()
    B, S, d, V = 17, 1024, 8, 100  # 17408 tokens > 16384
    x = torch.zeros(8, device="cuda")
    with pytest.raises(nnt.NNTError) as e:
        nnt.op_embedding_bwd_noalloc(x, S + 1, x, x, x, B, S, d, V)
    assert e.value.status == nnt.ERR_INVALID_ARG
