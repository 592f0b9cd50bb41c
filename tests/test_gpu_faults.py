"""Failure detection without a GPU fault (GPU).

Failures are injected on the host (nnt_set_fault_injection): an allocation
that fails, an async copy that cannot be submitted, a host wait that runs out.
Each must surface as its error code and leave the library usable: a model
whose creation failed is fully released, and a model whose call failed still
steps correctly afterwards. On the device, a bounded mbarrier wait that
nothing completes must give up after its limit, record the wait-timeout bit
in the error word and return, with the context still usable.
"""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

from oracle import gpt2 as O  # noqa: E402
from tile_task_transformer_gb300 import nnt, synth  # noqa: E402

pytestmark = pytest.mark.gpu

TINY = O.GPT2Config(n_layer=2, d_model=64, n_head=4, d_ff=256, vocab=256, seq=32, batch=2)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    nnt.lib()


@pytest.fixture(autouse=True)
def _disarm():
    yield
    for k in range(4):
        nnt.set_fault_injection(k, 0)


def make(**kw):
    c = TINY
    return nnt.Model(c.n_layer, c.d_model, c.n_head, c.d_ff, c.vocab, c.seq, c.batch, dtype=nnt.F32,
                     tiles={"seq_tile": 16, "embd_tile": 32}, seed=5, init_std=0.02, **kw)


WIN = synth.token_windows(5, TINY.batch, TINY.seq, TINY.vocab)


def reference_loss():
    m = make()
    loss = m.forward(WIN)
    m.close()
    return loss


@pytest.mark.parametrize("nth", [1, 3, 7])
def test_device_allocation_failure_is_oom_and_releases_everything(nth):
    ref = reference_loss()
    torch.cuda.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    nnt.set_fault_injection(nnt.FAULT_DEVICE_ALLOC, nth)
    with pytest.raises(nnt.NNTError) as e:
        make()
    assert e.value.status == nnt.ERR_OOM
    assert "injected" in str(e.value)
    torch.cuda.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0  # every earlier allocation was freed
    nnt.set_fault_injection(nnt.FAULT_DEVICE_ALLOC, 0)
    assert make().forward(WIN) == ref


def test_pinned_host_allocation_failure_is_oom():
    nnt.set_fault_injection(nnt.FAULT_HOST_ALLOC, 1)
    with pytest.raises(nnt.NNTError) as e:
        make()
    assert e.value.status == nnt.ERR_OOM


def test_offloaded_moments_allocation_failure_is_oom():
    # a device budget this small puts the AdamW moments in pinned host memory:
    # the loss word is pinned allocation 1, the two moment pools 2 and 3
    nnt.set_fault_injection(nnt.FAULT_HOST_ALLOC, 3)
    with pytest.raises(nnt.NNTError) as e:
        make(allow_host_offload=True, hbm_budget_bytes=1)
    assert e.value.status == nnt.ERR_OOM


def test_copy_submission_failure_leaves_model_usable():
    ref = reference_loss()
    m = make()
    nnt.set_fault_injection(nnt.FAULT_COPY, 1)  # the token upload of the next forward
    with pytest.raises(nnt.NNTError) as e:
        m.forward(WIN)
    assert e.value.status == nnt.ERR_CUDA
    assert m.forward(WIN) == ref
    nnt.set_fault_injection(nnt.FAULT_COPY, 2)  # the loss read-back
    with pytest.raises(nnt.NNTError) as e:
        m.forward(WIN)
    assert e.value.status == nnt.ERR_CUDA
    with pytest.raises(nnt.NNTError) as e:  # the forward did not complete: no backward
        m.backward()
    assert e.value.status == nnt.ERR_STATE
    assert m.forward(WIN) == ref
    m.backward()
    m.close()


def test_host_wait_timeout_then_recovery():
    ref = reference_loss()
    m = make()
    nnt.set_fault_injection(nnt.FAULT_EVENT_WAIT, 1)
    with pytest.raises(nnt.NNTError) as e:
        m.forward(WIN)
    assert e.value.status == nnt.ERR_TIMEOUT
    assert m.forward(WIN) == ref
    m.backward()
    m.adamw_step()
    m.close()


def test_bounded_device_wait_gives_up_and_reports():
    nnt.read_device_error()
    nnt.op_wait_selftest(1_000_000, arrive=False)  # nothing completes the phase: 1 ms, then give up
    assert nnt.read_device_error() == 2
    nnt.op_wait_selftest(1_000_000, arrive=True)  # completed before the wait: no error
    assert nnt.read_device_error() == 0
    # the context is still usable: a tensor-core GEMM right after
    a = torch.randn(256, 128, device="cuda").to(torch.bfloat16)
    b = torch.randn(192, 128, device="cuda").to(torch.bfloat16)
    c = torch.empty(256, 192, device="cuda")
    nnt.op_gemm(a, 128, 0, b, 128, 0, c, 192, nnt.F32, 256, 192, 128, dtype=nnt.BF16, backend=0)
    torch.cuda.synchronize()
    ref = a.double() @ b.double().T
    assert ((c.double() - ref).abs().max() / ref.abs().max()).item() < 1e-5
    assert nnt.read_device_error() == 0
