"""The bench's bookkeeping on the CPU: max over ranks through a
world-size-2 gloo process group, the whole-job rate, and the reference arm
running on rank 0 alone. (On GPUs the same helpers run over NCCL, one rank per
GPU; every rank is an independent replica, so there is no data-path
collective.)"""
import argparse
import multiprocessing as mp
import os
import socket

import pytest

import bench

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(1.5 + rank, world, "cpu")
        q.put((rank, slowest, bench.job_rate(world, 4096, slowest)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_with_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert [p.exitcode for p in procs] == [0, 0]
    # both ranks see the slower rank's time and the same whole-job rate
    assert got == [(0, 2.5, 2 * 4096 / 2.5), (1, 2.5, 2 * 4096 / 2.5)]


def test_one_rank_is_its_own_max():
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25
    assert bench.job_rate(1, 4096, 0.5) == 8192.0


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    args = argparse.Namespace(workload="tiny", warmup=3, steps=2, gpus=2)
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""


@pytest.mark.parametrize("L,d,H,f,V,S,B", [(12, 768, 12, 3072, 50257, 1024, 4),
                                           (4, 8192, 64, 32768, 50257, 1024, 8),
                                           (2, 64, 4, 256, 256, 32, 2)])
def test_model_flops_agree_with_the_pinned_oracle_count(L, d, H, f, V, S, B):
    from oracle import gpt2 as O

    cfg = O.GPT2Config(n_layer=L, d_model=d, n_head=H, d_ff=f, vocab=V, seq=S, batch=B)
    assert bench.model_step_flops(L, d, H, f, V, S, B) == O.step_flops(cfg)
