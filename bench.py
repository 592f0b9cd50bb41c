"""Benchmark: GPT2 training step (forward + backward + fused AdamW) tokens/s on one GB300.

Default workload: the GPT2-small-shaped configuration of the NNTile README's
GPT example ("Minimal working GPT example": 12 layers, d_model 768, 12 heads,
d_ff 3072, vocab 50257, sequence 1024, minibatch 4; tiles seq 1024, embd 768,
inner 3072, head 12), bf16 GEMM operands with fp32 master weights and AdamW
states, synthetic uniform token ids and N(0, 0.02) weights.

Prints one JSON line. ``value``: tokens/s over K timed steps with the tokens
already on the device (CUDA events on the model's stream); ``e2e``: the same
through the C ABI with the token windows copied in from pinned host memory and
the loss read back every step. ``roofline``: the dominant kernel's achieved
rate against MEASURED_PEAKS.json. ``cpu_baseline``: the CPU oracle on a
bounded sample (one sequence) on the host cores.

``--impl reference`` times the CPU oracle alone (the reference arm).
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GPT2 train tokens/s on 1 GB300; tile-kernel % of HBM/TC roofline"

WORKLOADS = {
    # name: (n_layer, d_model, n_head, d_ff, vocab, seq, batch, dtype, tiles)
    "gpt2-small": (12, 768, 12, 3072, 50257, 1024, 4, "bf16",
                   {"seq_tile": 1024, "embd_tile": 768, "inner_tile": 3072, "head_tile": 12,
                    "batch_tile": 4}),
    "tiny": (2, 64, 4, 256, 256, 32, 2, "fp32", {"seq_tile": 16, "embd_tile": 32}),
    "wide-4": (4, 8192, 64, 32768, 50257, 1024, 8, "bf16",
               {"seq_tile": 1024, "embd_tile": 2048, "inner_tile": 4096, "head_tile": 16}),
    # 26.6B parameters: AdamW moments partly in pinned host memory, fused backward + AdamW
    "wide-8": (8, 16384, 128, 65536, 50257, 1024, 4, "bf16",
               {"seq_tile": 1024, "embd_tile": 2048, "inner_tile": 4096, "head_tile": 16}),
}

GEMM_TYPES = {"gemm_qkv", "gemm_qk", "gemm_pv", "gemm_attn_out", "gemm_fc_gelu", "gemm_mlp_proj",
              "gemm_lm_head", "gemm_lm_dx", "gemm_lm_dw", "gemm_dx", "gemm_dw", "gemm_attn_bwd"}
KERNEL_OF_TYPE = {t: "gemm_tc_kernel" for t in GEMM_TYPES}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def gemm_traffic(workload):
    """DRAM bytes (read + write) per GEMM launch from the committed ncu summary,
    or None when that summary was taken on another workload or on a different
    version of the kernel source."""
    import hashlib
    p = os.path.join(ROOT, "profiles", f"gemm_tc_traffic_{workload.replace('-', '_')}.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        d = json.load(fh)
    csrc = os.path.join(ROOT, "tile_task_transformer_gb300", "csrc")
    h = hashlib.sha256()
    for f in ("gemm_tc.cu", "gemm.cuh", "tc_ptx.cuh"):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return d["bytes_per_launch"] if h.hexdigest() == d.get("source_sha256") else None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self):
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], 0.0, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = max(mx, float(f[2]))
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        sm.sort()
        return {"sm_mhz": sm[len(sm) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def model_step_flops(L, d, H, f, V, S, B):
    """Model FLOPs of one training step: three times the forward products (the
    backward does two per forward product). Per layer the four weight products
    (QKV, output projection, FC, MLP projection), the tied LM head once, and the
    attention products QK^T and P V over causal pairs only; elementwise work is
    not counted."""
    T = B * S
    dense = 2.0 * T * (L * (4 * d * d + 2 * d * f) + d * V)
    attn = L * B * H * 2 * (2.0 * (d // H) * S * (S + 1) / 2)
    return 3.0 * (dense + attn)


def max_over_ranks(x, world, device):
    """The largest of the ranks' values of x, on every rank (x itself for one
    rank): the job is as slow as its slowest replica."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.item()


def job_rate(world, tokens_per_rank, seconds):
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank / seconds


def oracle_sample(name, seed, batch=1):
    """CPU oracle step on `batch` sequences of the workload; returns (tokens, seconds, cores)."""
    import numpy as np

    from oracle import gpt2 as O
    from tile_task_transformer_gb300 import synth

    L, d, H, f, V, S, _, _, _ = WORKLOADS[name]
    cfg = O.GPT2Config(n_layer=L, d_model=d, n_head=H, d_ff=f, vocab=V, seq=S, batch=batch)
    params = synth.gpt2_params(seed, L, d, f, V, S)
    win = synth.token_windows(seed, batch, S, V)
    t0 = time.perf_counter()
    loss, grads, new_p, _, _ = O.train_step(cfg, params, win)
    dt = time.perf_counter() - t0
    assert np.isfinite(loss)
    return batch * S, dt, os.cpu_count()


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    name = args.workload
    _, _, _, _, _, S, B, dtype, _ = WORKLOADS[name]
    for _ in range(args.warmup):
        oracle_sample(name, 1)
    tot_tok, tot_t, cores = 0, 0.0, os.cpu_count()
    for _ in range(args.steps):
        tok, dt, cores = oracle_sample(name, 1)
        tot_tok += tok
        tot_t += dt
    v = tot_tok / tot_t
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000 * tot_t / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{name} (oracle sample: 1 sequence of {S} tokens per step)",
                   "global_batch": 1, "seq_len": S, "parallelism": "none (CPU oracle)"},
        "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": f"one {name} training step on 1 sequence x {S} tokens, fp64 numpy"},
        "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


def run_gpu(args):
    import numpy as np
    import torch

    from tile_task_transformer_gb300 import nnt, synth

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    name = args.workload
    L, d, H, f, V, S, B, dtype, tiles = WORKLOADS[name]
    if args.tiles:
        tiles = {**tiles, **json.loads(args.tiles)}
    dt = nnt.BF16 if dtype == "bf16" else nnt.F32
    stream = torch.cuda.Stream()
    link = None
    if nnt.plan_memory(L, d, H, f, V, S, B, dtype=dt, tiles=tiles, allow_host_offload=True)[1]:
        # moments in pinned host memory: the host link bounds their AdamW tasks
        link = host_link_peaks(torch)
    t_create = time.perf_counter()
    model = nnt.Model(L, d, H, f, V, S, B, dtype=dt, tiles=tiles, seed=1 + rank, stream=stream,
                      n_streams=args.streams, use_cuda_graph=not args.no_graph,
                      allow_host_offload=True)
    t_create = time.perf_counter() - t_create
    st = model.stats()
    fused = not args.separate or st["offload_active"] == 1
    T = B * S
    win_host = synth.token_windows(1 + rank, B, S, V)
    tok_dev = torch.as_tensor(win_host.view(np.int16)).to("cuda")
    tok_pin = torch.as_tensor(win_host.view(np.int16)).pin_memory()
    hp = dict(lr=3e-4, eps=1e-8, weight_decay=0.1)

    def step(tokens, want_loss):
        loss = model.forward(tokens, want_loss=want_loss)
        if fused:
            model.backward_adamw(**hp)
        else:
            model.backward()
            model.adamw_step(**hp)
        return loss

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    # warm-up (also captures the CUDA graphs)
    for _ in range(max(args.warmup, 1)):
        step(tok_dev, False)
    torch.cuda.synchronize()

    # ---- device-timed region: tokens resident in HBM
    clocks = ClockSampler()
    clocks.start()
    barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step(tok_dev, False)
    e1.record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop()
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world, "cuda")
    value = job_rate(world, T, ms / 1000.0)

    # ---- end to end through the C ABI: pinned host tokens in, loss out, every step
    torch.cuda.synchronize()
    barrier()
    t0 = time.perf_counter()
    losses = []
    for _ in range(args.steps):
        losses.append(step(tok_pin, True))
    torch.cuda.synchronize()
    barrier()
    e2e_s = max_over_ranks((time.perf_counter() - t0) / args.steps, world, "cuda")
    e2e_value = job_rate(world, T, e2e_s)
    assert all(np.isfinite(losses)), losses

    # ---- per-task timing pass (CUDA events on each task's stream) for the roofline
    model.set_trace(True)
    for _ in range(2):
        step(tok_dev, True)
    times = model.task_times()
    model.set_trace(False)
    pk, pk_kind = peaks()
    by_kernel = {}
    for tname, rec in times.items():
        if rec["launches"] == 0:
            continue
        k = KERNEL_OF_TYPE.get(tname, tname)
        agg = by_kernel.setdefault(k, {"ms": 0.0, "launches": 0, "flops": 0.0, "bytes": 0.0})
        agg["ms"] += rec["ms"]
        agg["launches"] += rec["launches"]
        agg["flops"] += rec["flops"]
        agg["bytes"] += rec["bytes"]
    total_ms = sum(a["ms"] for a in by_kernel.values())
    dom = max(by_kernel, key=lambda k: by_kernel[k]["ms"])
    a = by_kernel[dom]
    if dom == "adamw_host_moments" and link:
        # m and v of the host-resident chunks cross the host link both ways
        # (8 B each way per parameter); peak: pinned copies, both ways at once
        st_now = model.stats()
        link_bytes = (st_now["h2d_bytes"] + st_now["d2h_bytes"]) - (st["h2d_bytes"] + st["d2h_bytes"])
        steps_run = max(args.warmup, 1) + 2 * args.steps + 2
        achieved = link_bytes / steps_run / (a["ms"] / 2 / 1e3) / 1e9
        roof = {"bound": "host_link", "achieved": achieved, "peak": link["both_gbs"],
                "unit": "GB/s", "frac": achieved / link["both_gbs"], "traffic": None,
                "kernel": dom, "peak_kind": "measured in this run: pinned cudaMemcpyAsync, "
                "1 GiB each way at once", "host_link_gbs": link}
    elif a["flops"] > 0:
        achieved = a["flops"] / (a["ms"] / 1e3) / 1e12
        peak = pk.get("bf16_tflops_sustained", pk["bf16_tflops"])
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "traffic": gemm_traffic(name), "kernel": dom,
                "peak_kind": f"{pk_kind} sustained bf16",
                "launches_per_step": a["launches"] // 2}
    else:
        achieved = a["bytes"] / (a["ms"] / 1e3) / 1e9
        peak = pk["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": None, "kernel": dom,
                "peak_kind": f"{pk_kind} copy"}
    kernel_table = {k: {"share": v["ms"] / total_ms, "launches": v["launches"],
                        "ms_per_step": v["ms"] / 2,
                        **({"tflops": v["flops"] / (v["ms"] / 1e3) / 1e12} if v["flops"] else {}),
                        **({"gbs": v["bytes"] / (v["ms"] / 1e3) / 1e9} if v["bytes"] and not v["flops"] else {})}
                    for k, v in sorted(by_kernel.items(), key=lambda kv: -kv[1]["ms"])}

    # ---- CPU oracle baseline (rank 0, N = 1 only): one sequence of the workload
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        tok, sec, cores = oracle_sample(name, 1 + rank)
        cpu = {"value": tok / sec, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"one {name} training step on 1 sequence x {S} tokens (fp64 numpy, "
                         f"{sec:.1f} s; the GPU step above runs {B} sequences, both rates are per token)"}

    type_table = {k: {"ms_per_step": v["ms"] / 2, "launches_per_step": v["launches"] // 2,
                      **({"tflops": v["flops"] / (v["ms"] / 1e3) / 1e12} if v["flops"] else {}),
                      **({"gbs": v["bytes"] / (v["ms"] / 1e3) / 1e9} if v["bytes"] else {})}
                  for k, v in sorted(times.items(), key=lambda kv: -kv[1]["ms"]) if v["launches"]}
    n_kernels = st["kernels_forward"] + st["kernels_backward"] + st["kernels_adamw"]
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if dt == nnt.BF16 else "f32", "data": "synthetic",
        "config": {"workload": f"{name}: L{L} d{d} H{H} ff{f} V{V} S{S} B{B}, tiles {tiles}",
                   "global_batch": B * world, "seq_len": S,
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": "working set >> L2 (activations and weights are several GB per step)",
                   "cuda_graph": not args.no_graph, "streams": args.streams,
                   "fused_backward_adamw": fused,
                   "host_offload": {"active": bool(st["offload_active"]),
                                    "pinned_gib": st["host_pinned_bytes"] / 2 ** 30,
                                    "h2d_gib_per_step": None, "d2h_gib_per_step": None}},
        "clocks": clk,
        "e2e": {"value": e2e_value, "unit": "tokens/s",
                "h2d_bytes_per_step": int(win_host.nbytes), "d2h_bytes_per_step": 4},
        "gpu_launches": int(n_kernels * args.steps),
        "roofline": roof,
        "kernels": kernel_table,
        "task_types": type_table,
        "model_tflops": None,
        "loss": float(losses[-1]),
        "device_gib": st["device_bytes"] / 2 ** 30,
        "create_s": t_create,
    }
    if st["offload_active"]:
        st2 = model.stats()
        nsteps = max(args.warmup, 1) + 2 * args.steps + 2
        line["config"]["host_offload"]["h2d_gib_per_step"] = st2["h2d_bytes"] / nsteps / 2 ** 30
        line["config"]["host_offload"]["d2h_gib_per_step"] = st2["d2h_bytes"] / nsteps / 2 ** 30
    line["model_tflops"] = world * model_step_flops(L, d, H, f, V, S, B) / (ms / 1e3) / 1e12
    if cpu:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line))
    model.close()
    return 0


# --------------------------------------------------------------------------
# capacity sweep: the largest wide GPT2 that completes a step on one GPU
# --------------------------------------------------------------------------

# (layers, d_model) at the 8-layer, 26.6B-parameter wide-8 scale and deeper;
# d_ff = 4 d, 128-wide heads, 4 x 1024 tokens, tiles as wide-8
CAPACITY_POINTS = ((8, 16384), (9, 16384), (12, 14336), (16, 12288), (11, 15360), (13, 14336),
                   (10, 16384))


def host_available():
    with open("/proc/meminfo") as fh:
        for line in fh:
            if line.startswith("MemAvailable:"):
                return int(line.split()[1]) * 1024
    return 0


def host_link_peaks(torch):
    """Pinned cudaMemcpyAsync throughput of the host link, 1 GiB per copy, best
    of 5 by CUDA events: host to device, device to host, and both at once (one
    copy each way on two streams; bytes of both over the time of the pair)."""
    n = 1 << 28
    h_in = torch.empty(n, dtype=torch.float32, pin_memory=True)
    h_out = torch.empty(n, dtype=torch.float32, pin_memory=True)
    d_in = torch.empty(n, dtype=torch.float32, device="cuda")
    d_out = torch.empty(n, dtype=torch.float32, device="cuda")
    s_up, s_down = torch.cuda.Stream(), torch.cuda.Stream()
    link = {}
    for name, pairs in (("h2d_gbs", ((d_in, h_in, s_up),)), ("d2h_gbs", ((h_out, d_out, s_down),)),
                        ("both_gbs", ((d_in, h_in, s_up), (h_out, d_out, s_down)))):
        best = 1e9
        for _ in range(5):
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _, _, st in pairs:
                st.wait_event(e0)
            for dst, src, st in pairs:
                with torch.cuda.stream(st):
                    dst.copy_(src, non_blocking=True)
            for _, _, st in pairs:
                torch.cuda.current_stream().wait_stream(st)
            e1.record()
            torch.cuda.synchronize()
            best = min(best, e0.elapsed_time(e1))
        link[name] = len(pairs) * n * 4 / (best / 1e3) / 1e9
    del h_in, h_out, d_in, d_out
    torch.cuda.empty_cache()
    return link


def run_capacity(args):
    """Each point's device and pinned-host footprint comes from the library's
    allocation plan first; only points inside both budgets are created and
    stepped (forward + backward with the fused AdamW). Also measures the
    pinned cudaMemcpyAsync peaks of the host link."""
    import numpy as np
    import torch

    from tile_task_transformer_gb300 import nnt, synth

    gib = 1 << 30
    link = host_link_peaks(torch)
    print(json.dumps({"capacity": "host_link", "pinned_copy_1gib": link}), flush=True)
    points = CAPACITY_POINTS
    if args.capacity_points:
        points = [tuple(int(v) for v in p.split("x")) for p in args.capacity_points.split(",")]
    for L, d in points:
        H, f, V, S, B = d // 128, 4 * d, 50257, 1024, 4
        ht = 16 if H % 16 == 0 else 8
        tiles = {"seq_tile": 1024, "embd_tile": 2048, "inner_tile": 4096, "head_tile": ht}
        n = sum(int(np.prod(sh)) for _, sh in synth.param_names_shapes(L, d, f, V, S))
        free, _ = torch.cuda.mem_get_info()
        dev_budget = free - 2 * gib
        host_budget = max(host_available() - 16 * gib, 0)
        dev, host = nnt.plan_memory(L, d, H, f, V, S, B, tiles=tiles, allow_host_offload=True,
                                    hbm_budget_bytes=dev_budget)
        line = {"capacity": f"L{L} d{d} H{H} ff{f} V{V} S{S} B{B}", "params": n,
                "plan_device_gib": dev / gib, "plan_host_gib": host / gib,
                "device_budget_gib": dev_budget / gib, "host_budget_gib": host_budget / gib,
                "admitted": bool(dev <= dev_budget and host <= host_budget)}
        if line["admitted"]:
            t0 = time.perf_counter()
            m = nnt.Model(L, d, H, f, V, S, B, dtype=nnt.BF16, tiles=tiles, seed=3, use_cuda_graph=True,
                          n_streams=2, allow_host_offload=True, hbm_budget_bytes=dev_budget,
                          host_budget_bytes=host_budget)
            line["create_s"] = time.perf_counter() - t0
            win = synth.token_windows(3, B, S, V)
            stream = torch.cuda.current_stream()
            times, losses = [], []
            for _ in range(2):  # the first step also captures the graphs
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                losses.append(m.forward(win))
                m.backward_adamw()
                e1.record(stream)
                torch.cuda.synchronize()
                times.append(e0.elapsed_time(e1) / 1e3)
            st = m.stats()
            line.update(completed=bool(np.isfinite(losses).all()), loss=losses, step_s=times[-1],
                        tokens_per_s=B * S / times[-1], device_gib=st["device_bytes"] / gib,
                        pinned_gib=st["host_pinned_bytes"] / gib)
            m.close()
        print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------
# tile-kernel sweep: the step's tile kernels alone on synthetic tiles
# --------------------------------------------------------------------------

SWEEP_ROWS = (256, 1024, 4096, 8192)
SWEEP_COLS = (768, 3072, 16384, 65536)
SWEEP_GEMM = (1024, 2048, 4096, 8192)


def run_sweep(args):
    """One JSON line per (kernel, shape): time per call (CUDA events, median of
    `--steps` calls after `--warmup`), algorithmic bytes or flops, and the
    fraction of the measured HBM copy / dense bf16 peak. Inputs N(0, 1), logits
    N(0, 3). Memory-bound inputs are at least 256 MiB where the shape allows,
    else the buffers are cycled to exceed L2."""
    import numpy as np
    import torch

    from tile_task_transformer_gb300 import nnt

    pk, pk_kind = peaks()
    torch.manual_seed(4)
    dev = "cuda"
    kernels = args.sweep_kernel.split(",") if args.sweep_kernel else [
        "layernorm_fwd", "layernorm_bwd", "softmax_fwd", "softmax_bwd", "gelu_fwd", "gelu_bwd",
        "cross_entropy", "adamw", "gemm", "flash_attention"]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def timeit(fn):
        for _ in range(args.warmup):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(args.steps):
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return float(np.median(ts))

    def emit(kernel, shape, dtype, ms, nbytes=None, flops=None):
        line = {"sweep": kernel, "shape": shape, "dtype": dtype, "ms": ms}
        if flops:
            tf = flops / (ms / 1e3) / 1e12
            line.update(tflops=tf, frac=tf / pk["bf16_tflops"], peak=f"{pk_kind} burst bf16")
        else:
            gbs = nbytes / (ms / 1e3) / 1e9
            line.update(gbs=gbs, frac=gbs / pk["hbm_gbs"], peak=f"{pk_kind} HBM copy")
        print(json.dumps(line), flush=True)

    rows_list = [int(x) for x in args.sweep_rows.split(",")] if args.sweep_rows else SWEEP_ROWS
    cols_list = [int(x) for x in args.sweep_cols.split(",")] if args.sweep_cols else SWEEP_COLS
    for dt_name, dt, tdt, es in (("f32", nnt.F32, torch.float32, 4), ("bf16", nnt.BF16, torch.bfloat16, 2)):
        if args.sweep_dtype and dt_name != args.sweep_dtype:
            continue
        for R in rows_list:
            for Cc in cols_list:
                if "layernorm_fwd" in kernels or "layernorm_bwd" in kernels:
                    if Cc <= 32768:
                        x = torch.randn(R, Cc, device=dev)
                        g = torch.randn(Cc, device=dev)
                        b = torch.randn(Cc, device=dev)
                        y = torch.empty(R, Cc, device=dev, dtype=tdt)
                        mu = torch.empty(R, device=dev)
                        rs = torch.empty(R, device=dev)
                        if "layernorm_fwd" in kernels:
                            ms = timeit(lambda: nnt.op_layernorm_fwd(x, g, b, y, mu, rs, R, Cc, 1e-5, dt))
                            emit("layernorm_fwd", [R, Cc], dt_name, ms, nbytes=R * Cc * (4 + es) + 8 * R)
                        if "layernorm_bwd" in kernels:
                            dy = torch.randn(R, Cc, device=dev)
                            dx = torch.empty(R, Cc, device=dev)
                            dxa = torch.empty(R, Cc, device=dev, dtype=tdt)
                            dg = torch.empty(Cc, device=dev)
                            db = torch.empty(Cc, device=dev)
                            ms = timeit(lambda: nnt.op_layernorm_bwd(dy, x, mu, rs, g, None, dx, dxa, dg, db,
                                                                     R, Cc, dt))
                            # algorithmic: read dy, x; write dx and its activation-dtype copy (rows
                            # over 1024 columns read dy, x a second time for the column sums)
                            emit("layernorm_bwd", [R, Cc], dt_name, ms, nbytes=R * Cc * (8 + 4 + es))
                        del x, y
                if ("gelu_fwd" in kernels or "gelu_bwd" in kernels):
                    n = R * Cc
                    u = torch.randn(n, device=dev)
                    gg = torch.empty(n, device=dev, dtype=tdt)
                    if "gelu_fwd" in kernels:
                        ms = timeit(lambda: nnt.op_gelu_fwd(u, gg, n, dt))
                        emit("gelu_fwd", [R, Cc], dt_name, ms, nbytes=n * (4 + es))
                    if "gelu_bwd" in kernels:
                        du = torch.empty(n, device=dev, dtype=tdt)
                        ms = timeit(lambda: nnt.op_gelu_bwd(gg, u, du, n, dt))
                        emit("gelu_bwd", [R, Cc], dt_name, ms, nbytes=n * (es + 4 + es))
                        del du
                    del u, gg
                if "cross_entropy" in kernels and Cc >= 3072:
                    ldz = (Cc + 3) // 4 * 4
                    lddz = (Cc + 7) // 8 * 8
                    z = torch.randn(R, ldz, device=dev) * 3
                    tg = torch.randint(0, Cc, (R,), device=dev, dtype=torch.int32).to(torch.int16)  # uint16 bits
                    dz = torch.empty(R, lddz, device=dev, dtype=tdt)
                    rl = torch.empty(R, device=dev)
                    loss = torch.empty(1, device=dev)
                    ms = timeit(lambda: nnt.op_cross_entropy(z, R, Cc, ldz, tg, 1, dz, lddz, rl, loss, dt))
                    emit("cross_entropy", [R, Cc], dt_name, ms, nbytes=R * Cc * (4 + es) + 2 * R)
                    del z, dz
        # causal softmax on [nmat, S, S] score tiles
        for S in (1024, 2048, 4096):
            if not ("softmax_fwd" in kernels or "softmax_bwd" in kernels):
                break
            nmat = max(1, (512 << 20) // (S * S * 4))
            s_ = torch.randn(nmat, S, S, device=dev)
            p_ = torch.empty(nmat, S, S, device=dev, dtype=tdt)
            causal = nmat * S * (S + 1) / 2
            if "softmax_fwd" in kernels:
                ms = timeit(lambda: nnt.op_softmax_causal_fwd(s_, p_, nmat, S, dt))
                emit("softmax_fwd", [nmat, S, S], dt_name, ms, nbytes=causal * (4 + es))
            if "softmax_bwd" in kernels:
                nnt.op_softmax_causal_fwd(s_, p_, nmat, S, dt)
                ds = torch.empty_like(p_)
                ms = timeit(lambda: nnt.op_softmax_causal_bwd(p_, s_, ds, nmat, S, 0.125, dt))
                emit("softmax_bwd", [nmat, S, S], dt_name, ms, nbytes=causal * (es + 4 + es))
                del ds
            del s_, p_
    if "adamw" in kernels:
        for n in (1 << 24, 1 << 26, 1 << 28):
            w, g_, m_, v_ = (torch.randn(n, device=dev) for _ in range(4))
            v_.abs_()
            wb = torch.empty(n, device=dev, dtype=torch.bfloat16)
            ms = timeit(lambda: nnt.op_adamw(w, g_, m_, v_, wb, n, 3e-4, 0.9, 0.999, 1e-8, 0.1, 0.1, 0.001))
            emit("adamw", [n], "f32", ms, nbytes=30 * n)
            del w, g_, m_, v_, wb
    if "gemm" in kernels:
        sizes = [int(x) for x in args.sweep_gemm.split(",")] if args.sweep_gemm else SWEEP_GEMM
        for N in sizes:
            A = torch.randn(N, N, device=dev).to(torch.bfloat16)
            B = torch.randn(N, N, device=dev).to(torch.bfloat16)
            Cm = torch.empty(N, N, device=dev, dtype=torch.bfloat16)
            ms = timeit(lambda: nnt.op_gemm(A, N, 0, B, N, 0, Cm, N, nnt.BF16, N, N, N, dtype=nnt.BF16))
            emit("gemm", [N, N, N], "bf16", ms, flops=2.0 * N ** 3)
            del A, B, Cm
    if "flash_attention" in kernels:
        # fused causal attention on [Z][S][hd] bf16 (GPT2-small and wide layer shapes);
        # algorithmic flops on the causal half: forward QK^T, PV; backward dV, dP, dQ, dK
        for Z, S, hd in ((48, 1024, 64), (128, 1024, 128)):
            q, k, v, do = (torch.randn(Z, S, hd, device=dev).to(torch.bfloat16) for _ in range(4))
            o = torch.empty_like(q)
            lse = torch.empty(Z, S, device=dev)
            dq, dk, dv = (torch.empty_like(q) for _ in range(3))
            pairs = Z * S * (S + 1) / 2
            ms = timeit(lambda: nnt.op_flash_attention_fwd(q, k, v, o, lse, Z, S, hd))
            emit("flash_attention_fwd", [Z, S, hd], "bf16", ms, flops=2 * 2.0 * hd * pairs)
            ms = timeit(lambda: nnt.op_flash_attention_bwd(q, k, v, o, do, lse, dq, dk, dv, Z, S, hd))
            emit("flash_attention_bwd", [Z, S, hd], "bf16", ms, flops=4 * 2.0 * hd * pairs)
            del q, k, v, do, o, dq, dk, dv
    print(json.dumps({"sweep_device_error": nnt.read_device_error()}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default="gpt2-small", choices=sorted(WORKLOADS))
    ap.add_argument("--streams", type=int, default=4)
    ap.add_argument("--tiles", default="", help='JSON object of tile sizes that override the '
                    'workload\'s, e.g. {"batch_tile": 2}')
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--separate", action="store_true",
                    help="backward, then AdamW over all parameters (default: AdamW fused into the "
                    "backward, each parameter chunk updated once its gradient is final)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep", action="store_true", help="tile-kernel sweep instead of the step")
    ap.add_argument("--capacity", action="store_true",
                    help="largest wide GPT2 that completes a step (plan first, then create and step)")
    ap.add_argument("--capacity-points", default="", help="comma list of LAYERSxD_MODEL")
    ap.add_argument("--sweep-kernel", default="", help="comma list (default: all)")
    ap.add_argument("--sweep-dtype", default="", choices=["", "f32", "bf16"])
    ap.add_argument("--sweep-rows", default="")
    ap.add_argument("--sweep-cols", default="")
    ap.add_argument("--sweep-gemm", default="", help="comma list of M=N=K")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "native":
        print("warning: fewer than 3 warm-up steps", file=sys.stderr)
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_sweep(args)
    if args.capacity:
        return run_capacity(args)
    return run_gpu(args)


if __name__ == "__main__":
    sys.exit(main())
