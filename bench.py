#!/usr/bin/env python
"""Benchmark of the Flint-shaped 4-bit sparse MoE FFN layer on B300.

Default: the headline workload is the 8192-token prefill chunk through one
Flint-shaped MoE layer (d=2048, f=512, 256 routed experts top-6 + 1 shared,
NVFP4 weights, Zipf-skewed router; the block-scaled FP4 tensor-core path),
the largest single-GPU configuration. The same run also times, as
sub-records with their own roofline, e2e and timing, the three decode
workloads: one layer at T=1 (NVFP4), one layer at T=64 (q4_1, Zipf), and the
47-layer stack at T=1. Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config 1..5] [--no-subrecords]
  python bench.py --impl reference ...   # the CPU oracle, timed on host cores
  python bench.py --head                 # the 4-bit output head and its sampler
  python bench.py --attn                 # one decode step of a sliding-window attention layer

A step is one pass of the layer (router, top-k, bucketing, expert gate/up,
down projection, combine) over the workload's tokens. Per-step device time is
taken with CUDA events on the launching stream around the forward only; the
L2 flush (a memset of twice the L2 size) runs between steps, outside those
events. With torchrun (N > 1) every rank runs an independent replica of the
workload on its own GPU (the layer does not shard); the reported time is the
maximum over ranks and the value counts the tokens of all ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from bit_quantized_expert_softmax_b300 import synth  # noqa: E402

METRIC = "MoE-layer tokens/s"
FALLBACK_HBM_GBS = 6400.0
FALLBACK_BF16_TFLOPS = 1800.0


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d.get("bf16_tflops", FALLBACK_BF16_TFLOPS)),
                "source": "measured"}
    return {"hbm_gbs": FALLBACK_HBM_GBS, "bf16_tflops": FALLBACK_BF16_TFLOPS, "source": "fallback"}


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Maximum of a float over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int, device=None) -> None:
    if world <= 1:
        return
    import torch.distributed as dist
    if device is not None and device.type == "cuda":
        dist.barrier(device_ids=[device.index])
    else:
        dist.barrier()


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines: list[str] = []
        self.thread = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=5)

    def summary(self) -> dict:
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax = float(parts[1])
            except ValueError:
                continue
            for n, v in zip(names, parts[4:8]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_id_for(device) -> str:
    import torch
    props = torch.cuda.get_device_properties(device)
    uuid = getattr(props, "uuid", None)
    if uuid is not None:
        s = str(uuid)
        return s if s.startswith("GPU-") else "GPU-" + s
    return str(device.index)


def source_digest(*paths) -> str:
    h = hashlib.sha256()
    for p in paths:
        with open(os.path.join(ROOT, p), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str, digest: str):
    """DRAM bytes per launch of `kernel` from a committed ncu capture, if the
    capture was taken on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as fh:
        d = json.load(fh)
    rec = d.get(f"{kernel}@{workload}")
    if not rec or rec.get("source_digest") != digest:
        return None
    return rec.get("dram_bytes_per_launch")


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i.get("num_threads", 1) for i in threadpool_info() if i.get("user_api") == "blas"]
        return max(n) if n else 1
    except Exception:
        return os.cpu_count() or 1


def fp4_peak(fm, device) -> dict:
    """Dense block-scaled FP4 tensor-core throughput of this GPU, measured by
    the library's probe (tcgen05.mma kind::mxf4nvf4, operands resident on
    chip, one CTA per SM): a short burst per MMA width and a ~0.5 s run
    under the clock sampler. The burst maximum is the FP4 roofline's peak."""
    burst = {}
    for n in (128, 256):
        ms, flops = fm.flint_moe_probe_fp4_peak(n, 4000 if n == 256 else 8000)
        burst[n] = flops / (ms * 1e-3) / 1e12
    n_best = max(burst, key=burst.get)
    iters = int(4000 * 500.0 / max(ms, 1e-3)) if n_best == 256 else int(8000 * 500.0 / max(ms, 1e-3))
    iters = max(1000, min(iters, (1 << 24) - 1))
    with ClockSampler(gpu_id_for(device)) as clk:
        ms_s, flops_s = fm.flint_moe_probe_fp4_peak(n_best, iters)
    sustained = flops_s / (ms_s * 1e-3) / 1e12
    c = clk.summary()
    return {"tflops": burst[n_best], "burst_tflops_by_n": {str(k): v for k, v in burst.items()},
            "sustained_tflops": sustained, "sustained_ms": ms_s, "mma": f"M=128, N={n_best}, K=64, cta_group::1",
            "clocks_sustained": c,
            "tflops_per_ghz_sustained": sustained / (c["sm_mhz"] / 1e3) if c.get("sm_mhz") else None,
            "source": "measured on this GPU by flint_moe_probe_fp4_peak (bench run)"}


# ---------------------------------------------------------------------------
# workload
# ---------------------------------------------------------------------------


def fp4_expert_path(cfg) -> bool:
    """Whether the library runs this workload's experts as block-scaled FP4
    GEMMs (NVFP4 weights, d=2048, f=512, more than 64 tokens); the bench
    checks this against the handle's own plan."""
    return cfg.wfmt == 0 and cfg.d == 2048 and cfg.f == 512 and cfg.tokens > 64


def algorithmic_bytes(cfg, n_active_experts: int, T: int) -> dict:
    """Bytes the layer must move once per step (weights of the experts it
    uses, router, activations), and those of its expert kernels: the 16-bit
    activation gate/up kernel, and the FP4 path's gate/up and down GEMMs
    (weights of the experts used, their NVFP4 activation rows in, h or the
    bf16 per-assignment contributions out), with the GEMMs' algorithmic FLOPs."""
    per_mat = cfg.codes_per_matrix + cfg.scales_per_matrix + (4 if cfg.wfmt == 0 else 0)
    selected = n_active_experts * 3 * per_mat
    router = cfg.router_bytes + cfg.n_experts * 4
    acts = 2 * T * cfg.d * 2
    P = T * (cfg.top_k + 1)
    gateup = n_active_experts * 2 * per_mat + T * cfg.d * 2 + P * cfg.f * 4
    # FP4 path: NVFP4 activation rows in (codes, E4M3 scales, fp32 row scale);
    # gate/up writes h in fp32, down writes one bf16 contribution row per
    # (token, expert) pair
    fp4_gemm1 = n_active_experts * 2 * per_mat + P * (cfg.d // 2 + cfg.d // 16 + 4) + P * cfg.f * 4
    fp4_gemm2 = n_active_experts * per_mat + P * (cfg.f // 2 + cfg.f // 16 + 4) + P * cfg.d * 2
    return {"selected_expert_bytes": selected, "layer_bytes": selected + router + acts,
            "gateup_kernel_bytes": gateup, "fp4_gemm1_bytes": fp4_gemm1, "fp4_gemm2_bytes": fp4_gemm2,
            "fp4_gemm1_flops": 2 * P * cfg.d * 2 * cfg.f, "fp4_gemm2_flops": 2 * P * cfg.f * cfg.d}


def e2e_pipelined(fm, m, T, x_pin, x_dev, o_dev, stream, K, world, device):
    """Per-step time (ms) of the forward through the public API with its host
    copies pipelined the way a serving loop runs them: the upload of step
    i+1 (pinned host -> device) and the download of step i-1 (device ->
    pinned host) run on their own streams while step i's forward runs, with
    two device buffer sets. Every step's copies are inside the timed region,
    which spans all K steps (events on the forward stream; the copy streams
    start after its first event and it waits for the last download). No L2
    flush: each step moves more than L2 through DRAM (large T only)."""
    import torch
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    xd = [x_dev, torch.empty_like(x_dev)]
    od = [o_dev, torch.empty_like(o_dev)]
    op = [torch.empty_like(x_pin).pin_memory() for _ in range(2)]
    in_done = [torch.cuda.Event() for _ in range(2)]
    fw_done = [torch.cuda.Event() for _ in range(2)]
    out_done = [torch.cuda.Event() for _ in range(2)]

    def step(i):
        b = i % 2
        if i >= 2:
            s_in.wait_event(fw_done[b])      # the forward two steps back has read xd[b]
        with torch.cuda.stream(s_in):
            xd[b].copy_(x_pin, non_blocking=True)
        in_done[b].record(s_in)
        stream.wait_event(in_done[b])
        if i >= 2:
            stream.wait_event(out_done[b])   # od[b] of two steps back is downloaded
        fm.flint_moe_forward(m.h, 0, xd[b].view(torch.bfloat16), T, od[b].view(torch.bfloat16), stream)
        fw_done[b].record(stream)
        s_out.wait_event(fw_done[b])
        with torch.cuda.stream(s_out):
            op[b].copy_(od[b], non_blocking=True)
        out_done[b].record(s_out)

    for i in range(3):
        step(i)
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(stream)
    s_in.wait_event(t0)
    s_out.wait_event(t0)
    for i in range(3, 3 + K):
        step(i)
    stream.wait_event(out_done[(2 + K) % 2])
    t1.record(stream)
    torch.cuda.synchronize()
    return max_over_ranks(t0.elapsed_time(t1) / K, world, device)


def run_ours(cfg, world, rank, local, steps: int, warmup: int, soak_s: float = 1.0):
    import torch
    from bit_quantized_expert_softmax_b300 import build
    build.build()
    from bit_quantized_expert_softmax_b300 import flint_moe as fm

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    T = cfg.tokens
    n_layers = cfg.n_layers
    m = fm.MoE(cfg, max_tokens=T, n_layers=n_layers, device=local)
    for i in range(n_layers):          # one layer in host memory at a time
        m.load(i, synth.make_layer(cfg, layer=i))
    bits = synth.make_hidden(cfg)
    x = fm.hidden_to_device(bits, local)
    out = torch.empty_like(x)
    stream = torch.cuda.current_stream(device)

    # routing of the workload (for the byte count): experts used + shared
    idx = torch.empty((T, cfg.top_k), dtype=torch.int32, device=device)
    fm.flint_moe_router(m.h, 0, x, T, None, idx, None)
    torch.cuda.synchronize()
    n_active = int(np.unique(idx.cpu().numpy()).size) + 1
    nbytes = algorithmic_bytes(cfg, n_active, T)
    if n_layers > 1:
        nbytes = {k: v * n_layers for k, v in nbytes.items()}   # per-layer routing differs; T=1 -> 7 each

    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=device)

    launches_per_forward = fm.flint_moe_forward_launches(m.h, T)
    plan = fm.flint_moe_tensor_core_plan(m.h, 0, T)
    assert bool(plan & 2) == fp4_expert_path(cfg), f"tensor-core plan {plan} for {cfg.name}"
    graph = None
    if n_layers > 1:
        xs = x.clone()
        # one CUDA graph per token for the whole stack
        n0 = fm.flint_moe_launch_count(m.h)
        fm.flint_moe_forward_stack(m.h, 0, n_layers, xs, T, stream)   # warm, outside capture
        torch.cuda.synchronize()
        stack_launches = fm.flint_moe_launch_count(m.h) - n0   # 1 for the one-launch kernel
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                fm.flint_moe_forward_stack(m.h, 0, n_layers, xs, T, torch.cuda.current_stream())
            torch.cuda.synchronize()
        except Exception as exc:   # capture refused: launch directly
            print(f"note: stack graph capture failed ({exc}); launching directly", file=sys.stderr)
            graph = None
            torch.cuda.synchronize()

        if graph is not None:
            def step():
                graph.replay()
        else:
            def step():
                fm.flint_moe_forward_stack(m.h, 0, n_layers, xs, T, stream)

        def reset():      # every step decodes the same token from the same input
            xs.copy_(x)
        launches_per_step = stack_launches
    else:
        def step():
            fm.flint_moe_forward(m.h, 0, x, T, out, stream)

        def reset():
            pass
        launches_per_step = launches_per_forward

    def timed(n_steps, profile=False):
        """n_steps steps, each: L2 flush, event, forward, event. A device-side
        sleep queued first lets the host run ahead, so the events time the
        device and not the host's launch latency."""
        st_ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_steps)]
        en_ev = [torch.cuda.Event(enable_timing=True) for _ in range(n_steps)]
        torch.cuda.synchronize()
        if profile:
            fm.flint_moe_profile_begin(m.h, n_steps)
        torch.cuda._sleep(50_000_000)            # ~25 ms of device time
        for i in range(n_steps):
            flush.zero_()
            reset()
            st_ev[i].record(stream)
            step()
            en_ev[i].record(stream)
        torch.cuda.synchronize()
        phases = fm.flint_moe_profile_end(m.h) if profile else None
        return [a.elapsed_time(b) for a, b in zip(st_ev, en_ev)], phases

    K = steps
    with ClockSampler(gpu_id_for(device)) as clk:
        # the sampler covers warm-up, an untimed soak of >= soak_s seconds of
        # the same steps, and the timed steps: its record describes the device
        # under this load even when the timed region itself is short
        for _ in range(warmup):
            flush.zero_()
            reset()
            step()
        torch.cuda.synchronize()
        status = fm.flint_moe_status(m.h)
        assert status == fm.FLINT_OK, f"device status {status} after warm-up"
        t_soak = time.perf_counter()
        while time.perf_counter() - t_soak < soak_s:
            for _ in range(50):
                flush.zero_()
                reset()
                step()
            torch.cuda.synchronize()
        barrier(world, device)
        torch.cuda.synchronize()
        launches0 = fm.flint_moe_launch_count(m.h)
        t0 = time.perf_counter()
        step_ms, _ = timed(K)
        wall = time.perf_counter() - t0
    barrier(world, device)
    launches = fm.flint_moe_launch_count(m.h) - launches0
    if graph is not None:
        launches = launches_per_step * K     # graph replays do not pass through the host counter
    status = fm.flint_moe_status(m.h)
    assert status == fm.FLINT_OK, f"device status {status} after the timed steps"
    ms = statistics.mean(step_ms)
    ms_max = max_over_ranks(ms, world, device)
    value = world * T / (ms_max / 1e3)
    phase_us = None
    if n_layers == 1 and launches_per_forward > 1:
        # per-kernel split of the multi-kernel path (a separate pass: the
        # extra events would otherwise sit inside the timed steps)
        _, (phase_ms, n_prof) = timed(min(K, 2000), profile=True)
        phase_us = {k: p_ / n_prof * 1e3 for k, p_ in zip(fm.PROFILE_PHASES, phase_ms)}

    # end to end through the public API: pinned host in -> forward -> pinned host out
    xh = fm.hidden_to_host(x).copy()
    x_pin = torch.from_numpy(xh.view(np.int16)).pin_memory()
    o_pin = torch.empty_like(x_pin).pin_memory()
    x_dev = torch.empty((T, cfg.d), dtype=torch.int16, device=device)
    o_dev = torch.empty_like(x_dev)
    Ke = min(K, 2000)
    es = [torch.cuda.Event(enable_timing=True) for _ in range(Ke)]
    ee = [torch.cuda.Event(enable_timing=True) for _ in range(Ke)]
    for i in range(Ke + 3):
        flush.zero_()
        j = i - 3
        if j >= 0:
            es[j].record(stream)
        x_dev.copy_(x_pin, non_blocking=True)
        if n_layers > 1:
            fm.flint_moe_forward_stack(m.h, 0, n_layers, x_dev.view(torch.bfloat16), T, stream)
            o_pin.copy_(x_dev, non_blocking=True)
        else:
            fm.flint_moe_forward(m.h, 0, x_dev.view(torch.bfloat16), T, o_dev.view(torch.bfloat16), stream)
            o_pin.copy_(o_dev, non_blocking=True)
        if j >= 0:
            ee[j].record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in zip(es, ee)), world, device)
    e2e_pipe_ms = e2e_pipelined(fm, m, T, x_pin, x_dev, o_dev, stream, min(K, 500), world, device) \
        if n_layers == 1 and T > 64 else None

    peaks = measured_peaks()
    res = {
        "step_ms": step_ms, "ms": ms_max, "value": value, "wall_s": wall, "launches": launches,
        "clocks": clk.summary(), "bytes": nbytes, "n_active": n_active,
        "e2e_value": world * T / (e2e_ms / 1e3), "e2e_ms": e2e_ms, "peaks": peaks,
        "e2e_pipe_ms": e2e_pipe_ms,
        "launches_per_forward": launches_per_forward, "phase_us": phase_us, "graph": graph is not None,
        "plan": plan,
    }
    m.close()
    return res


HEAD_MAX_T = 8   # tokens per output-head call (the library's limit)


def run_head(args, world, local):
    """The 4-bit output head and its sampler (temperature 1.0, top-k 20,
    top-p 0.95): one step = the head GEMV of the step's tokens + one draw per
    token, with L2 flushed between steps."""
    import torch
    from bit_quantized_expert_softmax_b300 import build
    build.build()
    from bit_quantized_expert_softmax_b300 import flint_moe as fm

    hcfg = synth.HEAD_CONFIGS["flint"]
    T, V, d = hcfg.tokens, hcfg.vocab, hcfg.d
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    m = fm.MoE(synth.LayerConfig(d=d, f=128, tokens=HEAD_MAX_T, name="head_host"), max_tokens=HEAD_MAX_T,
               device=local)
    hw = synth.make_head(hcfg)
    fm.flint_moe_load_lm_head(m.h, hw.codes, hw.scales, hw.tensor_scale)
    bits = synth.make_hidden(hcfg, tokens=T)
    x = fm.hidden_to_device(bits, local)
    logits = torch.empty((T, V), dtype=torch.float32, device=device)
    u = torch.from_numpy(synth.make_uniforms(T)).to(device)
    tokens = torch.empty((T,), dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=device)

    def step(x_in=x):
        fm.flint_moe_lm_head(m.h, x_in, T, logits, stream)
        fm.flint_moe_sample(m.h, logits, T, 1.0, 20, 0.95, u, tokens, None, stream)

    def timed(n, fn):
        st_ev = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        en_ev = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        torch.cuda.synchronize()
        torch.cuda._sleep(50_000_000)
        for i in range(n):
            flush.zero_()
            st_ev[i].record(stream)
            fn()
            en_ev[i].record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in zip(st_ev, en_ev)]

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    assert fm.flint_moe_status(m.h) == fm.FLINT_OK
    K = args.steps
    barrier(world, device)
    launches0 = fm.flint_moe_launch_count(m.h)
    with ClockSampler(gpu_id_for(device)) as clk:
        step_ms = timed(K, step)
    launches = fm.flint_moe_launch_count(m.h) - launches0
    barrier(world, device)
    gemv_ms = timed(min(K, 2000), lambda: fm.flint_moe_lm_head(m.h, x, T, logits, stream))
    assert fm.flint_moe_status(m.h) == fm.FLINT_OK
    ms = max_over_ranks(statistics.mean(step_ms), world, device)

    # end to end through the public API: pinned host x in, the drawn tokens out
    x_pin = torch.from_numpy(bits.view(np.int16)).pin_memory()
    t_pin = torch.empty((T,), dtype=torch.int32).pin_memory()
    x_dev = torch.empty((T, d), dtype=torch.int16, device=device)
    Ke = min(K, 2000)
    es = [torch.cuda.Event(enable_timing=True) for _ in range(Ke)]
    ee = [torch.cuda.Event(enable_timing=True) for _ in range(Ke)]
    for i in range(Ke + 3):
        flush.zero_()
        j = i - 3
        if j >= 0:
            es[j].record(stream)
        x_dev.copy_(x_pin, non_blocking=True)
        step(x_dev.view(torch.bfloat16))
        t_pin.copy_(tokens, non_blocking=True)
        if j >= 0:
            ee[j].record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in zip(es, ee)), world, device)
    m.close()
    w_bytes = V * d // 2 + V * d // 16
    return {"T": T, "V": V, "d": d, "ms": ms, "step_ms": step_ms, "gemv_us": statistics.mean(gemv_ms) * 1e3,
            "bytes": w_bytes + T * d * 2 + T * V * 4, "weight_bytes": w_bytes, "launches": launches,
            "clocks": clk.summary(), "e2e_ms": e2e_ms, "name": hcfg.name}


def head_cpu_baseline(seconds: float) -> dict:
    """The oracle's head and sampler on a bounded sample: the logits of a block
    of the head's rows per step, scaled to the whole vocabulary."""
    import oracle
    hcfg = synth.HEAD_CONFIGS["flint"]
    hw = synth.make_head(hcfg)
    rows = 8192
    el, n = 0.0, 0
    while el < seconds:
        bits = synth.make_hidden(hcfg, tokens=hcfg.tokens, stream=1 + n)
        r0 = (n * rows) % (hcfg.vocab - rows)
        t0 = time.perf_counter()
        lg = oracle.lm_head.head_logits(bits, hw.codes[r0:r0 + rows], hw.scales[r0:r0 + rows], hw.tensor_scale)
        oracle.lm_head.sample(lg.astype(np.float32), 1.0, 20, 0.95, np.full(hcfg.tokens, 0.5))
        el += time.perf_counter() - t0
        n += 1
    per_step = el / n * hcfg.vocab / rows
    return {"value": hcfg.tokens / per_step, "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"{n} steps of {rows} of the {hcfg.vocab} head rows (float64 oracle, {el:.1f} s), "
                      f"scaled to the whole head"}


def _oracle_rate(cfg, seconds: float, act_quant: bool, max_tokens: int | None = None) -> tuple[float, str]:
    """Tokens/s of the oracle (float64 numpy, as it stands) on a bounded
    sample of the workload, and a description of the sample."""
    import oracle
    T = cfg.tokens
    if cfg.n_layers > 1:
        # the stack: whole layers of it, one at a time, scaled to all layers
        el, n = 0.0, 0
        bits = synth.make_hidden(cfg, tokens=T, stream=1)
        while (el < seconds or n == 0) and n < cfg.n_layers:
            L = synth.make_layer(cfg, layer=n)
            t0 = time.perf_counter()
            r = oracle.moe.moe_layer(bits, L)
            bits = oracle.formats.bf16_bits(oracle.formats.bf16_round(
                oracle.formats.bf16_array(bits) + r.out_bf16))
            el += time.perf_counter() - t0
            n += 1
        return T / (el / n * cfg.n_layers), (f"{n} of the {cfg.n_layers} layers (T={T}) in {el:.1f} s, "
                                             f"scaled to the whole stack")
    L = synth.make_layer(cfg)
    Ts = T if max_tokens is None else min(T, max_tokens)
    done, steps = 0, 0
    t0 = time.perf_counter()
    while True:
        bits = synth.make_hidden(cfg, tokens=T, stream=1 + steps)
        r0 = (steps * Ts) % T
        oracle.moe.moe_layer(bits[r0:r0 + Ts], L, act_quant=act_quant)
        done += Ts
        steps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    what = "full steps of the workload" if Ts == T else f"samples of {Ts} of the workload's {T} tokens"
    return done / el, f"{steps} {what} ({done} tokens) in {el:.1f} s"


ONE_THREAD_ENV = {"OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1", "MKL_NUM_THREADS": "1",
                  "BLIS_NUM_THREADS": "1", "VECLIB_MAXIMUM_THREADS": "1", "NUMEXPR_NUM_THREADS": "1"}


def _oracle_rate_one_thread(cfg_id: int, seconds: float, act_quant: bool, max_tokens: int | None):
    """_oracle_rate in a child process whose BLAS pool has one thread (the
    pool size is fixed when numpy loads, so it is set in the child's
    environment)."""
    env = dict(os.environ, **ONE_THREAD_ENV)
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-rate", str(cfg_id), str(seconds),
           "1" if act_quant else "0", str(max_tokens or 0)]
    out = subprocess.run(cmd, env=env, capture_output=True, text=True, timeout=600, check=True).stdout
    d = json.loads(out.strip().splitlines()[-1])
    return d["value"], d["sample"]


def cpu_baseline(cfg, seconds: float, act_quant: bool = False, single_tokens: int | None = None) -> dict:
    """The CPU oracle (test infrastructure), timed as it stands on the host
    cores on a bounded sample of the workload, with the NVFP4 activation
    quantisation where the GPU path applies it: once with the BLAS pool at its
    default size (all cores) and once in a child process with one thread."""
    v_all, what_all = _oracle_rate(cfg, seconds, act_quant)
    cfg_id = next(i for i, c in synth.CONFIGS.items() if c.name == cfg.name)
    v_one, what_one = _oracle_rate_one_thread(cfg_id, seconds, act_quant, single_tokens)
    mode = "quantised activations (NVFP4)" if act_quant else "16-bit activations"
    return {"value": v_all, "unit": "tokens/s", "cores": blas_threads(), "nproc": os.cpu_count(), "kind": "oracle",
            "sample": f"float64 numpy oracle, {mode}, all cores: {what_all}",
            "single_thread": {"value": v_one, "unit": "tokens/s", "cores": 1,
                              "sample": f"one BLAS thread: {what_one}"}}


def kernel_roofline(cfg, res, peaks, fp4) -> dict:
    """roofline (dominant kernel), and the per-workload extras, of one run."""
    hbm = peaks["hbm_gbs"]
    nb = res["bytes"]
    out = {}
    layer_gbs = nb["layer_bytes"] / (res["ms"] * 1e-3) / 1e9
    hbm_src = "measured (MEASURED_PEAKS.json hbm_gbs)" if peaks["source"] == "measured" else "fallback 6.4 TB/s"
    if res["launches_per_forward"] == 1 and cfg.n_layers == 1:
        k_us, k_bytes = res["ms"] * 1e3, nb["layer_bytes"]
        kname = "decode_fused_kernel (the whole layer in one launch)"
        srcs = ("bit_quantized_expert_softmax_b300/csrc/decode_fused.cu", "bit_quantized_expert_softmax_b300/csrc/tiles.cuh",
                "bit_quantized_expert_softmax_b300/csrc/common.cuh")
        kkey = "decode_fused_kernel"
    elif res["phase_us"] is not None and res["plan"] & 2:
        # FP4 path: the gate/up GEMM (largest phase) against the measured FP4 peak
        ph = res["phase_us"]
        k_us = ph["gateup"]
        srcs = ("bit_quantized_expert_softmax_b300/csrc/moe_prefill.cu", "bit_quantized_expert_softmax_b300/csrc/gemm_fp4.cuh",
                "bit_quantized_expert_softmax_b300/csrc/umma.cuh", "bit_quantized_expert_softmax_b300/csrc/common.cuh")
        f1, f2 = nb["fp4_gemm1_flops"], nb["fp4_gemm2_flops"]
        achieved = f1 / (k_us * 1e-6) / 1e12
        g1_gbs = nb["fp4_gemm1_bytes"] / (k_us * 1e-6) / 1e9
        layer_tflops = (f1 + f2) / (res["ms"] * 1e-3) / 1e12
        # attainable: the slower of streaming the layer's bytes at the copy
        # bandwidth and its FP4 FLOPs at the measured peak
        t_bytes = nb["layer_bytes"] / (hbm * 1e9)
        t_flops = (f1 + f2) / (fp4["tflops"] * 1e12)
        out["roofline"] = {
            "bound": "tensor", "achieved": achieved, "peak": fp4["tflops"], "unit": "TFLOP/s",
            "frac": achieved / fp4["tflops"],
            "traffic": recorded_traffic("fp4_gemm_kernel<Gemm1>", cfg.name, source_digest(*srcs)),
            "kernel": "fp4_gemm_kernel<Gemm1> (expert gate/up, block-scaled FP4, SwiGLU epilogue)",
            "algorithmic_flops_per_launch": f1, "algorithmic_bytes_per_launch": nb["fp4_gemm1_bytes"],
            "avg_launch_us": k_us, "hbm_achieved_gbs": g1_gbs, "hbm_frac": g1_gbs / hbm,
            "peak_source": "measured: dense FP4 burst of this GPU (flint_moe_probe_fp4_peak, this run)",
        }
        out["tensor"] = {
            "gateup_tflops": achieved, "down_tflops": f2 / (ph["down_combine"] * 1e-6) / 1e12,
            "layer_tflops": layer_tflops, "layer_frac_of_fp4_peak": layer_tflops / fp4["tflops"],
            "layer_attainable_us": max(t_bytes, t_flops) * 1e6,
            "layer_frac_of_attainable": max(t_bytes, t_flops) / (res["ms"] * 1e-3),
            "down_hbm_frac": nb["fp4_gemm2_bytes"] / (ph["down_combine"] * 1e-6) / 1e9 / hbm,
        }
        out["phases_us"] = ph
        k_us = None
    elif res["phase_us"] is not None:
        k_us, k_bytes = res["phase_us"]["gateup"], nb["gateup_kernel_bytes"]
        ring = 8 < cfg.tokens <= 64 and os.environ.get("FLINT_MOE_RING_EXPERTS", "1") != "0"
        kkey = "gateup_ring_kernel" if ring else "gateup_kernel"
        kname = f"{kkey} (expert gate/up, SwiGLU)"
        srcs = ("bit_quantized_expert_softmax_b300/csrc/experts.cu", "bit_quantized_expert_softmax_b300/csrc/tiles.cuh",
                "bit_quantized_expert_softmax_b300/csrc/common.cuh")
        out["phases_us"] = {k: v for k, v in res["phase_us"].items()
                            if k in ("router_topk_bucket", "gateup", "down_combine")}
    else:
        # the stack (per-layer figures: the step's time and bytes over the
        # layers): one single-layer launch per layer, replayed from a CUDA
        # graph with FLINT_MOE_STACK_KERNEL=0; by default all layers in one
        # persistent launch
        one_launch = os.environ.get("FLINT_MOE_STACK_KERNEL", "1") != "0"
        k_us, k_bytes = res["ms"] * 1e3 / cfg.n_layers, nb["layer_bytes"] / cfg.n_layers
        kkey = "decode_stack_kernel" if one_launch else "decode_fused_kernel"
        kname = (f"{kkey} (per layer, one launch for the whole stack)" if one_launch
                 else f"{kkey} (per layer, inside the stack's CUDA graph)")
        srcs = ("bit_quantized_expert_softmax_b300/csrc/decode_fused.cu", "bit_quantized_expert_softmax_b300/csrc/tiles.cuh",
                "bit_quantized_expert_softmax_b300/csrc/common.cuh")
    if k_us is not None:
        achieved = k_bytes / (k_us * 1e-6) / 1e9
        out["roofline"] = {
            "bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
            "traffic": recorded_traffic(kkey, cfg.name, source_digest(*srcs)),
            "kernel": kname, "algorithmic_bytes_per_launch": k_bytes, "avg_launch_us": k_us,
            "peak_source": hbm_src,
        }
    out["layer_hbm"] = {"bytes_per_step": nb["layer_bytes"], "selected_expert_bytes_per_step": nb["selected_expert_bytes"],
                        "achieved_gbs": layer_gbs, "frac_of_measured": layer_gbs / hbm,
                        "selected_frac_of_measured": nb["selected_expert_bytes"] / (res["ms"] * 1e-3) / 1e9 / hbm,
                        "experts_read": res["n_active"]}
    return out


def workload_config(cfg) -> dict:
    return {"workload": f"{cfg.name}: {cfg.n_layers} MoE layer(s), d={cfg.d}, f={cfg.f}, "
                        f"{cfg.n_experts} routed experts top-{cfg.top_k} + 1 shared, "
                        f"{'NVFP4' if cfg.wfmt == 0 else 'q4_1'} weights, T={cfg.tokens}"
                        + (", Zipf(1.1) router bias" if cfg.bias == "zipf" else ""),
            "tokens_per_step": cfg.tokens,
            "l2": "flushed between steps (memset of 2x L2, outside the per-step events)"}


def record(cfg, res, peaks, fp4, world) -> dict:
    """The measured numbers of one workload: value, timing, roofline, e2e,
    launches and clocks."""
    r = {"value": res["value"], "unit": "tokens/s", "ms_per_step": res["ms"],
         "dtype": "nvfp4" if res["plan"] & 2 else ("q4_1 weights, f16 activations" if cfg.wfmt == 1
                                                   else "nvfp4 weights, f16 activations"),
         "config": workload_config(cfg)}
    r.update(kernel_roofline(cfg, res, peaks, fp4))
    r["e2e"] = {"value": res["e2e_value"], "unit": "tokens/s", "h2d_bytes_per_step": cfg.tokens * cfg.d * 2,
                "d2h_bytes_per_step": cfg.tokens * cfg.d * 2,
                "method": "per step: upload, forward, download in order on one stream (L2 flushed between "
                          "steps, outside the step's events)"}
    if res.get("e2e_pipe_ms"):
        # large T: the serving form, copies overlapped with the neighbouring
        # steps' forwards; the serial figure is kept beside it
        r["e2e"].update({
            "value": world * cfg.tokens / (res["e2e_pipe_ms"] / 1e3),
            "method": "pipelined: the upload of step i+1 and the download of step i-1 on their own streams "
                      "while step i's forward runs (two device buffer sets); every step's copies inside "
                      "the timed region spanning all steps",
            "serial_value": res["e2e_value"],
            "serial_method": "per step: upload, forward, download in order on one stream"})
    r["gpu_launches"] = int(res["launches"])
    r["clocks"] = res["clocks"]
    step_ms = np.array(res["step_ms"])
    r["step_ms_p10_p50_p90"] = [float(np.percentile(step_ms, q)) for q in (10, 50, 90)]
    return r


# sub-records of the default run: (config, timed steps, warm-up steps)
SUBRECORDS = [(2, 2000, 200), (3, 1000, 100), (4, 200, 10)]


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------


def reference_main(args, cfg, rank):
    """The reference arm: the CPU oracle as it stands, on the host cores, on
    the same workload, metric and unit; each timed step is a bounded sample
    (at most 2048 of the workload's tokens, rotating over the batch), the
    warm-up steps 64-token samples, the whole run capped at ~2.5 minutes."""
    if rank != 0:
        return
    import oracle
    budget = 150.0
    t_all = time.perf_counter()
    n_keep = min(cfg.n_layers, 4)     # a stack step is timed on its first layers and scaled
    layers = [synth.make_layer(cfg, layer=i) for i in range(n_keep)]
    aq = fp4_expert_path(cfg)
    Ts = min(cfg.tokens, 2048)
    for i in range(args.warmup):
        bits = synth.make_hidden(cfg, stream=100 + i)[:min(cfg.tokens, 64)]
        oracle.moe.moe_layer(bits, layers[0], act_quant=aq)
    steps = []
    for i in range(args.steps):
        bits = synth.make_hidden(cfg, stream=1 + i)
        r0 = (i * Ts) % cfg.tokens
        t0 = time.perf_counter()
        for L in layers:
            oracle.moe.moe_layer(bits[r0:r0 + Ts], L, act_quant=aq)
        steps.append((time.perf_counter() - t0) * cfg.n_layers / n_keep)
        if time.perf_counter() - t_all > budget and len(steps) >= 3:
            break
    ms = statistics.mean(steps) * 1e3
    value = Ts / (ms / 1e3)
    sample = (f"{len(steps)} steps, each the oracle on {Ts} of the workload's {cfg.tokens} tokens"
              + (f" through {n_keep} of the {cfg.n_layers} layers, scaled" if n_keep < cfg.n_layers else "")
              + f"; {args.warmup} warm-up steps of 64 tokens; run capped at {budget:.0f} s")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": len(steps), "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "oracle_mode": "quantised activations (NVFP4)" if aq else "16-bit activations",
            "data": "synthetic", "config": workload_config(cfg),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "kind": "oracle", "cores": blas_threads(),
                             "nproc": os.cpu_count(), "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    if len(sys.argv) == 6 and sys.argv[1] == "--oracle-rate":
        # child of cpu_baseline: one oracle timing, printed as JSON
        cfg = synth.CONFIGS[int(sys.argv[2])]
        mt = int(sys.argv[5])
        v, what = _oracle_rate(cfg, float(sys.argv[3]), sys.argv[4] == "1", max_tokens=mt or None)
        print(json.dumps({"value": v, "sample": what}))
        return
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps of the headline workload (default: about 1 s of device time)")
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", type=int, default=5, choices=sorted(synth.CONFIGS),
                    help="headline workload (default 5: the 8192-token prefill)")
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--soak", type=float, default=1.0,
                    help="seconds of untimed steps under the clock sampler just before the timed steps")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-subrecords", action="store_true",
                    help="time only the headline workload (default with --config other than 5)")
    ap.add_argument("--attn", action="store_true",
                    help="one decode step of a sliding-window attention layer (64 sequences) instead of an MoE config")
    ap.add_argument("--head", action="store_true",
                    help="the 4-bit output head (146,432 x 2048 NVFP4) and its sampler instead of an MoE config")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.head:
        head_main(args)
        return
    if args.attn:
        attn_main(args)
        return
    cfg = synth.CONFIGS[args.config]
    if args.steps is None:
        args.steps = {1: 20000, 2: 20000, 3: 10000, 4: 5000, 5: 3000}[args.config]
    world, rank, local = dist_env()
    if world != args.gpus and world > 1:
        print(f"warning: WORLD_SIZE={world} but --gpus {args.gpus}", file=sys.stderr)

    if args.impl == "reference":
        reference_main(args, cfg, rank)
        return

    import torch
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from bit_quantized_expert_softmax_b300 import build
    build.build()
    from bit_quantized_expert_softmax_b300 import flint_moe as fm
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    peaks = measured_peaks()
    fp4 = fp4_peak(fm, device)
    res = run_ours(cfg, world, rank, local, args.steps, args.warmup, soak_s=args.soak)
    subs = {}
    if args.config == 5 and not args.no_subrecords:
        for c, k, w in SUBRECORDS:
            scfg = synth.CONFIGS[c]
            subs[scfg.name] = (scfg, k, w, run_ours(scfg, world, rank, local, k, w, soak_s=min(0.5, args.soak)))
    if rank == 0:
        line = {
            "metric": METRIC, "value": res["value"], "unit": "tokens/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "data": "synthetic",
        }
        rec = record(cfg, res, peaks, fp4, world)
        line.update({k: v for k, v in rec.items() if k not in ("value", "unit", "ms_per_step")})
        line["fp4_peak"] = fp4
        if subs:
            line["subrecords"] = {}
            for name, (scfg, k, w, sres) in subs.items():
                sr = record(scfg, sres, peaks, fp4, world)
                sr.update({"steps": k, "warmup": w})
                line["subrecords"][name] = sr
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_baseline(cfg, args.cpu_seconds, act_quant=bool(res["plan"] & 2),
                                                single_tokens=512)
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


ATTN_B, ATTN_POS, ATTN_CAP = 64, 4096, 520   # sequences, position of the decoded token, cache slots


def run_attn(args, world, local):
    """One decode step of a sliding-window attention layer for ATTN_B
    sequences whose window is full (position 4096: 512 cached positions plus
    the new token), with L2 flushed between steps."""
    import torch
    from bit_quantized_expert_softmax_b300 import build
    build.build()
    from bit_quantized_expert_softmax_b300 import flint_moe as fm
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    rng = np.random.default_rng(0)
    B, H, KV, cap = ATTN_B, 32, 4, ATTN_CAP

    def bf16(shape, scale=1.0):
        return (torch.from_numpy(rng.standard_normal(shape).astype(np.float32) * scale)
                .to(torch.bfloat16).to(device))
    q, k, v = bf16((B, H, 128)), bf16((B, KV, 128)), bf16((B, KV, 128))
    kc, vc = bf16((B, KV, cap, 128)), bf16((B, KV, cap, 128))
    wq = torch.from_numpy((1 + 0.1 * rng.standard_normal(128)).astype(np.float32)).to(device)
    wk = torch.from_numpy((1 + 0.1 * rng.standard_normal(128)).astype(np.float32)).to(device)
    sinks = torch.from_numpy(rng.standard_normal(H).astype(np.float32)).to(device)
    pos = torch.full((B,), ATTN_POS, dtype=torch.int32, device=device)
    out = torch.empty((B, H, 128), dtype=torch.bfloat16, device=device)
    stream = torch.cuda.current_stream(device)
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    flush = torch.empty(max(2 * l2, 256 << 20) // 4, dtype=torch.float32, device=device)

    def step(qq=q, oo=out):
        fm.flint_moe_attn_decode(H, KV, 513, cap, True, B, qq, k, v, kc, vc, pos, wq, wk, sinks, oo, stream=stream)

    for _ in range(args.warmup):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    K = args.steps
    st_ev = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    en_ev = [torch.cuda.Event(enable_timing=True) for _ in range(K)]
    with ClockSampler(gpu_id_for(device)) as clk:
        t_soak = time.perf_counter()
        while time.perf_counter() - t_soak < args.soak:
            for _ in range(50):
                flush.zero_()
                step()
            torch.cuda.synchronize()
        torch.cuda._sleep(50_000_000)
        for i in range(K):
            flush.zero_()
            st_ev[i].record(stream)
            step()
            en_ev[i].record(stream)
        torch.cuda.synchronize()
    step_ms = [a.elapsed_time(b) for a, b in zip(st_ev, en_ev)]
    ms = max_over_ranks(statistics.mean(step_ms), world, device)
    # end to end: q, k, v from pinned host memory, the output back
    q_pin = q.cpu().pin_memory()
    o_pin = torch.empty_like(out, device="cpu").pin_memory()
    q_dev = torch.empty_like(q)
    Ke = min(K, 2000)
    es = [torch.cuda.Event(enable_timing=True) for _ in range(Ke)]
    ee = [torch.cuda.Event(enable_timing=True) for _ in range(Ke)]
    for i in range(Ke + 3):
        flush.zero_()
        j = i - 3
        if j >= 0:
            es[j].record(stream)
        q_dev.copy_(q_pin, non_blocking=True)
        step(q_dev, out)
        o_pin.copy_(out, non_blocking=True)
        if j >= 0:
            ee[j].record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(statistics.mean(a.elapsed_time(b) for a, b in zip(es, ee)), world, device)
    kv_bytes = B * KV * 512 * 128 * 2 * 2              # cached keys and values read
    io_bytes = B * (H + 2 * KV) * 128 * 2 + B * H * 128 * 2 + B * KV * 128 * 2 * 2
    return {"ms": ms, "step_ms": step_ms, "bytes": kv_bytes + io_bytes, "clocks": clk.summary(), "e2e_ms": e2e_ms,
            "B": B, "h2d": B * H * 128 * 2, "d2h": B * H * 128 * 2}


def attn_cpu_baseline(seconds: float) -> dict:
    import oracle.attention as OA
    rng = np.random.default_rng(1)
    cap = ATTN_CAP
    q = rng.standard_normal((32, 128))
    k = rng.standard_normal((4, 128))
    v = rng.standard_normal((4, 128))
    kc = oracle_bits(rng.standard_normal((4, cap, 128)))
    vc = oracle_bits(rng.standard_normal((4, cap, 128)))
    w = np.ones(128)
    sinks = rng.standard_normal(32)
    n, t0 = 0, time.perf_counter()
    while time.perf_counter() - t0 < seconds or n == 0:
        OA.decode_step(q, k, v, kc, vc, ATTN_POS, w, w, sinks)
        n += 1
    el = time.perf_counter() - t0
    return {"value": n / el, "unit": "tokens/s", "cores": blas_threads(), "nproc": os.cpu_count(), "kind": "oracle",
            "sample": f"{n} single-sequence decode steps through the float64 oracle in {el:.1f} s"}


def oracle_bits(v):
    import oracle
    return oracle.formats.bf16_bits(oracle.formats.bf16_round(v))


def attn_main(args):
    import torch
    if args.steps is None:
        args.steps = 2000
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    r = run_attn(args, world, local)
    if rank == 0:
        peaks = measured_peaks()
        hbm = peaks["hbm_gbs"]
        achieved = r["bytes"] / (r["ms"] * 1e-3) / 1e9
        line = {
            "metric": "attention decode tokens/s", "value": world * r["B"] / (r["ms"] / 1e3), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16 cache, f32 math",
            "data": "synthetic",
            "config": {"workload": f"sliding-window attention layer decode: {r['B']} sequences at position {ATTN_POS} "
                                   f"(513-token window full), 32 query / 4 key-value heads of 128, QK RMSNorm, "
                                   f"rotary positions, sinks, bf16 cache",
                       "tokens_per_step": r["B"],
                       "l2": "flushed between steps (memset of 2x L2, outside the per-step events)"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                         "traffic": recorded_traffic("attn_decode_kernel", f"attn_decode_B{r['B']}_pos{ATTN_POS}",
                                                     source_digest("bit_quantized_expert_softmax_b300/csrc/attention.cu")),
                         "kernel": "attn_decode_kernel (one step, the whole layer)",
                         "algorithmic_bytes_per_launch": r["bytes"], "avg_launch_us": r["ms"] * 1e3,
                         "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if peaks["source"] == "measured"
                         else "fallback 6.4 TB/s"},
            "e2e": {"value": world * r["B"] / (r["e2e_ms"] / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": r["h2d"],
                    "d2h_bytes_per_step": r["d2h"]},
            "gpu_launches": args.steps, "clocks": r["clocks"],
        }
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = attn_cpu_baseline(min(args.cpu_seconds, 10.0))
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def head_main(args):
    import torch
    if args.steps is None:
        args.steps = 5000
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    r = run_head(args, world, local)
    if rank == 0:
        peaks = measured_peaks()
        hbm = peaks["hbm_gbs"]
        achieved = r["bytes"] / (r["gemv_us"] * 1e-6) / 1e9
        srcs = ("bit_quantized_expert_softmax_b300/csrc/lm_head.cu", "bit_quantized_expert_softmax_b300/csrc/tiles.cuh",
                "bit_quantized_expert_softmax_b300/csrc/common.cuh")
        line = {
            "metric": METRIC + " (output head)", "value": world * r["T"] / (r["ms"] / 1e3), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "nvfp4 weights, f16 x",
            "data": "synthetic",
            "config": {"workload": f"{r['name']}: NVFP4 output head {r['V']} x {r['d']}, T={r['T']}, then one draw "
                                   f"per token at temperature 1.0, top-k 20, top-p 0.95",
                       "tokens_per_step": r["T"],
                       "l2": "flushed between steps (memset of 2x L2, outside the per-step events)"},
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                         "traffic": recorded_traffic("head_gemv_kernel", r["name"], source_digest(*srcs)),
                         "kernel": "head_gemv_kernel (NVFP4 GEMV, mma.sync with tokens as rows)",
                         "algorithmic_bytes_per_launch": r["bytes"], "avg_launch_us": r["gemv_us"],
                         "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs)" if peaks["source"] == "measured"
                         else "fallback 6.4 TB/s"},
            "e2e": {"value": world * r["T"] / (r["e2e_ms"] / 1e3), "unit": "tokens/s",
                    "h2d_bytes_per_step": r["T"] * r["d"] * 2, "d2h_bytes_per_step": r["T"] * 4},
            "gpu_launches": int(r["launches"]), "clocks": r["clocks"],
        }
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = head_cpu_baseline(args.cpu_seconds)
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
