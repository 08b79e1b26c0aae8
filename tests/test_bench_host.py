"""Host-side logic of bench.py: the max-over-ranks reduction and barrier used
for N > 1 replicas (world size 2, gloo, on CPU), byte accounting, and the
clock-sample summary."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from bit_quantized_expert_softmax_b300 import synth


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    bench.barrier(world)
    got = bench.max_over_ranks(1.5 + rank, world)
    q.put((rank, got))
    dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = dict(q.get(timeout=5) for _ in range(2))
    assert res == {0: 2.5, 1: 2.5}


def test_single_rank_reduction_is_identity():
    assert bench.max_over_ranks(3.25, 1) == 3.25


def test_algorithmic_bytes_decode_layer():
    cfg = synth.CONFIGS[2]
    b = bench.algorithmic_bytes(cfg, 7, 1)
    # 7 experts x 3 matrices x (512 KiB codes + 64 KiB scales + 4 B tensor scale)
    assert b["selected_expert_bytes"] == 7 * 3 * (524288 + 65536 + 4)
    assert b["layer_bytes"] == b["selected_expert_bytes"] + 256 * 2048 * 4 + 256 * 4 + 2 * 2048 * 2
    assert b["gateup_kernel_bytes"] == 7 * 2 * (524288 + 65536 + 4) + 2048 * 2 + 7 * 512 * 4


def test_clock_summary_parses_nvidia_smi_lines():
    c = bench.ClockSampler("0")
    c.lines = ["1965, 2032, 700.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
               "1980, 2032, 720.1, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
               "garbage"]
    s = c.summary()
    assert s["sm_mhz"] == pytest.approx(1972.5) and s["sm_max_mhz"] == 2032
    assert s["reasons"] == ["sw_power_cap"] and s["samples"] == 2


def _decode_res(e2e_pipe_ms):
    cfg = synth.CONFIGS[2]
    return cfg, {
        "value": 48000.0, "ms": 0.0206, "step_ms": [0.0206, 0.0207], "launches": 2000,
        "launches_per_forward": 1, "plan": 0, "phase_us": None,
        "bytes": bench.algorithmic_bytes(cfg, 7, 1), "clocks": {"samples": 0}, "n_active": 7,
        "e2e_value": 27000.0, "e2e_pipe_ms": e2e_pipe_ms,
    }


def test_record_e2e_serial_and_pipelined():
    """The e2e figure: the serial per-step form by default; with a pipelined
    per-step time, that form's value, the serial one kept beside it."""
    peaks = {"hbm_gbs": 6480.8, "source": "measured"}
    cfg, res = _decode_res(None)
    r = bench.record(cfg, res, peaks, None, 1)
    assert r["e2e"]["value"] == 27000.0 and "serial_value" not in r["e2e"]
    assert r["e2e"]["h2d_bytes_per_step"] == r["e2e"]["d2h_bytes_per_step"] == cfg.tokens * cfg.d * 2
    cfg, res = _decode_res(0.04)
    r = bench.record(cfg, res, peaks, None, 2)
    assert r["e2e"]["value"] == pytest.approx(2 * cfg.tokens / 0.04e-3)
    assert r["e2e"]["serial_value"] == 27000.0 and r["e2e"]["method"].startswith("pipelined")
