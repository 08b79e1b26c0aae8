"""Failure path of the kernels' bounded waits, and the FP4 tensor-core probe.

Every spin-wait in the kernels (mbarrier phases, grid barriers) has a limit;
when it runs out the kernel records FLINT_ETIMEOUT in the status word and
returns instead of hanging. Here a wait is made to run out on purpose, with a
short limit and nothing in flight, and the handle must report the timeout and
then compute a layer correctly again. No GPU is faulted or hung: the waits
are bounded by the limit the test passes.
"""
import numpy as np
import pytest

from bit_quantized_expert_softmax_b300 import synth
from oracle import moe as M
from tests.gpu_util import assert_out_close

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def fm():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from bit_quantized_expert_softmax_b300 import build
    build.build()
    from bit_quantized_expert_softmax_b300 import flint_moe
    flint_moe.lib()
    return flint_moe


@pytest.mark.parametrize("kind", [0, 1])
def test_wait_that_runs_out_reports_timeout_and_handle_recovers(fm, kind):
    cfg = synth.CONFIGS[1]
    layer = synth.make_layer(cfg)
    bits = synth.make_hidden(cfg)
    m = fm.MoE(cfg, max_tokens=cfg.tokens)
    try:
        m.load(0, layer)
        assert fm.flint_moe_status(m.h) == fm.FLINT_OK
        fm.flint_moe_debug_wait_timeout(m.h, kind, 1000)
        assert fm.flint_moe_status(m.h) == fm.FLINT_ETIMEOUT
        assert fm.flint_moe_status(m.h) == fm.FLINT_OK          # read and cleared
        # the single-launch decode kernel (grid barriers) and the multi-kernel
        # path both still compute the layer
        for T in (1, cfg.tokens):
            out = m.forward(fm.hidden_to_device(bits[:T]))
            torch.cuda.synchronize()
            assert fm.flint_moe_status(m.h) == fm.FLINT_OK
            ref = M.moe_layer(bits[:T], layer)
            assert_out_close(fm.hidden_to_host(out), ref.out, f"after timeout kind {kind}, T={T}")
    finally:
        m.close()


def test_wait_timeout_rejects_bad_arguments(fm):
    cfg = synth.CONFIGS[1]
    m = fm.MoE(cfg, max_tokens=4)
    try:
        for kind, limit in [(2, 10), (-1, 10), (0, 0), (1, (1 << 20) + 1)]:
            with pytest.raises(fm.FlintError) as ei:
                fm.flint_moe_debug_wait_timeout(m.h, kind, limit)
            assert ei.value.code == fm.FLINT_EINVAL
    finally:
        m.close()


@pytest.mark.parametrize("n", [128, 256])
def test_fp4_peak_probe_runs(fm, n):
    """The probe completes and reports a throughput between a tenth of and
    twice the nominal dense FP4 figure of a B300 (~15 PFLOP/s): it runs the
    MMAs it counts, and no more."""
    ms, flops = fm.flint_moe_probe_fp4_peak(n, 20000)
    assert ms > 0 and flops > 0
    tflops = flops / (ms * 1e-3) / 1e12
    assert 1500 < tflops < 30000, tflops
    with pytest.raises(fm.FlintError):
        fm.flint_moe_probe_fp4_peak(64, 10)
