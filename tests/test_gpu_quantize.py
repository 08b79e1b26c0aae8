"""GPU NVFP4 quantisation of bf16 weight matrices (one fp32 tensor scale per
matrix) against the oracle, bit for bit, and through the layer: weights
quantised on the GPU, loaded, dequantised by the export and run through a
forward, against the oracle on the same codes."""
import numpy as np
import pytest

from bit_quantized_expert_softmax_b300 import synth
from oracle import formats as F
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


def _bf16(v):
    return F.bf16_bits(F.bf16_round(np.asarray(v, dtype=np.float64)))


def _gpu_quant(fm, bits):
    R, K = bits.shape
    w = torch.from_numpy(bits.view(np.int16)).cuda()
    codes = torch.full((R, K // 2), 0xAA, dtype=torch.uint8, device="cuda")
    scales = torch.full((R, K // 16), 0xAA, dtype=torch.uint8, device="cuda")
    ts = torch.full((1,), -1.0, dtype=torch.float32, device="cuda")
    fm.flint_moe_quantize_nvfp4(w, R, K, codes, scales, ts)
    torch.cuda.synchronize()
    return codes.cpu().numpy(), scales.cpu().numpy(), np.float32(ts.item())


def _packed(codes):
    c = codes.astype(np.uint8)
    return (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)


@pytest.mark.parametrize("R,K,seed,mag", [(1, 16, 1, 1.0), (7, 48, 2, 1e-3), (64, 256, 3, 30.0),
                                          (512, 2048, 4, 0.02), (2048, 512, 5, 0.02)])
def test_quantize_bit_exact(fm, R, K, seed, mag):
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((R, K)) * mag * np.exp(rng.uniform(-2, 2, size=(R, 1)))
    if R > 2:
        v[1] = 0.0                                     # a zero row: zero blocks inside a non-zero matrix
        v[2, :16] = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0] * 2) * mag   # grid-aligned values
    bits = _bf16(v)
    codes, scales, ts = _gpu_quant(fm, bits)
    rc, rsb, rs, _ = M.quant_weight_nvfp4(F.bf16_array(bits).astype(np.float32))
    assert ts == rs
    assert np.array_equal(scales, rsb)
    assert np.array_equal(codes, _packed(rc))


def test_quantize_zero_matrix_and_bad_arguments(fm):
    codes, scales, ts = _gpu_quant(fm, np.zeros((3, 32), dtype=np.uint16))
    assert ts == 0.0 and not codes.any() and not scales.any()
    for R, K in [(0, 16), (4, 8), (4, 24)]:
        with pytest.raises(fm.FlintError) as ei:
            fm.flint_moe_quantize_nvfp4(None, R, K, None, None, None)
        assert ei.value.code == fm.FLINT_EINVAL


def test_quantized_weights_through_the_layer(fm):
    """bf16 expert weights of the tiny shape quantised on the GPU, loaded and
    run: the dequantisation export equals the oracle's dequantisation of the
    oracle's own quantisation, and the layer matches the oracle."""
    cfg = synth.CONFIGS[1]
    L = synth.make_layer(cfg)
    rng = np.random.default_rng(9)
    n = cfg.n_experts + 1
    codes = np.empty_like(L.codes)
    scales = np.empty_like(L.scales)
    tscale = np.empty_like(L.tensor_scale)
    for e in range(n):
        for mat in range(3):
            R, K = (cfg.f, cfg.d) if mat < 2 else (cfg.d, cfg.f)
            bits = _bf16(rng.standard_normal((R, K)) * 0.02)
            c, sb, ts = _gpu_quant(fm, bits) if (e < 3 or e == n - 1) else (None, None, None)
            rc, rsb, rs, _ = M.quant_weight_nvfp4(F.bf16_array(bits).astype(np.float32))
            if c is not None:
                assert np.array_equal(c, _packed(rc)) and np.array_equal(sb, rsb) and ts == rs
            codes[e, mat] = _packed(rc).reshape(-1)
            scales[e, mat] = rsb.reshape(-1)
            tscale[e, mat] = rs
    L.codes, L.scales, L.tensor_scale = codes, scales, tscale
    m = fm.MoE(cfg, max_tokens=cfg.tokens)
    try:
        m.load(0, L)
        out = torch.empty((cfg.d, cfg.f), dtype=torch.float32, device="cuda")
        fm.flint_moe_dequant(m.h, 0, n - 1, 2, out)
        torch.cuda.synchronize()
        want = M.dequant_matrix(L, n - 1, 2).astype(np.float32)
        assert np.array_equal(out.cpu().numpy(), want)
        bits = synth.make_hidden(cfg)
        got = fm.hidden_to_host(m.forward(fm.hidden_to_device(bits)))
        torch.cuda.synchronize()
        assert_out_close(got, M.moe_layer(bits, L).out, "layer on GPU-quantised weights")
    finally:
        m.close()
