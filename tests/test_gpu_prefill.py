"""The large-T expert path on the block-scaled FP4 tensor cores (NVFP4 weights,
d = 2048, f = 512): activation quantisation bit for bit, and whole layers
against the oracle's quantised-activation expert (activations entering each
projection are NVFP4 with a per-token fp32 scale; h is quantised from its
float32 value)."""
import dataclasses

import numpy as np
import pytest

from bit_quantized_expert_softmax_b300 import synth
from oracle import formats as F
from oracle import moe as M
from tests.gpu_util import assert_out_close, compare_routing

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


def _bf16_bits(v: np.ndarray) -> np.ndarray:
    return F.bf16_bits(F.bf16_round(v))


# ---------------------------------------------------------------------------
# a9: activation quantisation, bit for bit
# ---------------------------------------------------------------------------


def _act_rows(K: int, T: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    v = rng.standard_normal((T, K)) * np.exp(rng.uniform(-6, 6, size=(T, 1)))
    v[0] = 0.0                                      # zero row: scale 0, codes 0
    v[1] = 0.0
    v[1, 17] = -3.0                                 # one non-zero element
    # exact E2M1 ties: amax 336 gives s_t = 1/8; a block of max 1.5 gets the
    # scale byte of 2.0, S = 0.25, and these values sit halfway between codes
    v[2] = 0.0
    v[2, 0] = 336.0
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0]) * 0.25
    v[2, 16:24] = ties
    v[2, 24:32] = -ties
    v[3] = rng.standard_normal(K) * 1e-20           # tiny but normal fp32 scales
    v[4] = rng.standard_normal(K) * 1e30            # huge
    v[5, :] = np.where(rng.random(K) < 0.5, -1e-3, 1e-3)
    v[5, 100] = 50.0                                 # most blocks far below amax
    return _bf16_bits(v)


@pytest.mark.parametrize("K", [2048, 512])
def test_act_quant_bit_exact(fm, K):
    T = 37
    bits = _act_rows(K, T, K)
    x = fm.hidden_to_device(bits)
    codes = torch.empty((T, K // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty((T, K // 16), dtype=torch.uint8, device="cuda")
    rows = torch.empty((T,), dtype=torch.float32, device="cuda")
    fm.flint_moe_debug_act_quant(x, T, K, codes, scales, rows)
    torch.cuda.synchronize()
    want_codes, want_sb, want_rows, _ = M.quant_act_nvfp4(F.bf16_array(bits).astype(np.float32))
    packed = (want_codes[:, 0::2] | (want_codes[:, 1::2] << 4)).astype(np.uint8)
    got_rows = rows.cpu().numpy()
    assert np.array_equal(got_rows.view(np.uint32), want_rows.astype(np.float32).view(np.uint32))
    assert np.array_equal(scales.cpu().numpy(), want_sb)
    got = codes.cpu().numpy()
    bad = np.argwhere(got != packed)
    assert bad.size == 0, f"{len(bad)} code bytes differ, first at {bad[:4].tolist()}"


def test_act_quant_rejects_bad_arguments(fm):
    x = torch.zeros((4, 2048), dtype=torch.bfloat16, device="cuda")
    c = torch.empty((4, 1024), dtype=torch.uint8, device="cuda")
    s = torch.empty((4, 128), dtype=torch.uint8, device="cuda")
    r = torch.empty((4,), dtype=torch.float32, device="cuda")
    for K in (1024, 4096, 0):
        rc = fm.lib().flint_moe_debug_act_quant(x.data_ptr(), 4, K, c.data_ptr(), s.data_ptr(), r.data_ptr(), None)
        assert rc == fm.FLINT_EINVAL
    rc = fm.lib().flint_moe_debug_act_quant(x.data_ptr() + 2, 4, 2048, c.data_ptr(), s.data_ptr(), r.data_ptr(),
                                            None)
    assert rc == fm.FLINT_EINVAL


# ---------------------------------------------------------------------------
# the layer on the FP4 tensor-core path
# ---------------------------------------------------------------------------


def _prefill_parity(fm, cfg, T, sample=None, max_tokens=None):
    L = synth.make_layer(cfg)
    bits = synth.make_hidden(cfg, tokens=T)
    m = fm.MoE(cfg, max_tokens=max_tokens or T, n_layers=1)
    m.load(0, L)
    plan = fm.flint_moe_tensor_core_plan(m.h, 0, T)
    x = fm.hidden_to_device(bits)
    out = m.forward(x, 0)
    torch.cuda.synchronize()
    assert fm.flint_moe_status(m.h) == fm.FLINT_OK
    got = fm.hidden_to_host(out)
    idx = torch.empty((T, cfg.top_k), dtype=torch.int32, device="cuda")
    fm.flint_moe_router(m.h, 0, x, T, None, idx, None)
    torch.cuda.synchronize()
    m.close()
    rows = np.arange(T) if sample is None else np.asarray(sample)
    ref = M.moe_layer(bits[rows], L, act_quant=True)
    same = compare_routing(idx.cpu().numpy()[rows], ref.sel, ref.logits, cfg.top_k)
    assert same.mean() >= 0.95
    return plan, got[rows][same], ref.out[same], ref, bits[rows][same], L


def _flint(**kw):
    return dataclasses.replace(synth.CONFIGS[5], **kw)


@pytest.mark.parametrize("T,bias", [(65, "zipf"), (300, "none"), (1000, "zipf")])
def test_prefill_fp4_layer(fm, T, bias):
    """Ragged expert groups (many experts with one or two rows, a few with
    several 128-row tiles), full comparison of every token."""
    cfg = _flint(bias=bias, tokens=T)
    plan, got, want, _, _, _ = _prefill_parity(fm, cfg, T)
    assert plan & 2, "the FP4 expert path was not selected"
    assert_out_close(got, want, f"FP4 prefill T={T} bias={bias}")


def test_prefill_fp4_T8192_sampled(fm):
    """The full prefill workload; sampled tokens against the oracle, and the
    quantised-activation result must be measurably different from the exact
    (16-bit activation) product, so the comparison above is not vacuous."""
    cfg = _flint()
    rng = np.random.default_rng(0)
    sample = np.unique(np.concatenate([[0, 1, 8191], rng.choice(8192, 61, replace=False)]))
    plan, got, want, ref, bits, L = _prefill_parity(fm, cfg, 8192, sample=sample)
    assert plan == 3, plan
    assert_out_close(got, want, "FP4 prefill T=8192 (sampled tokens)")
    exact = M.moe_layer(bits, L).out
    rel = np.linalg.norm(F.bf16_array(got) - exact) / np.linalg.norm(exact)
    assert rel > 2e-2, f"W4A4 result within {rel:.2e} of the W4A16 product"


def test_prefill_fp4_small_T_inside_large_handle(fm):
    """A handle sized for 8192 tokens serves a 65-token call on the FP4 path
    (the workspace is carved for the handle's maximum, used for fewer)."""
    cfg = _flint(tokens=65)
    plan, got, want, _, _, _ = _prefill_parity(fm, cfg, 65, max_tokens=8192)
    assert plan & 2
    assert_out_close(got, want, "FP4 prefill T=65 in an 8192-token handle")


def test_prefill_fp4_not_selected_for_q4_1_or_other_shapes(fm):
    for cfg, T in [(_flint(wfmt=synth.WFMT_Q4_1), 128), (synth.CONFIGS[1], 128)]:
        m = fm.MoE(cfg, max_tokens=T, n_layers=1)
        m.load(0, synth.make_layer(cfg))
        assert fm.flint_moe_tensor_core_plan(m.h, 0, T) & 2 == 0
        assert fm.flint_moe_tensor_core_plan(m.h, 0, 64) == 0
        m.close()


def test_prefill_fp4_deterministic_and_stack_residual(fm):
    """The FP4 path sums each token's contributions in a fixed order, so two
    forwards agree bit for bit, and forward_stack adds the residual exactly
    as x1 = bf16(x0 + bf16(layer(x0)))."""
    cfg = _flint(tokens=200)
    L = synth.make_layer(cfg)
    bits = synth.make_hidden(cfg, tokens=200)
    m = fm.MoE(cfg, max_tokens=200, n_layers=1)
    m.load(0, L)
    x = fm.hidden_to_device(bits)
    single = fm.hidden_to_host(m.forward(x, 0))
    again = fm.hidden_to_host(m.forward(x, 0))
    assert np.array_equal(single, again)
    fm.flint_moe_forward_stack(m.h, 0, 1, x, 200, None)
    torch.cuda.synchronize()
    assert fm.flint_moe_status(m.h) == fm.FLINT_OK
    stacked = fm.hidden_to_host(x)
    m.close()
    want = F.bf16_bits(F.bf16_round(F.bf16_array(bits) + F.bf16_array(single)))
    assert np.array_equal(stacked, want)
