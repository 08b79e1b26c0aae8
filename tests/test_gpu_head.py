"""The 4-bit output head and its sampler on the GPU against the oracle.

Logits: the head decodes weights to fp16 exactly and rounds x to fp16 after a
power-of-two scale per token (relative error <= 2^-11 per element), then
accumulates in fp32; a logit's error is then ~2^-11 of the typical logit
magnitude, so the bar below (relative L2 <= 2e-3, max abs <= 1e-2 x RMS) has
a margin of about 4. The sampler is checked on the GPU's own fp32 logits (the
same input on both sides): the top-k indices exactly, and the drawn token
exactly unless u lies within 1e-5 of one of the draw's boundaries (the oracle
sums in float64, the kernel in float32).
"""
import numpy as np
import pytest

from bit_quantized_expert_softmax_b300 import synth
from oracle import lm_head as H

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


def _handle(fm, d):
    cfg = synth.LayerConfig(d=d, f=128, tokens=8, name="head_host")
    return fm.MoE(cfg, max_tokens=8)


def _gpu_logits(fm, hcfg, T, seed=0):
    hw = synth.make_head(hcfg, seed=seed)
    x = synth.make_hidden(hcfg, tokens=T, seed=seed)
    m = _handle(fm, hcfg.d)
    fm.flint_moe_load_lm_head(m.h, hw.codes, hw.scales, hw.tensor_scale)
    xd = fm.hidden_to_device(x)
    logits = torch.full((T, hcfg.vocab), float("nan"), dtype=torch.float32, device="cuda")
    fm.flint_moe_lm_head(m.h, xd, T, logits)
    torch.cuda.synchronize()
    assert fm.flint_moe_status(m.h) == fm.FLINT_OK
    return m, hw, x, logits


def _assert_logits_close(got, ref, what):
    got = np.asarray(got, dtype=np.float64)
    assert np.all(np.isfinite(got)), f"{what}: non-finite logits"
    rms = float(np.sqrt(np.mean(ref ** 2)))
    rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    mx = float(np.max(np.abs(got - ref)))
    assert rel <= 2e-3 and mx <= 1e-2 * rms, f"{what}: rel L2 {rel:.2e}, max abs {mx:.3e} (rms {rms:.3e})"


@pytest.mark.parametrize("d,V,T", [(512, 1000, 3), (2048, 2048, 1), (2048, 1024, 8), (1024, 8, 2), (640, 136, 5)])
def test_head_logits_match_oracle(fm, d, V, T):
    """Several units per warp, a ragged vocabulary (not a multiple of the
    grid's warps), one unit in all, every token count up to 8, and a width of
    5 k-tiles (one partial register chunk)."""
    hcfg = synth.HeadConfig(d=d, vocab=V, tokens=T, seed=d + V)
    m, hw, x, logits = _gpu_logits(fm, hcfg, T, seed=hcfg.seed)
    ref = H.head_logits(x, hw.codes, hw.scales, hw.tensor_scale)
    _assert_logits_close(logits.cpu().numpy(), ref, f"d={d} V={V} T={T}")
    again = torch.empty_like(logits)
    fm.flint_moe_lm_head(m.h, fm.hidden_to_device(x), T, again)
    torch.cuda.synchronize()
    assert torch.equal(logits, again), "head logits not deterministic"
    m.close()


def test_head_flint_size_sampled_rows(fm):
    """The full Flint-sized head (146,432 x 2048), one token; rows sampled
    across the vocabulary (first, last, and random) against the oracle."""
    hcfg = synth.HEAD_CONFIGS["flint"]
    m, hw, x, logits = _gpu_logits(fm, hcfg, 1)
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, 1, 7, 8, hcfg.vocab - 1], rng.choice(hcfg.vocab, 2000, replace=False)]))
    ref = H.head_logits(x, hw.codes[rows], hw.scales[rows], hw.tensor_scale)
    _assert_logits_close(logits.cpu().numpy()[:, rows], ref, "Flint head, sampled rows")
    m.close()


def _check_draws(fm, m, logits, temperature, top_k, top_p, u):
    T, V = logits.shape
    ud = torch.from_numpy(u).cuda()
    tokens = torch.full((T,), -1, dtype=torch.int32, device="cuda")
    topk = torch.full((T, top_k), -1, dtype=torch.int32, device="cuda")
    fm.flint_moe_sample(m.h, logits, T, temperature, top_k, top_p, ud, tokens, topk)
    torch.cuda.synchronize()
    assert fm.flint_moe_status(m.h) == fm.FLINT_OK
    L = logits.cpu().numpy()
    got_tok = tokens.cpu().numpy()
    got_sel = topk.cpu().numpy()
    for t in range(T):
        d = H.sample_token(L[t], temperature, top_k, top_p, float(u[t]))
        k = len(d.sel)
        assert list(got_sel[t, :k]) == list(d.sel), f"top-k differs for token {t}"
        if got_tok[t] != d.token:
            near = np.min(np.abs(d.cdf - u[t])) <= 1e-5 if d.kept > 1 else False
            excl = np.cumsum(np.concatenate([[0.0], d.p]))[:k]
            near = near or np.min(np.abs(excl - top_p)) <= 1e-5
            assert near, f"token {t}: drew {got_tok[t]}, oracle {d.token} (u {u[t]})"


@pytest.mark.parametrize("temperature,top_k,top_p", [(1.0, 20, 0.95), (0.7, 20, 0.5), (1.0, 32, 1.0),
                                                     (2.0, 5, 0.9), (1.0, 1, 0.95), (0.0, 20, 0.95)])
def test_sampler_matches_oracle_on_the_gpu_logits(fm, temperature, top_k, top_p):
    hcfg = synth.HeadConfig(d=512, vocab=5000, tokens=8, seed=11)
    m, hw, x, logits = _gpu_logits(fm, hcfg, 8, seed=hcfg.seed)
    for rep in range(4):
        u = synth.make_uniforms(8, seed=rep, stream=int(temperature * 10) + top_k)
        _check_draws(fm, m, logits, temperature, top_k, top_p, u)
    m.close()


def test_sampler_flint_size_and_defaults(fm):
    """The Flint-sized vocabulary (72 parts merged) at the serving defaults."""
    hcfg = synth.HEAD_CONFIGS["flint"]
    m, hw, x, logits = _gpu_logits(fm, hcfg, 1)
    for rep in range(8):
        _check_draws(fm, m, logits, 1.0, 20, 0.95, synth.make_uniforms(1, seed=rep))
    m.close()


def test_sampler_ties_lower_index_and_nan_last(fm):
    """Equal logits rank by index; a NaN logit ranks last and is reported."""
    hcfg = synth.HeadConfig(d=512, vocab=4096, tokens=2, seed=12)
    m, hw, x, logits = _gpu_logits(fm, hcfg, 2, seed=hcfg.seed)
    L = torch.full((2, 4096), -5.0, dtype=torch.float32, device="cuda")
    L[0, 3000] = 7.0
    L[0, 100] = 7.0           # tie with 3000: 100 first
    L[0, 2049] = 6.5          # a second part
    L[1, 5] = float("nan")
    L[1, 4095] = 1.0
    u = np.array([0.0, 0.0], dtype=np.float32)
    ud = torch.from_numpy(u).cuda()
    tokens = torch.full((2,), -1, dtype=torch.int32, device="cuda")
    topk = torch.full((2, 3), -1, dtype=torch.int32, device="cuda")
    fm.flint_moe_sample(m.h, L, 2, 1.0, 3, 1.0, ud, tokens, topk)
    torch.cuda.synchronize()
    assert fm.flint_moe_status(m.h) == fm.FLINT_EDEVICE
    sel = topk.cpu().numpy()
    assert list(sel[0]) == [100, 3000, 2049]
    assert sel[1, 0] == 4095 and 5 not in list(sel[1])
    assert tokens.cpu().numpy()[0] == 100
    m.close()


def test_head_rejects_bad_calls(fm):
    m = _handle(fm, 512)
    x = torch.zeros((9, 512), dtype=torch.bfloat16, device="cuda")
    lg = torch.zeros((9, 1000), dtype=torch.float32, device="cuda")
    L = fm.lib()
    assert L.flint_moe_lm_head(m.h, x.data_ptr(), 1, lg.data_ptr(), None) == fm.FLINT_ESTATE
    hw = synth.make_head(synth.HeadConfig(d=512, vocab=1000))
    with pytest.raises(fm.FlintError):
        fm.flint_moe_load_lm_head(m.h, hw.codes[:999], hw.scales[:999], hw.tensor_scale)   # not a multiple of 8
    fm.flint_moe_load_lm_head(m.h, hw.codes, hw.scales, hw.tensor_scale)
    assert L.flint_moe_lm_head(m.h, x.data_ptr(), 9, lg.data_ptr(), None) == fm.FLINT_EINVAL
    u = torch.zeros((9,), dtype=torch.float32, device="cuda")
    tok = torch.zeros((9,), dtype=torch.int32, device="cuda")
    for T, temp, k, p in [(1, 1.0, 33, 0.9), (1, 1.0, 0, 0.9), (1, 1.0, 20, 0.0), (1, 1.0, 20, 1.5),
                          (9, 1.0, 20, 0.9)]:
        assert L.flint_moe_sample(m.h, lg.data_ptr(), T, temp, k, p, u.data_ptr(), tok.data_ptr(), None,
                                  None) == fm.FLINT_EINVAL
    m.close()
