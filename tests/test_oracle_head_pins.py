"""Pins of the output-head oracle and its sampler against facts that do not
come from the oracle itself: brute force on tiny inputs, hand-worked draws,
and properties of an inverse-CDF sampler (frequencies, temperature scaling,
the greedy limit)."""
import math

import numpy as np
import pytest

from bit_quantized_expert_softmax_b300 import synth
from oracle import formats as F
from oracle import lm_head as H
from tests.conftest import read_golden


def test_head_logits_brute_force():
    """Scalar decode of every code and scale byte, summed in Python."""
    cfg = synth.HeadConfig(d=32, vocab=8, tokens=2, seed=3)
    hw = synth.make_head(cfg)
    x = synth.make_hidden(cfg)
    got = H.head_logits(x, hw.codes, hw.scales, hw.tensor_scale)
    ts = float(hw.tensor_scale)
    for t in range(cfg.tokens):
        xv = [F.bf16_value(int(b)) for b in x[t]]
        for v in range(cfg.vocab):
            s = 0.0
            for i in range(cfg.d):
                byte = int(hw.codes[v, i // 2])
                code = byte & 0xF if i % 2 == 0 else byte >> 4
                w = F.e2m1_value(code) * F.e4m3_value(int(hw.scales[v, i // 16])) * ts
                s += w * xv[i]
            assert got[t, v] == pytest.approx(s, rel=1e-12, abs=1e-12)


def test_head_logits_rows_and_tokens_not_transposed():
    """Changing one weight row changes only that vocabulary entry; changing
    one token changes only that token's row of logits."""
    cfg = synth.HeadConfig(d=64, vocab=16, tokens=3, seed=4)
    hw = synth.make_head(cfg)
    x = synth.make_hidden(cfg)
    base = H.head_logits(x, hw.codes, hw.scales, hw.tensor_scale)
    codes = hw.codes.copy()
    codes[5] ^= 0x11
    alt = H.head_logits(x, codes, hw.scales, hw.tensor_scale)
    changed = np.nonzero(np.any(alt != base, axis=0))[0]
    assert list(changed) == [5]
    x2 = x.copy()
    x2[1] ^= 0x0001
    alt = H.head_logits(x2, hw.codes, hw.scales, hw.tensor_scale)
    assert list(np.nonzero(np.any(alt != base, axis=1))[0]) == [1]


def _golden_draws():
    rows = []
    for r in read_golden("sampler_examples.txt"):
        f = [c for c in r if c != "|"]
        rows.append((np.array([float(v) for v in f[0].split(",")], dtype=np.float32), float(f[1]), int(f[2]),
                     float(f[3]), float(f[4]), int(f[5]), int(f[6])))
    return rows


@pytest.mark.parametrize("row", _golden_draws())
def test_sampler_hand_worked_draws(row):
    logits, tau, k, top_p, u, token, kept = row
    d = H.sample_token(logits, tau, k, top_p, u)
    assert d.token == token
    assert d.kept == kept


def test_sampler_first_boundary_is_the_logistic():
    """Two kept candidates whose logits differ by delta: the first boundary is
    1 / (1 + e^(-delta / temperature))."""
    for delta, tau in [(1.0, 1.0), (0.5, 0.7), (3.0, 2.0)]:
        d = H.sample_token(np.array([delta, 0.0, -50.0], dtype=np.float32), tau, 2, 1.0, 0.0)
        assert d.cdf[0] == pytest.approx(1.0 / (1.0 + math.exp(-delta / tau)), rel=1e-6)


def test_sampler_frequencies_follow_the_softmax():
    """With top-k and top-p not cutting, the draws over a fine grid of u hit
    each token with its softmax probability (to the grid's resolution)."""
    rng = np.random.default_rng(7)
    logits = rng.standard_normal(6).astype(np.float32) * 2
    tau = 1.3
    n = 20000
    us = (np.arange(n) + 0.5) / n
    counts = np.zeros(6)
    for u in us:
        counts[H.sample_token(logits, tau, 6, 1.0, u).token] += 1
    z = np.exp(logits.astype(np.float64) / tau)
    want = z / z.sum()
    assert np.max(np.abs(counts / n - want)) <= 2.0 / n


def test_sampler_top_p_keeps_the_smallest_prefix_reaching_p():
    rng = np.random.default_rng(8)
    for _ in range(50):
        logits = rng.standard_normal(30).astype(np.float32) * 3
        top_p = float(rng.uniform(0.05, 1.0))
        d = H.sample_token(logits, 1.0, 20, top_p, 0.3)
        # the kept prefix reaches top_p, and dropping its last member would not
        assert d.p[:d.kept].sum() >= top_p or d.kept == 20
        assert d.kept == 1 or d.p[:d.kept - 1].sum() < top_p
        # the top-20 are the 20 largest logits by value then index
        order = sorted(range(30), key=lambda i: (-float(logits[i]), i))[:20]
        assert list(d.sel) == order


def test_sampler_temperature_scales_the_logits():
    """Temperature tau on logits l draws like temperature 1 on l / tau
    (halving is exact in float32)."""
    rng = np.random.default_rng(9)
    logits = rng.standard_normal(40).astype(np.float32) * 4
    for u in np.linspace(0.0, 0.999, 37):
        a = H.sample_token(logits, 2.0, 20, 0.95, u)
        b = H.sample_token(logits / np.float32(2.0), 1.0, 20, 0.95, u)
        assert a.token == b.token and a.kept == b.kept


def test_sampler_greedy_is_the_cold_limit():
    rng = np.random.default_rng(10)
    for _ in range(20):
        logits = rng.standard_normal(100).astype(np.float32)
        g = H.sample_token(logits, 0.0, 20, 0.95, 0.5).token
        assert g == int(np.argmax(logits))
        assert H.sample_token(logits, 1e-4, 20, 0.95, 0.999).token == g
