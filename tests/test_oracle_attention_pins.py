"""Pins of the decode-attention oracle (oracle/attention.py) against closed
forms and invariants: the RMS of a normalised head, rotation properties of
the position embedding, the logistic closed form of a one-key attention with
a sink, the plain softmax attention it reduces to without a sink, the window
and the query-to-key-head grouping."""
import math

import numpy as np
import pytest

from oracle import attention as A
from oracle import formats as F


def test_rms_norm_has_unit_rms_and_ignores_scale():
    rng = np.random.default_rng(1)
    v = rng.standard_normal((5, 128)) * 3.0
    n = A.rms_norm(v, np.ones(128), eps=0.0)
    assert np.allclose(np.sqrt(np.mean(n * n, axis=1)), 1.0, rtol=1e-12)
    assert np.allclose(A.rms_norm(7.5 * v, np.ones(128), eps=0.0), n, rtol=1e-12)
    w = rng.standard_normal(128)
    assert np.allclose(A.rms_norm(v, w, eps=0.0), n * w, rtol=1e-12)


def test_rope_is_a_rotation_with_relative_positions():
    rng = np.random.default_rng(2)
    q, k = rng.standard_normal(128), rng.standard_normal(128)
    assert np.allclose(A.rope(q, 0), q)
    for pos in (1, 17, 1000):
        assert math.isclose(np.linalg.norm(A.rope(q, pos)), np.linalg.norm(q), rel_tol=1e-12)
    # the score of rotated q at m and k at n depends on m - n only
    for m, n in [(5, 3), (700, 100), (513, 0)]:
        a = A.rope(q, m) @ A.rope(k, n)
        b = A.rope(q, m - n) @ k
        assert math.isclose(a, b, rel_tol=1e-10, abs_tol=1e-10)
    # pair i of the two halves turns by theta^(-i/64) per position
    e = np.zeros(128)
    e[3] = 1.0
    r = A.rope(e, 1)
    ang = A.THETA ** (-3 / 64)
    assert math.isclose(r[3], math.cos(ang), rel_tol=1e-12) and math.isclose(r[67], math.sin(ang), rel_tol=1e-12)


def test_one_key_attention_is_logistic_in_the_sink():
    rng = np.random.default_rng(3)
    q, k, v = rng.standard_normal(128), rng.standard_normal(128), rng.standard_normal(128)
    s = q @ k / math.sqrt(128)
    for sink in (-3.0, 0.0, 2.5):
        got = A.attend(q, k[None, :], v[None, :], sink)
        assert np.allclose(got, v / (1.0 + math.exp(sink - s)), rtol=1e-12)


def test_attention_without_sink_is_softmax_attention():
    rng = np.random.default_rng(4)
    q = rng.standard_normal(128)
    keys, vals = rng.standard_normal((40, 128)), rng.standard_normal((40, 128))
    s = keys @ q / math.sqrt(128)
    p = np.exp(s - s.max())
    want = (p / p.sum()) @ vals
    assert np.allclose(A.attend(q, keys, vals, -1e30), want, rtol=1e-12)


def _step_inputs(seed, cap=600):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((32, 128))
    k = rng.standard_normal((4, 128))
    v = rng.standard_normal((4, 128))
    kc = F.bf16_bits(F.bf16_round(rng.standard_normal((4, cap, 128))))
    vc = F.bf16_bits(F.bf16_round(rng.standard_normal((4, cap, 128))))
    wq, wk = 1 + 0.1 * rng.standard_normal(128), 1 + 0.1 * rng.standard_normal(128)
    sinks = rng.standard_normal(32)
    return q, k, v, kc, vc, wq, wk, sinks


def test_window_covers_exactly_the_last_513_positions():
    q, k, v, kc, vc, wq, wk, sinks = _step_inputs(5)
    pos, cap = 550, kc.shape[1]
    base = A.decode_step(q, k, v, kc, vc, pos, wq, wk, sinks)[0]
    kc2, vc2 = kc.copy(), vc.copy()
    old = pos - 513                                   # just outside: changing it changes nothing
    kc2[:, old % cap] ^= 0x1234
    vc2[:, old % cap] ^= 0x1234
    assert np.array_equal(A.decode_step(q, k, v, kc2, vc2, pos, wq, wk, sinks)[0], base)
    kc3 = kc.copy()
    kc3[:, (pos - 512) % cap] ^= 0x0100                # the oldest position inside the window
    assert not np.allclose(A.decode_step(q, k, v, kc3, vc, pos, wq, wk, sinks)[0], base)
    # full attention (window 0) reads every earlier position
    full = A.decode_step(q, k, v, kc, vc, pos, wq, wk, sinks, window=0, rope_on=False)[0]
    kc4 = kc.copy()
    kc4[:, 0] ^= 0x0100
    assert not np.allclose(A.decode_step(q, k, v, kc4, vc, pos, wq, wk, sinks, window=0, rope_on=False)[0], full)


def test_query_heads_share_key_heads_in_groups_of_eight():
    q, k, v, kc, vc, wq, wk, sinks = _step_inputs(6)
    pos = 20
    base = A.decode_step(q, k, v, kc, vc, pos, wq, wk, sinks)[0]
    v2 = v.copy()
    v2[2] += 1.0                                      # the current value of key head 2 only
    out = A.decode_step(q, k, v2, kc, vc, pos, wq, wk, sinks)[0]
    changed = np.any(out != base, axis=1)
    assert np.array_equal(np.nonzero(changed)[0], np.arange(16, 24))


def test_first_token_attends_to_itself_only():
    q, k, v, kc, vc, wq, wk, sinks = _step_inputs(7)
    out, ks, vs = A.decode_step(q, k, v, kc, vc, 0, wq, wk, sinks)
    for h in range(32):
        g = h // 8
        qh = A.rms_norm(q[h], wq)
        kg = A.rms_norm(k[g], wk)
        s = qh @ kg / math.sqrt(128)                  # position 0: no rotation
        assert np.allclose(out[h], v[g] / (1.0 + math.exp(sinks[h] - s)), rtol=1e-12)
    assert np.array_equal(vs, F.bf16_bits(F.bf16_round(v)))
