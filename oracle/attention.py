"""Plain CPU oracle of one decode step of Flint-shaped attention (float64).

TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's
CPU-baseline leg may import this module. It shares no code with the CUDA path.

The Flint blog ("Recursive Flint 40B-A2.5B", section "The architecture is an
argument about memory bandwidth", Attention and Position-encoding bullets)
fixes the shape: 35 sliding-window layers whose window is 513 tokens (the
current token and the 512 before it) interleaved with 14 full-attention
layers; 32 query heads and 4 key-value heads of dimension 128; rotary
position embeddings on the sliding-window layers and none on the
full-attention layers; per-head QK RMSNorm and learned per-head attention
sinks. It gives no formulas; the readings used here are:

  norm   q_h <- rms(q_h) * w_q, k_g <- rms(k_g) * w_k over the head dimension,
         rms(v) = v / sqrt(mean(v^2) + eps), eps = 1e-6, one weight vector of
         length 128 for all query heads and one for all key heads
  rope   (sliding-window layers) the two halves of a head, (v[i], v[i+64]),
         rotated by the angle pos * theta^(-i/64), theta = 10000
  scores s_j = q_h . k_j / sqrt(128) over the window's keys (key head h // 8)
  sink   the head's learned logit joins the softmax denominator only:
         o_h = sum_j exp(s_j - m) v_j / (sum_j exp(s_j - m) + exp(sink_h - m)),
         m = max(max_j s_j, sink_h)
  cache  keys are stored after norm and rotation, values as projected, both
         bf16; the current token's own key and value enter its attention
         unrounded and are stored rounded
"""
from __future__ import annotations

import math

import numpy as np

from . import formats as F

HEAD_DIM = 128
N_HEADS = 32
N_KV = 4
WINDOW = 513
EPS = 1e-6
THETA = 10000.0


def rms_norm(v: np.ndarray, w: np.ndarray, eps: float = EPS) -> np.ndarray:
    """v / sqrt(mean(v^2) + eps) * w along the last axis (float64)."""
    v = np.asarray(v, dtype=np.float64)
    return v / np.sqrt(np.mean(v * v, axis=-1, keepdims=True) + eps) * np.asarray(w, dtype=np.float64)


def rope(v: np.ndarray, pos: int, theta: float = THETA) -> np.ndarray:
    """Rotate the pairs (v[i], v[i + D/2]) of the last axis by pos * theta^(-2i/D)."""
    v = np.asarray(v, dtype=np.float64)
    D = v.shape[-1]
    half = D // 2
    ang = pos * theta ** (-np.arange(half, dtype=np.float64) / half)
    c, s = np.cos(ang), np.sin(ang)
    a, b = v[..., :half], v[..., half:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


def attend(q: np.ndarray, keys: np.ndarray, vals: np.ndarray, sink: float) -> np.ndarray:
    """One head: softmax over the keys' scores with the sink in the denominator."""
    s = keys @ q / math.sqrt(q.shape[-1])
    m = max(float(s.max()) if s.size else -math.inf, float(sink))
    p = np.exp(s - m)
    return (p @ vals) / (p.sum() + math.exp(float(sink) - m))


def decode_step(q_raw, k_raw, v_new, k_cache_bits, v_cache_bits, pos: int, wq, wk, sinks,
                window: int = WINDOW, rope_on: bool = True, theta: float = THETA):
    """One token of one sequence through one attention layer.

    q_raw [32, 128], k_raw [4, 128], v_new [4, 128]: the projections (float
    values, e.g. of bf16). k_cache_bits / v_cache_bits [4, cap, 128]: bf16 bit
    patterns; position p lives in slot p % cap; slots of positions pos-1,
    pos-2, ... down to the window's start are read. window = 0 means all
    positions 0 .. pos (full attention). Returns (out [32, 128] float64,
    k_store [4, 128] and v_store [4, 128]: the bf16 bit patterns written to
    slot pos % cap)."""
    q = rms_norm(q_raw, wq)
    k = rms_norm(k_raw, wk)
    if rope_on:
        q = rope(q, pos, theta)
        k = rope(k, pos, theta)
    v = np.asarray(v_new, dtype=np.float64)
    cap = k_cache_bits.shape[1]
    first = 0 if window == 0 else max(0, pos - window + 1)
    prev = list(range(first, pos))
    kc = F.bf16_array(k_cache_bits)
    vc = F.bf16_array(v_cache_bits)
    n_h, n_kv = q.shape[0], k.shape[0]
    group = n_h // n_kv
    out = np.zeros((n_h, q.shape[1]))
    for g in range(n_kv):
        keys = np.concatenate([kc[g, [p % cap for p in prev]], k[g][None, :]], axis=0)
        vals = np.concatenate([vc[g, [p % cap for p in prev]], v[g][None, :]], axis=0)
        for h in range(g * group, (g + 1) * group):
            out[h] = attend(q[h], keys, vals, sinks[h])
    return out, F.bf16_bits(F.bf16_round(k)), F.bf16_bits(F.bf16_round(v))
