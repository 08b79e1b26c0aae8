"""Plain CPU oracle of the 4-bit output head and its sampling front-end (float64).

TEST INFRASTRUCTURE. Only the test suite and the benchmark's CPU-baseline leg
may import this module. It shares no code with the CUDA path.

What it computes. The Flint blog ("Recursive Flint 40B-A2.5B") says the
output layer, lm_head, ships quantised to 4 bits because with ~2.5B active
parameters per token it is a large share of the bytes read per token
(section "The quantisation recipe is the most transferable part"); the model
is NVFP4 (section "What actually shipped"). Its evaluation and serving
defaults are temperature 1.0, top-p 0.95 and top-k 20 (section "The three
scores, and the footnotes that come with them", Sampling bullet). It gives no
formulas; the readings used here are:

  head    logits[t, v] = sum_i x[t, i] * W[v, i], W the NVFP4 head [V x d]
          (E2M1 code x E4M3 scale per 16 along d x fp32 tensor scale)
  sample  per token, on the float32 logits:
          temperature <= 0  -> the largest logit (equal logits: lower index)
          otherwise
            S   = the top_k indices by descending logit, then ascending index
            p_j = exp((l[S_j] - l[S_0]) / temperature), normalised over S
            m   = the number of leading j whose exclusive cumulative sum
                  sum_{i<j} p_i is below top_p (at least 1): the smallest
                  prefix of S whose probability reaches top_p
            Z   = sum_{j<m} p_j
            token = S_r, r the first j < m with sum_{i<=j} p_i > u * Z
                  (r = m - 1 if rounding leaves none), u in [0, 1) drawn by
                  the caller
          Top-k is applied before top-p, and the draw is an inverse CDF of
          the kept, renormalised probabilities.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from . import formats as F


def head_logits(x_bf16_bits: np.ndarray, codes: np.ndarray, scales: np.ndarray, tensor_scale: float) -> np.ndarray:
    """float64 [T, V] = x [T, d] . W[V, d]^T, with W dequantised exactly."""
    x = F.bf16_array(np.asarray(x_bf16_bits, dtype=np.uint16)).astype(np.float64)
    W = F.dequant_nvfp4(codes, scales, tensor_scale)
    return x @ W.T


@dataclasses.dataclass
class Draw:
    token: int
    sel: np.ndarray        # int64 [k]: the top-k indices, descending logit
    p: np.ndarray          # float64 [k]: their normalised probabilities
    kept: int              # m: how many of them survive top-p
    cdf: np.ndarray        # float64 [m]: sum_{i<=j} p_i / Z, the draw's boundaries


def top_indices(logits32: np.ndarray, k: int) -> np.ndarray:
    """The k largest float32 logits of one token: descending value, ties by
    ascending index."""
    L = np.asarray(logits32, dtype=np.float32).astype(np.float64)
    order = np.lexsort((np.arange(L.size), -L))
    return order[:k]


def sample_token(logits32: np.ndarray, temperature: float, top_k: int, top_p: float, u: float) -> Draw:
    """One token's draw (see the module docstring)."""
    L = np.asarray(logits32, dtype=np.float32).astype(np.float64)
    if temperature <= 0.0:
        sel = top_indices(L, 1)
        return Draw(int(sel[0]), sel, np.ones(1), 1, np.ones(1))
    k = min(int(top_k), L.size)
    sel = top_indices(L, k)
    e = np.exp((L[sel] - L[sel[0]]) / float(temperature))
    p = e / e.sum()
    m = 0
    run = 0.0
    while m < k and (m == 0 or run < top_p):
        run += p[m]
        m += 1
    cum = np.cumsum(p[:m])
    Z = cum[-1]
    r = m - 1
    for j in range(m):
        if cum[j] > u * Z:
            r = j
            break
    return Draw(int(sel[r]), sel, p, m, cum / Z)


def sample(logits32: np.ndarray, temperature: float, top_k: int, top_p: float, u: np.ndarray) -> list[Draw]:
    """Draws for every token of a [T, V] logits array, u [T]."""
    L = np.asarray(logits32, dtype=np.float32)
    return [sample_token(L[t], temperature, top_k, top_p, float(u[t])) for t in range(L.shape[0])]
