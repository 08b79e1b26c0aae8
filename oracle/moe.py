"""Plain CPU oracle of the Flint-shaped sparse MoE FFN layer (float64).

TEST INFRASTRUCTURE. Only the test suite, the smoke check and the benchmark's
CPU-baseline leg may import this module. It shares no code with the CUDA path.

What the layer computes. The Flint blog ("Recursive Flint 40B-A2.5B", section
"The architecture is an argument about memory bandwidth", Sparsity and Active
parameters bullets) fixes the structure: 256 routed experts per MoE layer, 6
chosen per token, one always-on shared expert, 47 MoE layers out of 49. It
names 4-bit NVFP4 and q4_1 weights (section "What actually shipped") and says
decode streams weights. It gives no formulas; the readings used here are:

  a1  logits   L[t, e] = sum_i x[t, i] * W_r[e, i] + b[e]
  a2  routing  S_t = the 6 experts with the largest float32 logits (equal
               logits: lower expert index first), listed by descending logit;
               p = softmax(L[t, :]); w[t, j] = p[S_t[j]] / sum_{e in S_t} p[e]
  a3  buckets  counts per expert, exclusive offsets, and the stable order of
               the flat assignments a = t*6 + j by (expert, a)
  a4  weights  NVFP4 or q4_1 dequantisation (see formats.py)
  a5  gate/up  h = silu(W_gate x) * (W_up x), silu(z) = z / (1 + exp(-z))
  a6  down     y_e = W_down h
  a7  shared   the same expert function with the shared weights, weight 1
  a8  combine  out[t] = bf16( y_shared[t] + sum_j w[t, j] * y_{S_t[j]}[t] )
  stack        x_{l+1} = bf16( x_l + out_l )

Float arithmetic is float64 (exact for the dequantised weights). Two decisions
turn floats into integers and are taken in float32, the precision of the
kernels: the top-6 selection (on the float32-rounded logits) and, in the
activation-quantisation mode used for FP4 tensor-core prefill, the choice of
FP4 codes and E4M3 block scales.
"""
from __future__ import annotations

import dataclasses

import numpy as np

from . import formats as F

# ---------------------------------------------------------------------------
# a1: router logits
# ---------------------------------------------------------------------------


def router_logits(x: np.ndarray, w_router: np.ndarray, bias: np.ndarray | None) -> np.ndarray:
    """float64 [T, E] = x [T, d] . W_r[E, d]^T (+ b[E])."""
    x = np.asarray(x, dtype=np.float64)
    L = x @ np.asarray(w_router, dtype=np.float64).T
    if bias is not None:
        L = L + np.asarray(bias, dtype=np.float64)[None, :]
    return L


# ---------------------------------------------------------------------------
# a2: softmax -> top-k -> renormalise
# ---------------------------------------------------------------------------


def select_topk(logits32: np.ndarray, k: int) -> np.ndarray:
    """int32 [T, k]: per token the k experts with the largest float32 logits,
    by descending logit then ascending expert index."""
    L = np.asarray(logits32, dtype=np.float32)
    if not np.all(np.isfinite(L)):
        raise ValueError("non-finite router logit")
    T, E = L.shape
    order = np.empty((T, E), dtype=np.int64)
    idx = np.arange(E)
    for t in range(T):
        # lexsort: last key is primary -> sort by -L, then by index
        order[t] = np.lexsort((idx, -L[t].astype(np.float64)))
    return order[:, :k].astype(np.int32)


def route_weights(logits: np.ndarray, sel: np.ndarray) -> np.ndarray:
    """float64 [T, k]: softmax over all experts, then renormalised over the
    selected ones."""
    L = np.asarray(logits, dtype=np.float64)
    p = np.exp(L - L.max(axis=1, keepdims=True))
    p = p / p.sum(axis=1, keepdims=True)
    ps = np.take_along_axis(p, np.asarray(sel, dtype=np.int64), axis=1)
    return ps / ps.sum(axis=1, keepdims=True)


# ---------------------------------------------------------------------------
# a3: bucketing
# ---------------------------------------------------------------------------


@dataclasses.dataclass
class Buckets:
    counts: np.ndarray   # int32 [E]
    offsets: np.ndarray  # int32 [E+1], exclusive prefix sum of counts
    perm: np.ndarray     # int32 [T*k]: sorted position -> flat assignment a = t*k + j


def bucket(sel: np.ndarray, n_experts: int) -> Buckets:
    e = np.asarray(sel, dtype=np.int64).reshape(-1)
    a = np.arange(e.size)
    perm = np.lexsort((a, e))            # primary key expert, then assignment index
    counts = np.bincount(e, minlength=n_experts)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    return Buckets(counts.astype(np.int32), offsets.astype(np.int32), perm.astype(np.int32))


# ---------------------------------------------------------------------------
# a4-a7: experts
# ---------------------------------------------------------------------------


def silu(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def dequant_matrix(layer, expert: int, mat: int) -> np.ndarray:
    """float64 [R, K] weights of one matrix of one expert (E = shared)."""
    codes, sc, ts = layer.matrix(expert, mat)
    if layer.cfg.wfmt == 0:
        return F.dequant_nvfp4(codes, sc, ts)
    return F.dequant_q41(codes, sc)


def expert_forward(wg: np.ndarray, wu: np.ndarray, wd: np.ndarray, x: np.ndarray) -> np.ndarray:
    """SwiGLU expert on rows of x: y = W_down (silu(W_gate x) * (W_up x))."""
    g = x @ wg.T
    u = x @ wu.T
    h = silu(g) * u
    return h @ wd.T


# ---------------------------------------------------------------------------
# activation quantisation (FP4 tensor-core mode)
# ---------------------------------------------------------------------------


def quant_act_nvfp4(v: np.ndarray):
    """Quantise rows of v to NVFP4 with a per-row float32 scale.

    All decisions are taken in float32, the precision of the kernels:
      s_t  = amax_t / 2688                     (2688 = 6 * 448), float32
      sb_b = E4M3_rne( (amax_b / 6) / s_t )    per 16 consecutive elements
      S_b  = E4M3(sb_b) * s_t                  float32
      r_b  = 1 / S_b                           float32
      code = E2M1_rne( v * r_b )               ties to even, saturating at 6
    A row with amax 0, or a block with S_b == 0, gets all codes 0 and scale 0.
    Returns (codes uint8 [T, K], block scale bytes uint8 [T, K/16],
             row scales float32 [T], dequantised values float64 [T, K]).
    """
    v = np.asarray(v, dtype=np.float32)
    T, K = v.shape
    amax_t = np.abs(v).max(axis=1)
    s_t = (amax_t / np.float32(2688.0)).astype(np.float32)
    blocks = v.reshape(T, K // 16, 16)
    amax_b = np.abs(blocks).max(axis=2)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = ((amax_b / np.float32(6.0)).astype(np.float32) / s_t[:, None]).astype(np.float32)
    ratio = np.where(s_t[:, None] > 0, ratio, np.float32(0.0))
    sb = F.e4m3_encode_rne_nonneg(ratio)
    S = (F.E4M3_TABLE[sb].astype(np.float32) * s_t[:, None]).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        inv = (np.float32(1.0) / S).astype(np.float32)
        r = (blocks * inv[:, :, None]).astype(np.float32)
    r = np.where(S[:, :, None] > 0, r, np.float32(0.0))
    codes = F.e2m1_encode_rne(r)
    codes = np.where(S[:, :, None] > 0, codes, 0).astype(np.uint8)
    deq = (F.E2M1_TABLE[codes] * F.E4M3_TABLE[sb][:, :, None]
           * s_t.astype(np.float64)[:, None, None])
    return codes.reshape(T, K), sb, s_t, deq.reshape(T, K)


def quant_weight_nvfp4(w: np.ndarray):
    """Quantise one weight matrix [R, K] (float32 values, e.g. of bf16
    weights) to NVFP4 with one float32 tensor scale for the whole matrix.

    The pages ship NVFP4 weights ("Flint", the NVFP4 GGUF build) and give no
    quantisation procedure; the reading is the activation rule with the
    per-row scale replaced by the per-tensor one that NVFP4 weights carry, all
    decisions in float32:
      s    = amax(|w|) / 2688                   (2688 = 6 * 448), float32
      sb_b = E4M3_rne( (amax_b / 6) / s )       per 16 consecutive elements of a row
      S_b  = E4M3(sb_b) * s,  r_b = 1 / S_b     float32
      code = E2M1_rne( w * r_b )                ties to even, saturating at 6
    An all-zero matrix, or a block with S_b == 0, gets codes 0 and scale 0.
    Returns (codes uint8 [R, K] one code per element, scale bytes uint8
    [R, K/16], tensor scale float32, dequantised values float64 [R, K])."""
    v = np.asarray(w, dtype=np.float32)
    R, K = v.shape
    s = np.float32(np.abs(v).max() / np.float32(2688.0)) if v.size else np.float32(0.0)
    blocks = v.reshape(R, K // 16, 16)
    amax_b = np.abs(blocks).max(axis=2)
    if s > 0:
        ratio = ((amax_b / np.float32(6.0)).astype(np.float32) / s).astype(np.float32)
    else:
        ratio = np.zeros_like(amax_b, dtype=np.float32)
    sb = F.e4m3_encode_rne_nonneg(ratio)
    S = (F.E4M3_TABLE[sb].astype(np.float32) * s).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        inv = (np.float32(1.0) / S).astype(np.float32)
        r = (blocks * inv[:, :, None]).astype(np.float32)
    r = np.where(S[:, :, None] > 0, r, np.float32(0.0))
    codes = F.e2m1_encode_rne(r)
    codes = np.where(S[:, :, None] > 0, codes, 0).astype(np.uint8)
    deq = F.E2M1_TABLE[codes] * F.E4M3_TABLE[sb][:, :, None] * float(s)
    return codes.reshape(R, K), sb, s, deq.reshape(R, K)


def expert_forward_w4a4(wg, wu, wd, x: np.ndarray) -> np.ndarray:
    """Expert with NVFP4-quantised activations entering each projection.

    The pages fix NVFP4 for the weights only ("Flint", the list of the
    repository's builds); quantising the activations is the reading that the
    FP4 x FP4 tensor-core product needs. Each projection input is quantised
    straight from its value: x as given (bf16), and h = silu(g) * u as
    computed, with its quantisation decisions taken on float32 h like every
    other decision here.
    """
    xq = quant_act_nvfp4(x)[3]
    g = xq @ wg.T
    u = xq @ wu.T
    h = silu(g) * u
    hq = quant_act_nvfp4(h.astype(np.float32))[3]
    return hq @ wd.T


# ---------------------------------------------------------------------------
# a8: layer and stack
# ---------------------------------------------------------------------------


@dataclasses.dataclass
class LayerResult:
    logits: np.ndarray    # float64 [T, E]
    sel: np.ndarray       # int32 [T, k]
    weights: np.ndarray   # float64 [T, k]
    out: np.ndarray       # float64 [T, d] before the bf16 rounding
    out_bf16: np.ndarray  # float64 [T, d], bfloat16 values


def moe_layer(x_bf16_bits: np.ndarray, layer, act_quant: bool = False,
              zero_routed: bool = False) -> LayerResult:
    """One MoE layer on bf16 hidden states (uint16 bit patterns [T, d]).

    act_quant: NVFP4-quantise the activations entering each expert projection
    (the FP4 tensor-core prefill mode). zero_routed: drop every routed
    expert's contribution (used by a check, not by the layer).
    """
    cfg = layer.cfg
    x = F.bf16_array(x_bf16_bits)
    T = x.shape[0]
    L = router_logits(x, layer.router, layer.router_bias)
    sel = select_topk(L.astype(np.float32), cfg.top_k)
    w = route_weights(L, sel)
    fwd = expert_forward_w4a4 if act_quant else expert_forward

    def expert_weights(e):
        return tuple(dequant_matrix(layer, e, m) for m in range(3))

    out = fwd(*expert_weights(cfg.n_experts), x)          # a7: shared expert, weight 1
    contrib = np.zeros((T, cfg.top_k, cfg.d))
    if not zero_routed:
        for e in np.unique(sel):
            rows, slots = np.nonzero(sel == e)
            contrib[rows, slots] = fwd(*expert_weights(int(e)), x[rows])
    for j in range(cfg.top_k):                             # a8: slot order
        out = out + w[:, j:j + 1] * contrib[:, j]
    return LayerResult(L, sel, w, out, F.bf16_round(out))


def moe_stack(x_bf16_bits: np.ndarray, layers) -> tuple[np.ndarray, list]:
    """Decode stack: x_{l+1} = bf16(x_l + out_l); returns (final bits, per-layer results)."""
    bits = np.asarray(x_bf16_bits, dtype=np.uint16)
    results = []
    for layer in layers:
        r = moe_layer(bits, layer)
        results.append(r)
        nxt = F.bf16_round(F.bf16_array(bits) + r.out_bf16)
        bits = F.bf16_bits(nxt)
    return bits, results
