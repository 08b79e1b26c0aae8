"""Seeded synthetic inputs for the Flint-shaped 4-bit MoE layer.

This module only draws random numbers and packs them into the canonical
(host-side) layouts that ``flint_moe_load_weights`` and ``flint_moe_forward``
accept. It holds none of the layer's arithmetic: it never decodes a code,
never evaluates a weight, router, expert or combine. Both the CPU oracle (in
the tests) and the CUDA path consume exactly the arrays produced here.

Shapes follow the Flint blog ("Recursive Flint 40B-A2.5B", section "The
architecture is an argument about memory bandwidth", Sparsity bullet): 256
routed experts per MoE layer, 6 chosen per token, one always-on shared expert,
47 MoE layers. The hidden width d=2048 and expert width f=512 are the
Flint-shaped sizes (they reproduce the 39.8B total / ~2.2B active body).

Value recipe (all streams are numpy PCG64, seeded through SeedSequence with
the key (seed, layer, stream-id)):

* hidden x ~ N(0, 1) drawn in float32 and truncated to bfloat16 (top 16 bits).
* router W_r ~ N(0, 1/sqrt(d)) float32, shape [E, d] (one row per expert).
* router bias: none, or the Zipf(s=1.1) popularity skew
  b[e] = -1.1 * ln(rank_e) with rank a seeded permutation of 1..E.
* NVFP4 expert weights, drawn directly in the packed domain: E2M1 codes
  uniform over all 16 codes, E4M3 block-scale bytes uniform over 0x28..0x3F
  (0.25 .. 1.875), one fp32 tensor scale per matrix 0.00705 * U(0.75, 1.25).
  The second moment then matches N(0, 0.02) weights.
* q4_1 expert weights: q uniform in 0..15, per block of 32 an fp16
  d = 0.00434 * U(0.8, 1.2) and m = -7.5 * d * U(0.9, 1.1) (weights of mean ~0
  and standard deviation ~0.02).
* The 47-layer decode stack carries the hidden state from layer to layer with
  a residual add and no normalisation. SwiGLU makes an expert's output grow
  quadratically with its input, so with down-projection weights of standard
  deviation 0.02 the residual stream overflows within ~20 layers. The stack
  workload therefore draws its down-projection tensor scales 4x smaller
  (standard deviation ~0.005; `down_scale`), which keeps the hidden RMS
  between 1.0 and 1.2 over all 47 layers. Byte counts are unchanged.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

WFMT_NVFP4 = 0
WFMT_Q4_1 = 1

# stream ids inside one (seed, layer)
_S_ROUTER, _S_BIAS, _S_CODES, _S_SCALES, _S_TSCALE, _S_HIDDEN = range(6)


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    """Shape of one MoE layer and of the workload run through it."""
    d: int
    f: int
    n_experts: int = 256
    top_k: int = 6
    wfmt: int = WFMT_NVFP4
    bias: str = "none"          # "none" | "zipf"
    tokens: int = 1
    n_layers: int = 1
    seed: int = 0
    name: str = ""
    down_scale: float = 1.0     # multiplier of the down-projection weight scale

    @property
    def block(self) -> int:
        return 16 if self.wfmt == WFMT_NVFP4 else 32

    @property
    def scale_bytes_per_block(self) -> int:
        return 1 if self.wfmt == WFMT_NVFP4 else 4

    @property
    def codes_per_matrix(self) -> int:
        """Bytes of packed codes of one [f x d] or [d x f] matrix."""
        return self.f * self.d // 2

    @property
    def scales_per_matrix(self) -> int:
        """Bytes of block scales of one matrix."""
        return self.f * self.d // self.block * self.scale_bytes_per_block

    @property
    def expert_bytes(self) -> int:
        """Bytes of one expert's three packed matrices (codes + block scales + tensor scales)."""
        ts = 4 if self.wfmt == WFMT_NVFP4 else 0
        return 3 * (self.codes_per_matrix + self.scales_per_matrix + ts)

    @property
    def router_bytes(self) -> int:
        return self.n_experts * self.d * 4


# The five workloads of the layer (tiny parity case, single-token decode,
# batched q4_1 decode, 47-layer decode stack, 8192-token prefill chunk).
CONFIGS = {
    1: LayerConfig(d=512, f=128, tokens=4, name="tiny_d512_f128_T4_nvfp4"),
    2: LayerConfig(d=2048, f=512, tokens=1, name="flint_decode_T1_nvfp4"),
    3: LayerConfig(d=2048, f=512, tokens=64, wfmt=WFMT_Q4_1, bias="zipf",
                   name="flint_decode_T64_q4_1_zipf"),
    4: LayerConfig(d=2048, f=512, tokens=1, n_layers=47, down_scale=0.25, name="flint_stack47_T1_nvfp4"),
    5: LayerConfig(d=2048, f=512, tokens=8192, bias="zipf", name="flint_prefill_T8192_nvfp4_zipf"),
}


def _rng(seed: int, layer: int, stream: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, layer, stream])))


@dataclasses.dataclass
class LayerWeights:
    """Canonical host layout of one layer (what flint_moe_load_weights copies).

    router        float32 [E, d]
    router_bias   float32 [E] or None
    codes         uint8   [E+1, 3, f*d/2]   expert E is the shared expert;
                  matrix 0 = gate [f x d], 1 = up [f x d], 2 = down [d x f],
                  each row-major with two 4-bit codes per byte, low nibble first
    scales        uint8   [E+1, 3, f*d/block*bytes_per_block]
                  NVFP4: one E4M3 byte per 16 codes of a row
                  q4_1 : per 32 codes of a row, fp16 d then fp16 m (little endian)
    tensor_scale  float32 [E+1, 3] (NVFP4; all ones for q4_1)
    """
    cfg: LayerConfig
    router: np.ndarray
    router_bias: np.ndarray | None
    codes: np.ndarray
    scales: np.ndarray
    tensor_scale: np.ndarray

    def matrix(self, expert: int, mat: int):
        """(codes [R, K/2], scales, tensor_scale) of one matrix in its 2-D shape."""
        c = self.cfg
        R, K = (c.f, c.d) if mat < 2 else (c.d, c.f)
        codes = self.codes[expert, mat].reshape(R, K // 2)
        if c.wfmt == WFMT_NVFP4:
            sc = self.scales[expert, mat].reshape(R, K // 16)
        else:
            sc = self.scales[expert, mat].view(np.uint16).reshape(R, K // 32, 2)
        return codes, sc, self.tensor_scale[expert, mat]


def make_layer(cfg: LayerConfig, layer: int = 0, seed: int | None = None) -> LayerWeights:
    """Draw one layer's weights (deterministic in (seed, layer))."""
    seed = cfg.seed if seed is None else seed
    E, d, f = cfg.n_experts, cfg.d, cfg.f
    router = (_rng(seed, layer, _S_ROUTER).standard_normal((E, d), dtype=np.float32)
              * np.float32(1.0 / math.sqrt(d))).astype(np.float32)
    bias = None
    if cfg.bias == "zipf":
        rank = _rng(seed, layer, _S_BIAS).permutation(E) + 1
        bias = (-1.1 * np.log(rank.astype(np.float64))).astype(np.float32)
    n_codes = cfg.codes_per_matrix
    codes = _rng(seed, layer, _S_CODES).integers(0, 256, size=(E + 1, 3, n_codes), dtype=np.uint8)
    if cfg.wfmt == WFMT_NVFP4:
        scales = _rng(seed, layer, _S_SCALES).integers(
            0x28, 0x40, size=(E + 1, 3, cfg.scales_per_matrix), dtype=np.uint8)
        tscale = (np.float32(0.00705) * _rng(seed, layer, _S_TSCALE).uniform(
            0.75, 1.25, size=(E + 1, 3))).astype(np.float32)
        tscale[:, 2] *= np.float32(cfg.down_scale)
    else:
        n_blk = f * d // 32
        r = _rng(seed, layer, _S_SCALES)
        dscale = np.array([1.0, 1.0, cfg.down_scale])[None, :, None]
        dd = (0.00434 * dscale * r.uniform(0.8, 1.2, size=(E + 1, 3, n_blk))).astype(np.float16)
        mm = (-7.5 * dd.astype(np.float64) * r.uniform(0.9, 1.1, size=(E + 1, 3, n_blk))).astype(np.float16)
        dm = np.stack([dd.view(np.uint16), mm.view(np.uint16)], axis=-1)   # [E+1, 3, n_blk, 2]
        scales = np.ascontiguousarray(dm).view(np.uint8).reshape(E + 1, 3, n_blk * 4)
        tscale = np.ones((E + 1, 3), dtype=np.float32)
    return LayerWeights(cfg, router, bias, codes, scales, tscale)


# ---------------------------------------------------------------------------
# The 4-bit output head (lm_head) and the uniforms its sampler draws with
# ---------------------------------------------------------------------------
# The blog gives ~2.5B active parameters per token counting the output head
# and ~2.2B for the body ("The architecture is an argument about memory
# bandwidth", Active parameters bullet): a head of ~0.3B parameters, i.e. a
# vocabulary of ~0.3e9 / d = ~146k rows at d = 2048; 146,432 is that figure
# rounded to a multiple of 128.
#
# Head recipe: NVFP4 codes uniform over all 16 codes, E4M3 block-scale bytes
# uniform over 0x28..0x3F, tensor scale 0.0353 * U(0.75, 1.25): weights of
# standard deviation ~0.1, so that x ~ N(0, 1) gives logits of standard
# deviation ~4.5 and a peaked distribution in which top-p cuts inside the
# top-20.
_S_HEAD_CODES, _S_HEAD_SCALES, _S_HEAD_TSCALE, _S_UNIFORM = 20, 21, 22, 23


@dataclasses.dataclass(frozen=True)
class HeadConfig:
    d: int = 2048
    vocab: int = 146_432
    tokens: int = 1
    seed: int = 0
    name: str = ""


HEAD_CONFIGS = {
    "flint": HeadConfig(name="flint_lm_head_V146432_T1_nvfp4"),
    "small": HeadConfig(d=512, vocab=1000, tokens=3, name="lm_head_d512_V1000_T3_nvfp4"),
}


@dataclasses.dataclass
class HeadWeights:
    """Canonical host layout of the head: codes uint8 [V, d/2] (two E2M1 codes
    per byte, low nibble first), scales uint8 [V, d/16] (E4M3), tensor_scale
    float32."""
    cfg: HeadConfig
    codes: np.ndarray
    scales: np.ndarray
    tensor_scale: np.float32


def make_head(cfg: HeadConfig, seed: int | None = None) -> HeadWeights:
    seed = cfg.seed if seed is None else seed
    V, d = cfg.vocab, cfg.d
    codes = _rng(seed, 0, _S_HEAD_CODES).integers(0, 256, size=(V, d // 2), dtype=np.uint8)
    scales = _rng(seed, 0, _S_HEAD_SCALES).integers(0x28, 0x40, size=(V, d // 16), dtype=np.uint8)
    tscale = np.float32(0.0353 * _rng(seed, 0, _S_HEAD_TSCALE).uniform(0.75, 1.25))
    return HeadWeights(cfg, codes, scales, tscale)


def make_uniforms(tokens: int, seed: int = 0, stream: int = 0) -> np.ndarray:
    """float32 [tokens] in [0, 1): the sampler's random draws, one per token."""
    u = _rng(seed, 20_000 + stream, _S_UNIFORM).random(tokens).astype(np.float32)
    return np.minimum(u, np.nextafter(np.float32(1.0), np.float32(0.0)))


def make_hidden(cfg: LayerConfig, tokens: int | None = None, seed: int | None = None,
                stream: int = 0) -> np.ndarray:
    """Hidden states as bfloat16 bit patterns, uint16 [T, d]."""
    seed = cfg.seed if seed is None else seed
    T = cfg.tokens if tokens is None else tokens
    x = _rng(seed, 10_000 + stream, _S_HIDDEN).standard_normal((T, cfg.d), dtype=np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)
