"""Scalar decoders and encoders for the number formats of the 4-bit MoE layer.

TEST INFRASTRUCTURE. This module belongs to the CPU oracle: only the test suite,
the smoke check and the benchmark's CPU-baseline leg may import it. The product
path never calls it and has no fallback to it.

Format definitions (the Flint blog names NVFP4 and q4_1 but does not define
them; "Recursive Flint 40B-A2.5B", section "What actually shipped", bullets
"NVFP4 GGUF" and "Int4 GGUF"):

* E2M1 (FP4), OCP Microscaling Formats spec v1.0, section 5.3.3: sign bit 3,
  exponent bits 2..1 with bias 1, mantissa bit 0; exponent 0 is subnormal
  (value m * 0.5). Magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}; no inf/NaN.
* E4M3 ("fn" variant), OCP 8-bit floating point spec: sign bit 7, exponent
  bits 6..3 with bias 7, mantissa bits 2..0; exponent 0 is subnormal
  (m/8 * 2^-6); S.1111.111 is NaN; no infinities; max 448.
* NVFP4 weight: w = (E2M1(code) * E4M3(block scale)) * fp32 tensor scale, one
  E4M3 block scale per 16 consecutive elements of a row along the contraction
  axis, one fp32 tensor scale per matrix.
* q4_1 weight: w = d * q + m with q in 0..15 and fp16 d, m per block of 32
  consecutive elements along the contraction axis.

Everything here computes in float64. Products such as code*scale*tensor_scale
need at most 2+4+24 significant bits and d*q+m at most ~40, so the float64
results are exact and a single rounding to float32 gives the correctly rounded
float32 weight.
"""
from __future__ import annotations

import math

import numpy as np

# ---------------------------------------------------------------------------
# scalar decoders (closed forms, one element at a time)
# ---------------------------------------------------------------------------


def e2m1_value(code: int) -> float:
    """Value of a 4-bit E2M1 code (OCP MX v1.0, FP4 E2M1)."""
    code = int(code) & 0xF
    sign = -1.0 if code & 0x8 else 1.0
    exp = (code >> 1) & 0x3
    man = code & 0x1
    if exp == 0:
        return sign * man * 0.5
    return sign * math.ldexp(1.0 + man / 2.0, exp - 1)


def e4m3_value(byte: int) -> float:
    """Value of an E4M3 ("fn") byte; NaN for S.1111.111."""
    byte = int(byte) & 0xFF
    sign = -1.0 if byte & 0x80 else 1.0
    exp = (byte >> 3) & 0xF
    man = byte & 0x7
    if exp == 0xF and man == 0x7:
        return math.nan
    if exp == 0:
        return sign * math.ldexp(man / 8.0, -6)
    return sign * math.ldexp(1.0 + man / 8.0, exp - 7)


def fp16_value(bits: int) -> float:
    """Value of an IEEE binary16 bit pattern."""
    bits = int(bits) & 0xFFFF
    sign = -1.0 if bits & 0x8000 else 1.0
    exp = (bits >> 10) & 0x1F
    man = bits & 0x3FF
    if exp == 0x1F:
        return sign * math.inf if man == 0 else math.nan
    if exp == 0:
        return sign * math.ldexp(man, -24)
    return sign * math.ldexp(1.0 + man / 1024.0, exp - 15)


def bf16_value(bits: int) -> float:
    """Value of a bfloat16 bit pattern (the top half of a binary32)."""
    return float(np.array([int(bits) << 16], dtype=np.uint32).view(np.float32)[0])


# Lookup tables built from the closed forms above.
E2M1_TABLE = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)
E4M3_TABLE = np.array([e4m3_value(b) for b in range(256)], dtype=np.float64)
E2M1_MAGNITUDES = E2M1_TABLE[:8].copy()  # 0, .5, 1, 1.5, 2, 3, 4, 6


_FP16_TABLE: np.ndarray | None = None


def fp16_array(bits: np.ndarray) -> np.ndarray:
    """Vector form of fp16_value (float64 out), through a 65536-entry table."""
    global _FP16_TABLE
    if _FP16_TABLE is None:
        _FP16_TABLE = np.array([fp16_value(b) for b in range(1 << 16)], dtype=np.float64)
    return _FP16_TABLE[np.asarray(bits, dtype=np.uint16)]


def bf16_array(bits: np.ndarray) -> np.ndarray:
    """Values of bfloat16 bit patterns (float64 out)."""
    bits = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return bits.view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# rounding to bfloat16 (output stage of the layer)
# ---------------------------------------------------------------------------

_BF16_MAX = math.ldexp(2.0 - 2.0 ** -7, 127)


def bf16_round(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bfloat16, ties to even (one rounding).

    bfloat16 keeps 8 significant bits and the binary32 exponent range; the
    subnormal spacing is 2^-133. Values at or beyond the overflow threshold
    (max + half an ulp) become +-inf.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    nz = (x != 0) & np.isfinite(x)
    m, e = np.frexp(x[nz])          # x = m * 2^e, 0.5 <= |m| < 1
    # quantum of the bfloat16 grid at this magnitude: 2^(e-8), floored at 2^-133
    qexp = np.maximum(e - 8, -133)
    q = np.rint(np.ldexp(x[nz], -qexp))   # rint = round half to even
    r = np.ldexp(q, qexp)
    r = np.where(np.abs(x[nz]) >= math.ldexp(2.0 - 2.0 ** -8, 127), np.copysign(np.inf, r), r)
    out[nz] = r
    out[~np.isfinite(x)] = x[~np.isfinite(x)]
    out[x == 0] = x[x == 0]
    return out


def bf16_bits(x: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns of values that are already bfloat16-representable."""
    v = np.asarray(x, dtype=np.float64).astype(np.float32)
    return (v.view(np.uint32) >> 16).astype(np.uint16)


# ---------------------------------------------------------------------------
# weight dequantisation
# ---------------------------------------------------------------------------


def unpack_nibbles(codes: np.ndarray) -> np.ndarray:
    """[R, K/2] bytes -> [R, K] nibbles; element 2i is the low nibble of byte i."""
    codes = np.asarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = codes & 0xF
    out[..., 1::2] = codes >> 4
    return out


def dequant_nvfp4(codes: np.ndarray, scales: np.ndarray, tensor_scale: float) -> np.ndarray:
    """NVFP4 matrix -> float64 [R, K] (exact).

    codes  uint8 [R, K/2]  (two E2M1 codes per byte, low nibble first)
    scales uint8 [R, K/16] (E4M3 block scale for elements 16j..16j+15)
    tensor_scale float32
    """
    nib = unpack_nibbles(codes)
    R, K = nib.shape
    blk = np.repeat(E4M3_TABLE[np.asarray(scales, dtype=np.uint8)], 16, axis=1)
    assert blk.shape == (R, K)
    return (E2M1_TABLE[nib] * blk) * float(np.float32(tensor_scale))


def dequant_q41(codes: np.ndarray, dm: np.ndarray) -> np.ndarray:
    """q4_1 matrix -> float64 [R, K] (exact).

    codes uint8  [R, K/2]     (q values, low nibble first)
    dm    uint16 [R, K/32, 2] (fp16 bits of d and m for each block of 32)
    """
    q = unpack_nibbles(codes).astype(np.float64)
    R, K = q.shape
    dm = np.asarray(dm, dtype=np.uint16)
    d = np.repeat(fp16_array(dm[..., 0]), 32, axis=1)
    m = np.repeat(fp16_array(dm[..., 1]), 32, axis=1)
    assert d.shape == (R, K)
    return d * q + m


# ---------------------------------------------------------------------------
# round-to-nearest encoders used by the activation-quantisation mode
# ---------------------------------------------------------------------------


def e2m1_encode_rne(r: np.ndarray) -> np.ndarray:
    """float32 values -> E2M1 codes: nearest magnitude, ties to the even
    mantissa bit, saturating at 6; the sign bit copies the sign bit of r."""
    r = np.asarray(r, dtype=np.float32)
    a = np.abs(r).astype(np.float64)
    codes = np.zeros(a.shape, dtype=np.uint8)
    best = np.full(a.shape, np.inf)
    for c in range(8):
        dist = np.abs(a - E2M1_MAGNITUDES[c])
        # strictly closer wins; on an exact tie keep the code whose mantissa bit is 0
        take = (dist < best) | ((dist == best) & ((c & 1) == 0))
        codes = np.where(take, c, codes)
        best = np.where(take, dist, best)
    codes = np.where(a >= 6.0, 7, codes).astype(np.uint8)
    return codes | (np.signbit(r).astype(np.uint8) << 3)


# Non-negative, finite E4M3 values in increasing order with their bytes.
_E4M3_POS_BYTES = np.array([b for b in range(0x7F)], dtype=np.uint8)  # 0x00..0x7E
_E4M3_POS_VALUES = E4M3_TABLE[_E4M3_POS_BYTES]


def e4m3_encode_rne_nonneg(r: np.ndarray) -> np.ndarray:
    """Non-negative float32 values -> E4M3 bytes: nearest value, ties to even
    mantissa, saturating at 448."""
    a = np.asarray(r, dtype=np.float32).astype(np.float64)
    assert np.all(a >= 0)
    idx = np.searchsorted(_E4M3_POS_VALUES, a)            # first value >= a
    idx = np.clip(idx, 0, len(_E4M3_POS_VALUES) - 1)
    lo = np.clip(idx - 1, 0, None)
    up_v = _E4M3_POS_VALUES[idx]
    lo_v = _E4M3_POS_VALUES[lo]
    d_up = up_v - a
    d_lo = a - lo_v
    pick_up = (d_up < d_lo) | ((d_up == d_lo) & ((_E4M3_POS_BYTES[idx] & 1) == 0))
    pick_up |= (lo == idx)
    out = np.where(pick_up, _E4M3_POS_BYTES[idx], _E4M3_POS_BYTES[lo])
    out = np.where(a >= 448.0, 0x7E, out)
    return out.astype(np.uint8)
