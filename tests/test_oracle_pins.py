"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test checks one oracle function against an independent source: a value
the Flint blog prints, a hand-worked example, an independent library decoder
(ml_dtypes, numpy float16, torch bfloat16), a closed-form identity, or brute
force on tiny inputs. A plausible slip in the oracle (a dropped term, a wrong
sign, index or nibble order, a transposed operand) fails at least one of them.
"""
import math

import ml_dtypes
import numpy as np
import pytest
import torch

from bit_quantized_expert_softmax_b300 import synth
from oracle import formats as F
from oracle import moe as M
from tests.conftest import read_golden

# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------


def test_e2m1_table_matches_ocp_values_and_ml_dtypes():
    # OCP MX v1.0 table of FP4 E2M1 magnitudes
    assert list(F.E2M1_TABLE[:8]) == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    lib = np.arange(16, dtype=np.uint8).view(ml_dtypes.float4_e2m1fn).astype(np.float64)
    assert np.array_equal(F.E2M1_TABLE, lib)
    assert math.copysign(1.0, F.E2M1_TABLE[8]) == -1.0   # 0b1000 is -0


def test_e4m3_table_matches_ml_dtypes_all_bytes():
    lib = np.arange(256, dtype=np.uint8).view(ml_dtypes.float8_e4m3fn).astype(np.float64)
    nan = np.isnan(lib)
    assert np.array_equal(nan, np.isnan(F.E4M3_TABLE))
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.array_equal(F.E4M3_TABLE[~nan], lib[~nan])
    assert F.E4M3_TABLE[0x7E] == 448.0 and F.E4M3_TABLE[0x01] == 2.0 ** -9


def test_fp16_table_matches_numpy_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    lib = bits.view(np.float16).astype(np.float64)
    ours = F.fp16_array(bits)
    fin = np.isfinite(lib)
    assert np.array_equal(np.isnan(ours), np.isnan(lib))
    assert np.array_equal(ours[fin], lib[fin])
    assert np.array_equal(ours[np.isinf(lib)], lib[np.isinf(lib)])


def test_bf16_round_matches_torch_on_float32_inputs():
    rng = np.random.default_rng(1)
    v = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(3.0),
        (rng.standard_normal(2000) * 1e-39).astype(np.float32),            # subnormals
        np.array([3.3895314e38, 3.39e38, -3.4e38, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8,
                  0.0, -0.0], dtype=np.float32),
    ])
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    ours = F.bf16_round(v.astype(np.float64))
    assert np.array_equal(np.isinf(ours), np.isinf(ref))
    ok = np.isfinite(ref)
    assert np.array_equal(ours[ok], ref[ok])


def test_bf16_round_single_rounding_from_float64():
    # 1 + 2^-8 + 2^-30 lies just above the tie between 1 and 1 + 2^-7: nearest is 1 + 2^-7.
    # Rounding through float32 first would hit the tie exactly and give 1.0.
    assert F.bf16_round(np.array([1.0 + 2.0 ** -8 + 2.0 ** -30]))[0] == 1.0 + 2.0 ** -7
    assert F.bf16_round(np.array([1.0 + 2.0 ** -8]))[0] == 1.0          # tie -> even
    assert F.bf16_round(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 1.0 + 2.0 ** -6


# ---------------------------------------------------------------------------
# dequantisation
# ---------------------------------------------------------------------------


def test_dequant_hand_examples():
    rows = read_golden("dequant_examples.txt")
    assert len(rows) >= 8
    for r in rows:
        if r[0] == "nvfp4":
            code, sc, ts, want = int(r[1], 16), int(r[2], 16), float(r[3]), float(r[4])
            codes = np.zeros((1, 8), dtype=np.uint8)
            codes[0, 0] = code                       # element 0 = low nibble of byte 0
            scales = np.array([[sc]], dtype=np.uint8)
            got = F.dequant_nvfp4(codes, scales, np.float32(ts))[0, 0]
        else:
            dbits, mbits, q, want = int(r[1], 16), int(r[2], 16), int(r[3]), float(r[4])
            codes = np.zeros((1, 16), dtype=np.uint8)
            codes[0, 0] = q
            dm = np.array([[[dbits, mbits]]], dtype=np.uint16)
            got = F.dequant_q41(codes, dm)[0, 0]
        got32 = np.float32(got)
        assert got32 == np.float32(want), r
        assert math.copysign(1.0, got32) == math.copysign(1.0, want), r


def test_dequant_nvfp4_matches_elementwise_library_decode():
    rng = np.random.default_rng(2)
    R, K = 5, 64
    codes = rng.integers(0, 256, size=(R, K // 2), dtype=np.uint8)
    scales = rng.integers(0, 0x7F, size=(R, K // 16), dtype=np.uint8)
    ts = np.float32(0.37)
    ours = F.dequant_nvfp4(codes, scales, ts)
    for r in range(R):
        for k in range(K):
            byte = int(codes[r, k // 2])
            nib = (byte & 0xF) if k % 2 == 0 else (byte >> 4)
            c = float(np.array([nib], dtype=np.uint8).view(ml_dtypes.float4_e2m1fn)[0])
            s = float(np.array([scales[r, k // 16]], dtype=np.uint8).view(ml_dtypes.float8_e4m3fn)[0])
            assert ours[r, k] == c * s * float(ts)


def test_dequant_q41_matches_elementwise_numpy_float16():
    rng = np.random.default_rng(3)
    R, K = 3, 96
    codes = rng.integers(0, 256, size=(R, K // 2), dtype=np.uint8)
    d = rng.uniform(-0.1, 0.1, size=(R, K // 32)).astype(np.float16)
    m = rng.uniform(-1, 1, size=(R, K // 32)).astype(np.float16)
    dm = np.stack([d.view(np.uint16), m.view(np.uint16)], axis=-1)
    ours = F.dequant_q41(codes, dm)
    for r in range(R):
        for k in range(K):
            byte = int(codes[r, k // 2])
            q = (byte & 0xF) if k % 2 == 0 else (byte >> 4)
            want = float(d[r, k // 32]) * q + float(m[r, k // 32])
            assert ours[r, k] == want


# ---------------------------------------------------------------------------
# router, top-k, renormalisation, bucketing
# ---------------------------------------------------------------------------


def test_router_logits_brute_force_exact_sum():
    rng = np.random.default_rng(4)
    T, E, d = 3, 7, 40
    x = rng.standard_normal((T, d))
    W = rng.standard_normal((E, d)).astype(np.float32)
    b = rng.standard_normal(E).astype(np.float32)
    L = M.router_logits(x, W, b)
    for t in range(T):
        for e in range(E):
            want = math.fsum([x[t, i] * float(W[e, i]) for i in range(d)] + [float(b[e])])
            assert abs(L[t, e] - want) <= 1e-12 * max(1.0, abs(want))


def test_topk_brute_force_and_ties():
    rng = np.random.default_rng(5)
    T, E, k = 20, 32, 6
    L = rng.standard_normal((T, E)).astype(np.float32)
    L[0, [3, 9, 17]] = 5.0                 # three-way tie at the top
    L[1, :] = 0.0                          # all equal: experts 0..5
    L[2, [30, 31]] = L[2].max() + 1        # tie at the top between the two last experts
    got = M.select_topk(L, k)
    for t in range(T):
        want = sorted(range(E), key=lambda e: (-float(L[t, e]), e))[:k]
        assert list(got[t]) == want
    assert list(got[0, :3]) == [3, 9, 17]
    assert list(got[1]) == [0, 1, 2, 3, 4, 5]
    assert list(got[2, :2]) == [30, 31]


def test_route_weights_equal_softmax_over_selected_and_sum_to_one():
    rng = np.random.default_rng(6)
    L = rng.standard_normal((50, 256)) * 3
    sel = M.select_topk(L.astype(np.float32), 6)
    w = M.route_weights(L, sel)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-12, rtol=0)
    Ls = np.take_along_axis(L, sel.astype(np.int64), axis=1)
    alt = np.exp(Ls) / np.exp(Ls).sum(axis=1, keepdims=True)     # closed form
    assert np.allclose(w, alt, rtol=1e-12, atol=0)
    assert np.all(np.diff(w, axis=1) <= 1e-15)                   # descending logits -> descending weights


def test_bucket_brute_force_and_invariants():
    rng = np.random.default_rng(7)
    T, k, E = 37, 6, 16
    sel = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    b = M.bucket(sel, E)
    lists = [[] for _ in range(E)]
    for t in range(T):
        for j in range(k):
            lists[int(sel[t, j])].append(t * k + j)
    assert list(b.perm) == [a for e in range(E) for a in lists[e]]
    assert list(b.counts) == [len(l) for l in lists]
    assert b.offsets[0] == 0 and b.offsets[-1] == T * k
    assert np.all(np.diff(b.offsets) >= 0)
    assert sorted(b.perm) == list(range(T * k))


# ---------------------------------------------------------------------------
# experts, combine, layer
# ---------------------------------------------------------------------------


def test_swiglu_hand_example():
    # d = f = 16, x = e_5 (one-hot at input 5).
    # gate[2, 5] = 1.0, up[2, 5] = 2.0 (element 5 = high nibble of byte 2), down[3, 2] = 0.5.
    # g2 = 1, u2 = 2, h2 = silu(1)*2 = 2e/(1+e), y3 = 0.5*h2 = e/(1+e); every other y is 0.
    def mat(row, byte, code):
        c = np.zeros((16, 8), dtype=np.uint8)
        c[row, byte] = code
        return F.dequant_nvfp4(c, np.full((16, 1), 0x38, np.uint8), np.float32(1.0))
    wg, wu, wd = mat(2, 2, 0x20), mat(2, 2, 0x40), mat(3, 1, 0x01)
    x = np.zeros((1, 16))
    x[0, 5] = 1.0
    y = M.expert_forward(wg, wu, wd, x)
    assert abs(y[0, 3] - math.e / (1 + math.e)) < 1e-15
    assert np.count_nonzero(y) == 1
    # silu with a negative argument: silu(-1) = -1/(1+e)
    assert abs(M.silu(np.array([-1.0]))[0] + 1 / (1 + math.e)) < 1e-15


def _tiny_cfg(**kw):
    base = dict(d=64, f=32, n_experts=16, top_k=6, tokens=5, seed=11)
    base.update(kw)
    return synth.LayerConfig(**base)


@pytest.mark.parametrize("wfmt", [synth.WFMT_NVFP4, synth.WFMT_Q4_1])
def test_sparse_layer_equals_dense_masked_evaluation(wfmt):
    cfg = _tiny_cfg(wfmt=wfmt, bias="zipf")
    layer = synth.make_layer(cfg)
    xb = synth.make_hidden(cfg)
    r = M.moe_layer(xb, layer)
    x = F.bf16_array(xb)
    # brute force: every expert on every token, masked by the routing weights
    dense = np.zeros((cfg.tokens, cfg.d))
    for e in range(cfg.n_experts + 1):
        ws = [M.dequant_matrix(layer, e, m) for m in range(3)]
        for t in range(cfg.tokens):
            g = np.array([math.fsum(ws[0][i] * x[t]) for i in range(cfg.f)])
            u = np.array([math.fsum(ws[1][i] * x[t]) for i in range(cfg.f)])
            h = g / (1 + np.exp(-g)) * u
            y = np.array([math.fsum(ws[2][i] * h) for i in range(cfg.d)])
            if e == cfg.n_experts:
                coef = 1.0
            else:
                hit = np.nonzero(r.sel[t] == e)[0]
                coef = float(r.weights[t, hit[0]]) if hit.size else 0.0
            dense[t] += coef * y
    assert np.max(np.abs(dense - r.out)) <= 1e-12 * np.max(np.abs(dense))


@pytest.mark.parametrize("wfmt", [synth.WFMT_NVFP4, synth.WFMT_Q4_1])
def test_zero_routed_experts_reproduce_shared_expert_exactly(wfmt):
    cfg = _tiny_cfg(wfmt=wfmt)
    layer = synth.make_layer(cfg)
    layer.codes[: cfg.n_experts] = 0
    layer.scales[: cfg.n_experts] = 0           # q4_1: d = m = 0 as well
    xb = synth.make_hidden(cfg)
    r = M.moe_layer(xb, layer)
    ws = [M.dequant_matrix(layer, cfg.n_experts, m) for m in range(3)]
    shared = M.expert_forward(*ws, F.bf16_array(xb))
    assert np.array_equal(r.out_bf16, F.bf16_round(shared))


def test_stack_residual_is_bf16_of_sum():
    cfg = _tiny_cfg(n_layers=2)
    layers = [synth.make_layer(cfg, layer=i) for i in range(2)]
    xb = synth.make_hidden(cfg)
    bits, res = M.moe_stack(xb, layers)
    x1 = F.bf16_round(F.bf16_array(xb) + res[0].out_bf16)
    r1 = M.moe_layer(F.bf16_bits(x1), layers[1])
    x2 = F.bf16_round(x1 + r1.out_bf16)
    assert np.array_equal(F.bf16_array(bits), x2)


# ---------------------------------------------------------------------------
# activation quantisation (FP4 tensor-core mode)
# ---------------------------------------------------------------------------


def test_act_quant_hand_example():
    rows = read_golden("act_quant_examples.txt")
    v = np.zeros((1, 64), dtype=np.float32)
    want_codes = np.zeros((1, 64), dtype=np.uint8)
    want_scales = {}
    for r in rows:
        if r[0] == "input":
            v[0, 16 * int(r[1]) + int(r[2])] = float(r[3])
        elif r[0] == "code":
            want_codes[0, 16 * int(r[1]) + int(r[2])] = int(r[3], 16)
        elif r[0] == "scale":
            want_scales[int(r[1])] = int(r[2], 16)
        elif r[0] == "rowscale":
            want_row = float(r[1])
    codes, sb, s_t, deq = M.quant_act_nvfp4(v)
    assert s_t[0] == want_row
    assert [int(sb[0, b]) for b in range(4)] == [want_scales[b] for b in range(4)]
    assert np.array_equal(codes, want_codes)
    assert deq[0, 16] == 12.0 and deq[0, 17] == 4.0 and deq[0, 22] == -8.0


def test_act_quant_round_trip_of_representable_rows():
    rng = np.random.default_rng(8)
    # Rows built from codes with the top block scale at 448 so that s_t is exactly 1/8:
    # every value is code * E4M3(sb) / 8 and must come back unchanged.
    T, K = 6, 64
    codes = rng.integers(0, 16, size=(T, K)).astype(np.uint8)
    codes[:, 0] = 7                                   # amax element of block 0 = 6 * 448 / 8
    sbytes = rng.integers(0x20, 0x60, size=(T, K // 16)).astype(np.uint8)
    sbytes[:, 0] = 0x7E
    for b in range(1, K // 16):
        codes[:, 16 * b] = 7                          # each block reaches 6 * its scale
    vals = F.E2M1_TABLE[codes] * np.repeat(F.E4M3_TABLE[sbytes], 16, axis=1) / 8.0
    got_codes, got_sb, s_t, deq = M.quant_act_nvfp4(vals.astype(np.float32))
    assert np.all(s_t == np.float32(6 * 448 / 8 / 2688))
    assert np.array_equal(got_sb, sbytes)
    assert np.array_equal(deq, vals)


def test_act_quant_error_is_within_half_a_grid_step():
    rng = np.random.default_rng(9)
    v = rng.standard_normal((16, 256)).astype(np.float32)
    codes, sb, s_t, deq = M.quant_act_nvfp4(v)
    S = np.repeat(F.E4M3_TABLE[sb] * s_t[:, None], 16, axis=1)
    # largest gap of the E2M1 grid below 6 is 2 (between 4 and 6): error <= 1 * S,
    # and below 2 the gap is 0.5: error <= 0.25 * S
    err = np.abs(deq - v)
    small = np.abs(v) <= 2 * S
    assert np.all(err <= 1.0 * S + 1e-12)
    assert np.all(err[small] <= 0.25 * S[small] * (1 + 1e-6) + 1e-12)


def test_w4a4_expert_by_brute_force():
    """The quantised-activation expert against a scalar evaluation on a tiny
    case: exact sums (math.fsum) of the quantised operands, silu through
    math.exp, and h quantised from its float32 value (no other rounding
    between the two projections)."""
    import math

    rng = np.random.default_rng(10)
    f, d = 32, 48
    wg = rng.standard_normal((f, d)) * 0.2
    wu = rng.standard_normal((f, d)) * 0.2
    wd = rng.standard_normal((d, f)) * 0.2
    x = rng.standard_normal((3, d)).astype(np.float32)
    got = M.expert_forward_w4a4(wg, wu, wd, x)
    xq = M.quant_act_nvfp4(x)[3]
    for t in range(3):
        h = np.zeros(f, dtype=np.float32)
        for i in range(f):
            g = math.fsum(xq[t, j] * wg[i, j] for j in range(d))
            u = math.fsum(xq[t, j] * wu[i, j] for j in range(d))
            h[i] = np.float32(g / (1.0 + math.exp(-g)) * u)
        hq = M.quant_act_nvfp4(h[None, :])[3][0]
        for o in range(d):
            want = math.fsum(hq[i] * wd[o, i] for i in range(f))
            assert abs(got[t, o] - want) <= 1e-12 * max(1.0, abs(want)), (t, o)


# ---------------------------------------------------------------------------
# the Flint shape against the numbers the blog prints
# ---------------------------------------------------------------------------


def _golden_structure():
    return {r[0]: float(r[1]) for r in read_golden("flint_structure.txt")}


def test_flint_shape_parameter_counts_fit_the_blog():
    g = _golden_structure()
    cfg = synth.CONFIGS[4]
    d, f, E, k = cfg.d, cfg.f, cfg.n_experts, cfg.top_k
    assert (E, k, cfg.n_layers) == (g["routed_experts"], g["experts_per_token"], g["moe_layers"])
    assert g["layers"] - g["dense_layers"] == cfg.n_layers
    expert = 3 * d * f
    moe_total = cfg.n_layers * ((E + int(g["shared_experts"])) * expert + E * d)
    hq, hkv, dh = int(g["query_heads"]), int(g["kv_heads"]), int(g["head_dim"])
    attn = int(g["layers"]) * (2 * d * hq * dh + 2 * d * hkv * dh)
    moe_active = cfg.n_layers * ((k + 1) * expert + E * d)
    assert moe_total + attn <= g["total_params"]
    assert 0.95 * g["total_params"] <= moe_total + attn + 0.9e9   # room for embeddings, lm_head, 2 dense FFNs
    body = moe_active + attn
    assert 1.9e9 <= body <= g["active_body_params"]
    assert g["active_body_params"] - body < 0.3e9


def test_bits_per_parameter_against_file_sizes():
    g = _golden_structure()
    # NVFP4: 4 bits + one 8-bit scale per 16 -> 4.5 bits; q4_1: 4 bits + 32 bits per 32 -> 5 bits
    nv = g["total_params"] * 4.5 / 8 / 1e9
    q4 = g["total_params"] * 5.0 / 8 / 1e9
    assert abs(nv - g["nvfp4_file_gb"]) / g["nvfp4_file_gb"] < 0.05
    assert abs(q4 - g["q4_1_file_gb"]) / g["q4_1_file_gb"] < 0.05
    assert g["q4_1_file_gb"] > g["nvfp4_file_gb"]
    cfg = synth.CONFIGS[2]
    assert cfg.expert_bytes == 3 * (cfg.f * cfg.d // 2 + cfg.f * cfg.d // 16 + 4)
    assert synth.CONFIGS[3].expert_bytes == 3 * cfg.f * cfg.d * 5 // 8


# ---------------------------------------------------------------------------
# weight quantisation (NVFP4, one tensor scale per matrix)
# ---------------------------------------------------------------------------


def test_weight_quant_single_row_is_the_pinned_row_rule():
    """With one row the per-tensor scale is the per-row one, so the weight
    quantiser must reproduce the activation quantiser (itself pinned by the
    hand-worked golden examples) bit for bit."""
    rng = np.random.default_rng(21)
    for scale in (1e-3, 1.0, 37.0):
        v = (rng.standard_normal((1, 256)) * scale).astype(np.float32)
        c1, sb1, s1, d1 = M.quant_weight_nvfp4(v)
        c2, sb2, s2, d2 = M.quant_act_nvfp4(v)
        assert np.array_equal(c1, c2) and np.array_equal(sb1, sb2)
        assert np.float32(s1) == s2[0]
        assert np.array_equal(d1, d2)


def test_weight_quant_brute_force_nearest_grid_value():
    """Every element's code is the nearest point of its block's grid
    {E2M1 values} x S_b (ties to the even code), found by brute force over
    the 16 codes; the tensor scale and block bytes follow their definitions."""
    rng = np.random.default_rng(22)
    v = (rng.standard_normal((5, 64)) * np.exp(rng.uniform(-3, 3, size=(5, 1)))).astype(np.float32)
    v[2, 16:32] = 0.0                                     # an all-zero block
    codes, sb, s, deq = M.quant_weight_nvfp4(v)
    assert s == np.float32(np.float32(np.abs(v).max()) / np.float32(2688.0))
    for r in range(5):
        for b in range(4):
            blk = v[r, 16 * b:16 * b + 16]
            amax_b = np.float32(np.abs(blk).max())
            want_sb = F.e4m3_encode_rne_nonneg(np.array([np.float32(amax_b / np.float32(6.0)) / s],
                                                        dtype=np.float32))[0]
            assert sb[r, b] == want_sb
            S = np.float32(F.E4M3_TABLE[want_sb] * s)
            for i in range(16):
                if S == 0:
                    assert codes[r, 16 * b + i] == 0
                    continue
                x = np.float32(blk[i] * np.float32(np.float32(1.0) / S))
                dist = [abs(float(x) - F.e2m1_value(c)) for c in range(16)]
                best = min(dist)
                cands = [c for c in range(16) if dist[c] == best]
                if x > 6.0:
                    cands = [7]
                if x < -6.0:
                    cands = [15]
                got = int(codes[r, 16 * b + i])
                if len(cands) > 1:    # a tie: the even mantissa (code bit 0 clear); +-0 both fine
                    cands = [c for c in cands if c & 1 == 0] or cands
                assert got in cands or (F.e2m1_value(got) == 0.0 and best == abs(float(x))), (r, b, i, got, cands)


def test_weight_quant_round_trip_and_zero():
    rng = np.random.default_rng(23)
    # values already on one NVFP4 grid (every 16-block reaches the 6.0 code,
    # so every block scale byte is 448's) get their codes back exactly
    codes = rng.integers(0, 16, size=(4, 32))
    codes[:, 0] = 7
    codes[:, 16] = 15                                     # -6.0
    vals = F.E2M1_TABLE[codes] * 0.25
    c, sb, s, deq = M.quant_weight_nvfp4(vals.astype(np.float32))
    assert np.all(sb == 0x7E)
    assert np.array_equal(F.E2M1_TABLE[c], F.E2M1_TABLE[codes])   # +-0 may swap sign codes
    assert np.allclose(deq, vals, rtol=2.0 ** -22, atol=0)
    z = np.zeros((3, 48), dtype=np.float32)
    c, sb, s, deq = M.quant_weight_nvfp4(z)
    assert s == 0 and not c.any() and not sb.any() and not deq.any()
