"""Decode attention (flint_moe_attn_decode) against the oracle's decode step:
sliding-window layers (513-token window, rotary positions) with the cache's
ring wrapping, full-attention layers (no rotation), first positions, two
steps in a row through the written cache slot, and bad arguments."""
import numpy as np
import pytest

from oracle import attention as A
from oracle import formats as F

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


def _bits(v):
    return F.bf16_bits(F.bf16_round(np.asarray(v, dtype=np.float64)))


def _case(B, cap, seed, n_kv=4):
    rng = np.random.default_rng(seed)
    H = 8 * n_kv
    q = _bits(rng.standard_normal((B, H, 128)))
    k = _bits(rng.standard_normal((B, n_kv, 128)))
    v = _bits(rng.standard_normal((B, n_kv, 128)))
    kc = _bits(rng.standard_normal((B, n_kv, cap, 128)))
    vc = _bits(rng.standard_normal((B, n_kv, cap, 128)))
    wq = (1 + 0.1 * rng.standard_normal(128)).astype(np.float32)
    wk = (1 + 0.1 * rng.standard_normal(128)).astype(np.float32)
    sinks = rng.standard_normal(H).astype(np.float32)
    return q, k, v, kc, vc, wq, wk, sinks


def _dev16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda()


def _run(fm, window, cap, rope, pos, case, n_kv=4):
    q, k, v, kc, vc, wq, wk, sinks = case
    B = q.shape[0]
    dq, dk, dv = _dev16(q), _dev16(k), _dev16(v)
    dkc, dvc = _dev16(kc), _dev16(vc)
    dpos = torch.tensor(pos, dtype=torch.int32, device="cuda")
    out = torch.empty((B, 8 * n_kv, 128), dtype=torch.int16, device="cuda")
    fm.flint_moe_attn_decode(8 * n_kv, n_kv, window, cap, rope, B, dq, dk, dv, dkc, dvc, dpos,
                             torch.from_numpy(wq).cuda(), torch.from_numpy(wk).cuda(),
                             torch.from_numpy(sinks).cuda(), out)
    torch.cuda.synchronize()
    return out.cpu().numpy().view(np.uint16), dkc.cpu().numpy().view(np.uint16), dvc.cpu().numpy().view(np.uint16)


def _check(fm, window, cap, rope, pos, case, n_kv=4):
    q, k, v, kc, vc, wq, wk, sinks = case
    out, kc2, vc2 = _run(fm, window, cap, rope, pos, case, n_kv)
    for b, p in enumerate(pos):
        ref, ks, vs = A.decode_step(F.bf16_array(q[b]), F.bf16_array(k[b]), F.bf16_array(v[b]), kc[b], vc[b], p,
                                    wq, wk, sinks, window=window, rope_on=rope)
        got = F.bf16_array(out[b])
        rel = np.linalg.norm(got - ref) / np.linalg.norm(ref)
        assert rel <= 5e-3, (b, p, rel)
        assert np.max(np.abs(got - ref)) <= 3e-2 * np.sqrt(np.mean(ref ** 2)), (b, p)
        slot = p % cap
        # the stored key: the oracle's bf16 of the normed, rotated key (one
        # rounding step apart at most where fp32 and fp64 straddle a boundary)
        gk = F.bf16_array(kc2[b][:, slot])
        wk_ = F.bf16_array(ks)
        assert np.all(np.abs(gk - wk_) <= np.abs(wk_) * 2.0 ** -7 + 1e-30), (b, p)
        assert np.mean(kc2[b][:, slot] == ks) >= 0.98
        assert np.array_equal(vc2[b][:, slot], vs)
        others = np.ones(cap, dtype=bool)
        others[slot] = False
        assert np.array_equal(kc2[b][:, others], kc[b][:, others])   # nothing else written


def test_sliding_window_positions_and_ring_wrap(fm):
    pos = [0, 1, 63, 64, 300, 512, 513, 514, 700, 4099, 100000]
    cap = 520
    _check(fm, 513, cap, True, pos, _case(len(pos), cap, 1))


def test_full_attention_without_rotation(fm):
    pos = [0, 5, 200, 1023]
    cap = 1024
    _check(fm, 0, cap, False, pos, _case(len(pos), cap, 2))


def test_other_head_counts(fm):
    pos = [7, 513, 900]
    for n_kv in (1, 2, 8):
        _check(fm, 513, 513, True, pos, _case(len(pos), 513, 3 + n_kv, n_kv=n_kv), n_kv=n_kv)


def test_two_steps_through_the_cache(fm):
    """Step pos writes its key and value into the cache; step pos+1 reads them
    as a cached position, against the oracle run on the cache the GPU wrote."""
    cap = 516
    case = _case(2, cap, 9)
    q, k, v, kc, vc, wq, wk, sinks = case
    pos = [515, 20]
    out1, kc1, vc1 = _run(fm, 513, cap, True, pos, case)
    case2 = (q, k, v, kc1, vc1, wq, wk, sinks)
    _check(fm, 513, cap, True, [p + 1 for p in pos], case2)


def test_attn_rejects_bad_arguments(fm):
    for kw in [dict(window=513, cap=512), dict(window=-1, cap=10), dict(window=0, cap=0)]:
        with pytest.raises(fm.FlintError) as ei:
            fm.flint_moe_attn_decode(32, 4, kw["window"], kw["cap"], True, 1, *([None] * 10))
        assert ei.value.code == fm.FLINT_EINVAL
    with pytest.raises(fm.FlintError):
        fm.flint_moe_attn_decode(30, 4, 513, 513, True, 1, *([None] * 10))   # not 8 query heads per key head
