"""The allocation-free bucketing entry point (flint_moe_bucket_noalloc)
against the handle-based flint_moe_bucket.

Callers that cannot allocate device memory where they bucket tokens (a step
recorded under CUDA stream capture, memory owned by another allocator, a
runtime without the CUDA allocator) use the no-alloc entry point; it must give
exactly what flint_moe_bucket gives, call after call, although every call
reuses the same static scratch array.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _selection(T, k, E, seed):
    rng = np.random.default_rng(seed)
    p = 1.0 / np.arange(1, E + 1) ** 1.1           # skewed expert popularity
    p /= p.sum()
    sel = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)])
    return sel.astype(np.int32)


def test_bucket_noalloc_matches_bucket_on_two_calls_in_a_row():
    if not torch.cuda.is_available():
        pytest.fail("CUDA device required for -m gpu tests")
    from bit_quantized_expert_softmax_b300 import build
    build.build()
    from bit_quantized_expert_softmax_b300 import flint_moe as fm

    E, k, Tmax = 256, 6, 8192
    h = fm.flint_moe_create(512, 128, E, k, 1, fm.FLINT_W_NVFP4, Tmax, 1, 0)
    try:
        # two calls in a row; the second is smaller, so stale scratch from the
        # first would show up if a call read what it had not written
        for T, seed in [(8192, 11), (683, 12)]:
            idx = torch.from_numpy(_selection(T, k, E, seed)).cuda()
            off_ref = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
            perm_ref = torch.full((T * k,), -1, dtype=torch.int32, device="cuda")
            off_na = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
            perm_na = torch.full((T * k,), -1, dtype=torch.int32, device="cuda")
            fm.flint_moe_bucket(h, idx, T, off_ref, perm_ref)
            fm.flint_moe_bucket_noalloc(idx, T, k, E, off_na, perm_na)
            torch.cuda.synchronize()
            assert torch.equal(off_na, off_ref), T
            assert torch.equal(perm_na, perm_ref), T
            assert int(off_na[-1]) == T * k
    finally:
        fm.flint_moe_destroy(h)


def test_bucket_noalloc_rejects_sizes_beyond_its_scratch():
    from bit_quantized_expert_softmax_b300 import flint_moe as fm
    k = 8
    T = (1 << 19) // k + 1                       # one token past the 524288-assignment limit
    with pytest.raises(fm.FlintError) as ei:
        fm.flint_moe_bucket_noalloc(None, T, k, 256, None, None, stream=0)
    assert ei.value.code == fm.FLINT_EINVAL
    with pytest.raises(fm.FlintError) as ei:
        fm.flint_moe_bucket_noalloc(None, 4, 6, 257, None, None, stream=0)   # E above 256
    assert ei.value.code == fm.FLINT_EINVAL
