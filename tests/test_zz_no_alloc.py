"""The allocation-free bucketing entry point (flint_moe_bucket_noalloc).

Some callers cannot allocate device memory where they bucket tokens: their
device memory is already reserved by another allocator (a framework's caching
pool), their host runtime forbids allocating outside its own allocator, or
they cannot afford cudaMalloc's implicit device synchronisation. The no-alloc
entry point serves them with a static scratch array inside the library. It
must give exactly what the oracle's bucketing gives, and what the handle-based
flint_moe_bucket gives, call after call, although every call reuses the same
scratch array.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import numpy as np
import pytest

from oracle import moe as M

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


def _selection(T, k, E, seed):
    rng = np.random.default_rng(seed)
    p = 1.0 / np.arange(1, E + 1) ** 1.1           # skewed expert popularity
    p /= p.sum()
    sel = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)])
    return sel.astype(np.int32)


def _noalloc(fm, idx_np, T, k, E):
    idx = torch.from_numpy(np.ascontiguousarray(idx_np)).cuda()
    off = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    perm = torch.full((max(T * k, 1),), -1, dtype=torch.int32, device="cuda")
    fm.flint_moe_bucket_noalloc(idx, T, k, E, off, perm)
    torch.cuda.synchronize()
    return off.cpu().numpy(), perm.cpu().numpy()[:T * k]


def test_bucket_noalloc_matches_oracle_and_bucket_on_two_calls_in_a_row(fm):
    E, k, Tmax = 256, 6, 8192
    h = fm.flint_moe_create(512, 128, E, k, 1, fm.FLINT_W_NVFP4, Tmax, 1, 0)
    try:
        # two calls in a row; the second is smaller, so stale scratch from the
        # first would show up if a call read what it had not written
        for T, seed in [(8192, 11), (683, 12)]:
            sel = _selection(T, k, E, seed)
            ref = M.bucket(sel, E)
            off_na, perm_na = _noalloc(fm, sel, T, k, E)
            assert np.array_equal(off_na, ref.offsets), T
            assert np.array_equal(perm_na, ref.perm), T
            idx = torch.from_numpy(sel).cuda()
            off_h = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
            perm_h = torch.full((T * k,), -1, dtype=torch.int32, device="cuda")
            fm.flint_moe_bucket(h, idx, T, off_h, perm_h)
            torch.cuda.synchronize()
            assert np.array_equal(off_h.cpu().numpy(), off_na), T
            assert np.array_equal(perm_h.cpu().numpy(), perm_na), T
    finally:
        fm.flint_moe_destroy(h)


@pytest.mark.parametrize("E,k,T", [(32, 1, 5000), (96, 5, 1001), (200, 8, 777), (256, 6, 1), (1, 1, 3000),
                                   (256, 8, 65536)])
def test_bucket_noalloc_other_expert_counts(fm, E, k, T):
    """Expert counts and top-k values other than the Flint shape; the last case
    is the T*k limit of the scratch (524288 assignments)."""
    if E == 1:
        sel = np.zeros((T, k), dtype=np.int32)
    elif T * k > 100000:
        rng = np.random.default_rng(5)
        sel = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    else:
        sel = _selection(T, k, E, 100 + E + k)
    ref = M.bucket(sel, E)
    off, perm = _noalloc(fm, sel, T, k, E)
    assert np.array_equal(off, ref.offsets)
    assert np.array_equal(perm, ref.perm)


def test_bucket_noalloc_drops_out_of_range_indices(fm):
    """Out-of-range expert indices are dropped, as documented: offsets[E]
    falls short of T*k by their number, and the valid assignments are placed
    as the oracle places them among themselves."""
    E, k, T = 64, 4, 300
    sel = _selection(T, k, E, 7)
    bad = [(3, 1, -1), (10, 0, E), (299, 3, 1000)]
    for t, j, v in bad:
        sel[t, j] = v
    off, perm = _noalloc(fm, sel, T, k, E)
    assert int(off[E]) == T * k - len(bad)
    flat = sel.reshape(-1)
    ok = (flat >= 0) & (flat < E)
    keep = np.nonzero(ok)[0]
    order = keep[np.lexsort((keep, flat[keep]))]
    assert np.array_equal(perm[:off[E]], order)
    counts = np.bincount(flat[ok], minlength=E)
    assert np.array_equal(off, np.concatenate([[0], np.cumsum(counts)]))


def test_bucket_noalloc_rejects_sizes_beyond_its_scratch(fm):
    k = 8
    T = (1 << 19) // k + 1                       # one token past the 524288-assignment limit
    with pytest.raises(fm.FlintError) as ei:
        fm.flint_moe_bucket_noalloc(None, T, k, 256, None, None, stream=0)
    assert ei.value.code == fm.FLINT_EINVAL
    with pytest.raises(fm.FlintError) as ei:
        fm.flint_moe_bucket_noalloc(None, 4, 6, 257, None, None, stream=0)   # E above 256
    assert ei.value.code == fm.FLINT_EINVAL
