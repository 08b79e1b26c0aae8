"""The block-scaled FP4 tensor-core GEMM (tcgen05 kind::mxf4nvf4) against the
dequantised product computed by the oracle's NVFP4 decoder."""
import numpy as np
import pytest

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


def _operand(rng, R, K):
    codes = rng.integers(0, 256, size=(R, K // 2), dtype=np.uint8)
    scales = rng.integers(0x28, 0x48, size=(R, K // 16), dtype=np.uint8)
    return codes, scales


def _diagnose(got, a, b):
    """Which of a few plausible layout slips the result matches (for the
    failure message only)."""
    ac, asc = a
    bc, bsc = b
    out = []

    def swap(c):
        return ((c & 0xF) << 4) | (c >> 4)

    def rev_scales(s):
        return s.reshape(s.shape[0], -1, 4)[:, :, ::-1].reshape(s.shape)

    cands = {
        "nibbles swapped": (F.dequant_nvfp4(swap(ac), asc, 1.0), F.dequant_nvfp4(swap(bc), bsc, 1.0)),
        "scale bytes reversed per word": (F.dequant_nvfp4(ac, rev_scales(asc), 1.0),
                                          F.dequant_nvfp4(bc, rev_scales(bsc), 1.0)),
        "no block scales": (F.dequant_nvfp4(ac, np.full_like(asc, 0x38), 1.0),
                            F.dequant_nvfp4(bc, np.full_like(bsc, 0x38), 1.0)),
    }
    for name, (A, B) in cands.items():
        ref = A @ B.T
        out.append(f"{name}: rel {np.max(np.abs(got - ref)) / np.max(np.abs(ref)):.2e}")
    return "; ".join(out)


@pytest.mark.parametrize("M,N,K", [(128, 128, 256), (256, 128, 512), (128, 384, 1024), (512, 256, 2048), (4096, 1024, 512)])
def test_fp4_gemm_matches_dequantised_product(fm, M, N, K):
    rng = np.random.default_rng(M * 7 + N * 3 + K)
    a = _operand(rng, M, K)
    b = _operand(rng, N, K)
    dev = [torch.from_numpy(x).cuda() for x in (*a, *b)]
    d = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    fm.flint_moe_debug_fp4_gemm(dev[0], dev[1], dev[2], dev[3], M, N, K, d)
    torch.cuda.synchronize()
    got = d.cpu().numpy().astype(np.float64)
    A = F.dequant_nvfp4(a[0], a[1], 1.0)
    B = F.dequant_nvfp4(b[0], b[1], 1.0)
    ref = A @ B.T
    assert np.all(np.isfinite(got)), "non-finite output"
    rel = float(np.max(np.abs(got - ref)) / np.max(np.abs(ref)))
    assert rel <= 1e-5, f"relative error {rel:.3e}; " + _diagnose(got, a, b)
