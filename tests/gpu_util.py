"""Helpers for the GPU parity tests: tolerances and routing comparison."""
import numpy as np

from oracle import formats as F

# Output tolerance of the layer: relative L2 error <= 5e-3 and max abs error
# <= 3e-2 x RMS of the reference output. Router logits: |dL| <= 1e-4 x
# max(|L_ref|, RMS of the reference row).
OUT_REL_L2 = 5e-3
OUT_MAX_ABS_RMS = 3e-2
LOGIT_REL = 1e-4


def assert_out_close(got_bf16_bits: np.ndarray, ref: np.ndarray, what: str = "out") -> dict:
    got = F.bf16_array(got_bf16_bits)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = got - ref
    rms = float(np.sqrt(np.mean(ref ** 2)))
    rel_l2 = float(np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-300))
    max_abs = float(np.max(np.abs(err))) if err.size else 0.0
    stats = dict(rel_l2=rel_l2, max_abs=max_abs, rms=rms)
    assert rel_l2 <= OUT_REL_L2, f"{what}: rel L2 {rel_l2:.3e} > {OUT_REL_L2} ({stats})"
    assert max_abs <= OUT_MAX_ABS_RMS * rms, f"{what}: max abs {max_abs:.3e} > 3e-2*rms ({stats})"
    return stats


def assert_logits_close(got: np.ndarray, ref: np.ndarray) -> float:
    rms = np.sqrt(np.mean(ref ** 2, axis=1, keepdims=True))
    scale = np.maximum(np.abs(ref), rms)
    worst = float(np.max(np.abs(got - ref) / scale))
    assert worst <= LOGIT_REL, f"router logits: worst relative error {worst:.3e}"
    return worst


def compare_routing(got_idx: np.ndarray, ref_sel: np.ndarray, ref_logits: np.ndarray, k: int) -> np.ndarray:
    """The GPU's selection must equal the oracle's, except where reference
    logits are so close (within the logit tolerance) that float32 summation
    order may legitimately swap them: then the GPU list must still be a valid
    descending top-k of the reference logits within that tolerance. Returns
    the mask of tokens whose selected set equals the oracle's (the ones an
    output comparison is meaningful for)."""
    got_idx = np.asarray(got_idx)
    T = ref_logits.shape[0]
    rms = np.sqrt(np.mean(ref_logits ** 2, axis=1))
    same_set = np.zeros(T, dtype=bool)
    for t in range(T):
        if np.array_equal(got_idx[t], ref_sel[t]):
            same_set[t] = True
            continue
        tol = LOGIT_REL * max(float(np.max(np.abs(ref_logits[t]))), float(rms[t]))
        g = ref_logits[t, got_idx[t]]
        kth = np.sort(ref_logits[t])[::-1][k - 1]
        assert len(set(got_idx[t].tolist())) == k, f"token {t}: repeated expert"
        assert np.all(g >= kth - 2 * tol), f"token {t}: selected a non-top expert {got_idx[t]} vs {ref_sel[t]}"
        assert np.all(np.diff(g) <= 2 * tol), f"token {t}: not in descending order {got_idx[t]}"
        same_set[t] = set(got_idx[t].tolist()) == set(ref_sel[t].tolist())
    return same_set
