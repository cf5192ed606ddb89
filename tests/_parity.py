"""Comparison helpers shared by the GPU parity tests (no arithmetic of the method)."""

import numpy as np

MAX_ABS = 2e-2        # bf16 / tf32 outputs: max abs error
REL_FRO = 5e-3        # relative Frobenius error
LSE_ABS = 1e-3        # LSE abs error


def to_np(t):
    return t.detach().double().cpu().numpy()


def assert_attention_close(got, ref, got_lse=None, ref_lse=None, what=""):
    """Rows with LSE = -inf must match exactly with zero output; everything else
    within the tolerances above."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    if ref_lse is not None:
        got_lse = np.asarray(got_lse, dtype=np.float64)
        ref_lse = np.asarray(ref_lse, dtype=np.float64)
        empty = np.isneginf(ref_lse)
        assert np.array_equal(np.isneginf(got_lse), empty), f"{what}: -inf LSE rows differ"
        assert np.all(got[empty] == 0.0), f"{what}: empty rows must be zero"
        fin = ~empty
        lerr = np.abs(got_lse[fin] - ref_lse[fin]).max() if fin.any() else 0.0
        assert lerr <= LSE_ABS, f"{what}: LSE max abs error {lerr:.3g}"
    err = np.abs(got - ref).max() if got.size else 0.0
    denom = np.linalg.norm(ref)
    rel = np.linalg.norm(got - ref) / denom if denom > 0 else np.linalg.norm(got)
    assert err <= MAX_ABS, f"{what}: max abs error {err:.3g}"
    assert rel <= REL_FRO, f"{what}: relative Frobenius error {rel:.3g}"
    return err, rel
