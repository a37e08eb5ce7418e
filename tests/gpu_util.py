"""Shared helpers for the GPU parity tests (imported by tests only)."""
import numpy as np

from oracle import vfy_oracle as O

ATOL = 2e-2          # attention tolerance: |gpu - oracle| <= ATOL + RTOL * |oracle| elementwise
RTOL = 1e-2
NORMWISE = 1e-2      # and ||gpu - oracle||_2 / ||oracle||_2 <= NORMWISE


def attn_errors(got_bits, ref):
    g = O.bf16_to_f64(got_bits)
    diff = np.abs(g - ref)
    excess = diff - (ATOL + RTOL * np.abs(ref))
    nrm = np.linalg.norm(ref)
    normwise = np.linalg.norm(g - ref) / nrm if nrm > 0 else np.linalg.norm(g)
    return float(excess.max(initial=-1.0)), float(normwise), float(diff.max(initial=0.0))


def assert_attn_close(got_bits, ref, what=""):
    excess, normwise, maxabs = attn_errors(got_bits, ref)
    assert np.all(np.isfinite(O.bf16_to_f64(got_bits))), f"{what}: non-finite output"
    assert excess <= 0, f"{what}: elementwise tolerance exceeded, max abs err {maxabs:.3e}"
    assert normwise <= NORMWISE, f"{what}: normwise error {normwise:.3e}"


def assert_lse_close(got, ref, what=""):
    fin = np.isfinite(ref)
    assert np.array_equal(np.isneginf(got), np.isneginf(ref)), f"{what}: -inf pattern differs"
    if fin.any():
        err = np.abs(got[fin] - ref[fin])
        assert err.max() <= 2e-3 + 1e-3 * np.abs(ref[fin]).max(), f"{what}: LSE err {err.max():.3e}"
