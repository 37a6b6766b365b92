"""Shared helpers of the GPU parity tests: tolerances and comparisons."""
import numpy as np

# Attention output against the float64 oracle: elementwise |got - want| <=
# ATOL_MAX + BF16_REL * |want| (a bf16 output carries 8 significant bits, so
# rounding alone moves it by up to 2^-8 of its magnitude) and relative L2
# with P in bf16 / fp32 (the FP8-P bound is looser); LSE absolute.
ATOL_MAX = 2e-3
BF16_REL = 2.0 ** -8
# The stated bound with P in bf16 (max-abs 1e-2), used where a row may see
# only a few keys: bf16 rounding of P then moves O by up to ~2^-9 |v|.
ATOL_P_BF16 = 1e-2
REL_L2 = 5e-3
REL_L2_FP8_P = 2e-2
# Elementwise guard where P enters P.V as two E4M3 terms: below 2^-6 the
# terms are subnormal, the low term's step is 2^-10, so each key can move O
# by ~2^-10 |v| (|v| up to ~4 here) beyond the 2^-8 relative rounding.
ATOL_P_FP8 = 2e-2
LSE_ATOL = 1e-3


def bf16_to_f64(t):
    """torch bf16 tensor (any device) -> float64 numpy."""
    import torch
    return t.detach().to("cpu", torch.float32).numpy().astype(np.float64)


def rel_l2(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    den = np.linalg.norm(want)
    return float(np.linalg.norm(got - want) / (den if den > 0 else 1.0))


def assert_attention_close(got, want, rel=REL_L2, atol=ATOL_MAX, what="O"):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    excess = np.abs(got - want) - BF16_REL * np.abs(want)
    err = float(np.max(excess)) if got.size else 0.0
    r = rel_l2(got, want)
    assert err <= atol and r <= rel, (
        f"{what}: max(|err| - 2^-8 |want|) {err:.3e} (<= {atol}), rel-L2 {r:.3e} (<= {rel})")


def assert_lse_close(got, want, atol=LSE_ATOL):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    inf_w = np.isneginf(want)
    assert np.array_equal(np.isneginf(got), inf_w), "lse: -inf pattern differs"
    if (~inf_w).any():
        err = float(np.max(np.abs(got[~inf_w] - want[~inf_w])))
        assert err <= atol, f"lse max-abs {err:.3e} > {atol}"
