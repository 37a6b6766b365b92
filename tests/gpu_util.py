"""Shared helpers of the GPU parity tests: tolerances and comparisons.

The stated bound for every attention output is, elementwise,
|got - want| <= 1e-2 (MAX_ABS), with relative L2 <= 5e-3 when P is bf16 or
fp32 and <= 2e-2 when P enters P.V as FP8.  The outputs are bf16: at
|want| >= 4 the rounding of the exact result to bf16 alone can move it by
up to 2^-8 |want| > 1e-2 (half an ulp), so only there the bound adds that
half ulp.  Below 4 (every output of an N(0,1) workload but a few rows that
see one or two keys) it is the plain 1e-2.

With QPKV_PARITY_LOG set to a file name, every comparison appends one line
(test name, max-abs error, rel-L2) to it: the record of achieved errors.
"""
import json
import os

import numpy as np

MAX_ABS = 1e-2
BF16_REL = 2.0 ** -8
BF16_EXEMPT_FROM = 4.0
REL_L2 = 5e-3
REL_L2_FP8_P = 2e-2
# The FP8 decode additionally meets a tighter bound: its probabilities keep
# ~12 bits, so the error is the output's bf16 rounding plus at most 2e-3.
DECODE_TIGHT = 2e-3
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


def _record(what, max_abs, r):
    path = os.environ.get("QPKV_PARITY_LOG")
    if not path:
        return
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    with open(path, "a") as f:
        f.write(json.dumps({"test": test, "what": what, "max_abs": max_abs, "rel_l2": r}) + "\n")


def assert_attention_close(got, want, rel=REL_L2, max_abs=MAX_ABS, tight=None, what="O"):
    """Elementwise |got - want| <= max_abs (+ bf16 half ulp at |want| >= 4),
    rel-L2 <= rel, and with ``tight`` also |got - want| - 2^-8 |want| <= tight."""
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.isfinite(got).all(), f"{what}: non-finite values"
    err = np.abs(got - want)
    r = rel_l2(got, want)
    m = float(err.max()) if got.size else 0.0
    _record(what, m, r)
    allow = np.where(np.abs(want) >= BF16_EXEMPT_FROM, BF16_REL * np.abs(want), 0.0)
    over = float((err - allow).max()) if got.size else 0.0
    assert over <= max_abs and r <= rel, (
        f"{what}: max-abs {m:.3e} (bound {max_abs}, bf16 half ulp added only at |want| >= 4: "
        f"{over:.3e}), rel-L2 {r:.3e} (<= {rel})")
    if tight is not None and got.size:
        t = float((err - BF16_REL * np.abs(want)).max())
        assert t <= tight, f"{what}: |err| - 2^-8 |want| = {t:.3e} > {tight}"


def assert_lse_close(got, want, atol=LSE_ATOL):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    inf_w = np.isneginf(want)
    assert np.array_equal(np.isneginf(got), inf_w), "lse: -inf pattern differs"
    if (~inf_w).any():
        err = float(np.max(np.abs(got[~inf_w] - want[~inf_w])))
        assert err <= atol, f"lse max-abs {err:.3e} > {atol}"
