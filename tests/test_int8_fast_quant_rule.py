"""The INT8 cache write's fast quantisation rule, replayed on the CPU.

The write kernel codes y / s, with s = float32(amax / 127), as
RNE(float32(y * inv)) with inv = float32(127 * float32(1 / amax)). It does
so whenever that product is at most 0.4999 from its integer and s lies in
[1e-30, 1e30]; otherwise it takes the correctly rounded float32 division.
numpy's float32 arithmetic (IEEE, round to nearest even) replays both paths
here. Wherever the rule takes the fast code, it must equal the division's
code. The inputs are blocks of random values over 40 decades, plus values
placed inside and at the edges of the 1e-4 band around every half-integer.
No GPU; the GPU tests compare the kernel's bytes with the oracle."""
import numpy as np

F32 = np.float32
NEAR_HALF = F32(0.4999)


def _both_paths(y, amax):
    """(fast code, |product - fast code|, division code, fast path usable)."""
    s = F32(amax) / F32(127)
    inv = F32(127) * (F32(1) / F32(amax))
    p = (y * inv).astype(F32)
    fast = np.rint(p)
    dev = np.abs((p - fast).astype(F32))
    exact = np.clip(np.rint((y / s).astype(F32)), -127, 127)
    usable = F32(1e-30) <= s <= F32(1e30)
    return fast, dev, exact, usable


def _check_block(y):
    amax = F32(np.abs(y).max())
    if amax == 0:
        return 0, 0
    fast, dev, exact, usable = _both_paths(y, amax)
    if not usable:
        return 0, y.size
    take = dev <= NEAR_HALF
    assert np.array_equal(fast[take], exact[take])
    assert np.abs(fast[take]).max() <= 127
    return int(take.sum()), int((~take).sum())


def test_fast_codes_equal_the_division_on_random_blocks():
    rng = np.random.default_rng(20240611)
    taken = 0
    for _ in range(300):
        mag = F32(10.0) ** F32(rng.uniform(-20, 20))
        y = (rng.standard_normal(16384) * mag).astype(F32)
        t, _ = _check_block(y)
        taken += t
    assert taken > 4_000_000


def test_fast_codes_equal_the_division_next_to_half_integers():
    """Quotients k + 1/2 + d with |d| up to 2e-4, the band's edges included:
    the product decides where it is clear of the band, the division inside."""
    rng = np.random.default_rng(7)
    taken = fallback = 0
    for _ in range(200):
        amax = F32(rng.uniform(0.5, 2.0)) * F32(10.0) ** F32(rng.integers(-12, 12))
        s = F32(amax) / F32(127)
        k = rng.integers(-127, 127, 20000).astype(np.float64)
        d = np.concatenate([rng.uniform(-2e-4, 2e-4, 16000),
                            np.repeat([-1e-4, 1e-4, -1.2e-4, 1.2e-4], 1000)])
        y = ((k + 0.5 + d) * float(s)).astype(F32)
        y = np.clip(y, -amax, amax)
        y[0] = amax                                    # the block's maximum
        t, f = _check_block(y)
        taken += t
        fallback += f
    assert taken > 1_000_000 and fallback > 100_000


def test_exact_half_integer_quotients_take_the_division():
    """s a power of two: y = (k + 1/2) s exactly, a tie that RNE sends to the
    even code; the product is a tie too, so the rule must route it to the
    division, which agrees."""
    for e in (-20, -3, 0, 5):
        s = F32(2.0) ** e
        amax = F32(127) * s
        k = np.arange(-127, 127, dtype=np.float64)
        y = np.concatenate([((k + 0.5) * float(s)).astype(F32), [amax]]).astype(F32)
        fast, dev, exact, usable = _both_paths(y, amax)
        assert usable
        ties = dev[:-1] > NEAR_HALF
        assert ties.all()
        assert np.array_equal(exact[:-1], np.rint(k + 0.5))
