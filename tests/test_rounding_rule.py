"""The quantiser's division-free rounding rule, checked in IEEE float32 on
the host: with inv = fl(1/S) and y = fl(r inv), rint(y) equals
rint(fl(r / S)) unless y lies within |y| 2^-21 of a half-integer, where the
kernel takes the division itself.  Random (r, S) with S an fp16 value, and
r built to land a few ulps from half-integers, for INT2 and INT4 clamps."""
import numpy as np
import pytest


def _ieee(r, S, qmax):
    return np.clip(np.rint((r / S).astype(np.float32)), -qmax - 1, qmax)


def _rule(r, S, qmax):
    inv = (np.float32(1) / S).astype(np.float32)
    y = (r * inv).astype(np.float32)
    t = np.rint(y)
    near = (np.float32(0.5) - np.abs((y - t).astype(np.float32))) <= (np.abs(y) * np.float32(2.0 ** -21))
    t = np.where(near, np.rint((r / S).astype(np.float32)), t)
    return np.clip(t, -qmax - 1, qmax), near.mean()


@pytest.mark.parametrize("bits", [2, 4])
def test_division_free_codes_equal_ieee(bits):
    rng = np.random.default_rng(bits)
    qmax = np.float32((1 << (bits - 1)) - 1)
    S = rng.uniform(1e-3, 60.0, 1_000_000).astype(np.float16).astype(np.float32)
    S = S[S > 0]
    r = (rng.uniform(-qmax - 1.6, qmax + 1.6, S.size) * S).astype(np.float32)
    got, rate = _rule(r, S, qmax)
    np.testing.assert_array_equal(got, _ieee(r, S, qmax))
    assert rate < 1e-4
    # a few ulps either side of (k + 1/2) S, and exactly on it
    k = rng.integers(-int(qmax) - 2, int(qmax) + 2, S.size).astype(np.float32)
    base = ((k + np.float32(0.5)) * S).astype(np.float32)
    for steps in (0, 1, 3, 8):
        rr = base
        for _ in range(steps):
            rr = np.nextafter(rr, np.where(k >= 0, np.inf, -np.inf).astype(np.float32)).astype(np.float32)
        np.testing.assert_array_equal(_rule(rr, S, qmax)[0], _ieee(rr, S, qmax))
    # scales saturated at the fp16 maximum, and huge quotients (clamped)
    big = np.full(1000, 65504.0, np.float32)
    rr = (rng.standard_normal(1000) * 1e9).astype(np.float32)
    np.testing.assert_array_equal(_rule(rr, big, qmax)[0], _ieee(rr, big, qmax))
