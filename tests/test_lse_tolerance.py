"""The log-sum-exp tolerance of the attention checks (tests/_helpers.py,
lse_tolerance) is a bound, not a fit: on random rows it holds for the LSE
computed the way the kernel rounds its operands (keys and weights to fp16,
queries already exact in fp16), against the fp64 LSE of the same keys."""
import numpy as np

from _helpers import lse_tolerance


def _lse(s):
    m = s.max(axis=-1, keepdims=True)
    return (m + np.log(np.exp(s - m).sum(axis=-1, keepdims=True)))[..., 0]


def test_lse_tolerance_bounds_fp16_operand_rounding():
    rng = np.random.default_rng(5)
    worst = 0.0
    for trial in range(6):
        d, nq, nk = (64, 128)[trial % 2], 48, 300
        q = rng.standard_normal((nq, 1, d)) * 3.0
        q = q.astype(np.float16).astype(np.float64)          # the queries enter exactly
        k = rng.standard_normal((nk, 1, d)) * (1.0 + 20.0 * (rng.random((nk, 1, 1)) < 0.02))
        scale = 1.0 / np.sqrt(d)
        s_ref = scale * (q[:, 0] @ k[:, 0].T)
        k16 = k.astype(np.float16).astype(np.float64)        # K_hat rounded to fp16
        s16 = scale * (q[:, 0] @ k16[:, 0].T)
        m = s16.max(axis=1, keepdims=True)
        p16 = np.exp(s16 - m).astype(np.float16).astype(np.float64)   # weights rounded to fp16
        lse16 = m[:, 0] + np.log(p16.sum(axis=1))
        err = np.abs(lse16 - _lse(s_ref))
        tol = lse_tolerance(q, np.abs(k), 1)[0]
        assert (err <= tol).all(), (trial, (err - tol).max())
        worst = max(worst, float((err / tol).max()))
    assert worst < 1.0
