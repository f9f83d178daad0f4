"""Pins of the oracle's rms_norm then mul (page "docs/modules/forward.md", Technical
usage, "Other public pieces"; How it is verified, rms_norm_of_a_constant_row) against
closed forms and invariants (tests/norm_cases.py), plus rows that go through the
multi-row entry one by one."""
import numpy as np

import norm_cases
import oracle


def test_closed_forms_and_invariants():
    assert norm_cases.failures(lambda x, w, eps: oracle.rms_norm_mul(x, w, eps)) == []


def test_rows_are_independent():
    rng = np.random.default_rng(3)
    X = rng.normal(0, 1, (5, 96)).astype(np.float32)
    X[2] *= 1000.0
    X[3] = 0.25
    w = rng.normal(0, 1, 96).astype(np.float32)
    Y = oracle.rms_norm_mul(X, w, 1e-5)
    for r in range(5):
        assert np.array_equal(Y[r].view(np.uint32), oracle.rms_norm_mul(X[r], w, 1e-5).view(np.uint32))


def test_close_to_the_real_formula():
    """Within a few f32 ulps of x / sqrt(mean(x^2) + eps) * w computed in long double
    precision (the roundings the reading adds are a handful of ulps at most)."""
    rng = np.random.default_rng(4)
    for n in (1, 9, 576, 4096):
        x = rng.normal(0, 3, n).astype(np.float32)
        w = rng.normal(0, 1, n).astype(np.float32)
        eps = 1e-6
        ref = x.astype(np.float64) / np.sqrt(np.mean(x.astype(np.float64) ** 2) + np.float32(eps)) * w
        got = oracle.rms_norm_mul(x, w, eps).astype(np.float64)
        assert np.all(np.abs(got - ref) <= 4 * np.spacing(np.abs(ref).astype(np.float32)).astype(np.float64) + 1e-30)
