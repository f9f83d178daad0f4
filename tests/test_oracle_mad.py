"""Pins of the oracle's attention accumulator helpers (page "docs/modules/f16.md",
Technical usage: `mad` is ggml_vec_mad_f16, the V accumulator of flash attention;
`scale` is ggml_vec_scale_f16), checked against numpy's own IEEE arithmetic and its
float32 -> float16 conversion (nearest-even), which share nothing with the oracle.

- scale: one f32 multiply then f16 -- numpy's float32 product and astype(float16)
  give the reference for every f16 value and several scales, including powers of two
  (exact scaling into the subnormals and overflow to infinity).
- mad: one fused multiply-add in f32 then f16 (the reading taken where the page is
  silent).  Where the exact value acc + v*w is representable in double (the two terms
  within 2^+-15 of each other: at most 35 + 30 + 11 bits), rounding it once to float32
  is the fused result, so numpy's double sum rounded to float32 then float16 is an
  independent reference.  Closed forms: w = 0 leaves a non-zero acc unchanged; small
  integers give exact integer sums."""
import numpy as np
import pytest

import oracle

ALL = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
FINITE = ALL[np.isfinite(ALL.view(np.float16))]


def np_f16(x32):
    with np.errstate(over="ignore"):
        return np.asarray(x32, dtype=np.float32).astype(np.float16).view(np.uint16)


def test_scale_by_one_is_the_identity_on_every_value():
    nonnan = ALL[~np.isnan(ALL.view(np.float16))]
    assert np.array_equal(oracle.f16_scale(nonnan, 1.0), nonnan)


@pytest.mark.parametrize("s", [2.0, 0.5, 2.0 ** -20, 2.0 ** 14, -3.0, 0.1, 1.0 / 3.0, 1e-3, 123.456])
def test_scale_matches_numpy_float32_then_float16(s):
    x = FINITE.view(np.float16).astype(np.float32)
    with np.errstate(over="ignore"):
        want = np_f16(x * np.float32(s))
    assert np.array_equal(oracle.f16_scale(FINITE, s), want)


def test_mad_matches_the_exact_sum_rounded_once():
    rng = np.random.default_rng(11)
    n = 200000
    e_acc = rng.integers(-12, 12, n)
    acc = np_f16(rng.uniform(1, 2, n) * np.exp2(e_acc) * rng.choice([-1, 1], n))
    v = np_f16(rng.uniform(1, 2, n) * np.exp2(rng.integers(-6, 6, n)) * rng.choice([-1, 1], n))
    w = np.float32(rng.uniform(0.5, 1.0) * 0.7)
    got = np.empty(n, np.uint16)
    # one w per call, as the helper takes it
    got[:] = oracle.f16_mad(acc, v, w)
    a64 = acc.view(np.float16).astype(np.float64)
    p64 = v.view(np.float16).astype(np.float64) * np.float64(w)  # exact: 11 x 24 bits
    keep = np.abs(np.log2(np.abs(a64)) - np.log2(np.abs(p64) + 1e-300)) < 15  # the sum is exact in double
    want = np_f16((a64 + p64).astype(np.float32))
    assert keep.sum() > n // 2
    assert np.array_equal(got[keep], want[keep])


def test_mad_closed_forms():
    rng = np.random.default_rng(12)
    acc = FINITE[FINITE.view(np.float16) != 0]
    v = rng.choice(FINITE, acc.size)
    assert np.array_equal(oracle.f16_mad(acc, v, 0.0), acc)  # + (+-0): a non-zero value stays
    ai = rng.integers(-100, 100, 5000)
    vi = rng.integers(-100, 100, 5000)
    out = oracle.f16_mad(np_f16(ai), np_f16(vi), 3.0).view(np.float16).astype(np.float64)
    assert np.array_equal(out, (ai + 3 * vi).astype(np.float64))  # |sum| <= 400: exact in f16


def test_mad_is_one_rounding_not_two():
    """The reading: the product and the sum round once together.  Near cancellation
    (acc close to -v*w) the f32 rounding of a separate product can survive the final
    f16 rounding; on such cases the oracle gives the fused value (the exact double sum
    rounded once), not the two-step one."""
    rng = np.random.default_rng(13)
    n = 400000
    v = np_f16(rng.uniform(1, 2, n))
    w = np.float32(1.0 + rng.uniform(0, 2.0 ** -9))
    prod = v.view(np.float16).astype(np.float64) * np.float64(w)  # exact
    acc = np_f16(-prod.astype(np.float32))  # acc close to -v*w
    a64 = acc.view(np.float16).astype(np.float64)
    fused = np_f16((a64 + prod).astype(np.float32))  # the double sum is exact here
    two = np_f16((prod.astype(np.float32) + a64.astype(np.float32)).astype(np.float32))
    differ = fused != two
    assert differ.sum() > 0
    got = oracle.f16_mad(acc, v, w)
    assert np.array_equal(got[differ], fused[differ])
    assert np.array_equal(got, fused)


def test_mad_and_scale_specials():
    inf, ninf, nan = np_f16(np.inf)[()], np_f16(-np.inf)[()], np.uint16(0x7E00)
    one = np_f16(1.0)[()]
    assert oracle.f16_scale(np.array([inf], np.uint16), 2.0)[0] == inf
    assert oracle.f16_scale(np.array([inf], np.uint16), -1.0)[0] == ninf
    assert np.isnan(oracle.f16_mad(np.array([one], np.uint16), np.array([inf], np.uint16), 0.0).view(np.float16)[0])
    assert np.isnan(oracle.f16_mad(np.array([nan], np.uint16), np.array([one], np.uint16), 1.0).view(np.float16)[0])
    assert oracle.f16_mad(np.array([np_f16(65504.0)[()]], np.uint16), np.array([np_f16(16.0)[()]], np.uint16),
                          1.0)[0] == inf  # 65520 rounds to infinity
