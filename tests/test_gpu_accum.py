"""GPU parity of bm_f16_mad and bm_f16_scale (page "docs/modules/f16.md", Technical
usage: `mad` is ggml_vec_mad_f16, flash attention's V accumulator; `scale` is
ggml_vec_scale_f16) against the oracle, bit for bit on every non-NaN result: random
accumulators across the f16 range (subnormals, values near cancellation, overflow to
infinity), the 8-wide path and the one-element path (a 2-byte offset), ragged ends,
v aliasing acc, and n = 0."""
import numpy as np
import pytest

import oracle
from conftest import to_dev

pytestmark = pytest.mark.gpu


def f16(x):
    with np.errstate(over="ignore"):
        return np.asarray(x, np.float32).astype(np.float16).view(np.uint16)


def inputs(n, seed):
    rng = np.random.default_rng(seed)
    mag = np.exp2(rng.uniform(-26, 17, n)) * rng.choice([-1.0, 1.0], n)
    acc = f16(mag)
    v = f16(np.exp2(rng.uniform(-20, 10, n)) * rng.choice([-1.0, 1.0], n))
    half = n // 2
    w = np.float32(rng.uniform(0.3, 3.0))
    # near cancellation in half of them: acc ~ -v * w
    acc[:half] = f16(-(v[:half].view(np.float16).astype(np.float64) * np.float64(w)).astype(np.float32))
    return acc, v, w


def same(got, want):
    g, w_ = got.view(np.float16), want.view(np.float16)
    both_nan = np.isnan(g) & np.isnan(w_)
    return bool(np.all((got == want) | both_nan))


def dev_u16(a, offset=0):
    """a device f16 copy of `a`, starting `offset` elements into a larger buffer."""
    import torch
    buf = torch.zeros(a.size + offset + 8, dtype=torch.float16, device="cuda")
    t = buf[offset:offset + a.size]
    t.copy_(to_dev(a))
    return t


@pytest.mark.parametrize("n", [1, 7, 8, 9, 1000, (1 << 20) + 3])
@pytest.mark.parametrize("offset", [0, 1])
def test_mad_matches_the_oracle(bm, n, offset):
    acc, v, w = inputs(n, n + offset)
    a_dev, v_dev = dev_u16(acc, offset), dev_u16(v, offset)
    bm.bm_f16_mad(a_dev, v_dev, float(w))
    got = a_dev.cpu().numpy().view(np.uint16)
    assert same(got, oracle.f16_mad(acc, v, w))
    assert bm.bm_device_status() == 0


@pytest.mark.parametrize("n", [1, 7, 8, 9, 1000, (1 << 20) + 3])
@pytest.mark.parametrize("offset", [0, 1])
@pytest.mark.parametrize("s", [0.5, 3.0, 0.1, 1000.0, -2.5e-3])
def test_scale_matches_the_oracle(bm, n, offset, s):
    acc, _, _ = inputs(n, 2 * n + offset)
    a_dev = dev_u16(acc, offset)
    bm.bm_f16_scale(a_dev, s)
    got = a_dev.cpu().numpy().view(np.uint16)
    assert same(got, oracle.f16_scale(acc, s))


def test_mad_with_v_equal_to_acc_and_empty(bm):
    import torch
    acc, _, w = inputs(4099, 5)
    a_dev = dev_u16(acc)
    bm.bm_f16_mad(a_dev, a_dev, float(w))  # acc = fma(acc, w, acc)
    assert same(a_dev.cpu().numpy().view(np.uint16), oracle.f16_mad(acc, acc, w))
    e = torch.empty(0, dtype=torch.float16, device="cuda")
    bm.bm_f16_mad(e, e, 1.0)
    bm.bm_f16_scale(e, 1.0)
    assert bm.bm_device_status() == 0


def test_every_f16_value_scaled(bm):
    """scale over all 65,536 patterns (specials included: inf stays inf, NaN stays NaN)."""
    allv = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    for s in (1.0, 0.75, 2.0 ** -12, 2.0 ** 9):
        a_dev = dev_u16(allv)
        bm.bm_f16_scale(a_dev, s)
        assert same(a_dev.cpu().numpy().view(np.uint16), oracle.f16_scale(allv, s))
