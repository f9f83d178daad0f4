"""GPU parity over the full shape sweep of single products that exercises the
takes_sgemm boundaries (page f16.md, Technical usage: ncols >= 2 && rows % 4 == 0 &&
k % 8 == 0): rows in {12, 13, 4096, 14336} x k in {8, 31, 33, 1536, 4097, 8192} x
columns in {1, 2, 5, 512}, weights N(0, 0.02), activations N(0, 1) rounded to f16.

Every case goes through bm_f16_matmul and is held to its path's contract: vec_dot's
bits for one column and where takes_sgemm fails; tinyBLAS's bits on the bit-exact
kernel (up to bm_set_exact_sgemm_cols columns, default 2); the 4e-6 * sum|w*a| bound
on the tensor cores, whose cases run a second time with balanced k ranges forced.
Products the oracle finishes in seconds are compared whole, larger ones on a sample
that always holds the four corners."""
import functools
import itertools

import numpy as np
import pytest

import oracle
import synth
from conftest import bits32, to_dev

pytestmark = pytest.mark.gpu

ROWS, KS, NCOLS = (12, 13, 4096, 14336), (8, 31, 33, 1536, 4097, 8192), (1, 2, 5, 512)
TOL = 4e-6


@functools.lru_cache(maxsize=2)
def weights(rows, k):
    W = synth.normal_f16(0, "sweep.w.%d.%d" % (rows, k), 0.02, (rows, k))
    return W, to_dev(W)


def activations(k, ncols):
    return oracle.to_f16(synth.normal_f32(0, "sweep.x.%d" % k, 1.0, (ncols, k)))


@pytest.mark.parametrize("rows,k,ncols", list(itertools.product(ROWS, KS, NCOLS)))
def test_sweep(bm, rows, k, ncols):
    W, dW = weights(rows, k)
    X = activations(k, ncols)
    Y = bits32(bm.bm_f16_matmul(dW, to_dev(X))).reshape(ncols, rows)
    sgemm = bool(bm.bm_takes_sgemm(rows, k, ncols))
    assert sgemm == oracle.takes_sgemm(rows, k, ncols)
    cur = bm.bm_set_exact_sgemm_cols(0)  # read the setting in force and put it back
    bm.bm_set_exact_sgemm_cols(cur)
    exact = not sgemm or ncols <= cur
    if rows * k * ncols <= 2e8:
        ref = oracle.matmul(W, X)
        if exact:
            assert np.array_equal(Y, bits32(ref))
        else:
            err = np.abs(Y.view(np.float32).astype(np.float64) - ref.astype(np.float64))
            assert (err <= TOL * oracle.abs_matmul(W, X)).all()
        return
    rng = np.random.default_rng(rows * 7 + k * 3 + ncols)
    ri = np.concatenate([[0, rows - 1, 0, rows - 1], rng.integers(0, rows, 3000)])
    ci = np.concatenate([[0, ncols - 1, ncols - 1, 0], rng.integers(0, ncols, 3000)])
    ref, ab = oracle.matmul_sample(W, X, ri, ci, with_absdot=not exact)
    got = Y[ci, ri]
    if exact:
        assert np.array_equal(got, bits32(ref))
    else:
        err = np.abs(got.view(np.float32).astype(np.float64) - ref.astype(np.float64))
        assert (err <= TOL * ab).all()


@pytest.mark.parametrize("rows,k,ncols", [s for s in itertools.product(ROWS, KS, NCOLS)
                                           if s[2] > 2 and oracle.takes_sgemm(*s)])
def test_sweep_with_balanced_k_ranges(bm, rows, k, ncols):
    """The tensor-core cases of the sweep again with balanced k ranges forced (bm_set_stream_k(1)):
    the same bound against tinyBLAS's element."""
    old = bm.bm_set_stream_k(1)
    try:
        W, dW = weights(rows, k)
        X = activations(k, ncols)
        Y = bits32(bm.bm_f16_matmul(dW, to_dev(X))).reshape(ncols, rows).view(np.float32)
    finally:
        bm.bm_set_stream_k(old)
    if rows * k * ncols <= 2e8:
        ref = oracle.matmul(W, X)
        err = np.abs(Y.astype(np.float64) - ref.astype(np.float64))
        assert (err <= TOL * oracle.abs_matmul(W, X)).all()
        return
    rng = np.random.default_rng(rows * 11 + k + ncols)
    ri = np.concatenate([[0, rows - 1, 0, rows - 1], rng.integers(0, rows, 3000)])
    ci = np.concatenate([[0, ncols - 1, ncols - 1, 0], rng.integers(0, ncols, 3000)])
    ref, ab = oracle.matmul_sample(W, X, ri, ci, with_absdot=True)
    err = np.abs(Y[ci, ri].astype(np.float64) - ref.astype(np.float64))
    assert (err <= TOL * ab).all()
    assert bm.bm_device_status() == 0
