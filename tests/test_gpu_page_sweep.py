"""The pages' own verification sweep on the GPU (page f16.md, "How it is verified",
avx2_equals_the_scalar_models): every row length k from 8 to 1,536 (every tail of
k % 32 and k % 64 included), 1 to 6 columns, 12 and 13 rows (both sides of
takes_sgemm), plus 1,540 rows (a multiple of 4 spanning twelve 128-row tiles and a
ragged thirteenth, and 192 eight-row groups and a half group).

Every product goes through bm_f16_matmul and is held to its path's contract against
the oracle: vec_dot's bits for one column and wherever takes_sgemm fails; tinyBLAS's
bits on the exact CUDA-core kernel (2 columns by default, and 3..6 columns again
with bm_set_exact_sgemm_cols(8)); within 4e-6 * sum|w*a| on the tensor cores.
Outputs are NaN-filled before each call."""
import numpy as np
import pytest

import oracle
import synth
from conftest import to_dev

pytestmark = pytest.mark.gpu

TOL = 4e-6
KS = range(8, 1537)


def inputs(rows, k):
    W = synth.normal_f16(0, "page_sweep.w.%d.%d" % (rows, k), 0.02, (rows, k))
    X = oracle.to_f16(synth.normal_f32(0, "page_sweep.x.%d" % k, 1.0, (6, k)))
    return W, X


def sweep(bm, rows, ks, exact_cols):
    """Runs the products of every k in ks and 1..6 columns; returns the counts of
    elements checked bit for bit and within the bound."""
    import torch
    old = bm.bm_set_exact_sgemm_cols(exact_cols)
    n_exact = n_bound = 0
    try:
        for k in ks:
            W, X = inputs(rows, k)
            dW, dX = to_dev(W), to_dev(X)
            Ys = []
            for nc in range(1, 7):
                Y = torch.full((nc, rows), float("nan"), dtype=torch.float32, device="cuda")
                bm.bm_f16_matmul(dW, dX[:nc], Y)
                Ys.append(Y)
            got = [Y.cpu().numpy() for Y in Ys]
            for nc in range(1, 7):
                ref = oracle.matmul(W, X[:nc])
                tensor = oracle.takes_sgemm(rows, k, nc) and nc > exact_cols
                if tensor:
                    err = np.abs(got[nc - 1].astype(np.float64) - ref.astype(np.float64))
                    ok = np.isfinite(got[nc - 1]).all() and (err <= TOL * oracle.abs_matmul(W, X[:nc])).all()
                    assert ok, (rows, k, nc, "tensor cores")
                    n_bound += ref.size
                else:
                    assert np.array_equal(got[nc - 1].view(np.uint32), ref.view(np.uint32)), (rows, k, nc)
                    n_exact += ref.size
    finally:
        bm.bm_set_exact_sgemm_cols(old)
    assert bm.bm_device_status() == 0
    return n_exact, n_bound


@pytest.mark.parametrize("rows", [12, 13, 1540])
def test_every_k_from_8_to_1536(bm, rows):
    """The default path selection (exact tinyBLAS kernel up to 2 columns)."""
    n_exact, n_bound = sweep(bm, rows, KS, 2)
    assert n_exact > 0
    assert (n_bound > 0) == (rows % 4 == 0)


@pytest.mark.parametrize("rows", [12, 1540])
def test_tinyblas_bits_on_every_k_multiple_of_8(bm, rows):
    """takes_sgemm shapes of 3..6 columns on the exact CUDA-core kernel: tinyBLAS's
    bits (f16.md, Design notes, "sgemm_dot") at every k % 8 == 0 from 8 to 1536."""
    n_exact, n_bound = sweep(bm, rows, range(8, 1537, 8), 8)
    assert n_bound == 0 and n_exact > 0


def test_unaligned_rows_every_small_shape(bm):
    """One column, rows not 16-byte aligned (k % 8 != 0): every row count 1..16 and every
    such k from 9 to 100, so every offset of a row from its 16-byte boundary and the
    matrix's last, clamped window occur; vec_dot's bits (f16.md, Design notes, "vec_dot")."""
    import torch
    for rows in range(1, 17):
        for k in (k for k in range(9, 101) if k % 8):
            W = synth.normal_f16(0, "unaligned.w.%d.%d" % (rows, k), 0.02, (rows, k))
            x = oracle.to_f16(synth.normal_f32(0, "unaligned.x.%d" % k, 1.0, k))
            y = torch.full((rows,), float("nan"), dtype=torch.float32, device="cuda")
            bm.bm_f16_matvec(to_dev(W), to_dev(x), y)
            assert np.array_equal(y.cpu().numpy().view(np.uint32), oracle.matvec(W, x).view(np.uint32)), (rows, k)
    assert bm.bm_device_status() == 0
