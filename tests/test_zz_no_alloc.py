"""bm_f16_matmul_noalloc: the tensor-core product for callers that cannot allocate
device memory (an engine that reserved the whole device for its own arena, a
plugin inside a host that owns the allocator, a latency-critical thread that
must not block in an allocator).  It keeps its split-k partial sums in the
library's static device scratch instead of a temporary workspace.

Checked through the C ABI against bm_f16_matmul, within the same bound the other
tensor-core tests use, on two calls in a row (the second call finds the first
call's contents in the shared scratch).  This file is named to be collected
last, and needs nothing from earlier tests: it passes alone in a fresh process.
"""
import numpy as np
import pytest

import oracle
import synth
from conftest import to_dev

pytestmark = pytest.mark.gpu

TOL = 4e-6


def rnd_f16(tid, shape, sigma=0.02):
    return synth.normal_f16(0, tid, sigma, shape)


def act(tid, shape):
    return oracle.to_f16(synth.normal_f32(0, tid, 1.0, shape))


# split along k (the scratch in use) for 20..64 columns; 3..8 columns take the CUDA-core kernel
@pytest.mark.parametrize("rows,k,ncols", [(4096, 4096, 64), (4096, 4096, 32), (1024, 8192, 20), (4096, 4096, 8),
                                          (1024, 8192, 3), (1536, 576, 4)])
def test_noalloc_matches_matmul_twice(bm, rows, k, ncols):
    import torch
    W = rnd_f16(200, (rows, k))
    X = act(201, (ncols, k))
    dW, dX = to_dev(W), to_dev(X)
    old = bm.bm_set_stream_k(0)  # the plans this entry point takes (no balanced k ranges)
    try:
        ref = bm.bm_f16_matmul(dW, dX).cpu().numpy().astype(np.float64)
    finally:
        bm.bm_set_stream_k(old)
    rng = np.random.default_rng(rows + ncols)
    ri = np.concatenate([[0, rows - 1], rng.integers(0, rows, 500)])
    ci = np.concatenate([[ncols - 1, 0], rng.integers(0, ncols, 500)])
    _, ab = oracle.matmul_sample(W, X, ri, ci)
    bound = np.full((ncols, rows), np.inf)
    bound[ci, ri] = TOL * ab
    for _ in range(2):
        Y = torch.full((ncols, rows), float("nan"), dtype=torch.float32, device="cuda")
        bm.bm_f16_matmul_noalloc(dW, dX, Y)
        got = Y.cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        # same kernel and plan as bm_f16_matmul without balanced ranges: within the tensor-core
        # bound everywhere sampled, and identical
        assert (np.abs(got - ref)[ci, ri] <= bound[ci, ri]).all()
        assert np.array_equal(got, ref)
    assert bm.bm_device_status() == 0


def test_noalloc_refuses_products_beyond_its_scratch(bm):
    import torch
    rows, k, ncols = 1024, 65536, 512  # 16 tiles, 8 k-splits: 16 MiB of partial tiles, more than the scratch
    dW = to_dev(rnd_f16(202, (rows, k)))
    dX = to_dev(act(203, (ncols, k)))
    Y = torch.zeros((ncols, rows), dtype=torch.float32, device="cuda")
    with pytest.raises(bm.BmError) as e:
        bm.bm_f16_matmul_noalloc(dW, dX, Y)
    assert e.value.status == 1 and "scratch" in str(e.value)
    assert bool((Y == 0).all())  # nothing was launched


def test_noalloc_vec_dot_shapes(bm):
    """Shapes off the tinyBLAS path take the vec_dot kernels (no scratch at all)."""
    import torch
    rows, k, ncols = 13, 1000, 5
    W, X = rnd_f16(204, (rows, k)), act(205, (ncols, k))
    Y = torch.empty((ncols, rows), dtype=torch.float32, device="cuda")
    bm.bm_f16_matmul_noalloc(to_dev(W), to_dev(X), Y)
    assert np.array_equal(Y.cpu().numpy().view(np.uint32), oracle.matmul(W, X).view(np.uint32))
