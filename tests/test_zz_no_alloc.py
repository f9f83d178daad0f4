"""bm_f16_matmul_noalloc: the tensor-core product for callers that cannot allocate
device memory (an engine that reserved the whole device for its own arena, a
plugin inside a host that owns the allocator, a latency-critical thread that
must not block in an allocator).  It keeps its split-k partial sums in the
library's static device scratch instead of a temporary workspace, and where the
fastest plan's partials would not fit that scratch it takes a plan with fewer
k-splits.

Checked through the C ABI against bm_f16_matmul, within the same bound the other
tensor-core tests use, on two calls in a row (the second call finds the first
call's contents in the shared scratch).  bm_tc_plan shows which cases really
split along k.  This file is named to be collected last, and needs nothing from
earlier tests: it passes alone in a fresh process.
"""
import numpy as np
import pytest

import oracle
import synth
from conftest import to_dev

pytestmark = pytest.mark.gpu

TOL = 4e-6
SCRATCH = 8 << 20  # BM_NOALLOC_SCRATCH_BYTES


def rnd_f16(tid, shape, sigma=0.02):
    return synth.normal_f16(0, tid, sigma, shape)


def act(tid, shape):
    return oracle.to_f16(synth.normal_f32(0, tid, 1.0, shape))


def check_against_matmul(bm, rows, k, ncols, tid, calls=2, nsample=500):
    import torch
    W = rnd_f16(tid, (rows, k))
    X = act(tid + 1, (ncols, k))
    dW, dX = to_dev(W), to_dev(X)
    plan = bm.bm_tc_plan(rows, k, ncols, noalloc=True) if bm.bm_takes_sgemm(rows, k, ncols) else None
    old = bm.bm_set_stream_k(0)  # the plans this entry point takes (no balanced k ranges)
    try:
        same_plan = plan is not None and bm.bm_tc_plan(rows, k, ncols) == plan
        ref = bm.bm_f16_matmul(dW, dX).cpu().numpy().astype(np.float64)
    finally:
        bm.bm_set_stream_k(old)
    rng = np.random.default_rng(rows + ncols)
    ri = np.concatenate([[0, rows - 1], rng.integers(0, rows, nsample)])
    ci = np.concatenate([[ncols - 1, 0], rng.integers(0, ncols, nsample)])
    want, ab = oracle.matmul_sample(W, X, ri, ci)
    for _ in range(calls):
        Y = torch.full((ncols, rows), float("nan"), dtype=torch.float32, device="cuda")
        bm.bm_f16_matmul_noalloc(dW, dX, Y)
        got = Y.cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        # within the tensor-core bound of tinyBLAS's element everywhere sampled, and close
        # to bm_f16_matmul everywhere (identical where both take the same plan)
        assert (np.abs(got[ci, ri] - want.astype(np.float64)) <= TOL * ab).all()
        if same_plan or plan is None:
            assert np.array_equal(got, ref)
        else:
            # two plans, each within the bound: every element within twice a typical bound
            assert (np.abs(got - ref) <= 2 * TOL * float(ab.mean())).all()
    assert bm.bm_device_status() == 0
    return plan


# 20..64 columns split along k (the scratch in use); 3..8 columns take the CUDA-core kernel
# at the default exact-column setting only up to 2 columns, so 4 and 8 columns are tensor-core
@pytest.mark.parametrize("rows,k,ncols", [(4096, 4096, 64), (4096, 4096, 32), (1024, 8192, 20), (4096, 4096, 8),
                                          (1024, 8192, 3), (1536, 576, 4)])
def test_noalloc_matches_matmul_twice(bm, rows, k, ncols):
    check_against_matmul(bm, rows, k, ncols, 200)


def test_noalloc_uses_the_scratch(bm):
    """At least one product splits along k, and two different split products in a row
    (the second finds the first one's partials in the scratch) both come out right."""
    plans = [check_against_matmul(bm, 4096, 4096, 64, 210, calls=1),
             check_against_matmul(bm, 1024, 8192, 20, 212, calls=1),
             check_against_matmul(bm, 4096, 4096, 64, 210, calls=1)]
    assert any(p["splits"] > 1 and 0 < p["scratch_bytes"] <= SCRATCH for p in plans), plans


def test_noalloc_replans_products_beyond_its_scratch(bm):
    """The Llama-3-8B down product at 512 columns: the fastest plan's partial tiles
    exceed the scratch, so the no-allocation product takes one with fewer k-splits
    whose partials fit (at worst none), with the same results within the bound."""
    rows, k, ncols = 4096, 14336, 512
    fast = bm.bm_tc_plan(rows, k, ncols)
    plan = check_against_matmul(bm, rows, k, ncols, 220, calls=2, nsample=2000)
    assert plan["scratch_bytes"] <= SCRATCH and plan["balanced"] == 0
    if fast["splits"] > 1 and fast["balanced"] == 0:
        assert fast["scratch_bytes"] > SCRATCH  # the case the re-plan exists for
        assert plan["splits"] < fast["splits"]


def test_noalloc_vec_dot_shapes(bm):
    """Shapes off the tinyBLAS path take the vec_dot kernels (no scratch at all)."""
    import torch
    rows, k, ncols = 13, 1000, 5
    W, X = rnd_f16(204, (rows, k)), act(205, (ncols, k))
    Y = torch.empty((ncols, rows), dtype=torch.float32, device="cuda")
    bm.bm_f16_matmul_noalloc(to_dev(W), to_dev(X), Y)
    assert np.array_equal(Y.cpu().numpy().view(np.uint32), oracle.matmul(W, X).view(np.uint32))
