"""GPU parity of bm_f16_matmul_multi: up to four matrices sharing one activation (the
prefill Q/K/V or gate/up).  Each output is held to the contract of its own matrix's
path, as bm_f16_matmul's: the tensor-core matrices (sharing one launch) within
4e-6 * sum|w*a| of tinyBLAS's element, the others (vec_dot, or tinyBLAS's bits on the
CUDA-core kernel) bit for bit."""
import numpy as np
import pytest

import oracle
import synth
from conftest import bits32, to_dev

pytestmark = pytest.mark.gpu

TOL = 4e-6


def rnd_f16(tid, shape, sigma=0.02):
    return synth.normal_f16(0, tid, sigma, shape)


def act(tid, shape):
    return oracle.to_f16(synth.normal_f32(0, tid, 1.0, shape))


def check(bm, Y, W, X, exact_cols):
    """Y: (ncols, rows) float32 (torch); W, X numpy."""
    rows, k = W.shape
    ncols = X.shape[0]
    got = bits32(Y).reshape(ncols, rows)
    exact = not oracle.takes_sgemm(rows, k, ncols) or ncols <= exact_cols
    if rows * k * ncols <= 1.5e8:
        ref = oracle.matmul(W, X)
        if exact:
            assert np.array_equal(got, bits32(ref))
        else:
            err = np.abs(got.view(np.float32).astype(np.float64) - ref.astype(np.float64))
            assert (err <= TOL * oracle.abs_matmul(W, X)).all()
        return
    rng = np.random.default_rng(rows + k + ncols)
    ri = np.concatenate([[0, rows - 1, 0, rows - 1], rng.integers(0, rows, 2500)])
    ci = np.concatenate([[0, ncols - 1, ncols - 1, 0], rng.integers(0, ncols, 2500)])
    ref, ab = oracle.matmul_sample(W, X, ri, ci, with_absdot=not exact)
    if exact:
        assert np.array_equal(got[ci, ri], bits32(ref))
    else:
        err = np.abs(got[ci, ri].view(np.float32).astype(np.float64) - ref.astype(np.float64))
        assert (err <= TOL * ab).all()


CASES = [
    # (rows of each matrix, k, ncols)
    ((4096, 1024, 1024), 4096, 512),    # Llama-3-8B Q/K/V: splits
    ((14336, 14336), 4096, 512),        # gate/up: 256-row units
    ((2048, 1024, 1024), 1024, 512),    # Qwen3-0.6B Q/K/V
    ((3072, 3072), 1024, 200),          # gate/up at a ragged column count
    ((576, 192, 192), 576, 64),         # SmolLM2 Q/K/V
    ((1024, 13, 0, 1028), 1536, 48),    # a vec_dot matrix (13 rows) and an empty one among them
    ((4096, 1024, 1024), 4096, 2),      # two columns: tinyBLAS's bits on the CUDA-core kernel
    ((128, 256, 384, 512), 64, 17),     # four matrices, one k-block
]


@pytest.mark.parametrize("rows,k,ncols", CASES)
def test_matmul_multi(bm, rows, k, ncols):
    Ws = [rnd_f16("mm.%d.%d.%d" % (i, r, k), (r, k)) for i, r in enumerate(rows)]
    X = act("mm.x.%d" % k, (ncols, k))
    Ys = bm.bm_f16_matmul_multi([to_dev(W) for W in Ws], to_dev(X))
    cur = bm.bm_set_exact_sgemm_cols(0)
    bm.bm_set_exact_sgemm_cols(cur)
    for W, Y in zip(Ws, Ys):
        if W.shape[0]:
            check(bm, Y, W, X, cur)
    assert bm.bm_device_status() == 0


def test_matmul_multi_repeatable_and_in_a_pdl_graph(bm):
    """Same bits every run, eagerly and replayed from a CUDA graph under programmatic
    dependent launch behind a rounding kernel."""
    import torch
    rows, k, ncols = (4096, 1024, 1024), 4096, 512
    dWs = [to_dev(rnd_f16("mmg.%d" % i, (r, k))) for i, r in enumerate(rows)]
    xf = to_dev(synth.normal_f32(0, "mmg.x", 1.0, (ncols, k)))
    h = torch.empty((ncols, k), dtype=torch.float16, device="cuda")
    Ys = [torch.empty((ncols, r), dtype=torch.float32, device="cuda") for r in rows]
    s = torch.cuda.Stream()

    def step():
        bm.bm_to_f16(xf, h, stream=s)
        bm.bm_f16_matmul_multi(dWs, h, Ys, stream=s)

    with torch.cuda.stream(s):
        step()
    torch.cuda.synchronize()
    want = [bits32(Y).copy() for Y in Ys]
    old = bm.bm_set_pdl(True)
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            step()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            step()
        for Y in Ys:
            Y.fill_(float("nan"))
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
    finally:
        bm.bm_set_pdl(old)
    for Y, w in zip(Ys, want):
        assert np.array_equal(bits32(Y), w)
    assert bm.bm_device_status() == 0
