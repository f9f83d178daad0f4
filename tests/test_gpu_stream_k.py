"""GPU parity of the tensor-core products with balanced k ranges (bm_set_stream_k):
every SM takes an equal run of the k-blocks of all tiles laid end to end, and the SM
holding a tile's last k-block adds the lower SMs' pieces in k order.  Forced on, each
product stays within 4e-6 * sum|w*a| of tinyBLAS's element (the oracle), gives the
same bits on every call, in a CUDA graph replayed several times (the flags go back to
zero) and under programmatic dependent launch; forced off, the k-split and whole-tile
plans do the same."""
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


@pytest.fixture
def mode(bm, request):
    old = bm.bm_set_stream_k(request.param)
    yield request.param
    bm.bm_set_stream_k(old)


def check_within(Yt, W, X):
    Y = Yt.cpu().numpy()
    ncols, rows = Y.shape
    if rows * W.shape[1] * ncols <= 2e8:
        ref, ab = oracle.matmul(W, X), oracle.abs_matmul(W, X)
        err = np.abs(Y.astype(np.float64) - ref.astype(np.float64))
        assert (err <= TOL * ab).all(), "worst ratio %g" % float((err / np.maximum(ab, 1e-300)).max())
        return
    rng = np.random.default_rng(rows + ncols)
    ri = np.concatenate([[0, rows - 1, 0, rows - 1], rng.integers(0, rows, 2500)])
    ci = np.concatenate([[0, ncols - 1, ncols - 1, 0], rng.integers(0, ncols, 2500)])
    ref, ab = oracle.matmul_sample(W, X, ri, ci)
    err = np.abs(Y[ci, ri].astype(np.float64) - ref.astype(np.float64))
    assert (err <= TOL * ab).all(), "worst ratio %g" % float((err / np.maximum(ab, 1e-300)).max())


SHAPES = [
    (4096, 4096, 512),    # Llama-3-8B Q / O
    (14336, 4096, 512),   # gate: 256-row units
    (4096, 14336, 512),   # down: a tile spread over several SMs
    (1024, 1024, 512),
    (640, 2048, 300),     # ragged columns
    (132, 72, 17),        # fewer k-blocks than SMs
    (256, 4104, 255),     # k % 64 != 0
    (12, 8192, 512),      # one short row tile
    (4096, 1536, 33),
    (8, 65536, 13),       # one tile over every SM: its owner adds 147 pieces
    (2048, 1024, 12),
]


@pytest.mark.parametrize("mode", [1, 0], indirect=True)
@pytest.mark.parametrize("rows,k,ncols", SHAPES)
def test_within_bound_and_repeatable(bm, mode, rows, k, ncols):
    W, X = rnd_f16(140, (rows, k)), act(141, (ncols, k))
    dW, dX = to_dev(W), to_dev(X)
    Y1 = bm.bm_f16_matmul(dW, dX)
    Y2 = bm.bm_f16_matmul(dW, dX)
    assert bm.bm_device_status() == 0
    assert np.array_equal(bits32(Y1), bits32(Y2))
    check_within(Y1, W, X)


@pytest.mark.parametrize("mode", [1], indirect=True)
def test_exact_integers(bm, mode):
    """Small integers: every partial sum and every piece is an exact f32 integer, so
    any correct split of the k-blocks gives the exact product (a piece added twice,
    dropped or taken from the wrong slot cannot pass)."""
    rng = np.random.default_rng(5)
    for rows, k, ncols in [(4096, 4096, 512), (132, 4096, 19), (8, 65536, 13), (1540, 8192, 40)]:
        Wi = rng.integers(-3, 4, (rows, k)).astype(np.float16)
        Xi = rng.integers(-3, 4, (ncols, k)).astype(np.float16)
        Y = bm.bm_f16_matmul(to_dev(Wi.view(np.uint16)), to_dev(Xi.view(np.uint16))).cpu().numpy()
        ri = rng.integers(0, rows, 400)
        ci = rng.integers(0, ncols, 400)
        want = np.einsum("ij,ij->i", Wi[ri].astype(np.float64), Xi[ci].astype(np.float64))
        assert np.array_equal(Y[ci, ri].astype(np.float64), want)


@pytest.mark.parametrize("mode", [1], indirect=True)
def test_graph_replays_streams_and_pdl(bm, mode):
    """The flags are reset by the owners, so a graph replayed again and again gives the
    same bits; two products on two streams at once use separate workspaces; under
    programmatic dependent launch a chain of products gives the same bits."""
    import torch
    rows, k, ncols = 4096, 4096, 512
    Wa, Wb = to_dev(rnd_f16(142, (rows, k))), to_dev(rnd_f16(143, (rows, k)))
    Xa, Xb = to_dev(act(144, (ncols, k))), to_dev(act(145, (ncols, k)))
    ref_a = bits32(bm.bm_f16_matmul(Wa, Xa))
    ref_b = bits32(bm.bm_f16_matmul(Wb, Xb))
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    Ya = torch.empty((ncols, rows), dtype=torch.float32, device="cuda")
    Yb = torch.empty((ncols, rows), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    for _ in range(3):
        bm.bm_f16_matmul(Wa, Xa, Ya, stream=s1)
        bm.bm_f16_matmul(Wb, Xb, Yb, stream=s2)
    torch.cuda.synchronize()
    assert np.array_equal(bits32(Ya), ref_a) and np.array_equal(bits32(Yb), ref_b)

    old = bm.bm_set_pdl(True)
    try:
        Yc = torch.empty((ncols, rows), dtype=torch.float32, device="cuda")
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s1):
            bm.bm_f16_matmul(Wa, Xa, Ya, stream=s1)
            bm.bm_f16_matmul(Wb, Xb, Yb, stream=s1)
            bm.bm_f16_matmul(Wa, Xb, Yc, stream=s1)
        for _ in range(5):
            Ya.fill_(float("nan"))
            Yb.fill_(float("nan"))
            g.replay()
            torch.cuda.synchronize()
            assert np.array_equal(bits32(Ya), ref_a) and np.array_equal(bits32(Yb), ref_b)
        ref_c = bits32(bm.bm_f16_matmul(Wa, Xb))
        assert np.array_equal(bits32(Yc), ref_c)
    finally:
        bm.bm_set_pdl(old)
    assert bm.bm_device_status() == 0


@pytest.mark.parametrize("mode", [1], indirect=True)
def test_multi_matrix(bm, mode):
    """Q/K/V of the Llama-3-8B and Qwen3-0.6B shapes in one launch, the ranges running
    across the matrices' tiles."""
    import torch
    for rows, k, ncols in [((4096, 1024, 1024), 4096, 512), ((2048, 1024, 1024), 1024, 512),
                           ((128, 256, 384, 512), 64, 17)]:
        Ws = [rnd_f16(150 + i, (r, k)) for i, r in enumerate(rows)]
        X = act(155, (ncols, k))
        Ys = [torch.empty((ncols, r), dtype=torch.float32, device="cuda") for r in rows]
        bm.bm_f16_matmul_multi([to_dev(W) for W in Ws], to_dev(X), Ys)
        assert bm.bm_device_status() == 0
        for W, Y in zip(Ws, Ys):
            check_within(Y, W, X)
