"""GPU parity of the takes_sgemm products against the oracle's tinyBLAS element:
|Y - sgemm_dot| <= 4e-6 * sum_i |w_i * a_i| per element.

The bound is the one the product's contract states for the tensor-core path;
tinyBLAS's own result is one rounding order among many, so the tensor-core sum is
compared to it within that bound rather than bit for bit.  Products of at most
bm_set_exact_sgemm_cols columns (default 2) run on the CUDA-core kernel, which gives
tinyBLAS's bits (test_gpu_sgemm_exact.py checks them exactly); they must meet the
bound here too."""
import numpy as np
import pytest

import oracle
import synth
from conftest import bits32, to_dev

pytestmark = pytest.mark.gpu

TOL = 4e-6


def rnd_f16(tid, shape, sigma=0.02, seed=0):
    return synth.normal_f16(seed, tid, sigma, shape)


def act(tid, shape, seed=0):
    return oracle.to_f16(synth.normal_f32(seed, tid, 1.0, shape))


def check_within(Y, W, X, sample=None):
    """Y is (ncols, rows) float32 from the GPU."""
    ncols, rows = Y.shape
    if sample is None:
        ref = oracle.matmul(W, X)
        ab = oracle.abs_matmul(W, X)
        err = np.abs(Y.astype(np.float64) - ref.astype(np.float64))
        bad = err > TOL * ab
        assert not bad.any(), "worst ratio %g" % float((err / np.maximum(ab, 1e-300)).max())
        return float((err / np.maximum(ab, 1e-300)).max())
    ri, ci = sample
    ref, ab = oracle.matmul_sample(W, X, ri, ci)
    got = Y[ci, ri].astype(np.float64)
    err = np.abs(got - ref.astype(np.float64))
    assert (err <= TOL * ab).all(), "worst ratio %g" % float((err / np.maximum(ab, 1e-300)).max())
    return float((err / np.maximum(ab, 1e-300)).max())


GEMM_SHAPES = [
    (1536, 576, 4), (1536, 576, 2), (12, 1000, 2), (12, 8, 2), (4, 8, 2), (128, 64, 16), (132, 72, 17),
    (12, 1536, 5), (4096, 8, 512), (12, 8192, 512), (4096, 1536, 2), (4096, 1536, 5), (256, 4104, 255),
    (1024, 1024, 512), (640, 2048, 300), (4096, 4096, 3), (4096, 4096, 8), (4096, 4096, 64),
    # the narrowest tensor-core tiles (9..48 columns)
    (12, 1000, 9), (4, 16, 16), (4096, 4096, 16), (576, 1536, 9), (2048, 1024, 12), (8, 65536, 13),
    (300, 8200, 11), (12, 1000, 17), (4, 8, 20), (1536, 576, 24), (4096, 1536, 33), (4096, 4096, 32),
    (20, 4104, 48),
]


@pytest.mark.parametrize("rows,k,ncols", GEMM_SHAPES)
def test_tensor_core_within_bound(bm, rows, k, ncols):
    assert bm.bm_takes_sgemm(rows, k, ncols)
    W = rnd_f16(70, (rows, k))
    X = act(71, (ncols, k))
    Y = bm.bm_f16_matmul(to_dev(W), to_dev(X)).cpu().numpy()
    assert np.isfinite(Y).all()
    if rows * k * ncols <= 2e8:
        check_within(Y, W, X)
    else:
        rng = np.random.default_rng(rows * 7 + ncols)
        ri = np.concatenate([[0, rows - 1, rows - 1], rng.integers(0, rows, 3000)])
        ci = np.concatenate([[0, ncols - 1, 0], rng.integers(0, ncols, 3000)])
        check_within(Y, W, X, (ri, ci))


def test_tensor_core_exact_integers(bm):
    """Small integers: every partial sum is an exact f32 integer, so any correct
    accumulation order gives the exact integer product (catches layout, operand and
    tile-edge mistakes with no tolerance at all)."""
    rng = np.random.default_rng(2)
    for rows, k, ncols in [(132, 200, 19), (256, 72, 2), (1540, 576, 4)]:
        Wi = rng.integers(-8, 9, size=(rows, k))
        Xi = rng.integers(-8, 9, size=(ncols, k))
        W = Wi.astype(np.float16).view(np.uint16)
        X = Xi.astype(np.float16).view(np.uint16)
        Y = bm.bm_f16_matmul(to_dev(W), to_dev(X)).cpu().numpy()
        assert np.array_equal(Y, (Xi @ Wi.T).astype(np.float32))


def test_logits_multi_column_takes_the_product_path(bm):
    E = rnd_f16(72, (49152 // 8, 576))
    X = act(73, (4, 576))
    Y1 = bm.bm_f16_logits(to_dev(E), to_dev(X))
    Y2 = bm.bm_f16_matmul(to_dev(E), to_dev(X))
    assert np.array_equal(bits32(Y1), bits32(Y2))
    check_within(Y1.cpu().numpy(), E, X, (np.arange(0, 6144, 7), np.arange(0, 6144, 7) % 4))


def test_twelve_vs_thirteen_rows_pick_different_paths(bm):
    """The page's pair: 12 rows x 2 columns take tinyBLAS's path (exactly its 0.0 for
    example E1), 13 rows the vec_dot fallback (exactly 1.0); with 20 columns the
    12-row product runs on the tensor cores, within the bound of that 0.0."""
    k = 32
    w = np.zeros(k, np.uint16)
    a = np.zeros(k, np.uint16)
    w[0], a[0], w[8], a[8], w[16], a[16] = 0x6c00, 0x6c00, 0x3c00, 0x3c00, 0xec00, 0x6c00
    X = np.stack([a, a])
    Y13 = bits32(bm.bm_f16_matmul(to_dev(np.tile(w, (13, 1))), to_dev(X)))
    assert (Y13 == 0x3f800000).all()
    Y12 = bits32(bm.bm_f16_matmul(to_dev(np.tile(w, (12, 1))), to_dev(X)))
    assert (Y12 == 0).all()
    Y12t = bm.bm_f16_matmul(to_dev(np.tile(w, (12, 1))), to_dev(np.tile(a, (20, 1)))).cpu().numpy()
    assert (np.abs(Y12t.astype(np.float64) - 0.0) <= TOL * (2.0 ** 25 + 1)).all()


def test_repeatable(bm):
    W = to_dev(rnd_f16(74, (4096, 4096)))
    X = to_dev(act(75, (512, 4096)))
    a = bits32(bm.bm_f16_matmul(W, X))
    b = bits32(bm.bm_f16_matmul(W, X))
    assert np.array_equal(a, b)


def test_bounded_wait_gives_up_and_context_survives(bm):
    """A producer that withholds its load makes the consumer's wait run out; the
    kernel reports BM_ERR_TIMEOUT and the context keeps working."""
    import torch
    W = torch.zeros((128, 64), dtype=torch.float16, device="cuda")
    X = torch.zeros((16, 64), dtype=torch.float16, device="cuda")
    Y = torch.empty((16, 128), dtype=torch.float32, device="cuda")
    assert bm.bm_selftest_wait_timeout(W, X, Y) == 5
    assert bm.bm_device_status() == 0
    Wn = rnd_f16(76, (256, 64))
    Xn = act(77, (16, 64))
    Y2 = bm.bm_f16_matmul(to_dev(Wn), to_dev(Xn)).cpu().numpy()
    check_within(Y2, Wn, Xn)
    assert bm.bm_device_status() == 0


SPLIT_SHAPES = [(4096, 4096, 512), (4096, 14336, 512), (4096, 4096, 8), (1024, 8192, 2), (256, 16384, 37),
                (1024, 8192, 18), (4096, 14336, 64)]


@pytest.mark.parametrize("rows,k,ncols", SPLIT_SHAPES)
def test_split_k_shapes_within_bound_and_repeatable(bm, rows, k, ncols):
    """Shapes with few output tiles take k-splits (partials summed in split order):
    within the bound, and bit-identical on a second call (the counters reset)."""
    W = rnd_f16(80, (rows, k))
    X = act(81, (ncols, k))
    dW, dX = to_dev(W), to_dev(X)
    Y1 = bm.bm_f16_matmul(dW, dX)
    Y2 = bm.bm_f16_matmul(dW, dX)
    assert np.array_equal(bits32(Y1), bits32(Y2))
    rng = np.random.default_rng(k + ncols)
    ri = np.concatenate([[0, rows - 1], rng.integers(0, rows, 2000)])
    ci = np.concatenate([[ncols - 1, 0], rng.integers(0, ncols, 2000)])
    check_within(Y1.cpu().numpy(), W, X, (ri, ci))


def test_split_k_in_a_cuda_graph_and_concurrent_streams(bm):
    """The split-k workspace is stream-ordered: the product captures into a CUDA graph
    and two products on two streams at once do not share it."""
    import torch
    rows, k, ncols = 4096, 8192, 64
    Wa, Wb = rnd_f16(82, (rows, k)), rnd_f16(83, (rows, k))
    Xa, Xb = act(84, (ncols, k)), act(85, (ncols, k))
    dWa, dWb, dXa, dXb = to_dev(Wa), to_dev(Wb), to_dev(Xa), to_dev(Xb)
    ref_a = bits32(bm.bm_f16_matmul(dWa, dXa))
    ref_b = bits32(bm.bm_f16_matmul(dWb, dXb))
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    Ya = torch.empty((ncols, rows), dtype=torch.float32, device="cuda")
    Yb = torch.empty((ncols, rows), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    for _ in range(3):
        bm.bm_f16_matmul(dWa, dXa, Ya, stream=s1)
        bm.bm_f16_matmul(dWb, dXb, Yb, stream=s2)
    torch.cuda.synchronize()
    assert np.array_equal(bits32(Ya), ref_a) and np.array_equal(bits32(Yb), ref_b)
    g = torch.cuda.CUDAGraph()
    Ya.fill_(float("nan"))
    with torch.cuda.graph(g, stream=s1):
        bm.bm_f16_matmul(dWa, dXa, Ya, stream=s1)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(bits32(Ya), ref_a)
    assert bm.bm_device_status() == 0


@pytest.mark.parametrize("rows,k,ncols", [(4096, 4096, 512), (1536, 576, 64), (14336, 1024, 512), (1000, 8192, 40)])
def test_pdl_prefill_chain_matches_plain_launches(bm, rows, k, ncols):
    """A prefill-like chain -- rounding kernel, tensor-core product (split or not),
    rounding of that product's output, a second product -- under programmatic
    dependent launch, eagerly and replayed from a CUDA graph: the same bits as with
    plain launches, and within the bound."""
    import torch
    W1 = to_dev(rnd_f16(130, (rows, k)))
    W2 = to_dev(rnd_f16(131, (k, rows)))
    xf = to_dev(synth.normal_f32(0, 132, 1.0, (ncols, k)))
    h1 = torch.empty((ncols, k), dtype=torch.float16, device="cuda")
    Y1 = torch.empty((ncols, rows), dtype=torch.float32, device="cuda")
    h2 = torch.empty((ncols, rows), dtype=torch.float16, device="cuda")
    Y2 = torch.empty((ncols, k), dtype=torch.float32, device="cuda")
    s = torch.cuda.Stream()

    def chain():
        bm.bm_to_f16(xf, h1, stream=s)
        bm.bm_f16_matmul(W1, h1, Y=Y1, stream=s)
        bm.bm_to_f16(Y1, h2, stream=s)
        bm.bm_f16_matmul(W2, h2, Y=Y2, stream=s)

    old = bm.bm_set_pdl(False)
    try:
        with torch.cuda.stream(s):
            chain()
        torch.cuda.synchronize()
        want1, want2 = bits32(Y1).copy(), bits32(Y2).copy()
        bm.bm_set_pdl(True)
        for Y in (Y1, Y2):
            Y.fill_(float("nan"))
        with torch.cuda.stream(s):
            chain()
        torch.cuda.synchronize()
        assert np.array_equal(bits32(Y1), want1) and np.array_equal(bits32(Y2), want2)
        for Y in (Y1, Y2):
            Y.fill_(float("nan"))
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            chain()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(bits32(Y1), want1) and np.array_equal(bits32(Y2), want2)
    finally:
        bm.bm_set_pdl(old)
    assert bm.bm_device_status() == 0
    rng = np.random.default_rng(rows + ncols)
    ri = rng.integers(0, rows, 2000)
    ci = rng.integers(0, ncols, 2000)
    check_within(Y1.cpu().numpy(), rnd_f16(130, (rows, k)), h1.cpu().numpy().view(np.uint16), sample=(ri, ci))
