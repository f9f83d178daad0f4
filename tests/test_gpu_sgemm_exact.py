"""GPU parity of the CUDA-core tinyBLAS kernels (bm_takes_sgemm shapes of 2..8
columns, with bm_set_exact_sgemm_cols(8)) against the oracle, bit for bit: k_sgemm_ring
where the activation fits in shared memory (most shapes here), k_sgemm_stream where it
does not (1024 x 14336 at 7 columns, 8 x 65536 at 5).

Each output of these products is tinyBLAS's sgemm_dot (page f16.md, "Design
notes", "sgemm_dot"): eight lane chains in increasing t, folded
((l0+l4)+(l2+l6))+((l1+l5)+(l3+l7)).  The kernel keeps that order, so every bit
must equal oracle.matmul -- including the hand-derived examples of tests/golden/.
"""
import json
import os

import numpy as np
import pytest

import oracle
import synth
from conftest import GOLDEN, bits32, to_dev

pytestmark = pytest.mark.gpu

MAX_STREAM_COLS = 8


@pytest.fixture(autouse=True)
def exact_up_to_eight(bm):
    """Every takes_sgemm product of up to 8 columns on the bit-exact kernel."""
    old = bm.bm_set_exact_sgemm_cols(MAX_STREAM_COLS)
    yield
    bm.bm_set_exact_sgemm_cols(old)


def rnd_f16(tid, shape, sigma=0.02, seed=0):
    return synth.normal_f16(seed, tid, sigma, shape)


def act(tid, shape, seed=0):
    return oracle.to_f16(synth.normal_f32(seed, tid, 1.0, shape))


def exact_or_sampled(Y, W, X, limit=3e8, nsample=4000):
    """Y: (ncols, rows) uint32 bits from the GPU; compares every element when the oracle
    finishes in seconds, else a sample that always includes the corners."""
    ncols, rows = Y.shape
    if rows * W.shape[1] * ncols <= limit:
        assert np.array_equal(Y, bits32(oracle.matmul(W, X)))
        return
    rng = np.random.default_rng(rows + W.shape[1] + ncols)
    ri = np.concatenate([[0, rows - 1, 0, rows - 1], rng.integers(0, rows, nsample)])
    ci = np.concatenate([[0, ncols - 1, ncols - 1, 0], rng.integers(0, ncols, nsample)])
    ref, _ = oracle.matmul_sample(W, X, ri, ci, with_absdot=False)
    assert np.array_equal(Y[ci, ri], bits32(ref))


# every column count of the kernel; rows with and without a half group (rows % 8 == 4);
# k with a ragged last 64-element block, a single step, several stages, the maximum
STREAM_SHAPES = [(12, 1000, n) for n in range(2, MAX_STREAM_COLS + 1)] + [
    (4, 8, 2), (12, 8, 3), (4, 16, 8), (20, 72, 5), (1536, 576, 4), (1536, 576, 2), (4100, 1536, 3),
    (4096, 4104, 8), (4096, 4096, 6), (1024, 14336, 7), (576, 1536, 8), (2048, 1024, 6), (8, 65536, 5),
    (65532, 64, 2), (300, 8200, 7), (128256, 64, 3), (14336, 4096, 8),
]


@pytest.mark.parametrize("rows,k,ncols", STREAM_SHAPES)
def test_sgemm_stream_bit_exact(bm, rows, k, ncols):
    assert bm.bm_takes_sgemm(rows, k, ncols)
    W = rnd_f16(100, (rows, k))
    X = act(101, (ncols, k))
    Y = bits32(bm.bm_f16_matmul(to_dev(W), to_dev(X))).reshape(ncols, rows)
    exact_or_sampled(Y, W, X)


def golden_sgemm_examples():
    ex = json.load(open(os.path.join(GOLDEN, "reduction_examples.json")))["examples"]
    return [e for e in ex if e.get("sgemm") is not None]


@pytest.mark.parametrize("ex", golden_sgemm_examples(), ids=lambda e: e["name"])
@pytest.mark.parametrize("ncols", [2, 5, 8])
def test_gpu_reproduces_sgemm_worked_examples(bm, ex, ncols):
    """The hand-derived sgemm_dot bits, on the GPU: the example row repeated over 12
    rows (bm_takes_sgemm), inside a larger product of random rows."""
    k = ex["k"]
    w = np.zeros(k, dtype=np.uint16)
    a = np.zeros(k, dtype=np.uint16)
    for i, wb, ab in ex["terms"]:
        w[i] = int(wb, 16)
        a[i] = int(ab, 16)
    want = int(ex["sgemm"], 16)
    X = np.tile(a, (ncols, 1))
    Y = bits32(bm.bm_f16_matmul(to_dev(np.tile(w, (12, 1))), to_dev(X)))
    assert (Y == want).all()
    W = np.concatenate([rnd_f16(102, (36, k)), np.tile(w, (12, 1)), rnd_f16(103, (52, k))])
    Y = bits32(bm.bm_f16_matmul(to_dev(W), to_dev(X))).reshape(ncols, 100)
    assert (Y[:, 36:48] == want).all()
    assert np.array_equal(Y, bits32(oracle.matmul(W, X)))


def test_columns_are_independent(bm):
    """Column c of a product equals the same column computed among other columns (no
    column leaks into another slot of a thread)."""
    rows, k = 1536, 576
    W = to_dev(rnd_f16(104, (rows, k)))
    X = act(105, (MAX_STREAM_COLS, k))
    full = bits32(bm.bm_f16_matmul(W, to_dev(X))).reshape(MAX_STREAM_COLS, rows)
    for n in (2, 3, 4, 5, 6, 7):
        part = bits32(bm.bm_f16_matmul(W, to_dev(X[:n]))).reshape(n, rows)
        assert np.array_equal(part, full[:n])


def test_noalloc_and_logits_take_the_same_kernel(bm):
    import torch
    rows, k, ncols = 4096, 1024, 6
    E = rnd_f16(106, (rows, k))
    X = act(107, (ncols, k))
    a = bits32(bm.bm_f16_matmul(to_dev(E), to_dev(X)))
    b = bits32(bm.bm_f16_matmul_noalloc(to_dev(E), to_dev(X),
                                        torch.empty((ncols, rows), dtype=torch.float32, device="cuda")))
    c = bits32(bm.bm_f16_logits(to_dev(E), to_dev(X)))
    assert np.array_equal(a, b) and np.array_equal(a, c)
    exact_or_sampled(a.reshape(ncols, rows), E, X)


def test_output_guard_zones_untouched(bm):
    import torch
    rows, k, ncols = 1000, 576, 3
    W = rnd_f16(108, (rows, k))
    X = act(109, (ncols, k))
    buf = torch.full((rows * ncols + 64,), float("nan"), dtype=torch.float32, device="cuda")
    bm.bm_f16_matmul(to_dev(W), to_dev(X), Y=buf[32:32 + rows * ncols])
    b = buf.cpu().numpy()
    assert np.isnan(b[:32]).all() and np.isnan(b[32 + rows * ncols:]).all()
    assert np.array_equal(bits32(b[32:32 + rows * ncols]), bits32(oracle.matmul(W, X)).ravel())


def test_pdl_chain_in_a_graph_is_bit_exact(bm):
    """Prefill-like chain of few-column products with programmatic dependent launch,
    eager and captured in a CUDA graph, each product's activation written by the
    rounding kernel just ahead of it."""
    import torch
    hid, ffn, n = 576, 1536, 5
    Wq, Wg, Wd = rnd_f16(110, (hid, hid)), rnd_f16(111, (ffn, hid)), rnd_f16(112, (hid, ffn))
    acts = [synth.normal_f32(0, 113 + i, 1.0, (n, kk)) for i, kk in enumerate([hid, hid, ffn])]
    dW = [to_dev(w) for w in (Wq, Wg, Wd)]
    dA = [to_dev(a) for a in acts]
    dH = [torch.empty(a.shape, dtype=torch.float16, device="cuda") for a in acts]
    outs = [torch.empty((n, w.shape[0]), dtype=torch.float32, device="cuda") for w in (Wq, Wg, Wd)]
    s = torch.cuda.Stream()

    def chain():
        for i in range(3):
            bm.bm_to_f16(dA[i], dH[i], stream=s)
            bm.bm_f16_matmul(dW[i], dH[i], Y=outs[i], stream=s)

    want = [oracle.matmul(w, oracle.to_f16(a)) for w, a in zip((Wq, Wg, Wd), acts)]
    old = bm.bm_set_pdl(True)
    try:
        with torch.cuda.stream(s):
            chain()
        torch.cuda.synchronize()
        for o, w in zip(outs, want):
            assert np.array_equal(bits32(o), bits32(w))
        for o in outs:
            o.fill_(float("nan"))
        g = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            chain()
        for _ in range(3):
            g.replay()
        torch.cuda.synchronize()
        for o, w in zip(outs, want):
            assert np.array_equal(bits32(o), bits32(w))
    finally:
        bm.bm_set_pdl(old)
    assert bm.bm_device_status() == 0
