"""GPU parity of the bit-exact paths against the CPU oracle, through the C ABI.

- bm_to_f16: every one of the 2^32 f32 bit patterns (NaN inputs must give NaN).
- bm_f16_matvec / bm_f16_matvec_multi / bm_f16_logits (one column): bit for bit,
  including the hand-derived reduction examples of tests/golden/.
- bm_f16_matmul where takes_sgemm is false: vec_dot per element, bit for bit.
"""
import json
import os

import numpy as np
import pytest

import oracle
import synth
from conftest import GOLDEN, bits32, to_dev

pytestmark = pytest.mark.gpu


def rnd_f16(tid, shape, sigma=0.02, seed=0):
    return synth.normal_f16(seed, tid, sigma, shape)


def act(tid, shape, seed=0):
    return oracle.to_f16(synth.normal_f32(seed, tid, 1.0, shape))


# --------------------------------------------------------------------------- bm_to_f16


def test_to_f16_all_bit_patterns(bm):
    import torch
    chunk = 1 << 27
    for c in range(0, 1 << 32, chunk):
        pats = np.arange(c, c + chunk, dtype=np.uint64).astype(np.uint32)
        xf = pats.view(np.float32)
        got = bm.bm_to_f16(to_dev(xf)).cpu().numpy().view(np.uint16)
        ref = oracle.to_f16(xf)
        nan_in = np.isnan(xf)
        ok = (got == ref) | nan_in
        assert ok.all(), "first mismatch at f32 bits 0x%08x" % int(pats[~ok][0])
        g = got[nan_in]
        assert (((g & 0x7c00) == 0x7c00) & ((g & 0x3ff) != 0)).all(), "NaN input must give NaN"
        del pats, xf, got, ref
    torch.cuda.synchronize()


@pytest.mark.parametrize("n", [1, 7, 8, 9, 15, 16, 17, 576, 1000003, 512 * 14336])
def test_to_f16_ragged_lengths(bm, n):
    xf = synth.normal_f32(3, n, 1.0, n)
    xf[: min(n, 4)] *= 70000.0  # some overflow to inf
    got = bm.bm_to_f16(to_dev(xf)).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, oracle.to_f16(xf))


def test_to_f16_empty_is_a_no_op(bm):
    import torch
    x = torch.empty(0, dtype=torch.float32, device="cuda")
    h = bm.bm_to_f16(x)
    assert h.numel() == 0


# --------------------------------------------------------------------------- worked examples


def golden_examples():
    return json.load(open(os.path.join(GOLDEN, "reduction_examples.json")))["examples"]


def example_vectors(ex):
    k = ex["k"]
    w = np.zeros(k, dtype=np.uint16)
    a = np.zeros(k, dtype=np.uint16)
    for i, wb, ab in ex["terms"]:
        w[i] = int(wb, 16)
        a[i] = int(ab, 16)
    return w, a


@pytest.mark.parametrize("ex", golden_examples(), ids=lambda e: e["name"])
def test_gpu_reproduces_worked_examples(bm, ex):
    """The hand-derived vec_dot bits, on the GPU: one row, 13 rows (the fallback), and
    the same rows followed by random rows so the example sits inside a larger launch."""
    w, a = example_vectors(ex)
    k = w.size
    want = int(ex["vec_dot"], 16)
    y = bm.bm_f16_matvec(to_dev(w[None, :]), to_dev(a))
    assert bits32(y)[0] == want
    W = np.concatenate([np.tile(w, (13, 1)), rnd_f16(5, (51, k))])
    y = bits32(bm.bm_f16_matvec(to_dev(W), to_dev(a)))
    assert (y[:13] == want).all()
    assert np.array_equal(y, bits32(oracle.matvec(W, a)))
    # two columns, 13 rows: the vec_dot fallback must give the same bits per element
    Y = bits32(bm.bm_f16_matmul(to_dev(np.tile(w, (13, 1))), to_dev(np.stack([a, a]))))
    assert (Y == want).all()


# --------------------------------------------------------------------------- one column


ONE_COL_SHAPES = [
    (1536, 576), (13, 1000), (12, 1000), (1, 1), (1, 31), (3, 33), (7, 8), (8, 8), (9, 32), (17, 64),
    (576, 576), (192, 576), (576, 1536), (1024, 1024), (2048, 1024), (1024, 3072), (4096, 4096),
    (1024, 4096), (4096, 14336), (12, 4097), (13, 4097), (4096, 31), (4096, 33), (14336, 8),
    (300, 65536), (5, 65535), (1000, 4104), (1000, 4100),
]


@pytest.mark.parametrize("rows,k", ONE_COL_SHAPES)
def test_matvec_bit_exact(bm, rows, k):
    W = rnd_f16(10, (rows, k))
    x = act(11, k)
    y = bm.bm_f16_matvec(to_dev(W), to_dev(x))
    assert np.array_equal(bits32(y), bits32(oracle.matvec(W, x)))


@pytest.mark.parametrize("rows,k", [(4096, 1536), (12, 8192), (14336, 33)])
def test_logits_one_column_is_matvec(bm, rows, k):
    E = rnd_f16(12, (rows, k))
    x = act(13, k)
    y1 = bm.bm_f16_logits(to_dev(E), to_dev(x[None, :]))
    y2 = bm.bm_f16_matvec(to_dev(E), to_dev(x))
    assert np.array_equal(bits32(y1).reshape(-1), bits32(y2))
    assert np.array_equal(bits32(y2), bits32(oracle.matvec(E, x)))


@pytest.mark.parametrize("rows_list,k", [
    ((576, 192, 192), 576), ((1536, 1536), 576), ((2048, 1024, 1024), 1024), ((3072, 3072), 1024),
    ((4096, 1024, 1024), 4096), ((13, 1, 7, 300), 33), ((0, 5, 0), 64), ((8, 8, 8, 8), 4097),
])
def test_matvec_multi_equals_separate(bm, rows_list, k):
    Ws = [rnd_f16(20 + i, (r, k)) for i, r in enumerate(rows_list)]
    x = act(30, k)
    ys = bm.bm_f16_matvec_multi([to_dev(W) for W in Ws], to_dev(x))
    for W, y in zip(Ws, ys):
        assert np.array_equal(bits32(y), bits32(oracle.matvec(W, x)))


def test_output_guard_zones_untouched(bm):
    """Outputs written inside a larger buffer leave the bytes around them alone."""
    import torch
    rows, k = 1000, 4097
    W = rnd_f16(40, (rows, k))
    x = act(41, k)
    buf = torch.full((rows + 64,), float("nan"), dtype=torch.float32, device="cuda")
    canary = bits32(buf).copy()
    bm.bm_f16_matvec(to_dev(W), to_dev(x), y=buf[32:32 + rows])
    b = bits32(buf)
    assert np.array_equal(b[:32], canary[:32]) and np.array_equal(b[32 + rows:], canary[32 + rows:])
    assert np.array_equal(b[32:32 + rows], bits32(oracle.matvec(W, x)))
    rows2 = 1536
    W2 = rnd_f16(42, (rows2, 576))
    x2 = act(43, 576)
    buf2 = torch.full((rows2 + 64,), float("nan"), dtype=torch.float32, device="cuda")
    bm.bm_f16_matvec(to_dev(W2), to_dev(x2), y=buf2[32:32 + rows2])
    b2 = bits32(buf2)
    assert np.isnan(buf2[:32].cpu().numpy()).all() and np.isnan(buf2[32 + rows2:].cpu().numpy()).all()
    assert np.array_equal(b2[32:32 + rows2], bits32(oracle.matvec(W2, x2)))


def test_repeatable_across_streams(bm):
    import torch
    W = to_dev(rnd_f16(50, (4096, 4096)))
    x = to_dev(act(51, 4096))
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    y1 = bm.bm_f16_matvec(W, x, stream=s1)
    y2 = bm.bm_f16_matvec(W, x, stream=s2)
    torch.cuda.synchronize()
    assert np.array_equal(bits32(y1), bits32(y2))


# --------------------------------------------------------------------------- vec_dot fallback


FALLBACK_SHAPES = [
    (13, 1000, 2), (13, 1000, 4), (13, 1000, 5), (13, 1536, 512), (12, 31, 2), (12, 33, 5),
    (4096, 31, 512), (4096, 33, 2), (14336, 33, 5), (13, 8, 512), (7, 4097, 3), (12, 4097, 512),
    (1, 1, 2), (3, 40, 9),
]


@pytest.mark.parametrize("rows,k,ncols", FALLBACK_SHAPES)
def test_matmul_fallback_bit_exact(bm, rows, k, ncols):
    assert not bm.bm_takes_sgemm(rows, k, ncols)
    W = rnd_f16(60, (rows, k))
    X = act(61, (ncols, k))
    Y = bits32(bm.bm_f16_matmul(to_dev(W), to_dev(X))).reshape(ncols, rows)
    if rows * k * ncols <= 3e8:
        assert np.array_equal(Y, bits32(oracle.matmul(W, X)))
    else:
        rng = np.random.default_rng(rows + k + ncols)
        ri = np.concatenate([[0, rows - 1], rng.integers(0, rows, 4000)])
        ci = np.concatenate([[ncols - 1, 0], rng.integers(0, ncols, 4000)])
        ref, _ = oracle.matmul_sample(W, X, ri, ci, with_absdot=False)
        assert np.array_equal(Y[ci, ri], bits32(ref))


def test_device_status_clean(bm):
    assert bm.bm_device_status() == 0


# --------------------------------------------------------------------------- programmatic dependent launch


def test_pdl_chain_in_a_graph_is_bit_exact(bm):
    """A decode-like chain (round -> fused QKV -> round -> O -> round -> fused gate/up ->
    round -> down) with programmatic dependent launch on, eager and captured in a CUDA
    graph: every output equals the oracle bit for bit, and so does a repeat."""
    import torch
    hid, ffn = 576, 1536
    Wq, Wk, Wv = rnd_f16(80, (576, hid)), rnd_f16(81, (192, hid)), rnd_f16(82, (192, hid))
    Wo, Wg, Wu, Wd = rnd_f16(83, (hid, hid)), rnd_f16(84, (ffn, hid)), rnd_f16(85, (ffn, hid)), rnd_f16(86, (hid, ffn))
    acts = [synth.normal_f32(0, 90 + i, 1.0, n) for i, n in enumerate([hid, hid, hid, ffn])]
    dW = [to_dev(w) for w in (Wq, Wk, Wv, Wo, Wg, Wu, Wd)]
    dA = [to_dev(a) for a in acts]
    dH = [torch.empty(a.size, dtype=torch.float16, device="cuda") for a in acts]
    outs = [torch.empty(w.shape[0], dtype=torch.float32, device="cuda") for w in (Wq, Wk, Wv, Wo, Wg, Wu, Wd)]
    s = torch.cuda.Stream()

    def chain():
        bm.bm_to_f16(dA[0], dH[0], stream=s)
        bm.bm_f16_matvec_multi(dW[0:3], dH[0], outs[0:3], stream=s)
        bm.bm_to_f16(dA[1], dH[1], stream=s)
        bm.bm_f16_matvec(dW[3], dH[1], outs[3], stream=s)
        bm.bm_to_f16(dA[2], dH[2], stream=s)
        bm.bm_f16_matvec_multi(dW[4:6], dH[2], outs[4:6], stream=s)
        bm.bm_to_f16(dA[3], dH[3], stream=s)
        bm.bm_f16_matvec(dW[6], dH[3], outs[6], stream=s)

    hs = [oracle.to_f16(a) for a in acts]
    want = [oracle.matvec(Wq, hs[0]), oracle.matvec(Wk, hs[0]), oracle.matvec(Wv, hs[0]), oracle.matvec(Wo, hs[1]),
            oracle.matvec(Wg, hs[2]), oracle.matvec(Wu, hs[2]), oracle.matvec(Wd, hs[3])]
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


# --------------------------------------------------------------------------- fused rounding + products


@pytest.mark.parametrize("rows_list,k,store_h", [
    ((576, 192, 192), 576, True), ((1536, 1536), 576, False), ((576,), 1536, True), ((49152,), 576, False),
    ((4096, 1024, 1024), 4096, True), ((13, 5, 300, 1), 1000, True), ((7, 8), 33, True), ((20,), 8, False),
    ((4096,), 14336, True), ((300,), 65536, False),
])
def test_matvec_act_equals_round_then_matvec(bm, rows_list, k, store_h):
    import torch
    Ws = [rnd_f16(100 + i, (r, k)) for i, r in enumerate(rows_list)]
    xf = synth.normal_f32(0, 110, 1.0, k)
    xf[:3] = [70000.0, -1e-30, 3e-8]  # overflow, f32 subnormal, f16 subnormal
    h = torch.full((k,), float("nan"), dtype=torch.float16, device="cuda") if store_h else None
    ys = bm.bm_f16_matvec_act([to_dev(W) for W in Ws], to_dev(xf), h=h)
    hx = oracle.to_f16(xf)
    for W, y in zip(Ws, ys):
        assert np.array_equal(bits32(y), bits32(oracle.matvec(W, hx)))
    if store_h:
        assert np.array_equal(h.cpu().numpy().view(np.uint16), hx)


def test_matvec_act_unaligned_k_needs_h(bm):
    import torch
    W = to_dev(rnd_f16(120, (10, 33)))
    x = to_dev(synth.normal_f32(0, 121, 1.0, 33))
    with pytest.raises(bm.BmError):
        bm.bm_f16_matvec_act([W], x)
