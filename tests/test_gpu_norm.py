"""GPU parity of rms_norm then mul (page "docs/modules/forward.md", Technical usage,
"Other public pieces"), standalone (bm_rms_norm_mul) and as the fused decode front
end (bm_f16_matvec_norm: the norm, the f16 rounding and up to four one-column
products in one launch), against the oracle, bit for bit.

The one freedom the kernels take is in the mean of the squares: they sum the squares
exactly (integer fixed point) and divide by k to 2^-62, where the oracle adds doubles
in index order and divides in double.  The two means agree after rounding to f32
unless the exact mean lies within about (k + 4) * 2^-53 (relative) of an f32 rounding
boundary: `ambiguous_rows` finds such rows from the exact sum (math.fsum); every other
row must match the oracle bit for bit, and an ambiguous row (none occurs in these
seeded inputs) within 2 ulps.
"""
import math

import numpy as np
import pytest

import norm_cases
import oracle
import synth
from conftest import bits32, to_dev

pytestmark = pytest.mark.gpu

EPS = 1e-5


def _lsb_exponent(v):
    """e such that the nonzero double v is an odd multiple of 2^e."""
    m, e = math.frexp(v)
    M = int(m * 2.0 ** 53)
    return e - 53 + ((M & -M).bit_length() - 1)


def ambiguous_rows(X, k):
    """Rows whose f32 mean could depend on the order of the double sum of squares:
    the sum is not exact in every order (its bits span more than 53 places) and the
    exact mean lies within (k + 4) * 2^-53 (relative) of an f32 rounding boundary."""
    X = np.asarray(X, np.float32).reshape(-1, k)
    with np.errstate(over="ignore", invalid="ignore"):
        q = (X * X).astype(np.float64)  # each square is one f32 multiply (inf when it overflows)
    amb = np.zeros(X.shape[0], bool)
    rel = (k + 4) * 2.0 ** -53
    for r in range(X.shape[0]):
        if not np.isfinite(q[r]).all():
            continue  # an infinite or NaN square: the mean is +inf or NaN whatever the order
        s = math.fsum(q[r])
        nz = q[r][q[r] != 0]
        if s == 0 or math.frexp(s)[1] - min(_lsb_exponent(float(v)) for v in nz) <= 53:
            continue  # every partial sum is a multiple of the smallest bit and below 2^53 of it: exact
        lo, hi = s * (1 - rel) / k, s * (1 + rel) / k
        amb[r] = np.float32(lo) != np.float32(hi)
    return amb


def assert_norm_rows(got, want, X, k):
    got, want = np.asarray(got, np.float32).reshape(-1, k), np.asarray(want, np.float32).reshape(-1, k)
    amb = ambiguous_rows(X, k)
    assert np.array_equal(bits32(got[~amb]), bits32(want[~amb]))
    if amb.any():
        ulp = np.spacing(np.abs(want[amb]))
        assert np.all(np.abs(got[amb] - want[amb]) <= 2 * ulp)
    return int(amb.sum())


def residual(tid, shape, sigma=1.0, seed=0):
    return synth.normal_f32(seed, tid, sigma, shape)


def norm_weight(tid, k, seed=0):
    # RMS-norm weights of trained models sit around 1 with a spread; f32 as the files keep them
    return (1.0 + synth.normal_f32(seed, tid, 0.2, k)).astype(np.float32)


ROW_SHAPES = [(1, 576), (7, 576), (512, 576), (3, 4096), (64, 4096), (2, 8192), (5, 1), (3, 3), (4, 5),
              (2, 1000), (1, 65536), (300, 1024), (33, 2048), (9, 1536)]


@pytest.mark.parametrize("nrows,k", ROW_SHAPES)
def test_rms_norm_rows(bm, nrows, k):
    X = residual("resid.%d.%d" % (nrows, k), (nrows, k))
    X[0] *= 1000.0                      # rows of very different scale in one call
    if nrows > 2:
        X[2] *= 1e-3
    g = norm_weight("attn_norm.%d" % k, k)
    out, h = bm.bm_rms_norm_mul(to_dev(X), to_dev(g), EPS, h=to_dev(np.zeros((nrows, k), np.uint16)),
                                out=to_dev(np.zeros((nrows, k), np.float32)))
    want = oracle.rms_norm_mul(X, g, EPS)
    assert assert_norm_rows(out.cpu().numpy(), want, X, k) == 0
    got_h = h.cpu().numpy().view(np.uint16)
    amb = ambiguous_rows(X, k)
    assert np.array_equal(got_h[~amb], oracle.to_f16(want)[~amb])


def test_closed_forms_on_the_gpu(bm):
    """The oracle's pins (constant rows, exact scales, eps inside the root, the sum that
    is exact only in double, zero rows, sign and power-of-two invariants) hold on the GPU."""
    import torch

    def f(x, w, eps):
        x = np.ascontiguousarray(x, np.float32)
        out, _ = bm.bm_rms_norm_mul(to_dev(x), to_dev(np.ascontiguousarray(w, np.float32)), float(eps))
        torch.cuda.synchronize()
        return out.cpu().numpy()

    assert norm_cases.failures(f) == []


def test_unaligned_rows_take_the_scalar_path(bm):
    import torch
    nrows, k = 6, 576
    X = residual("resid.u", (nrows, k))
    g = norm_weight("norm.u", k)
    buf = torch.zeros(nrows * k + 1, dtype=torch.float32, device="cuda")
    buf[1:] = torch.from_numpy(X.ravel()).cuda()
    obuf = torch.full((nrows * k + 2,), float("nan"), dtype=torch.float32, device="cuda")
    hbuf = torch.zeros(nrows * k + 1, dtype=torch.float16, device="cuda")
    bm.bm_rms_norm_mul(buf[1:].view(nrows, k), to_dev(g), EPS, out=obuf[1:1 + nrows * k].view(nrows, k),
                       h=hbuf[1:].view(nrows, k))
    o = obuf.cpu().numpy()
    assert np.isnan(o[0]) and np.isnan(o[-1])
    want = oracle.rms_norm_mul(X, g, EPS)
    assert_norm_rows(o[1:1 + nrows * k], want, X, k)
    assert np.array_equal(hbuf[1:].cpu().numpy().view(np.uint16), oracle.to_f16(want).ravel())


def test_in_place_and_single_outputs(bm):
    import torch
    nrows, k = 4, 4096
    X = residual("resid.ip", (nrows, k))
    g = norm_weight("norm.ip", k)
    want = oracle.rms_norm_mul(X, g, EPS)
    x = to_dev(X)
    bm.bm_rms_norm_mul(x, to_dev(g), EPS, out=x)
    assert_norm_rows(x.cpu().numpy(), want, X, k)
    _, h = bm.bm_rms_norm_mul(to_dev(X), to_dev(g), EPS, want_out=False)
    assert np.array_equal(h.cpu().numpy().view(np.uint16), oracle.to_f16(want))
    torch.cuda.synchronize()


# (k, rows of each matrix): Q/K/V and gate/up of SmolLM2-135M, Qwen3-0.6B, Llama-3-8B
FRONT_ENDS = [
    (576, (576, 192, 192)), (576, (1536, 1536)), (1024, (2048, 1024, 1024)), (4096, (4096, 1024, 1024)),
    (4096, (14336, 14336)), (64, (8, 16, 24, 32)), (4104, (1000, 13)),
]


@pytest.mark.parametrize("k,rows", FRONT_ENDS)
def test_matvec_norm_front_end(bm, k, rows):
    import torch
    x = residual("resid.fe.%d" % k, k, sigma=3.0)
    g = norm_weight("norm.fe.%d" % k, k)
    Ws = [synth.normal_f16(0, "w.fe.%d.%d.%d" % (k, r, i), 0.02, (r, k)) for i, r in enumerate(rows)]
    n_out = torch.zeros(k, dtype=torch.float32, device="cuda")
    h = torch.zeros(k, dtype=torch.float16, device="cuda")
    ys = bm.bm_f16_matvec_norm([to_dev(W) for W in Ws], to_dev(x), to_dev(g), EPS, n_out=n_out, h=h)
    n_want = oracle.rms_norm_mul(x, g, EPS)
    assert ambiguous_rows(x, k).sum() == 0
    assert np.array_equal(bits32(n_out), bits32(n_want))
    h_want = oracle.to_f16(n_want)
    assert np.array_equal(h.cpu().numpy().view(np.uint16), h_want)
    for y, yw in zip(ys, oracle.matvec_multi(Ws, h_want)):
        assert np.array_equal(bits32(y), bits32(yw))
    assert bm.bm_device_status() == 0


def test_matvec_norm_without_optional_outputs(bm):
    k, rows = 576, (576, 192)
    x = residual("resid.no", k)
    g = norm_weight("norm.no", k)
    Ws = [synth.normal_f16(0, "w.no.%d" % i, 0.02, (r, k)) for i, r in enumerate(rows)]
    ys = bm.bm_f16_matvec_norm([to_dev(W) for W in Ws], to_dev(x), to_dev(g), EPS)
    h_want = oracle.to_f16(oracle.rms_norm_mul(x, g, EPS))
    for y, yw in zip(ys, oracle.matvec_multi(Ws, h_want)):
        assert np.array_equal(bits32(y), bits32(yw))


@pytest.mark.parametrize("k", [100, 7, 1])
def test_matvec_norm_ragged_k(bm, k):
    """k % 8 != 0: the standalone norm kernel writes h, then the lane-per-chain product."""
    import torch
    x = residual("resid.rg.%d" % k, k)
    g = norm_weight("norm.rg.%d" % k, k)
    Ws = [synth.normal_f16(0, "w.rg.%d.%d" % (k, i), 0.5, (r, k)) for i, r in enumerate((40, 3))]
    h = torch.zeros(k, dtype=torch.float16, device="cuda")
    n_out = torch.zeros(k, dtype=torch.float32, device="cuda")
    ys = bm.bm_f16_matvec_norm([to_dev(W) for W in Ws], to_dev(x), to_dev(g), EPS, n_out=n_out, h=h)
    n_want = oracle.rms_norm_mul(x, g, EPS)
    assert np.array_equal(bits32(n_out), bits32(n_want))
    h_want = oracle.to_f16(n_want)
    assert np.array_equal(h.cpu().numpy().view(np.uint16), h_want)
    for y, yw in zip(ys, oracle.matvec_multi(Ws, h_want)):
        assert np.array_equal(bits32(y), bits32(yw))


def test_fused_equals_norm_then_products(bm):
    """The fused launch and the two-launch route (bm_rms_norm_mul, bm_f16_matvec_multi)
    agree bit for bit -- the scale is computed in the same order by every CTA."""
    import torch
    k = 2048
    x = residual("resid.eq", k, sigma=7.0)
    g = norm_weight("norm.eq", k)
    Ws = [to_dev(synth.normal_f16(0, "w.eq.%d" % i, 0.02, (r, k))) for i, r in enumerate((2048, 512, 512))]
    ys = bm.bm_f16_matvec_norm(Ws, to_dev(x), to_dev(g), EPS)
    _, h = bm.bm_rms_norm_mul(to_dev(x), to_dev(g), EPS, want_out=False)
    ys2 = bm.bm_f16_matvec_multi(Ws, h)
    for a, b in zip(ys, ys2):
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_decode_front_end_graph_with_pdl(bm):
    """Token embedding -> first RMS norm with its weight -> Q/K/V, as one decode step's
    front end (forward.md, Design notes, steps three and four), chained with
    programmatic dependent launch, eagerly and replayed from a CUDA graph."""
    import torch
    vocab, k = 4000, 576
    E = synth.normal_f16(0, "embd.fe", 0.02, (vocab, k))
    g = norm_weight("norm.fe", k)
    Ws = [synth.normal_f16(0, "w.fe.qkv.%d" % i, 0.02, (r, k)) for i, r in enumerate((576, 192, 192))]
    dE, dg, dWs = to_dev(E), to_dev(g), [to_dev(W) for W in Ws]
    ids = torch.tensor([1234], dtype=torch.int32, device="cuda")
    emb = torch.empty((1, k), dtype=torch.float32, device="cuda")
    ys = [torch.empty(W.shape[0], dtype=torch.float32, device="cuda") for W in Ws]
    s = torch.cuda.Stream()

    def step():
        bm.bm_f16_get_rows(dE, ids, out=emb, stream=s)
        bm.bm_f16_matvec_norm(dWs, emb.view(-1), dg, EPS, ys=ys, stream=s)

    x = oracle.widen(E[1234])
    want = oracle.matvec_multi(Ws, oracle.to_f16(oracle.rms_norm_mul(x, g, EPS)))
    old = bm.bm_set_pdl(True)
    try:
        with torch.cuda.stream(s):
            step()
        torch.cuda.synchronize()
        for y, yw in zip(ys, want):
            assert np.array_equal(bits32(y), bits32(yw))
        for y in ys:
            y.fill_(float("nan"))
        g_ = torch.cuda.CUDAGraph()
        torch.cuda.synchronize()
        with torch.cuda.graph(g_, stream=s):
            step()
        for _ in range(3):
            g_.replay()
        torch.cuda.synchronize()
        for y, yw in zip(ys, want):
            assert np.array_equal(bits32(y), bits32(yw))
    finally:
        bm.bm_set_pdl(old)
    assert bm.bm_device_status() == 0


def _same_or_both_nan(got, want):
    got, want = np.asarray(got, np.float32), np.asarray(want, np.float32)
    nan = np.isnan(want)
    return np.array_equal(np.isnan(got), nan) and np.array_equal(bits32(got[~nan]), bits32(want[~nan]))


@pytest.mark.parametrize("k", [576, 4096, 6000, 33])
def test_special_rows(bm, k):
    """Rows that take the norm's rarely used steps, against the oracle: an infinite value
    (scale 0, so inf * 0 = NaN there and zeros elsewhere), a NaN, a value whose square
    overflows, values so small that every square is subnormal or tiny (the accumulation
    that keeps subnormal squares), a mean below the normal f32 range (the double
    fallback), and a zero row with eps > 0."""
    rng = np.random.default_rng(k)
    X = rng.normal(0, 1, (7, k)).astype(np.float32)
    X[0, 3] = np.inf
    X[1, k // 2] = np.nan
    X[2, 1] = np.float32(3e19)              # its square overflows to inf
    X[3] *= np.float32(1e-12)               # every square below 2^-63: subnormal handling kept
    X[4] *= np.float32(1e-21)               # squares subnormal or zero, mean below 2^-126
    X[5] = 0.0
    X[6] *= np.float32(1e-19)               # mean near the bottom of the normal range
    g = norm_weight("norm.special.%d" % k, k)
    for eps in (1e-5, 0.0):
        out, _ = bm.bm_rms_norm_mul(to_dev(X), to_dev(g), eps)
        want = oracle.rms_norm_mul(X, g, eps)
        got = out.cpu().numpy()
        amb = ambiguous_rows(np.nan_to_num(X, nan=0.0, posinf=0.0), k)
        for r in range(X.shape[0]):
            if amb[r] and r not in (0, 1, 2):
                continue
            assert _same_or_both_nan(got[r], want[r]), (eps, r)


def test_special_rows_fused(bm):
    """The fused front end takes the same steps (an infinite value and tiny rows)."""
    import torch
    k = 1024
    rng = np.random.default_rng(5)
    g = norm_weight("norm.special.fused", k)
    W = synth.normal_f16(0, "w.special", 0.02, (64, k))
    for scale, spike in ((1.0, np.inf), (1e-12, None), (1e-21, None)):
        x = (rng.normal(0, 1, k) * scale).astype(np.float32)
        if spike is not None:
            x[10] = spike
        n_out = torch.zeros(k, dtype=torch.float32, device="cuda")
        y = bm.bm_f16_matvec_norm([to_dev(W)], to_dev(x), to_dev(g), EPS, n_out=n_out)[0]
        n_want = oracle.rms_norm_mul(x, g, EPS)
        assert _same_or_both_nan(n_out.cpu().numpy(), n_want)
        y_want = oracle.matvec(W, oracle.to_f16(n_want))
        assert _same_or_both_nan(y.cpu().numpy(), y_want)
