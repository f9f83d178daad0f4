"""Pins of the CPU oracle against what the pages and the mathematics fix.

The oracle restates the page "docs/modules/f16.md" (bankML): section "Design
notes" (activation rounding, vec_dot and sgemm_dot orders) and section
"Technical usage" / "Matrix products" (takes_sgemm, mat_vec_par,
mat_vec_multi_par, mat_mul_par).  None of these tests recomputes the oracle's
own formula: they use hand-derived worked examples (tests/golden/), IEEE-754
closed forms, the C compiler's own f16 conversion, exact rational sums and
exact integer sums.
"""
import json
import os
import struct
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from conftest import GOLDEN


def f32_bits(x) -> int:
    return struct.unpack("<I", struct.pack("<f", float(x)))[0]


def bits_f32(u: int) -> float:
    return struct.unpack("<f", struct.pack("<I", u))[0]


def f16_value(h: int) -> Fraction:
    """IEEE binary16 closed form: (-1)^s 2^(e-15) (1 + m/1024), or m 2^-24."""
    s, e, m = (h >> 15) & 1, (h >> 10) & 31, h & 1023
    assert e != 31
    v = Fraction(m, 1 << 24) if e == 0 else Fraction(1024 + m, 1024) * Fraction(2) ** (e - 15)
    return -v if s else v


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------- widen


def test_widen_exhaustive_closed_form():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.widen(h)
    for v in range(65536):
        e = (v >> 10) & 31
        if e == 31:
            if v & 1023:
                assert np.isnan(got[v])
            else:
                assert np.isinf(got[v]) and (got[v] < 0) == bool(v >> 15)
            continue
        want = f16_value(v)
        assert Fraction(float(got[v])) == want, hex(v)
        if want == 0:
            assert f32_bits(got[v]) >> 31 == v >> 15  # signed zero kept


def test_widen_matches_compiler_f16():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle.widen(h)
    ref = h.view(np.float16).astype(np.float32)
    finite = ~np.isnan(ref)
    assert (got[finite].view(np.uint32) == ref[finite].view(np.uint32)).all()


def test_round_trip_every_non_nan_f16():
    h = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    nan = ((h & 0x7c00) == 0x7c00) & ((h & 0x3ff) != 0)
    back = oracle.to_f16(oracle.widen(h))
    assert (back[~nan] == h[~nan]).all()


# --------------------------------------------------------------------------- to_f16


def test_to_f16_boundary_cases():
    for fb, hb, why in load("to_f16_cases.json")["cases"]:
        x = np.array([bits_f32(int(fb, 16))], dtype=np.float32)
        got = int(oracle.to_f16(x)[0])
        assert got == int(hb, 16), (fb, hex(got), why)


def test_to_f16_exhaustive_vs_compiler_conversion():
    """All 2^32 f32 patterns (NaN excluded) against the C compiler's _Float16."""
    bad, first = oracle.check_to_f16_vs_compiler(0, 1 << 32)
    assert bad == 0, "first mismatch at f32 bits 0x%08x" % first


def test_to_f16_is_nearest_ties_to_even():
    """The result is the nearest f16 (by exact rationals), ties to the even code."""
    rng = np.random.default_rng(1)
    pats = rng.integers(0, 1 << 32, size=20000, dtype=np.uint64).astype(np.uint32)
    xs = pats.view(np.float32)
    xs = xs[np.isfinite(xs) & (np.abs(xs) < 65504)]
    hs = oracle.to_f16(xs)
    for x, h in zip(xs.tolist(), hs.tolist()):
        X = Fraction(x)
        v = f16_value(h)
        mag = h & 0x7fff
        # neighbours of the chosen code on the same side of zero
        cands = [f16_value((h & 0x8000) | c) for c in (mag - 1, mag + 1) if 0 <= c < 0x7c00]
        if mag == 0:
            cands.append(f16_value(0x8001 if h == 0 else 0x0001))
        d = abs(X - v)
        for c in cands:
            dc = abs(X - c)
            assert d < dc or (d == dc and (mag & 1) == 0), (x, hex(h))


# --------------------------------------------------------------------------- takes_sgemm


def test_takes_sgemm_truth_table():
    for rows, k, n, want in load("takes_sgemm_table.json")["table"]:
        assert oracle.takes_sgemm(rows, k, n) == bool(want), (rows, k, n)


# --------------------------------------------------------------------------- reductions


def example_vectors(ex):
    k = ex["k"]
    w = np.zeros(k, dtype=np.uint16)
    a = np.zeros(k, dtype=np.uint16)
    for i, wb, ab in ex["terms"]:
        w[i] = int(wb, 16)
        a[i] = int(ab, 16)
    return w, a


@pytest.mark.parametrize("ex", load("reduction_examples.json")["examples"], ids=lambda e: e["name"])
def test_worked_reduction_examples(ex):
    w, a = example_vectors(ex)
    assert f32_bits(oracle.vec_dot_ref(w, a)) == int(ex["vec_dot"], 16), ex["why"]
    if ex["sgemm"] is not None:
        assert f32_bits(oracle.sgemm_dot_ref(w, a)) == int(ex["sgemm"], 16), ex["why"]


def test_exact_integer_sums():
    """Small-integer inputs whose partial sums stay below 2^24 are summed exactly on
    both paths, whatever the order: any dropped, repeated or mis-signed term shows."""
    rng = np.random.default_rng(7)
    for k in [1, 7, 8, 31, 32, 33, 63, 64, 65, 96, 100, 255, 256, 1000, 1537]:
        wi = rng.integers(-16, 17, size=k)
        ai = rng.integers(-16, 17, size=k)
        w = wi.astype(np.float16).view(np.uint16)
        a = ai.astype(np.float16).view(np.uint16)
        exact = int(np.dot(wi, ai))
        assert float(oracle.vec_dot_ref(w, a)) == exact
        if k % 8 == 0:
            assert float(oracle.sgemm_dot_ref(w, a)) == exact


def gamma(n):
    u = Fraction(1, 1 << 24)
    return n * u / (1 - n * u)


def test_brute_force_error_bounds():
    """Against exact rational sums: recursive-summation bounds for each path's chain
    length (vec_dot: k/32 adds per chain + 5 reduction levels, then one rounding of
    the double; sgemm: k/8 adds per lane + 3 levels)."""
    rng = np.random.default_rng(11)
    for trial in range(60):
        k = int(rng.integers(1, 400))
        if trial % 3 == 0:
            k = 8 * max(1, k // 8)
        w = synth.normal_f16(trial, 0, 0.5, k)
        a = synth.normal_f16(trial, 1, 2.0, k)
        ps = [f16_value(int(x)) * f16_value(int(y)) for x, y in zip(w, a)]
        S = sum(ps, Fraction(0))
        A = sum((abs(p) for p in ps), Fraction(0))
        vd = Fraction(float(oracle.vec_dot_ref(w, a)))
        bound = gamma(k // 32 + 5) * A + Fraction(1, 1 << 23) * abs(S) + Fraction(1, 1 << 60)
        assert abs(vd - S) <= bound, (k, float(vd), float(S))
        if k % 8 == 0:
            sg = Fraction(float(oracle.sgemm_dot_ref(w, a)))
            assert abs(sg - S) <= gamma(k // 8 + 3) * A, (k, float(sg), float(S))
        ad = Fraction(oracle.abs_dot(w, a))
        assert abs(ad - A) <= A * Fraction(1, 1 << 40)


def test_fma_and_mul_add_agree_on_f16_products():
    """Every f16 x f16 product is exact in f32, so fma(w, a, c) == c + w*a: the
    oracle's plain multiply-then-add is the FMA chain of the page's kernels."""
    rng = np.random.default_rng(3)
    h = rng.integers(0, 1 << 16, size=(200000, 2), dtype=np.uint32).astype(np.uint16)
    fin = ((h & 0x7c00) != 0x7c00).all(axis=1)
    h = h[fin]
    w = [f16_value(int(x)) for x in h[:, 0]]
    a = [f16_value(int(x)) for x in h[:, 1]]
    wf = h[:, 0].view(np.float16).astype(np.float32)
    af = h[:, 1].view(np.float16).astype(np.float32)
    prod = (wf * af).astype(np.float32)
    for i in range(0, len(w), 97):
        assert Fraction(float(prod[i])) == w[i] * a[i]


# --------------------------------------------------------------------------- products


def int_matrix(rng, shape, lo=-8, hi=9):
    v = rng.integers(lo, hi, size=shape)
    return v, v.astype(np.float16).view(np.uint16)


def test_matmul_layout_and_path_by_shape():
    """out[c*rows + r] = dot(W[r], X[c]) (exact integers); the path follows the shape."""
    rng = np.random.default_rng(5)
    for rows, k, ncols in [(12, 40, 3), (13, 40, 3), (12, 33, 2), (8, 64, 1), (4, 8, 5)]:
        Wi, W = int_matrix(rng, (rows, k))
        Xi, X = int_matrix(rng, (ncols, k))
        Y = oracle.matmul(W, X)
        assert Y.shape == (ncols, rows)
        for c in range(ncols):
            for r in range(rows):
                assert float(Y[c, r]) == int(np.dot(Wi[r], Xi[c]))
        if ncols > 1:
            assert float(Y.reshape(-1)[1 * rows + 2]) == int(np.dot(Wi[2], Xi[1]))


def test_path_choice_12_vs_13_rows():
    """E1's row repeated: 12 rows x 2 columns take tinyBLAS (0.0), 13 rows fall back to
    vec_dot (1.0), one column is always vec_dot, and k % 8 != 0 falls back."""
    ex = {e["name"]: e for e in load("reduction_examples.json")["examples"]}["E1_two_reductions_differ"]
    w, a = example_vectors(ex)
    X2 = np.stack([a, a])
    for rows, X, want in [(12, X2, 0.0), (13, X2, 1.0), (12, a[None, :], 1.0), (16, X2, 0.0)]:
        W = np.tile(w, (rows, 1))
        Y = oracle.matmul(W, X)
        assert (Y == want).all(), (rows, X.shape)
        assert all(f32_bits(v) == f32_bits(want) for v in Y.reshape(-1))
    wp = np.concatenate([w, np.zeros(4, np.uint16)])
    ap = np.concatenate([a, np.zeros(4, np.uint16)])
    Y = oracle.matmul(np.tile(wp, (12, 1)), np.stack([ap, ap]))
    assert (Y == 1.0).all()


def test_matvec_multi_is_separate_matvecs():
    k = 96
    Ws = [synth.normal_f16(0, t, 0.02, (r, k)) for t, r in enumerate([20, 7, 7])]
    x = synth.normal_f16(0, 9, 1.0, k)
    ys = oracle.matvec_multi(Ws, x)
    for W, y in zip(Ws, ys):
        assert (y.view(np.uint32) == oracle.matvec(W, x).view(np.uint32)).all()


def test_matmul_sample_and_abs():
    rows, k, ncols = 16, 72, 3
    W = synth.normal_f16(1, 0, 0.02, (rows, k))
    X = synth.normal_f16(1, 1, 1.0, (ncols, k))
    Y = oracle.matmul(W, X)
    ri = np.array([0, 5, 15, 3])
    ci = np.array([0, 2, 1, 2])
    got, ab = oracle.matmul_sample(W, X, ri, ci)
    assert (got.view(np.uint32) == Y[ci, ri].view(np.uint32)).all()
    full = oracle.abs_matmul(W, X)
    assert np.array_equal(ab, full[ci, ri])


def test_thread_count_does_not_change_bits():
    """OpenMP splits whole elements only (the pages' invariant: the split decides who
    computes an element, never its bits)."""
    import subprocess
    import sys
    code = ("import numpy as np, oracle, synth; W = synth.normal_f16(0,0,0.02,(257,1000)); "
            "X = synth.normal_f16(0,1,1.0,(3,1000)); print(oracle.matmul(W,X).view(np.uint32).sum(dtype=np.uint64))")
    outs = set()
    for t in ("1", "3"):
        env = dict(os.environ, OMP_NUM_THREADS=t)
        r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                           cwd=os.path.dirname(os.path.dirname(GOLDEN)), check=True)
        outs.add(r.stdout.strip())
    assert len(outs) == 1


def test_output_rows_choose_the_path():
    """forward.md, "Why only the output rows leave the last layer": the last layer's
    products see only the output rows, so their count picks the path.  Over an FFN
    shape (1536 x 576), the last row alone takes vec_dot and the same row among 7
    takes sgemm_dot -- each element checked against the per-element reference of
    its path, and the two differ in some elements."""
    rows, k, n = 1536, 576, 7
    W = synth.normal_f16(0, "outids.gate", 0.02, (rows, k))
    X = oracle.to_f16(synth.normal_f32(0, "outids.x", 1.0, (n, k)))
    assert oracle.takes_sgemm(rows, k, n) and not oracle.takes_sgemm(rows, k, 1)
    all_rows = oracle.matmul(W, X)[n - 1]
    last_only = oracle.matmul(W, X[n - 1:])[0]
    for r in range(0, rows, 97):
        assert f32_bits(all_rows[r]) == f32_bits(oracle.sgemm_dot_ref(W[r], X[n - 1]))
        assert f32_bits(last_only[r]) == f32_bits(oracle.vec_dot_ref(W[r], X[n - 1]))
    differ = np.count_nonzero(all_rows.view(np.uint32) != last_only.view(np.uint32))
    assert 0 < differ < rows
