"""Closed-form cases of rms_norm then mul (page "docs/modules/forward.md", Technical
usage, "Other public pieces": rms_norm then mul, the sum of squares in double, no FMA;
How it is verified: the unit test on a constant row).

Each case is chosen so that every step is exact, and the expected output is written
down from the mathematics, not computed by the function under test:

- constant rows of a power of two c: every square is exact, the double sum n*c^2 is
  exact, the mean is c^2, its square root |c|, and out = sign(c) * w exactly;
- the row (6, 8, 0, ..., 0) of n = 25: sum 100, mean 4, scale exactly 1/2, so
  out = (3, 4, 0, ...) * w; with (3, 4, 0, ...) and eps = 3 the scale is 1/2 too
  (mean 1 + eps 3 = 4), which pins where eps goes;
- the row (4096, 1, ..., 1) of n = 4097: the squares sum to 2^24 + 4096 in double
  (exactly), the mean is exactly 4096 and the scale 1/64; summed in f32 every +1 would
  be lost against 2^24 and the mean would not be 4096;
- a zero row with eps > 0 gives signed zeros, x -> -x gives -out, and scaling x by a
  power of two leaves out unchanged (eps = 0) -- invariants of the formula.

`failures(f)` runs them all against f(x, w, eps) -> out (one f32 row) and returns the
names of the cases it gets wrong.
"""
import numpy as np


def _w(n, seed):
    return np.random.default_rng(seed).normal(0.0, 1.0, n).astype(np.float32)


def _same(a, b):
    return np.array_equal(np.asarray(a, np.float32).view(np.uint32), np.asarray(b, np.float32).view(np.uint32))


def cases():
    """(name, x, w, eps, expected or None, check) with check(out) -> bool."""
    out = []
    for n in (1, 7, 576, 4096):
        w = _w(n, n)
        for c in (1.0, -1.0, 2.0 ** -10, -(2.0 ** 12), 0.5):
            x = np.full(n, c, np.float32)
            want = (w if c > 0 else -w).astype(np.float32)
            out.append(("constant_row_%d_%g" % (n, c), x, w, 0.0, want))
    n = 25
    w = _w(n, 25)
    x = np.zeros(n, np.float32)
    x[:2] = (6.0, 8.0)
    want = np.zeros(n, np.float32)
    want[:2] = (3.0, 4.0)
    out.append(("six_eight_scale_half", x, w, 0.0, want * w))
    x2 = x.copy()
    x2[:2] = (-6.0, 8.0)
    want2 = want.copy()
    want2[0] = -3.0
    out.append(("six_eight_signed", x2, w, 0.0, want2 * w))
    x3 = np.zeros(n, np.float32)
    x3[:2] = (3.0, 4.0)
    want3 = np.zeros(n, np.float32)
    want3[:2] = (1.5, 2.0)
    out.append(("eps_inside_the_root", x3, w, 3.0, want3 * w))
    x4 = x3.copy()
    x4[5], x4[0] = 3.0, 0.0
    want4 = np.zeros(n, np.float32)
    want4[5], want4[1] = 1.5, 2.0
    out.append(("index_follows_x", x4, w, 3.0, want4 * w))
    n = 4097
    w = _w(n, 4097)
    x = np.ones(n, np.float32)
    x[0] = 4096.0
    want = (x / np.float32(64.0)) * w  # x / 64 is exact for these x
    out.append(("double_accumulation", x, w, 0.0, want.astype(np.float32)))
    return out


def failures(f):
    bad = []
    for name, x, w, eps, want in cases():
        if not _same(f(x, w, eps), want):
            bad.append(name)
    # a zero row with eps > 0: (0 * scale) * w, the zero taking w's sign
    n = 64
    w = _w(n, 64)
    z = f(np.zeros(n, np.float32), w, 1e-5)
    if not (np.all(z == 0) and np.array_equal(np.signbit(z), np.signbit(w))):
        bad.append("zero_row")
    rng = np.random.default_rng(11)
    for n in (3, 100, 576):
        x = rng.normal(0, 1, n).astype(np.float32)
        w = _w(n, n + 1)
        eps = np.float32(1e-6)
        y = f(x, w, eps)
        if not _same(f(-x, w, eps), -y):
            bad.append("odd_in_x_%d" % n)
        y0 = f(x, w, 0.0)
        for p in (-8, 5, 20):
            if not _same(f(x * np.float32(2.0 ** p), w, 0.0), y0):
                bad.append("scale_invariance_%d_%d" % (n, p))
    return bad
