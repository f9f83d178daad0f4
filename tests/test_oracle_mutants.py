"""Mistakes planted in a copy of the oracle (on the CPU) must be caught by the pins.

Each mutant is oracle.c with one plausible slip -- a transposed pairing, a dropped
term, a wrong sign or index, a float tail, a wrong rounding rule, a norm summed in
float or with eps in the wrong place -- compiled into
a temporary library and run through the same page-derived checks the pin tests
use.  The unmutated source passes every check; each mutant must fail at least one.
"""
import ctypes as C
import json
import os
import subprocess
import tempfile

import numpy as np
import pytest

import norm_cases
from conftest import GOLDEN, ROOT

SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    "accumulator_pairing": ("(acc[0][l] + acc[2][l]) + (acc[1][l] + acc[3][l])",
                            "(acc[0][l] + acc[1][l]) + (acc[2][l] + acc[3][l])"),
    "low_high_pairs": ("t[m] = v[m] + v[m + 4]", "t[m] = v[2 * m] + v[2 * m + 1]"),
    "hadd_pairs": ("float h0 = t[0] + t[1];                                 /* first horizontal add */\n    float h1 = t[2] + t[3];",
                   "float h0 = t[0] + t[2];\n    float h1 = t[1] + t[3];"),
    "tail_in_float": ("double sumf = (double)r;", "float sumf = r;"),
    "tail_after_R": ("double sumf = (double)r;\n    for (int64_t i = k32; i < k; i++) sumf += (double)(or_widen(w[i]) * or_widen(a[i]));",
                     "double sumf = 0.0;\n    for (int64_t i = k32; i < k; i++) sumf += (double)(or_widen(w[i]) * or_widen(a[i]));\n    sumf += (double)r;"),
    "lane_index_transposed": ("int64_t i = s + 8 * j + l;", "int64_t i = s + 4 * l + j;"),
    "dropped_first_step": ("for (int64_t s = 0; s < k32; s += 32)", "for (int64_t s = 32; s < k32; s += 32)"),
    "wrong_sign": ("acc[j][l] = acc[j][l] + or_widen(w[i]) * or_widen(a[i]);",
                   "acc[j][l] = acc[j][l] - or_widen(w[i]) * or_widen(a[i]);"),
    "negative_zero_start": ("for (int l = 0; l < 8; l++) acc[j][l] = 0.0f;", "for (int l = 0; l < 8; l++) acc[j][l] = -0.0f;"),
    "sgemm_hsum_pairs": ("((l[0] + l[4]) + (l[2] + l[6])) + ((l[1] + l[5]) + (l[3] + l[7]))",
                         "((l[0] + l[1]) + (l[2] + l[3])) + ((l[4] + l[5]) + (l[6] + l[7]))"),
    # (swapping neighbouring lanes or rotating them is not a mistake: the hsum is symmetric
    # under those relabelings and the bits never change, so they are not listed)
    "sgemm_lanes_1_4_swapped": ("l[q] = l[q] + or_widen(w[i + q]) * or_widen(a[i + q]);",
                                "l[q] = l[q] + or_widen(w[i + (q == 1 ? 4 : q == 4 ? 1 : q)]) * "
                                "or_widen(a[i + (q == 1 ? 4 : q == 4 ? 1 : q)]);"),
    "sgemm_reversed_chain": ("for (int64_t i = 0; i < k; i += 8)", "for (int64_t i = k - 8; i >= 0; i -= 8)"),
    "takes_sgemm_rows": ("n >= 2 && rows % 4 == 0 && k % 8 == 0", "n >= 2 && rows % 2 == 0 && k % 8 == 0"),
    "takes_sgemm_one_column": ("n >= 2 && rows % 4 == 0 && k % 8 == 0", "n >= 1 && rows % 4 == 0 && k % 8 == 0"),
    "to_f16_ties_away": ("if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1;",
                         "if (rem >= 0x1000u) h += 1;"),
    "to_f16_overflow_threshold": ("if (a >= 0x477ff000u) return sign | 0x7c00u;", "if (a >= 0x477fe000u) return sign | 0x7c00u;"),
    "to_f16_subnormal_shift": ("uint32_t shift = 126 - e;", "uint32_t shift = 125 - e;"),
    "widen_subnormal_scale": ("float v = (float)m * 0x1p-24f;", "float v = (float)m * 0x1p-25f;"),
    "matmul_layout_transposed": ("int64_t c = e / rows, r = e % rows;", "int64_t r = e / ncols, c = e % ncols;"),
    "norm_sum_in_float": ("    double sum = 0.0;\n    for (int64_t i = 0; i < n; i++) {\n        float sq = x[i] * x[i];\n"
                          "        sum += (double)sq;",
                          "    float sum = 0.0f;\n    for (int64_t i = 0; i < n; i++) {\n        float sq = x[i] * x[i];\n"
                          "        sum += sq;"),
    "norm_dropped_first_square": ("for (int64_t i = 0; i < n; i++) {\n        float sq",
                                  "for (int64_t i = 1; i < n; i++) {\n        float sq"),
    "norm_mean_over_n_minus_1": ("(float)(sum / (double)n)", "(float)(sum / (double)(n > 1 ? n - 1 : 1))"),
    "norm_eps_outside_root": ("1.0f / sqrtf(mean + eps)", "1.0f / sqrtf(mean) + eps"),
    "norm_no_root": ("1.0f / sqrtf(mean + eps)", "1.0f / (mean + eps)"),
    "norm_sign_lost": ("float y = x[i] * scale;", "float y = fabsf(x[i]) * scale;"),
    "norm_weight_reversed": ("out[i] = y * w[i];", "out[i] = y * w[n - 1 - i];"),
    "norm_weight_dropped": ("out[i] = y * w[i];", "out[i] = y;"),
    "mad_two_roundings": ("acc[i] = or_to_f16(fmaf(or_widen(v[i]), w, or_widen(acc[i])));",
                          "acc[i] = or_to_f16(or_widen(v[i]) * w + or_widen(acc[i]));"),
    "mad_roles_swapped": ("acc[i] = or_to_f16(fmaf(or_widen(v[i]), w, or_widen(acc[i])));",
                          "acc[i] = or_to_f16(fmaf(or_widen(acc[i]), w, or_widen(v[i])));"),
    "mad_last_element_skipped": ("for (int64_t i = 0; i < n; i++) acc[i] = or_to_f16(fmaf(",
                                 "for (int64_t i = 0; i + 1 < n; i++) acc[i] = or_to_f16(fmaf("),
    "scale_divides": ("acc[i] = or_to_f16(or_widen(acc[i]) * s);", "acc[i] = or_to_f16(or_widen(acc[i]) / s);"),
}


def build(src_text, d, name):
    c = os.path.join(d, name + ".c")
    so = os.path.join(d, name + ".so")
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O2", "-std=gnu11", "-ffp-contract=off", "-fno-fast-math", "-fopenmp", "-fPIC",
                    "-shared", "-I", os.path.join(ROOT, "oracle"), "-o", so, c, "-lm"], check=True)
    L = C.CDLL(so)
    u16p, f32p = C.POINTER(C.c_uint16), C.POINTER(C.c_float)
    L.or_vec_dot_ref.argtypes = [u16p, u16p, C.c_int64]; L.or_vec_dot_ref.restype = C.c_float
    L.or_sgemm_dot_ref.argtypes = [u16p, u16p, C.c_int64]; L.or_sgemm_dot_ref.restype = C.c_float
    L.or_takes_sgemm.argtypes = [C.c_int64] * 3; L.or_takes_sgemm.restype = C.c_int
    L.or_to_f16.argtypes = [C.c_float]; L.or_to_f16.restype = C.c_uint16
    L.or_widen.argtypes = [C.c_uint16]; L.or_widen.restype = C.c_float
    L.or_matmul.argtypes = [u16p, C.c_int64, C.c_int64, u16p, C.c_int64, f32p]; L.or_matmul.restype = None
    L.or_rms_norm_mul.argtypes = [f32p, f32p, C.c_int64, C.c_float, f32p]; L.or_rms_norm_mul.restype = None
    L.or_f16_mad.argtypes = [u16p, u16p, C.c_float, C.c_int64]; L.or_f16_mad.restype = None
    L.or_f16_scale.argtypes = [u16p, C.c_float, C.c_int64]; L.or_f16_scale.restype = None
    return L


def f32_bits(x):
    return int(np.array([x], dtype=np.float32).view(np.uint32)[0])


def failures(L):
    """Run the page-derived checks; return the names of those that fail."""
    bad = []
    P = lambda a: a.ctypes.data_as(C.POINTER(C.c_uint16))
    ex = json.load(open(os.path.join(GOLDEN, "reduction_examples.json")))["examples"]
    for e in ex:
        k = e["k"]
        w = np.zeros(k, np.uint16)
        a = np.zeros(k, np.uint16)
        for i, wb, ab in e["terms"]:
            w[i], a[i] = int(wb, 16), int(ab, 16)
        if f32_bits(L.or_vec_dot_ref(P(w), P(a), k)) != int(e["vec_dot"], 16):
            bad.append("example:" + e["name"])
        if e["sgemm"] is not None and f32_bits(L.or_sgemm_dot_ref(P(w), P(a), k)) != int(e["sgemm"], 16):
            bad.append("example_sgemm:" + e["name"])
    for fb, hb, _ in json.load(open(os.path.join(GOLDEN, "to_f16_cases.json")))["cases"]:
        x = np.array([int(fb, 16)], np.uint32).view(np.float32)[0]
        if L.or_to_f16(float(x)) != int(hb, 16):
            bad.append("to_f16:" + fb)
    for h in list(range(0, 1024, 37)) + [0x3c00, 0x0400, 0x7bff, 0x8001]:
        s, e_, m = (h >> 15) & 1, (h >> 10) & 31, h & 1023
        want = (m * 2.0 ** -24 if e_ == 0 else (1 + m / 1024) * 2.0 ** (e_ - 15)) * (-1 if s else 1)
        if float(L.or_widen(h)) != want:
            bad.append("widen:%x" % h)
    for rows, k, n, want in json.load(open(os.path.join(GOLDEN, "takes_sgemm_table.json")))["table"]:
        if L.or_takes_sgemm(rows, k, n) != want:
            bad.append("takes_sgemm")
    rng = np.random.default_rng(7)
    for k in (7, 32, 33, 100, 256):
        wi, ai = rng.integers(-16, 17, size=k), rng.integers(-16, 17, size=k)
        w, a = wi.astype(np.float16).view(np.uint16), ai.astype(np.float16).view(np.uint16)
        if float(L.or_vec_dot_ref(P(w), P(a), k)) != int(np.dot(wi, ai)):
            bad.append("integer_sum:%d" % k)
    for rows, k, ncols in ((12, 40, 3), (13, 40, 3)):
        Wi, Xi = rng.integers(-8, 9, size=(rows, k)), rng.integers(-8, 9, size=(ncols, k))
        W, X = Wi.astype(np.float16).view(np.uint16), Xi.astype(np.float16).view(np.uint16)
        Y = np.empty((ncols, rows), np.float32)
        L.or_matmul(P(W), rows, k, P(X), ncols, Y.ctypes.data_as(C.POINTER(C.c_float)))
        if not np.array_equal(Y, (Xi @ Wi.T).astype(np.float32)):
            bad.append("matmul_layout")

    def norm(x, w, eps):
        x, w = np.ascontiguousarray(x, np.float32), np.ascontiguousarray(w, np.float32)
        out = np.empty_like(x)
        F = lambda a: a.ctypes.data_as(C.POINTER(C.c_float))
        L.or_rms_norm_mul(F(x), F(w), x.size, float(np.float32(eps)), F(out))
        return out

    bad += ["norm:" + b for b in norm_cases.failures(norm)]

    # mad and scale against numpy's float32 arithmetic and float16 conversion
    def f16(x):
        with np.errstate(over="ignore"):
            return np.asarray(x, np.float32).astype(np.float16).view(np.uint16)

    hs = np.arange(0, 1 << 16, 7, dtype=np.uint32).astype(np.uint16)
    hs = hs[np.isfinite(hs.view(np.float16))]
    for sc in (0.5, 3.0, 0.1):
        got = hs.copy()
        L.or_f16_scale(P(got), float(np.float32(sc)), got.size)
        with np.errstate(over="ignore"):
            if not np.array_equal(got, f16(hs.view(np.float16).astype(np.float32) * np.float32(sc))):
                bad.append("scale:%g" % sc)
    v = f16(rng.uniform(1, 2, 20000))
    wm = np.float32(1.00123456)  # 24 significant bits: v * wm is not exact in f32
    prod = v.view(np.float16).astype(np.float64) * np.float64(wm)
    acc = f16(-prod.astype(np.float32))  # near cancellation: the f32 rounding of a product shows
    acc[::2] = f16(rng.uniform(-4, 4, acc[::2].size))
    want = f16((acc.view(np.float16).astype(np.float64) + prod).astype(np.float32))
    got = acc.copy()
    L.or_f16_mad(P(got), P(v), float(wm), got.size)
    if not np.array_equal(got, want):
        bad.append("mad")
    return bad


@pytest.fixture(scope="module")
def workdir():
    with tempfile.TemporaryDirectory() as d:
        yield d


def test_unmutated_oracle_passes_every_check(workdir):
    assert failures(build(open(SRC).read(), workdir, "clean")) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(workdir, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert old in src, "mutation site not found: " + name
    bad = failures(build(src.replace(old, new, 1), workdir, name))
    assert bad, "mutant %s passed every check" % name
