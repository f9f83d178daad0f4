"""The C-ABI boundary without a GPU: the library builds and loads, exports every
symbol include/bm.h declares, and rejects bad arguments on the host before any
CUDA call (every case here returns before the library touches the device)."""
import ctypes as C
import json
import os
import re

import pytest

from conftest import GOLDEN, ROOT

HEADER = os.path.join(ROOT, "include", "bm.h")


@pytest.fixture(scope="module")
def L():
    from f16_weight_gemv_gb300 import _build
    import f16_weight_gemv_gb300 as bm
    _build.build()
    return bm.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bm_\w+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ["bm_to_f16", "bm_f16_matvec", "bm_f16_matvec_multi", "bm_f16_matmul", "bm_f16_logits",
              "bm_takes_sgemm", "bm_status_string", "bm_last_error", "bm_device_status"]:
        assert n in names


def test_library_exports_every_declared_symbol(L):
    import f16_weight_gemv_gb300 as bm
    for name in declared_functions():
        assert hasattr(L, name), name
        assert name in bm.EXPORTS, name
        assert hasattr(bm, name), name  # same name in the Python binding


def test_takes_sgemm_through_the_abi(L):
    table = json.load(open(os.path.join(GOLDEN, "takes_sgemm_table.json")))["table"]
    for rows, k, n, want in table:
        assert L.bm_takes_sgemm(rows, k, n) == want, (rows, k, n)


def test_status_strings(L):
    for s in range(6):
        assert L.bm_status_string(s)
    assert L.bm_status_string(99) == b"unknown status"


A = 0x100000  # a 16-byte aligned fake device address; never dereferenced here


def st(L, name, *args):
    return getattr(L, name)(*args)


def test_to_f16_host_checks(L):
    assert st(L, "bm_to_f16", A, A + 4096, -1, None) == 1
    assert st(L, "bm_to_f16", A, A + 4096, 0, None) == 0
    assert st(L, "bm_to_f16", None, A, 8, None) == 1
    assert L.bm_last_error()
    assert st(L, "bm_to_f16", A + 4, A + 4096, 8, None) == 2
    assert st(L, "bm_to_f16", A, A + 4098, 8, None) == 2
    assert st(L, "bm_to_f16", A, A + 16, 8, None) == 1  # h overlaps x


def test_matvec_host_checks(L):
    f = "bm_f16_matvec"
    assert st(L, f, A, 16, 0, A + 2 ** 20, A + 2 ** 21, None) == 1            # k = 0
    assert st(L, f, A, 16, 65537, A + 2 ** 24, A + 2 ** 25, None) == 1      # k > BM_MAX_K
    assert st(L, f, A, -1, 64, A + 2 ** 20, A + 2 ** 21, None) == 1
    assert st(L, f, A, 0, 64, A + 2 ** 20, A + 2 ** 21, None) == 0           # empty: nothing launched
    assert L.bm_last_error() == b""
    assert st(L, f, None, 16, 64, A + 2 ** 20, A + 2 ** 21, None) == 1
    assert st(L, f, A + 2, 16, 64, A + 2 ** 20, A + 2 ** 21, None) == 2
    assert st(L, f, A, 16, 64, A + 2 ** 20 + 8, A + 2 ** 21, None) == 2
    assert st(L, f, A, 16, 64, A + 2 ** 20, A + 2 ** 21 + 2, None) == 2
    assert st(L, f, A, 16, 64, A + 2 ** 20, A + 64, None) == 1               # y inside W
    assert st(L, f, A, 2 ** 62, 64, A + 2 ** 20, A + 2 ** 21, None) == 1     # size overflow


def test_matvec_multi_host_checks(L):
    f = L.bm_f16_matvec_multi
    W = (C.c_void_p * 5)(A, A + 2 ** 20, A + 2 ** 21, A + 2 ** 22, A + 2 ** 23)
    y = (C.c_void_p * 5)(A + 2 ** 24, A + 2 ** 24 + 4096, A + 2 ** 24 + 8192, A + 2 ** 24 + 12288, A + 2 ** 25)
    rows = (C.c_int64 * 5)(16, 16, 16, 16, 16)
    assert f(0, W, rows, 64, A + 2 ** 26, y, None) == 1
    assert f(5, W, rows, 64, A + 2 ** 26, y, None) == 1
    assert f(2, None, rows, 64, A + 2 ** 26, y, None) == 1
    yo = (C.c_void_p * 2)(A + 2 ** 24, A + 2 ** 24 + 32)                    # outputs overlap
    assert f(2, W, rows, 64, A + 2 ** 26, yo, None) == 1
    z = (C.c_int64 * 2)(0, 0)
    assert f(2, W, z, 64, A + 2 ** 26, y, None) == 0                         # all empty


def test_matmul_host_checks(L):
    for f in ("bm_f16_matmul", "bm_f16_logits"):
        assert st(L, f, A, 16, 64, A + 2 ** 20, 0, A + 2 ** 21, None) == 0
        assert st(L, f, A, 16, 64, A + 2 ** 20, -3, A + 2 ** 21, None) == 1
        assert st(L, f, A, 16, 64, A + 2 ** 20 + 4, 2, A + 2 ** 21, None) == 2
        assert st(L, f, A, 16, 64, A + 2 ** 20, 2, A + 2 ** 20 + 64, None) == 1  # Y overlaps X
        assert st(L, f, A, 2 ** 40, 64, A + 2 ** 20, 2 ** 30, A + 2 ** 21, None) == 1


def test_get_rows_host_checks(L):
    f = L.bm_f16_get_rows
    assert f(A, 16, 64, A + 2 ** 20, 0, A + 2 ** 21, None) == 0                 # n = 0: nothing to do
    assert f(A, 16, 64, A + 2 ** 20, -1, A + 2 ** 21, None) == 1
    assert f(A, 0, 64, A + 2 ** 20, 3, A + 2 ** 21, None) == 1                  # empty table
    assert f(None, 16, 64, A + 2 ** 20, 3, A + 2 ** 21, None) == 1
    assert f(A + 2, 16, 64, A + 2 ** 20, 3, A + 2 ** 21, None) == 2             # table misaligned
    assert f(A, 16, 64, A + 2 ** 20 + 4, 3, A + 2 ** 21, None) == 2             # ids misaligned
    assert f(A, 16, 64, A + 2 ** 20, 3, A + 2 ** 21 + 2, None) == 2             # output misaligned
    assert f(A, 16, 64, A + 2 ** 20, 3, A + 64, None) == 1                      # output overlaps the table


def test_exact_sgemm_cols_setting(L):
    """bm_set_exact_sgemm_cols clamps to 0..8 and returns the previous value (host only)."""
    old = L.bm_set_exact_sgemm_cols(5)
    assert 0 <= old <= 8
    assert L.bm_set_exact_sgemm_cols(100) == 5
    assert L.bm_set_exact_sgemm_cols(-3) == 8
    assert L.bm_set_exact_sgemm_cols(old) == 0


def test_product_path_is_cuda_only():
    """The binding has no CPU fallback: it loads libbm.so or fails, and never imports the oracle."""
    import f16_weight_gemv_gb300 as bm
    src = open(bm.__file__).read() + open(os.path.join(os.path.dirname(bm.__file__), "_build.py")).read()
    assert "import oracle" not in src and "from oracle" not in src
    csrc = os.path.join(os.path.dirname(bm.__file__), "csrc")
    for fn in os.listdir(csrc):
        assert "oracle.h" not in open(os.path.join(csrc, fn)).read()


def test_matvec_act_host_checks(L):
    f = L.bm_f16_matvec_act
    W = (C.c_void_p * 2)(A, A + 2 ** 20)
    y = (C.c_void_p * 2)(A + 2 ** 24, A + 2 ** 24 + 4096)
    rows = (C.c_int64 * 2)(16, 16)
    x, h = A + 2 ** 26, A + 2 ** 27
    assert f(0, W, rows, 64, x, h, y, None) == 1
    assert f(2, W, rows, 0, x, h, y, None) == 1
    assert f(2, W, rows, 64, None, h, y, None) == 1
    assert f(2, W, rows, 64, x + 4, h, y, None) == 2
    assert f(2, W, rows, 64, x, h + 2, y, None) == 2
    assert f(2, W, rows, 64, x, x + 16, y, None) == 1      # h overlaps x
    yo = (C.c_void_p * 2)(A + 2 ** 24, x + 8)               # y overlaps x
    assert f(2, W, rows, 64, x, h, yo, None) == 1


def test_matmul_noalloc_host_checks(L):
    f = "bm_f16_matmul_noalloc"
    assert st(L, f, A, 16, 64, A + 2 ** 20, 0, A + 2 ** 21, None) == 0
    assert st(L, f, A, 16, 0, A + 2 ** 20, 2, A + 2 ** 21, None) == 1
    assert st(L, f, A + 2, 16, 64, A + 2 ** 20, 2, A + 2 ** 21, None) == 2
    assert st(L, f, A, 16, 64, A + 2 ** 20, 2, A + 2 ** 20 + 64, None) == 1


def test_matvec_norm_host_checks(L):
    f = L.bm_f16_matvec_norm
    W = (C.c_void_p * 2)(A, A + 2 ** 20)
    y = (C.c_void_p * 2)(A + 2 ** 24, A + 2 ** 24 + 4096)
    rows = (C.c_int64 * 2)(16, 16)
    x, g, n, h = A + 2 ** 26, A + 2 ** 26 + 2 ** 16, A + 2 ** 26 + 2 ** 17, A + 2 ** 27
    assert f(0, W, rows, 64, x, g, 1e-5, n, h, y, None) == 1
    assert f(2, W, rows, 64, x, None, 1e-5, n, h, y, None) == 1          # no norm weight
    assert f(2, W, rows, 64, x, g + 4, 1e-5, n, h, y, None) == 2         # g misaligned
    assert f(2, W, rows, 64, x, g, 1e-5, n + 8, h, y, None) == 2         # n_out misaligned
    assert f(2, W, rows, 64, x, g, 1e-5, x + 16, h, y, None) == 1        # n_out overlaps x
    assert f(2, W, rows, 64, x, g, 1e-5, g, h, y, None) == 1             # n_out overlaps g
    assert f(2, W, rows, 64, x, g, 1e-5, n, g + 64, y, None) == 1        # h overlaps g
    yo = (C.c_void_p * 2)(A + 2 ** 24, g + 32)                             # y overlaps g
    assert f(2, W, rows, 64, x, g, 1e-5, n, h, yo, None) == 1
    assert f(2, W, rows, 60, x, g, 1e-5, n, None, y, None) == 1          # k % 8 != 0 needs h


def test_rms_norm_host_checks(L):
    f = L.bm_rms_norm_mul
    x, g, o, h = A, A + 2 ** 20, A + 2 ** 21, A + 2 ** 22
    assert f(x, g, 0, 64, 1e-5, o, h, None) == 0                          # no rows: nothing to do
    assert f(x, g, -1, 64, 1e-5, o, h, None) == 1
    assert f(x, g, 4, 0, 1e-5, o, h, None) == 1
    assert f(x, None, 4, 64, 1e-5, o, h, None) == 1
    assert f(x, g, 4, 64, 1e-5, None, None, None) == 1                    # no output
    assert f(x + 2, g, 4, 64, 1e-5, o, h, None) == 2
    assert f(x, g, 4, 64, 1e-5, o, h + 1, None) == 2
    assert f(x, g, 4, 64, 1e-5, x + 4, h, None) == 1                      # out overlaps x, not in place
    assert f(x, g, 4, 64, 1e-5, o, x + 256, None) == 1                    # h overlaps x
    assert f(x, g, 4, 64, 1e-5, g, None, None) == 1                       # out overlaps g


def test_matmul_multi_host_checks(L):
    f = L.bm_f16_matmul_multi
    W = (C.c_void_p * 2)(A, A + 2 ** 20)
    Y = (C.c_void_p * 2)(A + 2 ** 24, A + 2 ** 25)
    rows = (C.c_int64 * 2)(16, 16)
    X = A + 2 ** 26
    assert f(0, W, rows, 64, X, 8, Y, None) == 1
    assert f(5, W, rows, 64, X, 8, Y, None) == 1
    assert f(2, None, rows, 64, X, 8, Y, None) == 1
    assert f(2, W, rows, 0, X, 8, Y, None) == 1
    assert f(2, W, rows, 64, X + 2, 8, Y, None) == 2                    # X misaligned
    Yo = (C.c_void_p * 2)(A + 2 ** 24, A + 2 ** 24 + 64)                  # the outputs overlap
    assert f(2, W, rows, 64, X, 8, Yo, None) == 1
    assert f(2, W, rows, 64, X, 0, Y, None) == 0                        # no columns: nothing to do


def test_mad_and_scale_host_checks(L):
    f = "bm_f16_mad"
    assert st(L, f, A, A + 4096, 0.5, -1, None) == 1        # n < 0
    assert st(L, f, A, A + 4096, 0.5, 0, None) == 0         # nothing to do
    assert st(L, f, None, A + 4096, 0.5, 8, None) == 1
    assert st(L, f, A, None, 0.5, 8, None) == 1
    assert st(L, f, A + 1, A + 4096, 0.5, 8, None) == 2     # odd address
    assert st(L, f, A, A + 4097, 0.5, 8, None) == 2
    assert st(L, f, A, A + 8, 0.5, 8, None) == 1            # v overlaps acc without being it
    g = "bm_f16_scale"
    assert st(L, g, A, 2.0, -1, None) == 1
    assert st(L, g, A, 2.0, 0, None) == 0
    assert st(L, g, None, 2.0, 8, None) == 1
    assert st(L, g, A + 3, 2.0, 8, None) == 2


def test_tc_plan_host_checks(L):
    info = (C.c_int64 * 6)()
    assert st(L, "bm_tc_plan", 4096, 4096, 512, 0, None) == 1      # null info
    assert st(L, "bm_tc_plan", 13, 4096, 512, 0, info) == 1         # rows % 4 != 0: not a tensor-core product
    assert st(L, "bm_tc_plan", 4096, 33, 512, 0, info) == 1         # k % 8 != 0
    assert st(L, "bm_tc_plan", 4096, 4096, 1, 0, info) == 1         # one column
    assert st(L, "bm_tc_plan", 4096, 65544, 512, 0, info) == 1      # k > BM_MAX_K
    assert b"tensor-core" in L.bm_last_error()



def test_step_create_host_checks(L):
    import f16_weight_gemv_gb300 as bm
    calls = (bm.MatvecCall * 2)()
    out = C.c_void_p()
    assert st(L, "bm_step_create", calls, 1, None) == 1          # null step
    assert st(L, "bm_step_create", calls, 0, C.byref(out)) == 1  # no calls
    c = calls[0]
    c.nmat, c.k, c.x = 1, 4096, A + 2 ** 26
    c.W[0], c.rows[0], c.y[0] = A, 64, A + 2 ** 27
    c.nmat = 5
    assert st(L, "bm_step_create", calls, 1, C.byref(out)) == 1  # nmat outside 1..4
    c.nmat, c.k = 1, 4097
    assert st(L, "bm_step_create", calls, 1, C.byref(out)) == 1  # k % 8 != 0
    c.k, c.x = 4096, A + 2 ** 26 + 4
    assert st(L, "bm_step_create", calls, 1, C.byref(out)) == 2  # x not 16-byte aligned
    c.x, c.y[0] = A + 2 ** 26, A + 64                             # output inside W
    assert st(L, "bm_step_create", calls, 1, C.byref(out)) == 1
    c.y[0] = A + 2 ** 27
    d = calls[1]
    d.nmat, d.k, d.x = 1, 4096, A + 2 ** 26
    d.W[0], d.rows[0], d.y[0] = A + 2 ** 28, 64, A + 2 ** 28 + 128  # call 1 writes into its own weights
    assert st(L, "bm_step_create", calls, 2, C.byref(out)) == 1
    d.y[0] = A + 128                                               # call 1 writes into call 0's weights
    assert st(L, "bm_step_create", calls, 2, C.byref(out)) == 1
    assert b"weights" in L.bm_last_error()
    assert out.value is None
    assert st(L, "bm_step_run", None, None) == 1
    assert st(L, "bm_step_destroy", None) == 0
