"""GPU parity of the output-rows rule on the last layer (page "docs/modules/forward.md",
"Why only the output rows leave the last layer"): only the rows the engine outputs
(inp_out_ids: none, the last, or all) go through the last feed-forward products and
the logits, and for F16 their count picks the path -- one column is vec_dot, two or
more (bm_takes_sgemm) tinyBLAS.  The library selects by shape; these tests gather the
output rows on the device, as a caller does, and check every path against the oracle
bit for bit (the tinyBLAS path on the bit-exact kernel, bm_set_exact_sgemm_cols(8))."""
import numpy as np
import pytest

import oracle
import synth
from conftest import bits32, to_dev

pytestmark = pytest.mark.gpu

HID, FFN, VOCAB, NROWS = 576, 1536, 49152, 7


@pytest.fixture(autouse=True)
def exact_up_to_eight(bm):
    old = bm.bm_set_exact_sgemm_cols(8)
    yield
    bm.bm_set_exact_sgemm_cols(old)


def last_layer(bm, X, out_ids, Wg, Wd, E, sample_rows):
    """The FFN's gate and down products and the logits over the gathered output rows."""
    import torch
    idx = torch.tensor(out_ids, dtype=torch.int64, device="cuda")
    Xo = to_dev(X).index_select(0, idx).contiguous()
    n = len(out_ids)
    G = torch.empty((n, FFN), dtype=torch.float32, device="cuda")
    bm.bm_f16_matmul(to_dev(Wg), Xo, Y=G)
    Hd = to_dev(oracle.to_f16(synth.normal_f32(0, "outids.act_ffn", 1.0, (NROWS, FFN)))).index_select(0, idx)
    D = torch.empty((n, HID), dtype=torch.float32, device="cuda")
    bm.bm_f16_matmul(to_dev(Wd), Hd.contiguous(), Y=D)
    L = torch.empty((n, VOCAB), dtype=torch.float32, device="cuda")
    bm.bm_f16_logits(to_dev(E), Xo, Y=L)
    return bits32(G), bits32(D), bits32(L)[:, sample_rows]


def test_last_row_alone_versus_all_rows(bm):
    Wg = synth.normal_f16(0, "outids.gate", 0.02, (FFN, HID))
    Wd = synth.normal_f16(0, "outids.down", 0.02, (HID, FFN))
    E = synth.normal_f16(0, "outids.embd", 0.02, (VOCAB, HID))
    X = oracle.to_f16(synth.normal_f32(0, "outids.x", 1.0, (NROWS, HID)))
    Hd = oracle.to_f16(synth.normal_f32(0, "outids.act_ffn", 1.0, (NROWS, FFN)))
    rng = np.random.default_rng(3)
    vs = np.unique(np.concatenate([[0, VOCAB - 1], rng.integers(0, VOCAB, 3000)]))

    # all rows output: seven columns, tinyBLAS (bm_takes_sgemm) on every product
    assert bm.bm_takes_sgemm(FFN, HID, NROWS) and bm.bm_takes_sgemm(VOCAB, HID, NROWS)
    g_all, d_all, l_all = last_layer(bm, X, list(range(NROWS)), Wg, Wd, E, vs)
    assert np.array_equal(g_all, bits32(oracle.matmul(Wg, X)))
    assert np.array_equal(d_all, bits32(oracle.matmul(Wd, Hd)))
    ref, _ = oracle.matmul_sample(E, X, np.tile(vs, NROWS), np.repeat(np.arange(NROWS), vs.size), with_absdot=False)
    assert np.array_equal(l_all.reshape(-1), bits32(ref))

    # the last row only: one column, vec_dot
    g_one, d_one, l_one = last_layer(bm, X, [NROWS - 1], Wg, Wd, E, vs)
    assert np.array_equal(g_one[0], bits32(oracle.matvec(Wg, X[-1])))
    assert np.array_equal(d_one[0], bits32(oracle.matvec(Wd, Hd[-1])))
    ref, _ = oracle.matmul_sample(E, X[-1:], vs, np.zeros(vs.size, np.int64), with_absdot=False)
    assert np.array_equal(l_one[0], bits32(ref))

    # the same row, two paths: the bits differ in part of the elements, as the page says
    for one, allr in ((g_one[0], g_all[-1]), (d_one[0], d_all[-1]), (l_one[0], l_all[-1])):
        differ = np.count_nonzero(one != allr)
        assert 0 < differ < one.size


def test_two_output_rows_take_tinyblas(bm):
    """Two output rows are already a tinyBLAS product (and the exact kernel's default)."""
    import torch
    Wg = synth.normal_f16(0, "outids.gate", 0.02, (FFN, HID))
    X = oracle.to_f16(synth.normal_f32(0, "outids.x", 1.0, (NROWS, HID)))
    sel = [2, NROWS - 1]
    Xo = to_dev(X).index_select(0, torch.tensor(sel, device="cuda")).contiguous()
    G = bm.bm_f16_matmul(to_dev(Wg), Xo)
    assert np.array_equal(bits32(G), bits32(oracle.matmul(Wg, X[sel])))


def test_no_output_rows_launch_nothing(bm):
    import torch
    Wg = to_dev(synth.normal_f16(0, "outids.gate", 0.02, (FFN, HID)))
    Y = torch.empty((0, FFN), dtype=torch.float32, device="cuda")
    bm.bm_f16_matmul(Wg, torch.empty((0, HID), dtype=torch.float16, device="cuda"), Y=Y)
    assert Y.numel() == 0 and bm.bm_device_status() == 0
