"""GPU parity of bm_f16_get_rows (the token-embedding lookup: f16 rows widened to
f32, exactly; page f16.md, "Technical usage", dequantize_row / widen) against the
oracle's widening, bit for bit, on both kernel paths (16-byte chunks when hidden % 8
== 0 and the output is 16-byte aligned; one element per thread otherwise)."""
import numpy as np
import pytest

import oracle
import synth
from conftest import bits32, to_dev

pytestmark = pytest.mark.gpu


def ids_dev(ids):
    import torch
    return torch.from_numpy(np.ascontiguousarray(ids, dtype=np.int32)).cuda()


@pytest.mark.parametrize("hidden", [8, 1])
def test_every_f16_pattern(bm, hidden):
    """All 65536 bit patterns as a table; non-NaN values widen exactly, NaN stays NaN."""
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    E = pats.reshape(-1, hidden)
    ids = np.arange(E.shape[0])
    out = bm.bm_f16_get_rows(to_dev(E), ids_dev(ids)).cpu().numpy().reshape(-1)
    ref = oracle.widen(pats)
    nan = ((pats & 0x7C00) == 0x7C00) & ((pats & 0x3FF) != 0)
    assert np.array_equal(out.view(np.uint32)[~nan], ref.view(np.uint32)[~nan])
    assert np.isnan(out[nan]).all()
    assert bm.bm_device_status() == 0


@pytest.mark.parametrize("vocab,hidden,n", [
    (49152, 576, 1), (49152, 576, 7), (151936, 1024, 512), (128256, 4096, 3), (1000, 577, 40), (50, 31, 5),
])
def test_embedding_shapes(bm, vocab, hidden, n):
    E = synth.normal_f16(0, "embd.%d" % vocab, 0.02, (vocab, hidden))
    rng = np.random.default_rng(vocab + n)
    ids = np.concatenate([[0, vocab - 1], rng.integers(0, vocab, max(0, n - 2))])[:n]
    out = bm.bm_f16_get_rows(to_dev(E), ids_dev(ids)).cpu().numpy()
    assert np.array_equal(bits32(out), bits32(oracle.widen(E[ids])))
    assert bm.bm_device_status() == 0


def test_unaligned_output_takes_the_scalar_path(bm):
    import torch
    vocab, hidden, n = 300, 64, 9
    E = synth.normal_f16(0, "embd.u", 0.02, (vocab, hidden))
    ids = np.arange(n) * 7
    buf = torch.full((n * hidden + 2,), float("nan"), dtype=torch.float32, device="cuda")
    bm.bm_f16_get_rows(to_dev(E), ids_dev(ids), out=buf[1:1 + n * hidden])
    b = buf.cpu().numpy()
    assert np.isnan(b[0]) and np.isnan(b[-1])
    assert np.array_equal(bits32(b[1:1 + n * hidden]), bits32(oracle.widen(E[ids])).ravel())


def test_ids_out_of_range_are_reported_and_skipped(bm):
    import torch
    vocab, hidden = 100, 64
    E = synth.normal_f16(0, "embd.bad", 0.02, (vocab, hidden))
    ids = np.array([3, -1, 99, 100, 0, 2 ** 31 - 1], dtype=np.int64)
    out = torch.full((ids.size, hidden), float("nan"), dtype=torch.float32, device="cuda")
    bm.bm_f16_get_rows(to_dev(E), ids_dev(ids), out=out)
    assert bm.bm_device_status() == 1          # BM_ERR_INVALID_ARG, read and cleared
    assert bm.bm_device_status() == 0
    o = out.cpu().numpy()
    good = (ids >= 0) & (ids < vocab)
    assert np.array_equal(bits32(o[good]), bits32(oracle.widen(E[ids[good]])))
    assert np.isnan(o[~good]).all()            # rows of bad ids untouched


def test_empty(bm):
    import torch
    E = synth.normal_f16(0, "embd.e", 0.02, (10, 16))
    out = bm.bm_f16_get_rows(to_dev(E), torch.empty(0, dtype=torch.int32, device="cuda"))
    assert out.numel() == 0


def test_k_cache_rows_are_vec_dot(bm):
    """vec_dot_u16 (a K cache row against an f16 query; page f16.md, Technical usage)
    gives vec_dot's bits: scores over a K cache of 4096 positions x head_dim 64 / 128
    are bm_f16_matvec with the cache as the matrix."""
    for pos, hd in [(4096, 64), (513, 128), (1, 64), (33, 128)]:
        K = synth.normal_f16(0, "kcache.%d.%d" % (pos, hd), 1.0, (pos, hd))
        q = oracle.to_f16(synth.normal_f32(0, "q.%d" % hd, 1.0, hd))
        y = bm.bm_f16_matvec(to_dev(K), to_dev(q))
        assert np.array_equal(bits32(y), bits32(oracle.matvec(K, q)))
