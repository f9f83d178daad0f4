"""The binding's prepare(): calls recorded once (arguments checked and marshalled,
nothing launched) and replayed give the same bits as the same calls made through the
wrappers, follow in-place changes of their inputs, and keep the tensors they point
into alive; captured as one CUDA graph (Prepared.graph) they give the same bits again."""
import gc

import numpy as np
import pytest

import oracle
import synth
from conftest import bits32, to_dev

pytestmark = pytest.mark.gpu


def test_prepared_step_matches_eager_and_follows_inputs(bm):
    import torch
    k, rows = 576, (576, 192, 192)
    Ws = [to_dev(synth.normal_f16(0, "prep.w%d" % i, 0.02, (r, k))) for i, r in enumerate(rows)]
    E = to_dev(synth.normal_f16(0, "prep.e", 0.02, (4096, k)))
    x = to_dev(synth.normal_f32(0, "prep.x", 1.0, k))
    X = to_dev(synth.normal_f32(0, "prep.X", 1.0, (8, k)))
    s = torch.cuda.Stream()
    out = {}

    def step():
        out["y"] = bm.bm_f16_matvec_act(Ws, x, stream=s)
        out["h"] = bm.bm_to_f16(X, stream=s)
        out["Y"] = bm.bm_f16_matmul(Ws[0], out["h"], stream=s)
        out["L"] = bm.bm_f16_logits(E, out["h"], stream=s)

    pc = bm.prepare(step)
    assert len(pc) == 4
    torch.cuda.synchronize()
    for t in (*out["y"], out["Y"], out["L"]):
        t.fill_(float("nan"))  # nothing was launched while recording; replay fills them
    pc()
    torch.cuda.synchronize()
    got = [bits32(t).copy() for t in (*out["y"], out["Y"], out["L"])]
    with torch.cuda.stream(s):
        ys = bm.bm_f16_matvec_act(Ws, x, stream=s)
        h = bm.bm_to_f16(X, stream=s)
        Y = bm.bm_f16_matmul(Ws[0], h, stream=s)
        L = bm.bm_f16_logits(E, h, stream=s)
    torch.cuda.synchronize()
    for a, b in zip(got, [bits32(t) for t in (*ys, Y, L)]):
        assert np.array_equal(a, b)
    xh = oracle.to_f16(x.cpu().numpy())
    for W, y in zip(Ws, out["y"]):
        assert np.array_equal(bits32(y), bits32(oracle.matvec(W.cpu().numpy().view(np.uint16), xh)))
    x.mul_(2.0)  # in place: a replay reads the new values
    pc()
    torch.cuda.synchronize()
    xh2 = oracle.to_f16(x.cpu().numpy())
    assert np.array_equal(bits32(out["y"][0]), bits32(oracle.matvec(Ws[0].cpu().numpy().view(np.uint16), xh2)))
    assert bm.bm_device_status() == 0


def test_prepared_call_keeps_its_tensors(bm):
    """Outputs allocated inside the recorded thunk stay allocated for as long as the
    Prepared object lives, even with no other reference to them."""
    import torch
    k = 1024
    W = to_dev(synth.normal_f16(0, "prep.keep", 0.02, (512, k)))
    x = to_dev(oracle.to_f16(synth.normal_f32(0, "prep.keep.x", 1.0, k)))
    pc = bm.prepare(lambda: bm.bm_f16_matvec(W, x))
    gc.collect()
    junk = [torch.full((512,), 7.0, device="cuda") for _ in range(64)]  # would reuse freed blocks
    pc()
    torch.cuda.synchronize()
    y = pc._tensors[-1]
    assert np.array_equal(bits32(y), bits32(oracle.matvec(W.cpu().numpy().view(np.uint16), x.cpu().numpy().view(np.uint16))))
    del junk


def test_prepared_graph_matches_replay(bm):
    """The recorded calls captured as one graph: the same bits as the plain replay, on
    every replay, and in-place input changes are followed (the graph keeps the pointers)."""
    import torch
    k, rows = 576, (576, 192, 192)
    Ws = [to_dev(synth.normal_f16(0, "prepg.w%d" % i, 0.02, (r, k))) for i, r in enumerate(rows)]
    Wg = to_dev(synth.normal_f16(0, "prepg.g", 0.02, (1536, k)))
    x = to_dev(synth.normal_f32(0, "prepg.x", 1.0, k))
    X = to_dev(synth.normal_f32(0, "prepg.X", 1.0, (64, k)))
    s = torch.cuda.Stream()
    out = {}

    def step():
        out["y"] = bm.bm_f16_matvec_act(Ws, x, stream=s)
        out["h"] = bm.bm_to_f16(X, stream=s)
        out["Y"] = bm.bm_f16_matmul(Wg, out["h"], stream=s)  # tensor cores, may split k

    old = bm.bm_set_pdl(True)
    try:
        pc = bm.prepare(step)
        pc_graph = pc.graph(s)
        assert len(pc_graph) == 3
        with torch.cuda.stream(s):
            pc()
        torch.cuda.synchronize()
        want = [bits32(t).copy() for t in (*out["y"], out["Y"])]
        for _ in range(3):
            for t in (*out["y"], out["Y"]):
                t.fill_(float("nan"))
            torch.cuda.synchronize()
            with torch.cuda.stream(s):
                pc_graph()
            torch.cuda.synchronize()
            for a, t in zip(want, (*out["y"], out["Y"])):
                assert np.array_equal(a, bits32(t))
        x.mul_(-0.5)
        torch.cuda.synchronize()
        with torch.cuda.stream(s):
            pc_graph()
        torch.cuda.synchronize()
        xh = oracle.to_f16(x.cpu().numpy())
        assert np.array_equal(bits32(out["y"][1]), bits32(oracle.matvec(Ws[1].cpu().numpy().view(np.uint16), xh)))
    finally:
        bm.bm_set_pdl(old)
    assert bm.bm_device_status() == 0
