"""The entry points inside a CUDA graph: every call enqueues only kernels on
the caller's stream (no allocation, no synchronisation), so a training step
(lmhead_ce_fwd_bwd + bpb_reduce) and an evaluation step (masked
lmhead_ce_fwd + bpb_reduce) can be captured once and replayed.  Replays must
give bit-identical results to the same calls made eagerly."""
import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_util import dev_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lm():
    import lm_head_softcapped_lmhead_b300 as lm
    lm.lib()
    return lm


def capture(step):
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            step()
    torch.cuda.current_stream().wait_stream(side)
    return graph


def test_training_step_graph_replay_matches_eager(lm):
    N, V, d = 1000, 3000, 512
    inp = si.make_inputs(2, N=N, V=V, d=d)
    dd = dev_inputs(inp)
    ws = lm.workspace(N, V, d)
    nll, lse = torch.empty(N, device="cuda"), torch.empty(N, device="cuda")
    dh = torch.empty_like(dd["h"])
    dW = torch.zeros(V, d, device="cuda")
    acc = lm.bpb_acc()

    def step():
        lm.lmhead_ce_fwd_bwd(dd["h"], dd["W"], dd["tgt"], 30.0, 1.0 / N, nll, lse, dh=dh, dW=dW,
                             accumulate_dW=True, ws=ws)
        lm.bpb_reduce(nll, dd["nbytes"], acc, ws=ws)

    # Eager: two steps (dW and the bpb sums accumulate).  The first call also
    # does the library's one-time device set-up, outside any capture.
    step()
    step()
    assert lm.lmce_status(ws) == lm.LMCE_OK
    ref = [t.clone() for t in (nll, lse, dh, dW, acc)]

    # Captured once, replayed twice from the same starting state.
    graph = capture(step)
    nll.fill_(float("nan"))
    dh.fill_(float("nan"))
    dW.zero_()
    acc.zero_()
    graph.replay()
    graph.replay()
    torch.cuda.synchronize()
    assert lm.lmce_status(ws) == lm.LMCE_OK
    for got, want in zip((nll, lse, dh, dW, acc), ref):
        assert torch.equal(got, want)


def test_masked_eval_step_graph_replay_matches_eager(lm):
    N, V, d = 2 * si.WINDOW + 77, 2048, 512
    inp = si.make_inputs(4, N=N, V=V, d=d)
    dd = dev_inputs(inp)
    ws = lm.workspace(N, V, d, lm.LMCE_WS_MASKED)
    nll, lse = torch.empty(N, device="cuda"), torch.empty(N, device="cuda")
    acc = lm.bpb_acc()

    def step():
        lm.lmhead_ce_fwd(dd["h"], dd["W"], dd["tgt"], 30.0, nll, lse, row_mask=dd["mask"], ws=ws)
        lm.bpb_reduce(nll, dd["nbytes"], acc, row_mask=dd["mask"], ws=ws)

    step()
    assert lm.lmce_status(ws) == lm.LMCE_OK
    ref = [t.clone() for t in (nll, lse, acc)]
    graph = capture(step)
    nll.fill_(float("nan"))
    acc.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert lm.lmce_status(ws) == lm.LMCE_OK
    for got, want in zip((nll, lse, acc), ref):
        assert torch.equal(got, want)
    assert int(np.count_nonzero(inp["mask"])) == lm.read_bpb_acc(acc)[2]
