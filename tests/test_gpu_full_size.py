"""Full-size parity: the workloads at their full sizes, in the launch
configuration bench.py times, against oracle values stored in
tests/golden/full_size.json (written by tests/golden/make_golden.py --full,
which calls only the oracle).

* forward + backward batch (N = 16384) and training micro-batch (N = 65536),
  V = 8192, softcap 30, mean loss: the whole batch's bpb through bpb_reduce
  within 1e-5 relative (and its integer sums exactly), and dW on 8 vocabulary
  rows (the four most frequent Zipf targets, two mid-frequency and two rare
  ids) within 1e-2 relative Frobenius error, row by row;
* the int4 head (N = 65536): bpb through lmhead_ce_fwd_bwd_int4 + bpb_reduce;
* the sliding-window evaluation stream: 8 calls of 32 windows each, bpb
  accumulated across the calls in fp64 on the device; each call's sum of nll
  within 1e-5 relative, the stream's bpb within 1e-5, and a second run of the
  whole stream gives the same bits."""
import json
import os

import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_util import BPB_RTOL, GRAD_RTOL, dev_inputs, rel_fro

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "full_size.json")


@pytest.fixture(scope="module")
def lm():
    import lm_head_softcapped_lmhead_b300 as lm
    lm.lib()
    return lm


@pytest.fixture(scope="module")
def golden():
    with open(GOLDEN) as f:
        return json.load(f)


def check_sums(lm, acc, e):
    sn, sb, n = lm.read_bpb_acc(acc)
    assert (sb, n) == (e["sum_bytes"], e["n_scored"])
    assert abs(sn - e["sum_nll"]) <= BPB_RTOL * abs(e["sum_nll"])
    bpb = lm.lmce_bpb(acc)
    assert abs(bpb - e["bpb"]) <= BPB_RTOL * e["bpb"]


@pytest.mark.parametrize("cfg", [2, 3])
def test_train_batch_bpb_and_dW_rows(lm, golden, cfg):
    """The training step as bench.py runs it: lmhead_ce_fwd_bwd with dh (the
    one-pass forward + dh), bpb_reduce, then lmhead_ce_bwd with dW (given the
    forward's nll)."""
    e = golden[f"cfg{cfg}"]
    inp = si.make_inputs(cfg)
    assert (inp["N"], inp["seed"]) == (e["N"], e["seed"])
    d_inp = dev_inputs(inp)
    N, V, d = inp["N"], inp["V"], inp["d"]
    w = e["grad_scale"]
    ws = lm.workspace(N, V, d)
    nll = torch.empty(N, device="cuda")
    lse = torch.empty(N, device="cuda")
    dh = torch.empty_like(d_inp["h"])
    dW = torch.zeros((V, d), device="cuda")
    acc = lm.bpb_acc()
    lm.lmhead_ce_fwd_bwd(d_inp["h"], d_inp["W"], d_inp["tgt"], e["softcap"], w, nll, lse, dh=dh, ws=ws)
    lm.bpb_reduce(nll, d_inp["nbytes"], acc, ws=ws)
    lm.lmhead_ce_bwd(d_inp["h"], d_inp["W"], d_inp["tgt"], e["softcap"], lse, w, dW=dW, accumulate_dW=True, ws=ws,
                     nll=nll)
    assert lm.lmce_status(ws) == lm.LMCE_OK
    check_sums(lm, acc, e)
    got = dW[torch.tensor(e["vrows"], device="cuda")].double().cpu().numpy()
    ref = np.array(e["dW_rows"])
    for r, v in enumerate(e["vrows"]):
        assert rel_fro(got[r], ref[r]) <= GRAD_RTOL, (v, rel_fro(got[r], ref[r]))
    assert rel_fro(got, ref) <= GRAD_RTOL


def test_int4_batch_bpb(lm, golden):
    e = golden["cfg5"]
    inp = si.make_inputs(5)
    assert (inp["N"], inp["seed"]) == (e["N"], e["seed"])
    d_inp = dev_inputs(inp)
    N, V, d = inp["N"], inp["V"], inp["d"]
    ws = lm.workspace(N, V, d, lm.LMCE_WS_INT4)
    nll = torch.empty(N, device="cuda")
    lse = torch.empty(N, device="cuda")
    dh = torch.empty_like(d_inp["h"])
    acc = lm.bpb_acc()
    lm.lmhead_ce_fwd_bwd_int4(d_inp["h"], d_inp["Wq"], d_inp["scales"], si.INT4_GROUP, e["softcap"], d_inp["tgt"],
                              1.0 / N, nll, lse, dh, ws=ws)
    lm.bpb_reduce(nll, d_inp["nbytes"], acc, ws=ws)
    assert lm.lmce_status(ws) == lm.LMCE_OK
    check_sums(lm, acc, e)


def run_stream(lm, chunks):
    """Every chunk through lmhead_ce_fwd (row mask) + bpb_reduce into one
    stream accumulator; also each call's own sums."""
    stream_acc = lm.bpb_acc()
    per_call = []
    ws = None
    for inp in chunks:
        d_inp = dev_inputs(inp)
        N, V, d = inp["N"], inp["V"], inp["d"]
        if ws is None:
            ws = lm.workspace(N, V, d, lm.LMCE_WS_MASKED)
        nll = torch.empty(N, device="cuda")
        lm.lmhead_ce_fwd(d_inp["h"], d_inp["W"], d_inp["tgt"], si.SOFTCAP, nll, None, row_mask=d_inp["mask"], ws=ws)
        call_acc = lm.bpb_acc()
        lm.bpb_reduce(nll, d_inp["nbytes"], call_acc, row_mask=d_inp["mask"], ws=ws)
        lm.bpb_reduce(nll, d_inp["nbytes"], stream_acc, row_mask=d_inp["mask"], ws=ws)
        assert lm.lmce_status(ws) == lm.LMCE_OK
        per_call.append(lm.read_bpb_acc(call_acc))
    return stream_acc, per_call


def test_eval_stream_multi_call(lm, golden):
    st = golden["cfg4_stream"]
    chunks = [si.make_stream_chunk(c["k"]) for c in st["chunks"]]
    assert len(chunks) >= 4
    acc1, per_call = run_stream(lm, chunks)
    for c, (sn, sb, n) in zip(st["chunks"], per_call):
        assert (sb, n) == (c["sum_bytes"], c["n_scored"])
        assert abs(sn - c["sum_nll"]) <= BPB_RTOL * abs(c["sum_nll"])
    bpb = lm.lmce_bpb(acc1)
    assert abs(bpb - st["bpb"]) <= BPB_RTOL * st["bpb"]
    acc2, _ = run_stream(lm, chunks)
    assert torch.equal(acc1.view(torch.int64), acc2.view(torch.int64))
