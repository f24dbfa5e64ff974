"""Failure detection on the GPU without a fault: every in-kernel wait of the
library is bounded, and an expired wait raises LMCE_ETIMEOUT in the status
word and returns.  lmce_wait_selftest runs that bounded wait on an mbarrier
that never receives its arrival (a flag that nothing sets) with a short
limit: the status must read LMCE_ETIMEOUT, the context must stay usable, and
with the arrival given the same wait completes with LMCE_OK."""
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


def test_expired_wait_reports_timeout_and_context_survives(lm):
    inp = si.make_inputs(2, N=500, V=800, d=256)
    d_inp = dev_inputs(inp)
    ws = lm.workspace(500, 800, 256)
    before = torch.empty(500, device="cuda")
    lm.lmhead_ce_fwd(d_inp["h"], d_inp["W"], d_inp["tgt"], 30.0, before, None, ws=ws)
    assert lm.lmce_status(ws) == lm.LMCE_OK
    lm.lmce_wait_selftest(200000, arrive=False, ws=ws)      # ~0.1 ms of SM clock, nothing arrives
    assert lm.lmce_status(ws) == lm.LMCE_ETIMEOUT
    assert lm.lmce_status(ws) == lm.LMCE_OK                # lmce_status cleared it
    lm.lmce_wait_selftest(200000, arrive=True, ws=ws)
    assert lm.lmce_status(ws) == lm.LMCE_OK
    after = torch.empty(500, device="cuda")
    lm.lmhead_ce_fwd(d_inp["h"], d_inp["W"], d_inp["tgt"], 30.0, after, None, ws=ws)
    assert lm.lmce_status(ws) == lm.LMCE_OK
    assert torch.equal(before, after)
