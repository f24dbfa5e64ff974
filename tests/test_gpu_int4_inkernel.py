"""The int4 head dequantised inside the forward kernel
(lmhead_ce_fwd_int4_inkernel): converter warps turn the packed nibbles of
each ring stage into bf16 tiles bit-exactly, so nll and lse must be bit for
bit those of lmhead_ce_fwd_int4 (dequantise once, then the bf16 forward),
and match the oracle on the oracle's dequantised head.  Ragged shapes, an odd
number of 64-column chunks, a vocabulary below one tile, other group sizes,
a row mask, softcap 0 (the running-maximum form), W x 20, and the full size."""
import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_util import NLL_ATOL, dev_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lm():
    import lm_head_softcapped_lmhead_b300 as lm
    lm.lib()
    return lm


def both(lm, d_inp, Wq, sc, group, c, mask=None):
    N, d = d_inp["h"].shape
    V = Wq.shape[0]
    flags = lm.LMCE_WS_MASKED if mask is not None else 0
    ws_a = lm.workspace(N, V, d, flags | lm.LMCE_WS_INT4)
    ws_b = lm.workspace(N, V, d, flags)
    out = []
    for fn, ws in ((lm.lmhead_ce_fwd_int4, ws_a), (lm.lmhead_ce_fwd_int4_inkernel, ws_b)):
        nll = torch.full((N,), float("nan"), device="cuda")
        lse = torch.full((N,), float("nan"), device="cuda")
        fn(d_inp["h"], Wq, sc, group, c, d_inp["tgt"], nll, lse, row_mask=mask, ws=ws)
        assert lm.lmce_status(ws) == lm.LMCE_OK
        out.append((nll, lse))
    return out


@pytest.mark.parametrize("N,V,d,group,w_scale,c,masked", [
    (300, 700, 256, 64, 1.0, 30.0, False),
    (257, 1000, 512, 64, 20.0, 30.0, False),   # W x 20: exact-tanh chunks
    (200, 900, 192, 64, 1.0, 30.0, False),     # three 64-column chunks: a half-used last stage
    (130, 100, 128, 32, 1.0, 30.0, False),     # V below one tile, group 32
    (400, 600, 512, 128, 5.0, 30.0, True),     # group 128, row mask
    (300, 700, 256, 64, 60.0, 0.0, False),     # no cap: the running-maximum form
])
def test_inkernel_int4_bit_identical_and_oracle(lm, oracle_mod, N, V, d, group, w_scale, c, masked):
    inp = si.make_inputs(2, N=N, V=V, d=d, w_scale=w_scale)
    Wq, sc = si.quantize_int4_rtn(inp["W"], group)
    d_inp = dev_inputs(inp)
    mask = (np.arange(N) % 3 != 1).astype(np.uint8) if masked else None
    tm = None if mask is None else torch.from_numpy(mask).cuda()
    (na, la), (nb, lb) = both(lm, d_inp, torch.from_numpy(Wq).cuda(), torch.from_numpy(sc.view(np.int16)).cuda(),
                              group, c, tm)
    assert torch.equal(na, nb) and torch.equal(la, lb)
    Wdq = oracle_mod.dequant_int4(Wq, sc, d, group)
    ref, _ = oracle_mod.fwd(inp["h"], Wdq, inp["tgt"], c, mask=mask)
    assert np.abs(nb.cpu().numpy() - ref).max() <= NLL_ATOL


def test_inkernel_int4_full_size(lm, oracle_mod):
    """The quantised-head workload at full size (N = 65536, V = 8192, d = 512):
    bit for bit the dequantise-once forward, and the oracle on 32 sampled rows."""
    inp = si.make_inputs(5)
    d_inp = dev_inputs(inp)
    (na, la), (nb, lb) = both(lm, d_inp, d_inp["Wq"], d_inp["scales"], si.INT4_GROUP, 30.0)
    assert torch.equal(na, nb) and torch.equal(la, lb)
    rows = np.random.default_rng(5).choice(inp["N"], 32, replace=False)
    Wdq = oracle_mod.dequant_int4(inp["Wq"], inp["scales"], inp["d"], si.INT4_GROUP)
    ref, _ = oracle_mod.fwd(inp["h"], Wdq, inp["tgt"], 30.0, rows=rows)
    assert np.abs(nb.cpu().numpy()[rows] - ref).max() <= NLL_ATOL
