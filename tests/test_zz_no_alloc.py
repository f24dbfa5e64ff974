"""lmhead_ce_fwd_noalloc: the forward for callers that cannot give the library
device memory (a host process that owns all device memory through its own
pool, or a path that must not pay cudaMalloc's implicit synchronisation).
Its scratch is a static device array inside the library, so it takes no
workspace.  It runs the same kernels in the same launch shape as
lmhead_ce_fwd, so it must give the same bits; and its nll must match the
oracle on sampled rows.

Called through the C ABI with ctypes.  This file is collected last so that a
run stopping at the first failure has already run every other test; it also
passes on its own in a fresh process (the first call sets up the scratch)."""
import ctypes

import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_util import NLL_ATOL, dev_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lm():
    import lm_head_softcapped_lmhead_b300 as lm
    L = lm.lib()
    P, I64 = ctypes.c_void_p, ctypes.c_int64
    L.lmhead_ce_fwd_noalloc.argtypes = [P, I64, P, I64, I64, I64, P, ctypes.c_float, P, P, P]
    L.lmhead_ce_fwd_noalloc.restype = ctypes.c_int
    return lm


def noalloc_fwd(lm, d_inp, c, tgt=None):
    N, d = d_inp["h"].shape
    V = d_inp["W"].shape[0]
    tgt = d_inp["tgt"] if tgt is None else tgt
    nll = torch.full((N,), float("nan"), device="cuda")
    lse = torch.full((N,), float("nan"), device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rc = lm.lib().lmhead_ce_fwd_noalloc(ctypes.c_void_p(d_inp["h"].data_ptr()), d_inp["h"].stride(0),
                                        ctypes.c_void_p(d_inp["W"].data_ptr()), N, V, d,
                                        ctypes.c_void_p(tgt.data_ptr()), c,
                                        ctypes.c_void_p(nll.data_ptr()), ctypes.c_void_p(lse.data_ptr()), stream)
    assert rc == lm.LMCE_OK, lm.strerror(rc)
    return nll, lse


def workspace_fwd(lm, d_inp, c):
    N, d = d_inp["h"].shape
    V = d_inp["W"].shape[0]
    ws = lm.workspace(N, V, d)
    nll = torch.empty(N, device="cuda")
    lse = torch.empty(N, device="cuda")
    lm.lmhead_ce_fwd(d_inp["h"], d_inp["W"], d_inp["tgt"], c, nll, lse, ws=ws)
    assert lm.lmce_status(ws) == lm.LMCE_OK
    return nll, lse


def test_noalloc_matches_workspace_forward_two_calls(lm, oracle_mod):
    """Two calls in a row with different shapes share the static scratch; each
    gives bit for bit the nll and lse of lmhead_ce_fwd, and its nll matches
    the oracle on sampled rows within the nll tolerance."""
    cases = [si.make_inputs(3, N=5000, V=6000, d=512, w_scale=20.0),
             si.make_inputs(2, N=65536, V=8192, d=512)]
    for inp in cases:
        d_inp = dev_inputs(inp)
        a_nll, a_lse = noalloc_fwd(lm, d_inp, 30.0)
        torch.cuda.synchronize()
        b_nll, b_lse = workspace_fwd(lm, d_inp, 30.0)
        assert torch.all(torch.isfinite(a_nll))
        assert torch.equal(a_nll, b_nll) and torch.equal(a_lse, b_lse)
        rows = np.random.default_rng(inp["N"]).choice(inp["N"], 24, replace=False)
        ref_nll, _ = oracle_mod.fwd(inp["h"], inp["W"], inp["tgt"], 30.0, rows=rows)
        assert np.abs(a_nll.cpu().numpy()[rows] - ref_nll).max() <= NLL_ATOL


def test_noalloc_bad_target_row_is_nan(lm):
    """A target equal to V gives NaN in that row only; the other rows are
    those of a call with valid targets, and the next call (status word
    cleared at its start) is clean again."""
    inp = si.make_inputs(2, N=700, V=900, d=256)
    d_inp = dev_inputs(inp)
    good_nll, good_lse = noalloc_fwd(lm, d_inp, 30.0)
    bad = d_inp["tgt"].clone()
    bad[123] = 900
    nll, _ = noalloc_fwd(lm, d_inp, 30.0, tgt=bad)
    n = nll.cpu().numpy()
    assert np.isnan(n[123]) and np.isfinite(np.delete(n, 123)).all()
    assert np.array_equal(np.delete(n, 123), np.delete(good_nll.cpu().numpy(), 123))
    again, _ = noalloc_fwd(lm, d_inp, 30.0)
    assert torch.equal(again, good_nll)


def test_noalloc_rejects_sizes_beyond_its_scratch(lm):
    inp = si.make_inputs(2, N=64, V=64, d=64)
    d_inp = dev_inputs(inp)
    L = lm.lib()
    P = ctypes.c_void_p
    for N, V in ((65537, 64), (64, 8193)):
        rc = L.lmhead_ce_fwd_noalloc(P(d_inp["h"].data_ptr()), 64, P(d_inp["W"].data_ptr()), N, V, 64,
                                     P(d_inp["tgt"].data_ptr()), 30.0, P(d_inp["h"].data_ptr()), None, None)
        assert rc == lm.LMCE_EINVAL
    # only the fixed-shift form fits its scratch: no cap and caps above lmce_softcap_max(V) are refused
    for c in (0.0, 90.0):
        rc = L.lmhead_ce_fwd_noalloc(P(d_inp["h"].data_ptr()), 64, P(d_inp["W"].data_ptr()), 64, 64, 64,
                                     P(d_inp["tgt"].data_ptr()), c, P(d_inp["h"].data_ptr()), None, None)
        assert rc == lm.LMCE_ENOTSUP
