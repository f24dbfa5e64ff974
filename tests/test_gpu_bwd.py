"""Backward parity: dh and dW from the CUDA backward (through the C ABI)
against the fp64 oracle's analytic gradients on the same bf16 inputs."""
import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_util import GRAD_RTOL, dev_inputs, rel_fro, bf16_to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lm():
    import lm_head_softcapped_lmhead_b300 as lm
    lm.lib()
    return lm


def run_fwd_bwd(lm, d_inp, c, grad_scale, mask=None, want_dh=True, want_dW=True, dW_init=None, pass_nll=False):
    N, d = d_inp["h"].shape
    V = d_inp["W"].shape[0]
    ws = lm.workspace(N, V, d, lm.LMCE_WS_MASKED if mask is not None else 0)
    nll = torch.zeros(N, device="cuda")
    lse = torch.zeros(N, device="cuda")
    lm.lmhead_ce_fwd(d_inp["h"], d_inp["W"], d_inp["tgt"], c, nll, lse, row_mask=mask, ws=ws)
    dh = torch.full_like(d_inp["h"], float("nan")) if want_dh else None
    dW = None
    if want_dW:
        dW = torch.full((V, d), float("nan"), device="cuda") if dW_init is None else dW_init.clone()
    lm.lmhead_ce_bwd(d_inp["h"], d_inp["W"], d_inp["tgt"], c, lse, grad_scale, dh=dh, dW=dW,
                     accumulate_dW=dW_init is not None, row_mask=mask, ws=ws, nll=nll if pass_nll else None)
    assert lm.lmce_status(ws) == lm.LMCE_OK
    return nll, lse, dh, dW


@pytest.mark.parametrize("cfg,N,V,d,w_scale,c", [
    (2, 300, 700, 256, 1.0, 30.0),     # ragged
    (2, 512, 1024, 512, 1.0, 30.0),    # d = 512
    (2, 257, 1000, 512, 50.0, 30.0),   # W x 50: cap active
    (2, 200, 300, 64, 20.0, 2.0),      # c = 2, d = 64 (one K chunk)
    (2, 150, 260, 192, 1.0, 30.0),     # odd number of 64-chunks
    (1, 4096, 1024, 512, 1.0, 30.0),   # config 1 shape
])
def test_bwd_matches_oracle(lm, oracle_mod, cfg, N, V, d, w_scale, c):
    inp = si.make_inputs(cfg, N=N, V=V, d=d, w_scale=w_scale)
    w = 1.0 / N
    _, _, dh, dW = run_fwd_bwd(lm, dev_inputs(inp), c, w)
    _, ref_lse = oracle_mod.fwd(inp["h"], inp["W"], inp["tgt"], c)
    ref_dh, ref_dW = oracle_mod.bwd(inp["h"], inp["W"], inp["tgt"], c, ref_lse, w)
    assert rel_fro(bf16_to_f64(dh), ref_dh) <= GRAD_RTOL
    assert rel_fro(dW.cpu().numpy(), ref_dW) <= GRAD_RTOL


def test_bwd_accumulate_and_mask(lm, oracle_mod):
    N, V, d = 400, 600, 128
    inp = si.make_inputs(2, N=N, V=V, d=d, w_scale=10.0)
    mask = (np.arange(N) % 5 != 2).astype(np.uint8)
    M = int(mask.sum())
    d_inp = dev_inputs(inp)
    init = torch.randn(V, d, device="cuda") * 1e-3
    _, _, dh, dW = run_fwd_bwd(lm, d_inp, 30.0, 1.0 / M, mask=torch.from_numpy(mask).cuda(), dW_init=init)
    _, ref_lse = oracle_mod.fwd(inp["h"], inp["W"], inp["tgt"], 30.0, mask=mask)
    ref_dh, ref_dW = oracle_mod.bwd(inp["h"], inp["W"], inp["tgt"], 30.0, ref_lse, 1.0 / M, mask=mask)
    dh_np = bf16_to_f64(dh)
    assert np.all(dh_np[mask == 0] == 0)
    assert rel_fro(dh_np, ref_dh) <= GRAD_RTOL
    assert rel_fro(dW.cpu().numpy() - init.cpu().numpy(), ref_dW) <= GRAD_RTOL


def test_bwd_dh_only_and_dW_only(lm, oracle_mod):
    N, V, d = 260, 390, 256
    inp = si.make_inputs(2, N=N, V=V, d=d)
    d_inp = dev_inputs(inp)
    _, _, dh, _ = run_fwd_bwd(lm, d_inp, 30.0, 0.5, want_dW=False)
    _, _, _, dW = run_fwd_bwd(lm, d_inp, 30.0, 0.5, want_dh=False)
    _, ref_lse = oracle_mod.fwd(inp["h"], inp["W"], inp["tgt"], 30.0)
    ref_dh, ref_dW = oracle_mod.bwd(inp["h"], inp["W"], inp["tgt"], 30.0, ref_lse, 0.5)
    assert rel_fro(bf16_to_f64(dh), ref_dh) <= GRAD_RTOL
    assert rel_fro(dW.cpu().numpy(), ref_dW) <= GRAD_RTOL


def test_bwd_config2_full(lm, oracle_mod):
    """Config 2 at full size (N=16384, V=8192): dh on 24 sampled rows against
    the oracle, dW through <dh, h> = <dW, W> (holds at any size), and dW
    against the oracle on a 2048-row slice of the same inputs."""
    inp = si.make_inputs(2)
    N = inp["N"]
    d_inp = dev_inputs(inp)
    w = 1.0 / N
    _, lse, dh, dW = run_fwd_bwd(lm, d_inp, 30.0, w, pass_nll=True)
    rows = np.random.default_rng(1).choice(N, 24, replace=False)
    _, ref_lse = oracle_mod.fwd(inp["h"], inp["W"], inp["tgt"], 30.0, rows=rows)
    ref = oracle_mod.dh_rows(inp["h"], inp["W"], inp["tgt"], 30.0, rows, ref_lse, w)
    assert rel_fro(bf16_to_f64(dh)[rows], ref) <= GRAD_RTOL
    h64 = bf16_to_f64(d_inp["h"])
    W64 = bf16_to_f64(d_inp["W"])
    a = float((bf16_to_f64(dh) * h64).sum())
    b = float((dW.double().cpu().numpy() * W64).sum())
    assert abs(a - b) <= 2e-2 * max(abs(a), abs(b))


def test_bwd_deterministic(lm):
    inp = si.make_inputs(2, N=2048, V=2048, d=512)
    d_inp = dev_inputs(inp)
    r1 = run_fwd_bwd(lm, d_inp, 30.0, 1 / 2048)
    r2 = run_fwd_bwd(lm, d_inp, 30.0, 1 / 2048)
    assert torch.equal(r1[2], r2[2]) and torch.equal(r1[3], r2[3])


def test_bwd_confident_rows_with_nll(lm, oracle_mod):
    """Rows with p_t within about 1e-4 of 1: given the forward's nll, the
    target's p - 1 is expm1(-nll) and dh, dW stay within tolerance (from
    lse alone, s_t - lse cancels in fp32 there)."""
    from test_gpu_fwd_bwd import confident_inputs
    inp = confident_inputs()
    N = inp["N"]
    d_inp = dev_inputs(inp)
    for mask in (None, (np.arange(N) % 3 != 1).astype(np.uint8)):
        M = N if mask is None else int(mask.sum())
        mk = None if mask is None else torch.from_numpy(mask).cuda()
        _, _, dh, dW = run_fwd_bwd(lm, d_inp, 30.0, 1.0 / M, mask=mk, pass_nll=True)
        _, ref_lse = oracle_mod.fwd(inp["h"], inp["W"], inp["tgt"], 30.0, mask=mask)
        ref_dh, ref_dW = oracle_mod.bwd(inp["h"], inp["W"], inp["tgt"], 30.0, ref_lse, 1.0 / M, mask=mask)
        assert rel_fro(bf16_to_f64(dh), ref_dh) <= GRAD_RTOL
        assert rel_fro(dW.cpu().numpy(), ref_dW) <= GRAD_RTOL
