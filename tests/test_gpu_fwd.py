"""Forward parity: the CUDA forward (through the C ABI) against the fp64
oracle on the same bf16 inputs, element by element."""
import math

import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_util import NLL_ATOL, BPB_RTOL, dev_inputs, bf16_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lm():
    import lm_head_softcapped_lmhead_b300 as lm
    lm.lib()
    return lm


def run_fwd(lm, d_inp, softcap, mask=None, want_lse=True):
    N, d = d_inp["h"].shape
    V = d_inp["W"].shape[0]
    ws = lm.workspace(N, V, d, lm.LMCE_WS_MASKED if mask is not None else 0)
    nll = torch.full((N,), float("nan"), device="cuda")
    lse = torch.full((N,), float("nan"), device="cuda") if want_lse else None
    lm.lmhead_ce_fwd(d_inp["h"], d_inp["W"], d_inp["tgt"], softcap, nll, lse, row_mask=mask, ws=ws)
    assert lm.lmce_status(ws) == lm.LMCE_OK
    return nll.cpu().numpy(), (lse.cpu().numpy() if want_lse else None), ws


@pytest.mark.parametrize("cfg,N,V,d,w_scale,c", [
    (1, 4096, 1024, 512, 1.0, 30.0),     # config 1 at full size
    (1, 300, 1000, 512, 1.0, 30.0),      # ragged rows and vocab
    (2, 517, 777, 128, 1.0, 30.0),       # ragged, d = 128
    (2, 256, 8192, 512, 1.0, 30.0),      # V = 8192, several tiles
    (2, 384, 1100, 64, 1.0, 30.0),       # d = 64
    (2, 200, 640, 192, 1.0, 30.0),       # odd number of 64-chunks
    (2, 300, 1024, 512, 100.0, 30.0),    # W x 100: cap saturates
    (2, 257, 513, 256, 20.0, 1.0),       # c = 1: mostly the exact-tanh path
    (2, 129, 300, 128, 30.0, 50.0),      # c = 50
    (2, 300, 1024, 512, 100.0, 70.0),    # W x 100 at c = 70: S_other / e^{s_t} up to 5e58, past fp32
])
def test_fwd_matches_oracle(lm, oracle_mod, cfg, N, V, d, w_scale, c):
    inp = si.make_inputs(cfg, N=N, V=V, d=d, w_scale=w_scale)
    nll, lse, _ = run_fwd(lm, dev_inputs(inp), c)
    ref_nll, ref_lse = oracle_mod.fwd(inp["h"], inp["W"], inp["tgt"], c)
    assert np.all(np.isfinite(nll))
    assert np.abs(nll - ref_nll).max() <= NLL_ATOL
    assert np.abs(lse - ref_lse).max() <= NLL_ATOL
    b_ref, *_ = oracle_mod.bpb(ref_nll, inp["nbytes"])
    b_gpu, *_ = oracle_mod.bpb(nll.astype(np.float64), inp["nbytes"])
    assert abs(b_gpu - b_ref) <= BPB_RTOL * b_ref


def test_fwd_zero_hidden_is_ln_V(lm):
    """Closed form on the device: h = 0 gives nll = ln V for every row."""
    N, V, d = 333, 1500, 256
    inp = si.make_inputs(2, N=N, V=V, d=d)
    d_inp = dev_inputs(inp)
    d_inp["h"] = torch.zeros_like(d_inp["h"])
    nll, lse, _ = run_fwd(lm, d_inp, 30.0)
    assert np.abs(nll - math.log(V)).max() < 2e-5


def test_fwd_strided_h(lm, oracle_mod):
    """h with a row stride larger than d (a view into a wider buffer)."""
    N, V, d = 200, 700, 128
    inp = si.make_inputs(2, N=N, V=V, d=d)
    wide = torch.zeros((N, d + 64), dtype=torch.bfloat16, device="cuda")
    wide[:, :d] = bf16_dev(inp["h"])
    d_inp = dev_inputs(inp)
    d_inp["h"] = wide[:, :d]
    nll, _, _ = run_fwd(lm, d_inp, 30.0)
    ref, _ = oracle_mod.fwd(inp["h"], inp["W"], inp["tgt"], 30.0)
    assert np.abs(nll - ref).max() <= NLL_ATOL


def test_fwd_row_mask(lm, oracle_mod):
    """Sliding-window mask (last 64 rows of each 2048-row window scored) plus
    a ragged tail: masked rows give 0, scored rows match the oracle."""
    N, V, d = 2 * 2048 + 100, 1024, 512
    inp = si.make_inputs(4, N=N, V=V, d=d)
    mask = si.window_mask(N)
    mask[-3:] = 1
    d_inp = dev_inputs(inp)
    dm = torch.from_numpy(mask).cuda()
    nll, lse, _ = run_fwd(lm, d_inp, 30.0, mask=dm)
    ref, ref_lse = oracle_mod.fwd(inp["h"], inp["W"], inp["tgt"], 30.0, mask=mask)
    assert np.all(nll[mask == 0] == 0) and np.all(lse[mask == 0] == 0)
    assert np.abs(nll - ref).max() <= NLL_ATOL


def test_fwd_eval_stream_call_sampled(lm, oracle_mod):
    """One call of the sliding-window evaluation stream as `bench.py --table`
    times it: 512 windows of 2048 rows (1,048,576 rows, 32,768 scored; V=8192,
    d=512) through the compacting forward and bpb_reduce.  48 sampled scored
    rows against the oracle, every unscored row 0, and the device's bpb sums
    against the oracle's reduction of the device's nll."""
    N = 512 * si.WINDOW
    inp = si.make_inputs(4, N=N)
    mask = inp["mask"]
    d_inp = dev_inputs(inp)
    nll, lse, ws = run_fwd(lm, d_inp, 30.0, mask=d_inp["mask"])
    scored = np.nonzero(mask)[0]
    assert scored.size == 512 * si.STRIDE
    assert np.all(nll[mask == 0] == 0) and np.all(lse[mask == 0] == 0)
    assert np.all(np.isfinite(nll[scored]))
    rows = np.random.default_rng(4).choice(scored, 48, replace=False)
    ref, ref_lse = oracle_mod.fwd(inp["h"], inp["W"], inp["tgt"], 30.0, rows=rows)
    assert np.abs(nll[rows] - ref).max() <= NLL_ATOL
    assert np.abs(lse[rows] - ref_lse).max() <= NLL_ATOL
    acc = lm.bpb_acc()
    lm.bpb_reduce(torch.from_numpy(nll).cuda(), d_inp["nbytes"], acc, row_mask=d_inp["mask"], ws=ws)
    s_nll, s_bytes, n = lm.read_bpb_acc(acc)
    ref_bpb, ref_s_nll, ref_s_bytes, ref_n = oracle_mod.bpb(nll, inp["nbytes"], mask)
    assert (s_bytes, n) == (ref_s_bytes, ref_n)
    assert abs(s_nll - ref_s_nll) <= BPB_RTOL * abs(ref_s_nll)


def test_fwd_all_masked(lm):
    N, V, d = 300, 500, 128
    inp = si.make_inputs(2, N=N, V=V, d=d)
    dm = torch.zeros(N, dtype=torch.uint8, device="cuda")
    nll, lse, _ = run_fwd(lm, dev_inputs(inp), 30.0, mask=dm)
    assert np.all(nll == 0)


def test_fwd_bad_target_sets_status(lm):
    N, V, d = 130, 300, 64
    inp = si.make_inputs(2, N=N, V=V, d=d)
    d_inp = dev_inputs(inp)
    d_inp["tgt"][7] = V
    ws = lm.workspace(N, V, d)
    nll = torch.zeros(N, device="cuda")
    lm.lmhead_ce_fwd(d_inp["h"], d_inp["W"], d_inp["tgt"], 30.0, nll, None, ws=ws)
    assert lm.lmce_status(ws) == lm.LMCE_EDATA
    assert math.isnan(float(nll[7]))
    assert lm.lmce_status(ws) == lm.LMCE_OK  # the status word was cleared


def test_fwd_full_size_sampled(lm, oracle_mod):
    """Config 3 size (N=65536, V=8192) in the benchmark's launch
    configuration: 48 sampled rows against the oracle, and the bpb of all
    rows within the pages' statistical expectation."""
    inp = si.make_inputs(3)
    nll, lse, _ = run_fwd(lm, dev_inputs(inp), 30.0)
    rows = np.random.default_rng(0).choice(inp["N"], 48, replace=False)
    ref, ref_lse = oracle_mod.fwd(inp["h"], inp["W"], inp["tgt"], 30.0, rows=rows)
    assert np.abs(nll[rows] - ref).max() <= NLL_ATOL
    assert np.abs(lse[rows] - ref_lse).max() <= NLL_ATOL
    assert np.all(np.isfinite(nll))


def test_fwd_deterministic(lm):
    inp = si.make_inputs(2, N=1000, V=3000, d=512)
    d_inp = dev_inputs(inp)
    a, la, _ = run_fwd(lm, d_inp, 30.0)
    b, lb, _ = run_fwd(lm, d_inp, 30.0)
    assert np.array_equal(a, b) and np.array_equal(la, lb)
