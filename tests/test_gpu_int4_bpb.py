"""int4 head (bit-exact dequantisation, forward and dh against the oracle)
and the bits-per-byte reduction (against the oracle, deterministic)."""
import math

import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_util import NLL_ATOL, BPB_RTOL, GRAD_RTOL, dev_inputs, rel_fro, bf16_to_f64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lm():
    import lm_head_softcapped_lmhead_b300 as lm
    lm.lib()
    return lm


def test_dequant_bit_exact(lm, oracle_mod):
    inp = si.make_inputs(5, N=8, V=1000, d=512)
    d_inp = dev_inputs(inp)
    out = torch.empty((1000, 512), dtype=torch.bfloat16, device="cuda")
    lm.lmhead_int4_dequant(d_inp["Wq"], d_inp["scales"], 512, 64, out)
    torch.cuda.synchronize()
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    ref = oracle_mod.dequant_int4(inp["Wq"], inp["scales"], 512, 64)
    assert np.array_equal(got, ref)


def test_dequant_all_scales_bit_exact(lm, oracle_mod):
    """Every finite fp16 scale x every nibble, on the device."""
    sc = np.arange(65536, dtype=np.uint16)
    sc = sc[np.isfinite(sc.view(np.float16))]
    V, d = sc.size, 64
    q = np.arange(d) % 16
    nib = (np.where(q >= 8, q - 16, q) & 0xF).astype(np.uint8)
    Wq = np.tile((nib[0::2] | (nib[1::2] << 4)).astype(np.uint8), (V, 1))
    scales = sc.reshape(V, 1)
    out = torch.empty((V, d), dtype=torch.bfloat16, device="cuda")
    lm.lmhead_int4_dequant(torch.from_numpy(Wq).cuda(), torch.from_numpy(scales.view(np.int16)).cuda(), d, 64, out)
    torch.cuda.synchronize()
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, oracle_mod.dequant_int4(Wq, scales, d, 64))


@pytest.mark.parametrize("N,V", [(300, 1000), (2048, 8192)])
def test_int4_fwd_bwd_match_oracle(lm, oracle_mod, N, V):
    d = 512
    inp = si.make_inputs(5, N=N, V=V, d=d)
    d_inp = dev_inputs(inp)
    Wdeq = oracle_mod.dequant_int4(inp["Wq"], inp["scales"], d, 64)
    ws = lm.workspace(N, V, d, lm.LMCE_WS_INT4)
    nll = torch.zeros(N, device="cuda")
    lse = torch.zeros(N, device="cuda")
    lm.lmhead_ce_fwd_int4(d_inp["h"], d_inp["Wq"], d_inp["scales"], 64, 30.0, d_inp["tgt"], nll, lse, ws=ws)
    dh = torch.zeros_like(d_inp["h"])
    lm.lmhead_ce_bwd_int4(d_inp["h"], d_inp["Wq"], d_inp["scales"], 64, 30.0, d_inp["tgt"], lse, 1.0 / N, dh, ws=ws,
                          nll=nll)
    assert lm.lmce_status(ws) == lm.LMCE_OK
    ref_nll, ref_lse = oracle_mod.fwd(inp["h"], Wdeq, inp["tgt"], 30.0)
    assert np.abs(nll.cpu().numpy() - ref_nll).max() <= NLL_ATOL
    if N <= 300:
        ref_dh, _ = oracle_mod.bwd(inp["h"], Wdeq, inp["tgt"], 30.0, ref_lse, 1.0 / N, want_dW=False)
        assert rel_fro(bf16_to_f64(dh), ref_dh) <= GRAD_RTOL
    else:
        rows = np.arange(0, N, N // 16)
        ref = oracle_mod.dh_rows(inp["h"], Wdeq, inp["tgt"], 30.0, rows, ref_lse[rows], 1.0 / N)
        assert rel_fro(bf16_to_f64(dh)[rows], ref) <= GRAD_RTOL


@pytest.mark.parametrize("N,V,c,masked", [
    (300, 1000, 30.0, False),    # ragged N and V, the fused pass
    (257, 700, 70.0, False),     # softcap above 60: forward and dh as two passes
    (400, 600, 30.0, True),      # row mask
    (130, 100, 30.0, False),     # V below one 128-column tile
])
def test_int4_fused_fwd_bwd_matches_oracle(lm, oracle_mod, N, V, c, masked):
    d = 512
    inp = si.make_inputs(5, N=N, V=V, d=d)
    d_inp = dev_inputs(inp)
    mask = (np.arange(N) % 7 != 3).astype(np.uint8) if masked else None
    M = N if mask is None else int(mask.sum())
    Wdeq = oracle_mod.dequant_int4(inp["Wq"], inp["scales"], d, 64)
    ws = lm.workspace(N, V, d, lm.LMCE_WS_INT4 | (lm.LMCE_WS_MASKED if masked else 0))
    nll = torch.full((N,), float("nan"), device="cuda")
    lse = torch.full((N,), float("nan"), device="cuda")
    dh = torch.full_like(d_inp["h"], float("nan"))
    lm.lmhead_ce_fwd_bwd_int4(d_inp["h"], d_inp["Wq"], d_inp["scales"], 64, c, d_inp["tgt"], 1.0 / M, nll, lse, dh,
                              row_mask=None if mask is None else torch.from_numpy(mask).cuda(), ws=ws)
    assert lm.lmce_status(ws) == lm.LMCE_OK
    ref_nll, ref_lse = oracle_mod.fwd(inp["h"], Wdeq, inp["tgt"], c, mask=mask)
    assert np.abs(nll.cpu().numpy() - ref_nll).max() <= NLL_ATOL
    assert np.abs(lse.cpu().numpy() - ref_lse).max() <= NLL_ATOL
    ref_dh, _ = oracle_mod.bwd(inp["h"], Wdeq, inp["tgt"], c, ref_lse, 1.0 / M, mask=mask, want_dW=False)
    got = bf16_to_f64(dh)
    if mask is not None:
        assert np.all(got[mask == 0] == 0)
    assert rel_fro(got, ref_dh) <= GRAD_RTOL


def test_int4_fused_full_size_sampled(lm, oracle_mod):
    """The int4 head at full size (N=65536, V=8192, d=512): nll and dh of 32
    sampled rows against the oracle, and nll against the two-call path
    (lmhead_ce_fwd_int4 then lmhead_ce_bwd_int4) on every row."""
    inp = si.make_inputs(5)
    N, V, d = inp["N"], inp["V"], inp["d"]
    d_inp = dev_inputs(inp)
    ws = lm.workspace(N, V, d, lm.LMCE_WS_INT4)
    nll = torch.empty(N, device="cuda")
    lse = torch.empty(N, device="cuda")
    dh = torch.empty_like(d_inp["h"])
    lm.lmhead_ce_fwd_bwd_int4(d_inp["h"], d_inp["Wq"], d_inp["scales"], 64, 30.0, d_inp["tgt"], 1.0 / N, nll, lse,
                              dh, ws=ws)
    nll2 = torch.empty(N, device="cuda")
    lse2 = torch.empty(N, device="cuda")
    dh2 = torch.empty_like(d_inp["h"])
    lm.lmhead_ce_fwd_int4(d_inp["h"], d_inp["Wq"], d_inp["scales"], 64, 30.0, d_inp["tgt"], nll2, lse2, ws=ws)
    lm.lmhead_ce_bwd_int4(d_inp["h"], d_inp["Wq"], d_inp["scales"], 64, 30.0, d_inp["tgt"], lse2, 1.0 / N, dh2,
                          ws=ws, nll=nll2)
    assert lm.lmce_status(ws) == lm.LMCE_OK
    n = nll.cpu().numpy()
    assert np.all(np.isfinite(n))
    assert np.abs(n - nll2.cpu().numpy()).max() <= NLL_ATOL
    assert rel_fro(bf16_to_f64(dh), bf16_to_f64(dh2)) <= GRAD_RTOL
    Wdeq = oracle_mod.dequant_int4(inp["Wq"], inp["scales"], d, 64)
    rows = np.random.default_rng(5).choice(N, 32, replace=False)
    ref_nll, ref_lse = oracle_mod.fwd(inp["h"], Wdeq, inp["tgt"], 30.0, rows=rows)
    assert np.abs(n[rows] - ref_nll).max() <= NLL_ATOL
    ref = oracle_mod.dh_rows(inp["h"], Wdeq, inp["tgt"], 30.0, rows, ref_lse, 1.0 / N)
    assert rel_fro(bf16_to_f64(dh)[rows], ref) <= GRAD_RTOL


def test_bpb_reduce_matches_oracle_and_is_deterministic(lm, oracle_mod):
    rng = np.random.default_rng(4)
    N = 100003
    nll = (rng.random(N) * 12).astype(np.float32)
    nbytes = rng.integers(1, 13, size=N).astype(np.int32)
    mask = (rng.random(N) > 0.3).astype(np.uint8)
    ws = lm.workspace(1, 1, 64)
    outs = []
    for _ in range(3):
        acc = lm.bpb_acc()
        lm.bpb_reduce(torch.from_numpy(nll).cuda(), torch.from_numpy(nbytes).cuda(), acc,
                      row_mask=torch.from_numpy(mask).cuda(), ws=ws)
        outs.append(lm.read_bpb_acc(acc))
    assert outs[0] == outs[1] == outs[2]
    b_ref, sn, sb, n = oracle_mod.bpb(nll.astype(np.float64), nbytes, mask)
    assert outs[0][1] == sb and outs[0][2] == n
    assert abs(outs[0][0] - sn) <= 1e-12 * sn
    assert abs(lm.lmce_bpb(acc) - b_ref) <= 1e-12 * b_ref


def test_bpb_accumulates_across_calls_and_zero_bytes(lm):
    ws = lm.workspace(1, 1, 64)
    acc = lm.bpb_acc()
    nll = torch.full((1000,), math.log(1024), device="cuda")
    nb = torch.full((1000,), 4, dtype=torch.int32, device="cuda")
    lm.bpb_reduce(nll, nb, acc, ws=ws)
    lm.bpb_reduce(nll, nb, acc, ws=ws)
    sn, sb, n = lm.read_bpb_acc(acc)
    assert n == 2000 and sb == 8000
    assert lm.lmce_bpb(acc) == pytest.approx(10.0 / 4.0, rel=1e-6)
    empty = lm.bpb_acc()
    with pytest.raises(lm.LmceError):
        lm.lmce_bpb(empty)


def test_end_to_end_config1_bpb(lm, oracle_mod):
    """Config 1 end to end: forward + bpb_reduce against the oracle's bpb."""
    inp = si.make_inputs(1)
    d_inp = dev_inputs(inp)
    N, V, d = inp["N"], inp["V"], inp["d"]
    ws = lm.workspace(N, V, d)
    nll = torch.zeros(N, device="cuda")
    lm.lmhead_ce_fwd(d_inp["h"], d_inp["W"], d_inp["tgt"], 30.0, nll, None, ws=ws)
    acc = lm.bpb_acc()
    lm.bpb_reduce(nll, d_inp["nbytes"], acc, ws=ws)
    got = lm.lmce_bpb(acc)
    ref_nll, _ = oracle_mod.fwd(inp["h"], inp["W"], inp["tgt"], 30.0)
    b_ref, *_ = oracle_mod.bpb(ref_nll, inp["nbytes"])
    assert abs(got - b_ref) <= BPB_RTOL * b_ref
