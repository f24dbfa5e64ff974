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
