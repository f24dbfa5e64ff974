"""More storage formats of the tied table (asymmetric int4 with zero points,
int8 / int7 rows, fp16), the per-id byte-length bits per byte, softcap 0 (no
cap) and softcaps beyond the fixed-shift range, and the RMSNorm in front of
the head: every one through the C ABI against the fp64 oracle on the same
inputs.  Dequantisation is bit-exact over every code and every finite fp16
scale; the rest within the stated tolerances."""
import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_util import BPB_RTOL, GRAD_RTOL, NLL_ATOL, bf16_dev, bf16_to_f64, dev_inputs, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lm():
    import lm_head_softcapped_lmhead_b300 as lm
    lm.lib()
    return lm


def _finite_f16():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    return bits[np.isfinite(bits.view(np.float16))]


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _i16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()


# ---- dequantisation, bit-exact over the whole input domain ----------------------

def test_dequant_int4_asym_all_codes_zeros_scales(lm, oracle_mod):
    sc = _finite_f16()
    d, group = 64, 64
    row = np.repeat(np.arange(16), 4)           # every code, 4 times along d
    V = sc.size * 16                             # every scale with every zero point
    Q = np.tile(row, (V, 1))
    Wq = (Q[:, 0::2] | (Q[:, 1::2] << 4)).astype(np.uint8)
    scales = np.repeat(sc, 16)[:, None].copy()
    zeros = np.tile(np.arange(16, dtype=np.uint8), sc.size)[:, None].copy()
    want = oracle_mod.dequant_int4_asym(Wq, scales, zeros, d, group)
    q_t, s_t, z_t = torch.from_numpy(Wq).cuda(), _i16(scales), torch.from_numpy(zeros).cuda()
    out = torch.empty((V, d), dtype=torch.bfloat16, device="cuda")
    lm.lmhead_qhead_dequant(lm.qhead(lm.LMCE_QHEAD_INT4_ASYM, q_t, s_t, z_t, group), V, d, out)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(out), want)


def test_dequant_int8_rows_all_codes_scales(lm, oracle_mod):
    sc = _finite_f16()
    d = 256
    q = np.tile(np.arange(-128, 128, dtype=np.int8), (sc.size, 1))
    want = oracle_mod.dequant_int8_rows(q, sc)
    out = torch.empty((sc.size, d), dtype=torch.bfloat16, device="cuda")
    q_t = torch.from_numpy(q).cuda()
    lm.lmhead_qhead_dequant(lm.qhead(lm.LMCE_QHEAD_INT8_ROW, q_t, _i16(sc)), sc.size, d, out)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(out), want)


def test_dequant_fp16_all_patterns(lm, oracle_mod):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(128, 512)
    want = oracle_mod.dequant_f16(bits)
    out = torch.empty((128, 512), dtype=torch.bfloat16, device="cuda")
    lm.lmhead_qhead_dequant(lm.qhead(lm.LMCE_QHEAD_FP16, _i16(bits)), 128, 512, out)
    torch.cuda.synchronize()
    got = _bits(out)
    nan = np.isnan(bits.view(np.float16))
    assert np.array_equal(got[~nan], want[~nan])
    assert np.all(np.isnan(si.bf16_bits_to_f32(got[nan])))


# ---- forward / backward through a quantised head --------------------------------

def _head(lm, fmt, W_bits, group=64):
    """(lmce_qhead, tensors kept alive, the oracle's dequantised bf16 bits)."""
    import oracle
    d = W_bits.shape[1]
    if fmt == lm.LMCE_QHEAD_INT4_ASYM:
        Wq, sc, zp = si.quantize_int4_asym(W_bits, group)
        keep = (torch.from_numpy(Wq).cuda(), _i16(sc), torch.from_numpy(zp).cuda())
        return lm.qhead(fmt, *keep, group=group), keep, oracle.dequant_int4_asym(Wq, sc, zp, d, group)
    if fmt in (lm.LMCE_QHEAD_INT8_ROW, -7):
        q, sc = si.quantize_int8_rows(W_bits, 127 if fmt > 0 else 63)
        keep = (torch.from_numpy(q).cuda(), _i16(sc))
        return lm.qhead(lm.LMCE_QHEAD_INT8_ROW, *keep), keep, oracle.dequant_int8_rows(q, sc)
    if fmt == lm.LMCE_QHEAD_FP16:
        f = si.to_fp16_bits(W_bits)
        keep = (_i16(f),)
        return lm.qhead(fmt, *keep), keep, oracle.dequant_f16(f)
    Wq, sc = si.quantize_int4_rtn(W_bits, group)
    keep = (torch.from_numpy(Wq).cuda(), _i16(sc))
    return lm.qhead(fmt, *keep, group=group), keep, oracle.dequant_int4(Wq, sc, d, group)


FORMATS = [("int4", 1), ("int4_asym", 2), ("int8_row", 3), ("int7_row", -7), ("fp16", 4)]


@pytest.mark.parametrize("name,fmt", FORMATS)
def test_quantised_head_fwd_bwd(lm, oracle_mod, name, fmt):
    N, V, d, c = 300, 700, 256, 30.0
    inp = si.make_inputs(2, N=N, V=V, d=d, w_scale=20.0)
    hd, keep, Wdq = _head(lm, fmt, inp["W"])
    d_inp = dev_inputs(inp)
    ws = lm.workspace(N, V, d, lm.LMCE_WS_QHEAD)
    w = 1.0 / N
    nll, lse = torch.empty(N, device="cuda"), torch.empty(N, device="cuda")
    lm.lmhead_ce_fwd_q(d_inp["h"], hd, V, c, d_inp["tgt"], nll, lse, ws=ws)
    assert lm.lmce_status(ws) == lm.LMCE_OK
    ref_nll, ref_lse = oracle_mod.fwd(inp["h"], Wdq, inp["tgt"], c)
    assert np.abs(nll.cpu().numpy() - ref_nll).max() <= NLL_ATOL
    ref_dh, _ = oracle_mod.bwd(inp["h"], Wdq, inp["tgt"], c, ref_lse, w, want_dW=False)
    dh = torch.empty_like(d_inp["h"])
    lm.lmhead_ce_bwd_q(d_inp["h"], hd, V, c, d_inp["tgt"], lse, w, dh, ws=ws, nll=nll)
    assert lm.lmce_status(ws) == lm.LMCE_OK
    assert rel_fro(bf16_to_f64(dh), ref_dh) <= GRAD_RTOL
    nll2, lse2, dh2 = torch.empty_like(nll), torch.empty_like(lse), torch.empty_like(dh)
    lm.lmhead_ce_fwd_bwd_q(d_inp["h"], hd, V, c, d_inp["tgt"], w, nll2, lse2, dh2, ws=ws)
    assert lm.lmce_status(ws) == lm.LMCE_OK
    assert np.abs(nll2.cpu().numpy() - ref_nll).max() <= NLL_ATOL
    assert rel_fro(bf16_to_f64(dh2), ref_dh) <= GRAD_RTOL
    del keep


# ---- bits per byte with per-id byte lengths ---------------------------------------

def test_bpb_reduce_lut_matches_oracle(lm, oracle_mod):
    """Host-drawn nll values through bpb_reduce_lut against the oracle's bpb
    with bytes from the same table; a masked row and a row whose target is out
    of range (skipped, LMCE_EDATA)."""
    rng = np.random.default_rng(31)
    N, V = 70000, 8192
    nll = rng.random(N).astype(np.float32) * 12
    tgt = si.zipf_ids(rng, N, V, 1.1)
    mask = (rng.random(N) > 0.1).astype(np.uint8)
    lut = si.make_byte_lut(V)
    ws = lm.workspace(1, 1, 64)
    acc = lm.bpb_acc()
    t_nll, t_tgt = torch.from_numpy(nll).cuda(), torch.from_numpy(tgt).cuda()
    t_lut, t_mask = torch.from_numpy(lut).cuda(), torch.from_numpy(mask).cuda()
    lm.bpb_reduce_lut(t_nll, t_tgt, t_lut, acc, row_mask=t_mask, ws=ws)
    assert lm.lmce_status(ws) == lm.LMCE_OK
    b, sn, sb, n = oracle_mod.bpb_lut(nll.astype(np.float64), tgt, lut, mask)
    gsn, gsb, gn = lm.read_bpb_acc(acc)
    assert (gsb, gn) == (sb, n)
    assert abs(gsn - sn) <= 1e-12 * sn and abs(lm.lmce_bpb(acc) - b) <= 1e-12 * b
    # the same rows with bytes materialised per row give the same bits
    acc2 = lm.bpb_acc()
    lm.bpb_reduce(t_nll, torch.from_numpy(lut[tgt]).cuda(), acc2, row_mask=t_mask, ws=ws)
    assert torch.equal(acc.view(torch.int64), acc2.view(torch.int64))
    bad = tgt.copy()
    bad[5] = V
    mask[5] = 1
    acc3 = lm.bpb_acc()
    lm.bpb_reduce_lut(t_nll, torch.from_numpy(bad).cuda(), t_lut, acc3, row_mask=torch.from_numpy(mask).cuda(),
                      ws=ws)
    assert lm.lmce_status(ws) == lm.LMCE_EDATA
    assert lm.read_bpb_acc(acc3)[2] == int(mask.sum()) - 1


def test_bpb_lut_end_to_end(lm, oracle_mod):
    """Forward + bpb_reduce_lut against the oracle's forward + bpb with the
    same byte table (bits per byte within 1e-5 relative)."""
    inp = si.make_inputs(2, N=1500, V=3000, d=256, w_scale=10.0)
    d_inp = dev_inputs(inp)
    N, V, d = 1500, 3000, 256
    lut = si.make_byte_lut(V)
    ws = lm.workspace(N, V, d)
    nll = torch.empty(N, device="cuda")
    lm.lmhead_ce_fwd(d_inp["h"], d_inp["W"], d_inp["tgt"], 30.0, nll, None, ws=ws)
    acc = lm.bpb_acc()
    lm.bpb_reduce_lut(nll, d_inp["tgt"], torch.from_numpy(lut).cuda(), acc, ws=ws)
    assert lm.lmce_status(ws) == lm.LMCE_OK
    ref_nll, _ = oracle_mod.fwd(inp["h"], inp["W"], inp["tgt"], 30.0)
    b, *_ = oracle_mod.bpb_lut(ref_nll, inp["tgt"], lut)
    assert abs(lm.lmce_bpb(acc) - b) <= BPB_RTOL * b


# ---- softcap 0 (no cap) and softcaps beyond the fixed-shift range --------------------

@pytest.mark.parametrize("c,N,V,d,w_scale", [
    (0.0, 300, 700, 256, 100.0),    # no cap: logits up to ~150, e^s far beyond fp32
    (0.0, 257, 1000, 512, 5.0),
    (80.0, 300, 700, 256, 100.0),   # above lmce_softcap_max(700) = 79.45: running maximum
    (200.0, 130, 260, 128, 100.0),
    (79.5, 200, 1000, 512, 100.0),  # just above lmce_softcap_max(1000) = 79.09
])
def test_online_forward_matches_oracle(lm, oracle_mod, c, N, V, d, w_scale):
    inp = si.make_inputs(2, N=N, V=V, d=d, w_scale=w_scale)
    d_inp = dev_inputs(inp)
    ws = lm.workspace(N, V, d)
    nll, lse = torch.empty(N, device="cuda"), torch.empty(N, device="cuda")
    lm.lmhead_ce_fwd(d_inp["h"], d_inp["W"], d_inp["tgt"], c, nll, lse, ws=ws)
    assert lm.lmce_status(ws) == lm.LMCE_OK
    ref_nll, ref_lse = oracle_mod.fwd(inp["h"], inp["W"], inp["tgt"], c)
    if c == 0.0 and w_scale > 50:
        assert ref_lse.max() > 90.0   # the fixed shift could not hold these sums in fp32
    assert np.abs(nll.cpu().numpy() - ref_nll).max() <= NLL_ATOL
    assert np.abs(lse.cpu().numpy() - ref_lse).max() <= NLL_ATOL


@pytest.mark.parametrize("c", [0.0, 200.0])
def test_online_training_step_matches_oracle(lm, oracle_mod, c):
    """lmhead_ce_fwd_bwd at c = 0 and c = 200 (forward with a running maximum,
    then the dh and dW passes), with a row mask and dW accumulation."""
    N, V, d = 400, 600, 128
    inp = si.make_inputs(2, N=N, V=V, d=d, w_scale=40.0)
    mask = (np.arange(N) % 5 != 2).astype(np.uint8)
    M = int(mask.sum())
    d_inp = dev_inputs(inp)
    ws = lm.workspace(N, V, d, lm.LMCE_WS_MASKED)
    nll, lse = torch.empty(N, device="cuda"), torch.empty(N, device="cuda")
    dh = torch.empty_like(d_inp["h"])
    init = torch.randn(V, d, device="cuda") * 1e-3
    dW = init.clone()
    lm.lmhead_ce_fwd_bwd(d_inp["h"], d_inp["W"], d_inp["tgt"], c, 1.0 / M, nll, lse, dh=dh, dW=dW,
                         accumulate_dW=True, row_mask=torch.from_numpy(mask).cuda(), ws=ws)
    assert lm.lmce_status(ws) == lm.LMCE_OK
    ref_nll, ref_lse = oracle_mod.fwd(inp["h"], inp["W"], inp["tgt"], c, mask=mask)
    assert np.abs(nll.cpu().numpy() - ref_nll).max() <= NLL_ATOL
    ref_dh, ref_dW = oracle_mod.bwd(inp["h"], inp["W"], inp["tgt"], c, ref_lse, 1.0 / M, mask=mask)
    assert rel_fro(bf16_to_f64(dh), ref_dh) <= GRAD_RTOL
    assert rel_fro((dW - init).double().cpu().numpy(), ref_dW) <= GRAD_RTOL


# ---- RMSNorm in front of the head --------------------------------------------------

def _norm_inputs(N, V, d, seed=41, x_scale=2.0):
    rng = np.random.default_rng(seed)
    x = si.f32_to_bf16_bits((rng.standard_normal((N, d)) * x_scale).astype(np.float32))
    g = (1.0 + 0.1 * rng.standard_normal(d)).astype(np.float32)
    inp = si.make_inputs(2, N=N, V=V, d=d, w_scale=20.0)
    return x, g, inp


@pytest.mark.parametrize("with_gain", [True, False])
def test_rmsnorm_kernels_match_oracle(lm, oracle_mod, with_gain):
    N, d, eps = 1000, 512, 1e-6
    x, g, _ = _norm_inputs(N, 64, d)
    gg = g if with_gain else None
    tx = bf16_dev(x)
    tg = torch.from_numpy(g).cuda() if with_gain else None
    h = torch.empty_like(tx)
    rinv = torch.empty(N, device="cuda")
    lm.lmhead_rmsnorm_fwd(tx, tg, eps, h, rinv)
    ref_h, ref_r = oracle_mod.rmsnorm_fwd(x, gg, eps)
    assert np.abs(rinv.double().cpu().numpy() / ref_r - 1).max() <= 1e-6
    assert np.abs(bf16_to_f64(h) - ref_h).max() <= 2.0 ** -8 * np.abs(ref_h).max()
    rng = np.random.default_rng(42)
    dh_bits = si.f32_to_bf16_bits(rng.standard_normal((N, d)).astype(np.float32))
    dx = torch.empty_like(tx)
    dg = torch.zeros(d, device="cuda")
    ws = lm.workspace(N, 1, d, lm.LMCE_WS_RMSNORM)
    lm.lmhead_rmsnorm_bwd(tx, tg, rinv, bf16_dev(dh_bits), dx, dg, ws=ws)
    torch.cuda.synchronize()
    ref_dx, ref_dg = oracle_mod.rmsnorm_bwd(x, gg, eps, oracle_mod.widen_bf16(dh_bits))
    assert rel_fro(bf16_to_f64(dx), ref_dx) <= GRAD_RTOL
    assert rel_fro(dg.double().cpu().numpy(), ref_dg) <= 1e-5
    dg2 = dg.clone()
    lm.lmhead_rmsnorm_bwd(tx, tg, rinv, bf16_dev(dh_bits), dx, dg2, accumulate_dg=True, ws=ws)
    torch.cuda.synchronize()
    assert torch.equal(dg2, dg + dg)   # deterministic partials, added once more


@pytest.mark.parametrize("masked", [False, True])
def test_rmsnorm_head_training_step(lm, oracle_mod, masked):
    """lmhead_ce_fwd_bwd_rmsnorm (normalise, forward + dh, dW, then dx and dg)
    against the oracle's RMSNorm -> forward -> backward -> RMSNorm backward.
    The normalised rows enter the head as bf16 (the model's dtype; the
    forward + backward workload's hidden states are RMSNorm rows rounded to
    bf16), so the oracle's head runs on its RMSNorm output rounded once to
    bf16, and the RMSNorm backward takes the head's dh with respect to those
    rows."""
    N, V, d, c, eps = 600, 900, 256, 30.0, 1e-6
    x, g, inp = _norm_inputs(N, V, d)
    mask = (np.arange(N) % 4 != 1).astype(np.uint8) if masked else None
    M = N if mask is None else int(mask.sum())
    w = 1.0 / M
    tx = bf16_dev(x)
    tg = torch.from_numpy(g).cuda()
    d_inp = dev_inputs(inp)
    ws = lm.workspace(N, V, d, lm.LMCE_WS_RMSNORM | (lm.LMCE_WS_MASKED if masked else 0))
    nll, lse = torch.empty(N, device="cuda"), torch.empty(N, device="cuda")
    dx = torch.empty_like(tx)
    dg = torch.zeros(d, device="cuda")
    dW = torch.zeros((V, d), device="cuda")
    tm = None if mask is None else torch.from_numpy(mask).cuda()
    lm.lmhead_ce_fwd_bwd_rmsnorm(tx, tg, eps, d_inp["W"], d_inp["tgt"], c, w, nll, lse, dx=dx, dg=dg, dW=dW,
                                 row_mask=tm, ws=ws)
    assert lm.lmce_status(ws) == lm.LMCE_OK
    hn = oracle_mod.round_bf16(oracle_mod.rmsnorm_fwd(x, g, eps)[0])
    ref_nll, ref_lse = oracle_mod.fwd(hn, inp["W"], inp["tgt"], c, mask=mask)
    assert np.abs(nll.cpu().numpy() - ref_nll).max() <= NLL_ATOL
    ref_dhn, ref_dW = oracle_mod.bwd(hn, inp["W"], inp["tgt"], c, ref_lse, w, mask=mask)
    ref_dx, ref_dg = oracle_mod.rmsnorm_bwd(x, g, eps, ref_dhn)
    assert rel_fro(bf16_to_f64(dx), ref_dx) <= GRAD_RTOL
    assert rel_fro(dg.double().cpu().numpy(), ref_dg) <= GRAD_RTOL
    assert rel_fro(dW.double().cpu().numpy(), ref_dW) <= GRAD_RTOL
    nll_f = torch.empty(N, device="cuda")
    lm.lmhead_ce_fwd_rmsnorm(tx, tg, eps, d_inp["W"], d_inp["tgt"], c, nll_f, row_mask=tm, ws=ws)
    assert lm.lmce_status(ws) == lm.LMCE_OK
    assert np.abs(nll_f.cpu().numpy() - ref_nll).max() <= NLL_ATOL
