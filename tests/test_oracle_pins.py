"""Pins of the fp64 CPU oracle against facts fixed by mathematics, by an
independent library routine, or by brute force -- never against the oracle
itself.  CPU only.

Each test names the mistake it would catch.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import synth_inputs as si

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_case(rng, N, V, d, zscale, c):
    h = rng.standard_normal((N, d))
    W = rng.standard_normal((V, d)) * (zscale / math.sqrt(d))
    t = rng.integers(0, V, size=N)
    return h, W, t


# ---- number formats -------------------------------------------------------

def test_f16_decode_all_patterns(oracle_mod):
    """Every binary16 bit pattern decodes like numpy's float16 (catches a
    wrong exponent bias or a broken subnormal branch)."""
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle_mod.f16_to_f64(b) for b in bits])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isinf(got), np.isinf(ref))
    assert np.array_equal(np.isnan(got), np.isnan(ref))


def test_bf16_rounding_matches_torch(oracle_mod):
    """Round-to-nearest-even to bf16 agrees bit for bit with torch's
    float32 -> bfloat16 conversion on random values, exact ties, subnormals
    and overflow (catches round-half-up or truncation)."""
    rng = np.random.default_rng(7)
    with np.errstate(over="ignore"):
        big = (rng.standard_normal(5000) * 3e38).astype(np.float32)
    vals = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(5000) * 1e-38).astype(np.float32),
        big,
    ])
    # exact ties: a bf16 value plus half an ulp, for even and odd mantissas
    base = (rng.integers(0x3000, 0x5000, size=4000).astype(np.uint32) << 16)
    ties = (base | 0x8000).view(np.float32)
    vals = np.concatenate([vals, ties, np.float32([0.0, -0.0, 1.0, -1.0,
                                                  3.3895314e38, 1e-45])])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle_mod.f64_to_bf16_rne(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_round_bf16_array_matches_scalar_and_torch(oracle_mod):
    """The array form of the bf16 rounding equals the scalar one and torch's
    float64 -> bfloat16 on randoms, ties and edge values."""
    rng = np.random.default_rng(13)
    x = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-40, 39, 2000),
                        [0.0, -0.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 3.4e38, -1e-45, np.inf]])
    got = oracle_mod.round_bf16(x)
    assert np.array_equal(got, np.array([oracle_mod.f64_to_bf16_rne(float(v)) for v in x], dtype=np.uint16))
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


def test_widen_bf16_exact(oracle_mod):
    bits = np.arange(0, 65536, 7, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle_mod.widen_bf16(bits)
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])


# ---- int4 dequantisation: brute force over the whole domain ---------------

def test_dequant_int4_brute_force(oracle_mod):
    """All 16 nibbles x every finite fp16 scale, bit for bit against torch
    (q * scale is exact in fp32, then one RNE rounding to bf16).  Catches a
    swapped nibble order, a sign-extension slip or a double rounding."""
    sc_bits = np.arange(65536, dtype=np.uint16)
    sc_bits = sc_bits[np.isfinite(sc_bits.view(np.float16))]
    G = sc_bits.size                      # one group of 64 per scale
    d = 64
    # element k of each row holds nibble value (k % 16) as two's complement
    q = (np.arange(d) % 16)
    q = np.where(q >= 8, q - 16, q)
    nib = (q & 0xF).astype(np.uint8)
    row = (nib[0::2] | (nib[1::2] << 4)).astype(np.uint8)
    Wq = np.tile(row, (G, 1))
    scales = sc_bits.reshape(G, 1)
    got = oracle_mod.dequant_int4(Wq, scales, d=d, group=64)
    scf = torch.from_numpy(sc_bits.view(np.float16).astype(np.float32)).reshape(G, 1)
    prod = torch.from_numpy(q.astype(np.float32)).reshape(1, d) * scf
    ref = prod.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


# ---- forward: closed forms and an independent library routine ------------

@pytest.mark.parametrize("V", [1024, 8192])
def test_zero_logits_give_ln_V(oracle_mod, V):
    """h = 0 -> every softcapped logit is 0 -> nll = ln V exactly, and
    bpb = N log2 V / sum(bytes)."""
    N, d = 64, 512
    inp = si.make_inputs(2, N=N, V=V, d=d)
    h = np.zeros((N, d))
    nll, lse = oracle_mod.fwd(h, inp["W"], inp["tgt"], 30.0)
    assert np.allclose(nll, math.log(V), rtol=0, atol=1e-13)
    assert np.allclose(lse, math.log(V), rtol=0, atol=1e-13)
    b, sn, sb, n = oracle_mod.bpb(nll, inp["nbytes"])
    assert n == N and sb == int(inp["nbytes"].sum())
    assert b == pytest.approx(N * math.log2(V) / sb, rel=1e-14)


@pytest.mark.parametrize("V,expect", [(1024, 2.106067), (8192, 4.073739)])
def test_one_hot_logit_closed_form(oracle_mod, V, expect):
    """h_i = a e_k and W = e_t e_k^T: one logit of height a at the target and
    zeros elsewhere, so nll = ln(e^{c tanh(a/c)} + V - 1) - c tanh(a/c).
    a = 5, c = 30.  A non-target row gets ln(e^{c tanh(a/c)} + V - 1)."""
    a, c, d, k = 5.0, 30.0, 16, 3
    t_hot = 11
    W = np.zeros((V, d)); W[t_hot, k] = 1.0
    h = np.zeros((2, d)); h[:, k] = a
    tgt = np.array([t_hot, 0])
    nll, _ = oracle_mod.fwd(h, W, tgt, c)
    sa = c * math.tanh(a / c)
    assert nll[0] == pytest.approx(math.log(math.exp(sa) + V - 1) - sa, abs=1e-12)
    assert nll[0] == pytest.approx(expect, abs=5e-7)
    assert nll[1] == pytest.approx(math.log(math.exp(sa) + V - 1), abs=1e-12)


@pytest.mark.parametrize("c", [1.0, 2.0, 30.0, 50.0])
def test_matches_torch_cross_entropy(oracle_mod, c):
    """torch's fp64 cross_entropy of c*tanh(h W^T / c) is an independent
    implementation of the same definition (catches a dropped softcap, a
    wrong sign, a transposed operand or a wrong target index)."""
    rng = np.random.default_rng(11)
    h, W, t = _rand_case(rng, 37, 301, 24, zscale=3.0 * c, c=c)
    nll, lse = oracle_mod.fwd(h, W, t, c)
    z = torch.from_numpy(h) @ torch.from_numpy(W).T
    s = c * torch.tanh(z / c)
    ref = torch.nn.functional.cross_entropy(s, torch.from_numpy(t), reduction="none").numpy()
    assert np.allclose(nll, ref, rtol=0, atol=1e-12)
    assert np.allclose(lse, torch.logsumexp(s, dim=1).numpy(), rtol=0, atol=1e-12)


def test_large_cap_approaches_plain_ce(oracle_mod):
    """c -> infinity removes the cap: compare to plain cross_entropy(z)."""
    rng = np.random.default_rng(12)
    h, W, t = _rand_case(rng, 20, 50, 16, zscale=2.0, c=1.0)
    nll, _ = oracle_mod.fwd(h, W, t, 1e7)
    z = torch.from_numpy(h) @ torch.from_numpy(W).T
    ref = torch.nn.functional.cross_entropy(z, torch.from_numpy(t), reduction="none").numpy()
    assert np.allclose(nll, ref, rtol=0, atol=1e-9)


def test_saturated_cap_bounds(oracle_mod):
    """With W x 100 the cap saturates; any nll lies strictly between
    ln(1 + (V-1) e^{-2c}) and ln(1 + (V-1) e^{2c})."""
    inp = si.make_inputs(2, N=48, V=1024, w_scale=100.0)
    c = 30.0
    nll, _ = oracle_mod.fwd(inp["h"], inp["W"], inp["tgt"], c)
    V = 1024
    lo = math.log1p((V - 1) * math.exp(-2 * c))
    hi = math.log1p((V - 1) * math.exp(2 * c))
    assert np.all(nll > lo) and np.all(nll < hi)
    assert nll.max() > 10.0          # the cap really is active here


def test_rows_subset_and_mask(oracle_mod):
    """A row list returns exactly those rows; masked rows give 0 and leave the
    others unchanged."""
    inp = si.make_inputs(1, N=40, V=96, d=64)
    nll, lse = oracle_mod.fwd(inp["h"], inp["W"], inp["tgt"], 30.0)
    rows = np.array([5, 0, 39, 17])
    n2, l2 = oracle_mod.fwd(inp["h"], inp["W"], inp["tgt"], 30.0, rows=rows)
    assert np.array_equal(n2, nll[rows]) and np.array_equal(l2, lse[rows])
    mask = (np.arange(40) % 3 != 0).astype(np.uint8)
    n3, _ = oracle_mod.fwd(inp["h"], inp["W"], inp["tgt"], 30.0, mask=mask)
    assert np.all(n3[mask == 0] == 0)
    assert np.array_equal(n3[mask == 1], nll[mask == 1])


def test_bad_target_rejected(oracle_mod):
    inp = si.make_inputs(1, N=8, V=32, d=64)
    t = inp["tgt"].copy(); t[3] = 32
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.fwd(inp["h"], inp["W"], t, 30.0)
    mask = np.ones(8, np.uint8); mask[3] = 0       # masked: not an error
    oracle_mod.fwd(inp["h"], inp["W"], t, 30.0, mask=mask)


def test_permutation_invariances(oracle_mod):
    """Permuting vocab rows (and remapping targets) leaves nll unchanged;
    permuting rows permutes nll."""
    rng = np.random.default_rng(3)
    h, W, t = _rand_case(rng, 12, 40, 8, zscale=4.0, c=2.0)
    nll, _ = oracle_mod.fwd(h, W, t, 2.0)
    pv = rng.permutation(40)
    inv = np.argsort(pv)
    n2, _ = oracle_mod.fwd(h, W[pv], inv[t], 2.0)
    assert np.allclose(n2, nll, atol=1e-12)
    pr = rng.permutation(12)
    n3, _ = oracle_mod.fwd(h[pr], W, t[pr], 2.0)
    assert np.allclose(n3, nll[pr], atol=1e-12)


# ---- bits per byte --------------------------------------------------------

def test_bpb_uniform_and_mask(oracle_mod):
    """Uniform logits: bpb = (number of scored rows) log2 V / (their bytes),
    and masked rows drop out of both sums."""
    V, N = 1024, 100
    nll = np.full(N, math.log(V))
    nbytes = (np.arange(N) % 8 + 1).astype(np.int32)
    mask = (np.arange(N) % 4 == 0).astype(np.uint8)
    b, sn, sb, n = oracle_mod.bpb(nll, nbytes, mask)
    assert n == 25 and sb == int(nbytes[mask == 1].sum())
    assert b == pytest.approx(25 * math.log2(V) / sb, rel=1e-14)
    b0, *_ = oracle_mod.bpb(nll, nbytes, np.zeros(N, np.uint8))
    assert math.isnan(b0)


# ---- backward: finite differences and invariants ---------------------------

def _loss(oracle_mod, h, W, t, c, w, mask=None):
    nll, _ = oracle_mod.fwd(h, W, t, c, mask=mask)
    return w * nll.sum()


def test_gradients_match_finite_differences(oracle_mod):
    """Central differences (step 1e-5) of L = w * sum nll on N=3, V=7, d=5,
    c=2 with |z| ~ c so the cap is active: pins the analytic dh and dW (a
    dropped (1 - tanh^2) factor, a sign or a transposed product fails)."""
    rng = np.random.default_rng(5)
    N, V, d, c, w = 3, 7, 5, 2.0, 0.37
    h, W, t = _rand_case(rng, N, V, d, zscale=3.0, c=c)
    _, lse = oracle_mod.fwd(h, W, t, c)
    dh, dW = oracle_mod.bwd(h, W, t, c, lse, w)
    eps = 1e-5
    fd_h = np.zeros_like(h)
    for idx in np.ndindex(*h.shape):
        hp = h.copy(); hp[idx] += eps
        hm = h.copy(); hm[idx] -= eps
        fd_h[idx] = (_loss(oracle_mod, hp, W, t, c, w) - _loss(oracle_mod, hm, W, t, c, w)) / (2 * eps)
    fd_W = np.zeros_like(W)
    for idx in np.ndindex(*W.shape):
        Wp = W.copy(); Wp[idx] += eps
        Wm = W.copy(); Wm[idx] -= eps
        fd_W[idx] = (_loss(oracle_mod, h, Wp, t, c, w) - _loss(oracle_mod, h, Wm, t, c, w)) / (2 * eps)
    assert np.abs(dh - fd_h).max() <= 1e-8 * max(1.0, np.abs(fd_h).max())
    assert np.abs(dW - fd_W).max() <= 1e-8 * max(1.0, np.abs(fd_W).max())
    assert np.abs(fd_h).max() > 1e-2 and np.abs(fd_W).max() > 1e-2


def test_gradients_match_torch_autograd(oracle_mod):
    """A larger case against torch autograd of the same loss in fp64, with
    masked rows (independent differentiation of the definition)."""
    rng = np.random.default_rng(6)
    N, V, d, c, w = 17, 33, 12, 3.0, 1.0 / 13
    h, W, t = _rand_case(rng, N, V, d, zscale=5.0, c=c)
    mask = (rng.random(N) > 0.25).astype(np.uint8)
    _, lse = oracle_mod.fwd(h, W, t, c, mask=mask)
    dh, dW = oracle_mod.bwd(h, W, t, c, lse, w, mask=mask)
    th = torch.from_numpy(h).requires_grad_(True)
    tW = torch.from_numpy(W).requires_grad_(True)
    s = c * torch.tanh((th @ tW.T) / c)
    nll = torch.nn.functional.cross_entropy(s, torch.from_numpy(t), reduction="none")
    (w * (nll * torch.from_numpy(mask).double()).sum()).backward()
    assert np.allclose(dh, th.grad.numpy(), rtol=0, atol=1e-12)
    assert np.allclose(dW, tW.grad.numpy(), rtol=0, atol=1e-12)
    assert np.all(dh[mask == 0] == 0)


def test_gradient_inner_product_identity(oracle_mod):
    """<dh, h> = <dW, W>: both equal sum_ij dz_ij z_ij."""
    inp = si.make_inputs(2, N=64, V=200, d=64, w_scale=30.0)
    _, lse = oracle_mod.fwd(inp["h"], inp["W"], inp["tgt"], 30.0)
    dh, dW = oracle_mod.bwd(inp["h"], inp["W"], inp["tgt"], 30.0, lse, 1.0 / 64)
    h = oracle_mod.widen_bf16(inp["h"]); W = oracle_mod.widen_bf16(inp["W"])
    a, b = float((dh * h).sum()), float((dW * W).sum())
    assert a == pytest.approx(b, rel=1e-10)


def test_zero_hidden_gradient_closed_form(oracle_mod):
    """h = 0: p is uniform 1/V and tanh' = 1, so dh_i = w (mean_j W_j -
    W_{t_i}) and dW = 0."""
    inp = si.make_inputs(2, N=8, V=64, d=64)
    h = np.zeros((8, 64))
    W = oracle_mod.widen_bf16(inp["W"])
    _, lse = oracle_mod.fwd(h, W, inp["tgt"], 30.0)
    dh, dW = oracle_mod.bwd(h, W, inp["tgt"], 30.0, lse, 0.5)
    ref = 0.5 * (W.mean(axis=0)[None, :] - W[inp["tgt"]])
    assert np.allclose(dh, ref, rtol=0, atol=1e-15)
    assert np.all(dW == 0)


def test_dh_rows_matches_full(oracle_mod):
    inp = si.make_inputs(2, N=24, V=80, d=64, w_scale=20.0)
    _, lse = oracle_mod.fwd(inp["h"], inp["W"], inp["tgt"], 30.0)
    dh, _ = oracle_mod.bwd(inp["h"], inp["W"], inp["tgt"], 30.0, lse, 0.25, want_dW=False)
    rows = np.array([3, 0, 23])
    got = oracle_mod.dh_rows(inp["h"], inp["W"], inp["tgt"], 30.0, rows, lse[rows], 0.25)
    assert np.array_equal(got, dh[rows])


# ---- stored fixtures -------------------------------------------------------

def test_golden_fixtures(oracle_mod):
    """tests/golden/oracle_small.json was written by tests/golden/
    make_golden.py (which calls only the oracle); re-running the oracle
    must reproduce it, so an accidental change of the oracle shows up."""
    with open(os.path.join(GOLDEN, "oracle_small.json")) as f:
        g = json.load(f)
    for case in g["cases"]:
        inp = si.make_inputs(case["cfg"], N=case["N"], V=case["V"], d=case["d"],
                             w_scale=case["w_scale"])
        nll, lse = oracle_mod.fwd(inp["h"], inp["W"], inp["tgt"], case["softcap"])
        assert np.allclose(nll, case["nll"], rtol=0, atol=1e-12)
        b, *_ = oracle_mod.bpb(nll, inp["nbytes"])
        assert b == pytest.approx(case["bpb"], rel=1e-13)


# ---- tied table gradient through the input embedding ----------------------

def test_embed_bwd_permutation_places_rows(oracle_mod):
    """Ids forming a permutation put every gradient row, unchanged, in its
    token's row (catches indexing by position instead of by id)."""
    rng = np.random.default_rng(11)
    V, d = 37, 8
    ids = rng.permutation(V)
    g = rng.standard_normal((V, d))
    out = oracle_mod.embed_bwd(ids, g, V)
    assert np.array_equal(out[ids], g)


def test_embed_bwd_single_id_closed_form(oracle_mod):
    """All N rows on one id, row i = i * e_k: that token's row is
    N (N - 1) / 2 at component k and 0 elsewhere; every other row is 0
    (catches a dropped first or last row)."""
    N, V, d, k, v = 101, 5, 6, 2, 3
    g = np.zeros((N, d))
    g[:, k] = np.arange(N)
    out = oracle_mod.embed_bwd(np.full(N, v), g, V)
    want = np.zeros((V, d))
    want[v, k] = N * (N - 1) / 2
    assert np.array_equal(out, want)


def test_embed_bwd_invariants(oracle_mod):
    """Integer-valued rows (sums exact in fp64): reordering rows together
    with their ids changes nothing, the total over the table equals the total
    over the rows, and tokens that never occur get zero rows (catches rows
    added to the wrong token or lost)."""
    rng = np.random.default_rng(12)
    N, V, d = 500, 40, 16
    ids = si.zipf_ids(rng, N, V - 5, 1.1)  # the last 5 ids never occur
    g = rng.integers(-50, 51, size=(N, d)).astype(np.float64)
    out = oracle_mod.embed_bwd(ids, g, V)
    perm = rng.permutation(N)
    assert np.array_equal(oracle_mod.embed_bwd(ids[perm], g[perm], V), out)
    assert np.array_equal(out.sum(axis=0), g.sum(axis=0))
    assert np.all(out[V - 5:] == 0)
    counts = np.bincount(ids, minlength=V)
    assert np.array_equal(out[:, 0] != 0, (out[:, 0] != 0) & (counts > 0))


def test_embed_bwd_rejects_out_of_range_id(oracle_mod):
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.embed_bwd(np.array([0, 3]), np.ones((2, 4)), 3)
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.embed_bwd(np.array([-1]), np.ones((1, 4)), 3)


# ---- dW on listed vocabulary rows ------------------------------------------

@pytest.mark.parametrize("c", [30.0, 2.0, 0.0])
def test_dW_rows_matches_full(oracle_mod, c):
    """The per-row dW (for full-size sampled checks) equals the rows of the
    full backward, which finite differences pin; rows listed out of order
    and repeated, first and last included, with masked rows (catches a wrong
    vocabulary row, a dropped mask or a transposed product)."""
    inp = si.make_inputs(2, N=40, V=90, d=64, w_scale=20.0)
    mask = (np.arange(40) % 7 != 3).astype(np.uint8)
    _, lse = oracle_mod.fwd(inp["h"], inp["W"], inp["tgt"], c, mask=mask)
    _, dW = oracle_mod.bwd(inp["h"], inp["W"], inp["tgt"], c, lse, 0.3, mask=mask, want_dh=False)
    vrows = np.array([89, 0, 17, int(inp["tgt"][5]), 17])
    got = oracle_mod.dW_rows(inp["h"], inp["W"], inp["tgt"], c, lse, 0.3, vrows, mask=mask)
    assert np.allclose(got, dW[vrows], rtol=0, atol=1e-15)


# ---- no cap (softcap 0) ----------------------------------------------------

def test_uncapped_matches_torch_cross_entropy(oracle_mod):
    """softcap = 0 means no cap: nll equals torch's fp64 cross_entropy of the
    plain logits, and dh, dW equal torch autograd of that loss (catches a cap
    left in, or a (1 - tanh^2) factor left in the gradient)."""
    rng = np.random.default_rng(21)
    N, V, d, w = 13, 29, 10, 0.21
    h, W, t = _rand_case(rng, N, V, d, zscale=30.0, c=0.0)
    nll, lse = oracle_mod.fwd(h, W, t, 0.0)
    th = torch.from_numpy(h).requires_grad_(True)
    tW = torch.from_numpy(W).requires_grad_(True)
    ref = torch.nn.functional.cross_entropy(th @ tW.T, torch.from_numpy(t), reduction="none")
    assert np.allclose(nll, ref.detach().numpy(), rtol=0, atol=1e-11)
    assert ref.detach().numpy().max() > 20.0  # logits far beyond any cap of ~c = 30
    (w * ref.sum()).backward()
    dh, dW = oracle_mod.bwd(h, W, t, 0.0, lse, w)
    assert np.allclose(dh, th.grad.numpy(), rtol=0, atol=1e-11)
    assert np.allclose(dW, tW.grad.numpy(), rtol=0, atol=1e-11)
    rows = np.array([4, 0])
    assert np.allclose(oracle_mod.dh_rows(h, W, t, 0.0, rows, lse[rows], w), dh[rows], rtol=0, atol=1e-15)


# ---- bits per byte with per-id byte lengths ----------------------------------

def test_bpb_lut_closed_forms(oracle_mod):
    """A uniform table of b bytes gives sum nll / (ln 2 * b * n); with the
    table materialised per row (bytes_i = lut[t_i]) it equals the per-row
    bpb; masked rows count nothing (catches a table indexed by position
    instead of by target, or a mask ignored)."""
    rng = np.random.default_rng(22)
    N, V = 300, 50
    nll = rng.random(N) * 5
    t = rng.integers(0, V, N)
    mask = (rng.random(N) > 0.3).astype(np.uint8)
    b, sn, sb, n = oracle_mod.bpb_lut(nll, t, np.full(V, 3, np.int32), mask)
    M = int(mask.sum())
    assert (sb, n) == (3 * M, M)
    assert sn == pytest.approx(float(nll[mask == 1].sum()), rel=1e-15)
    assert b == pytest.approx(sn / (math.log(2) * 3 * M), rel=1e-15)
    lut = rng.integers(1, 13, V).astype(np.int32)
    b1 = oracle_mod.bpb_lut(nll, t, lut, mask)
    b2 = oracle_mod.bpb(nll, lut[t], mask)
    assert b1 == b2
    # zero logits: nll = ln V on every row, so bpb = n log2 V / sum lut[t]
    b3, *_ = oracle_mod.bpb_lut(np.full(N, math.log(V)), t, lut)
    assert b3 == pytest.approx(N * math.log2(V) / float(lut[t].sum()), rel=1e-13)
    with pytest.raises(oracle_mod.OracleError):
        oracle_mod.bpb_lut(nll, np.where(np.arange(N) == 7, V, t), lut)


# ---- more storage formats of the tied table ------------------------------------

def _all_finite_f16():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = bits.view(np.float16)
    return bits[np.isfinite(f)]


def test_dequant_int8_rows_brute_force(oracle_mod):
    """Every int8 code (-128..127) times every finite fp16 scale, bit-equal
    to torch: the fp32 product is exact (at most 7 + 11 significant bits),
    then torch's float -> bfloat16 is the one RNE rounding (catches a double
    rounding through bf16 scales, a sign or an unsigned byte read)."""
    sc = _all_finite_f16()
    q = np.arange(-128, 128, dtype=np.int8)
    V = sc.size
    Q = np.tile(q, (V, 1))
    got = oracle_mod.dequant_int8_rows(Q, sc)
    ref = (torch.from_numpy(Q.astype(np.float32))
           * torch.from_numpy(sc.view(np.float16).astype(np.float32))[:, None]).to(torch.bfloat16)
    assert np.array_equal(got, ref.view(torch.int16).numpy().view(np.uint16))


def test_dequant_int4_asym_brute_force(oracle_mod):
    """Every unsigned code and zero point (16 x 16) times every finite fp16
    scale, bit-equal to torch's (q - z) * s rounded once to bf16 (catches
    nibble order, a signed read of unsigned codes, or a zero point applied
    after the scale)."""
    sc = _all_finite_f16()
    d, group = 256, 256
    qs = np.arange(16)
    q_all, z_all = np.meshgrid(qs, qs, indexing="ij")
    q_row = q_all.reshape(-1)            # 256 codes along d
    z_vals = np.arange(16, dtype=np.uint8)
    V = sc.size * 16
    Q = np.tile(q_row, (V, 1))
    Wq = (Q[:, 0::2] | (Q[:, 1::2] << 4)).astype(np.uint8)
    scales = np.repeat(sc, 16)[:, None]
    zeros = np.tile(z_vals, sc.size)[:, None]
    got = oracle_mod.dequant_int4_asym(Wq, scales, zeros, d, group)
    ref = (torch.from_numpy((Q - zeros.astype(np.int64)).astype(np.float32))
           * torch.from_numpy(scales.view(np.float16).astype(np.float32))).to(torch.bfloat16)
    assert np.array_equal(got, ref.view(torch.int16).numpy().view(np.uint16))


def test_dequant_f16_all_patterns(oracle_mod):
    """All 65,536 fp16 patterns: bit-equal to torch's float16 -> bfloat16 for
    every non-NaN pattern, NaN stays NaN (catches truncation instead of RNE,
    lost subnormals or signs)."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle_mod.dequant_f16(bits)
    ref = torch.from_numpy(bits.view(np.float16)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(bits.view(np.float16))
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all(np.isnan(si.bf16_bits_to_f32(got[nan])))


# ---- RMSNorm in front of the head ---------------------------------------------

def test_rmsnorm_fwd_matches_torch_and_closed_forms(oracle_mod):
    """Against torch's fp64 rms_norm with a gain (an independent routine);
    a constant row a gives g * a / sqrt(a^2 + eps); with eps = 0 the output
    does not depend on the row's scale (catches a mean taken as a sum, eps
    outside the root, or the gain dropped)."""
    rng = np.random.default_rng(23)
    N, d, eps = 9, 24, 1e-6
    x = rng.standard_normal((N, d)) * 3
    g = rng.standard_normal(d)
    h, rinv = oracle_mod.rmsnorm_fwd(x, g, eps)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (d,), torch.from_numpy(g), eps)
    assert np.allclose(h, ref.numpy(), rtol=0, atol=1e-13)
    assert np.allclose(rinv, 1 / np.sqrt((x * x).mean(axis=1) + eps), rtol=1e-15)
    a = -0.7
    hc, _ = oracle_mod.rmsnorm_fwd(np.full((1, d), a), g, 0.01)
    assert np.allclose(hc[0], g * a / math.sqrt(a * a + 0.01), rtol=1e-15)
    h1, _ = oracle_mod.rmsnorm_fwd(x, None, 0.0)
    h2, _ = oracle_mod.rmsnorm_fwd(x * 37.5, None, 0.0)
    assert np.allclose(h1, h2, rtol=0, atol=1e-14)


def test_rmsnorm_bwd_finite_differences(oracle_mod):
    """Central differences (step 1e-6) of L = sum(R * rmsnorm(x; g)) for a
    fixed random R pin dx and dg; with no gain and eps = 0 every dx row is
    orthogonal to its x row (the output is scale-free) (catches a dropped
    r^3 term, a wrong sign or dg summed without the 1/r factor)."""
    rng = np.random.default_rng(24)
    N, d, eps = 3, 5, 1e-3
    x = rng.standard_normal((N, d))
    g = rng.standard_normal(d)
    R = rng.standard_normal((N, d))
    dx, dg = oracle_mod.rmsnorm_bwd(x, g, eps, R)

    def L(xx, gg):
        return float((R * oracle_mod.rmsnorm_fwd(xx, gg, eps)[0]).sum())

    step = 1e-6
    fd_x = np.zeros_like(x)
    for idx in np.ndindex(*x.shape):
        xp = x.copy(); xp[idx] += step
        xm = x.copy(); xm[idx] -= step
        fd_x[idx] = (L(xp, g) - L(xm, g)) / (2 * step)
    fd_g = np.zeros_like(g)
    for k in range(d):
        gp = g.copy(); gp[k] += step
        gm = g.copy(); gm[k] -= step
        fd_g[k] = (L(x, gp) - L(x, gm)) / (2 * step)
    assert np.abs(dx - fd_x).max() <= 1e-8 * max(1.0, np.abs(fd_x).max())
    assert np.abs(dg - fd_g).max() <= 1e-8 * max(1.0, np.abs(fd_g).max())
    dx0, _ = oracle_mod.rmsnorm_bwd(x, None, 0.0, R)
    assert np.abs((dx0 * x).sum(axis=1)).max() <= 1e-13


# ---- stored full-size fixtures ------------------------------------------------

def test_full_size_golden_reproduces(oracle_mod):
    """tests/golden/full_size.json (written by make_golden.py --full from the
    oracle only): re-running the oracle reproduces the forward + backward
    batch's sums and two of its dW rows, and two chunks of the evaluation
    stream, so an accidental change of the oracle shows up on CPU."""
    with open(os.path.join(GOLDEN, "full_size.json")) as f:
        g = json.load(f)
    e = g["cfg2"]
    inp = si.make_inputs(2)
    nll, lse = oracle_mod.fwd(inp["h"], inp["W"], inp["tgt"], e["softcap"])
    b, sn, sb, n = oracle_mod.bpb(nll, inp["nbytes"])
    assert (sb, n) == (e["sum_bytes"], e["n_scored"])
    assert sn == pytest.approx(e["sum_nll"], rel=1e-12) and b == pytest.approx(e["bpb"], rel=1e-12)
    sel = [0, 7]
    rows = oracle_mod.dW_rows(inp["h"], inp["W"], inp["tgt"], e["softcap"], lse, e["grad_scale"],
                              np.array([e["vrows"][i] for i in sel]))
    assert np.allclose(rows, np.array([e["dW_rows"][i] for i in sel]), rtol=1e-9, atol=1e-15)
    st = g["cfg4_stream"]
    for c in (st["chunks"][0], st["chunks"][-1]):
        ch = si.make_stream_chunk(c["k"])
        sel = np.nonzero(ch["mask"])[0]
        nll, _ = oracle_mod.fwd(ch["h"], ch["W"], ch["tgt"], st["softcap"], rows=sel)
        _, sn, sb, n = oracle_mod.bpb(nll, ch["nbytes"][sel])
        assert (sb, n) == (c["sum_bytes"], c["n_scored"])
        assert sn == pytest.approx(c["sum_nll"], rel=1e-12)
