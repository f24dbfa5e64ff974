"""Gradient of the tied table through the input embedding
(lmhead_tied_embed_bwd, through the C ABI) against the fp64 oracle.

Each element of the result is an fp32 sum, along a fixed tree, of the token's
bf16 rows (pieces of at most 32 rows summed in row order, groups of 16 pieces
added in order, the groups added in order, then one atomic addition into dW,
which flushes only subnormal results).  The classic bound for recursive
summation gives, per element, |gpu - exact| <= (n_v + 1) u (sum |g| + |dW0|)
with n_v the token's row count and u = 2^-24; the tests hold the GPU to that
bound, and to bit-identical repeats."""
import numpy as np
import pytest
import torch

import synth_inputs as si
from gpu_util import bf16_dev

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


@pytest.fixture(scope="module")
def lm():
    import lm_head_softcapped_lmhead_b300 as lm
    lm.lib()
    return lm


def run(lm, ids, g_bits, V, dW0, ld=None):
    N, d = g_bits.shape
    g = bf16_dev(g_bits)
    if ld is not None:
        wide = torch.zeros((N, ld), dtype=torch.bfloat16, device="cuda")
        wide[:, :d] = g
        g = wide[:, :d]
    dW = dW0.clone()
    ws = lm.workspace(N, V, d, lm.LMCE_WS_EMBED)
    lm.lmhead_tied_embed_bwd(torch.from_numpy(np.ascontiguousarray(ids)).cuda(), g, dW, ws=ws)
    return lm.lmce_status(ws), dW


def check(oracle_mod, ids, g_bits, V, dW0, dW, valid=None):
    """dW within the summation bound of dW0 + the oracle's sum."""
    if valid is not None:
        ids, g_bits = ids[valid], g_bits[valid]
    g = oracle_mod.widen_bf16(g_bits)
    ref = oracle_mod.embed_bwd(ids, g, V)
    absum = oracle_mod.embed_bwd(ids, np.abs(g), V)
    n = np.bincount(ids, minlength=V).astype(np.float64)[:, None]
    init = dW0.double().cpu().numpy()
    got = dW.double().cpu().numpy()
    bound = (n + 1) * U * (absum + np.abs(init)) * 1.001
    err = np.abs(got - (init + ref))
    assert np.all(err <= bound), float((err - bound).max())
    # Tokens that never occur keep their rows bit for bit.
    untouched = n[:, 0] == 0
    assert np.array_equal(got[untouched], init[untouched])


@pytest.mark.parametrize("N,V,d,ld", [
    (1000, 300, 64, None),     # ragged, d = 64
    (1, 5, 512, None),         # a single row
    (3000, 1, 128, None),      # one token owns every row (47 pieces)
    (777, 777, 256, None),     # every token once (a permutation below)
    (2500, 400, 192, 256),     # g with a row stride wider than d
    (30000, 20000, 64, None),  # 79 token blocks: the token scan looks back past one warp's 32 records;
                               # V above the eight-warp count walk: one warp's walk, counts in shared memory
    (20000, 50000, 64, None),  # V above the shared-memory count limit: counts in the histogram rows
])
def test_tied_embed_matches_oracle(lm, oracle_mod, N, V, d, ld):
    e = si.make_embed_inputs(N, V, d, seed=3000 + N)
    ids = e["ids"]
    if N == V:
        ids = np.random.default_rng(5).permutation(V).astype(np.int64)
    dW0 = torch.randn(V, d, device="cuda") * 1e-2
    st, dW = run(lm, ids, e["g"], V, dW0, ld=ld)
    assert st == lm.LMCE_OK
    check(oracle_mod, ids, e["g"], V, dW0, dW)


def test_tied_embed_hot_token_and_determinism(lm, oracle_mod):
    """Zipf ids over a small vocabulary (token 0 owns about a fifth of the
    rows, many pieces): within the bound, and the same bits on a repeat."""
    N, V, d = 20000, 500, 512
    e = si.make_embed_inputs(N, V, d, seed=3101)
    assert np.bincount(e["ids"])[0] > 64 * 20
    dW0 = torch.zeros(V, d, device="cuda")
    st, a = run(lm, e["ids"], e["g"], V, dW0)
    st2, b = run(lm, e["ids"], e["g"], V, dW0)
    assert st == st2 == lm.LMCE_OK
    assert torch.equal(a, b)
    check(oracle_mod, e["ids"], e["g"], V, dW0, a)


def test_tied_embed_bad_ids_are_skipped(lm, oracle_mod):
    N, V, d = 600, 50, 64
    e = si.make_embed_inputs(N, V, d, seed=3202)
    ids = e["ids"].copy()
    ids[7] = V
    ids[300] = -1
    dW0 = torch.zeros(V, d, device="cuda")
    st, dW = run(lm, ids, e["g"], V, dW0)
    assert st == lm.LMCE_EDATA
    valid = (ids >= 0) & (ids < V)
    check(oracle_mod, ids, e["g"], V, dW0, dW, valid=valid)


def test_tied_embed_training_batch_full(lm, oracle_mod):
    """The training micro-batch's input positions (N=65536, V=8192, d=512,
    Zipf ids) added to a head gradient, against the oracle on every element."""
    e = si.make_embed_inputs()
    dW0 = torch.randn(e["V"], e["d"], device="cuda") * 1e-3
    st, dW = run(lm, e["ids"], e["g"], e["V"], dW0)
    assert st == lm.LMCE_OK
    check(oracle_mod, e["ids"], e["g"], e["V"], dW0, dW)


def test_tied_embed_count_forms_agree(lm):
    """The stable sort is unique, so the three forms of the count kernel (eight
    warps with 16-bit counts for V <= 12288, one warp with counts in shared
    memory up to V = 32768, counts in the histogram rows above) give the same
    dW bits for the same ids; the extra vocabulary rows stay untouched."""
    N, V0, d = 20000, 12288, 128
    e = si.make_embed_inputs(N, V0, d, seed=3303)
    dW0 = torch.randn(V0, d, device="cuda") * 1e-2
    outs = []
    for V in (V0, V0 + 1, 40000):
        init = torch.zeros(V, d, device="cuda")
        init[:V0] = dW0
        st, dW = run(lm, e["ids"], e["g"], V, init)
        assert st == lm.LMCE_OK
        assert torch.equal(dW[V0:], init[V0:])
        outs.append(dW[:V0])
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[0], outs[2])
