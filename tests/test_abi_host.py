"""CPU-only checks of the C ABI: the library loads and exports every symbol
the header declares, and every host-detectable error is returned before any
CUDA call (these run without a GPU)."""
import ctypes
import math
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lmhead_ce.h")

OK, EINVAL, ENOTSUP, ECUDA, EDATA, ETIMEOUT = range(6)


@pytest.fixture(scope="module")
def L():
    from lm_head_softcapped_lmhead_b300 import build
    build.build()
    import lm_head_softcapped_lmhead_b300 as lm
    return lm.lib()


def header_functions():
    src = open(HEADER).read()
    return re.findall(r"^LMCE_API\s+[\w\s\*]+?\b(\w+)\s*\(", src, flags=re.M)


def test_every_declared_symbol_is_exported(L):
    names = header_functions()
    assert len(names) >= 14
    for n in names:
        assert hasattr(L, n), n
    import lm_head_softcapped_lmhead_b300 as lm
    assert set(lm.EXPORTS) == set(names)


def test_no_torch_types_in_header():
    src = open(HEADER).read()
    assert "torch" not in src.lower().replace("pytorch", "") and "at::" not in src


A = 0x10000  # a 16-byte aligned fake address: never dereferenced by these calls


def fwd(L, h=A, ldh=512, W=A, N=100, V=200, d=512, tgt=A, mask=None, c=30.0, nll=A, lse=None, ws=A,
        ws_bytes=1 << 40):
    P = ctypes.c_void_p
    return L.lmhead_ce_fwd(P(h), ldh, P(W), N, V, d, P(tgt), P(mask), c, P(nll), P(lse), P(ws), ws_bytes, None)


def test_fwd_host_validation(L):
    assert fwd(L, h=0) == EINVAL
    assert fwd(L, W=0) == EINVAL
    assert fwd(L, tgt=0) == EINVAL
    assert fwd(L, nll=0) == EINVAL
    assert fwd(L, ws=0) == EINVAL
    assert fwd(L, N=0) == EINVAL
    assert fwd(L, V=0) == EINVAL
    assert fwd(L, d=100, ldh=104) == ENOTSUP
    assert fwd(L, d=1024, ldh=1024) == ENOTSUP
    assert fwd(L, ldh=500) == EINVAL
    assert fwd(L, ldh=516) == EINVAL        # row pitch not a multiple of 16 bytes
    assert fwd(L, h=A + 2) == EINVAL        # misaligned base
    assert fwd(L, c=-1.0) == ENOTSUP        # softcap 0 means no cap; negative caps do not exist
    assert fwd(L, c=float("nan")) == ENOTSUP
    assert fwd(L, c=float("inf")) == ENOTSUP
    assert fwd(L, ws_bytes=100) == EINVAL   # workspace too small


def test_bwd_host_validation(L):
    P = ctypes.c_void_p

    def bwd(lse=A, w=1.0, dh=A, dW=A, d=512):
        return L.lmhead_ce_bwd(P(A), 512, P(A), 100, 200, d, P(A), None, 30.0, P(lse), None, w, P(dh), P(dW), 0,
                               P(A), 1 << 40, None)
    assert bwd(lse=0) == EINVAL
    assert bwd(dh=0, dW=0) == EINVAL
    assert bwd(w=float("nan")) == EINVAL
    assert bwd(dh=A + 4) == EINVAL
    assert bwd(d=96) == ENOTSUP


def test_fwd_bwd_host_validation(L):
    P = ctypes.c_void_p

    def fb(nll=A, lse=A, w=1.0, dh=A, dW=A, d=512, c=30.0, ws_bytes=1 << 40):
        return L.lmhead_ce_fwd_bwd(P(A), 512, P(A), 100, 200, d, P(A), None, c, w, P(nll), P(lse), P(dh), P(dW), 0,
                                   P(A), ws_bytes, None)
    assert fb(nll=0) == EINVAL
    assert fb(lse=0) == EINVAL               # the dW pass and the caller's backward need lse
    assert fb(w=float("inf")) == EINVAL
    assert fb(dh=A + 4) == EINVAL
    assert fb(dW=A + 8) == EINVAL
    assert fb(d=96) == ENOTSUP
    assert fb(c=-3.0) == ENOTSUP
    assert fb(ws_bytes=100) == EINVAL


def test_int4_host_validation(L):
    P = ctypes.c_void_p
    assert L.lmhead_int4_dequant(P(A), P(A), 10, 512, 10, P(A), None) == EINVAL    # group not /16
    assert L.lmhead_int4_dequant(P(A), P(A), 10, 512, 48, P(A), None) == EINVAL    # does not divide d
    assert L.lmhead_int4_dequant(P(0), P(A), 10, 512, 64, P(A), None) == EINVAL
    assert L.lmhead_int4_dequant(P(A + 3), P(A), 10, 512, 64, P(A), None) == EINVAL


def test_fwd_bwd_int4_host_validation(L):
    P = ctypes.c_void_p

    def fb(Wq=A, group=64, nll=A, lse=A, dh=A, w=1.0, d=512, c=30.0, ws_bytes=1 << 40):
        return L.lmhead_ce_fwd_bwd_int4(P(A), 512, P(Wq), P(A), group, 100, 200, d, P(A), None, c, w, P(nll),
                                        P(lse), P(dh), P(A), ws_bytes, None)
    assert fb(Wq=0) == EINVAL
    assert fb(group=48) == EINVAL            # does not divide d
    assert fb(nll=0) == EINVAL
    assert fb(lse=0) == EINVAL
    assert fb(dh=0) == EINVAL                # the int4 head is frozen: dh is the only gradient
    assert fb(dh=A + 4) == EINVAL
    assert fb(w=float("nan")) == EINVAL
    assert fb(c=-1.0) == ENOTSUP
    assert fb(ws_bytes=L.lmce_workspace_bytes(100, 200, 512, 0)) == EINVAL   # no room for the dequantised head


def test_tied_embed_host_validation(L):
    P = ctypes.c_void_p

    def eb(ids=A, g=A, ldg=512, N=100, V=200, d=512, dW=A, ws_bytes=1 << 40):
        return L.lmhead_tied_embed_bwd(P(ids), P(g), ldg, N, V, d, P(dW), P(A), ws_bytes, None)
    assert eb(ids=0) == EINVAL
    assert eb(g=0) == EINVAL
    assert eb(dW=0) == EINVAL
    assert eb(N=0) == EINVAL
    assert eb(V=0) == EINVAL
    assert eb(d=96) == ENOTSUP
    assert eb(ldg=500) == EINVAL              # below d
    assert eb(ldg=516) == EINVAL              # not a multiple of 8
    assert eb(g=A + 2) == EINVAL              # rows read as 16-byte vectors
    assert eb(dW=A + 4) == EINVAL
    assert eb(ws_bytes=L.lmce_workspace_bytes(100, 200, 512, 0)) == EINVAL  # no room for the sort
    assert L.lmce_workspace_bytes(100, 200, 512, 4) > L.lmce_workspace_bytes(100, 200, 512, 0)


def test_bpb_reduce_validation(L):
    P = ctypes.c_void_p
    assert L.bpb_reduce(P(0), P(A), None, 10, P(A), P(A), 1 << 20, None) == EINVAL
    assert L.bpb_reduce(P(A), P(A), None, 0, P(A), P(A), 1 << 20, None) == EINVAL
    assert L.bpb_reduce(P(A), P(A), None, 10, P(A), P(A), 16, None) == EINVAL


def test_host_bpb_helper(L):
    import lm_head_softcapped_lmhead_b300 as lm
    acc = lm._BpbAcc(10.0 * math.log(2.0), 5, 3)
    out = ctypes.c_double()
    assert L.lmce_bpb(ctypes.byref(acc), ctypes.byref(out)) == OK
    assert out.value == pytest.approx(2.0, rel=1e-15)
    zero = lm._BpbAcc(1.0, 0, 1)
    assert L.lmce_bpb(ctypes.byref(zero), ctypes.byref(out)) == EDATA


def test_workspace_and_softcap_bounds(L):
    import lm_head_softcapped_lmhead_b300 as lm
    a = lm.lmce_workspace_bytes(65536, 8192, 512)
    b = lm.lmce_workspace_bytes(65536, 8192, 512, lm.LMCE_WS_MASKED)
    c = lm.lmce_workspace_bytes(65536, 8192, 512, lm.LMCE_WS_INT4)
    assert 0 < a < b and a < c
    assert lm.lmce_workspace_bytes(0, 10, 64) == 0
    cm = lm.lmce_softcap_max(8192)
    # e^{-c} normal and V e^{c} finite in fp32, with margin
    assert 30.0 < cm < 88.7 - math.log(8192)
    assert math.exp(-cm) > 1.18e-38


def test_valid_call_without_gpu_fails_cleanly(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert fwd(L) == ECUDA
    assert L.lmce_last_cuda_error()


def test_strerror(L):
    for code in range(6):
        assert L.lmce_strerror(code)


def test_qhead_host_validation(L):
    """Quantised-head descriptions that fail before any launch."""
    import lm_head_softcapped_lmhead_b300 as lm
    P = ctypes.c_void_p

    def head(fmt=lm.LMCE_QHEAD_INT4, group=64, codes=A, scales=A, zeros=A):
        return lm._QHead(fmt, group, codes, scales, zeros)

    def deq(hd, V=10, d=512, out=A):
        return L.lmhead_qhead_dequant(ctypes.byref(hd), V, d, P(out), None)
    assert deq(head(fmt=7)) == EINVAL
    assert deq(head(codes=None)) == EINVAL
    assert deq(head(group=48)) == EINVAL
    assert deq(head(fmt=lm.LMCE_QHEAD_INT4_ASYM, zeros=None)) == EINVAL
    assert deq(head(fmt=lm.LMCE_QHEAD_INT8_ROW, codes=A + 8)) == EINVAL     # int8 codes: 16-byte vectors
    assert deq(head(fmt=lm.LMCE_QHEAD_INT8_ROW, scales=None)) == EINVAL
    assert deq(head(fmt=lm.LMCE_QHEAD_FP16, codes=A + 2)) == EINVAL
    assert deq(head(), d=96) == EINVAL
    assert deq(head(), out=A + 2) == EINVAL
    hd = head()
    assert L.lmhead_ce_fwd_q(P(A), 512, ctypes.byref(hd), 100, 200, 512, P(A), None, 30.0, P(0), None, P(A),
                             1 << 40, None) == EINVAL                      # nll required
    assert L.lmhead_ce_fwd_bwd_q(P(A), 512, ctypes.byref(hd), 100, 200, 512, P(A), None, 30.0, 1.0, P(A), P(A),
                                 P(0), P(A), 1 << 40, None) == EINVAL       # dh required
    assert L.lmhead_ce_bwd_q(P(A), 512, ctypes.byref(hd), 100, 200, 512, P(A), None, 30.0, P(A), None, 1.0, P(A),
                             P(A), 100, None) == EINVAL                     # workspace too small


def test_rmsnorm_host_validation(L):
    P = ctypes.c_void_p
    fwd_n = lambda x=A, ldx=512, d=512, h=A, rinv=A, eps=1e-6: L.lmhead_rmsnorm_fwd(  # noqa: E731
        P(x), ldx, None, eps, 100, d, P(h), 512, P(rinv), None)
    assert fwd_n(x=0) == EINVAL
    assert fwd_n(rinv=0) == EINVAL
    assert fwd_n(d=96, ldx=96) == ENOTSUP
    assert fwd_n(ldx=500) == EINVAL
    assert fwd_n(eps=-1.0) == EINVAL
    bwd_n = lambda dg=None, ws=A, ws_bytes=1 << 40, dx=A: L.lmhead_rmsnorm_bwd(  # noqa: E731
        P(A), 512, None, P(A), P(A), 512, 100, 512, P(dx), 512, P(dg), 0, P(ws), ws_bytes, None)
    assert bwd_n(dx=0) == EINVAL
    assert bwd_n(dg=A, ws=0) == EINVAL
    assert bwd_n(dg=A, ws_bytes=100) == EINVAL
    fb = lambda dx=A, dg=A, ws_bytes=1 << 40: L.lmhead_ce_fwd_bwd_rmsnorm(  # noqa: E731
        P(A), 512, None, 1e-6, P(A), 100, 200, 512, P(A), None, 30.0, 1.0, P(A), P(A), P(dx), 512, P(dg), P(A), 0,
        P(A), ws_bytes, None)
    assert fb(dx=0) == EINVAL                # the gain's gradient comes with dx
    assert fb(ws_bytes=100) == EINVAL


def test_bpb_lut_and_selftest_host_validation(L):
    P = ctypes.c_void_p
    lut = lambda lut_p=A, V=100, N=10: L.bpb_reduce_lut(P(A), P(A), P(lut_p), V, None, N, P(A), P(A),  # noqa: E731
                                                         1 << 20, None)
    assert lut(lut_p=0) == EINVAL
    assert lut(V=0) == EINVAL
    assert lut(N=0) == EINVAL
    assert L.lmce_wait_selftest(100, 0, P(0), 64, None) == EINVAL
    assert L.lmce_wait_selftest(-1, 0, P(A), 64, None) == EINVAL
    assert L.lmce_wait_selftest(100, 0, P(A), 8, None) == EINVAL
