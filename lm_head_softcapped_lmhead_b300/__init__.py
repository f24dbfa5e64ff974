"""Python binding of the liblmhead_ce C ABI (``include/lmhead_ce.h``).

Fused tied-LM-head + tanh-softcapped cross-entropy for B300 (sm_103a):
forward (nll, lse), backward (dh, dW), an int4 per-group head, and the
bits-per-byte reduction.  Every step runs in the library's CUDA kernels; this
module only marshals torch tensors (device memory, streams) into the C calls.
It never falls back to another implementation: if the shared library is
missing, importing the functions raises.

Function names match the C entry points.  Tensors are CUDA tensors:
h [N, d] bf16 (row stride may exceed d), W [V, d] bf16, tgt [N] int64,
row_mask [N] uint8 or None, nll / lse [N] fp32, dh like h, dW [V, d] fp32,
ws a uint8 workspace from :func:`workspace`.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "liblmhead_ce.so")

LMCE_OK, LMCE_EINVAL, LMCE_ENOTSUP, LMCE_ECUDA, LMCE_EDATA, LMCE_ETIMEOUT = range(6)
LMCE_WS_MASKED = 1
LMCE_WS_INT4 = 2
LMCE_WS_EMBED = 4
LMCE_WS_QHEAD = 2
LMCE_WS_RMSNORM = 8
LMCE_QHEAD_INT4, LMCE_QHEAD_INT4_ASYM, LMCE_QHEAD_INT8_ROW, LMCE_QHEAD_FP16 = 1, 2, 3, 4

EXPORTS = (
    "lmce_workspace_bytes", "lmce_workspace_init", "lmce_softcap_max", "lmhead_ce_fwd", "lmhead_ce_bwd",
    "lmhead_ce_fwd_int4", "lmhead_ce_bwd_int4", "bpb_reduce", "lmce_bpb", "lmhead_int4_dequant",
    "lmce_status", "lmce_last_cuda_error", "lmce_strerror", "lmce_launch_count", "lmhead_ce_fwd_noalloc",
    "lmhead_ce_fwd_bwd", "lmhead_ce_fwd_bwd_int4", "lmhead_tied_embed_bwd", "lmhead_ce_fwd_q", "lmhead_ce_bwd_q",
    "lmhead_ce_fwd_bwd_q", "lmhead_qhead_dequant", "lmhead_rmsnorm_fwd", "lmhead_rmsnorm_bwd",
    "lmhead_ce_fwd_rmsnorm", "lmhead_ce_fwd_bwd_rmsnorm", "bpb_reduce_lut", "lmce_wait_selftest",
    "lmhead_ce_fwd_int4_inkernel",
)

_lib = None


class LmceError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = f"{where}: {strerror(code)} (code {code})"
        if code == LMCE_ECUDA:
            msg += f": {last_cuda_error()}"
        super().__init__(msg)


class _QHead(ctypes.Structure):
    _fields_ = [("format", ctypes.c_int), ("group", ctypes.c_int), ("codes", ctypes.c_void_p),
                ("scales", ctypes.c_void_p), ("zeros", ctypes.c_void_p)]


class _BpbAcc(ctypes.Structure):
    _fields_ = [("sum_nll", ctypes.c_double), ("sum_bytes", ctypes.c_longlong),
                ("n_scored", ctypes.c_longlong)]


def lib():
    """The loaded liblmhead_ce.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m lm_head_softcapped_lmhead_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        P, I64, F, I, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int, ctypes.c_size_t
        sig = {
            "lmce_workspace_bytes": ([I64, I64, I64, ctypes.c_uint], SZ),
            "lmce_workspace_init": ([P, SZ, P], I),
            "lmce_softcap_max": ([I64], F),
            "lmhead_ce_fwd": ([P, I64, P, I64, I64, I64, P, P, F, P, P, P, SZ, P], I),
            "lmhead_ce_bwd": ([P, I64, P, I64, I64, I64, P, P, F, P, P, F, P, P, I, P, SZ, P], I),
            "lmhead_ce_fwd_bwd": ([P, I64, P, I64, I64, I64, P, P, F, F, P, P, P, P, I, P, SZ, P], I),
            "lmhead_ce_fwd_int4": ([P, I64, P, P, I, I64, I64, I64, P, P, F, P, P, P, SZ, P], I),
            "lmhead_ce_bwd_int4": ([P, I64, P, P, I, I64, I64, I64, P, P, F, P, P, F, P, P, SZ, P], I),
            "lmhead_ce_fwd_bwd_int4": ([P, I64, P, P, I, I64, I64, I64, P, P, F, F, P, P, P, P, SZ, P], I),
            "bpb_reduce": ([P, P, P, I64, P, P, SZ, P], I),
            "lmhead_tied_embed_bwd": ([P, P, I64, I64, I64, I64, P, P, SZ, P], I),
            "lmce_bpb": ([ctypes.POINTER(_BpbAcc), ctypes.POINTER(ctypes.c_double)], I),
            "lmhead_int4_dequant": ([P, P, I64, I64, I, P, P], I),
            "lmce_status": ([P, P, ctypes.POINTER(ctypes.c_int)], I),
            "lmce_last_cuda_error": ([], ctypes.c_char_p),
            "lmce_strerror": ([I], ctypes.c_char_p),
            "lmce_launch_count": ([], ctypes.c_ulonglong),
            "lmhead_ce_fwd_q": ([P, I64, ctypes.POINTER(_QHead), I64, I64, I64, P, P, F, P, P, P, SZ, P], I),
            "lmhead_ce_bwd_q": ([P, I64, ctypes.POINTER(_QHead), I64, I64, I64, P, P, F, P, P, F, P, P, SZ, P], I),
            "lmhead_ce_fwd_bwd_q": ([P, I64, ctypes.POINTER(_QHead), I64, I64, I64, P, P, F, F, P, P, P, P, SZ, P],
                                    I),
            "lmhead_qhead_dequant": ([ctypes.POINTER(_QHead), I64, I64, P, P], I),
            "lmhead_rmsnorm_fwd": ([P, I64, P, F, I64, I64, P, I64, P, P], I),
            "lmhead_rmsnorm_bwd": ([P, I64, P, P, P, I64, I64, I64, P, I64, P, I, P, SZ, P], I),
            "lmhead_ce_fwd_rmsnorm": ([P, I64, P, F, P, I64, I64, I64, P, P, F, P, P, P, SZ, P], I),
            "lmhead_ce_fwd_bwd_rmsnorm": ([P, I64, P, F, P, I64, I64, I64, P, P, F, F, P, P, P, I64, P, P, I, P, SZ,
                                           P], I),
            "bpb_reduce_lut": ([P, P, P, I64, P, I64, P, P, SZ, P], I),
            "lmce_wait_selftest": ([ctypes.c_longlong, I, P, SZ, P], I),
            "lmhead_ce_fwd_int4_inkernel": ([P, I64, P, P, I, I64, I64, I64, P, P, F, P, P, P, SZ, P], I),
        }
        for name, (args, res) in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def strerror(code: int) -> str:
    return lib().lmce_strerror(int(code)).decode()


def last_cuda_error() -> str:
    return lib().lmce_last_cuda_error().decode()


def lmce_launch_count() -> int:
    """Kernels enqueued by the library so far in this process."""
    return int(lib().lmce_launch_count())


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(rc: int, where: str):
    if rc != LMCE_OK:
        raise LmceError(rc, where)


def _bf16_bits(t, name):
    if t.dtype not in (torch.bfloat16, torch.int16, torch.uint16):
        raise TypeError(f"{name} must be bfloat16 (got {t.dtype})")
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be 2-D with unit stride along d")


def lmce_workspace_bytes(N: int, V: int, d: int, flags: int = 0) -> int:
    return int(lib().lmce_workspace_bytes(N, V, d, flags))


def lmce_softcap_max(V: int) -> float:
    return float(lib().lmce_softcap_max(V))


def workspace(N: int, V: int, d: int, flags: int = 0, device="cuda") -> torch.Tensor:
    """A zero-filled workspace of lmce_workspace_bytes(N, V, d, flags) bytes."""
    return torch.zeros(lmce_workspace_bytes(N, V, d, flags), dtype=torch.uint8, device=device)


def lmce_workspace_init(ws, stream=None):
    _check(lib().lmce_workspace_init(_p(ws), ws.numel(), _stream(stream)), "lmce_workspace_init")


def lmhead_ce_fwd(h, W, tgt, softcap, nll, lse=None, row_mask=None, ws=None, stream=None):
    _bf16_bits(h, "h")
    _bf16_bits(W, "W")
    N, d = h.shape
    V = W.shape[0]
    rc = lib().lmhead_ce_fwd(_p(h), h.stride(0), _p(W), N, V, d, _p(tgt), _p(row_mask), float(softcap),
                             _p(nll), _p(lse), _p(ws), ws.numel(), _stream(stream))
    _check(rc, "lmhead_ce_fwd")


def lmhead_ce_bwd(h, W, tgt, softcap, lse, grad_scale, dh=None, dW=None, accumulate_dW=False, row_mask=None,
                  ws=None, stream=None, nll=None):
    _bf16_bits(h, "h")
    _bf16_bits(W, "W")
    N, d = h.shape
    V = W.shape[0]
    if dh is not None and dh.stride(0) != h.stride(0):
        raise ValueError("dh must have the same row stride as h")
    rc = lib().lmhead_ce_bwd(_p(h), h.stride(0), _p(W), N, V, d, _p(tgt), _p(row_mask), float(softcap), _p(lse),
                             _p(nll), float(grad_scale), _p(dh), _p(dW), int(bool(accumulate_dW)), _p(ws),
                             ws.numel(), _stream(stream))
    _check(rc, "lmhead_ce_bwd")


def lmhead_ce_fwd_bwd(h, W, tgt, softcap, grad_scale, nll, lse, dh=None, dW=None, accumulate_dW=False,
                      row_mask=None, ws=None, stream=None):
    _bf16_bits(h, "h")
    _bf16_bits(W, "W")
    N, d = h.shape
    V = W.shape[0]
    if dh is not None and dh.stride(0) != h.stride(0):
        raise ValueError("dh must have the same row stride as h")
    rc = lib().lmhead_ce_fwd_bwd(_p(h), h.stride(0), _p(W), N, V, d, _p(tgt), _p(row_mask), float(softcap),
                                 float(grad_scale), _p(nll), _p(lse), _p(dh), _p(dW), int(bool(accumulate_dW)),
                                 _p(ws), ws.numel(), _stream(stream))
    _check(rc, "lmhead_ce_fwd_bwd")


def lmhead_ce_fwd_int4(h, Wq, scales, group, softcap, tgt, nll, lse=None, row_mask=None, ws=None, stream=None):
    _bf16_bits(h, "h")
    N, d = h.shape
    V = Wq.shape[0]
    rc = lib().lmhead_ce_fwd_int4(_p(h), h.stride(0), _p(Wq), _p(scales), int(group), N, V, d, _p(tgt),
                                  _p(row_mask), float(softcap), _p(nll), _p(lse), _p(ws), ws.numel(),
                                  _stream(stream))
    _check(rc, "lmhead_ce_fwd_int4")


def lmhead_ce_fwd_int4_inkernel(h, Wq, scales, group, softcap, tgt, nll, lse=None, row_mask=None, ws=None,
                                stream=None):
    """lmhead_ce_fwd_int4 with the dequantisation inside the forward kernel."""
    _bf16_bits(h, "h")
    N, d = h.shape
    V = Wq.shape[0]
    rc = lib().lmhead_ce_fwd_int4_inkernel(_p(h), h.stride(0), _p(Wq), _p(scales), int(group), N, V, d, _p(tgt),
                                           _p(row_mask), float(softcap), _p(nll), _p(lse), _p(ws), ws.numel(),
                                           _stream(stream))
    _check(rc, "lmhead_ce_fwd_int4_inkernel")


def lmhead_ce_bwd_int4(h, Wq, scales, group, softcap, tgt, lse, grad_scale, dh, row_mask=None, ws=None,
                       stream=None, nll=None):
    _bf16_bits(h, "h")
    N, d = h.shape
    V = Wq.shape[0]
    if dh.stride(0) != h.stride(0):
        raise ValueError("dh must have the same row stride as h")
    rc = lib().lmhead_ce_bwd_int4(_p(h), h.stride(0), _p(Wq), _p(scales), int(group), N, V, d, _p(tgt),
                                  _p(row_mask), float(softcap), _p(lse), _p(nll), float(grad_scale), _p(dh),
                                  _p(ws), ws.numel(), _stream(stream))
    _check(rc, "lmhead_ce_bwd_int4")


def lmhead_ce_fwd_bwd_int4(h, Wq, scales, group, softcap, tgt, grad_scale, nll, lse, dh, row_mask=None, ws=None,
                           stream=None):
    _bf16_bits(h, "h")
    N, d = h.shape
    V = Wq.shape[0]
    if dh.stride(0) != h.stride(0):
        raise ValueError("dh must have the same row stride as h")
    rc = lib().lmhead_ce_fwd_bwd_int4(_p(h), h.stride(0), _p(Wq), _p(scales), int(group), N, V, d, _p(tgt),
                                      _p(row_mask), float(softcap), float(grad_scale), _p(nll), _p(lse), _p(dh),
                                      _p(ws), ws.numel(), _stream(stream))
    _check(rc, "lmhead_ce_fwd_bwd_int4")


def lmhead_tied_embed_bwd(ids, g, dW, ws=None, stream=None):
    """dW[ids[i]] += g[i] for every row i (the tied table's gradient through
    the input embedding).  ids [N] int64, g [N, d] bf16, dW [V, d] fp32."""
    _bf16_bits(g, "g")
    N, d = g.shape
    V = dW.shape[0]
    if dW.dtype != torch.float32 or dW.dim() != 2 or dW.shape[1] != d or not dW.is_contiguous():
        raise ValueError("dW must be a contiguous [V, d] float32 tensor")
    rc = lib().lmhead_tied_embed_bwd(_p(ids), _p(g), g.stride(0), N, V, d, _p(dW), _p(ws), ws.numel(),
                                     _stream(stream))
    _check(rc, "lmhead_tied_embed_bwd")


def bpb_acc(device="cuda") -> torch.Tensor:
    """A zeroed device accumulator (24 bytes) for bpb_reduce."""
    return torch.zeros(3, dtype=torch.float64, device=device)


def bpb_reduce(nll, nbytes, acc, row_mask=None, ws=None, stream=None):
    N = nll.numel()
    rc = lib().bpb_reduce(_p(nll), _p(nbytes), _p(row_mask), N, _p(acc), _p(ws), ws.numel(), _stream(stream))
    _check(rc, "bpb_reduce")


def read_bpb_acc(acc) -> tuple:
    """(sum_nll, sum_bytes, n_scored) from a device accumulator."""
    raw = acc.detach().cpu().contiguous()
    a = _BpbAcc.from_buffer_copy(raw.numpy().tobytes())
    return a.sum_nll, a.sum_bytes, a.n_scored


def lmce_bpb(acc) -> float:
    """bits per byte from a device accumulator (host helper of the ABI)."""
    sn, sb, n = read_bpb_acc(acc)
    a = _BpbAcc(sn, sb, n)
    out = ctypes.c_double()
    _check(lib().lmce_bpb(ctypes.byref(a), ctypes.byref(out)), "lmce_bpb")
    return out.value


def lmhead_int4_dequant(Wq, scales, d, group, out, stream=None):
    V = Wq.shape[0]
    rc = lib().lmhead_int4_dequant(_p(Wq), _p(scales), V, d, int(group), _p(out), _stream(stream))
    _check(rc, "lmhead_int4_dequant")


def lmce_status(ws, stream=None) -> int:
    """Synchronises the stream; returns and clears the device status code."""
    code = ctypes.c_int()
    _check(lib().lmce_status(_p(ws), _stream(stream), ctypes.byref(code)), "lmce_status")
    return code.value


# ---- quantised / fp16 heads ----------------------------------------------------
def qhead(fmt, codes, scales=None, zeros=None, group=64):
    """A head description for the *_q calls: fmt one of LMCE_QHEAD_*, codes /
    scales / zeros CUDA tensors (see include/lmhead_ce.h).  Keep the tensors
    alive while the calls that use it run."""
    return _QHead(int(fmt), int(group), codes.data_ptr(), None if scales is None else scales.data_ptr(),
                  None if zeros is None else zeros.data_ptr())


def lmhead_qhead_dequant(head, V, d, out, stream=None):
    _check(lib().lmhead_qhead_dequant(ctypes.byref(head), V, d, _p(out), _stream(stream)), "lmhead_qhead_dequant")


def lmhead_ce_fwd_q(h, head, V, softcap, tgt, nll, lse=None, row_mask=None, ws=None, stream=None):
    _bf16_bits(h, "h")
    N, d = h.shape
    rc = lib().lmhead_ce_fwd_q(_p(h), h.stride(0), ctypes.byref(head), N, V, d, _p(tgt), _p(row_mask),
                               float(softcap), _p(nll), _p(lse), _p(ws), ws.numel(), _stream(stream))
    _check(rc, "lmhead_ce_fwd_q")


def lmhead_ce_bwd_q(h, head, V, softcap, tgt, lse, grad_scale, dh, row_mask=None, ws=None, stream=None, nll=None):
    _bf16_bits(h, "h")
    N, d = h.shape
    if dh.stride(0) != h.stride(0):
        raise ValueError("dh must have the same row stride as h")
    rc = lib().lmhead_ce_bwd_q(_p(h), h.stride(0), ctypes.byref(head), N, V, d, _p(tgt), _p(row_mask),
                               float(softcap), _p(lse), _p(nll), float(grad_scale), _p(dh), _p(ws), ws.numel(),
                               _stream(stream))
    _check(rc, "lmhead_ce_bwd_q")


def lmhead_ce_fwd_bwd_q(h, head, V, softcap, tgt, grad_scale, nll, lse, dh, row_mask=None, ws=None, stream=None):
    _bf16_bits(h, "h")
    N, d = h.shape
    if dh.stride(0) != h.stride(0):
        raise ValueError("dh must have the same row stride as h")
    rc = lib().lmhead_ce_fwd_bwd_q(_p(h), h.stride(0), ctypes.byref(head), N, V, d, _p(tgt), _p(row_mask),
                                   float(softcap), float(grad_scale), _p(nll), _p(lse), _p(dh), _p(ws), ws.numel(),
                                   _stream(stream))
    _check(rc, "lmhead_ce_fwd_bwd_q")


# ---- RMSNorm in front of the head ------------------------------------------------
def lmhead_rmsnorm_fwd(x, g, eps, h, rinv, stream=None):
    _bf16_bits(x, "x")
    _bf16_bits(h, "h")
    N, d = x.shape
    rc = lib().lmhead_rmsnorm_fwd(_p(x), x.stride(0), _p(g), float(eps), N, d, _p(h), h.stride(0), _p(rinv),
                                  _stream(stream))
    _check(rc, "lmhead_rmsnorm_fwd")


def lmhead_rmsnorm_bwd(x, g, rinv, dh, dx, dg=None, accumulate_dg=False, ws=None, stream=None):
    _bf16_bits(x, "x")
    _bf16_bits(dh, "dh")
    _bf16_bits(dx, "dx")
    N, d = x.shape
    rc = lib().lmhead_rmsnorm_bwd(_p(x), x.stride(0), _p(g), _p(rinv), _p(dh), dh.stride(0), N, d, _p(dx),
                                  dx.stride(0), _p(dg), int(bool(accumulate_dg)), _p(ws),
                                  0 if ws is None else ws.numel(), _stream(stream))
    _check(rc, "lmhead_rmsnorm_bwd")


def lmhead_ce_fwd_rmsnorm(x, g, eps, W, tgt, softcap, nll, lse=None, row_mask=None, ws=None, stream=None):
    _bf16_bits(x, "x")
    _bf16_bits(W, "W")
    N, d = x.shape
    V = W.shape[0]
    rc = lib().lmhead_ce_fwd_rmsnorm(_p(x), x.stride(0), _p(g), float(eps), _p(W), N, V, d, _p(tgt), _p(row_mask),
                                     float(softcap), _p(nll), _p(lse), _p(ws), ws.numel(), _stream(stream))
    _check(rc, "lmhead_ce_fwd_rmsnorm")


def lmhead_ce_fwd_bwd_rmsnorm(x, g, eps, W, tgt, softcap, grad_scale, nll, lse, dx=None, dg=None, dW=None,
                              accumulate=False, row_mask=None, ws=None, stream=None):
    _bf16_bits(x, "x")
    _bf16_bits(W, "W")
    N, d = x.shape
    V = W.shape[0]
    rc = lib().lmhead_ce_fwd_bwd_rmsnorm(_p(x), x.stride(0), _p(g), float(eps), _p(W), N, V, d, _p(tgt),
                                         _p(row_mask), float(softcap), float(grad_scale), _p(nll), _p(lse), _p(dx),
                                         0 if dx is None else dx.stride(0), _p(dg), _p(dW), int(bool(accumulate)),
                                         _p(ws), ws.numel(), _stream(stream))
    _check(rc, "lmhead_ce_fwd_bwd_rmsnorm")


# ---- bits per byte with per-id byte lengths, bounded-wait self-test ----------------
def bpb_reduce_lut(nll, tgt, lut, acc, row_mask=None, ws=None, stream=None):
    N = nll.numel()
    rc = lib().bpb_reduce_lut(_p(nll), _p(tgt), _p(lut), lut.numel(), _p(row_mask), N, _p(acc), _p(ws), ws.numel(),
                              _stream(stream))
    _check(rc, "bpb_reduce_lut")


def lmce_wait_selftest(limit_cycles, arrive, ws, stream=None):
    rc = lib().lmce_wait_selftest(int(limit_cycles), int(bool(arrive)), _p(ws), ws.numel(), _stream(stream))
    _check(rc, "lmce_wait_selftest")
