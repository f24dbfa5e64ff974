"""fp64 CPU oracle for the softcapped LM-head cross-entropy path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s cpu_baseline / reference leg may import this package.  It
shares no code with the CUDA library: the arithmetic lives in ``oracle.c``
(plain loops in double precision), and this module only builds it with gcc
and marshals numpy arrays.

Functions and the passages they follow (page title, section):

* :func:`fwd` -- tied-head logits, tanh softcap, log-sum-exp, target NLL.
  "parameter-golf: ... Where Model Size Becomes the Game", "The Baseline Is a
  Map, Not the Destination" (loss = criterion(logits, y)); "HYDRA Golf" stack
  list and "parameter-golf README" leaderboard row "PR1736 + PolarNS + ...
  FusedCE" ("fused softcapped CE"); softcap read as s = c*tanh(z/c).
* :func:`bpb` -- bits per byte.  tproger news "OpenAI launched Parameter
  Golf", section "Rules and metric" (bits per byte on FineWeb validation,
  compression counted in bytes).
* :func:`bwd` / :func:`dh_rows` -- gradient of the (weighted) NLL sum with
  respect to the hidden states and the tied embedding ("[AGENT TASK] OpenAI
  Parameter Golf", section "Training loop": bf16 mixed-precision training).
* :func:`dequant_int4` -- per-group int4 head ("HYDRA Golf" stack list:
  "per-group compression" of int4 weights), symmetric, group 64, fp16 scales.
* :func:`dW_rows` -- the head's dW for listed vocabulary rows only (same
  definition as :func:`bwd`), for sampled checks at full size.
* :func:`bpb_lut` -- bits per byte with the byte count of each scored token
  from a per-id table ("parameter-golf README" leaderboard rows "SP8192 +
  CaseOps + ..." (byte-sidecar BPB accounting) and "CaseOps Tokenizer + ..."
  (validation byte sidecars); "HYDRA Golf" submission conditions:
  tokenizer-aware validation BPB).
* :func:`dequant_int8_rows`, :func:`dequant_int4_asym`, :func:`dequant_f16`
  -- more storage formats of the tied table ("parameter-golf README"
  leaderboard rows "Mixed Quant + Sliding Window Eval" (int8 embeddings),
  "VarLen Attention + Fused MLP + ..." (int7 embeddings), "fp16 Embed" (FP16
  tied embedding); "HYDRA Golf" stack list: "LQER asymmetric int4,
  per-group compression").
* :func:`rmsnorm_fwd` / :func:`rmsnorm_bwd` -- the normalisation in front of
  the head and its backward ("parameter-golf README" leaderboard row "11L
  Partial RoPE + LN Scale + EMA + XSA4": layerwise LN scale; RMSNorm with an
  optional gain).
* A softcap of 0 means no cap (s = z) in :func:`fwd`, :func:`bwd`,
  :func:`dh_rows` and :func:`dW_rows`.
* :func:`embed_bwd` -- the tied table's gradient through the input embedding:
  each position's embedding gradient is added to its token's row ("[AGENT
  TASK] OpenAI Parameter Golf", architecture experiments table, row "Tied
  embeddings": input/output embedding sharing; "parameter-golf README",
  leaderboard row "Naive Baseline": TiedEmbeddings).

Parity pins for every function live in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so with gcc (-O2 -fopenmp)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        # -ffp-contract=off: no fused multiply-adds, so the arithmetic is the
        # plain sequence written in the source.
        cmd = ["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
               "-std=c11", _SRC, "-o", _LIB + ".tmp", "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(_LIB + ".tmp", _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        D = ctypes.c_double
        lib.oracle_fwd_f64.argtypes = [P, P, I64, I64, I64, P, P, D, P, I64, P, P]
        lib.oracle_fwd_f64.restype = ctypes.c_int
        lib.oracle_bwd_f64.argtypes = [P, P, I64, I64, I64, P, P, D, P, D, P, P]
        lib.oracle_bwd_f64.restype = ctypes.c_int
        lib.oracle_dh_rows_f64.argtypes = [P, P, I64, I64, I64, P, P, D, P, I64, P, D, P]
        lib.oracle_dh_rows_f64.restype = ctypes.c_int
        lib.oracle_bpb.argtypes = [P, P, P, I64, P, P, P]
        lib.oracle_bpb.restype = ctypes.c_double
        lib.oracle_dequant_int4.argtypes = [P, P, I64, I64, I64, P]
        lib.oracle_dequant_int4.restype = ctypes.c_int
        lib.oracle_embed_bwd_f64.argtypes = [P, P, I64, I64, I64, P]
        lib.oracle_embed_bwd_f64.restype = ctypes.c_int
        lib.oracle_dW_rows_f64.argtypes = [P, P, I64, I64, I64, P, P, D, P, D, P, I64, P]
        lib.oracle_dW_rows_f64.restype = ctypes.c_int
        lib.oracle_bpb_lut.argtypes = [P, P, P, I64, P, I64, P, P, P, P]
        lib.oracle_bpb_lut.restype = ctypes.c_double
        lib.oracle_dequant_int8_rows.argtypes = [P, P, I64, I64, P]
        lib.oracle_dequant_int8_rows.restype = ctypes.c_int
        lib.oracle_dequant_int4_asym.argtypes = [P, P, P, I64, I64, I64, P]
        lib.oracle_dequant_int4_asym.restype = ctypes.c_int
        lib.oracle_dequant_f16.argtypes = [P, I64, P]
        lib.oracle_dequant_f16.restype = ctypes.c_int
        lib.oracle_rmsnorm_fwd_f64.argtypes = [P, P, D, I64, I64, P, P]
        lib.oracle_rmsnorm_fwd_f64.restype = ctypes.c_int
        lib.oracle_rmsnorm_bwd_f64.argtypes = [P, P, D, P, I64, I64, P, P]
        lib.oracle_rmsnorm_bwd_f64.restype = ctypes.c_int
        lib.oracle_f64_to_bf16_rne_array.argtypes = [P, P, I64]
        lib.oracle_f64_to_bf16_rne_array.restype = None
        lib.oracle_bf16_to_f64_array.argtypes = [P, P, I64]
        lib.oracle_bf16_to_f64_array.restype = None
        lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_f64.restype = ctypes.c_double
        lib.oracle_f64_to_bf16_rne.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_bf16_rne.restype = ctypes.c_uint16
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = ctypes.c_int
        _lib = lib
    return _lib


class OracleError(RuntimeError):
    pass


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def widen_bf16(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> float64, exactly."""
    bits = _c(bits, np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    _load().oracle_bf16_to_f64_array(_ptr(bits), _ptr(out), bits.size)
    return out


def f16_to_f64(bits: int) -> float:
    return float(_load().oracle_f16_to_f64(int(bits)))


def f64_to_bf16_rne(x: float) -> int:
    return int(_load().oracle_f64_to_bf16_rne(float(x)))


def round_bf16(x) -> np.ndarray:
    """float64 array -> bf16 bit patterns (uint16), round to nearest even."""
    x = _c(x, np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_f64_to_bf16_rne_array(_ptr(x), _ptr(out), x.size)
    return out


def _as_f64(x):
    """Accept float64 arrays as they are, uint16 arrays as bf16 bits."""
    if x.dtype == np.uint16:
        return widen_bf16(x)
    return _c(x, np.float64)


def fwd(h, W, tgt, softcap, mask=None, rows=None):
    """Per-row (nll, lse) in float64.  h: [N, d], W: [V, d] (float64 or bf16
    bits), tgt: [N] int64, mask: [N] uint8 or None, rows: optional index list
    (then outputs follow that list)."""
    h = _as_f64(h)
    W = _as_f64(W)
    N, d = h.shape
    V = W.shape[0]
    tgt = _c(tgt, np.int64)
    mask = _c(mask, np.uint8)
    rows = _c(rows, np.int64)
    n_out = N if rows is None else rows.size
    nll = np.zeros(n_out, dtype=np.float64)
    lse = np.zeros(n_out, dtype=np.float64)
    rc = _load().oracle_fwd_f64(_ptr(h), _ptr(W), N, V, d, _ptr(tgt), _ptr(mask),
                                float(softcap), _ptr(rows), 0 if rows is None else rows.size,
                                _ptr(nll), _ptr(lse))
    if rc != 0:
        raise OracleError(f"oracle_fwd_f64 returned {rc}")
    return nll, lse


def bwd(h, W, tgt, softcap, lse, grad_scale, mask=None, want_dh=True, want_dW=True):
    """(dh [N, d], dW [V, d]) in float64 for L = grad_scale * sum nll_i."""
    h = _as_f64(h)
    W = _as_f64(W)
    N, d = h.shape
    V = W.shape[0]
    tgt = _c(tgt, np.int64)
    mask = _c(mask, np.uint8)
    lse = _c(lse, np.float64)
    dh = np.zeros((N, d), dtype=np.float64) if want_dh else None
    dW = np.zeros((V, d), dtype=np.float64) if want_dW else None
    rc = _load().oracle_bwd_f64(_ptr(h), _ptr(W), N, V, d, _ptr(tgt), _ptr(mask),
                                float(softcap), _ptr(lse), float(grad_scale), _ptr(dh), _ptr(dW))
    if rc != 0:
        raise OracleError(f"oracle_bwd_f64 returned {rc}")
    return dh, dW


def dh_rows(h, W, tgt, softcap, rows, lse_rows, grad_scale, mask=None):
    """dh for the listed rows only, given those rows' lse."""
    h = _as_f64(h)
    W = _as_f64(W)
    N, d = h.shape
    V = W.shape[0]
    tgt = _c(tgt, np.int64)
    mask = _c(mask, np.uint8)
    rows = _c(rows, np.int64)
    lse_rows = _c(lse_rows, np.float64)
    out = np.zeros((rows.size, d), dtype=np.float64)
    rc = _load().oracle_dh_rows_f64(_ptr(h), _ptr(W), N, V, d, _ptr(tgt), _ptr(mask),
                                    float(softcap), _ptr(rows), rows.size, _ptr(lse_rows),
                                    float(grad_scale), _ptr(out))
    if rc != 0:
        raise OracleError(f"oracle_dh_rows_f64 returned {rc}")
    return out


def bpb(nll, nbytes, mask=None):
    """(bpb, sum_nll, sum_bytes, n_scored)."""
    nll = _c(nll, np.float64)
    nbytes = _c(nbytes, np.int32)
    mask = _c(mask, np.uint8)
    sn = ctypes.c_double()
    sb = ctypes.c_int64()
    n = ctypes.c_int64()
    v = _load().oracle_bpb(_ptr(nll), _ptr(nbytes), _ptr(mask), nll.size,
                           ctypes.byref(sn), ctypes.byref(sb), ctypes.byref(n))
    return float(v), float(sn.value), int(sb.value), int(n.value)


def dequant_int4(Wq, scales_f16_bits, d, group=64):
    """bf16 bits [V, d] of round_to_bf16(q * scale)."""
    Wq = _c(Wq, np.uint8)
    sc = _c(scales_f16_bits, np.uint16)
    V = Wq.shape[0]
    out = np.zeros((V, d), dtype=np.uint16)
    rc = _load().oracle_dequant_int4(_ptr(Wq), _ptr(sc), V, d, group, _ptr(out))
    if rc != 0:
        raise OracleError(f"oracle_dequant_int4 returned {rc}")
    return out


def embed_bwd(ids, g, V):
    """[V, d] float64: out[ids[i]] += g[i] for every row i, in row order, from
    zeros.  g: [N, d] float64 or bf16 bits; ids: [N] int64 in [0, V)."""
    g = _as_f64(g)
    ids = _c(ids, np.int64)
    N, d = g.shape
    out = np.zeros((V, d), dtype=np.float64)
    rc = _load().oracle_embed_bwd_f64(_ptr(ids), _ptr(g), N, V, d, _ptr(out))
    if rc != 0:
        raise OracleError(f"oracle_embed_bwd_f64 returned {rc}")
    return out


def dW_rows(h, W, tgt, softcap, lse, grad_scale, vrows, mask=None):
    """[len(vrows), d] float64: rows vrows of dW for L = grad_scale * sum nll_i
    (lse: every row's, as from :func:`fwd`)."""
    h = _as_f64(h)
    W = _as_f64(W)
    N, d = h.shape
    V = W.shape[0]
    tgt = _c(tgt, np.int64)
    mask = _c(mask, np.uint8)
    lse = _c(lse, np.float64)
    vrows = _c(vrows, np.int64)
    out = np.zeros((vrows.size, d), dtype=np.float64)
    rc = _load().oracle_dW_rows_f64(_ptr(h), _ptr(W), N, V, d, _ptr(tgt), _ptr(mask), float(softcap),
                                    _ptr(lse), float(grad_scale), _ptr(vrows), vrows.size, _ptr(out))
    if rc != 0:
        raise OracleError(f"oracle_dW_rows_f64 returned {rc}")
    return out


def bpb_lut(nll, tgt, lut, mask=None):
    """(bpb, sum_nll, sum_bytes, n_scored) with bytes_i = lut[tgt[i]]."""
    nll = _c(nll, np.float64)
    tgt = _c(tgt, np.int64)
    lut = _c(lut, np.int32)
    mask = _c(mask, np.uint8)
    sn = ctypes.c_double()
    sb = ctypes.c_int64()
    n = ctypes.c_int64()
    err = ctypes.c_int()
    v = _load().oracle_bpb_lut(_ptr(nll), _ptr(tgt), _ptr(lut), lut.size, _ptr(mask), nll.size,
                               ctypes.byref(sn), ctypes.byref(sb), ctypes.byref(n), ctypes.byref(err))
    if err.value != 0:
        raise OracleError(f"oracle_bpb_lut: error {err.value}")
    return float(v), float(sn.value), int(sb.value), int(n.value)


def dequant_int8_rows(q, scales_f16_bits):
    """bf16 bits [V, d] of round_to_bf16(q * scale_row); q int8 [V, d]."""
    q = _c(q, np.int8)
    sc = _c(scales_f16_bits, np.uint16)
    V, d = q.shape
    out = np.zeros((V, d), dtype=np.uint16)
    rc = _load().oracle_dequant_int8_rows(_ptr(q), _ptr(sc), V, d, _ptr(out))
    if rc != 0:
        raise OracleError(f"oracle_dequant_int8_rows returned {rc}")
    return out


def dequant_int4_asym(Wq, scales_f16_bits, zeros, d, group=64):
    """bf16 bits [V, d] of round_to_bf16((q - zero) * scale), unsigned codes."""
    Wq = _c(Wq, np.uint8)
    sc = _c(scales_f16_bits, np.uint16)
    zp = _c(zeros, np.uint8)
    V = Wq.shape[0]
    out = np.zeros((V, d), dtype=np.uint16)
    rc = _load().oracle_dequant_int4_asym(_ptr(Wq), _ptr(sc), _ptr(zp), V, d, group, _ptr(out))
    if rc != 0:
        raise OracleError(f"oracle_dequant_int4_asym returned {rc}")
    return out


def dequant_f16(w_f16_bits):
    """bf16 bits of round_to_bf16(w) for fp16 bits w (any shape)."""
    w = _c(w_f16_bits, np.uint16)
    out = np.zeros(w.shape, dtype=np.uint16)
    rc = _load().oracle_dequant_f16(_ptr(w), w.size, _ptr(out))
    if rc != 0:
        raise OracleError(f"oracle_dequant_f16 returned {rc}")
    return out


def rmsnorm_fwd(x, g, eps):
    """(h [N, d], rinv [N]) float64: h = g * x / sqrt(mean(x^2) + eps);
    x float64 or bf16 bits; g [d] or None (no gain)."""
    x = _as_f64(x)
    g = None if g is None else _as_f64(np.asarray(g))
    N, d = x.shape
    h = np.zeros((N, d), dtype=np.float64)
    rinv = np.zeros(N, dtype=np.float64)
    rc = _load().oracle_rmsnorm_fwd_f64(_ptr(x), _ptr(g), float(eps), N, d, _ptr(h), _ptr(rinv))
    if rc != 0:
        raise OracleError(f"oracle_rmsnorm_fwd_f64 returned {rc}")
    return h, rinv


def rmsnorm_bwd(x, g, eps, dh):
    """(dx [N, d], dg [d]) float64, given dh = dL/dh of :func:`rmsnorm_fwd`."""
    x = _as_f64(x)
    g = None if g is None else _as_f64(np.asarray(g))
    dh = _c(dh, np.float64)
    N, d = x.shape
    dx = np.zeros((N, d), dtype=np.float64)
    dg = np.zeros(d, dtype=np.float64)
    rc = _load().oracle_rmsnorm_bwd_f64(_ptr(x), _ptr(g), float(eps), _ptr(dh), N, d, _ptr(dx), _ptr(dg))
    if rc != 0:
        raise OracleError(f"oracle_rmsnorm_bwd_f64 returned {rc}")
    return dx, dg
