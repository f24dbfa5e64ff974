"""Seeded synthetic inputs shaped like the Parameter Golf head workloads.

This module is shared by the tests, the benchmark and the smoke check, and
it feeds both the CUDA library and the CPU oracle.  It holds no arithmetic
of the method itself (no logits, softcap, softmax, loss or gradient): only
random draws, the bf16 / fp16 input encodings and the harness-side int4
quantiser that produces the quantised head the library then dequantises.

Workload shapes follow the pages' models: d = 512, vocab 1024 ("parameter-
golf README", leaderboard row "Naive Baseline": 9 layers, 512 dim, 1024
vocab, tied embeddings) or vocab 8192 with sequences of 2048 ("HYDRA Golf"
site, "HEAD I Core GPT": 11 layers, 512d, seq 2048, vocab 8192 BPE).  The
real FineWeb tokens, tokenizer and trained weights are not used: every
tensor here is drawn from a seeded numpy PCG64 stream.

Recipe (seed = 1000 + config id unless given; four child streams spawned in
the fixed order h, W, targets, bytes):

===  ======================================================================
cfg  contents
===  ======================================================================
1    N=4096, V=1024.  h ~ N(0,1) drawn in fp32, RNE-rounded to bf16;
     W ~ N(0, 0.02^2) -> bf16; targets uniform in [0, V); bytes U{1..8}.
2    N=16384, V=8192.  h = RMSNorm(N(0,1) row) (no gain, eps 1e-6) -> bf16;
     W as cfg 1; targets Zipf(1.1) over ids; bytes U{1..12}.
3    N=65536, V=8192.  As cfg 2.
4    sliding-window eval: windows of 2048 rows, only the last 64 rows of
     each window scored (row mask); h, W, targets as cfg 2; bytes U{1..12}.
     A chunk holds 32 windows (65536 rows, 2048 scored).
5    N=65536, V=8192, as cfg 3 plus the head quantised to symmetric int4
     per group of 64 along d with fp16 scales (round to nearest, ties even).
===  ======================================================================
"""
from __future__ import annotations

import numpy as np

D_MODEL = 512
SOFTCAP = 30.0
WINDOW = 2048
STRIDE = 64
INT4_GROUP = 64

CONFIGS = {
    1: dict(N=4096, V=1024, h="normal", targets="uniform", bytes_hi=8),
    2: dict(N=16384, V=8192, h="rmsnorm", targets="zipf", bytes_hi=12),
    3: dict(N=65536, V=8192, h="rmsnorm", targets="zipf", bytes_hi=12),
    4: dict(N=65536, V=8192, h="rmsnorm", targets="zipf", bytes_hi=12, windows=True),
    5: dict(N=65536, V=8192, h="rmsnorm", targets="zipf", bytes_hi=12, int4=True),
}


def f32_to_bf16_bits(x) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); uint16 bits."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    rounded = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    out = rounded.astype(np.uint16)
    nan = np.isnan(x)
    if nan.any():
        out[nan] = 0x7FC0
    return out


def bf16_bits_to_f32(b) -> np.ndarray:
    b = np.ascontiguousarray(b, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


def zipf_ids(rng: np.random.Generator, n: int, V: int, s: float = 1.1) -> np.ndarray:
    """P(id = k-1) proportional to k^-s for k = 1..V, by inverse CDF."""
    k = np.arange(1, V + 1, dtype=np.float64)
    p = k ** (-s)
    cdf = np.cumsum(p)
    cdf /= cdf[-1]
    u = rng.random(n)
    ids = np.searchsorted(cdf, u, side="right")
    return np.minimum(ids, V - 1).astype(np.int64)


def window_mask(N: int, window: int = WINDOW, stride: int = STRIDE) -> np.ndarray:
    """1 on the last `stride` rows of every `window`-row window, else 0."""
    m = np.zeros(N, dtype=np.uint8)
    r = np.arange(N) % window
    m[r >= window - stride] = 1
    return m


def quantize_int4_rtn(W_bf16_bits: np.ndarray, group: int = INT4_GROUP):
    """Harness-side symmetric per-group int4 quantiser (input generation only).

    scale = fp16(max|w| / 7) per group of `group` along d;
    q = clamp(round_half_even(w / scale), -7, 7) (0 where scale == 0).
    Packed as two's-complement nibbles: element 2m in the low nibble of byte
    m, element 2m+1 in the high nibble.  Returns (Wq [V, d/2] uint8,
    scales [V, d/group] uint16 fp16 bits).
    """
    W = bf16_bits_to_f32(W_bf16_bits).astype(np.float64)
    V, d = W.shape
    g = W.reshape(V, d // group, group)
    amax = np.abs(g).max(axis=2)
    scale16 = (amax / 7.0).astype(np.float16)
    sc = scale16.astype(np.float64)[:, :, None]
    with np.errstate(divide="ignore", invalid="ignore"):
        q = np.where(sc > 0, np.rint(g / np.where(sc > 0, sc, 1.0)), 0.0)
    q = np.clip(q, -7, 7).astype(np.int64).reshape(V, d)
    nib = (q & 0xF).astype(np.uint8)
    Wq = (nib[:, 0::2] | (nib[:, 1::2] << 4)).astype(np.uint8)
    return Wq, scale16.view(np.uint16).copy()


def quantize_int4_asym(W_bf16_bits: np.ndarray, group: int = INT4_GROUP):
    """Harness-side asymmetric per-group int4 quantiser (input generation
    only): per group scale = fp16((max - min) / 15) and an integer zero point
    z = clamp(round(-min / scale), 0, 15); q = clamp(round(w / scale) + z, 0,
    15), unsigned nibbles (element 2m in the low nibble of byte m).  Returns
    (Wq [V, d/2] uint8, scales [V, d/group] fp16 bits, zeros [V, d/group] uint8)."""
    W = bf16_bits_to_f32(W_bf16_bits).astype(np.float64)
    V, d = W.shape
    g = W.reshape(V, d // group, group)
    lo, hi = g.min(axis=2), g.max(axis=2)
    scale16 = ((hi - lo) / 15.0).astype(np.float16)
    sc = scale16.astype(np.float64)
    safe = np.where(sc > 0, sc, 1.0)
    zero = np.clip(np.rint(-lo / safe), 0, 15)
    q = np.clip(np.rint(g / safe[:, :, None]) + zero[:, :, None], 0, 15)
    q = np.where(sc[:, :, None] > 0, q, zero[:, :, None]).astype(np.int64).reshape(V, d)
    Wq = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    return Wq, scale16.view(np.uint16).copy(), zero.astype(np.uint8)


def quantize_int8_rows(W_bf16_bits: np.ndarray, qmax: int = 127):
    """Harness-side per-row int8 quantiser (qmax = 63 gives int7 values in the
    same int8 storage): scale = fp16(max|w_row| / qmax), q = clamp(round(w /
    scale), -qmax, qmax).  Returns (q [V, d] int8, scales [V] fp16 bits)."""
    W = bf16_bits_to_f32(W_bf16_bits).astype(np.float64)
    amax = np.abs(W).max(axis=1)
    scale16 = (amax / qmax).astype(np.float16)
    sc = scale16.astype(np.float64)
    q = np.where(sc[:, None] > 0, np.rint(W / np.where(sc > 0, sc, 1.0)[:, None]), 0.0)
    return np.clip(q, -qmax, qmax).astype(np.int8), scale16.view(np.uint16).copy()


def to_fp16_bits(W_bf16_bits: np.ndarray) -> np.ndarray:
    """The table stored as fp16 (round to nearest even from the bf16 values)."""
    return bf16_bits_to_f32(W_bf16_bits).astype(np.float16).view(np.uint16).copy()


def make_inputs(cfg: int, seed: int | None = None, N: int | None = None,
                V: int | None = None, d: int = D_MODEL, w_scale: float = 1.0,
                h_scale: float = 1.0) -> dict:
    """Seeded inputs for config `cfg`; N, V, d may be shrunk for small tests.

    Returns a dict of numpy arrays: h (uint16 bf16 bits [N, d]), W (uint16
    [V, d]), tgt (int64 [N]), nbytes (int32 [N]), mask (uint8 [N] or None),
    and for cfg 5 Wq (uint8 [V, d/2]) and scales (uint16 fp16 [V, d/64]).
    w_scale / h_scale multiply the drawn values before rounding (W x 100
    drives the softcap into saturation).
    """
    spec = CONFIGS[cfg]
    N = spec["N"] if N is None else int(N)
    V = spec["V"] if V is None else int(V)
    seed = 1000 + cfg if seed is None else int(seed)
    rng_h, rng_w, rng_t, rng_b = [np.random.Generator(np.random.PCG64(s))
                                  for s in np.random.SeedSequence(seed).spawn(4)]
    x = rng_h.standard_normal((N, d), dtype=np.float32)
    if spec["h"] == "rmsnorm":
        x64 = x.astype(np.float64)
        x = (x64 / np.sqrt(np.mean(x64 * x64, axis=1, keepdims=True) + 1e-6)).astype(np.float32)
    if h_scale != 1.0:
        x = (x * np.float32(h_scale)).astype(np.float32)
    w = rng_w.standard_normal((V, d), dtype=np.float32) * np.float32(0.02 * w_scale)
    if spec["targets"] == "uniform":
        tgt = rng_t.integers(0, V, size=N, dtype=np.int64)
    else:
        tgt = zipf_ids(rng_t, N, V, 1.1)
    nbytes = rng_b.integers(1, spec["bytes_hi"] + 1, size=N, dtype=np.int64).astype(np.int32)
    out = dict(cfg=cfg, seed=seed, N=N, V=V, d=d, softcap=SOFTCAP,
               h=f32_to_bf16_bits(x), W=f32_to_bf16_bits(w), tgt=tgt,
               nbytes=nbytes, mask=None)
    if spec.get("windows"):
        out["mask"] = window_mask(N)
    if spec.get("int4"):
        out["Wq"], out["scales"] = quantize_int4_rtn(out["W"], INT4_GROUP)
    return out


STREAM_CHUNK_WINDOWS = 32  # a chunk of the evaluation stream: 32 windows, 65,536 rows, 2,048 scored


def stream_chunk_seed(k: int) -> int:
    """Seed of chunk k of the sliding-window evaluation stream (cfg 4)."""
    return 1004 + 1_000_003 * (int(k) + 1)


def make_stream_chunk(k: int, windows: int = STREAM_CHUNK_WINDOWS) -> dict:
    """Chunk k of the sliding-window evaluation stream: `windows` windows of
    2048 rows, the last 64 of each scored (row mask), drawn as cfg 4 with the
    chunk's own seed.  Same keys as make_inputs."""
    return make_inputs(4, seed=stream_chunk_seed(k), N=windows * WINDOW)


def make_byte_lut(V: int, seed: int = 3001, hi: int = 12) -> np.ndarray:
    """A synthetic per-id byte-length table (int32 [V], uniform in 1..hi).
    The real table comes from the tokenizer, which is not available; the
    lengths follow the configs' per-token byte counts (U{1..12})."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return rng.integers(1, hi + 1, size=V, dtype=np.int64).astype(np.int32)


def make_embed_inputs(N: int = 65536, V: int = 8192, d: int = D_MODEL, seed: int = 2001,
                      g_scale: float = 1e-2) -> dict:
    """Seeded inputs of the tied table's input-embedding gradient: the
    positions' token ids (Zipf(1.1) over the vocabulary, like the targets)
    and the loss gradient with respect to each position's embedding row
    (N(0, g_scale^2), rounded to bf16).  Returns ids (int64 [N]) and g
    (uint16 bf16 bits [N, d])."""
    rng_i, rng_g = [np.random.Generator(np.random.PCG64(s)) for s in np.random.SeedSequence(seed).spawn(2)]
    ids = zipf_ids(rng_i, N, V, 1.1)
    g = rng_g.standard_normal((N, d), dtype=np.float32) * np.float32(g_scale)
    return dict(ids=ids, g=f32_to_bf16_bits(g), N=N, V=V, d=d)
