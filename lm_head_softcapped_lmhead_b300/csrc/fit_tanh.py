"""Derives the tanh polynomial used by the softcap in the CUDA kernels.

Method: minimax (Remez exchange) fit, in relative error, of
    g(u) = tanh(sqrt(u)) / sqrt(u)      on u in [0, XMAX^2],
by a degree-DEG polynomial P, so that tanh(x) ~= x * P(x^2) for |x| <= XMAX.
Outside that range the kernels use tanh(x) = 1 - 2 / (exp(2x) + 1).
Run:  python fit_tanh.py   (prints the coefficients written into softcap_math.cuh
and the worst relative error, in exact arithmetic and evaluated in fp32).
"""
import numpy as np

XMAX = 0.3
DEG = 3


def g(u):
    u = np.asarray(u, dtype=np.float64)
    r = np.sqrt(np.maximum(u, 1e-300))
    return np.where(u > 0, np.tanh(r) / r, 1.0)


def remez(a, b, deg, iters=40):
    n = deg + 2
    k = np.arange(n)
    u = (a + b) / 2 - (b - a) / 2 * np.cos(np.pi * k / (n - 1))
    grid = np.linspace(a, b, 400001)
    for _ in range(iters):
        A = np.zeros((n, n))
        for i in range(n):
            A[i, :deg + 1] = u[i] ** np.arange(deg + 1)
            A[i, deg + 1] = (-1) ** i * g(u[i])
        c = np.linalg.solve(A, g(u))[:deg + 1]
        err = (np.polyval(c[::-1], grid) - g(grid)) / g(grid)
        segs = np.split(np.arange(grid.size), np.where(np.diff(np.sign(err)) != 0)[0] + 1)
        ext = sorted(seg[np.argmax(np.abs(err[seg]))] for seg in segs)
        if len(ext) > n:
            ext = sorted(sorted(ext, key=lambda i: -abs(err[i]))[:n])
        if len(ext) == n:
            u = grid[ext]
    return c, float(np.abs(err).max())


def main():
    c, e = remez(0.0, XMAX * XMAX, DEG)
    c32 = c.astype(np.float32)
    x = np.linspace(-XMAX, XMAX, 200001).astype(np.float32)
    u = x * x
    p = np.float32(c32[-1])
    for ci in c32[-2::-1]:
        p = (p * u + ci).astype(np.float32)
    t = (x * p).astype(np.float32)
    ref = np.tanh(x.astype(np.float64))
    nz = np.abs(ref) > 0
    e32 = float(np.max(np.abs(t[nz] - ref[nz]) / np.abs(ref[nz])))
    print(f"XMAX={XMAX} DEG={DEG} minimax rel err={e:.3e} fp32-evaluated rel err={e32:.3e}")
    for i, ci in enumerate(c32):
        print(f"  c{i} = {float(ci)!r}f")


if __name__ == "__main__":
    main()
