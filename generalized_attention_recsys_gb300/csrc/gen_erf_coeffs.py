"""Generates the erf / erfc coefficients used by act.cuh for GELU (run by hand).

GELU(z) = z * Phi(z), Phi(z) = erfc(-z / sqrt2) / 2.

Forward (16-bit P): two evaluations of Phi, mixed per column so that the FMA
and MUFU pipes share the work (act.cuh):

  * polynomial (FMA pipe only): erf(X v) ~ v * p(v^2) with v = x / X clamped
    to [-1, 1], p of degree 5, X chosen by scanning; the fit covers x in
    [0, 7] with the clamp applied, so the tail beyond X is part of the
    minimax error. Lawson's algorithm (iteratively reweighted least squares
    converging to the minimax fit) on a dense grid.
  * tanh form (one MUFU tanh per score): Phi(z) ~ (1 + tanh(a z + b z^3)) / 2.
    a and b are fitted to atanh(2 Phi - 1) with weights dPhi/dy = 2 Phi (1 - Phi),
    i.e. a linearised minimax fit of Phi itself (Lawson again), on |z| <= 6.

The report gives each fit's max |Phi error| in float64.

FastGELU forward with e4m3 P: its own tanh factor fitted the same way as
the erf polynomial: tanh(sqrt(2/pi) (z + 0.044715 z^3)) ~ v t(v^2) with
v = z / Z clamped to [-1, 1], t of degree 5, Z scanned, minimax over
z in [0, 10] with the clamp applied (|Phi error| is half the tanh error).

Backward (MUFU rcp + ex2): for x >= 0 the form of Abramowitz & Stegun,
Handbook of Mathematical Functions, 7.1.25 (Hastings' approximation):

    erfc(x) ~ t (b0 + b1 t + b2 t^2) exp(-x^2),   t = 1 / (1 + p x),

and Phi(z) = 1 - erfc(|z| / sqrt2) / 2 for z >= 0, erfc(|z| / sqrt2) / 2 for
z < 0. The reciprocal and the exponential run on the MUFU pipe, leaving about
ten FMA-pipe operations per element; exp(-z^2 / 2) is also the normal pdf
(up to 1/sqrt(2 pi)) that the GELU derivative needs.

The coefficients here are fitted afresh, not copied from the handbook: for each
p on a grid, b0..b2 minimise the maximum absolute error of erfc on [0, 9]
(Lawson's algorithm: iteratively reweighted least squares converging to the
minimax fit), and the best p is kept. The report gives that error and the
error of a float32 evaluation in the kernels' operation order:
max |erfc error| about 2e-5, so |Phi error| <= 1e-5.

    python gen_erf_coeffs.py
"""

from math import erf, erfc

import numpy as np

N_TERMS = 3
X_MAX = 9.0
POLY_TERMS = 6


def fit_poly(x_clamp: float, n: int, iters: int = 300) -> tuple[np.ndarray, float]:
    """erf(x) ~ v p(v^2), v = min(x / x_clamp, 1), minimax over x in [0, 7]; returns (p, max |erf error|)."""
    x = np.linspace(0.0, 7.0, 30001)
    y = np.array([erf(t) for t in x])
    v = np.minimum(x / x_clamp, 1.0)
    u = v * v
    basis = np.stack([v * u ** i for i in range(n)], axis=1)
    w = np.ones_like(x)
    for _ in range(iters):
        c, *_ = np.linalg.lstsq(basis * np.sqrt(w)[:, None], y * np.sqrt(w), rcond=None)
        err = np.abs(basis @ c - y)
        w = w * (err / err.max() + 1e-4)
        w /= w.mean()
    return c, float(np.abs(basis @ c - y).max())


def best_poly(n: int) -> tuple[float, np.ndarray, float]:
    best = None
    for xc in np.arange(2.0, 3.2, 0.05):
        c, e = fit_poly(float(xc), n, 150)
        if best is None or e < best[2]:
            best = (float(xc), c, e)
    c, e = fit_poly(best[0], n)
    return best[0], c, e


def fit_fast_gelu_poly(z_clamp: float, n: int, iters: int = 300) -> tuple[np.ndarray, float]:
    """tanh(u(z)) ~ v t(v^2), v = min(z / z_clamp, 1), minimax over z in [0, 10]; returns (t, max |tanh error|)."""
    z = np.linspace(0.0, 10.0, 40001)
    y = np.tanh(np.sqrt(2.0 / np.pi) * (z + 0.044715 * z ** 3))
    v = np.minimum(z / z_clamp, 1.0)
    u = v * v
    basis = np.stack([v * u ** i for i in range(n)], axis=1)
    w = np.ones_like(z)
    for _ in range(iters):
        c, *_ = np.linalg.lstsq(basis * np.sqrt(w)[:, None], y * np.sqrt(w), rcond=None)
        err = np.abs(basis @ c - y)
        w = w * (err / err.max() + 1e-4)
        w /= w.mean()
    return c, float(np.abs(basis @ c - y).max())


def best_fast_gelu_poly(n: int) -> tuple[float, np.ndarray, float]:
    best = None
    for zc in np.arange(2.8, 4.2, 0.05):
        c, e = fit_fast_gelu_poly(float(zc), n, 150)
        if best is None or e < best[2]:
            best = (float(zc), c, e)
    c, e = fit_fast_gelu_poly(best[0], n)
    return best[0], c, e


def fit_tanh_form(iters: int = 300) -> tuple[np.ndarray, float]:
    """Phi(z) ~ (1 + tanh(a z + b z^3)) / 2: returns ((a, b), max |Phi error|)."""
    z = np.linspace(1e-3, 6.0, 20001)
    phi = np.array([0.5 * erfc(-t / np.sqrt(2.0)) for t in z])
    y = np.arctanh(2.0 * phi - 1.0)
    dphi = 2.0 * phi * (1.0 - phi)  # dPhi / dy
    basis = np.stack([z, z ** 3], axis=1) * dphi[:, None]
    target = y * dphi
    w = np.ones_like(z)
    for _ in range(iters):
        c, *_ = np.linalg.lstsq(basis * np.sqrt(w)[:, None], target * np.sqrt(w), rcond=None)
        err = np.abs(basis @ c - target)
        w = w * (err / err.max() + 1e-4)
        w /= w.mean()
    zz = np.linspace(-12.0, 12.0, 240001)
    ref = np.array([0.5 * erfc(-t / np.sqrt(2.0)) for t in zz])
    approx = 0.5 * (1.0 + np.tanh(zz * (c[0] + c[1] * zz * zz)))
    return c, float(np.abs(approx - ref).max())


def fit(p: float, n: int, iters: int = 300) -> tuple[np.ndarray, float]:
    x = np.linspace(0.0, X_MAX, 40001)
    y = np.array([erfc(v) for v in x])
    t = 1.0 / (1.0 + p * x)
    basis = np.stack([t ** (i + 1) * np.exp(-x * x) for i in range(n)], axis=1)
    w = np.ones_like(x)
    for _ in range(iters):
        c, *_ = np.linalg.lstsq(basis * np.sqrt(w)[:, None], y * np.sqrt(w), rcond=None)
        err = np.abs(basis @ c - y)
        w = w * (err / err.max() + 1e-6)
        w /= w.mean()
    return c, float(np.abs(basis @ c - y).max())


def best_fit(n: int) -> tuple[float, np.ndarray, float]:
    best = None
    for p in np.linspace(0.30, 0.70, 81):
        c, e = fit(p, n, 120)
        if best is None or e < best[2]:
            best = (p, c, e)
    p0 = best[0]
    for p in np.linspace(p0 - 0.005, p0 + 0.005, 21):
        c, e = fit(p, n)
        if e < best[2]:
            best = (p, c, e)
    return best


def fp32_phi_error(p: float, c: np.ndarray) -> float:
    """Max |Phi error| of the kernels' float32 operation order (exact rcp/exp2 stand-ins)."""
    f = np.float32
    z = np.linspace(-12.0, 12.0, 480001).astype(np.float32)
    d = (np.abs(z) * f(p / np.sqrt(2.0)) + f(1.0)).astype(np.float32)
    t = (f(1.0) / d).astype(np.float32)
    h = [f(ci / 2.0) for ci in c]
    q = (t * ((t * h[2] + h[1]) * t + h[0])).astype(np.float32)
    w = ((z * f(-0.5 / np.log(2.0))) * z).astype(np.float32)
    e = np.exp2(w.astype(np.float64)).astype(np.float32)
    hh = (q * e).astype(np.float32)
    phi = np.where(z >= 0, f(1.0) - hh, hh).astype(np.float64)
    ref = np.array([0.5 * erfc(-float(v) / np.sqrt(2.0)) for v in z])
    return float(np.abs(phi - ref).max())


if __name__ == "__main__":
    xc, cp, ep = best_poly(POLY_TERMS)
    print(f"// erf(x) ~ v p(v^2), v = clamp(x / {xc:.2f}, -1, 1): max |erf error| {ep:.2e}, |Phi error| {ep / 2:.2e}")
    print(f"constexpr float kGeluPolyX = {float(np.float32(xc))!r}f;")
    for i, ci in enumerate(cp):
        print(f"//   p[{i}] = {float(np.float32(ci))!r}f")
    ct, et = fit_tanh_form()
    zc, cf, ef = best_fast_gelu_poly(POLY_TERMS)
    print(f"// FastGELU tanh factor ~ v t(v^2), v = clamp(z / {zc:.2f}, -1, 1): max |tanh error| {ef:.2e}, "
          f"|Phi error| {ef / 2:.2e}")
    print(f"constexpr float kFastGeluPolyZ = {float(np.float32(zc))!r}f;")
    for i, ci in enumerate(cf):
        print(f"//   t[{i}] = {float(np.float32(ci))!r}f")
    print(f"// Phi(z) ~ (1 + tanh(a z + b z^3)) / 2: max |Phi error| {et:.2e}")
    print(f"constexpr float kPhiTanhA = {float(np.float32(ct[0]))!r}f;")
    print(f"constexpr float kPhiTanhB = {float(np.float32(ct[1]))!r}f;")
    p, c, e = best_fit(N_TERMS)
    print(f"// p = {p!r}; max |erfc error| {e:.2e}; float32 max |Phi error| {fp32_phi_error(p, c):.2e}")
    print(f"constexpr float kErfcP = {float(np.float32(p))!r}f;")
    for i, ci in enumerate(c):
        print(f"constexpr float kErfcB{i} = {float(np.float32(ci))!r}f;")
