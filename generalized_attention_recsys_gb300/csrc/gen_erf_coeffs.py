"""Generates the polynomial erf coefficients used by act.cuh (run by hand).

erf(X v) is approximated on v in [-1, 1] by v * p(v^2), p of degree n-1, with
X = 3 (beyond |x| = 3 the kernel uses erf = +-1; erfc(3) = 2.2e-5). The
coefficients come from Lawson's algorithm (iteratively reweighted least
squares converging to the minimax fit) on a dense grid in double precision.
The printed report includes the error of the float32 Horner evaluation that
the kernel performs: max |erf error| about 2.2e-5, i.e. |Phi error| <= 1.1e-5.

    python gen_erf_coeffs.py
"""

from math import erf

import numpy as np

X = 3.0
N_TERMS = 9


def fit(x_max: float, n: int, iters: int = 200) -> np.ndarray:
    v = np.linspace(0.0, 1.0, 20001)
    y = np.array([erf(x_max * vi) for vi in v])
    u = v * v
    basis = np.stack([v * u ** i for i in range(n)], axis=1)
    w = np.ones_like(v)
    for _ in range(iters):
        c, *_ = np.linalg.lstsq(basis * np.sqrt(w)[:, None], y * np.sqrt(w), rcond=None)
        err = np.abs(basis @ c - y)
        w = w * (err / err.max() + 1e-4)
        w /= w.mean()
    return c


def fp32_error(c: np.ndarray, x_max: float) -> float:
    v = np.linspace(-1.3, 1.3, 200001).astype(np.float32)
    vc = np.clip(v, -1, 1).astype(np.float32)
    uu = (vc * vc).astype(np.float32)
    p = np.float32(c[-1])
    for ci in c[-2::-1]:
        p = (p * uu + np.float32(ci)).astype(np.float32)
    approx = (vc * p).astype(np.float32)
    ref = np.array([erf(x_max * float(x)) for x in v])
    return float(np.abs(approx - ref).max())


if __name__ == "__main__":
    c = fit(X, N_TERMS)
    print(f"// erf({X} v) ~ v * p(v^2), |v| <= 1; float32 max |erf error| {fp32_error(c, X):.2e}")
    print("constexpr float kErfPoly[%d] = {" % N_TERMS)
    print(",\n".join(f"    {float(np.float32(ci))!r}f" for ci in c))
    print("};")
