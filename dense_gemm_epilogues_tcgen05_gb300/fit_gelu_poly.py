"""Coefficients of the two normal-CDF forms the fused erf-GELU epilogue uses for
16-bit outputs (csrc/epilogue.cuh): a polynomial for F16 outputs
(gelu_erf_poly2) and a tanh form for BF16 outputs (gelu_erf_tanh2).

GELU(z) = z * Phi(z), Phi the standard normal CDF.  On |z| <= ZMAX,

    Phi(z) - 1/2  ~=  z * P(z^2),     P(s) = c0 + c1 s + ... + c6 s^6,

and z is clamped to +-ZMAX beyond (Phi(4) = 1 - 3.2e-5).  The coefficients are
a near-minimax fit of the absolute error in Phi: a least-squares fit in the
Chebyshev basis of s/ZMAX^2 on Chebyshev nodes, reweighted towards the points
of largest error (iteratively reweighted least squares), then expanded into
the monomial basis of s.  The script prints the coefficients as float32
literals and the largest error of the float32 Horner evaluation (with the
clamp) over z in [-12, 12] against scipy's erf.

The tanh form is Phi(z) ~ 1/2 + tanh(z (t1 + t3 z^2)) / 2 (odd in z, saturating,
so no clamp); t1 and t3 minimise the largest absolute error in Phi (Nelder-Mead
on the maximum over a dense grid, started from the tanh-GELU's constants).  Its
error printed here is with an exact tanh; the kernel's hardware tanh adds at
most half its relative error (about 2^-11) to Phi.  Run:

    python dense_gemm_epilogues_tcgen05_gb300/fit_gelu_poly.py
"""
from __future__ import annotations

import numpy as np
from numpy.polynomial import chebyshev as C
from numpy.polynomial import polynomial as P
from scipy.special import erf

ZMAX = 4.0
DEGREE = 6


def fit(degree: int = DEGREE, zmax: float = ZMAX, nodes: int = 4000, rounds: int = 80):
    """Coefficients c0..c_degree (float64) of P in s = z^2."""
    x = np.cos(np.pi * (np.arange(nodes) + 0.5) / nodes)      # Chebyshev nodes on [-1, 1]
    s = (x + 1.0) * 0.5 * zmax * zmax                           # s in [0, zmax^2]
    z = np.sqrt(s)
    target = 0.5 * erf(z / np.sqrt(2.0))                        # Phi(z) - 1/2
    u = 2.0 * s / (zmax * zmax) - 1.0                           # s mapped to [-1, 1]
    V = C.chebvander(u, degree) * z[:, None]                    # columns: z * T_k(u)
    w = np.ones(nodes)
    for _ in range(rounds):
        coef, *_ = np.linalg.lstsq(V * w[:, None], target * w, rcond=None)
        err = V @ coef - target
        w *= 1.0 + 4.0 * np.abs(err) / np.abs(err).max()
        w /= w.mean()
    # T_k(u) with u = a s + b  ->  monomials in s
    a, b = 2.0 / (zmax * zmax), -1.0
    mono_u = C.cheb2poly(coef)                                   # coefficients in u
    out = np.zeros(degree + 1)
    for k, ck in enumerate(mono_u):
        out[:k + 1] += ck * P.polypow([b, a], k)                 # (b + a s)^k
    return out


def evaluate_f32(c: np.ndarray, z: np.ndarray, zmax: float = ZMAX) -> np.ndarray:
    """Phi(z) - 1/2 as the kernel computes it: float32 clamp, square and Horner."""
    cf = c.astype(np.float32)
    zc = np.clip(z.astype(np.float32), np.float32(-zmax), np.float32(zmax))
    s = (zc * zc).astype(np.float32)
    p = np.full_like(s, cf[-1])
    for k in range(len(cf) - 2, -1, -1):
        p = (p * s + cf[k]).astype(np.float32)
    return (zc * p).astype(np.float32)


def max_error(c: np.ndarray) -> float:
    z = np.linspace(-12.0, 12.0, 2_400_001)
    return float(np.abs(evaluate_f32(c, z).astype(np.float64) - 0.5 * erf(z / np.sqrt(2.0))).max())


def tanh_phi_f32(t: np.ndarray, z: np.ndarray) -> np.ndarray:
    """Phi(z) - 1/2 of the tanh form as the kernel computes its argument (float32), exact tanh."""
    tf = t.astype(np.float32)
    zf = z.astype(np.float32)
    u = (zf * (tf[1] * (zf * zf) + tf[0]).astype(np.float32)).astype(np.float32)
    return 0.5 * np.tanh(u.astype(np.float64))


def fit_tanh():
    """(t1, t3) of the tanh form, minimax in the absolute error of Phi."""
    from scipy.optimize import minimize
    z = np.linspace(0.0, 10.0, 200_001)
    target = 0.5 * erf(z / np.sqrt(2.0))
    worst = lambda t: float(np.abs(0.5 * np.tanh(z * (t[0] + t[1] * z * z)) - target).max())
    start = np.array([np.sqrt(2.0 / np.pi), 0.044715 * np.sqrt(2.0 / np.pi)])
    r = minimize(worst, start, method="Nelder-Mead", options={"xatol": 1e-12, "fatol": 1e-12, "maxiter": 20000})
    return r.x


def tanh_max_error(t: np.ndarray) -> float:
    z = np.linspace(-12.0, 12.0, 2_400_001)
    return float(np.abs(tanh_phi_f32(t, z) - 0.5 * erf(z / np.sqrt(2.0))).max())


def main():
    c = fit()
    for k, ck in enumerate(c):
        print(f"c{k} = {float(np.float32(ck))!r:>24}f   // {ck:.17e}")
    print(f"max |Phi error| over z in [-12, 12] (float32 evaluation): {max_error(c):.3e}")
    t = fit_tanh()
    for name, tk in zip(("t1", "t3"), t):
        print(f"{name} = {float(np.float32(tk))!r:>24}f   // {tk:.17e}")
    print(f"tanh form: max |Phi error| over z in [-12, 12] (float32 argument, exact tanh): {tanh_max_error(t):.3e}")


if __name__ == "__main__":
    main()
