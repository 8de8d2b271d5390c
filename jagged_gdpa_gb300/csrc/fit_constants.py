"""Derives the numeric constants of the device activations in act.cuh.

Run as ``python jagged_gdpa_gb300/csrc/fit_constants.py``; it prints the
values that act.cuh hard-codes (with the fit's error), so that every constant
there can be re-derived from mathematics alone:

1. GELU(x) = x * Phi(x) is approximated as x * sigmoid(a*x + b*x^3).  a and b
   minimise the maximum absolute error against the exact erf form on
   [-16, 16] (starting from the tanh-form values a = 2*sqrt(2/pi),
   b = a * 0.044715 of Hendrycks & Gimpel, "Gaussian Error Linear Units").
2. 2^f on f in [-1/2, 1/2] by a degree-DEG polynomial minimising the maximum
   relative error (Lawson's iteratively reweighted least squares on a dense
   grid, which converges to the minimax fit).
3. The integer seed K for 1/a: as_float(K - as_int(a)) minimising the maximum
   relative error over one binade (the error is periodic in the exponent).
"""

import numpy as np
from scipy.optimize import minimize
from scipy.special import erf, expit

DEG = 3


def fit_gelu_sigmoid():
    x = np.linspace(-16.0, 16.0, 400001)
    g = 0.5 * x * (1.0 + erf(x / np.sqrt(2.0)))

    def maxerr(p):
        a, b = p
        return np.max(np.abs(x * expit(a * x + b * x ** 3) - g))

    a0 = 2.0 * np.sqrt(2.0 / np.pi)
    p0 = np.array([a0, a0 * 0.044715])
    res = minimize(maxerr, p0, method="Nelder-Mead",
                   options={"xatol": 1e-10, "fatol": 1e-12, "maxiter": 4000})
    return res.x, maxerr(p0), maxerr(res.x)


def fit_exp2(deg=DEG, iters=200):
    f = np.linspace(-0.5, 0.5, 20001)
    y = np.exp2(f)
    w = np.ones_like(f)
    V = np.vander(f, deg + 1, increasing=True)
    for _ in range(iters):
        W = w / y                                   # relative error weighting
        c, *_ = np.linalg.lstsq(V * W[:, None], y * W, rcond=None)
        err = np.abs(V @ c - y) / y
        w = w * err
        w = w / w.sum()
        w = np.sqrt(w) * np.sqrt(len(w))            # Lawson update (damped)
    err = np.max(np.abs(V @ c - y) / y)
    return c, err


def fit_rcp_seed():
    a = np.linspace(1.0, 2.0, 100001, dtype=np.float64)[:-1].astype(np.float32)
    ai = a.view(np.int32).astype(np.int64)
    best = None
    for k in range(0x7EF00000, 0x7EF40000, 0x100):
        y = (np.int64(k) - ai).astype(np.int32).view(np.float32).astype(np.float64)
        e = np.max(np.abs(y * a.astype(np.float64) - 1.0))
        if best is None or e < best[1]:
            best = (k, e)
    k0 = best[0]
    for k in range(k0 - 0x100, k0 + 0x100):
        y = (np.int64(k) - ai).astype(np.int32).view(np.float32).astype(np.float64)
        e = np.max(np.abs(y * a.astype(np.float64) - 1.0))
        if e < best[1]:
            best = (k, e)
    return best


if __name__ == "__main__":
    (a, b), e0, e1 = fit_gelu_sigmoid()
    print(f"GELU sigmoid form: a = {a:.9g}, b = {b:.9g}  (max abs err {e1:.3e}; tanh-form start {e0:.3e})")
    c, e = fit_exp2()
    print(f"exp2 degree {DEG} on [-1/2, 1/2]: " + ", ".join(f"{v:.9g}" for v in c) + f"  (max rel err {e:.3e})")
    k, e = fit_rcp_seed()
    print(f"reciprocal seed K = 0x{k:08X}  (max rel err {e:.3e}; two Newton steps: {e**4:.3e})")
