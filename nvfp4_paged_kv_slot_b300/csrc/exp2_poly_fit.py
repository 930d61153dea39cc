"""Derives the coefficients of the degree-3 polynomial that the prefill's
softmax uses for 2^f, f in [-1/2, 1/2], on the FMA pipe (exp2_fma in
prefill.cu).  Iteratively reweighted least squares on Chebyshev nodes
(Lawson's algorithm) approaches the minimax fit of the relative error;
coefficients are then rounded to fp32 and the fp32-evaluated error reported.

    python nvfp4_paged_kv_slot_b300/csrc/exp2_poly_fit.py
"""
import numpy as np


def fit(deg=3, nodes=4000, iters=60):
    k = np.arange(nodes)
    f = 0.5 * np.cos(np.pi * (k + 0.5) / nodes)
    a = np.vander(f, deg + 1, increasing=True) / np.exp2(f)[:, None]
    w = np.ones_like(f)
    for _ in range(iters):
        c, *_ = np.linalg.lstsq(a * w[:, None], w, rcond=None)
        e = np.abs(a @ c - 1.0)
        w = w * np.sqrt(e / e.max() + 1e-3)
        w /= w.mean()
    return c.astype(np.float32)


def fp32_rel_error(c):
    f = np.linspace(-0.5, 0.5, 200001).astype(np.float32)
    p = np.full_like(f, c[-1])
    for cc in c[-2::-1]:
        p = p * f + cc
    return float(np.abs(p.astype(np.float64) / np.exp2(f.astype(np.float64)) - 1).max())


if __name__ == "__main__":
    c = fit()
    print("coefficients c0..c3:", [float(x) for x in c])
    print("max relative error (fp32 Horner):", fp32_rel_error(c))
