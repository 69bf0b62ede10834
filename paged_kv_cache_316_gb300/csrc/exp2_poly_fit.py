"""Fit the polynomial p(f) ~ 2^f on [-1/2, 1/2] used by the prefill kernel to
compute part of its exponentials on the FMA pipe.

2^x = 2^n * 2^f with n = round(x), f = x - n in [-1/2, 1/2] (Cody-Waite
style range reduction); 2^f is approximated by the degree-4 polynomial that
interpolates 2^f at the 5 Chebyshev nodes of [-1/2, 1/2] (near-minimax).
Run this file to print the coefficients (c0..c4, float32) and the maximum
relative error of the float32 evaluation over a dense grid.
"""
import numpy as np


def fit(degree: int = 4):
    k = np.arange(degree + 1)
    nodes = 0.5 * np.cos((2 * k + 1) * np.pi / (2 * (degree + 1)))
    V = np.vander(nodes, degree + 1, increasing=True)
    return np.linalg.solve(V, np.exp2(nodes))


def eval_f32(c, f):
    c = c.astype(np.float32)
    f = f.astype(np.float32)
    acc = np.full_like(f, c[-1])
    for ci in c[-2::-1]:
        acc = (acc * f + ci).astype(np.float32)
    return acc


if __name__ == "__main__":
    c = fit()
    f = np.linspace(-0.5, 0.5, 200001)
    rel = np.abs(eval_f32(c, f).astype(np.float64) / np.exp2(f) - 1.0)
    print("coefficients:", ", ".join(f"{x:.9e}f" for x in c.astype(np.float32)))
    print("max relative error (float32 Horner):", rel.max())
