"""Coefficients of the polynomial that approximates 2^f on [-1/2, 1/2] in the softmax.

p(f) = 1 + c1 f + c2 f^2 + c3 f^3 + c4 f^4, with the constant term fixed at 1 so that
2^0 is exact, and c1..c4 chosen by the Remez exchange algorithm to minimise the maximum
RELATIVE error |p(f) / 2^f - 1| over the interval (equioscillation at 5 points). Degree 4
gives 3.6e-6 (2^-18); degree 3 only 4.3e-4, about the fp16 rounding of P itself.
Run: python gen_exp2_poly.py  -> prints the fp32 coefficients and the error.
"""

import numpy as np


def remez_exp2(degree=4, iters=60):
    a, b = -0.5, 0.5
    n_free = degree              # c1..c_degree
    m = n_free + 1               # reference points (one extra for the level E)
    x = 0.5 * (a + b) + 0.5 * (b - a) * np.cos(np.pi * np.arange(m)[::-1] / (m - 1))
    grid = np.linspace(a, b, 200001)
    for _ in range(iters):
        # (1 + sum c_k x^k) / 2^x - 1 = (-1)^i E  ->  sum c_k x^k - (-1)^i E 2^x = 2^x - 1
        A = np.zeros((m, m))
        for k in range(1, degree + 1):
            A[:, k - 1] = x ** k
        A[:, -1] = -((-1.0) ** np.arange(m)) * np.exp2(x)
        rhs = np.exp2(x) - 1.0
        sol = np.linalg.solve(A, rhs)
        c = sol[:-1]
        err = (1.0 + sum(c[k - 1] * grid ** k for k in range(1, degree + 1))) / np.exp2(grid) - 1.0
        # new reference: extrema of the error, one per sign change interval
        idx = [0]
        for i in range(1, len(grid) - 1):
            if (err[i] - err[i - 1]) * (err[i + 1] - err[i]) <= 0:
                idx.append(i)
        idx.append(len(grid) - 1)
        idx = np.array(sorted(set(idx)))
        if len(idx) >= m:
            order = np.argsort(-np.abs(err[idx]))[:m]
            x = np.sort(grid[idx[order]])
    return c, float(np.max(np.abs(err)))


if __name__ == "__main__":
    c, e = remez_exp2()
    c32 = c.astype(np.float32)
    f = np.linspace(-0.5, 0.5, 100001).astype(np.float32)
    p = np.float32(0)
    for ck in c32[::-1]:
        p = (p + ck) * f
    p = np.float32(1) + p
    rel = np.max(np.abs(p.astype(np.float64) / np.exp2(f.astype(np.float64)) - 1.0))
    print("  ".join("c%d = %.9ef" % (i + 1, ck) for i, ck in enumerate(c32)))
    print("max relative error: remez %.3e, fp32 evaluation %.3e (2^%.2f)" % (e, rel, np.log2(rel)))
