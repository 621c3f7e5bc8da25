"""Fit the polynomial used by exp2_poly() in prefill_bf16.cu.

Method (Cody-Waite range reduction + minimax polynomial):
  2^x = 2^j * 2^f  with  j = rint(x),  f = x - j  in [-1/2, 1/2].
  2^j is applied by adding j to the float's exponent field; 2^f comes from a
  polynomial p(f) of degree 4 whose maximum RELATIVE error on [-1/2, 1/2] is
  minimised with the Remez exchange algorithm (equioscillation of
  (p(f) - 2^f) / 2^f at degree+2 points).

Run: python fit_exp2_poly.py  -> prints float32 coefficients c0..c4 and the
relative error of the float32-rounded polynomial evaluated in float64.
"""
import numpy as np

DEG = 4
LO, HI = -0.5, 0.5


def remez(deg, iters=30):
    n = deg + 2
    # Chebyshev extrema as the starting reference.
    x = 0.5 * (LO + HI) + 0.5 * (HI - LO) * np.cos(np.pi * np.arange(n)[::-1] / (n - 1))
    grid = np.linspace(LO, HI, 200001)
    for _ in range(iters):
        f = np.exp2(x)
        # Solve sum_k c_k x^k - f = (-1)^i E f  (relative equioscillation).
        A = np.zeros((n, n))
        for k in range(deg + 1):
            A[:, k] = x ** k
        A[:, -1] = -((-1.0) ** np.arange(n)) * f
        sol = np.linalg.solve(A, f)
        c = sol[:-1]
        err = (np.polyval(c[::-1], grid) - np.exp2(grid)) / np.exp2(grid)
        # New reference: extrema of the error between sign changes.
        idx = [0]
        sign = np.sign(err)
        for i in range(1, len(grid)):
            if sign[i] != sign[idx[-1]]:
                idx.append(i)
            elif abs(err[i]) > abs(err[idx[-1]]):
                idx[-1] = i
        if len(idx) >= n:
            idx = sorted(idx, key=lambda i: -abs(err[i]))[:n] if len(idx) > n else idx
            x = np.sort(grid[idx])
    return c


def main():
    c = remez(DEG)
    c32 = c.astype(np.float32)
    grid = np.linspace(LO, HI, 400001)
    p = np.zeros_like(grid)
    for ck in c32[::-1].astype(np.float64):
        p = p * grid + ck
    rel = np.abs(p - np.exp2(grid)) / np.exp2(grid)
    for k, ck in enumerate(c32):
        print(f"c{k} = {float(ck)!r}f  ({float(ck).hex()})")
    print(f"max relative error of the float32 coefficients: {rel.max():.3e}")


if __name__ == "__main__":
    main()
