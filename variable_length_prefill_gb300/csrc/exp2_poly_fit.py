"""Fit the polynomial behind exp2_poly() in ptx.cuh.

exp2_poly(x) computes 2^x without the MUFU unit, for part of the softmax's
exponentials (the rest stay on ex2.approx), so that the two pipes share the
work.  Method:

* Range reduction (Cody and Waite's scheme, with a single constant because
  the base is 2): n = round-to-nearest(x), f = x - n, so f is in [-1/2, 1/2]
  and 2^x = 2^n * 2^f; 2^n is applied by adding n to the exponent field.
* 2^f ~ p(f) = 1 + f (c1 + f (c2 + f c3)): p(0) = 1 exactly, so a row's
  largest score still gets weight 1.  (c1, c2, c3) minimise the largest
  relative error max |p(f) / 2^f - 1| over [-1/2, 1/2]: a discrete Chebyshev
  (minimax) fit on a dense grid, solved as a linear program, which reaches the
  same equioscillating solution as the Remez exchange.

Run it to print the coefficients rounded to float32 and the relative error of
the float32 evaluation (fused multiply-adds, as the kernel does):

    python exp2_poly_fit.py
"""
import numpy as np
from scipy.optimize import linprog


def fit(degree: int = 3, grid: int = 20001):
    f = np.linspace(-0.5, 0.5, grid)
    f = f[f != 0.0]  # p(0) = 1 holds exactly; the error vanishes there
    t = np.exp2(f)
    # relative error e = (1 + sum_k c_k f^k) / 2^f - 1, linear in c
    A = np.stack([f ** k / t for k in range(1, degree + 1)], axis=1)
    b = 1.0 - 1.0 / t
    n = degree
    # variables (c_1..c_n, E): minimise E with |A c - b| <= E
    cost = np.zeros(n + 1)
    cost[-1] = 1.0
    A_ub = np.block([[A, -np.ones((A.shape[0], 1))], [-A, -np.ones((A.shape[0], 1))]])
    b_ub = np.concatenate([b, -b])
    r = linprog(cost, A_ub=A_ub, b_ub=b_ub, bounds=[(None, None)] * (n + 1), method="highs")
    assert r.success, r.message
    return r.x[:n], r.x[n]


def eval_f32(x: np.ndarray, c: np.ndarray) -> np.ndarray:
    """The kernel's float32 sequence: magic-number rounding, f = x - n, Horner
    with fused multiply-adds (emulated: exact product and sum in float64,
    one rounding to float32), exponent add."""
    x = np.maximum(x.astype(np.float32), np.float32(-127.0))
    magic = np.float32(12582912.0)  # 1.5 * 2^23: x + magic rounds x to an integer
    tt = (x + magic).astype(np.float32)
    nf = (tt - magic).astype(np.float32)
    fr = (x.astype(np.float64) - nf.astype(np.float64)).astype(np.float32)

    def fma(a, b, cc):
        return (a.astype(np.float64) * b.astype(np.float64) + np.float64(cc)).astype(np.float32)
    p = fma(np.full_like(fr, c[2]), fr, c[1])
    p = fma(p, fr, c[0])
    p = fma(p, fr, np.float32(1.0))
    bits = (p.view(np.uint32).astype(np.int64) + (tt.view(np.uint32).astype(np.int64) << 23))
    return (bits & 0xFFFFFFFF).astype(np.uint32).view(np.float32)


if __name__ == "__main__":
    c, e = fit()
    c32 = c.astype(np.float32)
    print("coefficients c1, c2, c3 (float32):", [float(v) for v in c32])
    print("hex:", [hex(int(v)) for v in c32.view(np.uint32)])
    print(f"minimax relative error of the exact polynomial: {e:.3e}")
    x = np.linspace(-126.0, 8.0, 4000001, dtype=np.float64).astype(np.float32)
    y = eval_f32(x, c32)
    rel = np.abs(y.astype(np.float64) / np.exp2(x.astype(np.float64)) - 1.0)
    print(f"float32 evaluation, x in [-126, 8]: max relative error {rel.max():.3e}")
