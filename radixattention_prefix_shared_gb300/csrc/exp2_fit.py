"""Fit the cubic used for 2^x on the FMA pipe in the extend kernel's softmax.

Method (range reduction + polynomial): write x = j + f with j = round(x) and
-1/2 <= f <= 1/2, so 2^x = 2^j * 2^f.  j is obtained by adding
1.5 * 2^23 (the float then holds round(x) in its low mantissa bits), 2^j is
applied by adding j to the float's exponent field, and 2^f is the cubic
p(f) = 1 + f*(c1 + f*(c2 + f*c3)) -- p(0) = 1 exactly -- whose coefficients
minimise the maximum relative error |p(f) / 2^f - 1| over a dense grid of
[-1/2, 1/2] (a linear program solved with scipy's HiGHS).  Run this file to
print the coefficients pasted into common.cuh and the error of the float32
evaluation; the unit test checks that bound.
"""
import numpy as np

MAGIC = np.float32(12582912.0)  # 1.5 * 2^23


def fit(n_grid: int = 4001):
    from scipy.optimize import linprog
    f = np.linspace(-0.5, 0.5, n_grid)
    t = np.exp2(f)
    A = np.stack([f, f ** 2, f ** 3], axis=1) / t[:, None]
    b = 1.0 - 1.0 / t                        # |A c - b| <= e  <=>  |p/2^f - 1| <= e
    ones = np.ones((n_grid, 1))
    A_ub = np.vstack([np.hstack([A, -ones]), np.hstack([-A, -ones])])
    b_ub = np.concatenate([b, -b])
    res = linprog(c=[0, 0, 0, 1], A_ub=A_ub, b_ub=b_ub,
                  bounds=[(None, None)] * 3 + [(0, None)], method="highs")
    assert res.success, res.message
    return res.x[:3], res.x[3]


def exp2_f32(x, c):
    """The kernel's float32 evaluation, step by step, on the host."""
    x = np.maximum(np.asarray(x, np.float32), np.float32(-125.0))
    t = (x + MAGIC).astype(np.float32)
    jf = (t - MAGIC).astype(np.float32)
    f = (x - jf).astype(np.float32)
    c1, c2, c3 = (np.float32(v) for v in c)
    p = (c3 * f + c2).astype(np.float32)
    p = (p * f + c1).astype(np.float32)
    p = (p * f + np.float32(1.0)).astype(np.float32)
    j = t.view(np.int32) - MAGIC.view(np.int32)
    return (p.view(np.int32) + (j << 23)).view(np.float32)


if __name__ == "__main__":
    c, e = fit()
    print("c1, c2, c3 =", ", ".join(f"{float(np.float32(v))!r}f" for v in c))
    print(f"max relative error of the cubic (LP) = {e:.3e}")
    x = np.linspace(-125, 8, 2_000_001, dtype=np.float32)
    err = np.max(np.abs(exp2_f32(x, c).astype(np.float64) / np.exp2(x.astype(np.float64)) - 1))
    print(f"max relative error of the float32 evaluation on [-125, 8] = {err:.3e}")
