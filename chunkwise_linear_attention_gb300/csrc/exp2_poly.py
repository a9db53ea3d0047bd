"""Coefficients of the polynomial p(f) ~ 2^f on [-1/2, 1/2] used by the selective scan's
2^x (selective_scan.cu: exp2_fma / exp2_fma2, which split x = k + f, k an integer).

p(f) = 1 + c1 f + ... + c6 f^6 with p(0) = 1 exactly, fitted to minimise the largest
relative error max |p(f) - 2^f| / 2^f by Lawson's iteratively reweighted least squares
(C. L. Lawson, "Contributions to the theory of linear least maximum approximation",
1961) on a dense grid.  The fit's own error is about 2e-9; evaluated in fp32 by Horner's
rule with fused multiply-adds the result is within 0.64 ulp of 2^f (checked here on
200001 points with exactly emulated fp32 FMAs).  Prints the coefficients as fp32."""
import numpy as np


def fit(deg=6, grid=20001, iters=200):
    f = np.linspace(-0.5, 0.5, grid)
    f = f[f != 0.0]
    y = 2.0 ** f
    w = np.ones_like(f)
    V = np.vander(f, deg, increasing=True) * f[:, None]  # f, f^2, ..., f^deg
    for _ in range(iters):
        c, *_ = np.linalg.lstsq(V * (w / y)[:, None], (y - 1.0) * w / y, rcond=None)
        err = np.abs(1.0 + V @ c - y) / y
        w = w * np.sqrt(err / err.max()) + 1e-12
    return c, err.max()


def fp32_horner_max_ulps(c):
    c32 = [np.float32(x) for x in c]

    def fma32(a, b, d):
        return np.float32(np.float64(a) * np.float64(b) + np.float64(d))

    worst = 0.0
    for x in np.linspace(-0.5, 0.5, 200001).astype(np.float32):
        p = c32[-1]
        for ci in reversed(c32[:-1]):
            p = fma32(p, x, ci)
        p = fma32(p, x, np.float32(1.0))
        worst = max(worst, abs(float(p) - 2.0 ** float(x)) / 2.0 ** float(x) / 2.0 ** -23)
    return worst


if __name__ == "__main__":
    c, e = fit()
    print("fit max relative error %.3e, fp32 Horner max %.2f ulp" % (e, fp32_horner_max_ulps(c)))
    for i, x in enumerate(c, 1):
        print("c%d = %.9ef" % (i, np.float32(x)))
