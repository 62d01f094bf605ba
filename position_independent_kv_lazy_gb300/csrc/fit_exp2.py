"""Fit the polynomial the prefill softmax uses for 2^f, f in [-1/2, 1/2].

The kernel splits x = j + f with j = round(x) (Cody-Waite reduction with the 1.5 * 2^23 rounding
constant) and forms 2^x = p(f) * 2^j, adding j to the exponent bits. p is a degree-5 polynomial
fitted here by minimising the relative error max |p(f) / 2^f - 1| with a few rounds of
iteratively reweighted least squares on Chebyshev nodes (a discrete Remez approximation), then
rounding the coefficients to float32. Run: python fit_exp2.py  (prints the C constants and the
max relative error in float32 Horner evaluation).
"""
import numpy as np


def fit(degree=5, n=4001, rounds=40):
    k = np.arange(n)
    f = 0.5 * np.cos(np.pi * (2 * k + 1) / (2 * n))           # Chebyshev nodes on [-1/2, 1/2]
    target = np.exp2(f)
    V = np.vander(f, degree + 1, increasing=True)
    w = np.ones(n)
    for _ in range(rounds):
        A = V * (w / target)[:, None]
        c, *_ = np.linalg.lstsq(A, w, rcond=None)
        err = np.abs(V @ c / target - 1)
        w = w * (1 + 30 * err / err.max())                        # push weight to the peaks
        w /= w.mean()
    return c


def horner_f32(c, f):
    c32 = np.asarray(c, dtype=np.float32)
    acc = np.full_like(f, c32[-1], dtype=np.float32)
    for a in c32[-2::-1]:
        acc = (acc * f + a).astype(np.float32)
    return acc


if __name__ == "__main__":
    c = fit()
    f = np.linspace(-0.5, 0.5, 200001, dtype=np.float32)
    rel = np.abs(horner_f32(c, f).astype(np.float64) / np.exp2(f.astype(np.float64)) - 1)
    print("// max relative error (float32 Horner): %.3e" % rel.max())
    for i, a in enumerate(np.asarray(c, dtype=np.float32)):
        print("constexpr float kExp2C%d = %.9ef;" % (i, a))
