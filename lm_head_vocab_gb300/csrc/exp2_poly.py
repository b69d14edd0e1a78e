"""Coefficients of the degree-5 polynomial for 2^f, f in [-1/2, 1/2], used by
the kernels' packed exp2 (f32x2 FMA pipe) next to the hardware ex2.

Method: Remez exchange on the relative error w(f) (2^f - p(f)), w = 2^-f, in
50-digit arithmetic; the coefficients are then rounded to fp32.  Run it to
print the coefficients and the error of the fp32 evaluation (Horner with
fused multiply-adds, emulated in double with one rounding per step):

    python lm_head_vocab_gb300/csrc/exp2_poly.py
"""
import mpmath as mp
import numpy as np

DEG = 5


def remez(deg, a, b, iters=30):
    f = lambda x: mp.power(2, x)
    w = lambda x: 1 / mp.power(2, x)
    n = deg + 2
    xs = [(a + b) / 2 + (b - a) / 2 * mp.cos(mp.pi * (n - 1 - i) / (n - 1)) for i in range(n)]
    c = None
    for _ in range(iters):
        A = mp.matrix(n, n)
        rhs = mp.matrix(n, 1)
        for i, x in enumerate(xs):
            for j in range(deg + 1):
                A[i, j] = x ** j
            A[i, deg + 1] = (-1) ** i / w(x)
            rhs[i] = f(x)
        sol = mp.lu_solve(A, rhs)
        c = [sol[j] for j in range(deg + 1)]
        grid = [a + (b - a) * k / 4000 for k in range(4001)]
        vals = [w(x) * (f(x) - sum(c[j] * x ** j for j in range(deg + 1))) for x in grid]
        ext, s0 = [], 0
        for k in range(1, len(grid)):
            if mp.sign(vals[k]) != mp.sign(vals[s0]) and vals[k] != 0:
                ext.append(grid[max(range(s0, k), key=lambda q: abs(vals[q]))])
                s0 = k
        ext.append(grid[max(range(s0, len(grid)), key=lambda q: abs(vals[q]))])
        if len(ext) != n:
            break
        xs = ext
    return c


def f32(x):
    return np.float32(x)


def fma32(a, b, c):
    return f32(np.float64(a) * np.float64(b) + np.float64(c))


def eval_fp32(coef, x):
    """2^x as the kernel forms it: n = rint(x), f = x - n, Horner on f, n added to the exponent."""
    x = f32(x)
    n = f32(np.rint(np.float64(x)))
    fr = f32(np.float64(x) - np.float64(n))
    p = coef[-1]
    for ck in coef[-2::-1]:
        p = fma32(p, fr, ck)
    return np.ldexp(np.float64(p), int(n))


def main():
    mp.mp.dps = 50
    c = remez(DEG, mp.mpf(-0.5), mp.mpf(0.5))
    coef = [f32(float(ci)) for ci in c]
    xs = np.linspace(-60.0, 20.0, 200001, dtype=np.float32)
    rel = max(abs(eval_fp32(coef, x) / 2.0 ** np.float64(x) - 1.0) for x in xs[::7])
    for k, ck in enumerate(coef):
        print(f"c{k} = {float(ck):.9e}f  (bits 0x{np.float32(ck).view(np.uint32):08x})")
    print(f"max relative error of the fp32 evaluation over a sample of [-60, 20]: {rel:.3e}")


if __name__ == "__main__":
    main()
