"""Error bound of the FMA-pipe exp2 the distillation passes use for part of the
teacher exponentials (f2_exp2_poly in lm_head_vocab_gb300/csrc/ptx.cuh).

The coefficients are read from the kernel source, the evaluation is emulated
step by step in fp32 (one rounding per add and per fused multiply-add, the
exponent added to the bits as the kernel does) and compared with 2^x in fp64
over the whole range the kernels admit, [-124, 126].  The bound is 2.5e-7
relative, about the accuracy of the hardware ex2.approx it stands in for."""
import os
import re

import numpy as np

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "lm_head_vocab_gb300", "csrc",
                   "ptx.cuh")


def _coefficients():
    txt = open(SRC).read()
    body = txt[txt.index("f2_exp2_poly(uint64_t x)"):]
    body = body[:body.index("\n}\n")]
    vals = [float(v.rstrip("f")) for v in re.findall(r"f2_pack\(([-0-9.e+]+f), \1\)", body)]
    # magic, -magic, -1, then c5, c4, c3, c2, c1, c0
    assert vals[:3] == [12582912.0, -12582912.0, -1.0], vals
    return [np.float32(v) for v in vals[3:][::-1]]   # c0 .. c5


def _fma32(a, b, c):
    return np.float32(np.float64(a) * np.float64(b) + np.float64(c))


def _exp2_kernel(coef, x):
    x = np.float32(x)
    t = np.float32(np.float64(x) + 12582912.0)          # round to nearest: n in the low bits
    n = np.float32(np.float64(t) - 12582912.0)
    f = _fma32(n, np.float32(-1.0), x)
    q = _fma32(f, coef[5], coef[4])
    for ck in (coef[3], coef[2], coef[1], coef[0]):
        q = _fma32(q, f, ck)
    bits = (int(np.float32(q).view(np.uint32)) + (int(t.view(np.uint32)) << 23)) & 0xffffffff
    return float(np.uint32(bits).view(np.float32))


def test_coefficients_parse():
    c = _coefficients()
    assert len(c) == 6 and abs(float(c[0]) - 1.0) < 1e-6 and abs(float(c[1]) - np.log(2.0)) < 1e-5


def test_relative_error_over_range():
    coef = _coefficients()
    rng = np.random.default_rng(0)
    xs = np.concatenate([rng.uniform(-124.0, 126.0, 40000), np.arange(-124.0, 126.0, 0.5),
                         np.arange(-124.0, 126.0, 1.0) + 0.49999997, np.linspace(-1, 1, 2001)]).astype(np.float32)
    worst = 0.0
    for x in xs:
        y = _exp2_kernel(coef, x)
        ref = 2.0 ** float(x)
        worst = max(worst, abs(y / ref - 1.0))
    assert worst <= 2.5e-7, worst


def test_integer_arguments_exact_power():
    coef = _coefficients()
    for n in range(-124, 127):
        y = _exp2_kernel(coef, np.float32(n))
        assert abs(y / 2.0 ** n - 1.0) <= 2.5e-7
