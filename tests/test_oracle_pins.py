"""Pins for the fp64 oracle: facts fixed by the pages and by mathematics, not by
the oracle itself.

Each test below checks the oracle against something independent of it:
the pages' worked example, closed forms, a 50-digit brute-force evaluation
with finite differences, or PyTorch fp64 autograd.  A dropped term, a wrong
sign, a wrong index or a transposed operand anywhere in the oracle fails at
least one of them.
"""
import math

import mpmath
import numpy as np
import pytest
import torch

import oracle
from oracle import Problem

mp = mpmath.mp


def f32_rows(rows):
    return np.ascontiguousarray(np.array(rows, dtype=np.float32))


def run(P):
    R, g = oracle.forward_backward(P, nthreads=1)
    return R, g


# --------------------------------------------------------------------------
# The pages' worked example: a row with target margin 20.
# torchtitan PR 5661, review "Example".
# --------------------------------------------------------------------------
@pytest.mark.parametrize("V", [2, 1000, 32000])
def test_worked_example_margin20(golden, V):
    gold = golden("worked_example_margin20.txt")
    margin = gold["margin"]
    # non-targets all at 0, target at margin + ln(V-1): z_t - lse_{j!=t} z = margin exactly
    z = np.zeros((1, V), dtype=np.float64)
    z[0, 0] = margin + math.log(V - 1)
    P = Problem(logits=z.astype(np.float32), V=V, targets=np.array([0]))
    R, g = run(P)
    lse_nt = math.log(V - 1)
    zt = float(np.float32(z[0, 0]))
    expected = float(mpmath.log1p(mpmath.exp(mpmath.mpf(lse_nt) - mpmath.mpf(zt))))
    digits = int(gold["significant_digits"])
    assert float(f"{R.nll[0]:.{digits}g}") == gold["nll"]
    assert float(f"{g[0, 0]:.{digits}g}") == gold["target_grad"]
    assert R.nll[0] == pytest.approx(expected, rel=1e-12)
    # target gradient is -p_nt = -sigmoid(lse_nt - z_t)
    assert g[0, 0] == pytest.approx(-expected, rel=1e-8)
    assert abs(g.sum() - gold["row_sum"]) <= 1e-12 * np.abs(g).sum()


def test_worked_example_v2_exact():
    # z = [20, 0], target 0: margin exactly 20 in any precision.
    P = Problem(logits=f32_rows([[20.0, 0.0]]), V=2, targets=np.array([0]))
    R, g = run(P)
    sp = float(mpmath.log1p(mpmath.exp(-20)))
    sig = float(1 / (1 + mpmath.exp(20)))
    assert R.nll[0] == pytest.approx(sp, rel=1e-14)
    assert g[0, 0] == pytest.approx(-sig, rel=1e-14)
    assert g[0, 1] == pytest.approx(sig, rel=1e-14)
    assert g.sum() == 0.0


# --------------------------------------------------------------------------
# The collapse the pages fix: fp32 lse - z_t is exactly 0 past ln 2^24.
# --------------------------------------------------------------------------
def test_collapse_threshold(golden):
    gold = golden("collapse_margin.txt")
    thr = math.log(2.0 ** 24)
    assert thr == pytest.approx(gold["threshold_approx"], abs=0.05)
    V = 2
    for margin in [10.0, 15.0, 16.0, 17.0, 20.0, 30.0, 40.0]:
        z = np.array([[margin, 0.0]], dtype=np.float32)
        # naive fp32 form: log(sum_j exp(z_j - m)) - (z_t - m), m the row max;
        # the sum rounds to exactly 1 once e^-margin < 2^-24
        m = z.max(axis=1, keepdims=True)
        shifted = z - m
        naive = (np.log(np.exp(shifted).sum(axis=1)) - shifted[:, 0]).astype(np.float32)[0]
        R, g = run(Problem(logits=z, V=V, targets=np.array([0])))
        exact = float(mpmath.log1p(mpmath.exp(-margin)))
        assert R.nll[0] == pytest.approx(exact, rel=1e-13)
        assert R.nll[0] > 0 and g[0, 0] < 0
        if margin > thr + 0.2:
            assert naive == 0.0, margin
        if margin < thr - 0.2:
            assert naive > 0.0, margin


# --------------------------------------------------------------------------
# Closed forms.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("V", [1, 2, 7, 1024, 32000])
@pytest.mark.parametrize("c", [0.0, -3.5, 10.0])
def test_uniform_logits(V, c):
    alpha = 1e-3
    T = 3
    z = np.full((T, V), c, dtype=np.float32)
    t = np.arange(T) % V
    P = Problem(logits=z, V=V, targets=t, z_alpha=alpha, teacher=(z + 1.5).astype(np.float32),
                kl_weight=0.7)
    R, g = run(P)
    lnV = math.log(V)
    np.testing.assert_allclose(R.nll, lnV, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(R.lse, c + lnV, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(R.kl, 0.0, atol=1e-14)
    assert R.ce == pytest.approx(lnV, rel=1e-13, abs=1e-15)
    assert R.z == pytest.approx(alpha * (c + lnV) ** 2, rel=1e-13, abs=1e-18)
    # gradient: (1/T) * [(1/V - onehot) + 2 alpha (c+lnV) / V]
    exp_g = np.full((T, V), (1.0 / V + 2 * alpha * (c + lnV) / V) / T)
    exp_g[np.arange(T), t] -= 1.0 / T
    np.testing.assert_allclose(g, exp_g, rtol=1e-12, atol=1e-15)


def bern_kl(du, dz):
    """KL(Bern(q) || Bern(p)) at 50 digits, q = sigmoid(du), p = sigmoid(dz)."""
    mp.dps = 50
    q = 1 / (1 + mpmath.exp(-mpmath.mpf(du)))
    p = 1 / (1 + mpmath.exp(-mpmath.mpf(dz)))
    return float(q * mpmath.log(q / p) + (1 - q) * mpmath.log((1 - q) / (1 - p)))


@pytest.mark.parametrize("seed", range(5))
def test_two_class_closed_form(seed):
    rng = np.random.default_rng(seed)
    T = 6
    z = rng.normal(0, 4, size=(T, 2)).astype(np.float32)
    u = rng.normal(0, 4, size=(T, 2)).astype(np.float32)
    t = rng.integers(0, 2, size=T)
    w_kl = 0.5
    P = Problem(logits=z, V=2, targets=t, teacher=u, kl_weight=w_kl)
    R, g = run(P)
    zd = z.astype(np.float64)
    ud = u.astype(np.float64)
    for r in range(T):
        tt, o = t[r], 1 - t[r]
        d = zd[r, o] - zd[r, tt]
        nll = float(mpmath.log1p(mpmath.exp(d)))
        assert R.nll[r] == pytest.approx(nll, rel=1e-13)
        sig = 1.0 / (1.0 + math.exp(-d))          # p of the other class
        p1 = 1.0 / (1.0 + math.exp(-(zd[r, 1] - zd[r, 0])))
        q1 = 1.0 / (1.0 + math.exp(-(ud[r, 1] - ud[r, 0])))
        assert R.kl[r] == pytest.approx(bern_kl(ud[r, 1] - ud[r, 0], zd[r, 1] - zd[r, 0]),
                                        rel=1e-11, abs=1e-14)
        # gradient with s_tok = 1/T
        g_ce = np.zeros(2)
        g_ce[tt] = -sig
        g_ce[o] = sig
        g_kl = np.array([-(p1 - q1), p1 - q1])
        np.testing.assert_allclose(g[r], (g_ce + w_kl * g_kl) / T, rtol=1e-11, atol=1e-16)


@pytest.mark.parametrize("tau", [0.1, 0.5, 3.0, 10.0])
def test_two_class_closed_form_temperature(tau):
    """Distillation at a temperature, two classes: KL(Bern(q) || Bern(p^tau)) with
    q = sigmoid((u1 - u0)/tau), p^tau = sigmoid((z1 - z0)/tau), and its gradient
    w_kl (p^tau - q)/tau, no tau^2 factor (the oracle's reading of the pages'
    distillation term)."""
    rng = np.random.default_rng(int(tau * 10))
    T = 6
    z = rng.normal(0, 2, size=(T, 2)).astype(np.float32)
    u = rng.normal(0, 2, size=(T, 2)).astype(np.float32)
    t = rng.integers(0, 2, size=T)
    w_kl = 0.5
    P = Problem(logits=z, V=2, targets=t, teacher=u, kl_weight=w_kl, temperature=tau, ce_weight=0.0)
    R, g = run(P)
    zd, ud = z.astype(np.float64), u.astype(np.float64)
    for r in range(T):
        du, dz = (ud[r, 1] - ud[r, 0]) / tau, (zd[r, 1] - zd[r, 0]) / tau
        assert R.kl[r] == pytest.approx(bern_kl(du, dz), rel=1e-10, abs=1e-14)
        p1 = 1.0 / (1.0 + math.exp(-dz))
        q1 = 1.0 / (1.0 + math.exp(-du))
        g_kl = np.array([-(p1 - q1), p1 - q1]) / tau
        np.testing.assert_allclose(g[r], w_kl * g_kl / T, rtol=1e-10, atol=1e-16)


@pytest.mark.parametrize("tau", [0.5, 3.0])
def test_torch_fp64_autograd_temperature(tau):
    """The same against PyTorch fp64: kl_div of the tempered log-softmaxes, and
    autograd through z for the gradient."""
    rng = np.random.default_rng(int(tau * 7))
    T, V = 12, 301
    z = rng.normal(0, 3, size=(T, V)).astype(np.float32)
    u = (z + rng.normal(0, 1, size=(T, V))).astype(np.float32)
    t = rng.integers(0, V, size=T)
    t[3] = -100
    w_kl = 0.5
    P = Problem(logits=z, V=V, targets=t, teacher=u, kl_weight=w_kl, temperature=tau)
    R, g = run(P)
    zt = torch.tensor(z, dtype=torch.float64, requires_grad=True)
    ut = torch.tensor(u, dtype=torch.float64)
    tt = torch.tensor(t)
    act = tt != -100
    N = int(act.sum())
    ce = torch.nn.functional.cross_entropy(zt, tt, ignore_index=-100, reduction="sum") / N
    kl = torch.nn.functional.kl_div(torch.log_softmax(zt[act] / tau, 1), torch.log_softmax(ut[act] / tau, 1),
                                    log_target=True, reduction="sum") / N
    (ce + w_kl * kl).backward()
    assert R.kl_loss == pytest.approx(kl.item(), rel=1e-10)
    np.testing.assert_allclose(g, zt.grad.numpy(), rtol=1e-9, atol=1e-15)


def test_problem_rejects_other_dtypes():
    """The oracle reads float32 or bf16 bits only; a float64 array is refused,
    not reinterpreted."""
    z = np.zeros((2, 4))
    with pytest.raises(TypeError):
        Problem(logits=z, V=4, targets=np.zeros(2, dtype=np.int64))
    with pytest.raises(TypeError):
        Problem(logits=z.astype(np.float32), V=4, targets=np.zeros(2, dtype=np.int64), teacher=z)


@pytest.mark.parametrize("tau", [0.25, 1.0, 4.0])
def test_kl_shift_invariance(tau):
    """Adding a constant to every teacher logit, or to every student logit, of a
    row changes neither distribution: the KL and its gradient stay as they were."""
    rng = np.random.default_rng(17)
    T, V = 5, 64
    # values on a 1/64 grid, so the shifted logits are exact in float32 too
    z = np.round(rng.normal(0, 2, size=(T, V)) * 64) / 64
    u = z + np.round(rng.normal(0, 1, size=(T, V)) * 64) / 64
    t = rng.integers(0, V, size=T)
    f = np.float32
    base = run(Problem(logits=z.astype(f), V=V, targets=t, teacher=u.astype(f), kl_weight=1.0, ce_weight=0.0,
                       temperature=tau))
    for dz, du in [(0.0, 7.5), (-3.25, 0.0), (2.0, -9.0)]:
        R, g = run(Problem(logits=(z + dz).astype(f), V=V, targets=t, teacher=(u + du).astype(f), kl_weight=1.0,
                           ce_weight=0.0, temperature=tau))
        np.testing.assert_allclose(R.kl, base[0].kl, rtol=1e-11, atol=1e-14)
        # absolute at the terms' scale: where p^tau - q cancels, fp64's rounding of
        # the shifted exponent arguments (of size ~40 at tau = 1/4) shows at 1e-15
        np.testing.assert_allclose(g, base[1], rtol=1e-10, atol=1e-14)


# --------------------------------------------------------------------------
# Invariant: CE, KL and GSPO parts of a row gradient sum to 0; z part to 2 a lse s.
# --------------------------------------------------------------------------
def test_row_sums():
    rng = np.random.default_rng(7)
    T, V = 8, 257
    z = rng.normal(0, 3, size=(T, V)).astype(np.float32)
    u = (z + rng.normal(0, 1, size=(T, V))).astype(np.float32)
    t = rng.integers(0, V, size=T)
    t[2] = -100
    alpha = 0.01
    P = Problem(logits=z, V=V, targets=t, teacher=u, kl_weight=0.5, z_alpha=alpha)
    R = oracle.forward(P, nthreads=1)
    act = R.active.astype(bool)
    for w_ce, a, w_kl in [(1, 0, 0), (0, alpha, 0), (0, 0, 0.5)]:
        P2 = Problem(logits=z, V=V, targets=t, teacher=u, kl_weight=w_kl, z_alpha=a, ce_weight=w_ce)
        g = oracle.grad_rows(P2, R)
        sums = g.sum(axis=1)
        expect = np.where(act, 2 * a * R.lse * R.s_tok, 0.0)
        np.testing.assert_allclose(sums, expect, atol=1e-15 * 50)
        assert np.all(g[~act] == 0.0)


# --------------------------------------------------------------------------
# SUM reduction over shards with the global denominator equals the token mean.
# xtuner PR 1963, description.
# --------------------------------------------------------------------------
def test_shard_sum_equals_token_mean():
    rng = np.random.default_rng(3)
    T, V = 24, 300
    z = rng.normal(0, 2, size=(T, V)).astype(np.float32)
    t = rng.integers(0, V, size=T)
    t[[1, 5, 6]] = -100
    full = Problem(logits=z, V=V, targets=t, z_alpha=1e-3)
    Rf, gf = run(full)
    N = Rf.n_active
    total = 0.0
    parts = []
    for lo, hi in [(0, 7), (7, 16), (16, 24)]:
        Ps = Problem(logits=z[lo:hi], V=V, targets=t[lo:hi], z_alpha=1e-3,
                     reduction=oracle.REDUCE_SUM, denominator=float(N))
        Rs, gs = run(Ps)
        total += Rs.total
        parts.append(gs)
    assert total == pytest.approx(Rf.total, rel=1e-12)
    assert np.array_equal(np.concatenate(parts), gf)


# --------------------------------------------------------------------------
# Brute force at 50 digits, gradient by central differences of the total loss.
# --------------------------------------------------------------------------
def mp_total(z, u, t, act, alpha, w_ce, w_kl, tau, seg, S, adv, old, eps_lo, eps_hi,
             reduction, denom, tadv=None):
    T = len(z)
    V = len(z[0])
    N = sum(1 for r in range(T) if act[r])
    s_tok = (mpmath.mpf(1) / N if N else mpmath.mpf(0)) if reduction == 1 else 1 / mpmath.mpf(denom)
    ce = zl = kl = mpmath.mpf(0)
    logp = [None] * T
    for r in range(T):
        if not act[r]:
            continue
        lse = mpmath.log(mpmath.fsum(mpmath.exp(x) for x in z[r]))
        logp[r] = z[r][t[r]] - lse
        ce += -logp[r]
        zl += alpha * lse ** 2
        if u is not None:
            la = mpmath.log(mpmath.fsum(mpmath.exp(x / tau) for x in u[r]))
            lb = mpmath.log(mpmath.fsum(mpmath.exp(x / tau) for x in z[r]))
            for j in range(V):
                lq = u[r][j] / tau - la
                kl += mpmath.exp(lq) * (lq - (z[r][j] / tau - lb))
    tot = s_tok * (w_ce * ce + zl + w_kl * kl)
    if tadv is not None:
        for r in range(T):
            if not act[r]:
                continue
            rho = mpmath.exp(logp[r] - old[r])
            c = min(max(rho, 1 - eps_lo), 1 + eps_hi)
            tot += s_tok * (-min(rho * tadv[r], c * tadv[r]))
    if seg is not None:
        n = [0] * S
        D = [mpmath.mpf(0)] * S
        for r in range(T):
            if act[r] and seg[r] >= 0:
                n[seg[r]] += 1
                D[seg[r]] += logp[r] - old[r]
        ne = sum(1 for i in range(S) if n[i])
        s_seg = (mpmath.mpf(1) / ne if ne else 0) if reduction == 1 else 1 / mpmath.mpf(denom)
        for i in range(S):
            if n[i] == 0:
                continue
            s = mpmath.exp(D[i] / n[i])
            c = min(max(s, 1 - eps_lo), 1 + eps_hi)
            tot += s_seg * (-min(s * adv[i], c * adv[i]))
    return tot


BRUTE_CASES = [
    # name, T, V, kw
    ("ce", 3, 4, dict()),
    ("ce_z", 3, 3, dict(z_alpha=0.05)),
    ("kl_tau1", 2, 4, dict(teacher=True, kl_weight=0.5, temperature=1.0)),
    ("kl_tau2", 2, 3, dict(teacher=True, kl_weight=0.7, temperature=2.0, z_alpha=0.01)),
    ("masked_sum", 3, 4, dict(mask=[1, 0, 1], reduction=0, denominator=5.0, z_alpha=0.02)),
    ("gspo", 3, 3, dict(gspo=True, ce_weight=0.0, z_alpha=0.01)),
    ("gspo_ce_sum", 3, 4, dict(gspo=True, ce_weight=1.0, reduction=0, denominator=3.0)),
    ("grpo", 4, 3, dict(grpo=True, ce_weight=0.0, z_alpha=0.01)),
    ("grpo_ce_masked", 4, 4, dict(grpo=True, ce_weight=1.0, mask=[1, 1, 0, 1])),
]


@pytest.mark.parametrize("name,T,V,kw", BRUTE_CASES, ids=[c[0] for c in BRUTE_CASES])
def test_brute_force_mpmath(name, T, V, kw):
    mp.dps = 50
    rng = np.random.default_rng(abs(hash(name)) % 2**31)
    z = rng.normal(0, 2, size=(T, V)).astype(np.float32)
    u = rng.normal(0, 2, size=(T, V)).astype(np.float32) if kw.get("teacher") else None
    t = rng.integers(0, V, size=T)
    mask = np.array(kw.get("mask", [1] * T), dtype=np.uint8)
    seg = old = adv = None
    S = 0
    eps_lo = eps_hi = 0.0
    if kw.get("gspo"):
        # two segments; seg 1 pushed well above 1+eps_hi with A>0 -> clipped, no gradient
        seg = np.array([0, 0, 1][:T] + [1] * (T - 3), dtype=np.int32)
        S = 2
        adv = np.array([0.8, 1.3], dtype=np.float32)
        eps_lo, eps_hi = 0.2, 0.2
        old = np.zeros(T, dtype=np.float32)
    P = Problem(logits=z, V=V, targets=t, loss_mask=mask, ce_weight=kw.get("ce_weight", 1.0),
                z_alpha=kw.get("z_alpha", 0.0), teacher=u, kl_weight=kw.get("kl_weight", 0.0),
                temperature=kw.get("temperature", 1.0), reduction=kw.get("reduction", 1),
                denominator=kw.get("denominator", 1.0))
    if kw.get("gspo"):
        R0 = oracle.forward(P, nthreads=1)
        # seg 0: ratio ~ exp(0.05) inside the band; seg 1: ratio ~ exp(1) clipped
        for r in range(T):
            if seg[r] == 0:
                old[r] = np.float32(R0.logp[r] - 0.05)
            else:
                old[r] = np.float32(R0.logp[r] - 1.0)
        P.segment_ids, P.num_segments, P.advantages, P.old_logprobs = seg, S, adv, old
        P.clip_eps_low, P.clip_eps_high = eps_lo, eps_hi
    tadv = None
    if kw.get("grpo"):
        # four tokens: two inside the band (one per sign of A), one clipped high
        # with A > 0 (no gradient), one above the band with A < 0 (flows)
        R0 = oracle.forward(P, nthreads=1)
        shifts = [0.05, -0.05, 1.0, 1.0][:T]
        tadv = np.array([0.7, -1.1, 1.3, -0.4][:T], dtype=np.float32)
        old = np.array([np.float32(R0.logp[r] - shifts[r]) for r in range(T)], dtype=np.float32)
        eps_lo, eps_hi = 0.2, 0.2
        P.token_advantages, P.old_logprobs = tadv, old
        P.clip_eps_low, P.clip_eps_high = eps_lo, eps_hi
    R, g = run(P)

    zm = [[mpmath.mpf(float(x)) for x in row] for row in z]
    um = None if u is None else [[mpmath.mpf(float(x)) for x in row] for row in u]
    act = R.active.astype(bool).tolist()
    args = dict(t=t.tolist(), act=act, alpha=mpmath.mpf(P.z_alpha), w_ce=mpmath.mpf(P.ce_weight),
                w_kl=mpmath.mpf(P.kl_weight), tau=mpmath.mpf(P.temperature),
                seg=None if seg is None else seg.tolist(), S=S,
                adv=None if adv is None else [mpmath.mpf(float(a)) for a in adv],
                old=None if old is None else [mpmath.mpf(float(o)) for o in old],
                eps_lo=mpmath.mpf(eps_lo), eps_hi=mpmath.mpf(eps_hi),
                reduction=P.reduction, denom=P.denominator,
                tadv=None if tadv is None else [mpmath.mpf(float(a)) for a in tadv])
    tot = mp_total(zm, um, **args)
    assert R.total == pytest.approx(float(tot), rel=1e-13, abs=1e-15)
    h = mpmath.mpf("1e-20")
    for r in range(T):
        for j in range(V):
            zp = [row[:] for row in zm]
            zn = [row[:] for row in zm]
            zp[r][j] += h
            zn[r][j] -= h
            fd = (mp_total(zp, um, **args) - mp_total(zn, um, **args)) / (2 * h)
            assert g[r, j] == pytest.approx(float(fd), rel=1e-11, abs=1e-14), (r, j)


# --------------------------------------------------------------------------
# Library special case: PyTorch fp64 cross_entropy / logsumexp / kl_div + autograd.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(3))
def test_torch_fp64_autograd(seed):
    rng = np.random.default_rng(100 + seed)
    T, V = 16, 515
    z = rng.normal(0, 3, size=(T, V)).astype(np.float32)
    u = (z + rng.normal(0, 1, size=(T, V))).astype(np.float32)
    t = rng.integers(0, V, size=T)
    t[[0, 9]] = -100
    alpha, w_kl = 1e-3, 0.5
    P = Problem(logits=z, V=V, targets=t, z_alpha=alpha, teacher=u, kl_weight=w_kl)
    R, g = run(P)

    zt = torch.tensor(z, dtype=torch.float64, requires_grad=True)
    ut = torch.tensor(u, dtype=torch.float64)
    tt = torch.tensor(t)
    act = tt != -100
    N = int(act.sum())
    ce = torch.nn.functional.cross_entropy(zt, tt, ignore_index=-100, reduction="sum") / N
    lse = torch.logsumexp(zt, dim=1)
    zl = (alpha * lse[act] ** 2).sum() / N
    kl = torch.nn.functional.kl_div(torch.log_softmax(zt[act], 1), torch.log_softmax(ut[act], 1),
                                    log_target=True, reduction="sum") / N
    total = ce + zl + w_kl * kl
    total.backward()
    assert R.ce == pytest.approx(ce.item(), rel=1e-12)
    assert R.z == pytest.approx(zl.item(), rel=1e-12)
    assert R.kl_loss == pytest.approx(kl.item(), rel=1e-10)
    assert R.total == pytest.approx(total.item(), rel=1e-12)
    np.testing.assert_allclose(g, zt.grad.numpy(), rtol=1e-9, atol=1e-15)


# --------------------------------------------------------------------------
# GSPO closed forms.
# --------------------------------------------------------------------------
def _gspo_problem(log_ratio, A, eps=(0.1, 0.1), T=5, V=11, seed=0):
    """One segment over all T rows whose mean log-ratio is log_ratio."""
    rng = np.random.default_rng(seed)
    z = rng.normal(0, 1, size=(T, V)).astype(np.float32)
    t = rng.integers(0, V, size=T)
    P = Problem(logits=z, V=V, targets=t, ce_weight=0.0)
    R0 = oracle.forward(P, nthreads=1)
    P.segment_ids = np.zeros(T, dtype=np.int32)
    P.num_segments = 1
    P.advantages = np.array([A], dtype=np.float32)
    P.old_logprobs = (R0.logp - log_ratio).astype(np.float64)
    P.clip_eps_low, P.clip_eps_high = eps
    return P


def test_gspo_ratio_one():
    A = 0.75
    P = _gspo_problem(0.0, A)
    P.old_logprobs = oracle.forward(P).logp.copy()     # exactly the new log-probs
    R, g = run(P)
    assert R.seam.ratio[0] == 1.0
    assert R.gspo == pytest.approx(-A, rel=1e-15)
    # gradient A/n (p - onehot): rows sum to 0, target entry negative for A > 0
    n = P.logits.shape[0]
    Pce = Problem(logits=P.logits, V=P.V, targets=P.targets)
    _, gce = run(Pce)                                  # (p - onehot) / n
    np.testing.assert_allclose(g, A * gce, rtol=1e-12, atol=1e-17)
    assert R.coef[0] == pytest.approx(A / n)


def test_gspo_clipped_high_positive_adv():
    eps_hi = 0.1
    P = _gspo_problem(0.5, 2.0, eps=(0.1, eps_hi))       # s = e^0.5 > 1.1
    R, g = run(P)
    assert R.seam.ratio[0] == pytest.approx(math.exp(0.5), rel=1e-6)
    assert R.seam.flag[0] == 0
    assert R.gspo == pytest.approx(-(1 + eps_hi) * 2.0, rel=1e-12)
    assert np.all(g == 0.0)


def test_gspo_clipped_low_negative_adv():
    eps_lo = 0.1
    P = _gspo_problem(-0.5, -1.5, eps=(eps_lo, 0.1))    # s = e^-0.5 < 0.9, A < 0
    R, g = run(P)
    assert R.seam.flag[0] == 0
    assert R.gspo == pytest.approx(-(1 - eps_lo) * -1.5, rel=1e-12)
    assert np.all(g == 0.0)


def test_gspo_unclipped_side_flows():
    # s above the band but A < 0: min picks s*A (unclipped), gradient flows
    P = _gspo_problem(0.5, -1.0, eps=(0.1, 0.1))
    R, g = run(P)
    assert R.seam.flag[0] == 1
    s = R.seam.ratio[0]
    assert R.gspo == pytest.approx(s * 1.0, rel=1e-12)
    assert np.abs(g).sum() > 0


def test_gspo_empty_segment_and_padding():
    P = _gspo_problem(0.0, 1.0, T=6)
    P.num_segments = 3
    P.segment_ids = np.array([0, 0, -1, 2, 2, 2], dtype=np.int32)
    P.advantages = np.array([1.0, 5.0, -1.0], dtype=np.float32)
    R = oracle.forward(P)
    assert R.seam.n.tolist() == [2, 0, 3]
    assert R.seam.nonempty == 2
    assert R.seam.loss[1] == 0.0
    assert R.coef[2] == 0.0


# --------------------------------------------------------------------------
# Masking and infinities (torchtitan PR 5661 "Numerics": ignored labels; test
# plan: ignored rows with a -inf fallback logit).
# --------------------------------------------------------------------------
def test_ignored_rows_and_neg_inf():
    V = 6
    z = np.array([[1.0, 2.0, -np.inf, 0.5, 0.0, 3.0],
                  [-np.inf, 1.0, 1.0, 1.0, 1.0, 1.0],
                  [0.0, -np.inf, -np.inf, -np.inf, -np.inf, -np.inf]], dtype=np.float32)
    t = np.array([1, -100, 0])
    mask = np.array([1, 1, 1], dtype=np.uint8)
    P = Problem(logits=z, V=V, targets=t, loss_mask=mask, z_alpha=0.1)
    R, g = run(P)
    assert R.n_active == 2
    assert np.all(g[1] == 0.0) and R.nll[1] == 0.0
    assert g[0, 2] == 0.0                                  # exp(-inf) = 0
    # row 2: every non-target is -inf -> NLL 0, p_t = 1, CE gradient 0
    assert R.nll[2] == 0.0 and R.lse[2] == 0.0
    assert np.all(np.isfinite(g))
    P.loss_mask = np.array([0, 1, 1], dtype=np.uint8)
    R2, g2 = run(P)
    assert R2.n_active == 1 and np.all(g2[0] == 0.0)


def test_single_class_row():
    P = Problem(logits=f32_rows([[4.0], [-2.0]]), V=1, targets=np.array([0, 0]), z_alpha=0.5)
    R, g = run(P)
    assert np.all(R.nll == 0.0)
    np.testing.assert_allclose(R.lse, [4.0, -2.0])
    # only the z-loss gradient survives: 2 a lse * p / N with p = 1
    np.testing.assert_allclose(g[:, 0], [2 * 0.5 * 4.0 / 2, 2 * 0.5 * -2.0 / 2])


# --------------------------------------------------------------------------
# Entropy side output: closed forms and a 50-digit evaluation.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("V", [1, 2, 9, 4096])
def test_entropy_uniform_is_log_v(V):
    z = np.full((3, V), 1.25, dtype=np.float32)
    H = oracle.entropy(Problem(logits=z, V=V, targets=np.zeros(3, dtype=np.int64)))
    np.testing.assert_allclose(H, math.log(V), rtol=1e-12, atol=1e-15)


def test_entropy_two_class_and_brute():
    mp.dps = 50
    rng = np.random.default_rng(11)
    z = rng.normal(0, 3, size=(5, 2)).astype(np.float32)
    H = oracle.entropy(Problem(logits=z, V=2, targets=np.zeros(5, dtype=np.int64)))
    for r in range(5):
        q = 1 / (1 + mpmath.exp(-(mpmath.mpf(float(z[r, 1])) - mpmath.mpf(float(z[r, 0])))))
        hb = -(q * mpmath.log(q) + (1 - q) * mpmath.log(1 - q))
        assert H[r] == pytest.approx(float(hb), rel=1e-12)
    z = rng.normal(0, 2, size=(3, 7)).astype(np.float32)
    H = oracle.entropy(Problem(logits=z, V=7, targets=np.array([0, -100, 3])))
    for r in (0, 2):
        zs = [mpmath.mpf(float(v)) for v in z[r]]
        lse = mpmath.log(mpmath.fsum(mpmath.exp(v) for v in zs))
        h = -mpmath.fsum(mpmath.exp(v - lse) * (v - lse) for v in zs)
        assert H[r] == pytest.approx(float(h), rel=1e-12)
    assert H[1] == 0.0


@pytest.mark.parametrize("margin", [40.0, 60.0, 90.0])
def test_entropy_confident_rows(margin):
    """A row whose largest logit leads by a wide margin: p of that entry is
    within 1e-17 of 1, so -log p must not round to 0 (50-digit reference)."""
    mp.dps = 60
    rng = np.random.default_rng(int(margin))
    z = rng.normal(0, 1, size=(2, 64)).astype(np.float32)
    z[0, 5] = np.float32(margin)
    z[1, :] = 0.0
    z[1, 9] = np.float32(margin)            # two-level row: closed form below
    H = oracle.entropy(Problem(logits=z, V=64, targets=np.zeros(2, dtype=np.int64)))
    zs = [mpmath.mpf(float(v)) for v in z[0]]
    lse = mpmath.log(mpmath.fsum(mpmath.exp(v) for v in zs))
    h = -mpmath.fsum(mpmath.exp(v - lse) * (v - lse) for v in zs)
    assert H[0] == pytest.approx(float(h), rel=1e-12)
    # one entry at m, 63 at 0: q = 63 e^-m / (1 + 63 e^-m) spread evenly over 63
    m = mpmath.mpf(float(margin))
    q = 63 * mpmath.exp(-m) / (1 + 63 * mpmath.exp(-m))
    hb = -((1 - q) * mpmath.log(1 - q) + q * mpmath.log(q / 63))
    assert H[1] == pytest.approx(float(hb), rel=1e-12)


# --------------------------------------------------------------------------
# bf16 inputs.  The workloads hand the oracle bf16 bit patterns; every pin
# above feeds fp32.  A bf16 value is the upper half of the fp32 with the same
# sign, exponent and top seven fraction bits, so each pattern below is written
# out with the value the bf16 format gives it (sign, 8-bit exponent biased by
# 127, 7-bit fraction; subnormals at exponent field 0).  Fed as bf16 bits, the
# oracle must give exactly the results of the same values fed as fp32, whose
# path the pins above fix.
# --------------------------------------------------------------------------
BF16_TABLE = [
    (0x3F80, 1.0),
    (0xC040, -3.0),
    (0x4120, 10.0),
    (0x4049, 3.140625),                 # 2 * (1 + 73/128)
    (0xBF00, -0.5),
    (0x3E80, 0.25),
    (0x4300, 128.0),
    (0xC2F6, -123.0),                   # -64 * (1 + 118/128)
    (0x0001, 2.0 ** -133),              # smallest subnormal: 2^-126 * 1/128
    (0x8001, -(2.0 ** -133)),
    (0x007F, 127 * 2.0 ** -133),        # largest subnormal
    (0x0080, 2.0 ** -126),              # smallest normal
    (0x7F7F, (2.0 - 2.0 ** -7) * 2.0 ** 127),   # largest finite
    (0xFF7F, -(2.0 - 2.0 ** -7) * 2.0 ** 127),
    (0x0000, 0.0),
    (0x8000, -0.0),
    (0xFF80, -math.inf),
]


def test_bf16_bits_decode_table():
    bits = np.array([b for b, _ in BF16_TABLE], dtype=np.uint16)
    vals = np.array([v for _, v in BF16_TABLE], dtype=np.float64)
    got = oracle.bf16_bits_to_f64(bits)
    assert np.array_equal(got, vals)
    assert np.array_equal(np.signbit(got), np.signbit(vals))


def _bf16_pair(rows):
    """The same rows as bf16 bit patterns and as fp32 values."""
    lut = dict(BF16_TABLE)
    b = np.array(rows, dtype=np.uint16)
    f = np.vectorize(lambda x: lut[int(x)])(b).astype(np.float32)
    return b, f


def test_bf16_inputs_match_fp32_bit_for_bit():
    rows = [
        [0x3F80, 0xC040, 0x4120, 0x4049, 0xBF00, 0x3E80, 0x0001, 0xFF80],
        [0x4300, 0xC2F6, 0x0080, 0x007F, 0x8001, 0x0000, 0x8000, 0x3F80],
        [0x7F7F, 0x3F80, 0xC040, 0x0000, 0xFF80, 0x4120, 0xBF00, 0x3E80],
        [0xC040, 0xC2F6, 0xFF7F, 0x4049, 0x3E80, 0x0080, 0x4300, 0xBF00],
    ]
    # teacher: the same patterns in another order (its decode is the same routine)
    teach = [r[3:] + r[:3] for r in rows]
    zb, zf = _bf16_pair(rows)
    ub, uf = _bf16_pair(teach)
    t = np.array([2, 1, 5, 6])
    for kw in (dict(z_alpha=1e-4), dict(z_alpha=1e-4, kl_weight=0.5)):
        use_t = "kl_weight" in kw
        Pb = Problem(logits=zb, V=8, targets=t, teacher=ub if use_t else None, **kw)
        Pf = Problem(logits=zf, V=8, targets=t, teacher=uf if use_t else None, **kw)
        Rb, gb = oracle.forward_backward(Pb, nthreads=1)
        Rf, gf = oracle.forward_backward(Pf, nthreads=1)
        for name in ("nll", "lse", "lse_nt", "kl"):
            assert np.array_equal(getattr(Rb, name), getattr(Rf, name)), name
        assert Rb.total == Rf.total
        assert np.array_equal(gb, gf)
        assert np.array_equal(oracle.entropy(Pb), oracle.entropy(Pf))
    # the value check that makes the comparison mean something: row 0 against
    # its 50-digit definition from the table's values
    mp.dps = 50
    z0 = [mpmath.mpf(v) if math.isfinite(v) else None for v in zf[0].astype(np.float64)]
    terms = [mpmath.exp(v) for j, v in enumerate(z0) if j != 2 and v is not None]
    nll = mpmath.log1p(mpmath.fsum(terms) / mpmath.exp(z0[2]))
    Rb = oracle.forward(Problem(logits=zb[:1], V=8, targets=t[:1]))
    assert Rb.nll[0] == pytest.approx(float(nll), rel=1e-14)
