"""GPU parity for distillation at a temperature tau != 1.

The distillation term is read as the forward KL(q || p^tau) with
q = softmax(u / tau), p^tau = softmax(z / tau) and gradient
kl_weight (p^tau - q) / tau, no tau^2 factor (Fast-LLM PR 552, the list of
combinable losses, names distillation and fixes no more).  The kernel takes tau
through its own instantiation; these tests hold it to the fp64 oracle with the
tolerances of the tau = 1 path (tests/test_gpu_parity.py): losses relative
1e-5, lse and log-probs as there, the per-row KL relative 1e-4 / absolute
2e-6, bf16 gradients within 1 ulp plus the mixed-sign allowance, fp32
gradients absolute 1e-6.  Each tau is an fp32 value, so both sides use the same
temperature.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_util import Case, check_grad, compare_all, grad_to_f64, rel, run, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda", 0)


@pytest.fixture(scope="module")
def handle(dev):
    from lm_head_vocab_gb300 import LMLoss
    h = LMLoss(0, max_T=1 << 16, max_segments=1 << 10)
    yield h
    h.close()


def _case(dev, tau, shape, **params):
    w = workloads.get("ce_z_kl_bf16")
    if shape:
        w = w.with_shape(**shape)
    return Case(replace(w, temperature=float(np.float32(tau)), **params), dev)


def _bits(g):
    return g.view(torch.int16) if g.dtype == torch.bfloat16 else g


SHAPES = [
    dict(T=64, V=262144),             # the distillation workload's vocabulary, cluster of 10
    dict(T=40, V=5001),               # rows not 16-byte aligned, one CTA per row
    dict(T=48, V=32003, ld=32016),    # ragged tail, padded stride
]


@pytest.mark.parametrize("tau", [0.5, 2.0])
@pytest.mark.parametrize("shape", SHAPES, ids=[f"T{s['T']}-V{s['V']}" for s in SHAPES])
def test_tau_parity(dev, handle, tau, shape):
    case = _case(dev, tau, shape)
    R, g_ref, scale = oracle.forward_backward(case.P, with_scale=True)
    inp, out = run(handle, case)
    compare_all(case, out, R, g_ref, f"tau {tau} {shape}", scale)
    # in place gives the same bits as out of place (over the V columns; the
    # padding of a strided row stays as it was)
    V = case.w.V
    inp2 = dict(inp, logits=inp["logits"].clone())
    _, out2 = run(handle, case, grad="inplace", inp=inp2)
    assert torch.equal(_bits(out2.grad[:, :V]), _bits(out.grad[:, :V]))
    assert torch.equal(_bits(out2.grad[:, V:]), _bits(inp["logits"][:, V:]))
    assert torch.equal(out2.loss, out.loss)
    # the same call again gives the same bits
    _, out3 = run(handle, case, inp=inp)
    assert torch.equal(_bits(out3.grad[:, :V]), _bits(out.grad[:, :V]))


@pytest.mark.parametrize("tau", [0.1, 0.25, 4.0, 10.0])
def test_tau_range(dev, handle, tau):
    """Temperatures further from 1: sharp (0.1: p^tau is nearly one-hot on
    rows with a clear maximum) and flat (10: nearly uniform)."""
    case = _case(dev, tau, dict(T=32, V=50000))
    R, g_ref, scale = oracle.forward_backward(case.P, with_scale=True)
    _, out = run(handle, case)
    compare_all(case, out, R, g_ref, f"tau {tau}", scale)


def test_tau_one_unchanged_by_the_tau_path(dev, handle):
    """tau = 1 takes the instantiation without a temperature; a tau one fp32
    ulp away takes the other one and must agree with it to the tolerances."""
    case1 = _case(dev, 1.0, dict(T=32, V=40000))
    caseb = _case(dev, float(np.nextafter(np.float32(1.0), np.float32(2.0))), dict(T=32, V=40000))
    inp = case1.device_inputs()
    _, o1 = run(handle, case1, inp=inp)
    _, ob = run(handle, caseb, inp=inp)
    R, g_ref, scale = oracle.forward_backward(case1.P, with_scale=True)
    compare_all(case1, o1, R, g_ref, "tau 1", scale)
    compare_all(caseb, ob, R, g_ref, "tau 1 + ulp", scale)
    np.testing.assert_allclose(ob.kl.cpu().numpy(), o1.kl.cpu().numpy(), rtol=1e-4, atol=2e-6)


@pytest.mark.parametrize("tau", [0.5, 2.0])
def test_tau_forward_only(dev, handle, tau):
    """Statistics pass alone (no gradient buffer) with masked rows."""
    case = _case(dev, tau, dict(T=96, V=70001))
    R = oracle.forward(case.P)
    inp = case.device_inputs()
    out = handle.forward_backward(inp["logits"], inp["targets"], inp["loss_mask"],
                                  teacher_logits=inp["teacher_logits"], grad=None,
                                  want=("logp", "lse", "kl", "count"), **case.kwargs())
    torch.cuda.synchronize()
    assert handle.device_error() == 0
    compare_all(case, out, R, None, f"forward only, tau {tau}")
    # the fused call agrees to the oracle's tolerance: it runs more threads per
    # CTA, so its partial sums are added in another order, and the KL (formed from
    # terms of about ln V) may move by a few ulps of those terms
    _, full = run(handle, case, inp=inp)
    np.testing.assert_allclose(full.kl.cpu().numpy(), out.kl.cpu().numpy(), rtol=1e-4, atol=2e-6)
    np.testing.assert_allclose(full.loss.cpu().numpy(), out.loss.cpu().numpy(), rtol=1e-5)


def test_tau_mostly_masked_rows(dev, handle):
    """Nine rows in ten ignored: clusters skip most rows."""
    w = workloads.get("ce_z_kl_bf16").with_shape(T=1024, V=30000)
    w = replace(w, temperature=2.0, mask_count=int(0.9 * 1024))
    case = Case(w, dev)
    R, g_ref, scale = oracle.forward_backward(case.P, with_scale=True)
    _, out = run(handle, case)
    assert R.n_active == 1024 - int(0.9 * 1024)
    compare_all(case, out, R, g_ref, "tau 2, 90% masked", scale)


@pytest.mark.parametrize("tau", [0.5, 3.0])
@pytest.mark.parametrize("T,V", [(33, 1027), (16, 50000)])
def test_tau_fp32(dev, handle, tau, T, V):
    rng = np.random.default_rng(T * 7 + V)
    z = (rng.normal(0, 2, size=(T, V))).astype(np.float32)
    u = (z + rng.normal(0, 1, size=(T, V))).astype(np.float32)
    t = rng.integers(0, V, size=T)
    t[3] = -100
    P = oracle.Problem(logits=z, V=V, targets=t, teacher=u, kl_weight=0.5, z_alpha=1e-3,
                       temperature=float(np.float32(tau)))
    out = handle.forward_backward(to_device(z, dev), torch.from_numpy(t).to(dev),
                                  teacher_logits=to_device(u, dev), kl_weight=0.5, z_alpha=1e-3,
                                  temperature=tau, grad="new", want=("logp", "lse", "kl", "count"))
    torch.cuda.synchronize()
    assert handle.device_error() == 0
    R, g_ref = oracle.forward_backward(P)
    assert rel(float(out.loss[0]), R.total) <= 1e-5 and rel(float(out.loss[3]), R.kl_loss) <= 1e-5
    act = R.active.astype(bool)
    np.testing.assert_allclose(out.kl.cpu().numpy()[act], R.kl[act], rtol=1e-4, atol=2e-6)
    check_grad(grad_to_f64(out.grad), g_ref, False, f"fp32 tau {tau}")


def _kl_call(dev, handle, z, u, t, tau, **kw):
    zb = workloads.bf16_round(z.astype(np.float32))
    ub = workloads.bf16_round(u.astype(np.float32))
    args = dict(kl_weight=0.5, z_alpha=1e-3)
    args.update(kw)
    P = oracle.Problem(logits=zb, V=z.shape[1], targets=t, teacher=ub, temperature=float(np.float32(tau)), **args)
    out = handle.forward_backward(to_device(zb, dev), torch.from_numpy(t).to(dev),
                                  teacher_logits=to_device(ub, dev), temperature=tau, grad="new",
                                  want=("logp", "lse", "kl", "count", "entropy"), **args)
    torch.cuda.synchronize()
    assert handle.device_error() == 0
    return P, out


def _check(P, out, what, kl_atol=2e-6):
    """Losses and per-row outputs against the oracle.  The KL slot is held to
    relative 1e-5 or, for a KL near 0, to the per-row absolute bound summed
    over the rows (no fp32 evaluation of a KL of 1e-6 from logits of magnitude
    ten keeps five significant digits)."""
    R, g_ref, scale = oracle.forward_backward(P, with_scale=True)
    assert rel(float(out.loss[0]), R.total) <= 1e-5, (what, float(out.loss[0]), R.total)
    err_kl = abs(float(out.loss[3]) - R.kl_loss)
    assert err_kl <= 1e-5 * abs(R.kl_loss) + kl_atol * R.s_tok * R.n_active, (what, float(out.loss[3]), R.kl_loss)
    act = R.active.astype(bool)
    np.testing.assert_allclose(out.kl.cpu().numpy()[act], R.kl[act], rtol=1e-4, atol=kl_atol)
    np.testing.assert_allclose(out.lse.cpu().numpy()[act], R.lse[act], rtol=2e-6, atol=2e-6)
    _, used = check_grad(grad_to_f64(out.grad), g_ref, True, what, scale)
    assert used <= 1e-3 * g_ref.size, (what, used)
    return R


@pytest.mark.parametrize("tau", [0.5, 1.0, 2.0])
def test_tau_neg_inf_logits(dev, handle, tau):
    """-inf teacher logits (the guarded cross-term sum), -inf student logits
    where the teacher is -inf too (0 log 0 = 0), and a row whose only finite
    logit, student and teacher, is the target's (both distributions one-hot on
    it: KL 0)."""
    rng = np.random.default_rng(21)
    T, V = 8, 9000
    z = rng.normal(0, 2, size=(T, V))
    u = z + rng.normal(0, 1, size=(T, V))
    t = rng.integers(0, V, size=T)
    u[0, 17] = -np.inf
    u[1, :4000] = -np.inf
    z[2, 100:200] = -np.inf
    u[2, 100:200] = -np.inf
    z[3, :] = -np.inf
    u[3, :] = -np.inf
    z[3, t[3]] = 0.5
    u[3, t[3]] = 2.0
    P, out = _kl_call(dev, handle, z, u, t, tau)
    R = _check(P, out, f"-inf logits, tau {tau}")
    kl = out.kl.cpu().numpy()
    assert np.all(np.isfinite(kl))
    assert R.kl[3] == 0.0 and abs(kl[3]) <= 5e-7   # ln Su of a sum that is 1 to within an ulp or two


@pytest.mark.parametrize("tau", [0.5, 1.0, 2.0])
def test_tau_infinite_kl(dev, handle, tau):
    """A student logit of -inf where the teacher's is finite puts no student
    mass where the teacher has some: that row's KL is +inf on both sides, and
    its gradient stays finite (a p + b (p^tau - q) with p^tau = p = 0 there)."""
    rng = np.random.default_rng(23)
    T, V = 4, 5000
    z = rng.normal(0, 2, size=(T, V))
    u = z + rng.normal(0, 1, size=(T, V))
    t = rng.integers(0, V, size=T)
    z[1, (t[1] + 7) % V] = -np.inf
    zb = workloads.bf16_round(z.astype(np.float32))
    ub = workloads.bf16_round(u.astype(np.float32))
    P = oracle.Problem(logits=zb, V=V, targets=t, teacher=ub, kl_weight=0.5, temperature=float(np.float32(tau)))
    out = handle.forward_backward(to_device(zb, dev), torch.from_numpy(t).to(dev),
                                  teacher_logits=to_device(ub, dev), kl_weight=0.5, temperature=tau,
                                  grad="new", want=("kl",))
    torch.cuda.synchronize()
    assert handle.device_error() == 0
    R, g_ref, scale = oracle.forward_backward(P, with_scale=True)
    kl = out.kl.cpu().numpy()
    assert np.isposinf(R.kl[1]) and np.isposinf(kl[1])
    others = [0, 2, 3]
    np.testing.assert_allclose(kl[others], R.kl[others], rtol=1e-4, atol=2e-6)
    assert np.isposinf(float(out.loss[3])) and np.isposinf(float(out.loss[0]))
    check_grad(grad_to_f64(out.grad), g_ref, True, f"infinite KL, tau {tau}", scale)


@pytest.mark.parametrize("tau", [0.5, 2.0])
def test_tau_entropy_unchanged(dev, handle, tau):
    """The entropy output is that of softmax(z), whatever the temperature."""
    rng = np.random.default_rng(5)
    T, V = 24, 30000
    z = rng.normal(0, 2, size=(T, V))
    u = z + rng.normal(0, 1, size=(T, V))
    t = rng.integers(0, V, size=T)
    P, out = _kl_call(dev, handle, z, u, t, tau)
    _check(P, out, f"entropy, tau {tau}")
    act = oracle.active_mask(t, None).astype(bool)
    H = oracle.entropy(P, act)
    h = out.entropy.cpu().numpy().astype(np.float64)
    err = np.abs(h - H)
    assert np.all(err <= 5e-5 * np.abs(H) + 1e-7)


@pytest.mark.parametrize("kw", [dict(ce_weight=-0.5), dict(kl_weight=0.0), dict(kl_weight=-0.3),
                                dict(ce_weight=0.0, z_alpha=0.0)],
                         ids=["ce_negative", "kl_zero", "kl_negative", "kl_only"])
def test_tau_coefficient_signs(dev, handle, kw):
    """Coefficients of either sign: a < 0 or b <= 0 take the general gradient
    form; a = 0 (distillation alone) the fast one with no p term."""
    rng = np.random.default_rng(31)
    T, V = 16, 20000
    z = rng.normal(0, 2, size=(T, V))
    u = z + rng.normal(0, 1, size=(T, V))
    t = rng.integers(0, V, size=T)
    P, out = _kl_call(dev, handle, z, u, t, 2.0, **kw)
    _check(P, out, f"signs {kw}")


def test_tau_confident_rows(dev, handle):
    """Targets that dominate by 20 to 60 nats in the student and by 10 in the
    teacher: both distributions are nearly one-hot on the target, so the KL is
    small (about 1e-6 at tau = 0.5) next to the logits' offsets, and must not
    come from the difference of two large terms."""
    rng = np.random.default_rng(41)
    T, V = 12, 32000
    z = rng.normal(0, 1, size=(T, V))
    u = z + rng.normal(0, 1, size=(T, V))
    t = rng.integers(0, V, size=T)
    for r in range(T):
        z[r, t[r]] = z[r].max() + 20.0 + 40.0 * r / (T - 1)
        u[r, t[r]] = u[r].max() + 10.0
    for tau in (0.5, 1.0, 2.0):
        P, out = _kl_call(dev, handle, z, u, t, tau)
        # KL of 1e-6 and below: held to 5e-7 absolute per row
        _check(P, out, f"confident, tau {tau}", kl_atol=5e-7)


@pytest.mark.parametrize("cluster,threads,nbuf", [(2, 128, 1), (4, 256, 2), (8, 512, 1), (4, 1024, 2), (16, 128, 1)])
def test_tau_launch_shapes(dev, handle, cluster, threads, nbuf):
    """Launch shapes other than the default one at tau = 2 (two staged rows,
    1024 threads, a cluster of 16) agree with the oracle and with the default."""
    case = _case(dev, 2.0, dict(T=40, V=65536))
    inp = case.device_inputs()
    _, ref = run(handle, case, inp=inp)
    handle.set_launch_config(cluster, threads, nbuf)
    try:
        _, out = run(handle, case, inp=inp)
    finally:
        handle.set_launch_config(0, 0, 0)
    R, g_ref, scale = oracle.forward_backward(case.P, with_scale=True)
    compare_all(case, out, R, g_ref, f"tau 2, shape {cluster}x{threads}x{nbuf}", scale)
    np.testing.assert_allclose(out.kl.cpu().numpy(), ref.kl.cpu().numpy(), rtol=1e-5, atol=1e-7)
