"""Parity at the workloads' full sizes, in the launch configuration the benchmark
times (the library's default shape).

Rows are generated on the host in chunks and copied to the device; the oracle
then checks what it can compute one row at a time:
  * ce_z_bf16 (8192 x 32000): every row's gradient and the losses;
  * confident_bf16 (16384 x 128256): the losses over all rows, sampled rows'
    gradients, and the properties of every planted row (NLL > 0, target
    gradient < 0, the row summing to ~0) from the per-row outputs;
  * gspo_z_bf16 (32768 x 151936): the full seam (segment counts and flags
    bit-exact), the losses, and sampled rows' gradients;
  * ce_z_kl_bf16 (65536 x 262144, student and teacher 34 GB each), at the
    workload's temperature 1 and at 2: every row's statistics (log-prob, lse,
    KL) and the five losses against the oracle, run on each chunk of rows as it
    is generated (the host never holds the whole 68 GB), and sampled rows'
    gradients.
Tolerances are the same as in test_gpu_parity.py.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_util import check_grad, grad_to_f64, rel

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

CHUNK = 2048


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda", 0)


def _bf16(a):
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)


def upload(w, dev, keep_host=False, on_chunk=None):
    """Device logits (and teacher) for workload w, generated in row chunks;
    on_chunk(first_row, logits_rows, teacher_rows) sees each chunk on the host."""
    tg, mg = w.targets(), w.margins()
    L = torch.empty((w.T, w.row_stride), dtype=torch.bfloat16, device=dev)
    U = torch.empty_like(L) if w.teacher_sigma is not None else None
    host = np.empty((w.T, w.row_stride), dtype=np.uint16) if keep_host else None
    for a in range(0, w.T, CHUNK):
        n = min(CHUNK, w.T - a)
        x = w.logits_rows(a, n, targets=tg, margins=mg)
        L[a:a + n].copy_(_bf16(x))
        u = w.teacher_rows(a, n, x) if U is not None else None
        if u is not None:
            U[a:a + n].copy_(_bf16(u))
        if host is not None:
            host[a:a + n] = x
        if on_chunk is not None:
            on_chunk(a, x, u)
    return L, U, host


def host_rows(w, rows):
    """The given rows regenerated on the host (logits, teacher)."""
    tg, mg = w.targets(), w.margins()
    xs, us = [], []
    for r in rows:
        x = w.logits_rows(int(r), 1, targets=tg, margins=mg)
        xs.append(x)
        if w.teacher_sigma is not None:
            us.append(w.teacher_rows(int(r), 1, x))
    return np.concatenate(xs), (np.concatenate(us) if us else None)


def sample_rows(w, k=24, seed=5):
    rng = np.random.default_rng(seed)
    rows = {0, w.T - 1}
    m = w.margins()
    rows |= set(np.where(np.isfinite(m))[0][:6].tolist())
    rows |= set(w.masked_rows()[:3].tolist())
    rows |= set(rng.integers(0, w.T, size=k).tolist())
    return np.array(sorted(rows))


def call(dev, w, L, U, grad="inplace", seg=None, S=0, adv=None, old=None):
    from lm_head_vocab_gb300 import LMLoss
    h = LMLoss(0, max_T=w.T, max_segments=max(1, S))
    tg = torch.from_numpy(w.targets()).to(dev)
    mk = None if w.loss_mask() is None else torch.from_numpy(w.loss_mask()).to(dev)
    kw = dict(ce_weight=w.ce_weight, z_alpha=w.z_alpha, kl_weight=w.kl_weight, temperature=w.temperature,
              reduction="sum" if w.reduction == "sum_active" else "token_mean", denominator=w.denominator())
    if seg is not None:
        kw.update(segment_ids=seg, num_segments=S, advantages=adv, old_logprobs=old,
                  clip_eps_low=w.clip_eps_low, clip_eps_high=w.clip_eps_high)
    out = h.forward_backward(L, tg, mk, teacher_logits=U, grad=grad,
                             want=("logp", "lse", "kl", "count", "seg"), **kw)
    torch.cuda.synchronize()
    assert h.device_error() == 0
    h.close()
    return out


def sampled_oracle(w, rows, coef=None):
    """Oracle statistics and gradient of the sampled rows, with the full batch's scale."""
    x, u = host_rows(w, rows)
    t = w.targets()[rows]
    m = None if w.loss_mask() is None else w.loss_mask()[rows]
    n_act = w.n_active()
    P = oracle.Problem(logits=x, V=w.V, targets=t, loss_mask=m, ce_weight=w.ce_weight, z_alpha=w.z_alpha,
                       teacher=u, kl_weight=w.kl_weight, temperature=w.temperature,
                       reduction=oracle.REDUCE_SUM,
                       denominator=float(w.denominator() if w.reduction == "sum_active" else n_act))
    R = oracle.forward(P)
    if coef is not None:
        R.coef = coef
    g, gs = oracle.grad_rows(P, R, with_scale=True)
    return R, g, gs


def check_rows(out, w, rows, R, g, gs):
    act = R.active.astype(bool)
    logp = out.logp.cpu().numpy()[rows].astype(np.float64)
    lse = out.lse.cpu().numpy()[rows].astype(np.float64)
    np.testing.assert_allclose(lse[act], R.lse[act], rtol=2e-6, atol=2e-6)
    np.testing.assert_allclose(logp[act], R.logp[act], rtol=2e-5, atol=1e-6)
    if out.kl is not None:
        np.testing.assert_allclose(out.kl.cpu().numpy()[rows][act], R.kl[act], rtol=1e-4, atol=2e-6)
    gg = grad_to_f64(out.grad[torch.from_numpy(rows).to(out.grad.device), :w.V])
    # the mixed-sign allowance only with a teacher
    check_grad(gg, g, True, w.name, gs if out.kl is not None else None)


def test_ce_z_bf16_full(dev):
    w = workloads.get("ce_z_bf16")
    L, U, host = upload(w, dev, keep_host=True)
    out = call(dev, w, L, U, grad="inplace")
    P = oracle.Problem(logits=host, V=w.V, targets=w.targets(), z_alpha=w.z_alpha,
                       reduction=oracle.REDUCE_SUM, denominator=w.denominator())
    R, g, gs = oracle.forward_backward(P, with_scale=True)
    loss = out.loss.cpu().numpy()
    assert rel(float(loss[0]), R.total) <= 1e-5
    assert rel(float(loss[1]), R.ce) <= 1e-5 and rel(float(loss[2]), R.z) <= 1e-5
    assert int(out.count[0]) == R.n_active
    check_grad(grad_to_f64(out.grad), g, True, "ce_z_bf16 full")


def test_confident_bf16_full(dev):
    w = workloads.get("confident_bf16")
    L, U, host = upload(w, dev, keep_host=True)
    out = call(dev, w, L, U, grad="inplace")
    R = oracle.forward(oracle.Problem(logits=host, V=w.V, targets=w.targets()))
    assert rel(float(out.loss[0]), R.total) <= 1e-5
    logp = out.logp.cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(logp, R.logp, rtol=2e-5, atol=1e-6)
    # every planted row: NLL > 0 (no collapse), target gradient < 0, row sums to ~0
    m = w.margins()
    planted = np.where(np.isfinite(m))[0]
    assert np.all(logp[planted] < 0.0)
    t = torch.from_numpy(w.targets()).to(dev)
    pr = torch.from_numpy(planted).to(dev)
    gt = out.grad[pr, t[pr]].float()
    assert bool(torch.all(gt < 0))
    rows_g = out.grad[pr].float()
    assert bool(torch.all(rows_g.sum(1).abs() <= 2.0 ** -8 * rows_g.abs().sum(1)))
    rows = sample_rows(w)
    Rs, g, gs = sampled_oracle(w, rows)
    check_rows(out, w, rows, Rs, g, gs)


def test_gspo_z_bf16_full(dev):
    w = workloads.get("gspo_z_bf16")
    L, U, host = upload(w, dev, keep_host=True)
    seg, S, adv = w.segments()
    t = w.targets()
    R0 = oracle.forward(oracle.Problem(logits=host, V=w.V, targets=t))
    old = (R0.logp + w.old_logp_noise()).astype(np.float32)
    P = oracle.Problem(logits=host, V=w.V, targets=t, ce_weight=w.ce_weight, z_alpha=w.z_alpha,
                       segment_ids=seg, num_segments=S, advantages=adv, old_logprobs=old,
                       clip_eps_low=w.clip_eps_low, clip_eps_high=w.clip_eps_high)
    R = oracle.forward(P)
    out = call(dev, w, L, U, grad="inplace", seg=torch.from_numpy(seg).to(dev), S=S,
               adv=torch.from_numpy(adv).to(dev), old=torch.from_numpy(old).to(dev))
    loss = out.loss.cpu().numpy()
    for k, ref in enumerate([R.total, R.ce, R.z, R.kl_loss, R.gspo]):
        if ref != 0.0:
            assert rel(float(loss[k]), ref) <= 1e-5, (k, loss[k], ref)
    assert np.array_equal(out.seg_count.cpu().numpy(), R.seam.n)
    s = R.seam.ratio
    lo, hi = 1 - w.clip_eps_low, 1 + w.clip_eps_high
    amb = (np.abs(s - lo) < 1e-6 * lo) | (np.abs(s - hi) < 1e-6 * hi)
    assert np.array_equal(out.seg_flag.cpu().numpy()[~amb], R.seam.flag[~amb])
    rows = sample_rows(w)
    Psub = oracle.Problem(logits=host[rows], V=w.V, targets=t[rows], ce_weight=w.ce_weight, z_alpha=w.z_alpha,
                          reduction=oracle.REDUCE_SUM, denominator=float(R.n_active))
    Rs = oracle.forward(Psub)
    Rs.coef = R.coef[rows]
    g, gs = oracle.grad_rows(Psub, Rs, with_scale=True)
    check_rows(out, w, rows, Rs, g, gs)


@pytest.mark.parametrize("tau", [1.0, 2.0])
def test_ce_z_kl_bf16_full(dev, tau):
    """At the workload's own temperature 1, and at 2 (the other instantiation)."""
    from dataclasses import replace
    w = replace(workloads.get("ce_z_kl_bf16"), temperature=tau)
    tg, mk = w.targets(), w.loss_mask()
    nll, lse, kl = (np.zeros(w.T) for _ in range(3))
    act = oracle.active_mask(tg, mk).astype(bool)

    def oracle_chunk(a, x, u):
        # the oracle's per-row statistics of this chunk, from the same host bits
        n = len(x)
        R = oracle.forward(oracle.Problem(logits=x, V=w.V, targets=tg[a:a + n], loss_mask=mk[a:a + n],
                                          z_alpha=w.z_alpha, teacher=u, kl_weight=w.kl_weight,
                                          temperature=w.temperature))
        nll[a:a + n], lse[a:a + n], kl[a:a + n] = R.nll, R.lse, R.kl

    L, U, _ = upload(w, dev, on_chunk=oracle_chunk)
    out = call(dev, w, L, U, grad="inplace")
    del U
    # the five losses: token mean over the active rows of each term, from the
    # oracle's fp64 per-row values
    n = int(act.sum())
    assert int(out.count[0]) == n == w.n_active()
    ce = float(np.sum(nll)) / n
    z = w.z_alpha * float(np.sum(lse * lse)) / n
    klm = float(np.sum(kl)) / n
    ref = [w.ce_weight * ce + z + w.kl_weight * klm, ce, z, klm, 0.0]
    loss = out.loss.cpu().numpy().astype(np.float64)
    for k in range(4):
        assert rel(loss[k], ref[k]) <= 1e-5, (k, loss[k], ref[k])
    assert loss[4] == 0.0
    # every row's statistics
    logp_g = out.logp.cpu().numpy().astype(np.float64)
    lse_g = out.lse.cpu().numpy().astype(np.float64)
    kl_g = out.kl.cpu().numpy().astype(np.float64)
    assert np.all(logp_g[~act] == 0.0) and np.all(lse_g[~act] == 0.0) and np.all(kl_g[~act] == 0.0)
    np.testing.assert_allclose(lse_g[act], lse[act], rtol=2e-6, atol=2e-6)
    np.testing.assert_allclose(logp_g[act], -nll[act], rtol=2e-5, atol=1e-6)
    np.testing.assert_allclose(kl_g[act], kl[act], rtol=1e-4, atol=2e-6)
    # sampled rows' gradients
    rows = sample_rows(w)
    Rs, g, gs = sampled_oracle(w, rows)
    check_rows(out, w, rows, Rs, g, gs)
