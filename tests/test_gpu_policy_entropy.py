"""GPU parity for the per-token entropy output and the token-level GRPO term.

Entropy: H_r = -sum_j p_j log p_j of softmax(z_r), against the oracle's fp64
sum.  The kernel forms it as p_t NLL + p_nt (ln S - B/S + softplus(-d)), whose
terms are all non-negative, so the bound is relative: 5e-5 of H plus 1e-7
absolute (fp32 sums of about log V in magnitude).

GRPO: per-token advantages and old log-probs, clipped surrogate
-min(rho A, clamp(rho, 1-eps_lo, 1+eps_hi) A).  Whether a token's gradient
flows is an fp32 decision in the kernel and an fp64 one in the oracle; rows
whose ratio lies within 1e-5 of a clip bound may take either branch and are
left out of the gradient comparison (the loss is continuous there).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_util import Case, check_grad, grad_to_f64, rel, to_device

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
    h = LMLoss(0, max_T=1 << 16, max_segments=1 << 12)
    yield h
    h.close()


ENTROPY_CASES = [
    ("ce_fp32_small", None),
    ("ce_z_bf16", dict(T=256, V=32000)),
    ("ce_z_bf16", dict(T=64, V=32003, ld=32016)),
    ("confident_bf16", dict(T=128, V=128256)),
    ("ce_z_kl_bf16", dict(T=64, V=262144)),
    ("ce_z_kl_bf16", dict(T=40, V=5001)),
]


def _case(dev, name, shape):
    w = workloads.get(name)
    if shape:
        w = w.with_shape(**shape)
    return Case(w, dev)


def _call(handle, case, inp, want, grad="new", **extra):
    kw = case.kwargs()
    kw.update(extra)
    out = handle.forward_backward(inp["logits"], inp["targets"], inp["loss_mask"],
                                  teacher_logits=inp["teacher_logits"], grad=grad, want=want, **kw)
    torch.cuda.synchronize()
    assert handle.device_error() == 0
    return out


def check_entropy(h_gpu, h_ref, act, what):
    assert np.all(h_gpu[~act] == 0.0), what
    assert np.all(np.isfinite(h_gpu[act])), what
    err = np.abs(h_gpu[act] - h_ref[act])
    bound = 5e-5 * np.abs(h_ref[act]) + 1e-7
    assert np.all(err <= bound), f"{what}: worst {float(np.max(err / bound)):.2f} of the bound"


@pytest.mark.parametrize("name,shape", ENTROPY_CASES, ids=[f"{n}-{s}" for n, s in ENTROPY_CASES])
def test_entropy_parity(dev, handle, name, shape):
    case = _case(dev, name, shape)
    inp = case.device_inputs()
    out = _call(handle, case, inp, want=("logp", "lse", "entropy"))
    act = oracle.active_mask(case.P.targets, case.P.loss_mask).astype(bool)
    H = oracle.entropy(case.P, act)
    check_entropy(out.entropy.cpu().numpy().astype(np.float64), H, act, f"{name} {shape}")
    # asking for the entropy changes no other output
    base = _call(handle, case, inp, want=("logp", "lse"))
    assert torch.equal(out.loss, base.loss)
    assert torch.equal(out.logp, base.logp) and torch.equal(out.lse, base.lse)
    V = case.w.V   # columns past V of a padded row are not written
    g1 = out.grad[:, :V].view(torch.int16) if out.grad.dtype == torch.bfloat16 else out.grad[:, :V]
    g0 = base.grad[:, :V].view(torch.int16) if base.grad.dtype == torch.bfloat16 else base.grad[:, :V]
    assert torch.equal(g1, g0)


def test_entropy_forward_only_and_neg_inf(dev, handle):
    V = 300
    z = np.random.default_rng(3).normal(size=(5, V)) * 3.0
    z[0, 7] = -np.inf            # one masked vocabulary entry
    z[1, :] = -np.inf            # an ignored row
    z[2, 1:] = -np.inf           # all mass on the target: H = 0
    z[2, 0] = 1.0
    z[3, 10] = 60.0              # a confident row: H tiny, no cancellation allowed
    z[4, :150] = -np.inf         # half the vocabulary masked
    t = np.array([3, -100, 0, 10, 200])
    x = z.astype(np.float32)
    P = oracle.Problem(logits=x, V=V, targets=t)
    act = oracle.active_mask(t, None).astype(bool)
    H = oracle.entropy(P, act)
    logits = to_device(x, dev)
    out = handle.forward_backward(logits, torch.from_numpy(t).to(dev), grad=None, want=("entropy",))
    torch.cuda.synchronize()
    assert handle.device_error() == 0
    h = out.entropy.cpu().numpy().astype(np.float64)
    assert h[2] == 0.0
    check_entropy(h, H, act, "-inf and confident rows")
    assert 0.0 < h[3] < 1e-18          # about 1e-20 here


def _grpo_inputs(case, eps=(0.2, 0.28), sigma=0.25, seed=11):
    """Token advantages: the segment's advantage on each of its tokens (0 on
    padding), the usual GRPO broadcast; old log-probs: the oracle's log-prob
    plus seeded noise, so that a share of tokens fall outside the clip range."""
    w = case.w
    seg, S, adv = w.segments()
    tok_adv = np.where(seg >= 0, adv[np.maximum(seg, 0)], 0.0).astype(np.float32)
    R0 = oracle.forward(oracle.Problem(logits=case.x, V=w.V, targets=case.targets, loss_mask=case.mask))
    noise = np.random.default_rng(seed).normal(0.0, sigma, size=w.T)
    old = (R0.logp + noise).astype(np.float32)
    P = oracle.Problem(logits=case.x, V=w.V, targets=case.targets, loss_mask=case.mask,
                       ce_weight=w.ce_weight, z_alpha=w.z_alpha,
                       reduction=case.P.reduction, denominator=case.P.denominator,
                       token_advantages=tok_adv, old_logprobs=old,
                       clip_eps_low=eps[0], clip_eps_high=eps[1])
    return P, tok_adv, old


def _policy_mag(P, R):
    """s_tok * sum |min(rho A, clamp(rho) A)|: the scale of the policy sum's rounding."""
    act = R.active.astype(bool)
    rho = np.exp(R.logp - P.old_logprobs.astype(np.float64))
    A = P.token_advantages.astype(np.float64)
    lo, hi = 1 - P.clip_eps_low, 1 + P.clip_eps_high
    return R.s_tok * float(np.sum(np.abs(np.minimum(rho * A, np.clip(rho, lo, hi) * A)[act])))


@pytest.mark.parametrize("reduction", ["token_mean", "sum"])
def test_grpo_parity(dev, handle, reduction):
    w = workloads.get("gspo_z_bf16").with_shape(T=1024, V=151936, packed_len=256)
    case = Case(w, dev)
    P, tok_adv, old = _grpo_inputs(case)
    if reduction == "sum":
        P.reduction, P.denominator = oracle.REDUCE_SUM, 3000.0
    else:
        P.reduction, P.denominator = oracle.REDUCE_TOKEN_MEAN, 1.0
    R, g_ref = oracle.forward_backward(P)
    inp = case.device_inputs()
    out = handle.forward_backward(
        inp["logits"], inp["targets"], inp["loss_mask"], ce_weight=w.ce_weight, z_alpha=w.z_alpha,
        token_advantages=torch.from_numpy(tok_adv).to(dev), old_logprobs=torch.from_numpy(old).to(dev),
        clip_eps_low=P.clip_eps_low, clip_eps_high=P.clip_eps_high, reduction=reduction,
        denominator=P.denominator, grad="new", want=("logp", "lse", "count"))
    torch.cuda.synchronize()
    assert handle.device_error() == 0
    act = R.active.astype(bool)
    rho = np.exp(R.logp - old.astype(np.float64))
    lo, hi = 1 - P.clip_eps_low, 1 + P.clip_eps_high
    clipped = act & ((rho < lo) | (rho > hi))
    assert 0.05 * act.sum() < clipped.sum() < 0.6 * act.sum()    # both branches are exercised
    loss = out.loss.cpu().numpy().astype(np.float64)
    # the policy sum mixes signs: bound its error by the summed magnitudes
    mag = _policy_mag(P, R)
    assert abs(loss[4] - R.gspo) <= 1e-5 * mag, (loss[4], R.gspo, mag)
    assert abs(loss[0] - R.total) <= 1e-5 * (abs(R.total) + mag)
    assert rel(loss[1], R.ce) <= 1e-5 and rel(loss[2], R.z) <= 1e-5
    amb = act & ((np.abs(rho - lo) < 1e-5 * lo) | (np.abs(rho - hi) < 1e-5 * hi))
    keep = ~amb
    check_grad(grad_to_f64(out.grad[torch.from_numpy(np.where(keep)[0]).to(dev)]), g_ref[keep], True, "grpo")


@pytest.mark.parametrize("tau", [1.0, 2.0])
def test_grpo_with_teacher(dev, handle, tau):
    """The token-level policy term together with distillation (at temperature
    1 and 2): the policy coefficient of a row joins the cross-entropy's in the
    gradient, the teacher's term stays as it is."""
    from dataclasses import replace
    w = replace(workloads.get("ce_z_kl_bf16").with_shape(T=256, V=30011), temperature=tau)
    case = Case(w, dev)
    rng = np.random.default_rng(31)
    tok_adv = rng.normal(0, 1, size=w.T).astype(np.float32)
    R0 = oracle.forward(oracle.Problem(logits=case.x, V=w.V, targets=case.targets, loss_mask=case.mask))
    old = (R0.logp + rng.normal(0.0, 0.25, size=w.T)).astype(np.float32)
    P = oracle.Problem(logits=case.x, V=w.V, targets=case.targets, loss_mask=case.mask, ce_weight=w.ce_weight,
                       z_alpha=w.z_alpha, teacher=case.u, kl_weight=w.kl_weight, temperature=w.temperature,
                       token_advantages=tok_adv, old_logprobs=old, clip_eps_low=0.2, clip_eps_high=0.28)
    R, g_ref, scale = oracle.forward_backward(P, with_scale=True)
    inp = case.device_inputs()
    out = handle.forward_backward(
        inp["logits"], inp["targets"], inp["loss_mask"], teacher_logits=inp["teacher_logits"],
        ce_weight=w.ce_weight, z_alpha=w.z_alpha, kl_weight=w.kl_weight, temperature=w.temperature,
        token_advantages=torch.from_numpy(tok_adv).to(dev), old_logprobs=torch.from_numpy(old).to(dev),
        clip_eps_low=0.2, clip_eps_high=0.28, grad="new", want=("logp", "lse", "kl", "count"))
    torch.cuda.synchronize()
    assert handle.device_error() == 0
    act = R.active.astype(bool)
    rho = np.exp(R.logp - old.astype(np.float64))
    lo, hi = 0.8, 1.28
    clipped = act & ((rho < lo) | (rho > hi))
    assert 0.05 * act.sum() < clipped.sum() < 0.8 * act.sum()    # both branches are exercised
    loss = out.loss.cpu().numpy().astype(np.float64)
    mag = _policy_mag(P, R)
    assert abs(loss[4] - R.gspo) <= 1e-5 * mag, (loss[4], R.gspo, mag)
    assert abs(loss[0] - R.total) <= 1e-5 * (abs(R.total) + mag)
    assert rel(loss[1], R.ce) <= 1e-5 and rel(loss[2], R.z) <= 1e-5 and rel(loss[3], R.kl_loss) <= 1e-5
    np.testing.assert_allclose(out.kl.cpu().numpy()[act], R.kl[act], rtol=1e-4, atol=2e-6)
    amb = act & ((np.abs(rho - lo) < 1e-5 * lo) | (np.abs(rho - hi) < 1e-5 * hi))
    keep = np.where(~amb)[0]
    check_grad(grad_to_f64(out.grad[torch.from_numpy(keep).to(dev)]), g_ref[keep], True,
               f"grpo with teacher, tau {tau}", scale[keep])


def test_grpo_forward_only_matches_fused(dev, handle):
    """The policy loss from the statistics-only launch equals the fused one."""
    w = workloads.get("gspo_z_bf16").with_shape(T=512, V=40000, packed_len=128)
    case = Case(w, dev)
    P, tok_adv, old = _grpo_inputs(case, seed=12)
    inp = case.device_inputs()
    kw = dict(ce_weight=w.ce_weight, z_alpha=w.z_alpha, token_advantages=torch.from_numpy(tok_adv).to(dev),
              old_logprobs=torch.from_numpy(old).to(dev), clip_eps_low=P.clip_eps_low,
              clip_eps_high=P.clip_eps_high, want=("logp",))
    a = handle.forward_backward(inp["logits"], inp["targets"], inp["loss_mask"], grad="new", **kw)
    b = handle.forward_backward(inp["logits"], inp["targets"], inp["loss_mask"], grad=None, **kw)
    torch.cuda.synchronize()
    assert handle.device_error() == 0
    assert torch.equal(a.loss, b.loss) and torch.equal(a.logp, b.logp)
    R = oracle.forward(P)
    assert abs(float(a.loss[4]) - R.gspo) <= 1e-5 * _policy_mag(P, R)


def test_grpo_with_gspo_is_rejected(dev, handle):
    from lm_head_vocab_gb300._lib import LMLossError
    z = torch.zeros((4, 64), dtype=torch.bfloat16, device=dev)
    t = torch.tensor([1, 2, 3, 4], device=dev)
    one = torch.ones(4, device=dev)
    with pytest.raises(LMLossError):
        handle.forward_backward(z, t, segment_ids=torch.zeros(4, dtype=torch.int32, device=dev), num_segments=1,
                                advantages=torch.ones(1, device=dev), old_logprobs=one,
                                token_advantages=one, grad="new")
