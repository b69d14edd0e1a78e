"""GPU parity for vocabulary-split rows: a row's columns spread over K shards
(separate [T, V_k] matrices), statistics per shard, one merge, gradient per
shard.  The merged losses, log-probs and lse, and the shards' gradients laid
side by side, are compared with the fp64 oracle of the whole row, with the
tolerances of test_gpu_parity.py."""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_util import check_grad, grad_to_f64, rel, to_device

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
    h = LMLoss(0, max_T=1 << 14, max_segments=1)
    yield h
    h.close()


def run_shards(handle, dev, x, targets, mask, cuts, dtype, z_alpha, reduction="token_mean", denominator=1.0):
    """Split host logits x [T, V] at `cuts`, run the three shard steps, return
    (merged outputs, gradient of the whole row as float64)."""
    T, V = x.shape
    bounds = [0] + list(cuts) + [V]
    tg = torch.from_numpy(targets).to(dev)
    mk = None if mask is None else torch.from_numpy(mask).to(dev)
    shards = []
    for k in range(len(bounds) - 1):
        a, b = bounds[k], bounds[k + 1]
        shards.append((a, to_device(np.ascontiguousarray(x[:, a:b]), dev)))
    parts = [handle.shard_stats(z, tg, mk, v0=v0, V_total=V) for v0, z in shards]
    out = handle.shard_merge(parts, tg, mk, V_total=V, z_alpha=z_alpha, reduction=reduction,
                             denominator=denominator)
    grads = [handle.shard_grad(z, tg, mk, v0=v0, V_total=V, z_alpha=z_alpha, reduction=reduction,
                               denominator=denominator) for v0, z in shards]
    torch.cuda.synchronize()
    g = np.concatenate([grad_to_f64(gk) for gk in grads], axis=1)
    return out, g


CASES = [
    ("ce_z_bf16", dict(T=96, V=50021), [20000], 1e-4),
    ("ce_z_bf16", dict(T=64, V=32000), [7, 16000, 31990], 1e-4),       # a 7-wide shard, a 10-wide one
    ("confident_bf16", dict(T=64, V=128256), [64128], 0.0),            # two V_local halves
    ("ce_fp32_small", None, [300, 301], 0.0),                         # a one-column shard
]


@pytest.mark.parametrize("name,shape,cuts,alpha", CASES, ids=[f"{c[0]}-{c[2]}" for c in CASES])
def test_shards_match_whole_row_oracle(dev, handle, name, shape, cuts, alpha):
    w = workloads.get(name)
    if shape:
        w = w.with_shape(**shape)
    x = w.logits_rows(0, w.T)
    t = w.targets()
    m = w.loss_mask()
    bf16 = w.dtype == "bf16"
    P = oracle.Problem(logits=x, V=w.V, targets=t, loss_mask=m, z_alpha=alpha)
    R, g_ref = oracle.forward_backward(P)
    out, g = run_shards(handle, dev, x, t, m, cuts, w.dtype, alpha)
    assert handle.device_error() == 0
    loss = out.loss.cpu().numpy().astype(np.float64)
    assert rel(loss[0], R.total) <= 1e-5 and rel(loss[1], R.ce) <= 1e-5
    if alpha:
        assert rel(loss[2], R.z) <= 1e-5
    assert loss[3] == 0.0 and loss[4] == 0.0
    assert int(out.count[0]) == R.n_active
    act = R.active.astype(bool)
    logp = out.logp.cpu().numpy().astype(np.float64)
    lse = out.lse.cpu().numpy().astype(np.float64)
    assert np.all(logp[~act] == 0.0) and np.all(lse[~act] == 0.0)
    np.testing.assert_allclose(lse[act], R.lse[act], rtol=2e-6, atol=2e-6)
    np.testing.assert_allclose(logp[act], R.logp[act], rtol=2e-5, atol=1e-6)
    check_grad(g, g_ref, bf16, f"{name} shards {cuts}")   # no teacher: no mixed-sign allowance


def test_shards_agree_with_whole_row_call(dev, handle):
    """The shard path and the one-call path give the same losses to rounding and
    gradients within one bf16 ulp of each other."""
    w = workloads.get("ce_z_bf16").with_shape(T=128, V=40000)
    x = w.logits_rows(0, w.T)
    t = w.targets()
    out, g = run_shards(handle, dev, x, t, None, [13000, 26000], "bf16", 1e-4, reduction="sum",
                        denominator=float(w.n_active()))
    whole = handle.forward_backward(to_device(x, dev), torch.from_numpy(t).to(dev), grad="new",
                                    z_alpha=1e-4, reduction="sum", denominator=float(w.n_active()))
    torch.cuda.synchronize()
    assert rel(float(out.loss[0]), float(whole.loss[0])) <= 1e-6
    gw = grad_to_f64(whole.grad)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(gw), 2.0 ** -126))) - 7)
    assert np.all(np.abs(g - gw) <= ulp)


def test_confident_row_target_in_one_shard(dev, handle):
    """A row whose target leads every other column by 30 nats: the shard holding
    it and the shards without it merge to NLL = softplus(lse_nt - z_t) > 0 (no
    collapse), and the target gradient stays negative."""
    rng = np.random.default_rng(4)
    T, V = 4, 9000
    z = rng.normal(0, 2, size=(T, V)).astype(np.float32)
    t = np.array([10, 4500, 8999, 3])
    for r in range(T):
        z[r, t[r]] = z[r].max() + 30.0
    x = workloads.bf16_round(z)
    P = oracle.Problem(logits=x, V=V, targets=t)
    R, g_ref = oracle.forward_backward(P)
    out, g = run_shards(handle, dev, x, t, None, [3000, 6000], "bf16", 0.0)
    logp = out.logp.cpu().numpy().astype(np.float64)
    assert np.all(logp < 0.0)
    np.testing.assert_allclose(logp, R.logp, rtol=2e-5, atol=1e-12)
    assert all(g[r, t[r]] < 0 for r in range(T))
    check_grad(g, g_ref, True, "confident shards")


def test_shard_target_out_of_range_sets_error(dev, handle):
    from lm_head_vocab_gb300._lib import LMLOSS_ERR_BAD_TARGET
    x = np.zeros((3, 100), dtype=np.float32)
    t = np.array([1, 100, 50])
    run_shards(handle, dev, x, t, None, [40], "fp32", 0.0)
    assert handle.device_error() == LMLOSS_ERR_BAD_TARGET


def test_shard_calls_reject_teacher(dev, handle):
    from lm_head_vocab_gb300 import _lib
    from lm_head_vocab_gb300._lib import LMLossError
    z = torch.zeros((2, 64), dtype=torch.bfloat16, device=dev)
    tg = torch.tensor([1, 2], device=dev)
    a, _out, _keep = handle.build_args(z, tg, teacher_logits=z.clone(), kl_weight=0.5, grad=None, want=())
    part = torch.empty((2, 4), device=dev)
    st = _lib.load().lmloss_shard_stats(handle.handle, a, 0, 64, part.data_ptr(), 0)
    assert st == _lib.LMLOSS_ERR_UNSUPPORTED
    with pytest.raises(LMLossError):
        handle.shard_stats(z, tg, v0=10, V_total=64)            # shard past the vocabulary
