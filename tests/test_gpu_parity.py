"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on the
same seeded inputs, element by element.

Tolerances (from the arithmetic, fixed here):
  losses            relative 1e-5;
  bf16 gradients    within 1 bf16 ulp of the fp64 value (a value below 2^-126
                    may flush to 0); where the definition sums terms of mixed
                    sign (distillation's a p - b q; at the target column the CE
                    or policy term against the z / KL term), plus 2^-17 of the
                    terms' summed magnitude (see tests/gpu_util.py), used by at
                    most 1e-3 of the elements;
  fp32 gradients    absolute 1e-6;
  integer outputs   bit-exact (active count, segment counts, segment flags
                    away from a clip bound, masked rows exactly 0).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_util import WANT, Case, check_grad, compare_all, grad_to_f64, rel, run, to_device

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
    h = LMLoss(0, max_T=1 << 17, max_segments=1 << 14)
    yield h
    h.close()


SMALL = [
    ("ce_fp32_small", None),
    ("ce_z_bf16", dict(T=256, V=32000)),
    ("ce_z_bf16", dict(T=97, V=32003)),            # rows not 16-byte aligned
    ("ce_z_bf16", dict(T=64, V=32003, ld=32016)),  # ragged tail, padded stride
    ("confident_bf16", dict(T=128, V=128256)),
    ("gspo_z_bf16", dict(T=1024, V=151936, packed_len=256)),
    ("ce_z_kl_bf16", dict(T=64, V=262144)),
    ("ce_z_kl_bf16", dict(T=40, V=5001)),
    ("ce_fp32_small", dict(T=33, V=1027)),          # fp32, unaligned rows
]


def _case(dev, name, shape):
    w = workloads.get(name)
    if shape:
        w = w.with_shape(**shape)
    return Case(w, dev)


@pytest.mark.parametrize("name,shape", SMALL, ids=[f"{n}-{s}" for n, s in SMALL])
def test_parity_small(dev, handle, name, shape):
    case = _case(dev, name, shape)
    R, g_ref, scale = oracle.forward_backward(case.P, with_scale=True)
    inp, out = run(handle, case)
    compare_all(case, out, R, g_ref, f"{name} {shape}", scale)
    if case.w.has_gspo:
        sc = out.seg_count.cpu().numpy()
        assert np.array_equal(sc, R.seam.n)
        assert out.count.cpu().numpy()[1] == R.seam.nonempty
        flag = out.seg_flag.cpu().numpy()
        s = R.seam.ratio
        lo, hi = 1 - case.w.clip_eps_low, 1 + case.w.clip_eps_high
        amb = (np.abs(s - lo) < 1e-6 * lo) | (np.abs(s - hi) < 1e-6 * hi)
        assert np.array_equal(flag[~amb], R.seam.flag[~amb])
        # the ratio inherits the fp32 log-probs' error (about 1e-6 of |logp| ~ 12)
        np.testing.assert_allclose(out.seg_ratio.cpu().numpy()[R.seam.n > 0], s[R.seam.n > 0], rtol=2e-5)
    # in place gives the same bits as out of place over the V columns, and leaves
    # the padding of a strided row as it was
    logits2 = inp["logits"].clone()
    inp2 = dict(inp, logits=logits2)
    _, out2 = run(handle, case, grad="inplace", inp=inp2)
    V = case.w.V
    bits = (lambda g: g.view(torch.int16)) if out.grad.dtype == torch.bfloat16 else (lambda g: g)
    assert torch.equal(bits(out2.grad[:, :V]), bits(out.grad[:, :V]))
    assert torch.equal(bits(out2.grad[:, V:]), bits(inp["logits"][:, V:]))
    assert torch.equal(out2.loss, out.loss)


def test_confident_rows_properties(dev, handle):
    """Planted margins 15..40: NLL > 0, target gradient < 0, rows sum to ~0."""
    case = _case(dev, "confident_bf16", dict(T=256, V=128256))
    _, out = run(handle, case)
    m = case.w.margins()
    planted = np.where(np.isfinite(m))[0]
    assert len(planted) > 50
    logp = out.logp.cpu().numpy()
    g = grad_to_f64(out.grad)
    t = case.targets
    for r in planted:
        assert logp[r] < 0.0
        assert g[r, t[r]] < 0.0
        assert abs(g[r].sum()) <= 2.0 ** -8 * np.abs(g[r]).sum()


def test_kl_allowance_is_rare(dev, handle):
    """The distillation gradient needs the cancellation allowance on only a tiny
    fraction of elements; everything else is within 1 bf16 ulp."""
    case = _case(dev, "ce_z_kl_bf16", dict(T=32, V=262144))
    R, g_ref, scale = oracle.forward_backward(case.P, with_scale=True)
    _, out = run(handle, case)
    worst, used = check_grad(grad_to_f64(out.grad), g_ref, True, "kl", scale)
    assert used <= 1e-3 * g_ref.size, used


def test_deterministic_repeat(dev, handle):
    case = _case(dev, "ce_z_kl_bf16", dict(T=48, V=70000))
    inp = case.device_inputs()
    _, a = run(handle, case, inp=inp)
    _, b = run(handle, case, inp=inp)
    assert torch.equal(a.grad.view(torch.int16), b.grad.view(torch.int16))
    assert torch.equal(a.loss, b.loss)


def test_back_to_back_calls_match_synchronised_calls(dev, handle):
    """Calls of different kinds queued on one stream with no host sync between
    them (each kernel may start while the one before it finishes) give the same
    bits as the same calls with a sync after each."""
    cases = [_case(dev, "ce_z_bf16", dict(T=2048, V=32000)),
             _case(dev, "gspo_z_bf16", dict(T=1024, V=151936, packed_len=256)),
             _case(dev, "ce_z_kl_bf16", dict(T=64, V=262144)),
             _case(dev, "confident_bf16", dict(T=512, V=128256))]
    inps = [c.device_inputs() for c in cases]

    def call(c, inp, grad):
        return handle.forward_backward(
            inp["logits"], inp["targets"], inp["loss_mask"], teacher_logits=inp["teacher_logits"],
            segment_ids=inp.get("segment_ids"), advantages=inp.get("advantages"),
            old_logprobs=inp.get("old_logprobs"), grad=grad, want=WANT, **c.kwargs())

    order = [(k, g) for _ in range(2) for k in range(len(cases)) for g in ("new", None)]
    ref = []
    for k, g in order:
        ref.append(call(cases[k], inps[k], g))
        torch.cuda.synchronize()
    got = [call(cases[k], inps[k], g) for k, g in order]
    torch.cuda.synchronize()
    assert handle.device_error() == 0
    for (k, g), a, b in zip(order, ref, got):
        assert torch.equal(a.loss, b.loss), (k, g)
        assert torch.equal(a.logp, b.logp) and torch.equal(a.lse, b.lse), (k, g)
        assert torch.equal(a.count, b.count), (k, g)
        if g is not None:
            assert torch.equal(a.grad.view(torch.int16), b.grad.view(torch.int16)), (k, g)


@pytest.mark.parametrize("name,shape", [("ce_z_bf16", dict(T=512, V=32000)),
                                        ("ce_z_kl_bf16", dict(T=48, V=70000))])
def test_cuda_graph_capture_and_replay(dev, handle, name, shape):
    """A whole call captured in a CUDA graph and replayed on new input values
    gives the bits of direct calls on those values."""
    case = _case(dev, name, shape)
    inp = case.device_inputs()
    kw = case.kwargs()
    want = ("logp", "lse", "count")
    x = inp["logits"].clone()
    u = None if inp["teacher_logits"] is None else inp["teacher_logits"].clone()
    tg = inp["targets"].clone()
    mk = None if inp["loss_mask"] is None else inp["loss_mask"].clone()

    def call():
        return handle.forward_backward(x, tg, mk, teacher_logits=u, grad="new", want=want, **kw)

    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        call()                                   # warm-up outside the capture
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        captured = call()
    gen = torch.Generator(device=dev)
    for k in range(3):
        gen.manual_seed(100 + k)
        x.copy_((inp["logits"].float() + torch.randn(x.shape, device=dev, generator=gen)).to(x.dtype))
        if u is not None:
            u.copy_((inp["teacher_logits"].float() + torch.randn(u.shape, device=dev, generator=gen)).to(u.dtype))
        tg.copy_(torch.randint(0, case.w.V, tg.shape, device=dev, generator=gen))
        graph.replay()
        torch.cuda.synchronize()
        direct = call()
        torch.cuda.synchronize()
        assert handle.device_error() == 0
        assert torch.equal(captured.loss, direct.loss), k
        assert torch.equal(captured.logp, direct.logp) and torch.equal(captured.lse, direct.lse), k
        assert torch.equal(captured.count, direct.count), k
        assert torch.equal(captured.grad.view(torch.int16), direct.grad.view(torch.int16)), k


@pytest.mark.parametrize("cluster,threads,nbuf", [(1, 256, 1), (2, 512, 2), (3, 512, 1), (4, 256, 2),
                                                  (8, 512, 2), (16, 128, 1)])
def test_launch_shapes(dev, handle, cluster, threads, nbuf):
    case = _case(dev, "ce_z_bf16", dict(T=96, V=50021))
    R, g_ref = oracle.forward_backward(case.P)
    handle.set_launch_config(cluster, threads, nbuf)
    try:
        _, out = run(handle, case)
        info = handle.call_info()
        assert info["cluster"] == cluster and info["threads"] == threads and info["nbuf"] == nbuf
        compare_all(case, out, R, g_ref, f"shape {cluster},{threads},{nbuf}")
    finally:
        handle.set_launch_config(0, 0, 0)


@pytest.mark.parametrize("tau", [1.0, 2.0])
def test_gspo_with_teacher(dev, handle, tau):
    """GSPO together with distillation (and cross-entropy): the statistics pass
    keeps the teacher's row statistics for the gradient pass that follows the
    seam.  Every output against the oracle, the seam's counts and flags as in
    the GSPO parity case."""
    from dataclasses import replace
    w = workloads.get("gspo_z_bf16").with_shape(T=1024, V=40000, packed_len=256)
    w = replace(w, teacher_sigma=1.0, kl_weight=0.5, temperature=tau, ce_weight=0.3)
    case = Case(w, dev)
    R, g_ref, scale = oracle.forward_backward(case.P, with_scale=True)
    inp, out = run(handle, case)
    compare_all(case, out, R, g_ref, f"gspo with teacher, tau {tau}", scale)
    assert np.array_equal(out.seg_count.cpu().numpy(), R.seam.n)
    flag = out.seg_flag.cpu().numpy()
    ratio = R.seam.ratio
    lo, hi = 1 - w.clip_eps_low, 1 + w.clip_eps_high
    amb = (np.abs(ratio - lo) < 1e-6 * lo) | (np.abs(ratio - hi) < 1e-6 * hi)
    assert np.array_equal(flag[~amb], R.seam.flag[~amb])
    assert handle.call_info()["path"] == 2


FP32_CASES = [
    ("gspo_z_bf16", dict(T=512, V=20011, packed_len=128), {}),
    ("gspo_z_bf16", dict(T=512, V=20011, packed_len=128),
     dict(teacher_sigma=1.0, kl_weight=0.5, temperature=2.0, ce_weight=0.3)),
    ("confident_bf16", dict(T=64, V=30001), {}),
    ("ce_z_kl_bf16", dict(T=48, V=20011), {}),
]


@pytest.mark.parametrize("name,shape,params", FP32_CASES,
                         ids=["gspo", "gspo_teacher_tau2", "confident", "ce_z_kl"])
def test_fp32_paths(dev, handle, name, shape, params):
    """The fp32 instantiations on the paths the bf16 workloads take: GSPO's
    three passes (with and without a teacher), planted confident rows, and
    distillation; gradients within 1e-6 absolute, as for ce_fp32_small."""
    from dataclasses import replace
    w = replace(workloads.get(name).with_shape(**shape), dtype="fp32", **params)
    case = Case(w, dev)
    R, g_ref, scale = oracle.forward_backward(case.P, with_scale=True)
    _, out = run(handle, case)
    compare_all(case, out, R, g_ref, f"fp32 {name} {params}", scale)
    if w.has_gspo:
        assert np.array_equal(out.seg_count.cpu().numpy(), R.seam.n)


def test_launch_config_rejects_unbuilt_shapes(dev, handle):
    """Only the block sizes the library is built for are accepted."""
    from lm_head_vocab_gb300.lmloss import LMLossError
    for cluster, threads, nbuf in [(0, 384, 0), (0, 64, 0), (17, 0, 0), (0, 0, 3), (-1, 0, 0)]:
        with pytest.raises(LMLossError):
            handle.set_launch_config(cluster, threads, nbuf)
    handle.set_launch_config(0, 0, 0)


@pytest.mark.parametrize("name,shape", [("ce_z_kl_bf16", dict(T=1024, V=30000)),
                                        ("ce_z_bf16", dict(T=2048, V=32000)),
                                        ("confident_bf16", dict(T=2048, V=8000))])
def test_mostly_masked_rows(dev, handle, name, shape):
    """Nine rows in ten ignored: the persistent clusters run through long
    stretches of rows with no statistics to exchange, where the per-row records
    must still keep a cluster's CTAs in step (a CTA that ran two rows ahead would
    overwrite a peer's record slot)."""
    case = _case(dev, name, shape)
    rng = np.random.default_rng(7)
    case.targets[rng.random(case.w.T) < 0.9] = -100      # the oracle's Problem shares this array
    R, g_ref, scale = oracle.forward_backward(case.P, with_scale=True)
    _, out = run(handle, case)
    compare_all(case, out, R, g_ref, f"{name} mostly masked", scale)
    assert int(out.count[0]) == R.n_active < 0.2 * case.w.T


def test_shard_sum_bitwise(dev, handle):
    """Rows split into shards, each called with SUM over the global active count,
    give the full token-mean call's gradient bit for bit, and losses that add up."""
    case = _case(dev, "ce_z_bf16", dict(T=200, V=32000))
    inp = case.device_inputs()
    w = case.w
    _, full = handle_run_mean(handle, case, inp)
    N = float(case.P.denominator)   # workload reduction is SUM over the active count
    parts = []
    tot = 0.0
    for lo, hi in [(0, 77), (77, 150), (150, 200)]:
        out = handle.forward_backward(inp["logits"][lo:hi], inp["targets"][lo:hi], None, z_alpha=w.z_alpha,
                                      reduction="sum", denominator=N, grad="new")
        torch.cuda.synchronize()
        parts.append(out.grad)
        tot += float(out.loss[0])
    assert torch.equal(torch.cat(parts).view(torch.int16), full.grad.view(torch.int16))
    assert rel(tot, float(full.loss[0])) <= 1e-6


def handle_run_mean(handle, case, inp):
    out = handle.forward_backward(inp["logits"], inp["targets"], None, z_alpha=case.w.z_alpha,
                                  reduction="token_mean", grad="new")
    torch.cuda.synchronize()
    return inp, out


# ------------------------------------------------------------------- edges
def _tiny_problem(dev, handle, z, t, dtype, mask=None, **kw):
    x = z.astype(np.float32)
    host = workloads.bf16_round(x) if dtype == "bf16" else x
    P = oracle.Problem(logits=host, V=z.shape[1], targets=t, loss_mask=mask, **kw)
    R, g_ref = oracle.forward_backward(P)
    logits = to_device(host, dev)
    out = handle.forward_backward(logits, torch.from_numpy(t).to(dev),
                                  None if mask is None else torch.from_numpy(mask).to(dev),
                                  grad="new", want=("logp", "lse", "count"),
                                  reduction="token_mean" if P.reduction == 1 else "sum",
                                  denominator=P.denominator, z_alpha=P.z_alpha)
    torch.cuda.synchronize()
    return P, R, g_ref, out


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_extreme_margins(dev, handle, dtype):
    """Target margins of 20 to 130 nats.  While the NLL e^d is a normal fp32 number
    (d above about -87) it matches the oracle to the per-row tolerance; while it
    is an fp32 subnormal (d down to about -103) it stays above 0 and within a
    few subnormal steps of the oracle; below that it is 0 (never negative, never
    NaN).  The target gradient is never positive."""
    rng = np.random.default_rng(11)
    margins = np.array([20.0, 40.0, 60.0, 70.0, 80.0, 85.0, 95.0, 100.0, 130.0])
    T, V = len(margins), 4099
    z = rng.normal(0, 1, size=(T, V))
    t = rng.integers(0, V, size=T)
    for r in range(T):
        z[r, t[r]] = z[r].max() + margins[r]
    P, R, g_ref, out = _tiny_problem(dev, handle, z, t, dtype)
    assert handle.device_error() == 0
    assert rel(float(out.loss[0]), R.total) <= 1e-5
    logp = out.logp.cpu().numpy().astype(np.float64)
    nll_ref = -R.logp
    assert np.all(np.isfinite(logp)) and np.all(logp <= 0.0)
    normal = nll_ref >= 2.0 ** -126
    sub = (nll_ref < 2.0 ** -126) & (nll_ref >= 2.0 ** -148)
    under = nll_ref < 2.0 ** -150
    assert normal.sum() >= 4 and sub.sum() >= 2 and under.sum() >= 1, (normal, sub, under)
    np.testing.assert_allclose(logp[normal], R.logp[normal], rtol=2e-5, atol=0)
    assert np.all(logp[normal] < 0.0)
    # subnormal NLL: nonzero, within a relative 1e-3 or four subnormal steps
    assert np.all(logp[sub] < 0.0), (logp[sub], R.logp[sub])
    err = np.abs(-logp[sub] - nll_ref[sub])
    assert np.all(err <= np.maximum(1e-3 * nll_ref[sub], 4 * 2.0 ** -149)), (logp[sub], R.logp[sub])
    assert np.all(-logp[under] <= 2.0 ** -149)
    g = grad_to_f64(out.grad)
    assert all(g[r, t[r]] <= 0.0 for r in range(T))
    check_grad(g, g_ref, dtype == "bf16", f"margins {dtype}")


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("V", [1, 2, 3, 7, 8, 9, 17])
def test_small_vocab(dev, handle, dtype, V):
    rng = np.random.default_rng(V)
    T = 13
    z = rng.normal(0, 3, size=(T, V))
    t = rng.integers(0, V, size=T)
    t[3] = -100
    P, R, g_ref, out = _tiny_problem(dev, handle, z, t, dtype, z_alpha=0.01)
    assert handle.device_error() == 0
    assert rel(float(out.loss[0]), R.total) <= 1e-5 or abs(R.total) < 1e-30
    check_grad(grad_to_f64(out.grad), g_ref, dtype == "bf16", f"V={V}")


def test_all_rows_masked_and_empty(dev, handle):
    z = np.random.default_rng(0).normal(size=(5, 300))
    t = np.full(5, -100)
    P, R, g_ref, out = _tiny_problem(dev, handle, z, t, "bf16")
    assert torch.all(out.loss == 0) and torch.all(out.grad.float() == 0)
    assert int(out.count[0]) == 0
    # T = 0
    logits = torch.empty((0, 300), dtype=torch.bfloat16, device=dev)
    out = handle.forward_backward(logits, torch.empty(0, dtype=torch.int64, device=dev), grad="new")
    torch.cuda.synchronize()
    assert torch.all(out.loss == 0)


def test_neg_inf_logits(dev, handle):
    V = 40
    z = np.random.default_rng(1).normal(size=(4, V))
    z[0, 5] = -np.inf           # active row, a -inf non-target
    z[1, :] = -np.inf           # ignored row full of -inf
    z[2, 1:] = -np.inf          # every non-target is -inf: NLL 0, p_t = 1
    z[2, 0] = 0.5
    t = np.array([3, -100, 0, 7])
    P, R, g_ref, out = _tiny_problem(dev, handle, z, t, "bf16")
    assert handle.device_error() == 0
    g = grad_to_f64(out.grad)
    assert np.all(np.isfinite(g))
    check_grad(g, g_ref, True, "-inf rows")
    assert rel(float(out.loss[0]), R.total) <= 1e-5


def test_bad_target_sets_device_error(dev, handle):
    from lm_head_vocab_gb300._lib import LMLOSS_ERR_BAD_TARGET
    z = torch.zeros((3, 64), dtype=torch.bfloat16, device=dev)
    t = torch.tensor([1, 64, 2], device=dev)
    out = handle.forward_backward(z, t, grad="new")
    torch.cuda.synchronize()
    assert handle.device_error() == LMLOSS_ERR_BAD_TARGET
    assert handle.device_error() == 0            # read clears it
    assert torch.isnan(out.loss[0])
    assert torch.all(out.grad[0].float() != 0) and torch.isnan(out.grad[1].float()).all()


def test_bad_segment_sets_device_error(dev, handle):
    from lm_head_vocab_gb300._lib import LMLOSS_ERR_BAD_SEGMENT
    T, V = 4, 100
    z = torch.zeros((T, V), dtype=torch.bfloat16, device=dev)
    t = torch.tensor([1, 2, 3, 4], device=dev)
    seg = torch.tensor([0, 0, 1, 5], dtype=torch.int32, device=dev)
    adv = torch.ones(2, device=dev)
    old = torch.zeros(T, device=dev)
    handle.forward_backward(z, t, segment_ids=seg, num_segments=2, advantages=adv, old_logprobs=old,
                            ce_weight=0.0, grad="new")
    torch.cuda.synchronize()
    assert handle.device_error() == LMLOSS_ERR_BAD_SEGMENT


def test_bounded_wait_gives_up_and_device_stays_usable(dev, handle):
    """A wait on a barrier nothing arrives at ends with LMLOSS_ERR_TIMEOUT after
    its limit; the context stays usable (a normal call right after works)."""
    from lm_head_vocab_gb300 import _lib
    assert _lib.lmloss_selftest_bounded_wait(handle.handle, 200_000) == _lib.LMLOSS_ERR_TIMEOUT
    case = _case(dev, "ce_z_bf16", dict(T=16, V=1000))
    R, g_ref = oracle.forward_backward(case.P)
    _, out = run(handle, case)
    compare_all(case, out, R, g_ref, "after the wait self-test")


def test_forward_only_with_teacher(dev, handle):
    """Statistics mode with a teacher and masked rows (no gradient requested)."""
    case = _case(dev, "ce_z_kl_bf16", dict(T=300, V=20000))
    R = oracle.forward(case.P)
    inp = case.device_inputs()
    out = handle.forward_backward(inp["logits"], inp["targets"], inp["loss_mask"],
                                  teacher_logits=inp["teacher_logits"], grad=None,
                                  want=("logp", "lse", "kl", "count"), **case.kwargs())
    torch.cuda.synchronize()
    assert handle.device_error() == 0
    compare_all(case, out, R, None, "forward only with teacher")


def _kl_problem(dev, handle, z, u, t):
    """bf16 student and teacher, KL weight 0.5, z-loss 1e-3."""
    zb = workloads.bf16_round(z.astype(np.float32))
    ub = workloads.bf16_round(u.astype(np.float32))
    P = oracle.Problem(logits=zb, V=z.shape[1], targets=t, teacher=ub, kl_weight=0.5, z_alpha=1e-3)
    out = handle.forward_backward(to_device(zb, dev), torch.from_numpy(t).to(dev),
                                  teacher_logits=to_device(ub, dev), kl_weight=0.5, z_alpha=1e-3,
                                  grad="new", want=("logp", "lse", "kl", "count"))
    torch.cuda.synchronize()
    return P, out


@pytest.mark.parametrize("spread", [30.0, 140.0])
def test_kl_teacher_range(dev, handle, spread):
    """Teacher rows whose logits span `spread` nats (140: the smallest teacher
    probabilities underflow fp32 and flush to 0 in the exponentials)."""
    rng = np.random.default_rng(int(spread))
    T, V = 24, 40000
    z = rng.normal(0, 2, size=(T, V))
    u = z + rng.normal(0, 1, size=(T, V))
    cols = rng.integers(0, V, size=(T, 50))
    for r in range(T):
        u[r, cols[r]] = u[r].max() - spread
    t = rng.integers(0, V, size=T)
    P, out = _kl_problem(dev, handle, z, u, t)
    assert handle.device_error() == 0
    R, g_ref, scale = oracle.forward_backward(P, with_scale=True)
    assert rel(float(out.loss[0]), R.total) <= 1e-5 and rel(float(out.loss[3]), R.kl_loss) <= 1e-5
    np.testing.assert_allclose(out.kl.cpu().numpy(), R.kl, rtol=1e-4, atol=2e-6)
    check_grad(grad_to_f64(out.grad), g_ref, True, f"teacher spread {spread}", scale)


def test_kl_teacher_nan_propagates(dev, handle):
    """A NaN teacher logit makes that row's KL and gradient NaN, and no other row's."""
    rng = np.random.default_rng(9)
    T, V = 6, 3000
    z = rng.normal(0, 2, size=(T, V))
    u = z + rng.normal(0, 1, size=(T, V))
    u[2, 1234] = np.nan
    t = rng.integers(0, V, size=T)
    P, out = _kl_problem(dev, handle, z, u, t)
    assert handle.device_error() == 0
    g = out.grad.float().cpu().numpy()
    kl = out.kl.cpu().numpy()
    assert np.isnan(kl[2]) and np.all(np.isnan(g[2]))
    others = [r for r in range(T) if r != 2]
    assert np.all(np.isfinite(kl[others])) and np.all(np.isfinite(g[others]))
    assert np.isnan(float(out.loss[0]))
