"""Logits in host memory: lmloss_forward_backward_host copies the rows in
chunks on a stream of the handle's own and starts each chunk's kernel as soon
as it has landed.  Every output must be the bits of lmloss_forward_backward on
the same data (a row's computation does not depend on the chunking; the token
count and the loss reduction run once over all rows), for several chunkings,
both reductions, forward only, a teacher, GRPO's per-token inputs, GSPO, the
entropy and padded rows; and the copies must follow the caller's earlier work on
its stream."""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_util import Case, compare_all

pytestmark = pytest.mark.gpu

WANT = ("logp", "lse", "kl", "count", "entropy")


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda", 0)


@pytest.fixture(scope="module")
def handle(dev):
    from lm_head_vocab_gb300 import LMLoss
    h = LMLoss(0, max_T=4096, max_segments=4096)
    yield h
    h.close()


def _bits(t):
    if t is None:
        return None
    t = t.contiguous()
    return (t.view(torch.int16) if t.dtype == torch.bfloat16 else t.view(torch.int32)).cpu().numpy()


def _same(a, b, what, V):
    for k in ("loss", "logp", "lse", "kl", "entropy", "grad"):
        x, y = getattr(a, k), getattr(b, k)
        assert (x is None) == (y is None), (what, k)
        if x is not None:
            if k == "grad":   # the V columns (padding columns are never written)
                x, y = x[:, :V], y[:, :V]
            assert np.array_equal(_bits(x), _bits(y)), (what, k)
    assert torch.equal(a.count, b.count), what


def _chunks(T, chunk_rows):
    # the library's rule: chunk_rows rows a chunk (0: T / 8), at most 64 chunks
    rows = chunk_rows if chunk_rows > 0 else -(-T // 8)
    if -(-T // rows) > 64:
        rows = -(-T // 64)
    return -(-T // rows)


CASES = [
    ("ce_z_bf16", dict(T=1000, V=32000), {}, "new", [0, 1, 7, 128, 999, 1000, 4096]),
    ("ce_z_bf16", dict(T=257, V=4099), {}, "inplace", [0, 64]),
    ("ce_z_kl_bf16", dict(T=300, V=30011), {}, "new", [0, 37]),
    ("ce_z_kl_bf16", dict(T=300, V=30011), dict(temperature=2.0), None, [0, 100]),
    ("confident_bf16", dict(T=512, V=50000), {}, "inplace", [0, 3]),
    ("ce_fp32_small", dict(T=64, V=1024), {}, "new", [0, 5]),
]


@pytest.mark.parametrize("name,shape,params,grad,chunks", CASES,
                         ids=["ce_z", "ce_z_unaligned_inplace", "distill", "distill_tau2_fwd", "confident_inplace",
                              "fp32"])
def test_same_bits_as_device_call(dev, handle, name, shape, params, grad, chunks):
    w = replace(workloads.get(name).with_shape(**shape), **params)
    case = Case(w, dev)
    inp = case.device_inputs()
    kw = case.kwargs()
    hx = inp["logits"].cpu().pin_memory()
    hu = None if inp["teacher_logits"] is None else inp["teacher_logits"].cpu().pin_memory()
    pristine = inp["logits"].clone()
    ref = handle.forward_backward(inp["logits"], inp["targets"], inp["loss_mask"],
                                  teacher_logits=inp["teacher_logits"], grad=grad, want=WANT, **kw)
    if grad == "inplace":
        ref.grad = ref.grad.clone()
    torch.cuda.synchronize()
    assert handle.device_error() == 0
    ref_info = handle.call_info()
    for rows in chunks:
        # device buffers that the call fills from the host tensors
        d_x = torch.full_like(pristine, float("nan"))
        d_u = None if hu is None else torch.full_like(inp["teacher_logits"], float("nan"))
        out = handle.forward_backward_host(hx, d_x, inp["targets"], inp["loss_mask"], host_teacher=hu,
                                           chunk_rows=rows, teacher_logits=d_u, grad=grad, want=WANT, **kw)
        torch.cuda.synchronize()
        assert handle.device_error() == 0
        info = handle.call_info()
        # one staged-row launch per chunk in place of the single one
        assert info["launches"] == ref_info["launches"] - 1 + _chunks(w.T, rows), (info, ref_info, rows)
        _same(out, ref, f"{name} chunk_rows {rows}", w.V)
        if grad != "inplace":
            # the device buffer holds the copied logits
            assert np.array_equal(_bits(d_x[:, :w.V]), _bits(pristine[:, :w.V]))
    R, g_ref, scale = oracle.forward_backward(case.P, with_scale=True) if grad else (oracle.forward(case.P), None, None)
    if grad:
        compare_all(case, out, R, g_ref, f"host {name}", scale)


def test_grpo_inputs_follow_their_rows(dev, handle):
    """GRPO's per-token advantages and old log-probs are indexed by row: each
    chunk reads its own."""
    w = workloads.get("ce_z_bf16").with_shape(T=600, V=20011)
    case = Case(w, dev)
    inp = case.device_inputs()
    rng = np.random.default_rng(5)
    adv = torch.from_numpy(rng.normal(0, 1, size=w.T).astype(np.float32)).to(dev)
    old = torch.from_numpy(rng.normal(-8, 1, size=w.T).astype(np.float32)).to(dev)
    kw = dict(case.kwargs(), token_advantages=adv, old_logprobs=old, clip_eps_low=0.2, clip_eps_high=0.28)
    ref = handle.forward_backward(inp["logits"], inp["targets"], inp["loss_mask"], grad="new", want=WANT, **kw)
    hx = inp["logits"].cpu().pin_memory()
    d_x = torch.empty_like(inp["logits"])
    out = handle.forward_backward_host(hx, d_x, inp["targets"], inp["loss_mask"], chunk_rows=97, grad="new",
                                       want=WANT, **kw)
    torch.cuda.synchronize()
    assert handle.device_error() == 0
    _same(out, ref, "grpo", w.V)


def test_copies_follow_earlier_work_on_the_stream(dev, handle):
    """Back-to-back in-place steps on one stream: each call's copies wait for the
    previous call's kernels to finish writing their gradient into the same
    device buffer, so every step sees its own logits."""
    w = workloads.get("ce_z_bf16").with_shape(T=2048, V=32000)
    case = Case(w, dev)
    inp = case.device_inputs()
    kw = case.kwargs()
    ref = handle.forward_backward(inp["logits"].clone(), inp["targets"], inp["loss_mask"], grad="inplace",
                                  want=WANT, **kw)
    torch.cuda.synchronize()
    hx = inp["logits"].cpu().pin_memory()
    d_x = torch.empty_like(inp["logits"])
    s = torch.cuda.Stream(dev)
    outs = []
    with torch.cuda.stream(s):
        for _ in range(4):
            o = handle.forward_backward_host(hx, d_x, inp["targets"], inp["loss_mask"], chunk_rows=256,
                                             grad="inplace", want=WANT, stream=s, **kw)
            outs.append((o.loss.clone(), o.logp.clone()))
    s.synchronize()
    assert handle.device_error() == 0
    for loss, logp in outs:
        assert torch.equal(loss, ref.loss) and torch.equal(logp, ref.logp)
    assert np.array_equal(_bits(d_x[:, :w.V]), _bits(ref.grad[:, :w.V]))


@pytest.mark.parametrize("teacher", [False, True], ids=["gspo", "gspo_teacher"])
def test_gspo(dev, handle, teacher):
    """GSPO: the chunks run the statistics pass as they land; the seam and the
    gradient pass follow over all rows.  Same bits as the device call."""
    w = workloads.get("gspo_z_bf16").with_shape(T=1024, V=20011, packed_len=256)
    if teacher:
        w = replace(w, teacher_sigma=1.0, kl_weight=0.5, temperature=2.0, ce_weight=0.3)
    case = Case(w, dev)
    inp = case.device_inputs()
    kw = case.kwargs()
    g = dict(segment_ids=inp["segment_ids"], advantages=inp["advantages"], old_logprobs=inp["old_logprobs"])
    want = WANT + ("seg",)
    ref = handle.forward_backward(inp["logits"], inp["targets"], inp["loss_mask"],
                                  teacher_logits=inp["teacher_logits"], grad="new", want=want, **g, **kw)
    torch.cuda.synchronize()
    hx = inp["logits"].cpu().pin_memory()
    hu = None if inp["teacher_logits"] is None else inp["teacher_logits"].cpu().pin_memory()
    d_u = None if hu is None else torch.empty_like(inp["teacher_logits"])
    out = handle.forward_backward_host(hx, torch.empty_like(inp["logits"]), inp["targets"], inp["loss_mask"],
                                       host_teacher=hu, teacher_logits=d_u, chunk_rows=100, grad="new",
                                       want=want, **g, **kw)
    torch.cuda.synchronize()
    assert handle.device_error() == 0
    assert handle.call_info()["path"] == 2
    _same(out, ref, "gspo", w.V)
    for k in ("seg_count", "seg_ratio", "seg_flag", "seg_loss"):
        assert torch.equal(getattr(out, k), getattr(ref, k)), k


def test_rejects_unpaired_host_teacher(dev, handle):
    w = workloads.get("ce_z_bf16").with_shape(T=64, V=4096)
    case = Case(w, dev)
    inp = case.device_inputs()
    hx = inp["logits"].cpu().pin_memory()
    with pytest.raises(ValueError):
        handle.forward_backward_host(hx, torch.empty_like(inp["logits"]), inp["targets"], host_teacher=hx,
                                     grad="new")


def test_padded_rows(dev, handle):
    """Rows with padding (ld > V): each chunk copies its rows' full stride and
    the last row's V columns; outputs as the device call's."""
    rng = np.random.default_rng(11)
    T, V, ld = 203, 5000, 5016
    x = rng.normal(0, 2, size=(T, ld)).astype(np.float32)
    full = torch.from_numpy(x).to(dev).to(torch.bfloat16)
    x_dev = full[:, :V]
    t = torch.from_numpy(rng.integers(0, V, size=T)).to(dev)
    ref = handle.forward_backward(x_dev, t, z_alpha=1e-4, grad="new", want=WANT)
    hx = torch.empty((T, ld), dtype=torch.bfloat16).pin_memory()
    hx.copy_(full.cpu())
    hx = hx[:, :V]
    d_x = torch.full((T, ld), float("nan"), dtype=torch.bfloat16, device=dev)[:, :V]
    out = handle.forward_backward_host(hx, d_x, t, chunk_rows=50, z_alpha=1e-4, grad="new", want=WANT)
    torch.cuda.synchronize()
    assert handle.device_error() == 0
    _same(out, ref, "padded rows", V)


def test_cuda_graph_capture_and_replay(dev, handle):
    """The host-buffer call captured in a CUDA graph (its copy stream joins the
    capture through the events) and replayed after new values are written into
    the pinned host buffer: each replay gives the bits of a direct device call
    on those values."""
    w = workloads.get("ce_z_bf16").with_shape(T=512, V=32000)
    case = Case(w, dev)
    inp = case.device_inputs()
    kw = case.kwargs()
    want = ("logp", "lse", "count")
    hx = inp["logits"].cpu().pin_memory()
    x = torch.empty_like(inp["logits"])

    def call():
        return handle.forward_backward_host(hx, x, inp["targets"], inp["loss_mask"], chunk_rows=100, grad="new",
                                            want=want, **kw)

    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        call()                                   # creates the copy stream and events, outside the capture
    torch.cuda.current_stream(dev).wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        captured = call()
    gen = torch.Generator().manual_seed(3)
    for k in range(3):
        hx.copy_((inp["logits"].float().cpu() + torch.randn(hx.shape, generator=gen)).to(hx.dtype))
        graph.replay()
        torch.cuda.synchronize()
        direct = handle.forward_backward(hx.to(dev), inp["targets"], inp["loss_mask"], grad="new", want=want, **kw)
        torch.cuda.synchronize()
        assert handle.device_error() == 0
        assert torch.equal(captured.loss, direct.loss), k
        assert torch.equal(captured.logp, direct.logp) and torch.equal(captured.lse, direct.lse), k
        assert torch.equal(captured.grad.view(torch.int16), direct.grad.view(torch.int16)), k
