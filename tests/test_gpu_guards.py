"""Out-of-bounds writes and input mutation, checked without a sanitizer: every
output buffer of a call sits between guard bands of a known byte pattern that
must survive the call, the logits must be untouched unless the gradient is
written in place, and odd shapes (T = 1, V not a multiple of the vector width,
rows not 16-byte aligned, a vocabulary-shard tail) are included."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_util import check_grad, grad_to_f64, rel, to_device

pytestmark = pytest.mark.gpu

GUARD = 4096          # bytes on each side of every output
PATTERN = 0x5A


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda", 0)


@pytest.fixture(scope="module")
def handle(dev):
    from lm_head_vocab_gb300 import LMLoss
    h = LMLoss(0, max_T=4096, max_segments=64)
    yield h
    h.close()


class Guarded:
    """A device buffer of `nbytes` with GUARD bytes of PATTERN on both sides."""

    def __init__(self, nbytes, dev):
        self.n = nbytes
        self.raw = torch.full((nbytes + 2 * GUARD,), PATTERN, dtype=torch.uint8, device=dev)

    @property
    def ptr(self):
        return self.raw.data_ptr() + GUARD

    def view(self, dtype, shape):
        return self.raw[GUARD:GUARD + self.n].view(dtype).view(shape)

    def intact(self):
        lo = self.raw[:GUARD]
        hi = self.raw[GUARD + self.n:]
        return bool(torch.all(lo == PATTERN)) and bool(torch.all(hi == PATTERN))


def _problem(T, V, ld, dtype, seed, teacher=False):
    rng = np.random.default_rng(seed)
    z = rng.normal(0, 2, size=(T, ld)).astype(np.float32)
    u = (z + rng.normal(0, 1, size=(T, ld))).astype(np.float32) if teacher else None
    t = rng.integers(0, V, size=T)
    if T > 2:
        t[1] = -100
    if dtype == "bf16":
        z = workloads.bf16_round(z)
        u = None if u is None else workloads.bf16_round(u)
    return z, u, t


SHAPES = [(1, 1000, 1000), (1, 7, 7), (3, 9, 9), (5, 4099, 4111), (17, 32003, 32008), (64, 50021, 50021)]


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("T,V,ld", SHAPES, ids=[f"{s[0]}x{s[1]}/{s[2]}" for s in SHAPES])
@pytest.mark.parametrize("teacher", [False, True])
def test_outputs_stay_in_bounds_and_input_untouched(dev, handle, dtype, T, V, ld, teacher):
    z, u, t = _problem(T, V, ld, dtype, seed=T * 7 + V, teacher=teacher)
    logits_full = to_device(z, dev)
    logits = logits_full[:, :V]
    teach = None if u is None else to_device(u, dev)[:, :V]
    tg = torch.from_numpy(t).to(dev)
    before = logits_full.clone()
    esz = 2 if dtype == "bf16" else 4
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    g = Guarded(T * ld * esz, dev)
    grad = g.view(tdt, (T, ld))[:, :V]
    a, out, keep = handle.build_args(logits, tg, teacher_logits=teach, kl_weight=0.5 if teacher else 0.0,
                                     z_alpha=1e-3, grad=grad, want=("logp", "lse", "kl", "entropy", "count"))
    bufs = {}
    for name, nbytes in [("loss_out", 20), ("logp_out", 4 * T), ("lse_out", 4 * T), ("entropy_out", 4 * T),
                         ("count_out", 16)] + ([("kl_out", 4 * T)] if teacher else []):
        bufs[name] = Guarded(nbytes, dev)
        setattr(a, name, bufs[name].ptr)
    handle.call(a)
    torch.cuda.synchronize()
    assert handle.device_error() == 0
    assert g.intact(), "gradient guard band overwritten"
    for name, b in bufs.items():
        assert b.intact(), f"{name} guard band overwritten"
    assert torch.equal(logits_full, before), "logits modified although the gradient went elsewhere"
    # the padding columns of the gradient buffer are not written either
    if ld > V:
        pad = g.view(tdt, (T, ld))[:, V:].contiguous().view(torch.uint8)
        assert bool(torch.all(pad == PATTERN))
    # and the values are right
    P = oracle.Problem(logits=z, V=V, targets=t, teacher=u, kl_weight=0.5 if teacher else 0.0, z_alpha=1e-3)
    R, g_ref, scale = oracle.forward_backward(P, with_scale=True)
    loss = bufs["loss_out"].view(torch.float32, (5,)).cpu().numpy().astype(np.float64)
    assert rel(loss[0], R.total) <= 1e-5
    check_grad(grad_to_f64(grad), g_ref, dtype == "bf16", f"guarded {T}x{V}", scale if teacher else None)


def test_in_place_only_touches_the_row_columns(dev, handle):
    """In place with a padded stride: the gradient overwrites columns [0, V) of
    each row and leaves the padding columns alone."""
    T, V, ld = 9, 3001, 3008
    z, _, t = _problem(T, V, ld, "bf16", seed=3)
    full = to_device(z, dev)
    pad_before = full[:, V:].clone()
    out = handle.forward_backward(full[:, :V], torch.from_numpy(t).to(dev), grad="inplace")
    torch.cuda.synchronize()
    assert torch.equal(full[:, V:], pad_before)
    P = oracle.Problem(logits=z, V=V, targets=t)
    R, g_ref = oracle.forward_backward(P)
    check_grad(grad_to_f64(full[:, :V]), g_ref, True, "in place padded")


def test_shard_partials_stay_in_bounds(dev, handle):
    from lm_head_vocab_gb300 import _lib
    T, V = 33, 1000
    z, _, t = _problem(T, V, V, "bf16", seed=5)
    tg = torch.from_numpy(t).to(dev)
    shard = to_device(np.ascontiguousarray(z[:, 400:]), dev)
    part = Guarded(16 * T, dev)
    a, _out, _keep = handle.build_args(shard, tg, grad=None, want=())
    st = _lib.load().lmloss_shard_stats(handle.handle, a, 400, V, ctypes.c_void_p(part.ptr),
                                        torch.cuda.current_stream(dev).cuda_stream)
    assert st == _lib.LMLOSS_OK
    torch.cuda.synchronize()
    assert part.intact()
