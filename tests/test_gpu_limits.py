"""The largest rows the library serves, and a clean refusal just past them.

A row is staged across a cluster of at most 16 CTAs, each holding its slice of
the row (and of the teacher's) in its shared memory, so the largest
vocabulary follows from the device's opt-in shared memory per block:
16 slices of (limit - 3072 header bytes) / (element size x arrays), rounded
down to whole 16-byte vectors.  At that size every output matches the oracle;
one vector more returns LMLOSS_ERR_UNSUPPORTED before anything is launched.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.gpu_util import check_grad, grad_to_f64, rel, to_device

pytestmark = pytest.mark.gpu

HDR = 3072          # the staged-row kernel's header bytes ahead of the slices
CLUSTER_MAX = 16


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda", 0)


@pytest.fixture(scope="module")
def handle(dev):
    from lm_head_vocab_gb300 import LMLoss
    h = LMLoss(0, max_T=64, max_segments=1)
    yield h
    h.close()


def v_max(arrays: int, esz: int = 2) -> int:
    """Largest V whose 16 slices each fit one CTA's opt-in shared memory."""
    optin = torch.cuda.get_device_properties(0).shared_memory_per_block_optin
    per_array = (optin - HDR) // arrays // 128 * 128       # slices are padded to 128 bytes
    cols = per_array // esz // (16 // esz) * (16 // esz)   # whole 16-byte vectors
    return CLUSTER_MAX * cols


def _case(V, T, teacher, seed):
    rng = np.random.default_rng(seed)
    z = workloads.bf16_round(rng.normal(0, 2, size=(T, V)).astype(np.float32))
    u = workloads.bf16_round((z.view(np.uint16).astype(np.uint32) << 16).view(np.float32)
                             + rng.normal(0, 1, size=(T, V)).astype(np.float32)) if teacher else None
    t = rng.integers(0, V, size=T)
    t[-1] = V - 1                     # a target in the last column of the last slice
    return z, u, t


@pytest.mark.parametrize("teacher", [False, True], ids=["ce_z", "ce_z_kl"])
def test_largest_vocabulary(dev, handle, teacher):
    V = v_max(2 if teacher else 1)
    T = 3
    z, u, t = _case(V, T, teacher, seed=V % 1000)
    P = oracle.Problem(logits=z, V=V, targets=t, teacher=u, kl_weight=0.5 if teacher else 0.0, z_alpha=1e-4)
    R, g_ref, scale = oracle.forward_backward(P, with_scale=True)
    out = handle.forward_backward(to_device(z, dev), torch.from_numpy(t).to(dev),
                                  teacher_logits=None if u is None else to_device(u, dev),
                                  kl_weight=0.5 if teacher else 0.0, z_alpha=1e-4, grad="new",
                                  want=("logp", "lse", "kl", "count"))
    torch.cuda.synchronize()
    assert handle.device_error() == 0
    info = handle.call_info()
    assert info["cluster"] == CLUSTER_MAX
    loss = out.loss.cpu().numpy().astype(np.float64)
    assert rel(loss[0], R.total) <= 1e-5
    np.testing.assert_allclose(out.lse.cpu().numpy(), R.lse, rtol=2e-6, atol=2e-6)
    if teacher:
        np.testing.assert_allclose(out.kl.cpu().numpy(), R.kl, rtol=1e-4, atol=2e-6)
    check_grad(grad_to_f64(out.grad), g_ref, True, f"V = {V}", scale if teacher else None)


@pytest.mark.parametrize("teacher", [False, True], ids=["ce_z", "ce_z_kl"])
def test_one_vector_more_is_refused(dev, handle, teacher):
    from lm_head_vocab_gb300.lmloss import LMLossError
    from lm_head_vocab_gb300 import _lib
    V = v_max(2 if teacher else 1) + CLUSTER_MAX * 8
    T = 2
    x = torch.zeros((T, V), dtype=torch.bfloat16, device=dev)
    t = torch.zeros(T, dtype=torch.int64, device=dev)
    with pytest.raises(LMLossError) as e:
        handle.forward_backward(x, t, teacher_logits=x.clone() if teacher else None,
                                kl_weight=0.5 if teacher else 0.0, grad="new")
    assert e.value.status == _lib.LMLOSS_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert handle.device_error() == 0
