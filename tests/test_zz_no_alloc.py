"""The allocation-free entry point gives the regular entry point's results.

lmloss_forward_backward_noalloc serves callers that may not allocate device
memory once they are running, such as an inference-engine plugin whose enqueue
step must not allocate, or a service that plans all of its device memory at
start-up: cudaMalloc can synchronise the device and can fail under memory
pressure.  Its workspace is a fixed array inside the library.

This file is named so that pytest collects it last: a run that stops at the
first failure has then already run every other test.  It builds what it needs
itself, so it also passes when run alone in a fresh process.
"""
import re

import numpy as np
import pytest
import torch

import workloads
from tests.gpu_util import Case, bf16_ulp, grad_to_f64, rel

pytestmark = pytest.mark.gpu

WANT = ("logp", "lse", "kl", "count", "seg")
CASES = [
    ("ce_z_bf16", dict(T=256, V=32000)),
    ("gspo_z_bf16", dict(T=512, V=8192, packed_len=128)),
    ("ce_z_kl_bf16", dict(T=64, V=20000)),
]


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    torch.cuda.set_device(0)
    return torch.device("cuda", 0)


def _call(h, case, inp, entry):
    """One call through the C ABI; entry is 'regular' (handle) or 'noalloc'."""
    from lm_head_vocab_gb300 import _lib
    args, out, keep = h.build_args(
        inp["logits"], inp["targets"], inp["loss_mask"], teacher_logits=inp["teacher_logits"],
        segment_ids=inp.get("segment_ids"), advantages=inp.get("advantages"),
        old_logprobs=inp.get("old_logprobs"), grad="new", want=WANT, **case.kwargs())
    stream = torch.cuda.current_stream()
    if entry == "regular":
        st = _lib.lmloss_forward_backward(h.handle, args, stream.cuda_stream)
    else:
        st = _lib.lmloss_forward_backward_noalloc(args, stream.cuda_stream)
    assert st == _lib.LMLOSS_OK, _lib.lmloss_status_string(st)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("name,shape", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_regular_twice(dev, name, shape):
    from lm_head_vocab_gb300 import LMLoss
    case = Case(workloads.get(name).with_shape(**shape), dev)
    inp = case.device_inputs()
    h = LMLoss(0, max_T=case.w.T, max_segments=max(1, case.S))
    try:
        ref = _call(h, case, inp, "regular")
        assert h.device_error() == 0
        for _ in range(2):      # two calls in a row share the fixed workspace
            out = _call(h, case, inp, "noalloc")
            lr, lo = ref.loss.cpu().numpy(), out.loss.cpu().numpy()
            for k in range(5):
                assert (lr[k] == 0 and lo[k] == 0) or rel(float(lo[k]), float(lr[k])) <= 1e-5, (k, lo, lr)
            assert torch.equal(out.count, ref.count)
            gr, go = grad_to_f64(ref.grad), grad_to_f64(out.grad)
            assert np.all(np.abs(go - gr) <= bf16_ulp(gr)), "gradient beyond 1 bf16 ulp of the regular call"
            np.testing.assert_allclose(out.logp.cpu().numpy(), ref.logp.cpu().numpy(), rtol=1e-6, atol=1e-7)
            np.testing.assert_allclose(out.lse.cpu().numpy(), ref.lse.cpu().numpy(), rtol=1e-6, atol=1e-7)
            if case.w.has_gspo:
                assert torch.equal(out.seg_count, ref.seg_count)
                assert torch.equal(out.seg_flag, ref.seg_flag)
    finally:
        h.close()


def test_noalloc_rejects_oversized_calls(dev):
    from lm_head_vocab_gb300 import LMLoss, _lib
    h = LMLoss(0, max_T=16, max_segments=1)
    try:
        logits = torch.zeros((16, 64), dtype=torch.bfloat16, device=dev)
        targets = torch.zeros(16, dtype=torch.int64, device=dev)
        args, out, keep = h.build_args(logits, targets, grad="new", want=())
        limit = int(re.search(r"#define LMLOSS_NOALLOC_MAX_T (\d+)", open(_lib.HEADER).read()).group(1))
        args.T = limit + 1      # beyond the fixed workspace: rejected before any launch
        st = _lib.lmloss_forward_backward_noalloc(args, torch.cuda.current_stream().cuda_stream)
        assert st == _lib.LMLOSS_ERR_INVALID_ARG
    finally:
        h.close()
