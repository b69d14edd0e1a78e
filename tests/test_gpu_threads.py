"""Handles used from several host threads at once.

Two threads, each with its own handle and its own CUDA stream, call the library
at the same time on workloads of different shapes: different kernel
instantiations, shared-memory sizes and cluster shapes.  The kernels' launch
attributes are process-wide, so this is where one thread could lower a limit
under the other's launch.  Every call must succeed, and each thread's results
must be the bits of the same call made alone.  (The allocation-free entry point
shares one workspace and is documented as not reentrant; it is not used here.)
"""
import threading

import pytest
import torch

import workloads
from tests.gpu_util import Case

pytestmark = pytest.mark.gpu

WANT = ("logp", "lse", "kl", "count")


@pytest.fixture(scope="module")
def dev():
    import __graft_entry__
    __graft_entry__.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    return torch.device("cuda", 0)


def _bits(t):
    return t.view(torch.int16) if t.dtype == torch.bfloat16 else t


def _call(h, case, inp, stream=None):
    return h.forward_backward(inp["logits"], inp["targets"], inp["loss_mask"],
                              teacher_logits=inp["teacher_logits"], grad="new", want=WANT,
                              stream=stream, **case.kwargs())


def test_two_threads_two_handles(dev):
    from lm_head_vocab_gb300 import LMLoss
    cases = [Case(workloads.get("ce_z_kl_bf16").with_shape(T=192, V=65536), dev),
             Case(workloads.get("ce_z_bf16").with_shape(T=1024, V=5001), dev)]
    inps = [c.device_inputs() for c in cases]
    # each call alone first
    refs = []
    for c, inp in zip(cases, inps):
        h = LMLoss(0, max_T=c.w.T, max_segments=1)
        refs.append(_call(h, c, inp))
        torch.cuda.synchronize()
        assert h.device_error() == 0
        h.close()

    calls = 24
    results = [None, None]
    errors = []
    start = threading.Barrier(2)

    def worker(k):
        try:
            torch.cuda.set_device(0)
            h = LMLoss(0, max_T=cases[k].w.T, max_segments=1)
            s = torch.cuda.Stream()
            start.wait()
            with torch.cuda.stream(s):
                outs = [_call(h, cases[k], inps[k], stream=s) for _ in range(calls)]
            s.synchronize()
            results[k] = (outs[0], outs[-1], h.device_error())
            h.close()
        except Exception as e:   # reported to the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(k,)) for k in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for k in range(2):
        first, last, err = results[k]
        assert err == 0
        for out in (first, last):
            assert torch.equal(_bits(out.grad), _bits(refs[k].grad)), f"thread {k}: gradient bits differ"
            assert torch.equal(out.loss, refs[k].loss), (k, out.loss, refs[k].loss)
            assert torch.equal(out.logp, refs[k].logp) and torch.equal(out.lse, refs[k].lse)
            if out.kl is not None:
                assert torch.equal(out.kl, refs[k].kl)
