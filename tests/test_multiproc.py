"""Row sharding over ranks (world size 2, gloo, CPU).

Each rank takes its own rows of a batch twice as tall, as bench.py does under
torchrun, and reduces with SUM over the global active count computed on the
host from the seeds.  The ranks' losses, summed with an all_reduce, equal the
full batch's token-mean loss, and each rank's gradient rows equal the full
batch's rows (xtuner PR 1963 "[FSDP][Loss] Switch gradient reduction to SUM":
each rank's loss is its local component of the global token mean).  The fp64
oracle stands in for the device path, so no GPU is needed.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _small(name):
    import workloads
    base = workloads.get(name)
    return base.with_shape(48, 777)


def _worker(rank, world, port, name, out_dir):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import oracle
    w = _small(name)
    sl = bench.RankSlice(w, rank, world)
    x, u = sl.host_rows(w.T)
    t, m, n_glob = sl.targets, sl.mask, sl.n_active_global
    kw = bench.call_kwargs(w, world, n_glob)
    assert kw["reduction"] == "sum" and kw["denominator"] == float(n_glob)
    P = oracle.Problem(logits=x, V=w.V, targets=t, loss_mask=m, ce_weight=w.ce_weight, z_alpha=w.z_alpha,
                       teacher=u, kl_weight=w.kl_weight, reduction=oracle.REDUCE_SUM,
                       denominator=kw["denominator"])
    R, g = oracle.forward_backward(P, nthreads=1)
    tot = torch.tensor([R.total], dtype=torch.float64)
    dist.all_reduce(tot)
    cnt = torch.tensor([R.n_active], dtype=torch.int64)
    dist.all_reduce(cnt)
    np.save(os.path.join(out_dir, f"g{rank}.npy"), g)
    np.save(os.path.join(out_dir, f"tot{rank}.npy"), np.array([tot.item(), float(cnt.item()), float(n_glob)]))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("name", ["ce_z_bf16", "ce_z_kl_bf16", "confident_bf16"])
def test_row_sharding_gloo(tmp_path, name):
    import oracle
    port = _free_port()
    mp.start_processes(_worker, args=(WORLD, port, name, str(tmp_path)), nprocs=WORLD, start_method="spawn")
    w = _small(name)
    wg = w.with_shape(w.T * WORLD, w.V)
    tg = wg.targets()
    x = wg.logits_rows(0, wg.T, targets=tg)
    u = wg.teacher_rows(0, wg.T, x)
    P = oracle.Problem(logits=x, V=w.V, targets=tg, loss_mask=wg.loss_mask(), ce_weight=w.ce_weight,
                       z_alpha=w.z_alpha, teacher=u, kl_weight=w.kl_weight, reduction=oracle.REDUCE_TOKEN_MEAN)
    R, g = oracle.forward_backward(P, nthreads=1)
    parts = [np.load(tmp_path / f"g{r}.npy") for r in range(WORLD)]
    info = [np.load(tmp_path / f"tot{r}.npy") for r in range(WORLD)]
    for tot, cnt, n_glob in info:
        assert tot == pytest.approx(R.total, rel=1e-12)
        assert int(cnt) == R.n_active == int(n_glob)
    assert np.array_equal(np.concatenate(parts), g)
