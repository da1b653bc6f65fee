"""Data-parallel sharding arithmetic of the path, on CPU with two gloo ranks.

Rows are independent, so a batch splits over ranks.  Each rank holds its own
rows and the full W.  The exchange is: an all-reduce of the valid count
(the normaliser), then an all-reduce of the loss sum and of dW.  dX rows
need no exchange.  A shard run with the library's ``norm_count`` = global
count produces exactly the per-rank terms below; here the terms come from
the oracle (its per-shard results rescaled from the local to the global
count), and their reduction over two gloo ranks must equal the oracle on
the whole batch.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

IGN = -100


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_dir):
    import oracle
    from flce_synth import make_case
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}",
                            rank=rank, world_size=world)
    X, W, t = make_case(37, 24, 90, "fp32", seed=41, ignore_num=20, w_std=0.4)
    rows = np.array_split(np.arange(37), world)[rank]
    Xs, ts = X[rows].contiguous(), t[rows].contiguous()
    n_local = torch.tensor([int((ts != IGN).sum())], dtype=torch.int64)
    n_global = n_local.clone()
    dist.all_reduce(n_global)                       # exchange 1: the normaliser
    r = oracle.flce(Xs, W, ts, IGN)
    scale = float(n_local.item()) / float(n_global.item())
    loss_sum = torch.tensor([r["loss"] * scale], dtype=torch.float64)
    dW = torch.from_numpy(r["dW"] * scale)
    dist.all_reduce(loss_sum)                       # exchange 2: loss and dW
    dist.all_reduce(dW)
    dX_rows = r["dX"] * scale                       # rows stay on their rank
    np.save(os.path.join(out_dir, f"dx{rank}.npy"), dX_rows)
    if rank == 0:
        np.save(os.path.join(out_dir, "dw.npy"), dW.numpy())
        np.save(os.path.join(out_dir, "loss.npy"), loss_sum.numpy())
        np.save(os.path.join(out_dir, "n.npy"), n_global.numpy())
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_shards_reduce_to_the_whole_batch(tmp_path):
    import oracle
    from flce_synth import make_case
    oracle.build()
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    X, W, t = make_case(37, 24, 90, "fp32", seed=41, ignore_num=20, w_std=0.4)
    ref = oracle.flce(X, W, t, IGN)
    assert int(np.load(tmp_path / "n.npy")[0]) == ref["n_valid"]
    assert abs(float(np.load(tmp_path / "loss.npy")[0]) - ref["loss"]) <= 1e-13
    np.testing.assert_allclose(np.load(tmp_path / "dw.npy"), ref["dW"], rtol=1e-11, atol=1e-15)
    dX = np.vstack([np.load(tmp_path / f"dx{r}.npy") for r in range(world)])
    np.testing.assert_allclose(dX, ref["dX"], rtol=1e-11, atol=1e-15)
