"""Data-parallel sharding of the path, on CPU with two gloo ranks.

Rows are independent, so a batch splits over ranks.  Each rank holds its own
rows and the full W.  The exchange is: an all-reduce of the valid count (the
normaliser), then one call per rank with ``norm_count`` set to that global
count, then an all-reduce of the loss and of dW.  dX rows need no exchange.
On a GPU the call is the library's ``flce_fwd_bwd_ex(norm_count=...)``
(checked against the oracle shard by shard in
``tests/test_gpu_shards.py``); here, with no GPU, each rank makes the same
call on the oracle, whose ``norm_count`` follows the same reading, and the
reduction over two gloo ranks must equal the oracle on the whole batch.
"""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

IGN = -100
CASE = dict(N=37, H=24, V=90)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _case():
    from flce_synth import make_case
    return make_case(CASE["N"], CASE["H"], CASE["V"], "fp32", seed=41, ignore_num=20,
                     w_std=0.4)


def _rank_main(rank, world, port, out_dir):
    import oracle
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}",
                            rank=rank, world_size=world)
    X, W, t = _case()
    rows = np.array_split(np.arange(CASE["N"]), world)[rank]
    Xs, ts = X[rows].contiguous(), t[rows].contiguous()
    n_global = torch.tensor([int((ts != IGN).sum())], dtype=torch.int64)
    dist.all_reduce(n_global)                       # exchange 1: the normaliser
    r = oracle.flce(Xs, W, ts, IGN, norm_count=int(n_global.item()))
    loss = torch.tensor([r["loss"]], dtype=torch.float64)
    dW = torch.from_numpy(r["dW"])
    dist.all_reduce(loss)                           # exchange 2: loss and dW
    dist.all_reduce(dW)
    np.save(os.path.join(out_dir, f"dx{rank}.npy"), r["dX"])  # rows stay on their rank
    if rank == 0:
        np.save(os.path.join(out_dir, "dw.npy"), dW.numpy())
        np.save(os.path.join(out_dir, "loss.npy"), loss.numpy())
        np.save(os.path.join(out_dir, "n.npy"), n_global.numpy())
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_shards_reduce_to_the_whole_batch(tmp_path):
    import oracle
    oracle.build()
    world = 2
    mp.spawn(_rank_main, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    X, W, t = _case()
    ref = oracle.flce(X, W, t, IGN)
    assert int(np.load(tmp_path / "n.npy")[0]) == ref["n_valid"]
    assert abs(float(np.load(tmp_path / "loss.npy")[0]) - ref["loss"]) <= 1e-13
    np.testing.assert_allclose(np.load(tmp_path / "dw.npy"), ref["dW"], rtol=1e-11, atol=1e-15)
    dX = np.vstack([np.load(tmp_path / f"dx{r}.npy") for r in range(world)])
    np.testing.assert_allclose(dX, ref["dX"], rtol=1e-11, atol=1e-15)
