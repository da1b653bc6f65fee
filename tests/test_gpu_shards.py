"""The sharded (data-parallel) variant on the CUDA path: a batch split into
row shards, each shard run through the C ABI's ``flce_fwd_bwd_ex`` with
``norm_count`` set to the whole batch's valid count, exactly as one rank of a
data-parallel job would after an all-reduce of the count.

The shards' losses and dW add up, and their dX rows stack, to the oracle's
results on the whole batch (within the path's tolerances); each shard also
matches the oracle's own shard call (``oracle.flce(..., norm_count=n)``).
The shards run one after the other on one GPU; the exchange itself (count,
loss and dW all-reduces) is exercised with gloo ranks on CPU in
``tests/test_sharding_cpu.py``.
"""
import numpy as np
import pytest
import torch

import oracle
from flce_synth import make_case
from parity_util import assert_grad, assert_loss

pytestmark = pytest.mark.gpu
IGN = -100
DEV = "cuda"


def _run_shards(flce, X, W, t, bounds, vocab_chunk=0):
    n_global = int((t != IGN).sum())
    Wd = W.to(DEV)
    loss_sum, dW_sum, dX_rows, per_shard = 0.0, None, [], []
    for a, b in bounds:
        Xs, ts = X[a:b].contiguous(), t[a:b].contiguous()
        loss, nval, dX, dW = flce.flce_fwd_bwd_ex(Xs.to(DEV), Wd, ts.to(DEV), IGN, sync=True,
                                                  norm_count=n_global, vocab_chunk=vocab_chunk)
        assert int(nval.item()) == int((ts != IGN).sum())
        loss_sum += loss.item()
        dW_sum = dW.double() if dW_sum is None else dW_sum + dW.double()
        dX_rows.append(dX.float().cpu())
        per_shard.append((Xs, ts, loss.item(), dX.float().cpu().numpy(), dW.cpu().numpy()))
    return n_global, loss_sum, dW_sum.cpu().numpy(), torch.cat(dX_rows).numpy(), per_shard


@pytest.mark.parametrize("N,H,V,dtype,ign_pct,bounds,vc", [
    (700, 256, 3000, "bf16", 10, [(0, 300), (300, 301), (301, 700)], 0),
    (1000, 192, 2500, "bf16", 10, [(0, 500), (500, 1000)], 512),
    (389, 100, 1300, "fp32", 10, [(0, 130), (130, 260), (260, 389)], 768),
])
def test_shards_add_up_to_the_whole_batch(cuda_lib, N, H, V, dtype, ign_pct, bounds, vc):
    X, W, t = make_case(N, H, V, dtype, seed=3 * N + V, ignore_num=ign_pct,
                        w_std=0.05 if dtype == "bf16" else 0.1)
    n, loss_sum, dW, dX, per_shard = _run_shards(cuda_lib, X, W, t, bounds, vc)
    ref = oracle.flce(X, W, t, IGN)
    assert n == ref["n_valid"]
    assert_loss(loss_sum, ref["loss"])
    assert_grad(dW, ref["dW"], "dW summed over shards")
    assert_grad(dX, ref["dX"], "dX stacked over shards")
    for Xs, ts, loss, dXs, dWs in per_shard:
        r = oracle.flce(Xs, W, ts, IGN, norm_count=n)
        assert_loss(loss, r["loss"], "shard loss")
        if int((ts != IGN).sum()):
            assert_grad(dXs, r["dX"], "shard dX")
            assert_grad(dWs, r["dW"], "shard dW")


def test_a_shard_with_no_valid_row(cuda_lib):
    """A shard whose rows are all ignored contributes 0 to the loss and to dW
    and has zero dX rows, also with a global normaliser."""
    X, W, t = make_case(200, 128, 900, "bf16", seed=5, ignore_num=0)
    t[50:120] = IGN
    n, loss_sum, dW, dX, per_shard = _run_shards(cuda_lib, X, W, t,
                                                 [(0, 50), (50, 120), (120, 200)])
    _, ts, loss_mid, dX_mid, dW_mid = per_shard[1]
    assert int((ts != IGN).sum()) == 0
    assert loss_mid == 0.0
    assert not np.any(dX_mid) and not np.any(dW_mid)
    ref = oracle.flce(X, W, t, IGN)
    assert n == ref["n_valid"]
    assert_loss(loss_sum, ref["loss"])
    assert_grad(dW, ref["dW"], "dW summed over shards")
    assert_grad(dX, ref["dX"], "dX stacked over shards")
