"""The asynchronous entry point inside a CUDA graph.

A training step captured in a CUDA graph replays the path with no host work
per launch.  flce_fwd_bwd_ex (sync off) makes only stream-ordered calls
(workspace allocation and release, memsets, kernel launches with
programmatic dependencies), so it can be captured; replays on new input
values in the same buffers must reproduce an eager call bit for bit (every
kernel of the path is deterministic)."""
import pytest
import torch

import oracle
from flce_synth import make_case
from parity_util import assert_grad, assert_loss

pytestmark = pytest.mark.gpu
IGN = -100
DEV = "cuda"
SHAPE = (600, 256, 5000)  # three vocabulary chunks of 2048 columns, ragged last one


def _fill(bufs, seed):
    X, W, t = make_case(*SHAPE, "bf16", seed=seed, ignore_num=30, w_std=0.3)
    for b, v in zip(bufs, (X, W, t)):
        b.copy_(v.to(DEV))
    return X, W, t


@pytest.mark.parametrize("own_workspace", [False, True])
def test_graph_replay_matches_eager(cuda_lib, own_workspace):
    N, H, V = SHAPE
    Xd = torch.empty((N, H), dtype=torch.bfloat16, device=DEV)
    Wd = torch.empty((V, H), dtype=torch.bfloat16, device=DEV)
    td = torch.empty(N, dtype=torch.int64, device=DEV)
    bufs = (Xd, Wd, td)
    _fill(bufs, 70)
    kw = dict(vocab_chunk=2048)
    if own_workspace:
        need = cuda_lib.flce_workspace_bytes(N, H, V, True, vocab_chunk=2048)
        kw["workspace"] = torch.empty(need, dtype=torch.uint8, device=DEV)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside the capture
        for _ in range(2):
            cuda_lib.flce_fwd_bwd_ex(Xd, Wd, td, IGN, **kw)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    info = {}
    with torch.cuda.graph(graph):
        loss, nval, dX, dW = cuda_lib.flce_fwd_bwd_ex(Xd, Wd, td, IGN, info=info, **kw)

    for seed in (71, 72):
        X, W, t = _fill(bufs, seed)
        graph.replay()
        torch.cuda.synchronize()
        assert int(info["status"].item()) == 0
        e_loss, e_nval, e_dX, e_dW = cuda_lib.flce_fwd_bwd_ex(Xd, Wd, td, IGN, sync=True, **kw)
        assert loss.item() == e_loss.item()
        assert int(nval.item()) == int(e_nval.item())
        assert torch.equal(dX, e_dX) and torch.equal(dW, e_dW)
        ref = oracle.flce(X, W, t, IGN)
        assert int(nval.item()) == ref["n_valid"]
        assert_loss(loss.item(), ref["loss"])
        assert_grad(dX.float().cpu().numpy(), ref["dX"], "dX (graph)")
        assert_grad(dW.cpu().numpy(), ref["dW"], "dW (graph)")
