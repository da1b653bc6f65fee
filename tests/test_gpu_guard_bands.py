"""Guard bands around every buffer the library writes: the stand-in for a
memory checker's out-of-bounds detection.

Each output (dX, dW, lse, row losses, a caller workspace, the CE gradient)
is the middle of a larger device buffer whose bytes on both sides are filled
with a canary pattern.  After calls on ragged shapes (N, H and V tails,
several chunks, bf16 and fp32, a one-word vocabulary, a 16-byte row) every
canary byte must be untouched, the read-only inputs unchanged, and the
results still equal to the oracle's.
"""
import pytest
import torch

import oracle
from flce_synth import make_case, targets
from parity_util import assert_grad, assert_loss

pytestmark = pytest.mark.gpu
IGN = -100
DEV = "cuda"
PAD = 4096          # bytes of canary on each side (keeps 256-byte alignment)
CANARY = 0xA5


class Guarded:
    """A device tensor of `shape`/`dtype` at the middle of a canary-filled
    uint8 buffer."""

    def __init__(self, shape, dtype):
        n = 1
        for s in shape:
            n *= s
        self.nbytes = n * torch.empty((), dtype=dtype).element_size()
        self.buf = torch.full((PAD + self.nbytes + PAD,), CANARY, dtype=torch.uint8, device=DEV)
        self.t = self.buf[PAD:PAD + self.nbytes].view(dtype).view(*shape)

    def intact(self) -> bool:
        head = self.buf[:PAD]
        tail = self.buf[PAD + self.nbytes:]
        return bool((head == CANARY).all().item()) and bool((tail == CANARY).all().item())


def _inputs(N, H, V, dtype, seed, ign_pct=10):
    X, W, t = make_case(N, H, V, dtype, seed=seed, ignore_num=ign_pct,
                        w_std=0.05 if dtype == "bf16" else 0.1)
    if V == 1:
        t[t != IGN] = 0
    return X, W, t


@pytest.mark.parametrize("N,H,V,dtype,vc", [
    (300, 200, 1000, "bf16", 256),    # four chunks, the last one 232 columns wide
    (513, 136, 3000, "bf16", 512),    # N, H and V tails, six chunks
    (389, 100, 1300, "fp32", 768),    # tf32 path, odd N (padded transposes)
    (70, 64, 1, "bf16", 0),           # a one-word vocabulary
    (1, 8, 257, "bf16", 0),           # one token, 16-byte rows, V one past a tile
    (2050, 136, 777, "bf16", 256),    # 9 pair row-tiles, K tail of 8
])
def test_fused_call_stays_inside_its_buffers(cuda_lib, N, H, V, dtype, vc):
    X, W, t = _inputs(N, H, V, dtype, seed=N + H + V)
    Xd, Wd, td = X.to(DEV), W.to(DEV), t.to(DEV)
    X0, W0, t0 = Xd.clone(), Wd.clone(), td.clone()
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    gdX, gdW = Guarded((N, H), tdt), Guarded((V, H), torch.float32)
    glse, grows = Guarded((N,), torch.float32), Guarded((N,), torch.float32)
    need = cuda_lib.flce_workspace_bytes(N, H, V, True, dtype=tdt, vocab_chunk=vc)
    gws = Guarded((need,), torch.uint8)
    loss, nval, dX, dW = cuda_lib.flce_fwd_bwd_ex(
        Xd, Wd, td, IGN, sync=True, dX=gdX.t, dW=gdW.t, lse_out=glse.t,
        loss_rows_out=grows.t, workspace=gws.t, vocab_chunk=vc)
    for name, g in (("dX", gdX), ("dW", gdW), ("lse", glse), ("row losses", grows),
                    ("workspace", gws)):
        assert g.intact(), f"a write landed outside {name}"
    assert torch.equal(Xd, X0) and torch.equal(Wd, W0) and torch.equal(td, t0)
    ref = oracle.flce(X, W, t, IGN)
    assert int(nval.item()) == ref["n_valid"]
    assert_loss(loss.item(), ref["loss"])
    assert_loss(glse.t.cpu().numpy(), ref["lse"], "lse")
    assert_loss(grows.t.cpu().numpy(), ref["loss_rows"], "row losses")
    if V > 1:
        assert_grad(gdX.t.float().cpu().numpy(), ref["dX"], "dX")
        assert_grad(gdW.t.cpu().numpy(), ref["dW"], "dW")


def test_loss_only_call_stays_inside_its_buffers(cuda_lib):
    N, H, V = 333, 128, 1234
    X, W, t = _inputs(N, H, V, "bf16", seed=5)
    glse, grows = Guarded((N,), torch.float32), Guarded((N,), torch.float32)
    loss, nval = cuda_lib.flce_fwd(X.to(DEV), W.to(DEV), t.to(DEV), IGN, sync=True,
                                   lse_out=glse.t, loss_rows_out=grows.t)
    assert glse.intact() and grows.intact()
    ref = oracle.flce(X, W, t, IGN, grads=False)
    assert_loss(loss.item(), ref["loss"])
    assert_loss(glse.t.cpu().numpy(), ref["lse"], "lse")


@pytest.mark.parametrize("N,V,dtype,inplace", [
    (37, 1001, "bf16", False),    # rows not 16-byte multiples: the scalar path
    (64, 3000, "fp32", False),
    (50, 4096, "bf16", True),     # gradient written over the logits
    (9, 1, "fp32", False),
])
def test_ce_on_logits_stays_inside_its_buffers(cuda_lib, N, V, dtype, inplace):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    S, _, _ = make_case(N, V, 1, dtype, seed=N + V, x_std=3.0)  # logits ~ N(0, 9)
    t = torch.from_numpy(targets(N, V, "uniform", N + V, 10))
    gS = Guarded((N, V), tdt)
    gS.t.copy_(S.to(DEV))
    gdS = gS if inplace else Guarded((N, V), tdt)
    glse = Guarded((N,), torch.float32)
    loss, nval, dS = cuda_lib.flce_ce_fwd_bwd(gS.t, t.to(DEV), IGN, sync=True, dlogits=gdS.t,
                                              lse_out=glse.t)
    assert gS.intact() and gdS.intact() and glse.intact()
    if not inplace:
        assert torch.equal(gS.t.cpu(), S)
    ref = oracle.ce(S, t, IGN)
    assert int(nval.item()) == ref["n_valid"]
    assert_loss(loss.item(), ref["loss"])
    assert_loss(glse.t.cpu().numpy(), ref["lse"], "lse")
    if V > 1:
        assert_grad(gdS.t.float().cpu().numpy(), ref["dS"], "dS")
