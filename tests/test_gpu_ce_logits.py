"""GPU parity of cross-entropy on materialised logits (flce_ce_fwd_bwd)
against the fp64 oracle's oracle_ce, element by element."""
import numpy as np
import pytest
import torch

import oracle
from flce_synth import make_case, normal_tensor
from parity_util import assert_grad, assert_loss

pytestmark = pytest.mark.gpu
IGN = -100
DEV = "cuda"


def _logits(N, V, dtype, seed, std=2.0):
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    return normal_tensor((N, V), std, seed, 9, dt)


def _targets(N, V, seed, ignore_num):
    _, _, t = make_case(N, 8, V, "fp32", seed=seed, ignore_num=ignore_num)
    return t


@pytest.mark.parametrize("N,V,dtype,ign", [
    # 16-byte vector path (rows 16-byte aligned, V * elt % 16 == 0)
    (4, 256, "fp32", 0),            # rows shorter than one pass of the CTA
    (300, 1000, "bf16", 10),        # vector tail only
    (129, 32000, "bf16", 20),       # unrolled body and tail
    (33, 128256, "bf16", 3),        # a Llama-3-sized row
    (40, 60000, "bf16", 10),
    (17, 128256, "fp32", 0),        # fp32 row of 513 KB
    (301, 4096, "fp32", 30),        # 2 rows on most CTAs
    (700, 20000, "bf16", 5),        # several rows per CTA
    # scalar path (a row is not a multiple of 16 bytes)
    (257, 777, "bf16", 5),
    (64, 5003, "fp32", 0),
])
def test_ce_matches_oracle(cuda_lib, N, V, dtype, ign):
    S = _logits(N, V, dtype, seed=N + V)
    t = _targets(N, V, seed=V, ignore_num=ign)
    ref = oracle.ce(S, t, IGN)
    lse = torch.empty(N, device=DEV)
    rows = torch.empty(N, device=DEV)
    loss, nval, dS = cuda_lib.flce_ce_fwd_bwd(S.to(DEV), t.to(DEV), IGN, sync=True,
                                              lse_out=lse, loss_rows_out=rows)
    assert int(nval.item()) == ref["n_valid"]
    assert_loss(loss.item(), ref["loss"])
    assert_loss(lse.cpu().numpy(), ref["lse"], "lse")
    assert_loss(rows.cpu().numpy(), ref["loss_rows"], "row loss")
    assert_grad(dS.float().cpu().numpy(), ref["dS"], "dS")


@pytest.mark.parametrize("N,V,dtype", [
    (64, 32000, "bf16"),    # vector path, one CTA per row
    (40, 60000, "fp32"),    # vector path, rows split across a cluster
    (50, 777, "bf16"),      # scalar path
])
def test_ce_masked_logits(cuda_lib, N, V, dtype):
    """-inf (masked) logits: a long run at the start of even rows, so that
    whole batches a thread reads first are masked, and every 7th column of odd
    rows.  Masked entries add nothing to lse and get a zero gradient."""
    S = _logits(N, V, dtype, seed=N + 3 * V)
    masked = torch.zeros((N, V), dtype=torch.bool)
    masked[0::2, : V // 3] = True
    masked[1::2, 0::7] = True
    S[masked] = float("-inf")
    i = torch.arange(N, dtype=torch.int64)
    t = V // 3 + (i * 7919) % (V - V // 3)
    t = torch.where(t % 7 == 0, t + 1, t).clamp(max=V - 1)
    t[t % 7 == 0] -= 2
    t[::9] = IGN
    assert not masked[i[t != IGN], t[t != IGN]].any()
    ref = oracle.ce(S, t, IGN)
    assert np.isfinite(ref["loss"])
    lse = torch.empty(N, device=DEV)
    loss, nval, dS = cuda_lib.flce_ce_fwd_bwd(S.to(DEV), t.to(DEV), IGN, sync=True, lse_out=lse)
    assert int(nval.item()) == ref["n_valid"]
    assert_loss(loss.item(), ref["loss"])
    assert_loss(lse.cpu().numpy(), ref["lse"], "lse")
    got = dS.float().cpu()
    assert torch.isfinite(got).all()
    assert (got[masked] == 0).all()
    assert_grad(got.numpy(), ref["dS"], "dS")


@pytest.mark.parametrize("dtype,scale", [("bf16", -0.5), ("fp32", -2.0), ("bf16", 0.0),
                                         ("bf16", 3.0)])
def test_ce_grad_scale_signs(cuda_lib, dtype, scale):
    """dS for a negative, a zero and a positive grad_scale.  A positive scale
    is folded into the exponent; any other multiplies the softmax (the two
    forms of the gradient pass).  Against the oracle's dS times the scale."""
    N, V = 37, 20000
    S = _logits(N, V, dtype, seed=71)
    t = _targets(N, V, seed=72, ignore_num=10)
    ref = oracle.ce(S, t, IGN)
    loss, nval, dS = cuda_lib.flce_ce_fwd_bwd(S.to(DEV), t.to(DEV), IGN, sync=True,
                                              grad_scale=scale)
    assert int(nval.item()) == ref["n_valid"]
    assert_loss(loss.item(), ref["loss"])
    got = dS.float().cpu().numpy()
    if scale == 0.0:
        assert not got.any()
    else:
        assert_grad(got, scale * ref["dS"], f"dS x {scale}")


def test_ce_in_place_and_loss_only(cuda_lib):
    S = _logits(200, 3000, "bf16", seed=61)
    t = _targets(200, 3000, seed=62, ignore_num=10)
    ref = oracle.ce(S, t, IGN)
    buf = S.to(DEV)
    loss, _, dS = cuda_lib.flce_ce_fwd_bwd(buf, t.to(DEV), IGN, sync=True, inplace=True)
    assert dS.data_ptr() == buf.data_ptr()
    assert_loss(loss.item(), ref["loss"])
    assert_grad(buf.float().cpu().numpy(), ref["dS"], "in-place dS")
    S2 = S.to(DEV)
    loss2, _, none = cuda_lib.flce_ce_fwd_bwd(S2, t.to(DEV), IGN, sync=True, grad=False)
    assert none is None and loss2.item() == loss.item()
    assert torch.equal(S2.cpu(), S)  # the logits are untouched without a gradient


def test_ce_in_place_long_rows(cuda_lib):
    """In place with long rows and two rows on some CTAs: each element is
    read twice (statistics, then gradient) and then overwritten."""
    S = _logits(180, 50000, "bf16", seed=67)
    t = _targets(180, 50000, seed=68, ignore_num=7)
    ref = oracle.ce(S, t, IGN)
    buf = S.to(DEV)
    loss, _, _ = cuda_lib.flce_ce_fwd_bwd(buf, t.to(DEV), IGN, sync=True, inplace=True)
    assert_loss(loss.item(), ref["loss"])
    assert_grad(buf.float().cpu().numpy(), ref["dS"], "in-place dS")


def test_ce_matches_fused_path_on_the_same_logits(cuda_lib):
    """S = X W^T materialised in fp32: CE on S equals the fused loss (same
    definition, different kernels)."""
    X, W, t = make_case(300, 128, 2000, "bf16", seed=63, ignore_num=10)
    Xd, Wd, td = X.to(DEV), W.to(DEV), t.to(DEV)
    S = (Xd.float() @ Wd.float().t()).contiguous()
    a = cuda_lib.flce_ce_fwd_bwd(S, td, IGN, sync=True)
    b = cuda_lib.flce_fwd_bwd_ex(Xd, Wd, td, IGN, sync=True)
    assert_loss(a[0].item(), b[0].item())
    assert_grad((a[2] @ Wd.float()).cpu().numpy(), b[2].float().cpu().numpy(), "dS W vs dX")


def test_ce_edge_cases(cuda_lib):
    S = _logits(50, 400, "bf16", seed=64).to(DEV)
    t = torch.full((50,), IGN, dtype=torch.int64, device=DEV)
    loss, nval, dS = cuda_lib.flce_ce_fwd_bwd(S, t, IGN, sync=True)
    assert loss.item() == 0.0 and nval.item() == 0 and dS.abs().max().item() == 0.0
    t[3] = 400
    with pytest.raises(cuda_lib.FlceError) as ei:
        cuda_lib.flce_ce_fwd_bwd(S, t, IGN, sync=True)
    assert ei.value.status == cuda_lib.FLCE_ERR_TARGET
    e = cuda_lib.flce_ce_fwd_bwd(torch.zeros((0, 400), device=DEV),
                                 torch.zeros(0, dtype=torch.int64, device=DEV), IGN, sync=True)
    assert e[0].item() == 0.0 and e[1].item() == 0


def test_ce_autograd_module(cuda_lib):
    S = _logits(100, 900, "fp32", seed=65)
    t = _targets(100, 900, seed=66, ignore_num=10)
    ref = oracle.ce(S, t, IGN)
    x = S.to(DEV).requires_grad_(True)
    loss = cuda_lib.CrossEntropyLoss(IGN)(x, t.to(DEV))
    (2.0 * loss).backward()
    assert_loss(loss.item(), ref["loss"])
    assert_grad(x.grad.cpu().numpy(), 2.0 * ref["dS"], "2 dS")
