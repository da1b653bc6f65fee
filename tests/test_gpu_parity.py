"""GPU parity: the CUDA path through the C ABI against the fp64 CPU oracle,
element by element, at sizes the oracle finishes in seconds; plus the edge
cases (ragged tiles, targets in the last partial vocabulary tile, all rows
ignored, N = 0, bad targets) and the error paths of the boundary."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from flce_synth import make_case
from parity_util import assert_grad, assert_loss

pytestmark = pytest.mark.gpu
IGN = -100
DEV = "cuda"


def _gpu(X, W, t):
    return X.to(DEV), W.to(DEV), t.to(DEV)


def _check_full(flce, X, W, t, vocab_chunk=0, ignore_index=IGN):
    Xd, Wd, td = _gpu(X, W, t)
    N = X.shape[0]
    lse = torch.empty(N, device=DEV)
    rows = torch.empty(N, device=DEV)
    info = {}
    loss, nval, dX, dW = flce.flce_fwd_bwd_ex(Xd, Wd, td, ignore_index, sync=True,
                                              lse_out=lse, loss_rows_out=rows,
                                              vocab_chunk=vocab_chunk, info=info)
    ref = oracle.flce(X, W, t, ignore_index)
    assert int(nval.item()) == ref["n_valid"]
    assert_loss(loss.item(), ref["loss"])
    if N:
        assert_loss(lse.cpu().numpy(), ref["lse"], "lse")
        assert_loss(rows.cpu().numpy(), ref["loss_rows"], "row loss")
        assert_grad(dX.float().cpu().numpy(), ref["dX"], "dX")
    assert_grad(dW.cpu().numpy(), ref["dW"], "dW")
    assert int(info["status"].item()) == 0
    return info


CASES = [
    # N, H, V, dtype, ignored %, vocab_chunk
    (4, 128, 256, "fp32", 0, 0),        # the overview's worked-example shape
    (1, 64, 256, "bf16", 0, 0),         # one row
    (127, 64, 255, "bf16", 10, 0),      # all ragged, V below one vocabulary tile
    (300, 192, 1000, "bf16", 10, 0),    # ragged M, K, V tails
    (513, 320, 3000, "bf16", 5, 512),   # six chunks, ragged last chunk
    (700, 320, 3000, "fp32", 10, 512),  # tf32 path with chunks
    (256, 4096, 2048, "bf16", 2, 0),    # long K (64 stages of the ring)
    (2050, 136, 777, "bf16", 30, 256),  # 17 row tiles, K tail of 8, 4 chunks
    (389, 100, 1300, "fp32", 20, 768),  # fp32 with odd N (transpose padding)
]


@pytest.mark.parametrize("N,H,V,dtype,ign,vc", CASES)
def test_fwd_bwd_matches_oracle(cuda_lib, N, H, V, dtype, ign, vc):
    X, W, t = make_case(N, H, V, dtype, seed=N + V, ignore_num=ign,
                        w_std=0.088 if dtype == "fp32" else 0.02)
    info = _check_full(cuda_lib, X, W, t, vocab_chunk=vc)
    if vc:
        assert info["vocab_chunk"] == vc


def _random_cases(n=24, seed=20261202):
    """Seeded shapes: every N, H and V tail, ignored rows, explicit chunk
    widths (0 = planner) and both element types (fp32 runs on tf32)."""
    rng = np.random.default_rng(seed)
    out = []
    for k in range(n):
        dtype = "fp32" if k % 4 == 3 else "bf16"
        N = int(rng.integers(1, 900))
        H = int(rng.integers(1, 48)) * (4 if dtype == "fp32" else 8)  # 16-byte rows
        V = int(rng.integers(2, 6000))
        ign = min(int(rng.integers(0, 40)), N)
        vc = int(rng.choice([0, 256, 512, 1280, 2048]))
        out.append((N, H, V, dtype, ign, vc))
    return out


@pytest.mark.parametrize("N,H,V,dtype,ign,vc", _random_cases())
def test_randomized_shapes(cuda_lib, N, H, V, dtype, ign, vc):
    X, W, t = make_case(N, H, V, dtype, seed=7 * N + V, ignore_num=ign, w_std=0.05)
    _check_full(cuda_lib, X, W, t, vocab_chunk=vc)


def test_large_logits_range(cuda_lib):
    """W scaled up so logits span about +-40: the max-shifted sums must hold."""
    X, W, t = make_case(200, 256, 1500, "bf16", seed=9, ignore_num=5, w_std=0.15)
    _check_full(cuda_lib, X, W, t)


def test_targets_in_last_partial_tile(cuda_lib):
    X, W, _ = make_case(130, 64, 700, "bf16", seed=11)
    t = torch.arange(130, dtype=torch.int64) % 188 + 512  # every target in [512, 700)
    t[5] = IGN
    _check_full(cuda_lib, X, W, t)
    t2 = torch.full((130,), 699, dtype=torch.int64)     # the very last column
    _check_full(cuda_lib, X, W, t2, vocab_chunk=256)


def test_single_word_vocabulary(cuda_lib):
    """V = 1: the softmax is exactly 1, so the exact loss and gradients are 0.
    The kernels form 2^(S log2 e - lse2) with lse2 rounded in fp32, so they
    may leave a residual of a few ulp of the unit-size terms."""
    X, W, t = make_case(70, 64, 1, "bf16", seed=17)
    t[:] = 0
    loss, nval, dX, dW = cuda_lib.flce_fwd_bwd_ex(*_gpu(X, W, t), IGN, sync=True)
    assert int(nval.item()) == 70
    assert abs(loss.item()) <= 1e-4
    assert dX.float().abs().max().item() <= 1e-5 * W.float().abs().max().item()
    assert dW.abs().max().item() <= 1e-5 * X.float().abs().max().item()


@pytest.mark.parametrize("N,H,V,vc", [
    (90, 64, 2, 0),          # two words: the oracle's loss is the softplus closed form
    (50, 8, 300, 0),         # the narrowest bf16 rows (16 bytes): one K block, mostly fill
    (32, 256, 256000, 0),    # a 256k vocabulary in one chunk (1000 vocabulary tiles)
    (32, 256, 256000, 65536),  # the same in four chunks, ragged last one
])
def test_vocabulary_and_width_extremes(cuda_lib, N, H, V, vc):
    X, W, t = make_case(N, H, V, "bf16", seed=N + H, ignore_num=3, w_std=0.3)
    _check_full(cuda_lib, X, W, t, vocab_chunk=vc)


def test_more_tiles_than_units_in_every_gemm(cuda_lib):
    """4096 x 2048 x 8192: 128 dX pair tiles (16 x 8) for 76 CTA pairs, so
    units run two dX tiles each and the dX GEMM uses both TMEM accumulator
    buffers and the ring's phase flips across tiles; pass 2 and dW also have
    more tiles than units.  Once with the planner's chunk width and once with
    2048-column chunks (dX then takes the fp32 TMA reduce-add path over
    several tiles per unit).  Every output element against the oracle."""
    N, H, V = 4096, 2048, 8192
    X, W, t = make_case(N, H, V, "bf16", seed=4242, ignore_num=3, t_dist="zipf")
    ref = oracle.flce(X, W, t, IGN)
    Xd, Wd, td = _gpu(X, W, t)
    for vc in (0, 2048):
        info = {}
        lse = torch.empty(N, device=DEV)
        loss, nval, dX, dW = cuda_lib.flce_fwd_bwd_ex(Xd, Wd, td, IGN, sync=True,
                                                      lse_out=lse, vocab_chunk=vc, info=info)
        assert int(nval.item()) == ref["n_valid"]
        assert_loss(loss.item(), ref["loss"])
        assert_loss(lse.cpu().numpy(), ref["lse"], "lse")
        assert_grad(dX.float().cpu().numpy(), ref["dX"], f"dX (chunk {info['vocab_chunk']})")
        assert_grad(dW.cpu().numpy(), ref["dW"], f"dW (chunk {info['vocab_chunk']})")
        if vc:
            assert info["vocab_chunk"] == vc


def test_shift_invariance_with_large_row_offsets(cuda_lib):
    """W + 1 b^T adds x_i . b to every logit of row i (here up to about +-45):
    softmax, loss, dW and dX are unchanged because each row of G sums to 0,
    and lse_i moves by x_i . b.  W and b sit on grids (k/256, |k| <= 16, and
    m/16, |m| <= 8) on which W + 1 b^T is exact in bf16.  The shifted problem
    on the GPU must match the oracle's unshifted one."""
    N, H, V = 300, 2048, 3000
    g = torch.Generator().manual_seed(77)
    X, _, t = make_case(N, H, V, "bf16", seed=77, ignore_num=10)
    Wk = torch.randint(-16, 17, (V, H), generator=g).double() / 256
    b = torch.randint(-8, 9, (H,), generator=g).double() / 16
    W = Wk.to(torch.bfloat16)
    Ws = (Wk + b[None, :]).to(torch.bfloat16)
    assert torch.equal(Ws.double(), Wk + b[None, :])  # exact in bf16
    lse = torch.empty(N, device=DEV)
    loss, nval, dX, dW = cuda_lib.flce_fwd_bwd_ex(*_gpu(X, Ws, t), IGN, sync=True, lse_out=lse)
    ref = oracle.flce(X, W, t, IGN)
    shift = (X.double() @ b).numpy()
    assert np.abs(shift).max() > 20.0
    assert int(nval.item()) == ref["n_valid"]
    assert_loss(loss.item(), ref["loss"])
    assert_loss(lse.cpu().numpy(), ref["lse"] + shift, "lse")
    assert_grad(dX.float().cpu().numpy(), ref["dX"], "dX")
    assert_grad(dW.cpu().numpy(), ref["dW"], "dW")


@pytest.mark.parametrize("N,H,V,dtype,vc", [
    (513, 320, 3000, "bf16", 512),
    (389, 100, 1300, "fp32", 768),
])
def test_int32_targets(cuda_lib, N, H, V, dtype, vc):
    """target_is_int32: the ids given as int32 give bit for bit the results of
    the same call with int64 ids (fused path, loss-only path, host-buffer
    entry, CE on logits), the fused results match the oracle, and an int32
    id outside [0, V) is reported as a bad target."""
    X, W, t = make_case(N, H, V, dtype, seed=N + 31, ignore_num=10,
                        w_std=0.05 if dtype == "bf16" else 0.1)
    Xd, Wd, td = _gpu(X, W, t)
    t32 = td.to(torch.int32)
    a = cuda_lib.flce_fwd_bwd_ex(Xd, Wd, td, IGN, sync=True, vocab_chunk=vc)
    b = cuda_lib.flce_fwd_bwd_ex(Xd, Wd, t32, IGN, sync=True, vocab_chunk=vc)
    assert a[0].item() == b[0].item() and int(a[1].item()) == int(b[1].item())
    assert torch.equal(a[2], b[2]) and torch.equal(a[3], b[3])
    ref = oracle.flce(X, W, t, IGN)
    assert int(b[1].item()) == ref["n_valid"]
    assert_loss(b[0].item(), ref["loss"])
    assert_grad(b[2].float().cpu().numpy(), ref["dX"], "dX")
    assert_grad(b[3].cpu().numpy(), ref["dW"], "dW")
    fa = cuda_lib.flce_fwd(Xd, Wd, td, IGN, sync=True)
    fb = cuda_lib.flce_fwd(Xd, Wd, t32, IGN, sync=True)
    assert fa[0].item() == fb[0].item()
    loss_h, dX_h, dW_h = cuda_lib.flce_fwd_bwd_host(X.pin_memory(), W.pin_memory(),
                                                    t.to(torch.int32).pin_memory(), IGN,
                                                    vocab_chunk=vc)
    assert loss_h == a[0].item()
    assert torch.equal(dX_h, a[2].cpu()) and torch.equal(dW_h, a[3].cpu())
    S = (Xd.float() @ Wd.float().t()).to(Xd.dtype).contiguous()
    ca = cuda_lib.flce_ce_fwd_bwd(S, td, IGN, sync=True)
    cb = cuda_lib.flce_ce_fwd_bwd(S, t32, IGN, sync=True)
    assert ca[0].item() == cb[0].item() and torch.equal(ca[2], cb[2])
    bad = t32.clone()
    bad[N // 2] = V
    with pytest.raises(cuda_lib.FlceError) as ei:
        cuda_lib.flce_fwd_bwd_ex(Xd, Wd, bad, IGN, sync=True)
    assert ei.value.status == cuda_lib.FLCE_ERR_TARGET


def test_launch_sequence(cuda_lib):
    """Per-launch trace of a three-chunk call: pass 1, combine, then pass 2,
    dW and dX per chunk, then the bf16 conversion of dX."""
    X, W, t = make_case(300, 128, 2000, "bf16", seed=18, ignore_num=10)
    tr = cuda_lib.Trace(capacity=16)
    cuda_lib.flce_fwd_bwd_ex(*_gpu(X, W, t), IGN, sync=True, vocab_chunk=768, trace=tr)
    kinds = [k for k, _ in tr.launches()]
    assert kinds == ["logits_lse", "combine"] + ["logits_grad", "dw", "dx"] * 3 + ["convert"]


def test_concurrent_calls_on_two_streams(cuda_lib):
    """Calls are reentrant: two asynchronous calls in flight at once on two
    streams, each with the library's own scratch, give exactly the result of
    a lone call (the combine's ticket and scalars live in each call's
    scratch)."""
    X, W, t = make_case(700, 256, 6000, "bf16", seed=19, ignore_num=25)
    Xd, Wd, td = _gpu(X, W, t)
    ref = cuda_lib.flce_fwd_bwd_ex(Xd, Wd, td, IGN, sync=True, vocab_chunk=1024)
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    outs = []
    torch.cuda.synchronize()
    for k, st in enumerate(streams):
        with torch.cuda.stream(st):
            for _ in range(3):  # several calls queued on each stream
                outs.append(cuda_lib.flce_fwd_bwd_ex(Xd, Wd, td, IGN, vocab_chunk=1024))
    torch.cuda.synchronize()
    for loss, nval, dX, dW in outs:
        assert loss.item() == ref[0].item() and int(nval.item()) == int(ref[1].item())
        assert torch.equal(dX, ref[2]) and torch.equal(dW, ref[3])


def test_workspace_budget_is_honoured(cuda_lib):
    """A caller budget below what one 2048-column chunk needs gets the
    2048-column plan; the result matches the oracle."""
    X, W, t = make_case(300, 128, 5000, "bf16", seed=20, ignore_num=10)
    info = {}
    ref = oracle.flce(X, W, t, IGN)
    loss, nval, dX, dW = cuda_lib.flce_fwd_bwd_ex(*_gpu(X, W, t), IGN, sync=True,
                                                  workspace_budget=1 << 20, info=info)
    assert info["vocab_chunk"] == 2048
    assert info["workspace_bytes"] == cuda_lib.flce_workspace_bytes(300, 128, 5000, True,
                                                                    vocab_chunk=2048)
    assert int(nval.item()) == ref["n_valid"]
    assert_loss(loss.item(), ref["loss"])
    assert_grad(dX.float().cpu().numpy(), ref["dX"], "dX")
    assert_grad(dW.cpu().numpy(), ref["dW"], "dW")


def test_all_ignored_gives_zero(cuda_lib):
    X, W, _ = make_case(64, 64, 512, "bf16", seed=12)
    t = torch.full((64,), IGN, dtype=torch.int64)
    loss, nval, dX, dW = cuda_lib.flce_fwd_bwd_ex(*_gpu(X, W, t), IGN, sync=True)
    assert loss.item() == 0.0 and nval.item() == 0
    assert dX.abs().max().item() == 0.0 and dW.abs().max().item() == 0.0


def test_single_valid_row(cuda_lib):
    X, W, _ = make_case(96, 64, 512, "bf16", seed=13)
    t = torch.full((96,), IGN, dtype=torch.int64)
    t[77] = 3
    _check_full(cuda_lib, X, W, t)


def test_empty_batch(cuda_lib):
    X = torch.zeros((0, 64), dtype=torch.bfloat16, device=DEV)
    W = torch.randn(300, 64, device=DEV).to(torch.bfloat16)
    t = torch.zeros((0,), dtype=torch.int64, device=DEV)
    dW = torch.full((300, 64), 7.0, device=DEV)
    loss, nval, dX, dW = cuda_lib.flce_fwd_bwd_ex(X, W, t, IGN, sync=True, dW=dW)
    assert loss.item() == 0.0 and nval.item() == 0
    assert dW.abs().max().item() == 0.0


def test_custom_ignore_index(cuda_lib):
    X, W, t = make_case(150, 64, 600, "bf16", seed=14, ignore_num=20, ignore_index=0)
    _check_full(cuda_lib, X, W, t, ignore_index=0)


def test_bad_target_reports_error(cuda_lib):
    X, W, _ = make_case(40, 64, 300, "bf16", seed=15)
    for bad in (300, -1, 10 ** 9):
        t = torch.zeros(40, dtype=torch.int64)
        t[17] = bad
        with pytest.raises(cuda_lib.FlceError) as ei:
            cuda_lib.flce_fwd_bwd_ex(*_gpu(X, W, t), IGN, sync=True)
        assert ei.value.status == cuda_lib.FLCE_ERR_TARGET
    # asynchronous form: the status lands in the device word
    t = torch.zeros(40, dtype=torch.int64)
    t[0] = 300
    info = {}
    cuda_lib.flce_fwd_bwd_ex(*_gpu(X, W, t), IGN, sync=False, info=info)
    torch.cuda.synchronize()
    assert int(info["status"].item()) == cuda_lib.FLCE_ERR_TARGET
    # a good call afterwards is unaffected
    t[0] = 5
    _check_full(cuda_lib, X, W, t)


def test_loss_only_entry(cuda_lib):
    X, W, t = make_case(333, 128, 1234, "bf16", seed=16, ignore_num=15)
    Xd, Wd, td = _gpu(X, W, t)
    lse = torch.empty(333, device=DEV)
    rows = torch.empty(333, device=DEV)
    info = {}
    loss, nval = cuda_lib.flce_fwd(Xd, Wd, td, IGN, sync=True, lse_out=lse,
                                   loss_rows_out=rows, info=info)
    ref = oracle.flce(X, W, t, IGN, grads=False)
    assert nval.item() == ref["n_valid"]
    assert_loss(loss.item(), ref["loss"])
    assert_loss(lse.cpu().numpy(), ref["lse"], "lse")
    assert_loss(rows.cpu().numpy(), ref["loss_rows"], "row loss")
    # the loss-only plan holds no gradient chunk
    assert info["workspace_bytes"] < cuda_lib.flce_workspace_bytes(333, 128, 1234, True)


def test_simple_and_host_entry_points(cuda_lib):
    X, W, t = make_case(257, 64, 900, "bf16", seed=17, ignore_num=10)
    ref = oracle.flce(X, W, t, IGN)
    loss, dX, dW = cuda_lib.flce_fwd_bwd(*_gpu(X, W, t), IGN)
    assert_loss(loss, ref["loss"])
    assert_grad(dX.float().cpu().numpy(), ref["dX"], "dX")
    assert_grad(dW.cpu().numpy(), ref["dW"], "dW")
    loss_h, dX_h, dW_h = cuda_lib.flce_fwd_bwd_host(X.pin_memory(), W.pin_memory(),
                                                    t.pin_memory(), IGN)
    assert loss_h == loss
    assert torch.equal(dX_h, dX.cpu()) and torch.equal(dW_h, dW.cpu())


@pytest.mark.parametrize("N,H,V,dtype,vc,pinned", [
    (700, 256, 9000, "bf16", 2048, True),   # 5 chunks, 8 W pieces, dW rows sent per chunk
    (300, 128, 3000, "bf16", 0, False),     # pageable host memory
    (100, 64, 2000, "fp32", 512, True),     # fp32 (tf32) path
])
def test_host_entry_overlapped_copies(cuda_lib, N, H, V, dtype, vc, pinned):
    X, W, t = make_case(N, H, V, dtype, seed=N + H, ignore_num=10,
                        w_std=0.088 if dtype == "fp32" else 0.02)
    dev = cuda_lib.flce_fwd_bwd_ex(*_gpu(X, W, t), IGN, sync=True, vocab_chunk=vc)
    if pinned:
        X, W, t = X.pin_memory(), W.pin_memory(), t.pin_memory()
    loss, dX, dW = cuda_lib.flce_fwd_bwd_host(X, W, t, IGN, vocab_chunk=vc)
    assert loss == dev[0].item()
    assert torch.equal(dX, dev[2].cpu()) and torch.equal(dW, dev[3].cpu())
    ref = oracle.flce(X, W, t, IGN)
    assert_loss(loss, ref["loss"])
    assert_grad(dW.numpy(), ref["dW"], "dW")


def test_deterministic(cuda_lib):
    X, W, t = make_case(600, 256, 4000, "bf16", seed=18, ignore_num=5)
    Xd, Wd, td = _gpu(X, W, t)
    a = cuda_lib.flce_fwd_bwd_ex(Xd, Wd, td, IGN, sync=True, vocab_chunk=1024)
    b = cuda_lib.flce_fwd_bwd_ex(Xd, Wd, td, IGN, sync=True, vocab_chunk=1024)
    assert a[0].item() == b[0].item()
    assert torch.equal(a[2], b[2]) and torch.equal(a[3], b[3])


def test_grad_scale_and_norm_count(cuda_lib):
    X, W, t = make_case(300, 128, 800, "bf16", seed=19, ignore_num=10)
    Xd, Wd, td = _gpu(X, W, t)
    base = cuda_lib.flce_fwd_bwd_ex(Xd, Wd, td, IGN, sync=True)
    sc = cuda_lib.flce_fwd_bwd_ex(Xd, Wd, td, IGN, sync=True, grad_scale=0.25)
    assert sc[0].item() == base[0].item()
    torch.testing.assert_close(sc[3], base[3] * 0.25, rtol=1e-2, atol=1e-7)
    n = int(base[1].item())
    nc = cuda_lib.flce_fwd_bwd_ex(Xd, Wd, td, IGN, sync=True, norm_count=2 * n)
    assert abs(nc[0].item() - base[0].item() / 2) <= 1e-6 * base[0].item()
    torch.testing.assert_close(nc[3], base[3] * 0.5, rtol=1e-2, atol=1e-7)


def test_autograd_module(cuda_lib):
    X, W, t = make_case(200, 128, 700, "bf16", seed=20, ignore_num=10)
    ref = oracle.flce(X, W, t, IGN)
    w = W.to(DEV).requires_grad_(True)
    x = X.to(DEV).requires_grad_(True)
    loss = cuda_lib.LinearCrossEntropyLoss(IGN)(w, x, t.to(DEV))
    (3.0 * loss).backward()
    assert_loss(loss.item(), ref["loss"])
    assert_grad(x.grad.float().cpu().numpy(), 3.0 * ref["dX"], "3 dX")
    assert_grad(w.grad.float().cpu().numpy(), 3.0 * ref["dW"], "3 dW")


@pytest.mark.parametrize("sdt,ddt", [(torch.float32, torch.bfloat16), (torch.float32, torch.float32),
                                     (torch.bfloat16, torch.bfloat16),
                                     (torch.bfloat16, torch.float32)])
def test_scale_convert(cuda_lib, sdt, ddt):
    """flce_scale_convert (the autograd backward's grad_output scaling and dW
    cast): bit for bit the fp32 product rounded to the destination type, on
    aligned buffers, on buffers one element off 16-byte alignment (the
    element-by-element path), with a length that is not a multiple of 8,
    without a scale, and in place."""
    g = torch.Generator().manual_seed(3)
    n = 100003
    src = (torch.randn(n + 1, generator=g) * 5).to(sdt).to(DEV)
    scale = torch.tensor([-0.3712], device=DEV)
    for off in (0, 1):
        a = src[off:off + n]
        ref = (a.float() * scale).to(ddt)
        out = torch.empty(n + 1, dtype=ddt, device=DEV)[off:off + n]
        cuda_lib.scale_convert(a, out, scale)
        assert torch.equal(out, ref)
    out = torch.empty(n, dtype=ddt, device=DEV)
    cuda_lib.scale_convert(src[:n], out)
    assert torch.equal(out, src[:n].float().to(ddt))
    if sdt == ddt:
        buf = src[:n].clone()
        cuda_lib.scale_convert(buf, buf, scale)
        assert torch.equal(buf, (src[:n].float() * scale).to(ddt))
    lib = cuda_lib.load_library()
    codes = {torch.float32: cuda_lib.FLCE_FP32, torch.bfloat16: cuda_lib.FLCE_BF16}
    base = torch.empty(64, dtype=torch.float32, device=DEV)
    rc = lib.flce_scale_convert(base.data_ptr(), codes[torch.float32], base.data_ptr() + 8,
                                codes[torch.float32], 32, None, None)
    assert rc == cuda_lib.FLCE_ERR_ARG  # a shifted overlap is refused


def test_caller_workspace(cuda_lib):
    X, W, t = make_case(300, 128, 2000, "bf16", seed=21, ignore_num=10)
    need = cuda_lib.flce_workspace_bytes(300, 128, 2000, True, vocab_chunk=512)
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    ref = oracle.flce(X, W, t, IGN)
    Xd, Wd, td = _gpu(X, W, t)
    loss, _, dX, dW = cuda_lib.flce_fwd_bwd_ex(Xd, Wd, td, IGN, sync=True, workspace=ws,
                                               vocab_chunk=512)
    assert_loss(loss.item(), ref["loss"])
    assert_grad(dW.cpu().numpy(), ref["dW"], "dW")
    with pytest.raises(cuda_lib.FlceError) as ei:
        cuda_lib.flce_fwd_bwd_ex(Xd, Wd, td, IGN, sync=True, workspace=ws[:need // 2],
                                 vocab_chunk=512)
    assert ei.value.status == cuda_lib.FLCE_ERR_WORKSPACE


def test_argument_errors(cuda_lib):
    lib = cuda_lib.load_library()
    X, W, t = _gpu(*make_case(16, 64, 256, "bf16", seed=22))
    dX = torch.empty_like(X)
    dW = torch.empty(256, 64, device=DEV)
    loss = ctypes.c_float()
    call = lambda *a: lib.flce_fwd_bwd(*a)  # noqa: E731
    assert call(None, W.data_ptr(), t.data_ptr(), 16, 64, 256, IGN, ctypes.byref(loss),
                dX.data_ptr(), dW.data_ptr()) == cuda_lib.FLCE_ERR_ARG
    assert call(X.data_ptr(), W.data_ptr(), t.data_ptr(), 16, 64, 0, IGN, ctypes.byref(loss),
                dX.data_ptr(), dW.data_ptr()) == cuda_lib.FLCE_ERR_ARG
    assert call(X.data_ptr(), W.data_ptr(), t.data_ptr(), 16, 64, 256, IGN, None,
                dX.data_ptr(), dW.data_ptr()) == cuda_lib.FLCE_ERR_ARG
    # H * 2 bytes = 24 is not a multiple of 16
    X12 = torch.zeros(16, 12, dtype=torch.bfloat16, device=DEV)
    W12 = torch.zeros(256, 12, dtype=torch.bfloat16, device=DEV)
    assert call(X12.data_ptr(), W12.data_ptr(), t.data_ptr(), 16, 12, 256, IGN,
                ctypes.byref(loss), dX.data_ptr(), dW.data_ptr()) == cuda_lib.FLCE_ERR_ALIGN
    # misaligned X pointer
    assert call(X.data_ptr() + 2, W.data_ptr(), t.data_ptr(), 15, 64, 256, IGN,
                ctypes.byref(loss), dX.data_ptr(), dW.data_ptr()) == cuda_lib.FLCE_ERR_ALIGN
    with pytest.raises(cuda_lib.FlceError) as ei:
        cuda_lib.flce_fwd_bwd_ex(X, W, t, IGN, sync=True, vocab_chunk=300)
    assert ei.value.status == cuda_lib.FLCE_ERR_ARG
    assert lib.flce_last_error()  # a message was left for the caller
