"""The allocation-free loss entry point, flce_fwd_noalloc, called through the
C ABI and compared with flce_fwd on two calls in a row.

flce_fwd_noalloc serves callers that cannot allocate device memory where the
loss is computed (memory planned up front in their own arena, a plugin step
that may not allocate, a latency-bound loop).  Its scratch is a fixed static
array inside the library, shared by all calls; this file is collected last so
that a run stopping at its first failure has run every other test already.
"""
import ctypes

import pytest
import torch

import oracle
from flce_synth import make_case
from parity_util import assert_loss

pytestmark = pytest.mark.gpu
IGN = -100
DEV = "cuda"


def _noalloc(lib, X, W, t, dtype_code):
    N, H = X.shape
    V = W.shape[0]
    loss = torch.full((), float("nan"), dtype=torch.float32, device=DEV)
    lse = torch.full((N,), float("nan"), dtype=torch.float32, device=DEV)
    nval = torch.full((), -1, dtype=torch.int64, device=DEV)
    status = torch.full((), -1, dtype=torch.int32, device=DEV)
    rc = lib.flce_fwd_noalloc(X.data_ptr(), W.data_ptr(), t.data_ptr(), N, H, V, IGN,
                              dtype_code, loss.data_ptr(), lse.data_ptr(), nval.data_ptr(),
                              status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return rc, loss, lse, nval, status


def test_noalloc_matches_fwd_on_two_calls_in_a_row(cuda_lib):
    lib = cuda_lib.load_library()
    # a larger call first, then a smaller one that reuses the scratch the
    # first call left behind
    cases = [(1500, 256, 9000, "bf16", 33), (333, 128, 2100, "bf16", 34)]
    for N, H, V, dtype, seed in cases:
        X, W, t = make_case(N, H, V, dtype, seed=seed, ignore_num=10)
        X, W, t = X.to(DEV), W.to(DEV), t.to(DEV)
        assert cuda_lib.flce_workspace_bytes(N, H, V, with_grads=False) < 32 * 2 ** 20
        ref_lse = torch.empty(N, device=DEV)
        ref_loss, ref_nv = cuda_lib.flce_fwd(X, W, t, IGN, sync=True, lse_out=ref_lse)
        rc, loss, lse, nval, status = _noalloc(lib, X, W, t, cuda_lib.FLCE_BF16)
        assert rc == cuda_lib.FLCE_OK, lib.flce_last_error()
        assert int(status.item()) == cuda_lib.FLCE_OK
        assert int(nval.item()) == int(ref_nv.item())
        assert_loss(loss.item(), ref_loss.item())
        assert_loss(lse.cpu().numpy(), ref_lse.cpu().numpy(), "lse")


def test_noalloc_fp32_matches_fwd_and_the_oracle(cuda_lib):
    lib = cuda_lib.load_library()
    X, W, t = make_case(333, 128, 2100, "fp32", seed=35, ignore_num=10, w_std=0.1)
    Xd, Wd, td = X.to(DEV), W.to(DEV), t.to(DEV)
    ref_lse = torch.empty(333, device=DEV)
    ref_loss, ref_nv = cuda_lib.flce_fwd(Xd, Wd, td, IGN, sync=True, lse_out=ref_lse)
    for _ in range(2):
        rc, loss, lse, nval, status = _noalloc(lib, Xd, Wd, td, cuda_lib.FLCE_FP32)
        assert rc == cuda_lib.FLCE_OK, lib.flce_last_error()
        assert int(status.item()) == cuda_lib.FLCE_OK
        assert int(nval.item()) == int(ref_nv.item())
        assert_loss(loss.item(), ref_loss.item())
        assert_loss(lse.cpu().numpy(), ref_lse.cpu().numpy(), "lse")
    orc = oracle.flce(X, W, t, IGN, grads=False)
    assert int(nval.item()) == orc["n_valid"]
    assert_loss(loss.item(), orc["loss"])
    assert_loss(lse.cpu().numpy(), orc["lse"], "lse vs oracle")


def test_noalloc_python_wrapper(cuda_lib):
    X, W, t = make_case(700, 192, 5000, "bf16", seed=36, ignore_num=10)
    Xd, Wd, td = X.to(DEV), W.to(DEV), t.to(DEV)
    ref_lse = torch.empty(700, device=DEV)
    ref_loss, ref_nv = cuda_lib.flce_fwd(Xd, Wd, td, IGN, sync=True, lse_out=ref_lse)
    lse = torch.empty(700, device=DEV)
    loss, nval, status = cuda_lib.flce_fwd_noalloc(Xd, Wd, td, IGN, lse_out=lse)
    torch.cuda.synchronize()
    assert int(status.item()) == cuda_lib.FLCE_OK
    assert int(nval.item()) == int(ref_nv.item())
    assert_loss(loss.item(), ref_loss.item())
    assert_loss(lse.cpu().numpy(), ref_lse.cpu().numpy(), "lse")
    with pytest.raises(ValueError):  # a too-short lse buffer is refused before the call
        cuda_lib.flce_fwd_noalloc(Xd, Wd, td, IGN, lse_out=torch.empty(699, device=DEV))


def test_noalloc_leaves_device_memory_unchanged(cuda_lib):
    """Once the first call on the device has looked up the static array,
    further calls take no device memory at all: the device's free memory is
    the same before and after them."""
    lib = cuda_lib.load_library()
    X, W, t = make_case(1500, 256, 9000, "bf16", seed=37, ignore_num=10)
    Xd, Wd, td = X.to(DEV), W.to(DEV), t.to(DEV)
    rc, *_ = _noalloc(lib, Xd, Wd, td, cuda_lib.FLCE_BF16)  # the first call sets up
    assert rc == cuda_lib.FLCE_OK
    loss = torch.empty((), dtype=torch.float32, device=DEV)
    lse = torch.empty(1500, dtype=torch.float32, device=DEV)
    nval = torch.empty((), dtype=torch.int64, device=DEV)
    status = torch.empty((), dtype=torch.int32, device=DEV)
    stream = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        rc = lib.flce_fwd_noalloc(Xd.data_ptr(), Wd.data_ptr(), td.data_ptr(), 1500, 256, 9000,
                                  IGN, cuda_lib.FLCE_BF16, loss.data_ptr(), lse.data_ptr(),
                                  nval.data_ptr(), status.data_ptr(), stream)
        assert rc == cuda_lib.FLCE_OK, lib.flce_last_error()
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert int(status.item()) == cuda_lib.FLCE_OK


def test_noalloc_rejects_a_problem_beyond_its_scratch(cuda_lib):
    lib = cuda_lib.load_library()
    X = torch.zeros((8, 64), dtype=torch.bfloat16, device=DEV)
    W = torch.zeros((8, 64), dtype=torch.bfloat16, device=DEV)
    t = torch.zeros(8, dtype=torch.int64, device=DEV)
    loss = torch.empty((), dtype=torch.float32, device=DEV)
    # N = 65536 tokens over V = 128256 needs ~131 MB of scratch: rejected
    # before any launch (the small buffers above are never read)
    rc = lib.flce_fwd_noalloc(X.data_ptr(), W.data_ptr(), t.data_ptr(), 65536, 64, 128256, IGN,
                              cuda_lib.FLCE_BF16, loss.data_ptr(), None, None, None, None)
    assert rc == cuda_lib.FLCE_ERR_WORKSPACE
    assert b"static scratch" in lib.flce_last_error()
