"""Failure detection on the GPU without a fault: the bounded wait every
kernel of the library uses must give up after its limit, report
FLCE_ERR_TIMEOUT through the status word, and leave the context usable."""
import time

import pytest
import torch

from flce_synth import make_case
from parity_util import assert_loss

pytestmark = pytest.mark.gpu


def test_wait_expiry_is_reported_and_the_context_survives(cuda_lib):
    lib = cuda_lib.load_library()
    t0 = time.perf_counter()
    rc = lib.flce_selftest_wait_expiry(50_000_000)  # 50 ms
    dt = time.perf_counter() - t0
    assert rc == cuda_lib.FLCE_ERR_TIMEOUT, lib.flce_last_error()
    assert 0.04 <= dt < 5.0
    assert b"bounded wait" in lib.flce_last_error()
    # the device still answers: a normal call right after is correct
    X, W, t = make_case(64, 64, 512, "bf16", seed=71)
    a = cuda_lib.flce_fwd_bwd_ex(X.cuda(), W.cuda(), t.cuda(), -100, sync=True)
    b = cuda_lib.flce_fwd_bwd_ex(X.cuda(), W.cuda(), t.cuda(), -100, sync=True)
    assert_loss(a[0].item(), b[0].item())
    assert torch.cuda.synchronize() is None


def test_selftest_rejects_bad_limits(cuda_lib):
    lib = cuda_lib.load_library()
    assert lib.flce_selftest_wait_expiry(0) == cuda_lib.FLCE_ERR_ARG
    assert lib.flce_selftest_wait_expiry(3_000_000_000) == cuda_lib.FLCE_ERR_ARG
