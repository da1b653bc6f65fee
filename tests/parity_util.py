"""Tolerances and comparison helpers shared by the GPU parity tests.

Tolerances (fixed for this path): loss |d| <= 1e-3 |ref| + 1e-4; dX and dW
each max|d| <= 2e-2 max|ref| with cosine similarity >= 0.9999; the count of
valid rows bit-exact.  lse uses the loss tolerance row by row.
"""
import numpy as np

LOSS_RTOL, LOSS_ATOL = 1e-3, 1e-4
GRAD_MAX_REL, GRAD_COS = 2e-2, 0.9999


def loss_ok(got: float, ref: float) -> bool:
    return abs(got - ref) <= LOSS_RTOL * abs(ref) + LOSS_ATOL


def assert_loss(got, ref, what="loss"):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    bound = LOSS_RTOL * np.abs(ref) + LOSS_ATOL
    bad = np.abs(got - ref) > bound
    assert not bad.any(), (f"{what}: {int(bad.sum())} entries out of tolerance, worst "
                           f"|d|={np.abs(got - ref).max():.3e} vs bound {bound.max():.3e}")


def grad_stats(got, ref):
    got = np.asarray(got, dtype=np.float64).ravel()
    ref = np.asarray(ref, dtype=np.float64).ravel()
    err = float(np.abs(got - ref).max()) if got.size else 0.0
    mx = float(np.abs(ref).max()) if ref.size else 0.0
    ng, nr = np.linalg.norm(got), np.linalg.norm(ref)
    cos = float(got @ ref / (ng * nr)) if ng > 0 and nr > 0 else (1.0 if ng == nr else 0.0)
    return err, mx, cos


def assert_grad(got, ref, what):
    err, mx, cos = grad_stats(got, ref)
    if mx == 0.0:
        assert err == 0.0, f"{what}: reference is zero but max|got| = {err:.3e}"
        return
    assert err <= GRAD_MAX_REL * mx, f"{what}: max|d| {err:.3e} > {GRAD_MAX_REL} * {mx:.3e}"
    assert cos >= GRAD_COS, f"{what}: cosine {cos:.6f} < {GRAD_COS}"


def assert_grad_blocks(got, ref, what, rows_per_block: int = 4096):
    """assert_grad for a large gradient, block of rows by block of rows (no
    full float64 copy of ``got``): the same criteria (max|d| against max|ref|
    over the whole array, and the cosine over the whole array).  ``got`` is a
    torch tensor (any device) or a numpy array, ``ref`` a float64 array of the
    same shape."""
    import torch
    R = ref.shape[0]
    err = mx = dot = ng2 = nr2 = 0.0
    for a in range(0, R, rows_per_block):
        b = min(a + rows_per_block, R)
        g = got[a:b]
        g = g.double().cpu().numpy() if isinstance(g, torch.Tensor) else np.asarray(g, np.float64)
        r = ref[a:b]
        err = max(err, float(np.abs(g - r).max()) if g.size else 0.0)
        mx = max(mx, float(np.abs(r).max()) if r.size else 0.0)
        dot += float((g * r).sum())
        ng2 += float((g * g).sum())
        nr2 += float((r * r).sum())
    if mx == 0.0:
        assert err == 0.0, f"{what}: reference is zero but max|got| = {err:.3e}"
        return
    cos = dot / np.sqrt(ng2 * nr2) if ng2 > 0 and nr2 > 0 else 0.0
    assert err <= GRAD_MAX_REL * mx, f"{what}: max|d| {err:.3e} > {GRAD_MAX_REL} * {mx:.3e}"
    assert cos >= GRAD_COS, f"{what}: cosine {cos:.6f} < {GRAD_COS}"
