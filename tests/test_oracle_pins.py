"""Pins for the CPU oracle: facts the mathematics fixes, independent of the
oracle's own code.  CPU only.

What the oracle computes is the plain definition of softmax cross-entropy on
the LM-head logits S = X W^T, mean over rows whose target is not the ignore
index, with the exact gradients (Liger-Kernel project overview,
"Método de API de Baixo Nível" and "Cálculo Preciso").  Each pin below is
chosen so that a plausible slip (a dropped term, a sign, an index, a
transposed operand, the wrong normaliser) fails at least one of them.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from flce_synth import WORKLOADS, make_case, make_inputs

GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")))
IGN = -100


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# --------------------------------------------------------------------------- W = 0
@pytest.mark.parametrize("V", [2, 256, 32000, 128256, 152064])
def test_zero_weight_loss_is_log_V(V):
    """W = 0: every logit is 0, so each row's loss is log V exactly."""
    N, H = 3, 8
    X = _rand((N, H), 1)
    W = np.zeros((V, H))
    t = np.array([0, V - 1, V // 2], dtype=np.int64)
    r = oracle.flce(X, W, t, grads=(V <= 256))
    ref = GOLDEN["log_V"][str(V)]
    assert abs(r["loss"] - ref) <= 4e-16 * ref
    assert abs(ref - math.log(V)) <= 4e-16 * ref
    np.testing.assert_allclose(r["lse"], ref, rtol=4e-16)


def test_zero_weight_gradients_closed_form():
    """W = 0: dX = 0 and dW_j = (1/n) sum_valid (1/V - [j = t_i]) x_i."""
    N, H, V = 7, 5, 11
    X = _rand((N, H), 2)
    W = np.zeros((V, H))
    t = np.array([3, IGN, 0, 10, 3, IGN, 7], dtype=np.int64)
    r = oracle.flce(X, W, t, IGN)
    n = 5
    assert r["n_valid"] == n
    np.testing.assert_array_equal(r["dX"], 0.0)
    expect = np.zeros((V, H))
    for i in range(N):
        if t[i] == IGN:
            continue
        expect += np.outer(np.full(V, 1.0 / V), X[i]) / n
        expect[t[i]] -= X[i] / n
    np.testing.assert_allclose(r["dW"], expect, rtol=1e-13, atol=1e-15)


# ------------------------------------------------------------------ G = dW^T with X = I
def test_identity_input_exposes_G_against_scipy_softmax():
    """X = I (N = H) makes dW = G^T, so G is visible: each valid row sums to 0,
    ignored rows are exactly 0, and G = (softmax(S) - onehot)/n_valid with the
    softmax taken from scipy."""
    from scipy.special import softmax
    N = H = 6
    V = 9
    X = np.eye(N)
    W = _rand((V, H), 3, 2.0)
    t = np.array([4, IGN, 8, 0, 4, IGN], dtype=np.int64)
    r = oracle.flce(X, W, t, IGN)
    G = r["dW"].T
    assert G.shape == (N, V)
    np.testing.assert_allclose(G.sum(axis=1), 0.0, atol=1e-15)
    np.testing.assert_array_equal(G[t == IGN], 0.0)
    S = W.T  # S_ij = sum_h I_ih W_jh = W_ji
    P = softmax(S, axis=1)
    n = int((t != IGN).sum())
    for i in range(N):
        if t[i] == IGN:
            continue
        e = P[i].copy()
        e[t[i]] -= 1.0
        np.testing.assert_allclose(G[i], e / n, rtol=1e-12, atol=1e-16)
    # dX_i = sum_j G_ij w_j  -> with X = I the same G gives dX = G W
    np.testing.assert_allclose(r["dX"], G @ W, rtol=1e-12, atol=1e-15)


# --------------------------------------------------------------------------- V = 2
def test_two_class_softplus():
    """V = 2: row loss = softplus(S_other - S_target) = logaddexp(0, d)."""
    N, H = 9, 4
    X = _rand((N, H), 4)
    W = _rand((2, H), 5)
    t = np.array([0, 1, 1, 0, IGN, 1, 0, 0, 1], dtype=np.int64)
    r = oracle.flce(X, W, t, IGN)
    S = X @ W.T
    for i in range(N):
        if t[i] == IGN:
            assert r["loss_rows"][i] == 0.0
            continue
        d = S[i, 1 - t[i]] - S[i, t[i]]
        assert abs(r["loss_rows"][i] - np.logaddexp(0.0, d)) <= 1e-13
    valid = t != IGN
    assert abs(r["loss"] - r["loss_rows"][valid].mean()) <= 1e-14


# ------------------------------------------------------------------------ invariants
def test_loss_nonnegative_and_rows_sum_zero():
    X, W, t = make_case(33, 24, 70, "fp32", seed=11, w_std=0.5, ignore_num=10)
    r = oracle.flce(X, W, t, IGN)
    assert r["loss"] >= 0.0
    assert (r["loss_rows"] >= 0.0).all()
    # sum_j dW_j = sum_i (sum_j G_ij) x_i = 0
    assert np.abs(r["dW"].sum(axis=0)).max() <= 1e-14 * np.abs(r["dW"]).max() * 70
    # rows of dX for ignored targets are exactly zero
    ign = (t == IGN).numpy()
    assert ign.sum() == 3
    np.testing.assert_array_equal(r["dX"][ign], 0.0)


def test_shift_invariance():
    """W + 1 b^T adds x_i.b to every logit of row i: softmax, loss and dW are
    unchanged, and dX = G (W + 1 b^T) = G W because each row of G sums to 0."""
    N, H, V = 6, 5, 13
    X = _rand((N, H), 6)
    W = _rand((V, H), 7)
    b = _rand((H,), 8)
    t = np.array([1, 12, IGN, 5, 5, 0], dtype=np.int64)
    a = oracle.flce(X, W, t, IGN)
    s = oracle.flce(X, W + b[None, :], t, IGN)
    assert abs(a["loss"] - s["loss"]) <= 1e-13
    np.testing.assert_allclose(s["dW"], a["dW"], rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(s["dX"], a["dX"], rtol=1e-11, atol=1e-14)


def test_duplicated_batch():
    """Repeating the batch keeps the mean loss and dW, and halves each dX row
    (the normaliser doubles): pins the 1/n_valid scaling."""
    N, H, V = 5, 7, 10
    X = _rand((N, H), 9)
    W = _rand((V, H), 10)
    t = np.array([2, IGN, 9, 0, 4], dtype=np.int64)
    a = oracle.flce(X, W, t, IGN)
    d = oracle.flce(np.vstack([X, X]), W, np.concatenate([t, t]), IGN)
    assert d["n_valid"] == 2 * a["n_valid"]
    assert abs(d["loss"] - a["loss"]) <= 1e-14
    np.testing.assert_allclose(d["dW"], a["dW"], rtol=1e-12, atol=1e-16)
    np.testing.assert_allclose(d["dX"][:N], a["dX"] / 2, rtol=1e-12, atol=1e-16)


def test_all_ignored_and_empty():
    """Reading taken: no valid row gives loss 0 and zero gradients."""
    N, H, V = 4, 3, 5
    X = _rand((N, H), 12)
    W = _rand((V, H), 13)
    t = np.full(N, IGN, dtype=np.int64)
    r = oracle.flce(X, W, t, IGN)
    assert r["loss"] == 0.0 and r["n_valid"] == 0
    np.testing.assert_array_equal(r["dX"], 0.0)
    np.testing.assert_array_equal(r["dW"], 0.0)
    e = oracle.flce(np.zeros((0, H)), W, np.zeros(0, dtype=np.int64), IGN)
    assert e["loss"] == 0.0 and e["n_valid"] == 0 and e["dW"].shape == (V, H)


def test_bad_target_rejected():
    X = _rand((2, 3), 14)
    W = _rand((4, 3), 15)
    with pytest.raises(oracle.OracleError):
        oracle.flce(X, W, np.array([0, 4]), IGN)
    with pytest.raises(oracle.OracleError):
        oracle.flce(X, W, np.array([-1, 0]), IGN)
    # a custom ignore index is honoured
    r = oracle.flce(X, W, np.array([7, 1]), 7)
    assert r["n_valid"] == 1


# ----------------------------------------------------------------------- brute force
def test_brute_force_every_target_assignment():
    """N = 3, V = 4, H = 2: every assignment of targets (including ignored rows)
    against a 50-digit mpmath evaluation of the unshifted definition; gradients
    against 50-digit central differences of that same evaluation."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    N, H, V = 3, 2, 4
    X = np.round(_rand((N, H), 16), 3)
    W = np.round(_rand((V, H), 17), 3)

    def mp_loss(Xm, Wm, t):
        tot, n = mp.mpf(0), 0
        for i in range(N):
            if t[i] == IGN:
                continue
            s = [mp.fsum(Xm[i][h] * Wm[j][h] for h in range(H)) for j in range(V)]
            tot += mp.log(mp.fsum(mp.exp(v) for v in s)) - s[t[i]]
            n += 1
        return tot / n if n else mp.mpf(0)

    Xm = [[mp.mpf(float(v)) for v in row] for row in X]
    Wm = [[mp.mpf(float(v)) for v in row] for row in W]
    eps = mp.mpf(10) ** -20
    for assign in itertools.product([IGN, 0, 1, 2, 3], repeat=N):
        t = np.array(assign, dtype=np.int64)
        r = oracle.flce(X, W, t, IGN)
        ref = mp_loss(Xm, Wm, t)
        assert abs(r["loss"] - float(ref)) <= 1e-14 * max(1.0, abs(float(ref)))
        if assign not in [(0, 1, 2), (IGN, 3, 3), (2, IGN, IGN), (IGN, IGN, IGN)]:
            continue
        for (i, h) in itertools.product(range(N), range(H)):
            Xp = [row[:] for row in Xm]; Xp[i][h] += eps
            Xn = [row[:] for row in Xm]; Xn[i][h] -= eps
            g = (mp_loss(Xp, Wm, t) - mp_loss(Xn, Wm, t)) / (2 * eps)
            assert abs(r["dX"][i, h] - float(g)) <= 1e-14
        for (j, h) in itertools.product(range(V), range(H)):
            Wp = [row[:] for row in Wm]; Wp[j][h] += eps
            Wn = [row[:] for row in Wm]; Wn[j][h] -= eps
            g = (mp_loss(Xm, Wp, t) - mp_loss(Xm, Wn, t)) / (2 * eps)
            assert abs(r["dW"][j, h] - float(g)) <= 1e-14


# ---------------------------------------------------------------- finite differences
def test_finite_differences_worked_example():
    """Central differences of the oracle's loss against every entry of dX and
    dW on the overview's worked example (N=4, H=128, V=256, float32 inputs
    widened to double)."""
    w = WORKLOADS["tiny_worked_4x128x256_fp32"]
    X, W, t = make_inputs(w)
    X = X.double().numpy().copy()
    W = W.double().numpy().copy()
    r = oracle.flce(X, W, t, IGN)
    h = 1e-5
    # dX: every entry
    fd = np.zeros_like(X)
    for idx in np.ndindex(X.shape):
        x0 = X[idx]
        X[idx] = x0 + h; lp = oracle.flce(X, W, t, IGN, grads=False)["loss"]
        X[idx] = x0 - h; lm = oracle.flce(X, W, t, IGN, grads=False)["loss"]
        X[idx] = x0
        fd[idx] = (lp - lm) / (2 * h)
    assert np.abs(fd - r["dX"]).max() <= 1e-8 * np.abs(r["dX"]).max() + 1e-10
    # dW: every entry; perturbing W[j, k] moves only logit column j
    fdw = np.zeros_like(W)
    for idx in np.ndindex(W.shape):
        w0 = W[idx]
        W[idx] = w0 + h; lp = oracle.flce(X, W, t, IGN, grads=False)["loss"]
        W[idx] = w0 - h; lm = oracle.flce(X, W, t, IGN, grads=False)["loss"]
        W[idx] = w0
        fdw[idx] = (lp - lm) / (2 * h)
    assert np.abs(fdw - r["dW"]).max() <= 1e-8 * np.abs(r["dW"]).max() + 1e-10


# ------------------------------------------------------------- library special case
@pytest.mark.parametrize("case", [
    dict(N=4, H=128, V=256, dtype="fp32", ignore_num=0, seed=1000),
    dict(N=37, H=40, V=301, dtype="bf16", ignore_num=20, seed=3),
    dict(N=64, H=96, V=1000, dtype="bf16", ignore_num=5, seed=4, t_dist="zipf"),
])
def test_against_torch_float64_autograd(case):
    """torch float64 F.linear + F.cross_entropy(ignore_index, mean) + autograd."""
    args = dict(case)
    X, W, t = make_case(args.pop("N"), args.pop("H"), args.pop("V"), **args)
    r = oracle.flce(X, W, t, IGN)
    Xd = X.double().requires_grad_(True)
    Wd = W.double().requires_grad_(True)
    loss = torch.nn.functional.cross_entropy(torch.nn.functional.linear(Xd, Wd), t,
                                             ignore_index=IGN, reduction="mean")
    loss.backward()
    assert abs(r["loss"] - loss.item()) <= 1e-12 * abs(loss.item())
    np.testing.assert_allclose(r["dX"], Xd.grad.numpy(), rtol=1e-9, atol=1e-15)
    np.testing.assert_allclose(r["dW"], Wd.grad.numpy(), rtol=1e-9, atol=1e-15)


def test_row_and_vocab_subsets_match_full():
    X, W, t = make_case(29, 16, 77, "bf16", seed=21, ignore_num=10, w_std=0.3)
    full = oracle.flce(X, W, t, IGN)
    rows = [0, 5, 28, 13]
    sub = oracle.flce_rows(X, W, t, rows, IGN)
    assert sub["n_valid"] == full["n_valid"]
    np.testing.assert_allclose(sub["lse"], full["lse"][rows], rtol=1e-15)
    np.testing.assert_allclose(sub["loss_rows"], full["loss_rows"][rows], rtol=1e-15)
    np.testing.assert_allclose(sub["dX"], full["dX"][rows], rtol=1e-13, atol=1e-18)
    voc = [76, 0, 40]
    dw = oracle.flce_dw_rows(X, W, t, voc, IGN)
    np.testing.assert_allclose(dw, full["dW"][voc], rtol=1e-13, atol=1e-18)


# ------------------------------------------------------------------ generator counts
@pytest.mark.parametrize("name", list(WORKLOADS))
def test_workload_valid_counts(name):
    """n_valid = N - floor(p N) exactly, from the generator's recipe."""
    from flce_synth import targets
    w = WORKLOADS[name]
    t = targets(w.N, w.V, w.t_dist, w.seed, w.ignore_num, 100, w.ignore_index)
    assert oracle.count_valid(t, IGN) == GOLDEN["ignored_counts"][name]
    valid = t[t != IGN]
    assert valid.min() >= 0 and valid.max() < w.V


# ------------------------------------------------- CE on materialised logits
def test_ce_zero_logits_is_log_V():
    """All-zero logits: every valid row's loss is log V, dS = (1/V - onehot)/n."""
    V = 256
    S = np.zeros((5, V))
    t = np.array([0, 255, IGN, 7, 7], dtype=np.int64)
    r = oracle.ce(S, t, IGN)
    assert abs(r["loss"] - GOLDEN["log_V"]["256"]) <= 1e-15 * 6
    expect = np.where((t != IGN)[:, None], np.full((5, V), 1.0 / V), 0.0)
    for i in range(5):
        if t[i] != IGN:
            expect[i, t[i]] -= 1.0
    np.testing.assert_allclose(r["dS"], expect / 4, rtol=1e-14, atol=1e-18)


def test_ce_agrees_with_fused_oracle_through_the_chain_rule():
    """CE on S = X W^T (formed in float64) equals the fused oracle's loss, and
    its dS maps to the fused gradients: dX = dS W, dW = dS^T X."""
    X, W, t = make_case(23, 16, 50, "fp32", seed=51, ignore_num=15, w_std=0.5)
    Xd, Wd = X.double().numpy(), W.double().numpy()
    f = oracle.flce(X, W, t, IGN)
    c = oracle.ce(Xd @ Wd.T, t, IGN)
    assert abs(c["loss"] - f["loss"]) <= 1e-13
    assert c["n_valid"] == f["n_valid"]
    np.testing.assert_allclose(c["lse"], f["lse"], rtol=1e-14)
    np.testing.assert_allclose(c["dS"] @ Wd, f["dX"], rtol=1e-11, atol=1e-16)
    np.testing.assert_allclose(c["dS"].T @ Xd, f["dW"], rtol=1e-11, atol=1e-16)


def test_ce_against_torch_cross_entropy():
    S = torch.randn(40, 300, dtype=torch.float64, generator=torch.Generator().manual_seed(5)) * 3
    t = torch.randint(0, 300, (40,), generator=torch.Generator().manual_seed(6))
    t[::7] = IGN
    r = oracle.ce(S, t, IGN)
    Sg = S.clone().requires_grad_(True)
    loss = torch.nn.functional.cross_entropy(Sg, t, ignore_index=IGN)
    loss.backward()
    assert abs(r["loss"] - loss.item()) <= 1e-12 * loss.item()
    np.testing.assert_allclose(r["dS"], Sg.grad.numpy(), rtol=1e-10, atol=1e-16)
    np.testing.assert_allclose(r["dS"].sum(axis=1), 0.0, atol=1e-15)


def test_ce_masked_columns_equal_deleted_columns():
    """A -inf (masked) logit is a column that is not there: CE over a row with
    masked columns equals CE over the row with those columns deleted (loss,
    lse, the visible gradient), and the masked columns' gradient is 0."""
    g = torch.Generator().manual_seed(11)
    S = torch.randn(12, 90, dtype=torch.float64, generator=g) * 2
    keep = torch.ones(90, dtype=torch.bool)
    keep[:30] = False
    keep[45::4] = False
    vis = torch.nonzero(keep).ravel()
    t_vis = torch.randint(0, len(vis), (12,), generator=g)
    t = vis[t_vis]
    t[5] = IGN
    t_vis[5] = IGN
    Sm = S.clone()
    Sm[:, ~keep] = float("-inf")
    a = oracle.ce(Sm, t, IGN)
    b = oracle.ce(S[:, keep].contiguous(), t_vis, IGN)
    assert abs(a["loss"] - b["loss"]) <= 1e-14 * b["loss"]
    np.testing.assert_allclose(a["lse"], b["lse"], rtol=1e-14)
    np.testing.assert_allclose(a["dS"][:, keep.numpy()], b["dS"], rtol=1e-13, atol=1e-17)
    assert (a["dS"][:, ~keep.numpy()] == 0).all()


# --------------------------------------------- row / vocabulary subset functions
def test_subset_functions_zero_weight_closed_forms():
    """W = 0 pins the sampled-row and sampled-dW-row functions on their own:
    lse = log V, row loss = log V, dX rows = 0, dW rows in closed form."""
    N, H, V = 9, 6, 300
    X = _rand((N, H), 71)
    W = np.zeros((V, H))
    t = np.array([0, 299, IGN, 5, 5, 17, IGN, 150, 2], dtype=np.int64)
    rows = [8, 0, 2, 5]
    r = oracle.flce_rows(X, W, t, rows, IGN)
    np.testing.assert_allclose(r["lse"], math.log(V), rtol=1e-15)
    np.testing.assert_allclose(r["loss_rows"], [math.log(V), math.log(V), 0.0, math.log(V)],
                               rtol=1e-15)
    np.testing.assert_array_equal(r["dX"], 0.0)
    voc = [5, 0, 299, 42]
    dw = oracle.flce_dw_rows(X, W, t, voc, IGN)
    n = int((t != IGN).sum())
    for k, j in enumerate(voc):
        expect = sum((1.0 / V - (1.0 if t[i] == j else 0.0)) * X[i]
                     for i in range(N) if t[i] != IGN) / n
        np.testing.assert_allclose(dw[k], expect, rtol=1e-13, atol=1e-16)


def test_subset_functions_against_torch_autograd():
    X, W, t = make_case(20, 12, 40, "fp32", seed=72, ignore_num=20, w_std=0.7)
    Xd = X.double().requires_grad_(True)
    Wd = W.double().requires_grad_(True)
    torch.nn.functional.cross_entropy(torch.nn.functional.linear(Xd, Wd), t,
                                      ignore_index=IGN).backward()
    rows = [19, 3, 0, 11]
    r = oracle.flce_rows(X, W, t, rows, IGN)
    np.testing.assert_allclose(r["dX"], Xd.grad.numpy()[rows], rtol=1e-10, atol=1e-16)
    voc = [39, 1, 20]
    np.testing.assert_allclose(oracle.flce_dw_rows(X, W, t, voc, IGN), Wd.grad.numpy()[voc],
                               rtol=1e-10, atol=1e-16)


# ------------------------------------------------------- data-parallel shards
def test_shard_normaliser():
    """norm_count > 0 divides by the whole batch's valid count instead of the
    call's own: equal to the default when it is the call's own count; each
    shard matches torch float64 autograd of the sum-reduced cross-entropy
    divided by norm_count; and three row shards' losses and dW add up to the
    whole batch's while their dX rows stack to its dX."""
    X, W, t = make_case(41, 12, 70, "fp32", seed=91, ignore_num=9, w_std=0.5)
    whole = oracle.flce(X, W, t, IGN)
    n = whole["n_valid"]
    own = oracle.flce(X, W, t, IGN, norm_count=n)
    assert own["loss"] == whole["loss"]
    np.testing.assert_array_equal(own["dW"], whole["dW"])
    np.testing.assert_array_equal(own["dX"], whole["dX"])
    parts = np.array_split(np.arange(41), 3)
    loss_sum, dW_sum, dX_rows = 0.0, np.zeros_like(whole["dW"]), []
    for rows in parts:
        Xs, ts = X[rows].contiguous(), t[rows].contiguous()
        r = oracle.flce(Xs, W, ts, IGN, norm_count=n)
        assert r["n_valid"] == int((ts != IGN).sum())
        Xt = Xs.double().requires_grad_(True)
        Wt = W.double().requires_grad_(True)
        ref = torch.nn.functional.cross_entropy(torch.nn.functional.linear(Xt, Wt), ts,
                                                ignore_index=IGN, reduction="sum") / n
        ref.backward()
        assert abs(r["loss"] - ref.item()) <= 1e-13 * abs(ref.item())
        np.testing.assert_allclose(r["dX"], Xt.grad.numpy(), rtol=1e-10, atol=1e-15)
        np.testing.assert_allclose(r["dW"], Wt.grad.numpy(), rtol=1e-10, atol=1e-15)
        loss_sum += r["loss"]
        dW_sum += r["dW"]
        dX_rows.append(r["dX"])
    assert abs(loss_sum - whole["loss"]) <= 1e-13 * whole["loss"]
    np.testing.assert_allclose(dW_sum, whole["dW"], rtol=1e-11, atol=1e-16)
    np.testing.assert_allclose(np.vstack(dX_rows), whole["dX"], rtol=1e-12, atol=1e-16)


# -------------------------------------------------------------- planted mistakes
MUTATIONS = [
    # (name, original text in flce_oracle.c, planted replacement)
    ("one-hot sign in dW", "(t[i] == j ? 1.0 : 0.0);\n        g /= den;",
     "(t[i] == j ? -1.0 : 0.0);\n        g /= den;"),
    ("normaliser N instead of n_valid", "*loss = nv > 0 ? acc / den : 0.0;\n  if (lse)",
     "*loss = nv > 0 ? acc / (double)N : 0.0;\n  if (lse)"),
    ("transposed operand in dX", "dxi[h] += g * elem(W, type, j * H + h);\n        }\n      }\n      free",
     "dxi[h] += g * elem(X, type, i * H + h);\n        }\n      }\n      free"),
    ("dropped max shift", "for (int64_t j = 0; j < V; ++j) s += exp(srow[j] - m);",
     "for (int64_t j = 0; j < V; ++j) s += exp(srow[j]);"),
]


@pytest.mark.parametrize("name,orig,planted", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_pins_catch_a_planted_mistake(tmp_path, name, orig, planted):
    """Compile a copy of the oracle with one plausible slip planted (the
    oracle itself is untouched) and check that the pins reject it."""
    import ctypes
    import subprocess
    src = open(os.path.join(os.path.dirname(oracle.__file__), "flce_oracle.c")).read()
    assert src.count(orig) == 1, name
    p = tmp_path / "mutant.c"
    p.write_text(src.replace(orig, planted))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", str(so),
                    str(p), "-lm"], check=True)
    lib = ctypes.CDLL(str(so))
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.oracle_flce.argtypes = [vp, vp, i32, vp, i64, i64, i64, i64, i64, vp, vp, vp, vp, vp,
                                vp]
    lib.oracle_flce.restype = i32

    def run(X, W, t):
        X = np.ascontiguousarray(X, dtype=np.float64)
        W = np.ascontiguousarray(W, dtype=np.float64)
        t = np.ascontiguousarray(t, dtype=np.int64)
        N, H = X.shape
        V = W.shape[0]
        loss, nv = np.zeros(1), np.zeros(1, dtype=np.int64)
        lse, lr = np.zeros(N), np.zeros(N)
        dX, dW = np.zeros((N, H)), np.zeros((V, H))
        ptr = lambda a: a.ctypes.data_as(vp)  # noqa: E731
        lib.oracle_flce(ptr(X), ptr(W), 0, ptr(t), N, H, V, IGN, 0, ptr(loss), ptr(nv), ptr(lse),
                        ptr(lr), ptr(dX), ptr(dW))
        return loss[0], dX, dW

    # the torch float64 reference and the large-logit case (max shift matters)
    Xc, Wc, tc = make_case(30, 10, 50, "fp32", seed=73, ignore_num=20, w_std=0.5)
    Xt = Xc.double().requires_grad_(True)
    Wt = Wc.double().requires_grad_(True)
    ref = torch.nn.functional.cross_entropy(torch.nn.functional.linear(Xt, Wt), tc,
                                            ignore_index=IGN)
    ref.backward()
    loss, dX, dW = run(Xc.double().numpy(), Wc.double().numpy(), tc.numpy())
    big_loss, _, _ = run(Xc.double().numpy() * 100, Wc.double().numpy() * 100, tc.numpy())
    caught = (abs(loss - ref.item()) > 1e-9 or
              not np.allclose(dX, Xt.grad.numpy(), rtol=1e-8, atol=1e-14) or
              not np.allclose(dW, Wt.grad.numpy(), rtol=1e-8, atol=1e-14) or
              not np.isfinite(big_loss))
    assert caught, f"the pins did not catch: {name}"
