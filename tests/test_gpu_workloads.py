"""GPU parity at the workloads' full sizes, in the launch configuration the
benchmark times (default planner, default stream, bf16).

Each workload's inputs are drawn once and its full GPU call is made once (a
class-scoped fixture, one test class per workload, so one workload is
resident at a time); the tests then compare that run with the oracle:
  * small head (2048 x 2048 x 32000): the whole problem in full (loss, count,
    lse, row losses, dX, dW);
  * Qwen2-7B head and long-context head: the first 1024 tokens as a problem
    of their own on the GPU against the oracle's run on those 1024 rows
    (loss, count, lse, row losses, dX, dW in full); and rows 0-1023 of the
    full GPU run against the same oracle run (lse and row losses directly, dX
    rescaled by the ratio of the two valid counts);
  * Llama-3-8B head: dW rows of the full run (every row of the first targets,
    the vocabulary edges, random rows) against the oracle over all 8192
    tokens, and a 64-token prefix problem;
  * every workload: sampled token rows of the full run (lse, row loss, dX
    row), the count bit-exact against N - floor(p N), the loss rechecked on
    the host from the GPU's lse and host-double target logits, sum_j dW_j = 0,
    and the workspace bound.
"""
import json
import os
from types import SimpleNamespace

import numpy as np
import pytest
import torch

import oracle
from flce_synth import WORKLOADS, make_inputs
from parity_util import (GRAD_COS, GRAD_MAX_REL, assert_grad, assert_grad_blocks,
                         assert_loss)

pytestmark = pytest.mark.gpu
IGN = -100
DEV = "cuda"
GOLDEN = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "closed_forms.json")))
SMALL = "small_head_2048x2048x32000"
LLAMA = "llama3_8b_head_8192x4096x128256"
QWEN = "qwen2_7b_head_16384x3584x152064"
LONG = "long_context_65536x4096x128256"


def _sample_rows(t: torch.Tensor, k: int = 10, seed: int = 0):
    N = t.shape[0]
    rng = np.random.default_rng(seed)
    rows = {0, 1, N - 1, N // 2}
    ign = torch.nonzero(t == IGN).flatten().tolist()
    if ign:
        rows.add(ign[0])
    rows.update(rng.choice(N, size=k, replace=False).tolist())
    return sorted(rows)


def _make_run(name, cuda_lib):
    """Inputs of one workload and its full GPU call."""
    w = WORKLOADS[name]
    X, W, t = make_inputs(w)
    Xd, Wd, td = X.to(DEV), W.to(DEV), t.to(DEV)
    lse = torch.empty(w.N, device=DEV)
    rows_out = torch.empty(w.N, device=DEV)
    info = {}
    loss, nval, dX, dW = cuda_lib.flce_fwd_bwd_ex(Xd, Wd, td, IGN, sync=True, lse_out=lse,
                                                  loss_rows_out=rows_out, info=info)
    return SimpleNamespace(name=name, w=w, X=X, W=W, t=t, Xd=Xd, Wd=Wd, td=td,
                           loss=loss.item(), n=int(nval.item()), dX=dX, dW=dW, lse=lse,
                           rows_out=rows_out, info=info, cache={})


def _prefix_oracle(r, P):
    """The oracle on the first P tokens as a problem of their own (cached)."""
    key = ("prefix", P)
    if key not in r.cache:
        r.cache[key] = oracle.flce(r.X[:P].contiguous(), r.W, r.t[:P].contiguous(), IGN)
    return r.cache[key]


@pytest.fixture(scope="class")
def run(request, cuda_lib):
    """The full run of the requesting class's workload (class attribute NAME),
    made once per class."""
    r = _make_run(request.cls.NAME, cuda_lib)
    yield r
    r.__dict__.clear()
    torch.cuda.empty_cache()


class _EveryWorkload:
    """Checks made on every workload's full run."""
    NAME = None

    def test_count_loss_recheck_and_properties(self, run):
        """Count bit-exact; the loss and every row loss rechecked on the host
        from the GPU's lse and target logits S_{i,t_i} = x_i . w_{t_i} taken in
        double from the inputs; sum_j dW_j = 0; finite outputs; the workspace
        bound."""
        r = run
        w = r.w
        assert r.n == GOLDEN["ignored_counts"][r.name]
        valid = (r.t != IGN)
        tv = torch.where(valid, r.t, torch.zeros_like(r.t))
        s_t = torch.empty(w.N, dtype=torch.float64)
        for a in range(0, w.N, 8192):  # x_i . w_{t_i} in double, on the host
            b = min(a + 8192, w.N)
            s_t[a:b] = (r.X[a:b].double() * r.W[tv[a:b]].double()).sum(dim=1)
        lse = r.lse.double().cpu()
        host_rows = torch.where(valid, lse - s_t, torch.zeros_like(lse))
        assert_loss(r.rows_out.cpu().numpy(), host_rows.numpy(), "row losses vs host recheck")
        assert_loss(r.loss, host_rows.sum().item() / r.n, "loss vs host recheck")
        assert abs(r.loss - r.rows_out.double().sum().item() / r.n) <= 1e-5 * r.loss
        col_sum = r.dW.double().sum(dim=0).abs()
        col_abs = r.dW.double().abs().sum(dim=0)
        assert (col_sum <= 1e-2 * col_abs + 1e-12).all(), "sum_j dW_j is not ~0"
        assert torch.isfinite(r.dX.float()).all() and torch.isfinite(r.dW).all()
        # one sixteenth of the N x V fp32 logits, where the fp32 dX accumulator
        # itself fits under it
        bound = w.N * w.V * 4 // 16
        if w.N * w.H * 4 < bound // 2:
            assert r.info["workspace_bytes"] <= bound

    def test_sampled_rows_against_oracle(self, run):
        r = run
        rows = _sample_rows(r.t, seed=r.w.seed)
        ref = oracle.flce_rows(r.X, r.W, r.t, rows, IGN)
        assert ref["n_valid"] == r.n
        assert_loss(r.lse[rows].cpu().numpy(), ref["lse"], "lse rows")
        assert_loss(r.rows_out[rows].cpu().numpy(), ref["loss_rows"], "row losses")
        assert_grad(r.dX[rows].float().cpu().numpy(), ref["dX"], "dX rows")


# ------------------------------------------------------------------ small head
class TestSmallHead(_EveryWorkload):
    NAME = SMALL

    def test_in_full(self, run):
        """2048 x 2048 x 32000: the full GPU run against the oracle's full
        run, every output element."""
        r = run
        ref = oracle.flce(r.X, r.W, r.t, IGN)
        assert r.n == ref["n_valid"]
        assert_loss(r.loss, ref["loss"])
        assert_loss(r.lse.cpu().numpy(), ref["lse"], "lse")
        assert_loss(r.rows_out.cpu().numpy(), ref["loss_rows"], "row losses")
        assert_grad(r.dX.float().cpu().numpy(), ref["dX"], "dX")
        assert_grad_blocks(r.dW, ref["dW"], "dW")


# ---------------------------------------------------------- Llama-3-8B head
def _dw_vocab_rows(r, k_random=13, k_targets=8):
    rng = np.random.default_rng(r.w.seed)
    tv = r.t[r.t != IGN].tolist()
    return sorted(set(tv[:k_targets]) | {0, r.w.V - 1, r.w.V // 2} |
                  set(rng.choice(r.w.V, k_random, replace=False).tolist()))


class TestLlama3Head(_EveryWorkload):
    NAME = LLAMA

    def test_full_run_dw_rows(self, run):
        """dW rows of the full 8192-token run (the first targets' rows, the
        vocabulary edges, random rows) against the oracle over all 8192
        tokens."""
        r = run
        vocab = _dw_vocab_rows(r)
        assert len(vocab) >= 16
        ref = oracle.flce_dw_rows(r.X, r.W, r.t, vocab, IGN)
        assert_grad(r.dW[vocab].cpu().numpy(), ref, "dW rows of the full run")
        for k, j in enumerate(vocab):  # and each row on its own
            got = r.dW[j].double().cpu().numpy()
            err = np.abs(got - ref[k]).max()
            assert err <= GRAD_MAX_REL * np.abs(ref[k]).max(), f"dW row {j}"
            cos = float(got @ ref[k] / (np.linalg.norm(got) * np.linalg.norm(ref[k])))
            assert cos >= GRAD_COS, f"dW row {j}: cosine {cos}"

    def test_prefix_64_in_full(self, run, cuda_lib):
        """The first 64 tokens as a problem of their own: loss, lse and dX in
        full, and 24 dW rows, against the oracle."""
        r = run
        Np = 64
        Xp, tp = r.X[:Np].contiguous(), r.t[:Np].contiguous()
        lse = torch.empty(Np, device=DEV)
        loss, nval, dX, dW = cuda_lib.flce_fwd_bwd_ex(Xp.to(DEV), r.Wd, tp.to(DEV), IGN,
                                                      sync=True, lse_out=lse)
        ref = oracle.flce_rows(Xp, r.W, tp, list(range(Np)), IGN)
        assert int(nval.item()) == ref["n_valid"]
        valid = (tp != IGN).numpy()
        assert_loss(loss.item(), ref["loss_rows"][valid].sum() / ref["n_valid"])
        assert_loss(lse.cpu().numpy(), ref["lse"], "lse")
        assert_grad(dX.float().cpu().numpy(), ref["dX"], "dX")
        rng = np.random.default_rng(r.w.seed)
        tv = tp[tp != IGN].tolist()
        vocab = sorted(set(tv[:8]) | {0, r.w.V - 1, r.w.V // 2} |
                       set(rng.choice(r.w.V, 13, replace=False).tolist()))
        ref_dw = oracle.flce_dw_rows(Xp, r.W, tp, vocab, IGN)
        assert_grad(dW[vocab].cpu().numpy(), ref_dw, "dW rows")

    def test_linearity_and_determinism(self, run, cuda_lib):
        """dW of the full batch equals the count-weighted dW of its two
        halves, and a second run of the full workload is bitwise identical."""
        r = run
        again = cuda_lib.flce_fwd_bwd_ex(r.Xd, r.Wd, r.td, IGN, sync=True)
        assert r.loss == again[0].item()
        assert torch.equal(r.dX, again[2]) and torch.equal(r.dW, again[3])
        del again
        h = r.w.N // 2
        a = cuda_lib.flce_fwd_bwd_ex(r.Xd[:h].contiguous(), r.Wd, r.td[:h].contiguous(), IGN,
                                     sync=True)
        b = cuda_lib.flce_fwd_bwd_ex(r.Xd[h:].contiguous(), r.Wd, r.td[h:].contiguous(), IGN,
                                     sync=True)
        na, nb = (int(v[1].item()) for v in (a, b))
        nf = r.n
        assert nf == na + nb
        comb = (na * a[3].double() + nb * b[3].double()) / nf
        assert_grad(r.dW.double().cpu().numpy(), comb.cpu().numpy(), "dW split")
        lc = (na * a[0].item() + nb * b[0].item()) / nf
        assert abs(r.loss - lc) <= 1e-5 * lc
        assert_grad(r.dX[:h].float().cpu().numpy(), (a[2].float() * na / nf).cpu().numpy(),
                    "dX first half")

    def test_loss_only_matches_full_call(self, run, cuda_lib):
        """flce_fwd runs the same pass 1 and combine as the full call: the
        loss, the count and the per-row lse agree bit for bit at full size."""
        r = run
        lse_b = torch.empty(r.w.N, device=DEV)
        loss, nval = cuda_lib.flce_fwd(r.Xd, r.Wd, r.td, IGN, sync=True, lse_out=lse_b)
        assert loss.item() == r.loss and int(nval.item()) == r.n
        assert torch.equal(r.lse, lse_b)

    def test_ce_on_materialised_logits_sampled_rows(self, run, cuda_lib):
        """Cross-entropy on the full 8192 x 128256 bf16 logits of the workload
        (S = X W^T by cuBLAS, input staging only): sampled rows of lse, row
        loss and dS against the oracle on those rows, the count against the
        closed form, and sum_j dS_ij = 0 on every row."""
        r = run
        w = r.w
        S = (r.Xd @ r.Wd.t()).contiguous()
        lse = torch.empty(w.N, device=DEV)
        rows_out = torch.empty(w.N, device=DEV)
        loss, nval, dS = cuda_lib.flce_ce_fwd_bwd(S, r.td, IGN, sync=True, lse_out=lse,
                                                  loss_rows_out=rows_out)
        n = int(nval.item())
        assert n == GOLDEN["ignored_counts"][r.name]
        rows = _sample_rows(r.t, seed=w.seed)
        ref = oracle.ce(S[rows].cpu(), r.t[rows], IGN)
        n_sub = ref["n_valid"]
        assert_loss(lse[rows].cpu().numpy(), ref["lse"], "lse rows")
        assert_loss(rows_out[rows].cpu().numpy(), ref["loss_rows"], "row losses")
        # the oracle normalises the subset by its own count
        assert_grad(dS[rows].float().cpu().numpy() * n / n_sub, ref["dS"], "dS rows")
        assert abs(loss.item() - rows_out.double().sum().item() / n) <= 1e-5 * loss.item()
        row_sums = dS.float().sum(dim=1).abs()
        # bf16 rounding of the target entry alone can leave 2^-9 / n per row
        assert (row_sums <= 1e-2 / n).all(), "a dS row does not sum to ~0"
        del S, dS


# ------------------------------------------- Qwen2-7B head, long-context head
class _Prefix1024(_EveryWorkload):
    """The configurations whose oracle check is a separate 1024-row run."""

    def test_prefix_1024_in_full(self, run, cuda_lib):
        """The first 1024 tokens as a problem of their own: the GPU call
        against the oracle's run on the same 1024 rows, every output
        element."""
        r = run
        P = 1024
        Xp, tp = r.Xd[:P].contiguous(), r.td[:P].contiguous()
        lse = torch.empty(P, device=DEV)
        rows_out = torch.empty(P, device=DEV)
        loss, nval, dX, dW = cuda_lib.flce_fwd_bwd_ex(Xp, r.Wd, tp, IGN, sync=True,
                                                      lse_out=lse, loss_rows_out=rows_out)
        ref = _prefix_oracle(r, P)
        assert int(nval.item()) == ref["n_valid"]
        assert_loss(loss.item(), ref["loss"])
        assert_loss(lse.cpu().numpy(), ref["lse"], "lse")
        assert_loss(rows_out.cpu().numpy(), ref["loss_rows"], "row losses")
        assert_grad(dX.float().cpu().numpy(), ref["dX"], "dX")
        del dX
        assert_grad_blocks(dW, ref["dW"], "dW")
        ref["dW"] = None  # 4+ GB of float64: not needed by the next test

    def test_full_run_rows_0_to_1023(self, run):
        """Rows 0-1023 of the full GPU run against the oracle's 1024-row run:
        lse and row losses do not depend on the other rows; dX rows do only
        through the normaliser, so the full run's rows times n_full / n_prefix
        must equal the prefix problem's dX."""
        r = run
        P = 1024
        ref = _prefix_oracle(r, P)
        assert_loss(r.lse[:P].cpu().numpy(), ref["lse"], "lse rows 0-1023")
        assert_loss(r.rows_out[:P].cpu().numpy(), ref["loss_rows"], "row losses 0-1023")
        scaled = r.dX[:P].double().cpu().numpy() * (r.n / ref["n_valid"])
        assert_grad(scaled, ref["dX"], "dX rows 0-1023 (rescaled)")


class TestQwen2Head(_Prefix1024):
    NAME = QWEN


class TestLongContextHead(_Prefix1024):
    NAME = LONG
