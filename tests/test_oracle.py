"""Pins for the fp64 oracle: closed forms, invariants, finite differences,
library routines and brute force. None of these retypes the oracle's formulas;
each checks it against something that the mathematics fixes independently.

A mutation test at the end plants plausible mistakes in a copy of the oracle
(on the CPU) and checks that at least one pin catches each of them.
"""
import math
import types

import numpy as np
import pytest
import torch

from oracle import lce_oracle as O

IGN = -100


def _rand(N, D, V, seed, n_ign=0, w_std=0.3):
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((N, D))
    W = rng.standard_normal((V, D)) * w_std
    y = rng.integers(0, V, size=N)
    if n_ign:
        y[rng.permutation(N)[:n_ign]] = IGN
    return H, W, y


# ---------------------------------------------------------------- closed forms

def check_w_zero(orc):
    """W = 0: every logit is 0, so lse = log V, loss = log V, dH = 0 and
    dW[v] = sum_{valid i} (1/V - 1[y_i = v]) H_i / N_valid (uniform softmax)."""
    N, D, V = 12, 6, 10
    rng = np.random.default_rng(1)
    H = rng.standard_normal((N, D))
    W = np.zeros((V, D))
    y = rng.integers(0, V, size=N)
    y[[2, 7]] = IGN
    r = orc.forward_backward(H, W, y)
    assert r["n_valid"] == 10
    assert abs(r["loss"] - math.log(V)) < 1e-12
    assert np.allclose(r["lse"], math.log(V), atol=1e-12)
    assert np.abs(r["dH"]).max() == 0.0
    # expected dW by explicit loops
    exp = np.zeros((V, D))
    for i in range(N):
        if y[i] == IGN:
            continue
        for v in range(V):
            coef = 1.0 / V - (1.0 if v == y[i] else 0.0)
            exp[v] += coef * H[i] / 10
    assert np.allclose(r["dW"], exp, atol=1e-13)


def test_w_zero_closed_form():
    check_w_zero(O)


def test_two_class_logistic_closed_form():
    """V = 2 reduces to logistic regression: loss = log(1 + exp(-(z_y - z_other)))."""
    rng = np.random.default_rng(3)
    N, D = 9, 4
    H = rng.standard_normal((N, D))
    W = rng.standard_normal((2, D))
    y = rng.integers(0, 2, size=N)
    r = O.forward_backward(H, W, y)
    z = H @ W.T
    margin = z[np.arange(N), y] - z[np.arange(N), 1 - y]
    assert abs(r["loss"] - np.mean(np.log1p(np.exp(-margin)))) < 1e-12
    # dL/dz_y = -sigmoid(-margin)/N
    sig = 1.0 / (1.0 + np.exp(margin))
    g_y = -sig / N
    dH_exp = g_y[:, None] * (W[y] - W[1 - y])
    assert np.allclose(r["dH"], dH_exp, atol=1e-13)


def test_identical_rows_give_uniform_softmax():
    """If every vocabulary row of W is the same vector, Z is constant along V."""
    rng = np.random.default_rng(4)
    N, D, V = 7, 5, 13
    H = rng.standard_normal((N, D))
    w = rng.standard_normal(D)
    W = np.tile(w, (V, 1))
    y = rng.integers(0, V, size=N)
    loss, lse, nv, _ = O.forward(H, W, y)
    assert abs(loss - math.log(V)) < 1e-12
    assert np.allclose(lse, H @ w + math.log(V), atol=1e-12)


# ------------------------------------------------------------------ invariants

def check_invariants(orc, seed=5):
    H, W, y = _rand(20, 7, 11, seed, n_ign=3)
    r = orc.forward_backward(H, W, y, dloss=1.7)
    # rows of softmax - onehot sum to 0  =>  sum over v of dW[v, :] is 0
    assert np.abs(r["dW"].sum(axis=0)).max() < 1e-13
    # ignored rows: zero dH
    ign = y == IGN
    assert np.abs(r["dH"][ign]).max() == 0.0
    # perturbing ignored rows' H changes neither the loss nor dW
    H2 = H.copy()
    H2[ign] += 5.0
    r2 = orc.forward_backward(H2, W, y, dloss=1.7)
    assert abs(r2["loss"] - r["loss"]) < 1e-13
    assert np.allclose(r2["dW"], r["dW"], atol=1e-13)
    # loss equals the mean over the valid subset
    rs = orc.forward_backward(H[~ign], W, y[~ign], dloss=1.7)
    assert abs(rs["loss"] - r["loss"]) < 1e-13
    assert np.allclose(rs["dW"], r["dW"], atol=1e-13)
    assert np.allclose(rs["dH"], r["dH"][~ign], atol=1e-13)
    # shift invariance: adding the same u to every vocabulary row of W
    u = np.random.default_rng(seed + 1).standard_normal(W.shape[1])
    r3 = orc.forward_backward(H, W + u[None, :], y, dloss=1.7)
    assert abs(r3["loss"] - r["loss"]) < 1e-12
    assert np.allclose(r3["dH"], r["dH"], atol=1e-12)
    assert np.allclose(r3["dW"], r["dW"], atol=1e-12)
    # permuting the rows permutes lse and dH and leaves loss and dW
    p = np.random.default_rng(seed + 2).permutation(len(y))
    r4 = orc.forward_backward(H[p], W, y[p], dloss=1.7)
    assert abs(r4["loss"] - r["loss"]) < 1e-13
    assert np.allclose(r4["lse"], r["lse"][p], atol=1e-13)
    assert np.allclose(r4["dH"], r["dH"][p], atol=1e-13)
    assert np.allclose(r4["dW"], r["dW"], atol=1e-13)
    # dloss is linear
    r5 = orc.forward_backward(H, W, y, dloss=1.0)
    assert np.allclose(r5["dH"] * 1.7, r["dH"], atol=1e-14)


def test_invariants():
    check_invariants(O)


def test_all_rows_ignored():
    H, W, y = _rand(5, 4, 6, 8)
    y[:] = IGN
    r = O.forward_backward(H, W, y)
    assert r["loss"] == 0.0 and r["n_valid"] == 0
    assert not np.any(r["dH"]) and not np.any(r["dW"])
    assert np.all(np.isfinite(r["lse"]))


def test_out_of_range_labels_are_counted_and_dropped():
    H, W, y = _rand(8, 4, 6, 9)
    y2 = y.copy()
    y2[1] = 6          # == V, out of range
    y2[4] = -3         # negative, not ignore_index
    r = O.forward_backward(H, W, y2)
    assert r["n_bad"] == 2 and r["n_valid"] == 6
    y3 = y.copy()
    y3[[1, 4]] = IGN
    r3 = O.forward_backward(H, W, y3)
    assert abs(r["loss"] - r3["loss"]) < 1e-14
    assert np.allclose(r["dW"], r3["dW"])


# ------------------------------------------------------- finite differences

def check_fd(orc):
    """Central finite differences of dloss * loss at N=4, D=8, V=16 with an
    ignored row and dloss != 1 agree with dH and dW to 1e-6."""
    N, D, V = 4, 8, 16
    H, W, y = _rand(N, D, V, 11, w_std=0.5)
    y[2] = IGN
    dloss = 0.7
    r = orc.forward_backward(H, W, y, dloss=dloss)

    def f(Hx, Wx):
        return dloss * orc.forward(Hx, Wx, y)[0]

    eps = 1e-5
    for (A, G) in ((H, r["dH"]), (W, r["dW"])):
        num = np.zeros_like(A)
        for idx in np.ndindex(A.shape):
            Ap = A.copy(); Ap[idx] += eps
            Am = A.copy(); Am[idx] -= eps
            if A is H:
                num[idx] = (f(Ap, W) - f(Am, W)) / (2 * eps)
            else:
                num[idx] = (f(H, Ap) - f(H, Am)) / (2 * eps)
        assert np.abs(num - G).max() <= 1e-6
    # lse against a finite difference identity: d lse_i / d z_ij = softmax_ij,
    # so d lse_i / d H_i = softmax_i W
    Z = H @ W.T
    P = np.exp(Z - Z.max(1, keepdims=True)); P /= P.sum(1, keepdims=True)
    for i in range(N):
        g = np.zeros(D)
        for d in range(D):
            Hp = H.copy(); Hp[i, d] += eps
            Hm = H.copy(); Hm[i, d] -= eps
            g[d] = (orc.forward(Hp, W, y)[1][i] - orc.forward(Hm, W, y)[1][i]) / (2 * eps)
        assert np.abs(g - P[i] @ W).max() <= 1e-6


def test_finite_differences():
    check_fd(O)


# ------------------------------------------------------- library routines

def check_torch(orc, seed=13):
    """torch.nn.functional.cross_entropy(ignore_index=-100, mean) + autograd, fp64."""
    H, W, y = _rand(33, 9, 21, seed, n_ign=4)
    Ht = torch.tensor(H, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    loss = torch.nn.functional.cross_entropy(Ht @ Wt.T, torch.tensor(y), ignore_index=IGN)
    (loss * 2.5).backward()
    r = orc.forward_backward(H, W, y, dloss=2.5)
    assert abs(r["loss"] - loss.item()) < 1e-12
    assert np.allclose(r["dH"], Ht.grad.numpy(), atol=1e-13)
    assert np.allclose(r["dW"], Wt.grad.numpy(), atol=1e-13)
    lse_t = torch.logsumexp(torch.tensor(H) @ torch.tensor(W).T, dim=1).numpy()
    assert np.allclose(r["lse"], lse_t, atol=1e-12)


def test_vs_torch_cross_entropy():
    check_torch(O)


def test_lse_vs_scipy_logsumexp_large_logits():
    from scipy.special import logsumexp
    rng = np.random.default_rng(2)
    Z = rng.standard_normal((6, 50)) * 300.0     # exp would overflow without the max shift
    assert np.allclose(O.row_logsumexp(Z), logsumexp(Z, axis=1), rtol=0, atol=1e-10)


def test_brute_force_python_loops():
    """Pure-Python loops with math.exp/math.log on a 3x2x4 case."""
    H = [[0.5, -1.0], [2.0, 0.25], [-0.75, 1.5]]
    W = [[0.1, 0.2], [-0.3, 0.4], [0.5, -0.6], [0.0, 0.7]]
    y = [2, IGN, 0]
    N, D, V = 3, 2, 4
    z = [[sum(H[i][d] * W[v][d] for d in range(D)) for v in range(V)] for i in range(N)]
    lse = [math.log(sum(math.exp(z[i][v]) for v in range(V))) for i in range(N)]
    nv = 2
    loss = sum(lse[i] - z[i][y[i]] for i in range(N) if y[i] != IGN) / nv
    g = [[(math.exp(z[i][v] - lse[i]) - (1.0 if v == y[i] else 0.0)) / nv if y[i] != IGN else 0.0
          for v in range(V)] for i in range(N)]
    dH = [[sum(g[i][v] * W[v][d] for v in range(V)) for d in range(D)] for i in range(N)]
    dW = [[sum(g[i][v] * H[i][d] for i in range(N)) for d in range(D)] for v in range(V)]
    r = O.forward_backward(np.array(H), np.array(W), np.array(y))
    assert abs(r["loss"] - loss) < 1e-14
    assert np.allclose(r["lse"], lse, atol=1e-14)
    assert np.allclose(r["dH"], dH, atol=1e-15)
    assert np.allclose(r["dW"], dW, atol=1e-15)


def test_expected_loss_at_init_tiny_workload():
    """For H ~ N(0,1), W ~ N(0, s^2) the logits of a row are ~N(0, |h|^2 s^2); then
    E[lse] ~= log V + D s^2 / 2 and E[z_y] = 0, so the mean loss is near
    log 32000 + 512 * 0.02^2 / 2 = 10.4757 (tiny workload, 256 rows)."""
    from lce_synth import workload_inputs
    H, W, y = workload_inputs("tiny")
    loss, lse, nv, nb = O.forward(H, W, y)
    assert nv == 256 and nb == 0
    assert abs(loss - (math.log(32000) + 512 * 0.02 ** 2 / 2)) < 0.05


# ------------------------------------------------------- reduction variants

def test_reductions_vs_torch():
    """torch cross_entropy with reduction sum / none (+ autograd, fp64), and a
    per-row upstream gradient for 'none'."""
    H, W, y = _rand(25, 7, 19, 31, n_ign=3)
    rng = np.random.default_rng(32)
    g_rows = rng.standard_normal(25)
    for red, dl in (("sum", 0.6), ("none", g_rows)):
        Ht = torch.tensor(H, requires_grad=True)
        Wt = torch.tensor(W, requires_grad=True)
        out = torch.nn.functional.cross_entropy(Ht @ Wt.T, torch.tensor(y), ignore_index=IGN,
                                                reduction=red)
        (out * torch.as_tensor(dl)).sum().backward()
        r = O.forward_backward(H, W, y, dloss=dl, reduction=red)
        assert np.allclose(r["loss"], out.detach().numpy(), atol=1e-12)
        assert np.allclose(r["dH"], Ht.grad.numpy(), atol=1e-13)
        assert np.allclose(r["dW"], Wt.grad.numpy(), atol=1e-13)


def test_reduction_relations_and_fd():
    """sum = mean * N_valid; the per-row losses sum to it and are 0 on ignored
    rows; a per-row dloss equal everywhere matches 'sum'; finite differences of
    sum_i dloss_i L_i give the 'none' gradients."""
    H, W, y = _rand(6, 5, 9, 33, n_ign=2, w_std=0.5)
    m = O.forward_backward(H, W, y, reduction="mean")
    s_ = O.forward_backward(H, W, y, reduction="sum", dloss=2.0)
    n = O.forward_backward(H, W, y, reduction="none", dloss=np.full(6, 2.0))
    assert abs(s_["loss"] - m["loss"] * m["n_valid"]) < 1e-12
    assert abs(np.sum(n["loss"]) - s_["loss"]) < 1e-12
    assert np.all(n["loss"][y == IGN] == 0.0)
    assert np.allclose(n["dH"], s_["dH"], atol=1e-15) and np.allclose(n["dW"], s_["dW"], atol=1e-15)
    g = np.random.default_rng(34).standard_normal(6)
    r = O.forward_backward(H, W, y, reduction="none", dloss=g)
    f = lambda Hx: float(np.dot(g, O.forward_backward(Hx, W, y, reduction="none")["loss"]))
    eps = 1e-5
    num = np.zeros_like(H)
    for idx in np.ndindex(H.shape):
        Hp = H.copy(); Hp[idx] += eps
        Hm = H.copy(); Hm[idx] -= eps
        num[idx] = (f(Hp) - f(Hm)) / (2 * eps)
    assert np.abs(num - r["dH"]).max() <= 1e-6


# ------------------------------------------------------- CE over given logits

@pytest.mark.parametrize("reduction", ["mean", "sum", "none"])
def test_ce_from_logits_vs_torch(reduction):
    rng = np.random.default_rng(41)
    N, V = 19, 37
    Z = rng.standard_normal((N, V)) * 4.0
    y = rng.integers(0, V, size=N)
    y[[3, 11]] = IGN
    dl = rng.standard_normal(N) if reduction == "none" else 1.3
    Zt = torch.tensor(Z, requires_grad=True)
    out = torch.nn.functional.cross_entropy(Zt, torch.tensor(y), ignore_index=IGN,
                                            reduction=reduction)
    (out * torch.as_tensor(dl)).sum().backward()
    r = O.ce_from_logits(Z, y, dloss=dl, reduction=reduction)
    assert np.allclose(r["loss"], out.detach().numpy(), atol=1e-12)
    assert np.allclose(r["dZ"], Zt.grad.numpy(), atol=1e-14)
    assert np.allclose(r["lse"], torch.logsumexp(torch.tensor(Z), 1).numpy(), atol=1e-12)


def check_ce_torch(orc, reduction="mean"):
    """ce_from_logits against torch cross_entropy(ignore_index=-100) + autograd, fp64."""
    rng = np.random.default_rng(41)
    N, V = 19, 37
    Z = rng.standard_normal((N, V)) * 4.0
    y = rng.integers(0, V, size=N)
    y[[3, 11]] = IGN
    dl = rng.standard_normal(N) if reduction == "none" else 1.3
    Zt = torch.tensor(Z, requires_grad=True)
    out = torch.nn.functional.cross_entropy(Zt, torch.tensor(y), ignore_index=IGN,
                                            reduction=reduction)
    (out * torch.as_tensor(dl)).sum().backward()
    r = orc.ce_from_logits(Z, y, dloss=dl, reduction=reduction)
    assert np.allclose(r["loss"], out.detach().numpy(), atol=1e-12)
    assert np.allclose(r["dZ"], Zt.grad.numpy(), atol=1e-14)
    assert np.allclose(r["lse"], torch.logsumexp(torch.tensor(Z), 1).numpy(), atol=1e-12)


def check_ce_matches_projection_path(orc):
    """With Z = H W^T, the CE over logits gives the fused path's loss and lse, and
    dZ W / dZ^T H are its dH / dW (the chain rule through the projection)."""
    H, W, y = _rand(23, 7, 29, 5, n_ign=3)
    r = orc.forward_backward(H, W, y, dloss=0.6)
    c = orc.ce_from_logits(H @ W.T, y, dloss=0.6)
    assert abs(c["loss"] - r["loss"]) < 1e-12
    assert np.allclose(c["lse"], r["lse"], atol=1e-12)
    assert np.allclose(c["dZ"] @ W, r["dH"], atol=1e-13)
    assert np.allclose(c["dZ"].T @ H, r["dW"], atol=1e-13)


def test_ce_from_logits_matches_projection_path():
    check_ce_matches_projection_path(O)


CE_MUTATIONS = {
    "CE dropped onehot": ("dZ[idx, y[idx]] -= 1.0", "pass"),
    "CE loss sign": ("row_loss[idx] = lse[idx] - Z[idx, y[idx]]", "row_loss[idx] = Z[idx, y[idx]] - lse[idx]"),
    "CE ignored rows not zeroed": ("dZ[~valid] = 0.0", "pass"),
    "CE softmax without lse": ("dZ = np.exp(Z - lse[:, None]) if N else np.zeros((0, V))",
                               "dZ = np.exp(Z) if N else np.zeros((0, V))"),
    "CE sum scaled as mean": ("row_scale = np.full(N, float(dloss))\n",
                              "row_scale = np.full(N, float(dloss) / max(n_valid, 1))\n"),
}


@pytest.mark.parametrize("name", sorted(CE_MUTATIONS))
def test_ce_pins_catch_planted_mistakes(name):
    old, new = CE_MUTATIONS[name]
    m = _mutant(old, new)
    caught = 0
    for pin in (lambda o: check_ce_torch(o, "mean"), lambda o: check_ce_torch(o, "sum"),
                lambda o: check_ce_torch(o, "none"), check_ce_matches_projection_path):
        try:
            with np.errstate(all="ignore"):
                pin(m)
        except Exception:
            caught += 1
    assert caught >= 1, f"no pin caught mutation {name!r}"


def test_ce_from_logits_rows_sum_to_zero_and_large_logits():
    """Rows of dZ sum to 0 for valid rows; logits near +-1000 stay finite."""
    rng = np.random.default_rng(42)
    Z = rng.standard_normal((8, 50)) * 400.0
    y = rng.integers(0, 50, size=8)
    r = O.ce_from_logits(Z, y, reduction="sum")
    assert np.all(np.isfinite(r["dZ"])) and np.all(np.isfinite(r["lse"]))
    assert np.abs(r["dZ"].sum(axis=1)).max() < 1e-12


# ------------------------------------------------------- final RMSNorm

def _norm_case(seed, N=7, D=12, eps=1e-5):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((N, D)) * np.exp(rng.standard_normal((N, 1)) * 0.7)
    gamma = 1.0 + 0.3 * rng.standard_normal(D)
    dH = rng.standard_normal((N, D))
    return X, gamma, dH, eps


def check_rmsnorm_torch(orc, seed=51):
    """Forward and backward against torch.nn.functional.rms_norm + autograd, fp64."""
    X, gamma, dH, eps = _norm_case(seed)
    Xt = torch.tensor(X, requires_grad=True)
    gt = torch.tensor(gamma, requires_grad=True)
    Ht = torch.nn.functional.rms_norm(Xt, (X.shape[1],), gt, eps=eps)
    (Ht * torch.tensor(dH)).sum().backward()
    H, rstd = orc.rmsnorm_forward(X, gamma, eps)
    dX, dgamma = orc.rmsnorm_backward(X, gamma, eps, dH)
    assert np.allclose(H, Ht.detach().numpy(), atol=1e-13)
    assert np.allclose(dX, Xt.grad.numpy(), atol=1e-12)
    assert np.allclose(dgamma, gt.grad.numpy(), atol=1e-12)
    assert np.allclose(rstd, 1.0 / np.sqrt((X ** 2).mean(axis=1) + eps), atol=1e-14)


def check_rmsnorm_fd(orc, seed=52):
    """Central finite differences of L = sum(dH * RMSNorm(X)) in X and gamma."""
    X, gamma, dH, eps = _norm_case(seed, N=3, D=5)
    f = lambda X_, g_: float(np.sum(dH * orc.rmsnorm_forward(X_, g_, eps)[0]))
    dX, dgamma = orc.rmsnorm_backward(X, gamma, eps, dH)
    h = 1e-6
    for idx in np.ndindex(X.shape):
        Xp = X.copy(); Xp[idx] += h
        Xm = X.copy(); Xm[idx] -= h
        assert abs((f(Xp, gamma) - f(Xm, gamma)) / (2 * h) - dX[idx]) < 1e-7
    for j in range(gamma.size):
        gp = gamma.copy(); gp[j] += h
        gm = gamma.copy(); gm[j] -= h
        assert abs((f(X, gp) - f(X, gm)) / (2 * h) - dgamma[j]) < 1e-7


def test_rmsnorm_vs_torch():
    check_rmsnorm_torch(O)


def test_rmsnorm_finite_differences():
    check_rmsnorm_fd(O)


def test_rmsnorm_page_closed_form_with_uniform_gamma():
    """With the same gamma on every channel the page's closed form (gamma / RMS
    outside, sum_i x_i dL/dy_i inside) is exact; the oracle agrees with it there."""
    X, _, dH, eps = _norm_case(53)
    gamma = np.full(X.shape[1], 1.7)
    dX, _ = O.rmsnorm_backward(X, gamma, eps, dH)
    d = X.shape[1]
    rms = np.sqrt((X ** 2).mean(axis=1) + eps)[:, None]
    page = gamma / rms * (dH - X * np.sum(X * dH, axis=1, keepdims=True) / (d * rms ** 2))
    assert np.allclose(dX, page, atol=1e-12)


def test_rmsnorm_scale_invariance_without_eps():
    """eps = 0: RMSNorm(c x) = RMSNorm(x), so dX is orthogonal to x in every row."""
    X, gamma, dH, _ = _norm_case(54)
    H1, _ = O.rmsnorm_forward(X, gamma, 0.0)
    H2, _ = O.rmsnorm_forward(3.5 * X, gamma, 0.0)
    assert np.allclose(H1, H2, atol=1e-13)
    dX, _ = O.rmsnorm_backward(X, gamma, 0.0, dH)
    assert np.abs(np.sum(dX * X, axis=1)).max() < 1e-12


def check_norm_composition_torch(orc, seed=55):
    """RMSNorm -> X W^T -> cross_entropy(ignore_index) in fp64 autograd against
    norm_forward_backward without the bf16 rounding of H."""
    rng = np.random.default_rng(seed)
    N, D, V = 21, 10, 17
    X = rng.standard_normal((N, D)) * 2.0
    gamma = 1.0 + 0.2 * rng.standard_normal(D)
    W = rng.standard_normal((V, D)) * 0.5
    y = rng.integers(0, V, size=N)
    y[[2, 9]] = IGN
    Xt = torch.tensor(X, requires_grad=True)
    gt = torch.tensor(gamma, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    H = torch.nn.functional.rms_norm(Xt, (D,), gt, eps=1e-6)
    loss = torch.nn.functional.cross_entropy(H @ Wt.T, torch.tensor(y), ignore_index=IGN)
    (loss * 0.8).backward()
    r = orc.norm_forward_backward(X, gamma, 1e-6, W, y, dloss=0.8, round_h=False)
    assert abs(r["loss"] - loss.item()) < 1e-12
    assert np.allclose(r["dX"], Xt.grad.numpy(), atol=1e-13)
    assert np.allclose(r["dgamma"], gt.grad.numpy(), atol=1e-13)
    assert np.allclose(r["dW"], Wt.grad.numpy(), atol=1e-13)


def test_norm_composition_vs_torch():
    check_norm_composition_torch(O)


def test_norm_round_h_is_bf16_of_exact_h():
    rng = np.random.default_rng(56)
    X = rng.standard_normal((6, 16))
    gamma = 1.0 + 0.1 * rng.standard_normal(16)
    W = rng.standard_normal((9, 16)) * 0.1
    y = rng.integers(0, 9, size=6)
    r = O.norm_forward_backward(X, gamma, 1e-5, W, y)
    H, _ = O.rmsnorm_forward(X, gamma, 1e-5)
    expect = torch.tensor(H).to(torch.bfloat16).double().numpy()
    assert np.array_equal(r["H"], expect)
    assert np.abs(r["H"] - H).max() <= 2.0 ** -8 * np.abs(H).max()


NORM_MUTATIONS = {
    "gamma outside the sum (page literal)": (
        "    u = dH * g[None, :]\n    c = np.sum(u * X, axis=1)\n    dX = rstd[:, None] * u - X * (rstd ** 3 * c / d)[:, None]",
        "    u = dH * g[None, :]\n    c = np.sum(dH * X, axis=1)\n    dX = rstd[:, None] * u - X * g[None, :] * (rstd ** 3 * c / d)[:, None]"),
    "r instead of r^3": ("dX = rstd[:, None] * u - X * (rstd ** 3 * c / d)[:, None]",
                         "dX = rstd[:, None] * u - X * (rstd * c / d)[:, None]"),
    "dgamma without rstd": ("dgamma = np.sum(dH * X * rstd[:, None], axis=0)", "dgamma = np.sum(dH * X, axis=0)"),
    "sum instead of mean of squares": ("    ms = np.mean(X * X, axis=1)\n", "    ms = np.sum(X * X, axis=1)\n"),
    "eps outside the sqrt": ("    rstd = 1.0 / np.sqrt(ms + eps)\n", "    rstd = 1.0 / (np.sqrt(ms) + eps)\n"),
    "backward drops the cross term": ("dX = rstd[:, None] * u - X * (rstd ** 3 * c / d)[:, None]",
                                      "dX = rstd[:, None] * u"),
}


@pytest.mark.parametrize("name", sorted(NORM_MUTATIONS))
def test_norm_pins_catch_planted_mistakes(name):
    old, new = NORM_MUTATIONS[name]
    m = _mutant(old, new)
    caught = 0
    for pin in (check_rmsnorm_torch, check_rmsnorm_fd, check_norm_composition_torch):
        try:
            with np.errstate(all="ignore"):
                pin(m)
        except Exception:
            caught += 1
    assert caught >= 1, f"no pin caught mutation {name!r}"


# ------------------------------------------------------- sampled helpers

def test_sampled_helpers_match_full():
    H, W, y = _rand(40, 6, 30, 17, n_ign=5)
    r = O.forward_backward(H, W, y, dloss=0.9)
    rows = np.array([0, 3, 7, 11, 39])
    lse, zy = O.rows_lse_and_target(H, W, y, rows)
    assert np.allclose(lse, r["lse"][rows], atol=1e-14)
    valid = y[rows] != IGN
    Z = H @ W.T
    assert np.allclose(zy[valid], Z[rows[valid], y[rows[valid]]], atol=1e-14)
    assert np.all(np.isnan(zy[~valid]))
    dH = O.rows_dH(H, W, y, rows, r["n_valid"], dloss=0.9)
    assert np.allclose(dH, r["dH"][rows], atol=1e-15)
    vrows = np.array([0, 5, 29])
    dW = O.cols_dW(H, W, y, vrows, r["lse"], r["n_valid"], dloss=0.9)
    assert np.allclose(dW, r["dW"][vrows], atol=1e-15)


def test_blocking_does_not_change_results(monkeypatch):
    H, W, y = _rand(37, 5, 19, 21, n_ign=2)
    r1 = O.forward_backward(H, W, y)
    monkeypatch.setattr(O, "_block_rows", lambda V: 4)
    r2 = O.forward_backward(H, W, y)
    assert abs(r1["loss"] - r2["loss"]) < 1e-13
    for k in ("lse", "dH", "dW"):
        assert np.allclose(r1[k], r2[k], atol=1e-14)


# ------------------------------------------------------- mutation check

MUTATIONS = {
    "dropped onehot term": ("G[idx, yb[idx]] -= 1.0", "pass"),
    "wrong onehot sign": ("G[idx, yb[idx]] -= 1.0", "G[idx, yb[idx]] += 1.0"),
    "divide by N not N_valid": ("row_scale = np.full(N, (float(dloss) / n_valid) if n_valid else 0.0)",
                                "row_scale = np.full(N, float(dloss) / N)"),
    "ignored rows not zeroed": ("G[~v] = 0.0", "pass"),
    "dW transposed operand": ("dW += G.T @ H[s:e]", "dW += (H[s:e].T @ G).T[::-1]"),
    "lse without log": ("return m + np.log(np.exp(Z - m[:, None]).sum(axis=1))",
                        "return m + np.exp(Z - m[:, None]).sum(axis=1)"),
    "max not added back": ("return m + np.log(np.exp(Z - m[:, None]).sum(axis=1))",
                           "return np.log(np.exp(Z - m[:, None]).sum(axis=1))"),
    "loss sign": ("row_loss[s:e][idx] = lse_b[idx] - Z[idx, yb[idx]]",
                  "row_loss[s:e][idx] = Z[idx, yb[idx]] - lse_b[idx]"),
    "dH uses W transposed wrong": ("dH[s:e] = G @ W", "dH[s:e] = G @ W[::-1]"),
}


def _mutant(old, new):
    import inspect
    src = inspect.getsource(O)
    assert old in src, old
    m = types.ModuleType("mutant")
    exec(compile(src.replace(old, new), "mutant", "exec"), m.__dict__)
    return m


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistakes(name):
    old, new = MUTATIONS[name]
    m = _mutant(old, new)
    pins = (check_w_zero, check_invariants, check_fd, check_torch)
    caught = 0
    for pin in pins:
        try:
            with np.errstate(all="ignore"):
                pin(m)
        except Exception:
            caught += 1
    assert caught >= 1, f"no pin caught mutation {name!r}"
