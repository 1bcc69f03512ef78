"""fp64 CPU oracle for the fused chunked linear + cross-entropy loss.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports, calls or links
this file; only the tests, the smoke check and the benchmark's CPU-baseline leg
do. It shares no code, table or helper with the CUDA path.

What it computes is the plain definition of linear projection + softmax
cross-entropy with the mean over non-ignored rows, because the pages claim the
fused method reaches exactly that result ("Unsloth Architecture: Manual Triton
Backpropagation, Fused Cross-Entropy, and 80% VRAM Cut", pillar 4 "Zero
Approximation Loss"). So the oracle materialises the logits (in row blocks,
to bound host memory; the blocking changes no arithmetic) and follows the steps
in the order the pages state them:

  1. Z = H W^T  -- the LM-head projection ("Arquitectura interna de Unsloth y
     optimizacion en Triton", section 3 "Fused Cross Entropy"; "Unsloth
     Architecture ...", section "The Un-Fused Cross-Entropy Logit Disaster").
  2. lse_i = m_i + log sum_j exp(Z_ij - m_i), m_i = max_j Z_ij -- subtract the
     row maximum, then log-sum-exp (same section 3 of the Spanish page).
  3. L_i = lse_i - Z_{i,y_i}; loss = sum over valid rows / N_valid
     ("Unsloth Architecture ...", pillar 1 "Fused Chunked Cross-Entropy Loss").
  4. dL/dZ_ij = (softmax(Z)_ij - 1[j = y_i]) * dloss / N_valid, zero rows for
     ignored samples (section 3 of the Spanish page; pillar 1).
  5. dH = G W and dW = G^T H -- backpropagation into both the hidden states and
     the vocabulary projection (section 3 of the Spanish page).

Readings where the pages are silent:
  * ignore_index rows (y == ignore_index) are dropped from the mean; the
    normaliser is N_valid (the pages divide by the token count, which is the
    same when nothing is ignored).
  * labels outside [0, V) that are not ignore_index are treated as ignored
    and reported through the returned ``n_bad``.
  * N_valid == 0 gives loss 0 and zero gradients.
  * the loss uses lse - z_y exactly, with no clamp of p.
  * dloss is a scalar upstream gradient multiplying G.
  * reduction variants (a library option the pages do not discuss): "mean"
    (the pages' normalised loss), "sum" (sum over valid rows, G scaled by dloss)
    and "none" (per-row losses, 0 for ignored rows; dloss is then a per-row
    vector and row i of G is scaled by dloss[i]).

The module also holds the final RMSNorm that produces H and its backward
(rmsnorm_forward / rmsnorm_backward / norm_forward_backward), the step before
the LM head in the same pages.

Pins: tests/test_oracle.py checks this module against closed forms (W = 0),
invariants (row sums of G, column sums of dW, shift invariance, ignored rows),
central finite differences, scipy's logsumexp and torch's cross_entropy in fp64.
"""
from __future__ import annotations

import numpy as np

IGNORE_INDEX = -100


def as_f64(a) -> np.ndarray:
    """Upcast a torch tensor (any float dtype, incl. bf16) or array to fp64 numpy."""
    if hasattr(a, "detach"):
        a = a.detach().to("cpu")
        if not a.is_floating_point():
            return a.numpy()
        import torch  # only for the dtype conversion of bf16 tensors
        return a.to(torch.float64).numpy()
    return np.asarray(a, dtype=np.float64)


def as_labels(y) -> np.ndarray:
    """Labels as an int64 numpy vector (accepts torch tensors, lists, arrays)."""
    if hasattr(y, "detach"):
        y = y.detach().to("cpu").numpy()
    return np.asarray(y).astype(np.int64)


def valid_rows(y: np.ndarray, V: int, ignore_index: int = IGNORE_INDEX):
    """Rows that take part in the loss, and the count of out-of-range labels."""
    y = as_labels(y)
    in_range = (y >= 0) & (y < V)
    bad = (~in_range) & (y != ignore_index)
    return in_range & (y != ignore_index), int(bad.sum())


def logits(H: np.ndarray, W: np.ndarray) -> np.ndarray:
    """Step 1: Z = H W^T in fp64."""
    return H @ W.T


def row_logsumexp(Z: np.ndarray) -> np.ndarray:
    """Step 2: per-row log-sum-exp with the row maximum subtracted first."""
    m = Z.max(axis=1)
    return m + np.log(np.exp(Z - m[:, None]).sum(axis=1))


def _block_iter(n: int, block: int):
    for s in range(0, n, block):
        yield s, min(s + block, n)


def _block_rows(V: int) -> int:
    # keep a block of fp64 logits near 256 MB
    return max(1, min(4096, (256 << 20) // (8 * max(V, 1))))


def forward(H, W, y, ignore_index: int = IGNORE_INDEX):
    """Loss and per-row lse (steps 1-3). Returns (loss, lse[N], n_valid, n_bad)."""
    H = as_f64(H)
    W = as_f64(W)
    y = as_labels(y)
    N, V = H.shape[0], W.shape[0]
    valid, n_bad = valid_rows(y, V, ignore_index)
    n_valid = int(valid.sum())
    lse = np.empty(N, dtype=np.float64)
    total = 0.0
    for s, e in _block_iter(N, _block_rows(V)):
        Z = logits(H[s:e], W)
        lse[s:e] = row_logsumexp(Z)
        v = valid[s:e]
        idx = np.nonzero(v)[0]
        total += float(np.sum(lse[s:e][idx] - Z[idx, y[s:e][idx]]))
    loss = total / n_valid if n_valid else 0.0
    return loss, lse, n_valid, n_bad


def forward_backward(H, W, y, ignore_index: int = IGNORE_INDEX, dloss=1.0,
                     reduction: str = "mean"):
    """Steps 1-5. Returns dict(loss, lse[N], dH[N,D], dW[V,D], n_valid, n_bad), fp64.

    reduction "mean": loss = sum / N_valid, G scaled by dloss / N_valid;
    "sum": loss = sum, G scaled by dloss; "none": loss is the per-row vector and
    dloss a per-row vector scaling the rows of G."""
    H = as_f64(H)
    W = as_f64(W)
    y = as_labels(y)
    N, D = H.shape
    V = W.shape[0]
    valid, n_bad = valid_rows(y, V, ignore_index)
    n_valid = int(valid.sum())
    if reduction == "mean":
        row_scale = np.full(N, (float(dloss) / n_valid) if n_valid else 0.0)
    elif reduction == "sum":
        row_scale = np.full(N, float(dloss))
    elif reduction == "none":
        row_scale = np.broadcast_to(np.asarray(dloss, dtype=np.float64), (N,)).copy()
    else:
        raise ValueError(f"unknown reduction {reduction!r}")
    lse = np.empty(N, dtype=np.float64)
    row_loss = np.zeros(N, dtype=np.float64)
    dH = np.zeros((N, D), dtype=np.float64)
    dW = np.zeros((V, D), dtype=np.float64)
    for s, e in _block_iter(N, _block_rows(V)):
        Z = logits(H[s:e], W)
        lse_b = row_logsumexp(Z)
        lse[s:e] = lse_b
        v = valid[s:e]
        idx = np.nonzero(v)[0]
        yb = y[s:e]
        row_loss[s:e][idx] = lse_b[idx] - Z[idx, yb[idx]]
        # step 4: G = (softmax - onehot) * scale, ignored rows zero
        G = np.exp(Z - lse_b[:, None])
        G[idx, yb[idx]] -= 1.0
        G *= row_scale[s:e, None]
        G[~v] = 0.0
        # step 5
        dH[s:e] = G @ W
        dW += G.T @ H[s:e]
    total = float(np.sum(row_loss))
    if reduction == "mean":
        loss = total / n_valid if n_valid else 0.0
    elif reduction == "sum":
        loss = total
    else:
        loss = row_loss
    return dict(loss=loss, lse=lse, dH=dH, dW=dW, n_valid=n_valid, n_bad=n_bad)


def ce_from_logits(Z, y, ignore_index: int = IGNORE_INDEX, dloss=1.0, reduction: str = "mean"):
    """Steps 2-4 on logits the caller already has (no projection): lse, the loss
    under `reduction`, and dZ = (softmax(Z) - onehot(y)) * scale. fp64."""
    Z = as_f64(Z)
    y = as_labels(y)
    N, V = Z.shape
    valid, n_bad = valid_rows(y, V, ignore_index)
    n_valid = int(valid.sum())
    lse = row_logsumexp(Z) if N else np.zeros(0)
    idx = np.nonzero(valid)[0]
    row_loss = np.zeros(N)
    row_loss[idx] = lse[idx] - Z[idx, y[idx]]
    if reduction == "mean":
        row_scale = np.full(N, (float(dloss) / n_valid) if n_valid else 0.0)
        loss = float(row_loss.sum()) / n_valid if n_valid else 0.0
    elif reduction == "sum":
        row_scale = np.full(N, float(dloss))
        loss = float(row_loss.sum())
    elif reduction == "none":
        row_scale = np.broadcast_to(np.asarray(dloss, dtype=np.float64), (N,)).copy()
        loss = row_loss
    else:
        raise ValueError(f"unknown reduction {reduction!r}")
    dZ = np.exp(Z - lse[:, None]) if N else np.zeros((0, V))
    dZ[idx, y[idx]] -= 1.0
    dZ *= row_scale[:, None]
    dZ[~valid] = 0.0
    return dict(loss=loss, lse=lse, dZ=dZ, n_valid=n_valid, n_bad=n_bad)


# ---------------------------------------------------------------------------
# The final RMSNorm that produces H ("Unsloth Architecture: Manual Triton
# Backpropagation, Fused Cross-Entropy, and 80% VRAM Cut", pillar 3 "Fused
# RMSNorm & SwiGLU Kernels": the normalisation x / sqrt(mean x^2 + eps) * gamma
# and its hand-derived gradient with respect to x).
# ---------------------------------------------------------------------------

def rmsnorm_forward(X, gamma, eps: float):
    """h = x * rstd * gamma per row, rstd = 1 / sqrt(mean_i x_i^2 + eps).
    Returns (H [N, D], rstd [N]) in fp64."""
    X = as_f64(X)
    g = as_f64(gamma)
    ms = np.mean(X * X, axis=1)
    rstd = 1.0 / np.sqrt(ms + eps)
    return X * rstd[:, None] * g[None, :], rstd


def rmsnorm_backward(X, gamma, eps: float, dH):
    """Gradient of RMSNorm for the upstream gradient dH. Returns (dX, dgamma), fp64.

    With r = rstd of the row and u = gamma * dH (elementwise):
        dx = r * u - x * r^3 * (sum_i u_i x_i) / d,      dgamma = sum_rows dH * x * r.
    Reading: the page writes the leading factor as gamma / RMS(x) and the inner
    sum as sum_i x_i dL/dy_i; that is this expression when every channel has the
    same gamma. For a general gamma the derivative needs gamma inside the sum,
    as here (pinned against autograd and finite differences)."""
    X = as_f64(X)
    g = as_f64(gamma)
    dH = as_f64(dH)
    d = X.shape[1]
    rstd = 1.0 / np.sqrt(np.mean(X * X, axis=1) + eps)
    u = dH * g[None, :]
    c = np.sum(u * X, axis=1)
    dX = rstd[:, None] * u - X * (rstd ** 3 * c / d)[:, None]
    dgamma = np.sum(dH * X * rstd[:, None], axis=0)
    return dX, dgamma


def round_bf16(a: np.ndarray) -> np.ndarray:
    """Round fp64 values to bf16 (nearest even) and back to fp64."""
    import torch  # the rounding only
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16).to(torch.float64).numpy()


def norm_forward_backward(X, gamma, eps: float, W, y, ignore_index: int = IGNORE_INDEX,
                          dloss=1.0, reduction: str = "mean", round_h: bool = True):
    """RMSNorm -> LM head + cross-entropy -> backward into X, gamma and W.

    H = RMSNorm(X); with round_h the normalised hidden state is rounded to bf16,
    the dtype it is stored in and multiplied by the projection (the rounding is
    passed through unchanged by the backward). Then steps 1-5 on H, and dX,
    dgamma from rmsnorm_backward with the fp64 dH.
    Returns dict(loss, lse, dX, dgamma, dW, rstd, H, n_valid, n_bad)."""
    H, rstd = rmsnorm_forward(X, gamma, eps)
    if round_h:
        H = round_bf16(H)
    r = forward_backward(H, W, y, ignore_index=ignore_index, dloss=dloss, reduction=reduction)
    dX, dgamma = rmsnorm_backward(X, gamma, eps, r["dH"])
    return dict(loss=r["loss"], lse=r["lse"], dX=dX, dgamma=dgamma, dW=r["dW"], rstd=rstd, H=H,
                n_valid=r["n_valid"], n_bad=r["n_bad"])


# ---------------------------------------------------------------------------
# Sampled outputs for workloads too large to materialise on the host in a test.
# Each one is the same definition restricted to the requested rows / columns.
# ---------------------------------------------------------------------------

def rows_lse_and_target(H, W, y, rows, ignore_index: int = IGNORE_INDEX):
    """lse_i and z_{i,y_i} (nan when row i is not valid) for the selected rows."""
    H = as_f64(H)
    W = as_f64(W)
    y = as_labels(y)
    rows = np.asarray(rows, dtype=np.int64)
    Z = logits(H[rows], W)
    lse = row_logsumexp(Z)
    valid, _ = valid_rows(y[rows], W.shape[0], ignore_index)
    zy = np.full(len(rows), np.nan)
    zy[valid] = Z[np.nonzero(valid)[0], y[rows][valid]]
    return lse, zy


def rows_dH(H, W, y, rows, n_valid: int, ignore_index: int = IGNORE_INDEX, dloss: float = 1.0):
    """dH for the selected rows: (softmax(Z_i) - onehot(y_i)) * dloss/N_valid times W."""
    H = as_f64(H)
    W = as_f64(W)
    y = as_labels(y)
    rows = np.asarray(rows, dtype=np.int64)
    Z = logits(H[rows], W)
    lse = row_logsumexp(Z)
    G = np.exp(Z - lse[:, None])
    valid, _ = valid_rows(y[rows], W.shape[0], ignore_index)
    idx = np.nonzero(valid)[0]
    G[idx, y[rows][idx]] -= 1.0
    G *= dloss / n_valid if n_valid else 0.0
    G[~valid] = 0.0
    return G @ W


def cols_dW(H, W, y, vrows, lse_all, n_valid: int, ignore_index: int = IGNORE_INDEX,
            dloss: float = 1.0):
    """dW rows for the selected vocabulary ids, given every row's lse.

    dW[v] = sum_i G[i, v] H[i], G[i, v] = (exp(z_iv - lse_i) - 1[y_i = v]) * dloss/N_valid.
    """
    H = as_f64(H)
    W = as_f64(W)
    y = as_labels(y)
    vrows = np.asarray(vrows, dtype=np.int64)
    lse_all = np.asarray(lse_all, dtype=np.float64)
    Zc = H @ W[vrows].T                      # [N, len(vrows)]
    G = np.exp(Zc - lse_all[:, None])
    valid, _ = valid_rows(y, W.shape[0], ignore_index)
    G -= (y[:, None] == vrows[None, :]) & valid[:, None]
    G *= dloss / n_valid if n_valid else 0.0
    G[~valid] = 0.0
    return G.T @ H
