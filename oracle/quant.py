"""Per-vector TurboQuant quantization of keys and values (oracle, fp64).

TEST INFRASTRUCTURE (see ``oracle/__init__``).

[BLOG] §1.2:
  stage 1 (PolarQuant): multiply by a random orthogonal matrix, then quantize every
  rotated coordinate independently with an MSE-optimal Lloyd-Max quantizer of (b-1) bits;
  stage 2 (QJL): r = x - DEQUANT_mse(Q_mse(x)); project r with a random Gaussian S;
  keep only sign(S r), and ||r||_2 as the scale used at reconstruction.
[3BITS] "Python + HuggingFace": quantize returns (indices, norms) per vector.

Keys get both stages with (b-1) bits in stage 1; values get stage 1 only, with b bits.

Readings (the pages leave these open):
* The stored norm is n = ||x||_2 and the quantizer sees yhat = Pi x / n.  A zero vector
  has n = 0 and takes yhat = 0 (so every code is L/2, the cell right of the middle
  boundary 0), r = 0, gamma = 0 and every sign bit 1.
* DEQUANT_mse(idx, n) = n Pi^T c[idx]; the residual is formed in the original frame,
  r = x - n Pi^T c[idx], with n in fp64.
* A sign bit is 1 when (S r)_i >= 0 (ties to 1).
* n and gamma = ||r||_2 are stored rounded to fp32.
* Inputs are bf16 values widened exactly to fp64 (the caller passes them widened).
"""
import numpy as np

from . import codebook as cbmod


def _norms_and_yhat(X, Pi):
    X = np.asarray(X, dtype=np.float64)
    n = np.sqrt(np.sum(X * X, axis=1))
    Y = X @ Pi.T                                   # rows: (Pi x)^T
    safe = np.where(n > 0, n, 1.0)
    yhat = np.where(n[:, None] > 0, Y / safe[:, None], 0.0)
    return n, yhat


def mse_stage(X, Pi, centroids, boundaries):
    """Stage 1 for every row x of X: (idx [N,d] int, n [N] fp64, yhat [N,d])."""
    n, yhat = _norms_and_yhat(X, Pi)
    idx = cbmod.encode(yhat, boundaries)
    return idx, n, yhat


def dequant_mse(idx, n, Pi, centroids):
    """n Pi^T c[idx] for every row (original frame)."""
    return np.asarray(n, dtype=np.float64)[:, None] * (np.asarray(centroids)[idx] @ Pi)


def qjl_stage(X, idx, n, Pi, S, centroids):
    """Stage 2 given stage-1 codes: (sigma [N,m] uint8, gamma [N] fp64, z = S r [N,m])."""
    X = np.asarray(X, dtype=np.float64)
    r = X - dequant_mse(idx, n, Pi, centroids)
    gamma = np.sqrt(np.sum(r * r, axis=1))
    z = r @ S.T
    sigma = (z >= 0).astype(np.uint8)
    return sigma, gamma, z


def quantize_keys(X, Pi, S, cb_k):
    """Keys: dict(idx, n (fp32), gamma (fp32), sigma, plus fp64 intermediates yhat, z)."""
    c, t = cb_k
    idx, n, yhat = mse_stage(X, Pi, c, t)
    sigma, gamma, z = qjl_stage(X, idx, n, Pi, S, c)
    return dict(idx=idx, n=n.astype(np.float32), gamma=gamma.astype(np.float32),
                sigma=sigma, yhat=yhat, z=z, n64=n, gamma64=gamma)


def quantize_keys_mse(X, Pi, cb_k):
    """Keys without the QJL stage ([3BITS] "Python + HuggingFace": the stage-1 quantizer
    returns indices and norms): dict(idx, n (fp32), sigma None, gamma None, plus yhat)."""
    c, t = cb_k
    idx, n, yhat = mse_stage(X, Pi, c, t)
    return dict(idx=idx, n=n.astype(np.float32), sigma=None, gamma=None, yhat=yhat, n64=n)


def quantize_values(X, Pi, cb_v):
    """Values: dict(idx, n (fp32), plus fp64 yhat)."""
    c, t = cb_v
    idx, n, yhat = mse_stage(X, Pi, c, t)
    return dict(idx=idx, n=n.astype(np.float32), yhat=yhat, n64=n)


QJL_CONST = np.sqrt(np.pi / 2.0)


def reconstruct_keys(idx, n, sigma, gamma, Pi, S, centroids):
    """khat = n Pi^T c[idx] + gamma * sqrt(pi/2)/m * S^T (2 sigma - 1)   (original frame).

    The constant: for s ~ N(0, I), E[<s,q> sign<s,r>] = sqrt(2/pi) <q,r>/||r||, so the
    factor sqrt(pi/2) makes the QJL term an unbiased estimate of <q, r>."""
    m = S.shape[0]
    signs = 2.0 * np.asarray(sigma, dtype=np.float64) - 1.0
    g = np.asarray(gamma, dtype=np.float64)
    return dequant_mse(idx, n, Pi, centroids) + (g * QJL_CONST / m)[:, None] * (signs @ S)


def reconstruct_keys_any(tok_k, Pi, S, centroids):
    """khat for keys with the QJL stage (sigma present) or without it (sigma None: stage 1
    only, khat = n Pi^T c[idx])."""
    if tok_k.get("sigma") is None:
        return dequant_mse(tok_k["idx"], tok_k["n"], Pi, centroids)
    return reconstruct_keys(tok_k["idx"], tok_k["n"], tok_k["sigma"], tok_k["gamma"], Pi, S, centroids)


def reconstruct_values(idx, n, Pi, centroids):
    return dequant_mse(idx, n, Pi, centroids)
