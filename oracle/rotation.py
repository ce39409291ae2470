"""The method's seeded random matrices (oracle side).

TEST INFRASTRUCTURE (see ``oracle/__init__``).

[BLOG] §1.2, stage 1: every KV vector is multiplied by a random orthogonal matrix, which
spreads information evenly over the coordinates.  Stage 2: the residual is projected by a
random Gaussian matrix S.  [3BITS] "Как работает TurboQuant" (idea one) says the same of
the rotation.

Readings:
* "Random orthogonal" is taken as Haar-distributed: Pi = Q diag(sign R_ii) where G = Q R
  is the QR factorisation of a d x d matrix G of i.i.d. N(0,1) entries (sign(0) = +1).
  With the signs fixed, Q is the unique orthogonal factor whose R has a positive
  diagonal, so any correct QR routine yields the same Pi up to rounding.
* G and S are filled row-major from the Gaussian streams of ``oracle.rng``.
* One Pi and one S per (d, m, seed), shared by every head and by keys and values; the
  rotated vector is y = Pi x and the projection is z = S r.
"""
import numpy as np

from . import rng


def gaussian_matrix(stream_seed, rows, cols):
    return rng.gaussians(stream_seed, rows * cols).reshape(rows, cols)


def haar_rotation(d, seed):
    """Pi (d x d, fp64): Q of the QR of the seeded Gaussian matrix, columns sign-fixed."""
    g = gaussian_matrix(rng.rotation_stream_seed(seed), d, d)
    q, r = np.linalg.qr(g)            # LAPACK Householder QR (a library primitive)
    s = np.sign(np.diag(r))
    s[s == 0] = 1.0
    return q * s[None, :]


def qjl_matrix(m, d, seed):
    """S (m x d, fp64) with i.i.d. N(0,1) entries."""
    return gaussian_matrix(rng.projection_stream_seed(seed), m, d)
