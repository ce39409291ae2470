"""Lloyd-Max scalar quantizer for one coordinate of a rotated, normalised vector (oracle).

TEST INFRASTRUCTURE (see ``oracle/__init__``).

[BLOG] §1.2, stage 1: after the rotation each coordinate is quantized independently with
an MSE-optimal (Lloyd-Max) scalar quantizer of (b-1) bits.  [3BITS] "Как работает
TurboQuant" (idea two): the distribution of the rotated coordinates is known in advance,
so the optimal grid is computed once and stored; no calibration data is used.

Readings:
* The quantizer acts on yhat = (Pi x) / ||x||, a coordinate of a uniformly random unit
  vector of R^d.  Its exact density is f(t) = (1 - t^2)^((d-3)/2) / B(1/2, (d-1)/2) on
  [-1, 1] (t^2 ~ Beta(1/2, (d-1)/2)).  [3BITS] calls it "close to normal"; N(0, 1/d) is
  its large-d limit and is used only as a check.  The exact density depends on d alone,
  which keeps the codebook data-oblivious.
* Lloyd-Max conditions: every interior boundary is the midpoint of its two neighbouring
  centroids, and every centroid is the conditional mean of its cell.  Solved by the
  Lloyd iteration (alternate the two conditions) from equal-mass cells until no centroid
  moves by more than 1e-10, then by Newton steps on the same conditions (the Lloyd map
  contracts slowly for many levels, rho ~ 0.995 at 32 levels, so plain iteration stalls
  at its rounding floor well before 1e-12 of the fixed point).  The density is symmetric
  and log-concave for d >= 3, so the optimum is unique and symmetric (Fleischer 1964);
  every step keeps the exact antisymmetry c[k] = -c[L-1-k], which makes the middle
  boundary exactly 0.
* Keys use L = 2^(b-1) levels; values use L = 2^b levels (the value path has no QJL stage).
* A code is idx = #{k : yhat >= t_k} over the interior boundaries (a value equal to a
  boundary takes the upper cell).

Cell mass uses the regularised incomplete beta function (SciPy, a library primitive);
the cell's first moment has the closed form int t (1-t^2)^a dt = -(1-t^2)^(a+1) / (2(a+1)).
"""
import numpy as np
from scipy import special


def _alpha(d):
    return (d - 3) / 2.0


def _log_norm(d):
    # log of B(1/2, (d-1)/2) = int_{-1}^{1} (1 - t^2)^((d-3)/2) dt
    return special.betaln(0.5, (d - 1) / 2.0)


def cdf(t, d):
    """P(Y <= t) for one coordinate Y of a uniform unit vector in R^d."""
    t = np.clip(np.asarray(t, dtype=np.float64), -1.0, 1.0)
    half = 0.5 * special.betainc(0.5, (d - 1) / 2.0, t * t)
    return np.where(t >= 0, 0.5 + half, 0.5 - half)


def ppf(p, d):
    """Inverse of ``cdf``."""
    p = np.asarray(p, dtype=np.float64)
    x = special.betaincinv(0.5, (d - 1) / 2.0, np.abs(2.0 * p - 1.0))
    return np.sign(p - 0.5) * np.sqrt(x)


def first_moment(a, b, d):
    """int_a^b t f(t) dt (closed form)."""
    al = _alpha(d)
    g = lambda t: -np.power(np.clip(1.0 - np.asarray(t) ** 2, 0.0, None), al + 1.0) / (2.0 * (al + 1.0))
    return (g(b) - g(a)) / np.exp(_log_norm(d))


def second_moment(a, b, d):
    """int_a^b t^2 f(t) dt, from the Beta(3/2, (d-1)/2) law of t^2 on each half-line."""
    # E[Y^2 ; Y in [0, x]] = (1/2) E[T ; T <= x^2] with T = Y^2 ~ Beta(1/2, (d-1)/2)
    #                      = (1/2) (1/d) I_{x^2}(3/2, (d-1)/2)
    def s(t):
        t = np.clip(np.asarray(t, dtype=np.float64), -1.0, 1.0)
        v = 0.5 / d * special.betainc(1.5, (d - 1) / 2.0, t * t)
        return np.sign(t) * v
    return s(b) - s(a)


def density(t, d):
    t = np.asarray(t, dtype=np.float64)
    return np.power(np.clip(1.0 - t * t, 0.0, None), _alpha(d)) / np.exp(_log_norm(d))


def lloyd_map(c, d):
    """One Lloyd step: boundaries at centroid midpoints, then cell conditional means."""
    t = 0.5 * (c[:-1] + c[1:])
    edges = np.concatenate(([-1.0], t, [1.0]))
    mass = cdf(edges[1:], d) - cdf(edges[:-1], d)
    tc = first_moment(edges[:-1], edges[1:], d) / mass
    return 0.5 * (tc - tc[::-1]), edges, mass


def _lloyd_jacobian(c, d):
    """d T(c) / d c for the Lloyd map T (tridiagonal)."""
    L = len(c)
    tc, edges, mass = lloyd_map(c, d)
    f = density(edges, d)
    # dT_k/dt_k (lower edge) and dT_k/dt_{k+1} (upper edge); end edges are fixed
    lo = f[:-1] * (tc - edges[:-1]) / mass
    hi = f[1:] * (edges[1:] - tc) / mass
    J = np.zeros((L, L))
    for k in range(L):
        if k > 0:
            J[k, k - 1] += 0.5 * lo[k]
            J[k, k] += 0.5 * lo[k]
        if k < L - 1:
            J[k, k] += 0.5 * hi[k]
            J[k, k + 1] += 0.5 * hi[k]
    return tc, J


def lloyd_max(d, levels, lloyd_tol=1e-10, max_iter=200000, newton_steps=20):
    """Centroids c[0..L-1] (ascending) and interior boundaries t[1..L-1] for the density of
    one coordinate of a uniform unit vector in R^d.  Returns (centroids, boundaries, iters)."""
    if d < 3:
        raise ValueError("d >= 3 required")
    L = int(levels)
    if L == 1:
        return np.zeros(1), np.zeros(0), 0
    t = ppf(np.arange(1, L) / L, d)                  # equal-mass start
    edges = np.concatenate(([-1.0], t, [1.0]))
    c = first_moment(edges[:-1], edges[1:], d) / (cdf(edges[1:], d) - cdf(edges[:-1], d))
    c = 0.5 * (c - c[::-1])
    it = 0
    for it in range(1, max_iter + 1):                # Lloyd iteration
        c_new = lloyd_map(c, d)[0]
        delta = np.max(np.abs(c_new - c))
        c = c_new
        if delta < lloyd_tol:
            break
    for _ in range(newton_steps):                    # Newton on T(c) - c = 0
        tc, J = _lloyd_jacobian(c, d)
        step = np.linalg.solve(J - np.eye(L), -(tc - c))
        step = 0.5 * (step - step[::-1])
        c = c + step
        it += 1
        if np.max(np.abs(step)) <= 1e-17:
            break
    t = 0.5 * (c[:-1] + c[1:])
    return c, t, it


def distortion(c, t, d):
    """Per-coordinate MSE E[(Y - c[idx(Y)])^2] of the quantizer (c, t) under the density."""
    edges = np.concatenate(([-1.0], np.asarray(t), [1.0]))
    a, b = edges[:-1], edges[1:]
    m0 = cdf(b, d) - cdf(a, d)
    m1 = first_moment(a, b, d)
    m2 = second_moment(a, b, d)
    return float(np.sum(m2 - 2.0 * c * m1 + c * c * m0))


def encode(yhat, boundaries):
    """idx = #{k : yhat >= t_k}."""
    return np.searchsorted(np.asarray(boundaries), yhat, side="right")


_CACHE = {}


def codebook(d, levels):
    """Cached (centroids, boundaries) for (d, L)."""
    key = (int(d), int(levels))
    if key not in _CACHE:
        c, t, _ = lloyd_max(d, levels)
        _CACHE[key] = (c, t)
    return _CACHE[key]
