// Host-side constants of the method: seeded random matrices and Lloyd-Max codebooks.
//
// [BLOG] "Технология TurboQuant и её применение с локальными LLM", section 1.2: every KV
// vector is rotated by a random orthogonal matrix, each rotated coordinate is quantized by
// an MSE-optimal Lloyd-Max scalar quantizer, and the residual is sketched by the signs of
// a random Gaussian projection.  [3BITS] "3 бита вместо 16 ...", "Как работает
// TurboQuant": the codebook is computed once for the known coordinate distribution and
// stored; no calibration.
//
// Everything here is fp64 and runs once per context, off the hot path.
#include <cmath>
#include <cstring>
#include <vector>

#include "tq_internal.h"

namespace tq {

// ---- SplitMix64 (Steele, Lea & Flood 2014; finaliser constants as published by Vigna) ----
// Output i of the stream seeded with s is mix(s + (i+1) * golden_gamma).
static inline uint64_t splitmix_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
  z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
  return z ^ (z >> 31);
}

// Fills out[0..count) with N(0,1) draws: uniforms u = (x >> 11) * 2^-53 taken in pairs
// (u1, u2); Box-Muller with w = 1 - u1 in (0, 1] gives sqrt(-2 ln w) cos(2 pi u2), then
// the matching sin.
void gaussian_stream(uint64_t stream_seed, size_t count, double* out) {
  const uint64_t gamma = 0x9E3779B97F4A7C15ULL;
  uint64_t state = stream_seed;
  const double two_pi = 6.283185307179586476925286766559;
  for (size_t i = 0; i < count; i += 2) {
    state += gamma;
    double u1 = (double)(splitmix_mix(state) >> 11) * 0x1.0p-53;
    state += gamma;
    double u2 = (double)(splitmix_mix(state) >> 11) * 0x1.0p-53;
    double rad = std::sqrt(-2.0 * std::log(1.0 - u1));
    double th = two_pi * u2;
    out[i] = rad * std::cos(th);
    if (i + 1 < count) out[i + 1] = rad * std::sin(th);
  }
}

// ---- Haar rotation: Householder QR of a Gaussian matrix, signs of diag(R) moved into Q ----
// Returns Pi row-major (y = Pi x).  With diag(R) > 0 the Q factor is unique, so any correct
// QR gives the same Pi up to rounding.
void haar_rotation(int d, uint64_t seed, double* pi) {
  std::vector<double> a((size_t)d * d);
  gaussian_stream(2 * seed, a.size(), a.data());        // row-major G
  std::vector<double> vs((size_t)d * d, 0.0);            // Householder vector k in vs[k*d ..]
  std::vector<double> rdiag(d);
  for (int k = 0; k < d; ++k) {
    double norm2 = 0.0;
    for (int i = k; i < d; ++i) norm2 += a[(size_t)i * d + k] * a[(size_t)i * d + k];
    double x0 = a[(size_t)k * d + k];
    double alpha = (x0 >= 0.0 ? -1.0 : 1.0) * std::sqrt(norm2);
    double* v = &vs[(size_t)k * d];
    double vnorm2 = 0.0;
    for (int i = k; i < d; ++i) {
      v[i] = a[(size_t)i * d + k] - (i == k ? alpha : 0.0);
      vnorm2 += v[i] * v[i];
    }
    if (vnorm2 > 0.0) {
      double inv = 1.0 / std::sqrt(vnorm2);
      for (int i = k; i < d; ++i) v[i] *= inv;
      // A[k:, k:] -= 2 v (v^T A[k:, k:])
      for (int j = k; j < d; ++j) {
        double dot = 0.0;
        for (int i = k; i < d; ++i) dot += v[i] * a[(size_t)i * d + j];
        for (int i = k; i < d; ++i) a[(size_t)i * d + j] -= 2.0 * v[i] * dot;
      }
    }
    rdiag[k] = a[(size_t)k * d + k];
  }
  // Q = H_0 H_1 ... H_{d-1} I, applied from the right-most reflector inwards.
  std::vector<double> q((size_t)d * d, 0.0);
  for (int i = 0; i < d; ++i) q[(size_t)i * d + i] = 1.0;
  for (int k = d - 1; k >= 0; --k) {
    const double* v = &vs[(size_t)k * d];
    for (int j = 0; j < d; ++j) {
      double dot = 0.0;
      for (int i = k; i < d; ++i) dot += v[i] * q[(size_t)i * d + j];
      for (int i = k; i < d; ++i) q[(size_t)i * d + j] -= 2.0 * v[i] * dot;
    }
  }
  for (int i = 0; i < d; ++i)
    for (int j = 0; j < d; ++j) pi[(size_t)i * d + j] = q[(size_t)i * d + j] * (rdiag[j] < 0.0 ? -1.0 : 1.0);
}

void gaussian_projection(int m, int d, uint64_t seed, double* s) {
  gaussian_stream(2 * seed + 1, (size_t)m * d, s);
}

// ---- Lloyd-Max for f(t) = (1 - t^2)^a / Z on [-1, 1], a = (d - 3) / 2 ------------------

namespace {

// n-point Gauss-Legendre rule on [-1, 1]: nodes by Newton's method on P_n (three-term
// recurrence), weights 2 / ((1 - x^2) P_n'(x)^2).
struct Gauss {
  std::vector<double> x, w;
  static void legendre(int n, double z, double& pn, double& dpn) {
    double p0 = 1.0, p1 = z;
    for (int k = 2; k <= n; ++k) {
      double p2 = ((2.0 * k - 1.0) * z * p1 - (k - 1.0) * p0) / k;
      p0 = p1;
      p1 = p2;
    }
    pn = p1;
    dpn = n * (z * p1 - p0) / (z * z - 1.0);
  }
  explicit Gauss(int n) : x(n), w(n) {
    for (int i = 0; i < n; ++i) {
      double z = std::cos(M_PI * (i + 0.75) / (n + 0.5));
      for (int it = 0; it < 100; ++it) {
        double pn, dpn;
        legendre(n, z, pn, dpn);
        double dz = pn / dpn;
        z -= dz;
        if (std::fabs(dz) < 1e-17) break;
      }
      double pn, dpn;
      legendre(n, z, pn, dpn);
      x[i] = z;
      w[i] = 2.0 / ((1.0 - z * z) * dpn * dpn);
    }
  }
};

struct Sphere {
  int d;
  double a, log_z;
  const Gauss& g;
  Sphere(int d_, const Gauss& g_) : d(d_), a((d_ - 3) / 2.0), g(g_) {
    // Z = B(1/2, (d-1)/2) = Gamma(1/2) Gamma((d-1)/2) / Gamma(d/2)
    log_z = std::lgamma(0.5) + std::lgamma((d - 1) / 2.0) - std::lgamma(d / 2.0);
  }
  double dens(double t) const {
    double u = 1.0 - t * t;
    return u <= 0.0 ? 0.0 : std::exp(a * std::log(u) - log_z);
  }
  double rule(double lo, double hi) const {
    double c = 0.5 * (lo + hi), h = 0.5 * (hi - lo), s = 0.0;
    for (size_t i = 0; i < g.x.size(); ++i) s += g.w[i] * dens(c + h * g.x[i]);
    return s * h;
  }
  // Composite rule: panels no wider than a sixteenth of the density's width 2/sqrt(d),
  // on each of which the 24-point rule is exact to rounding (the integrand is smooth at
  // that scale: (1 - t^2)^a behaves like exp(-d t^2 / 2)).
  double mass(double lo, double hi) const {
    if (hi <= lo) return 0.0;
    const double panel = 0.125 / std::sqrt((double)d);
    int n = (int)std::ceil((hi - lo) / panel);
    if (n < 1) n = 1;
    const double h = (hi - lo) / n;
    double s = 0.0;
    for (int i = 0; i < n; ++i) s += rule(lo + i * h, lo + (i + 1) * h);
    return s;
  }
  // int_lo^hi t f(t) dt in closed form: antiderivative -(1-t^2)^(a+1) / (2 (a+1) Z)
  double first_moment(double lo, double hi) const {
    auto g1 = [&](double t) {
      double u = 1.0 - t * t;
      return u <= 0.0 ? 0.0 : -std::exp((a + 1.0) * std::log(u) - log_z) / (2.0 * (a + 1.0));
    };
    return g1(hi) - g1(lo);
  }
};

// Lloyd map: boundaries at centroid midpoints, then cell conditional means (antisymmetrised).
void lloyd_map(const Sphere& sp, const std::vector<double>& c, std::vector<double>& tc,
               std::vector<double>& edges, std::vector<double>& mass) {
  int L = (int)c.size();
  edges.assign(L + 1, 0.0);
  edges[0] = -1.0;
  edges[L] = 1.0;
  for (int k = 1; k < L; ++k) edges[k] = 0.5 * (c[k - 1] + c[k]);
  mass.assign(L, 0.0);
  std::vector<double> raw(L);
  for (int k = 0; k < L; ++k) {
    mass[k] = sp.mass(edges[k], edges[k + 1]);
    raw[k] = sp.first_moment(edges[k], edges[k + 1]) / mass[k];
  }
  tc.assign(L, 0.0);
  for (int k = 0; k < L; ++k) tc[k] = 0.5 * (raw[k] - raw[L - 1 - k]);
}

// Dense Gaussian elimination with partial pivoting (L <= 64).
bool solve(std::vector<double> A, std::vector<double> b, int n, std::vector<double>& x) {
  for (int col = 0; col < n; ++col) {
    int piv = col;
    for (int r = col + 1; r < n; ++r)
      if (std::fabs(A[r * n + col]) > std::fabs(A[piv * n + col])) piv = r;
    if (A[piv * n + col] == 0.0) return false;
    if (piv != col) {
      for (int k = 0; k < n; ++k) std::swap(A[col * n + k], A[piv * n + k]);
      std::swap(b[col], b[piv]);
    }
    for (int r = col + 1; r < n; ++r) {
      double f = A[r * n + col] / A[col * n + col];
      for (int k = col; k < n; ++k) A[r * n + k] -= f * A[col * n + k];
      b[r] -= f * b[col];
    }
  }
  x.assign(n, 0.0);
  for (int r = n - 1; r >= 0; --r) {
    double s = b[r];
    for (int k = r + 1; k < n; ++k) s -= A[r * n + k] * x[k];
    x[r] = s / A[r * n + r];
  }
  return true;
}

}  // namespace

// Centroids from an equal-mass start: Lloyd iteration until no centroid moves by 1e-10,
// then Newton steps on T(c) - c = 0 (the Lloyd map contracts slowly for many levels).
int lloyd_max(int d, int L, double* centroids, double* boundaries) {
  static const Gauss gauss(24);
  Sphere sp(d, gauss);
  // equal-mass start: invert the cumulative mass by bisection
  std::vector<double> edges(L + 1);
  edges[0] = -1.0;
  edges[L] = 1.0;
  for (int k = 1; k < L; ++k) {
    double target = (double)k / L, lo = -1.0, hi = 1.0;
    for (int it = 0; it < 200; ++it) {
      double mid = 0.5 * (lo + hi);
      double m = mid <= 0.0 ? 0.5 - sp.mass(mid, 0.0) : 0.5 + sp.mass(0.0, mid);
      (m < target ? lo : hi) = mid;
    }
    edges[k] = 0.5 * (lo + hi);
  }
  std::vector<double> c(L), tc, e2, mass;
  for (int k = 0; k < L; ++k) c[k] = sp.first_moment(edges[k], edges[k + 1]) / sp.mass(edges[k], edges[k + 1]);
  {
    std::vector<double> s(L);
    for (int k = 0; k < L; ++k) s[k] = 0.5 * (c[k] - c[L - 1 - k]);
    c = s;
  }
  bool done = false;
  for (int it = 0; it < 200000; ++it) {
    lloyd_map(sp, c, tc, e2, mass);
    double delta = 0.0;
    for (int k = 0; k < L; ++k) delta = std::fmax(delta, std::fabs(tc[k] - c[k]));
    c = tc;
    if (delta < 1e-10) {
      done = true;
      break;
    }
  }
  if (!done) return TQ_ENOTCONV;
  for (int step = 0; step < 20; ++step) {
    lloyd_map(sp, c, tc, e2, mass);
    std::vector<double> J((size_t)L * L, 0.0), rhs(L), x;
    for (int k = 0; k < L; ++k) {
      double lo = sp.dens(e2[k]) * (tc[k] - e2[k]) / mass[k];       // dT_k / d(lower edge)
      double hi = sp.dens(e2[k + 1]) * (e2[k + 1] - tc[k]) / mass[k];  // dT_k / d(upper edge)
      if (k > 0) {
        J[k * L + k - 1] += 0.5 * lo;
        J[k * L + k] += 0.5 * lo;
      }
      if (k < L - 1) {
        J[k * L + k] += 0.5 * hi;
        J[k * L + k + 1] += 0.5 * hi;
      }
      J[k * L + k] -= 1.0;
      rhs[k] = -(tc[k] - c[k]);
    }
    if (!solve(J, rhs, L, x)) return TQ_ENOTCONV;
    double mx = 0.0;
    for (int k = 0; k < L; ++k) {
      double st = 0.5 * (x[k] - x[L - 1 - k]);
      c[k] += st;
      mx = std::fmax(mx, std::fabs(st));
    }
    if (mx <= 1e-17) break;
  }
  for (int k = 0; k < L; ++k) centroids[k] = c[k];
  for (int k = 1; k < L; ++k) boundaries[k - 1] = 0.5 * (c[k - 1] + c[k]);
  return TQ_OK;
}

}  // namespace tq

extern "C" int tq_make_codebook(int d, int levels, double* centroids, double* boundaries) {
  if (d < 3 || d > 65536 || levels < 2 || levels > 64 || !centroids || !boundaries) return TQ_EINVAL;
  return tq::lloyd_max(d, levels, centroids, boundaries);
}

extern "C" int tq_make_rotation(int d, uint64_t seed, double* pi_out) {
  if (d < 1 || d > 4096 || !pi_out) return TQ_EINVAL;
  tq::haar_rotation(d, seed, pi_out);
  return TQ_OK;
}

extern "C" int tq_make_projection(int m, int d, uint64_t seed, double* s_out) {
  if (m < 1 || d < 1 || m > 4096 || d > 4096 || !s_out) return TQ_EINVAL;
  tq::gaussian_projection(m, d, seed, s_out);
  return TQ_OK;
}
