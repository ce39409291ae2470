// Exact re-evaluation of the quantizer's decisions next to a boundary.
//
// [BLOG] "Технология TurboQuant и её применение с локальными LLM", section 1.2 defines each
// code as the Lloyd-Max cell of yhat_j = (Pi x)_j / ||x|| and each QJL bit as the sign of
// (S r)_i with r = x - ||x|| Pi^T c[idx].  The kernels compute yhat and S r in fp32 (tensor-core
// hi/lo pieces or fp32 FMAs), whose error is far below a code cell but not zero, so a value
// that lands within kDeltaCode of a boundary (or a projection within kDeltaSign * ||r|| of
// zero) is taken again here in double-float arithmetic (an fp32 pair hi + lo, ~2^-44
// relative): the decision then equals the one of exact arithmetic, which the fp64 definition
// reaches too, except on a set of inputs of measure ~1e-15 per coordinate.
//
// Every function is warp-collective: all 32 lanes call it with the same row and coordinate,
// each lane holding the vector's coordinates lane * E ... lane * E + E - 1 (E = D / 32).
// Double-float steps follow Dekker (1971) and Knuth's TwoSum; the rounding-explicit
// intrinsics keep the compiler from contracting or reassociating them.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace tq {
namespace exact {

// A decision is re-taken when the fast value is within these margins.  The fast paths'
// errors: fp16 hi/lo tensor-core rotation <= ~2^-20 of ||x|| (piece rounding 2^-22, fp32
// accumulation of 16 MMAs), fp32 FMA rotation ~2^-25 typical; the residual projection
// ~2^-20 of ||r||.  The margins leave a factor of 4 or more above those bounds.
constexpr float kDeltaCode = 1.0f / 262144.0f;   // 2^-18, in units of yhat
constexpr float kDeltaSign = 1.0f / 16384.0f;    // 2^-14, relative to ||r||

struct F2 {
  float hi, lo;
};

__device__ __forceinline__ F2 two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, e};
}
__device__ __forceinline__ F2 fast_two_sum(float a, float b) {   // |a| >= |b| or a == 0
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ F2 add(F2 a, F2 b) {
  F2 s = two_sum(a.hi, b.hi);
  const F2 t = two_sum(a.lo, b.lo);
  s.lo = __fadd_rn(s.lo, t.hi);
  s = fast_two_sum(s.hi, s.lo);
  s.lo = __fadd_rn(s.lo, t.lo);
  return fast_two_sum(s.hi, s.lo);
}
__device__ __forceinline__ F2 neg(F2 a) { return {-a.hi, -a.lo}; }
// (a.hi + a.lo) * x, the leading product exact through the fused multiply-add
__device__ __forceinline__ F2 mul_f(F2 a, float x) {
  const float p = __fmul_rn(a.hi, x);
  float e = __fmaf_rn(a.hi, x, -p);
  e = __fmaf_rn(a.lo, x, e);
  return fast_two_sum(p, e);
}
__device__ __forceinline__ F2 mul(F2 a, F2 b) {
  const float p = __fmul_rn(a.hi, b.hi);
  float e = __fmaf_rn(a.hi, b.hi, -p);
  e = __fmaf_rn(a.hi, b.lo, e);
  e = __fmaf_rn(a.lo, b.hi, e);
  return fast_two_sum(p, e);
}
// The exact sum of the error-free pair operation is symmetric in its operands, so every lane
// of the butterfly ends with bit-identical results.
__device__ __forceinline__ F2 warp_sum(F2 v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const F2 w{__shfl_xor_sync(0xffffffffu, v.hi, o), __shfl_xor_sync(0xffffffffu, v.lo, o)};
    v = add(v, w);
  }
  return v;
}
// sqrt(a) for a > 0: one Newton correction of the fp32 root, s + (a - s^2) / (2 s).
__device__ __forceinline__ F2 sqrt_f2(F2 a) {
  if (!(a.hi > 0.f)) return {0.f, 0.f};
  const float s = __fsqrt_rn(a.hi);
  const float p = __fmul_rn(s, s);
  const float pe = __fmaf_rn(s, s, -p);
  const float r = __fadd_rn(__fsub_rn(__fsub_rn(a.hi, p), pe), a.lo);
  return fast_two_sum(s, __fdiv_rn(r, __fmul_rn(2.f, s)));
}
__device__ __forceinline__ bool nonneg(F2 a) { return a.hi > 0.f || (a.hi == 0.f && a.lo >= 0.f); }

// The lane's E = D / 32 coordinates of a bf16 vector in global memory (exact in fp32).
template <int D>
__device__ __forceinline__ void load_row(const __nv_bfloat16* row, int lane, float* x) {
  constexpr int E = D / 32;
  const __nv_bfloat16* p = row + lane * E;
  if constexpr (E == 2) {
    const __nv_bfloat162 v = *reinterpret_cast<const __nv_bfloat162*>(p);
    x[0] = __low2float(v);
    x[1] = __high2float(v);
  } else {
#pragma unroll
    for (int g = 0; g < E / 4; ++g) {
      const uint2 w = *reinterpret_cast<const uint2*>(p + 4 * g);
      x[4 * g + 0] = __uint_as_float(w.x << 16);
      x[4 * g + 1] = __uint_as_float(w.x & 0xFFFF0000u);
      x[4 * g + 2] = __uint_as_float(w.y << 16);
      x[4 * g + 3] = __uint_as_float(w.y & 0xFFFF0000u);
    }
  }
}

// ||x||: the squares of bf16 values are exact in fp32 (16 significant bits).
template <int D>
__device__ __forceinline__ F2 norm(const float* x) {
  F2 s{0.f, 0.f};
#pragma unroll
  for (int e = 0; e < D / 32; ++e) s = add(s, F2{__fmul_rn(x[e], x[e]), 0.f});
  return sqrt_f2(warp_sum(s));
}

// Lloyd-Max code of coordinate j: #{k : (Pi x)_j >= t_k ||x||} over nb <= 32 boundaries
// (th + tl), for ||x|| > 0.  pih / pil: Pi row-major as hi + lo.
template <int D>
__device__ __forceinline__ int code(const float* x, F2 n, const float* __restrict__ pih,
                                    const float* __restrict__ pil, int j, const float* __restrict__ th,
                                    const float* __restrict__ tl, int nb, int lane) {
  constexpr int E = D / 32;
  F2 y{0.f, 0.f};
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const int i = lane * E + e;
    y = add(y, mul_f(F2{pih[(size_t)j * D + i], pil[(size_t)j * D + i]}, x[e]));
  }
  y = warp_sum(y);
  bool ge = false;
  if (lane < nb) ge = nonneg(add(y, neg(mul(F2{th[lane], tl[lane]}, n))));
  return __popc(__ballot_sync(0xffffffffu, ge));
}

// QJL bit of projection row i: (S r)_i >= 0 with r = x - ||x|| Pi^T c[idx], taken as
// (S x)_i - ||x|| (S' c[idx])_i, S' = S Pi^T (equal in exact arithmetic).  codes: the lane's
// E codes of the vector; sh / sl: S row-major, qh / ql: S' row-major; ch / cl: centroids.
template <int D>
__device__ __forceinline__ bool sign(const float* x, F2 n, const int* codes, const float* __restrict__ sh,
                                     const float* __restrict__ sl, const float* __restrict__ qh,
                                     const float* __restrict__ ql, const float* __restrict__ ch,
                                     const float* __restrict__ cl, int i, int lane) {
  constexpr int E = D / 32;
  F2 a{0.f, 0.f}, b{0.f, 0.f};
#pragma unroll
  for (int e = 0; e < E; ++e) {
    const size_t o = (size_t)i * D + lane * E + e;
    a = add(a, mul_f(F2{sh[o], sl[o]}, x[e]));
    b = add(b, mul(F2{qh[o], ql[o]}, F2{ch[codes[e]], cl[codes[e]]}));
  }
  a = warp_sum(a);
  b = warp_sum(b);
  return nonneg(add(a, neg(mul(n, b))));
}

// The context's double-float tables (one device allocation, see tables_floats).
struct Tables {
  const float *pih, *pil, *sh, *sl, *qh, *ql, *tkh, *tkl, *tvh, *tvl, *ckh, *ckl;
  const float *nkt, *nvt;   // near tables of the key and value books (near_table)
};
__host__ __device__ inline Tables tables(const float* base, int d) {
  const size_t dd = (size_t)d * d;
  Tables t;
  t.pih = base;
  t.pil = base + dd;
  t.sh = base + 2 * dd;
  t.sl = base + 3 * dd;
  t.qh = base + 4 * dd;
  t.ql = base + 5 * dd;
  t.tkh = base + 6 * dd;
  t.tkl = t.tkh + 32;
  t.tvh = t.tkl + 32;
  t.tvl = t.tvh + 32;
  t.ckh = t.tvl + 32;
  t.ckl = t.ckh + 32;
  t.nkt = t.ckl + 32;
  t.nvt = t.nkt + 64;
  return t;
}
__host__ __device__ constexpr size_t tables_floats(int d) { return (size_t)6 * d * d + 6 * 32 + 2 * 64; }

// Near-boundary test of the fast path: cell idx of a code is [t_{idx-1}, t_idx), widened to
// [-2, t_0) and [t_{L-2}, 2) at the ends (|yhat| <= 1); the table holds (centre, half width -
// kDeltaCode) per cell, and yhat is near a boundary iff |yhat - centre| > half width - delta.
__host__ inline void near_table(const double* t, int levels, float* out /* 2 * levels */) {
  for (int k = 0; k < levels; ++k) {
    const double lo = k == 0 ? -2.0 : t[k - 1], hi = k == levels - 1 ? 2.0 : t[k];
    out[2 * k] = (float)(0.5 * (lo + hi));
    out[2 * k + 1] = (float)(0.5 * (hi - lo) - (double)kDeltaCode);
  }
}

}  // namespace exact
}  // namespace tq
