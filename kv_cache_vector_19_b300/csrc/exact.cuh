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

// E consecutive fp32 values at p (E = 2, 4 or 8), 8-byte aligned.
template <int E>
__device__ __forceinline__ void load_f(const float* __restrict__ p, float* v) {
  if constexpr (E == 2) {
    const float2 a = *reinterpret_cast<const float2*>(p);
    v[0] = a.x;
    v[1] = a.y;
  } else {
#pragma unroll
    for (int g = 0; g < E / 2; ++g) {
      const float2 a = *reinterpret_cast<const float2*>(p + 2 * g);
      v[2 * g] = a.x;
      v[2 * g + 1] = a.y;
    }
  }
}

// code() for the vector at `row` (global bf16), every load issued before the arithmetic so
// that one memory round trip serves the whole decision; ||x|| = 0 gives the middle code.
template <int D>
__device__ __forceinline__ int code_of_row(const __nv_bfloat16* row, const float* __restrict__ pih,
                                           const float* __restrict__ pil, int j, const float* __restrict__ th,
                                           const float* __restrict__ tl, int nb, int lane) {
  constexpr int E = D / 32;
  float x[E], ph[E], pl[E];
  load_row<D>(row, lane, x);
  load_f<E>(pih + (size_t)j * D + lane * E, ph);
  load_f<E>(pil + (size_t)j * D + lane * E, pl);
  const float bh = lane < nb ? th[lane] : 0.f, bl = lane < nb ? tl[lane] : 0.f;
  const F2 n = norm<D>(x);
  if (!(n.hi > 0.f)) return (nb + 1) / 2;
  F2 y{0.f, 0.f};
#pragma unroll
  for (int e = 0; e < E; ++e) y = add(y, mul_f(F2{ph[e], pl[e]}, x[e]));
  y = warp_sum(y);
  const bool ge = lane < nb && nonneg(add(y, neg(mul(F2{bh, bl}, n))));
  return __popc(__ballot_sync(0xffffffffu, ge));
}

// sign() for the vector at `row` with the lane's E codes, loads first as in code_of_row.
template <int D>
__device__ __forceinline__ bool sign_of_row(const __nv_bfloat16* row, const int* codes,
                                            const float* __restrict__ sh, const float* __restrict__ sl,
                                            const float* __restrict__ qh, const float* __restrict__ ql,
                                            const float* __restrict__ ch, const float* __restrict__ cl, int i,
                                            int lane) {
  constexpr int E = D / 32;
  float x[E], s_h[E], s_l[E], q_h[E], q_l[E], c_h[E], c_l[E];
  load_row<D>(row, lane, x);
  const size_t o = (size_t)i * D + lane * E;
  load_f<E>(sh + o, s_h);
  load_f<E>(sl + o, s_l);
  load_f<E>(qh + o, q_h);
  load_f<E>(ql + o, q_l);
#pragma unroll
  for (int e = 0; e < E; ++e) {
    c_h[e] = ch[codes[e]];
    c_l[e] = cl[codes[e]];
  }
  const F2 n = norm<D>(x);
  F2 a{0.f, 0.f}, b{0.f, 0.f};
#pragma unroll
  for (int e = 0; e < E; ++e) {
    a = add(a, mul_f(F2{s_h[e], s_l[e]}, x[e]));
    b = add(b, mul(F2{q_h[e], q_l[e]}, F2{c_h[e], c_l[e]}));
  }
  a = warp_sum(a);
  b = warp_sum(b);
  return nonneg(add(a, neg(mul(n, b))));
}

// Two-step forms for callers that hide the memory round trip: pre_*() issues every load of
// one decision into registers (warp-collective, no arithmetic), fin_*() takes it later.
// head_dim 128 (4 coordinates per lane); the bf16 values stay packed until they are used.
struct CodePre {
  uint2 xb;
  float ph[4], pl[4], bh, bl;
};
__device__ __forceinline__ void unpack4(uint2 w, float* x) {
  x[0] = __uint_as_float(w.x << 16);
  x[1] = __uint_as_float(w.x & 0xFFFF0000u);
  x[2] = __uint_as_float(w.y << 16);
  x[3] = __uint_as_float(w.y & 0xFFFF0000u);
}
__device__ __forceinline__ void pre_code(CodePre& p, const __nv_bfloat16* row, const float* __restrict__ pih,
                                         const float* __restrict__ pil, int j, const float* __restrict__ th,
                                         const float* __restrict__ tl, int nb, int lane) {
  p.xb = *reinterpret_cast<const uint2*>(row + lane * 4);
  load_f<4>(pih + (size_t)j * 128 + lane * 4, p.ph);
  load_f<4>(pil + (size_t)j * 128 + lane * 4, p.pl);
  p.bh = lane < nb ? th[lane] : 0.f;
  p.bl = lane < nb ? tl[lane] : 0.f;
}
__device__ __forceinline__ int fin_code(const CodePre& p, int nb, int lane) {
  float x[4];
  unpack4(p.xb, x);
  const F2 n = norm<128>(x);
  if (!(n.hi > 0.f)) return (nb + 1) / 2;
  F2 y{0.f, 0.f};
#pragma unroll
  for (int e = 0; e < 4; ++e) y = add(y, mul_f(F2{p.ph[e], p.pl[e]}, x[e]));
  y = warp_sum(y);
  const bool ge = lane < nb && nonneg(add(y, neg(mul(F2{p.bh, p.bl}, n))));
  return __popc(__ballot_sync(0xffffffffu, ge));
}
struct SignPre {
  uint2 xb;
  float sh[4], sl[4], qh[4], ql[4];
  uint32_t codes;   // the lane's 4 codes, 8 bits each
};
__device__ __forceinline__ void pre_sign(SignPre& p, const __nv_bfloat16* row, uint32_t codes,
                                         const float* __restrict__ sh, const float* __restrict__ sl,
                                         const float* __restrict__ qh, const float* __restrict__ ql, int i, int lane) {
  p.xb = *reinterpret_cast<const uint2*>(row + lane * 4);
  const size_t o = (size_t)i * 128 + lane * 4;
  load_f<4>(sh + o, p.sh);
  load_f<4>(sl + o, p.sl);
  load_f<4>(qh + o, p.qh);
  load_f<4>(ql + o, p.ql);
  p.codes = codes;
}
// ch / cl: the centroids as hi + lo (shared memory)
__device__ __forceinline__ bool fin_sign(const SignPre& p, const float* ch, const float* cl) {
  float x[4];
  unpack4(p.xb, x);
  const F2 n = norm<128>(x);
  F2 a{0.f, 0.f}, b{0.f, 0.f};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int c = (int)((p.codes >> (8 * e)) & 0xFFu);
    a = add(a, mul_f(F2{p.sh[e], p.sl[e]}, x[e]));
    b = add(b, mul(F2{p.qh[e], p.ql[e]}, F2{ch[c], cl[c]}));
  }
  a = warp_sum(a);
  b = warp_sum(b);
  return nonneg(add(a, neg(mul(n, b))));
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
