// Format version 2: separate key and value widths, keys with or without the QJL stage.
//
// [3BITS] "3 бита вместо 16: разбираем TurboQuant ...", "Python + HuggingFace": a cache object
// is built with key_bits and value_bits, and the stage-1 quantizer alone returns indices and
// norms; the same page notes that the llama.cpp forks switch the QJL stage off for keys.
// [BLOG] "Технология TurboQuant и её применение с локальными LLM", section 1.2 defines both
// stages.  A version-2 page keeps the version-1 regions, order and bit order with KB key code
// planes, VB value code planes and m sign bits per token; m = 0 (no QJL) drops the sign and
// gamma regions.  Version 1 is KB = b - 1, VB = b, m = d; such contexts take the version-1
// kernels, everything else comes here.
//
// CUDA cores, fp32, the plane counts and m read at run time: the quantizer of a page tile
// (Y = X Pi^T, Lloyd-Max codes, residual, Z = R S'^T, signs), the split decode with its
// prologue and the shared combine, and the dequantizer.  Decisions within the exact-decision
// band are taken again in double-float arithmetic (exact.cuh), as in the version-1 kernels.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "exact.cuh"
#include "layout.cuh"
#include "tq_internal.h"

namespace tq {
namespace kv2 {

struct Geom {   // one version-2 page
  int kb, vb, m;   // key code planes, value code planes, sign bits per token (0: no QJL)
  int off_kcodes, off_signs, off_nk, off_gamma, off_vcodes, off_nv, bytes;
};

Geom geom_of(const tq_ctx* c) {
  Geom g;
  const int d = c->d, P = kPage;
  g.kb = c->kb;
  g.vb = c->vb;
  g.m = c->m;
  g.off_kcodes = 0;
  g.off_signs = g.off_kcodes + g.kb * P * d / 8;
  g.off_nk = g.off_signs + P * g.m / 8;
  g.off_gamma = g.off_nk + 4 * P;
  g.off_vcodes = g.off_gamma + (g.m > 0 ? 4 * P : 0);
  g.off_nv = g.off_vcodes + g.vb * d * 4 * 4;
  g.bytes = g.off_nv + 4 * P;
  return g;
}

constexpr int kThreads = 256;
constexpr int kRows = 64;
constexpr int kMaxPlanes = 5;

// ---------------------------------------------------------------- quantizer

struct QArgs {
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  int kv_heads, n_tokens, max_tokens, pages_per_seq;
  const int32_t* start_pos;
  uint8_t* cache;
  const float* pit;   // [D][D] Pi^T
  const float* spt;   // [D][m] S'^T
  const float* ck;
  const float* tk;
  const float* cv;
  const float* tv;
  const float* exact;
  int* status;
  PageMap pm;
  KVLayout lay;         // element strides of k and v over (batch, KV head, token)
  Geom g;
};

// C[64][N] (row stride N+1) = A[64][D] (row stride D+1) * Bt[D][N]; 256 threads, each owns
// rows ty + 16 i (i < 4) and columns tx*4 + 64 cc + (0..3).
template <int D, int N>
__device__ __forceinline__ void gemm64(const float* __restrict__ A, const float* __restrict__ Bt,
                                       float* __restrict__ C) {
  constexpr int NC = N / 64;
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15;
  float acc[4][NC][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int cc = 0; cc < NC; ++cc)
#pragma unroll
      for (int u = 0; u < 4; ++u) acc[i][cc][u] = 0.f;
#pragma unroll 4
  for (int kk = 0; kk < D; ++kk) {
    float av[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) av[i] = A[(ty + 16 * i) * (D + 1) + kk];
#pragma unroll
    for (int cc = 0; cc < NC; ++cc) {
      const float4 bv = __ldg(reinterpret_cast<const float4*>(Bt + (size_t)kk * N + tx * 4 + 64 * cc));
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[i][cc][0] = fmaf(av[i], bv.x, acc[i][cc][0]);
        acc[i][cc][1] = fmaf(av[i], bv.y, acc[i][cc][1]);
        acc[i][cc][2] = fmaf(av[i], bv.z, acc[i][cc][2]);
        acc[i][cc][3] = fmaf(av[i], bv.w, acc[i][cc][3]);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int cc = 0; cc < NC; ++cc)
#pragma unroll
      for (int u = 0; u < 4; ++u) C[(ty + 16 * i) * (N + 1) + tx * 4 + 64 * cc + u] = acc[i][cc][u];
}

// Loads 64 bf16 rows (slots s0 .. s0+63 of the page) into fp32 rows of xs; rows outside
// [lo, hi) are zero.  Then one warp per row computes the fp32 norm.
template <int D>
__device__ __forceinline__ void load_rows(const __nv_bfloat16* __restrict__ src_seq, int64_t ts, int page, int start, int s0,
                                          int lo, int hi, float* xs, float* nrm) {
  const int tid = threadIdx.x;
  for (int e = tid; e < kRows * (D / 8); e += kThreads) {
    const int row = e / (D / 8), ch = e % (D / 8);
    const int slot = s0 + row;
    float f[8];
    if (slot >= lo && slot < hi) {
      const long tok = (long)page * 128 + slot - start;
      const uint4 raw = __ldg(reinterpret_cast<const uint4*>(src_seq + tok * ts) + ch);
      const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        f[2 * u] = __uint_as_float(w[u] << 16);
        f[2 * u + 1] = __uint_as_float(w[u] & 0xFFFF0000u);
      }
    } else {
#pragma unroll
      for (int u = 0; u < 8; ++u) f[u] = 0.f;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) xs[row * (D + 1) + ch * 8 + u] = f[u];
  }
  __syncthreads();
  const int warp = tid >> 5, lane = tid & 31;
  for (int row = warp; row < kRows; row += kThreads / 32) {
    float s = 0.f;
    for (int j = lane; j < D; j += 32) {
      const float x = xs[row * (D + 1) + j];
      s = fmaf(x, x, s);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) nrm[row] = sqrtf(s);
  }
  __syncthreads();
}

// Warp-collective: this warp's codes that the fast value put next to a boundary, taken again
// exactly; returns this thread's (possibly new) code.
template <int D>
__device__ __forceinline__ int resolve_codes(bool near, int idx, int row, int j, const __nv_bfloat16* src_seq,
                                             int64_t ts, int page, int start, int s0, const float* pih, const float* pil,
                                             const float* th, const float* tl, int nb, int lane) {
  uint32_t ev = __ballot_sync(0xffffffffu, near);
  while (ev) {
    const int L = __ffs(ev) - 1;
    ev &= ev - 1;
    const int rowL = __shfl_sync(0xffffffffu, row, L), jL = __shfl_sync(0xffffffffu, j, L);
    const int r = exact::code_of_row<D>(src_seq + ((long)page * 128 + s0 + rowL - start) * ts, pih, pil, jL, th, tl,
                                        nb, lane);
    if (lane == L) idx = r;
  }
  return idx;
}

// Fast Lloyd-Max code (boundary count) and whether it is within the exact-decision band
// (near table: one (centre, half width - delta) pair per cell).
__device__ __forceinline__ int fast_code(float yh, const float* t, int nb, const float2* cells, bool& near) {
  int idx = 0;
  for (int q = 0; q < nb; ++q) idx += (yh >= t[q]) ? 1 : 0;
  near = fabsf(yh - cells[idx].x) > cells[idx].y;
  return idx;
}

template <int D>
__global__ void __launch_bounds__(kThreads) quantize_kernel(QArgs a) {
  const Geom g = a.g;
  constexpr int KW = D / 32;
  const int LK = 1 << g.kb, LV = 1 << g.vb, SW = g.m / 32;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float* xs = reinterpret_cast<float*>(smem_raw);                 // [64][D+1]  X, later Z
  float* ys = xs + kRows * (D + 1);                                // [64][D+1]  Y, later R
  float* nrm = ys + kRows * (D + 1);                               // [64]
  float* gam = nrm + kRows;                                        // [64]
  float* s_ck = gam + kRows;                                       // [32]
  float* s_tk = s_ck + 32;
  float* s_cv = s_tk + 32;
  float* s_tv = s_cv + 32;
  float2* s_nk = reinterpret_cast<float2*>(s_tv + 32);              // [32]
  float2* s_nv = s_nk + 32;                                        // [32]
  uint8_t* kcode = reinterpret_cast<uint8_t*>(s_nv + 32);           // [64][D]
  uint8_t* vcode = kcode + kRows * D;                              // [128][D]

  const int tid = threadIdx.x, lane = tid & 31;
  const int b = blockIdx.z, h = blockIdx.y;
  const int start = a.start_pos[b];
  if (start < 0 || start > a.max_tokens - a.n_tokens) {
    if (tid == 0 && blockIdx.x == 0) atomicOr(a.status, kFlagBounds);
    return;
  }
  const int page = start / 128 + blockIdx.x;
  const int lo = max(start, page * 128) - page * 128;
  const int hi = min(start + a.n_tokens, page * 128 + 128) - page * 128;
  if (lo >= hi) return;

  const exact::Tables T = exact::tables(a.exact, D);
  for (int i = tid; i < LK; i += kThreads) s_ck[i] = a.ck[i];
  for (int i = tid; i < LK - 1; i += kThreads) s_tk[i] = a.tk[i];
  for (int i = tid; i < LV; i += kThreads) s_cv[i] = a.cv[i];
  for (int i = tid; i < LV - 1; i += kThreads) s_tv[i] = a.tv[i];
  for (int i = tid; i < 2 * LK; i += kThreads) reinterpret_cast<float*>(s_nk)[i] = T.nkt[i];
  for (int i = tid; i < 2 * LV; i += kThreads) reinterpret_cast<float*>(s_nv)[i] = T.nvt[i];

  const size_t seq = (size_t)b * a.kv_heads + h;
  uint8_t* pg = a.cache + a.pm.index((int)seq, a.kv_heads, a.pages_per_seq, page, a.status) * g.bytes;
  uint32_t* g_kc = reinterpret_cast<uint32_t*>(pg + g.off_kcodes);
  uint32_t* g_sg = reinterpret_cast<uint32_t*>(pg + g.off_signs);
  float* g_nk = reinterpret_cast<float*>(pg + g.off_nk);
  float* g_gm = reinterpret_cast<float*>(pg + g.off_gamma);
  uint32_t* g_vc = reinterpret_cast<uint32_t*>(pg + g.off_vcodes);
  float* g_nv = reinterpret_cast<float*>(pg + g.off_nv);
  const __nv_bfloat16* kseq = a.k + (b * a.lay.kb + h * a.lay.kh);   // token i at kseq + i kt
  const __nv_bfloat16* vseq = a.v + (b * a.lay.vb + h * a.lay.vh);
  __syncthreads();

  for (int half = 0; half < 2; ++half) {
    const int s0 = half * kRows;
    if (hi <= s0 || lo >= s0 + kRows) continue;
    // ---------------- keys ----------------
    load_rows<D>(kseq, a.lay.kt, page, start, s0, lo, hi, xs, nrm);
    gemm64<D, D>(xs, a.pit, ys);
    __syncthreads();
    for (int e = tid; e < kRows * D; e += kThreads) {
      const int row = e / D, j = e % D;
      const float n = nrm[row];
      const float y = ys[row * (D + 1) + j];
      const float yh = n > 0.f ? y / n : 0.f;
      bool near;
      int idx = fast_code(yh, s_tk, LK - 1, s_nk, near);
      idx = resolve_codes<D>(near && n > 0.f, idx, row, j, kseq, a.lay.kt, page, start, s0, T.pih, T.pil, T.tkh, T.tkl, LK - 1,
                             lane);
      kcode[row * D + j] = (uint8_t)idx;
      ys[row * (D + 1) + j] = y - n * s_ck[idx];   // r_rot = Pi r
    }
    __syncthreads();
    if (g.m > 0) {
      const int warp = tid >> 5;
      for (int row = warp; row < kRows; row += kThreads / 32) {
        float s = 0.f;
        for (int j = lane; j < D; j += 32) {
          const float r = ys[row * (D + 1) + j];
          s = fmaf(r, r, s);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) gam[row] = sqrtf(s);
      }
      gemm64<D, D>(ys, a.spt, xs);   // Z = R S'^T (m == D)
      __syncthreads();
      // projections next to zero: exact sign (stored back into Z as +-1)
      for (int e = tid; e < kRows * D; e += kThreads) {
        const int row = e / D, i = e % D;
        const float z = xs[row * (D + 1) + i];
        uint32_t ev = __ballot_sync(0xffffffffu, fabsf(z) < exact::kDeltaSign * gam[row]);
        while (ev) {
          const int L = __ffs(ev) - 1;
          ev &= ev - 1;
          const int rowL = __shfl_sync(0xffffffffu, row, L), iL = __shfl_sync(0xffffffffu, i, L);
          int codes[D / 32];
#pragma unroll
          for (int q = 0; q < D / 32; ++q) codes[q] = kcode[rowL * D + lane * (D / 32) + q];
          const bool sg = exact::sign_of_row<D>(kseq + ((long)page * 128 + s0 + rowL - start) * a.lay.kt, codes, T.sh, T.sl,
                                                T.qh, T.ql, T.ckh, T.ckl, iL, lane);
          if (lane == L) xs[row * (D + 1) + i] = sg ? 1.f : -1.f;
        }
      }
      __syncthreads();
    }
    // bit-pack the key-code planes (and the sign plane), one word per thread-iteration
    const int np = g.kb + (g.m > 0 ? 1 : 0);
    for (int e = tid; e < kRows * np * KW; e += kThreads) {
      const int row = e / (np * KW), rem = e % (np * KW);
      const int plane = rem / KW, w = rem % KW;
      const int slot = s0 + row;
      if (slot < lo || slot >= hi) continue;
      uint32_t word = 0;
#pragma unroll 8
      for (int bit = 0; bit < 32; ++bit) {
        const int j = coord_of<D>(w, bit);
        const uint32_t v = plane < g.kb ? (uint32_t)((kcode[row * D + j] >> plane) & 1)
                                        : (uint32_t)(xs[row * (D + 1) + j] >= 0.f);
        word |= v << bit;
      }
      if (plane < g.kb)
        g_kc[((size_t)plane * 128 + slot) * KW + w] = word;
      else
        g_sg[(size_t)slot * SW + w] = word;
    }
    for (int row = tid; row < kRows; row += kThreads) {
      const int slot = s0 + row;
      if (slot >= lo && slot < hi) {
        g_nk[slot] = nrm[row];
        if (g.m > 0) g_gm[slot] = gam[row];
      }
    }
    __syncthreads();
    // ---------------- values ----------------
    load_rows<D>(vseq, a.lay.vt, page, start, s0, lo, hi, xs, nrm);
    gemm64<D, D>(xs, a.pit, ys);
    __syncthreads();
    for (int e = tid; e < kRows * D; e += kThreads) {
      const int row = e / D, j = e % D;
      const float n = nrm[row];
      const float yh = n > 0.f ? ys[row * (D + 1) + j] / n : 0.f;
      bool near;
      int idx = fast_code(yh, s_tv, LV - 1, s_nv, near);
      idx = resolve_codes<D>(near && n > 0.f, idx, row, j, vseq, a.lay.vt, page, start, s0, T.pih, T.pil, T.tvh, T.tvl, LV - 1,
                             lane);
      vcode[(s0 + row) * D + j] = (uint8_t)idx;
    }
    for (int row = tid; row < kRows; row += kThreads) {
      const int slot = s0 + row;
      if (slot >= lo && slot < hi) g_nv[slot] = nrm[row];
    }
    __syncthreads();
  }
  // value-code words: [plane][coord][4], each over 32 slots of the page
  for (int e = tid; e < g.vb * D * 4; e += kThreads) {
    const int plane = e / (D * 4), rem = e % (D * 4), j = rem >> 2, c = rem & 3;
    uint32_t word = 0, mask = 0;
#pragma unroll 8
    for (int bit = 0; bit < 32; ++bit) {
      const int slot = slot_of(c, bit);
      if (slot >= lo && slot < hi) {
        mask |= 1u << bit;
        word |= (uint32_t)((vcode[slot * D + j] >> plane) & 1) << bit;
      }
    }
    uint32_t* dst = g_vc + ((size_t)plane * D + j) * 4 + c;
    if (mask == 0xffffffffu) {
      *dst = word;
    } else if (mask != 0u) {
      atomicAnd(dst, ~mask);
      atomicOr(dst, word);
    }
  }
}

template <int D>
constexpr size_t quant_smem_bytes() {
  return (size_t)2 * kRows * (D + 1) * 4 + 2 * kRows * 4 + (4 * 32 + 2 * 64) * 4 + (size_t)kRows * D + (size_t)128 * D;
}

template <int D>
int launch_q(const tq_ctx* c, const void* k, const void* v, int batch, int kv_heads, int n_tokens,
             const int32_t* start_pos, void* cache, int max_tokens, cudaStream_t st, const PageMap& pm,
             const KVLayout& lay) {
  QArgs a;
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.kv_heads = kv_heads;
  a.n_tokens = n_tokens;
  a.max_tokens = max_tokens;
  a.pages_per_seq = (max_tokens + 127) / 128;
  a.start_pos = start_pos;
  a.cache = static_cast<uint8_t*>(cache);
  a.pit = c->d_pit;
  a.spt = c->d_spt;
  a.ck = c->d_ck;
  a.tk = c->d_tk;
  a.cv = c->d_cv;
  a.tv = c->d_tv;
  a.exact = c->d_exact;
  a.status = c->d_status;
  a.pm = pm;
  a.lay = lay;
  a.g = geom_of(c);
  const dim3 grid((n_tokens + 127) / 128 + 1, kv_heads, batch);
  quantize_kernel<D><<<grid, kThreads, quant_smem_bytes<D>(), st>>>(a);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ECUDA;
}

// ---------------------------------------------------------------- decode

constexpr int kDThreads = 128;
constexpr int kMaxG = 16;

// q~ = Pi q and (with QJL) q_s = S q, one CTA of 4 D threads per (query head, batch).
template <int D>
__global__ void __launch_bounds__(4 * D) prologue_kernel(const float* __restrict__ q, const float* __restrict__ pit,
                                                         const float* __restrict__ st, float* __restrict__ qr,
                                                         float* __restrict__ qs, int q_heads, int m) {
  constexpr int KQ = D / 4;
  __shared__ float sq[D];
  __shared__ float s_a[4][D], s_s[4][D];
  const size_t row = (size_t)blockIdx.y * q_heads + blockIdx.x;
  const int j = threadIdx.x % D, part = threadIdx.x / D;
  if (part == 0) sq[j] = q[row * D + j];
  __syncthreads();
  float acc = 0.f, s = 0.f;
#pragma unroll
  for (int kk = 0; kk < KQ; ++kk) {
    const int k = part * KQ + kk;
    acc = fmaf(pit[(size_t)k * D + j], sq[k], acc);        // Pi[j][k] q[k]
    if (m > 0) s = fmaf(st[(size_t)k * D + j], sq[k], s);  // S[j][k] q[k]
  }
  s_a[part][j] = acc;
  s_s[part][j] = s;
  __syncthreads();
  if (part == 0) {
    qr[row * D + j] = (s_a[0][j] + s_a[1][j]) + (s_a[2][j] + s_a[3][j]);
    qs[row * D + j] = (s_s[0][j] + s_s[1][j]) + (s_s[2][j] + s_s[3][j]);
  }
}

struct DArgs {
  const float* qr;
  const float* qs;
  const uint8_t* cache;
  const int32_t* seq_lens;
  float* logits;
  float* part;          // [B][Hq][splits][2 + D]
  const float* ck;
  const float* cv;
  int* status;
  PageMap pm;
  float sparse_v;       // Sparse V threshold (0: dense)
  int q_heads, kv_heads, group, max_tokens, pages_per_seq, splits, pages_per_split;
  Geom g;
};

// One CTA per (split, KV head, batch): thread = token slot for the scores, = coordinate for PV.
template <int D>
__global__ void __launch_bounds__(kDThreads) split_kernel(DArgs a) {
  constexpr int KW = D / 32, CPT = (D + kDThreads - 1) / kDThreads;
  const Geom g = a.g;
  const int LK = 1 << g.kb, LV = 1 << g.vb, SW = g.m / 32;
  __shared__ float s_qr[kMaxG][D];
  __shared__ float s_qs[kMaxG][D];
  __shared__ float s_p[kMaxG][128];
  __shared__ float s_nv[128];
  __shared__ int s_keep[128];   // some head keeps the position's value (Sparse V)
  __shared__ float s_m[kMaxG], s_l[kMaxG], s_alpha[kMaxG];
  __shared__ float s_ck[32], s_cv[32];

  const int tid = threadIdx.x;
  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int G = a.group;
  int seq_len = a.seq_lens[b];
  if (seq_len > a.max_tokens || seq_len < 0) {
    if (tid == 0 && split == 0 && kvh == 0) atomicOr(a.status, kFlagBounds);
    seq_len = seq_len < 0 ? 0 : a.max_tokens;
  }
  const int h0 = kvh * G;
  for (int e = tid; e < G * D; e += kDThreads) {
    const int hh = e / D, j = e % D;
    const size_t row = (size_t)b * a.q_heads + h0 + hh;
    s_qr[hh][j] = a.qr[row * D + j];
    s_qs[hh][j] = a.qs[row * D + j];
  }
  if (tid < LK) s_ck[tid] = a.ck[tid];
  if (tid < LV) s_cv[tid] = a.cv[tid];
  if (tid < kMaxG) {
    s_m[tid] = -INFINITY;
    s_l[tid] = 0.f;
  }
  float o[kMaxG][CPT];
#pragma unroll
  for (int hh = 0; hh < kMaxG; ++hh)
#pragma unroll
    for (int u = 0; u < CPT; ++u) o[hh][u] = 0.f;
  __syncthreads();

  const float qjl_scale = g.m > 0 ? 1.2533141373155002512f / (float)g.m : 0.f;   // sqrt(pi/2) / m
  const float inv_sqrt_d = 1.0f / sqrtf((float)D);
  const bool sparse = a.sparse_v > 0.f;   // Sparse V bookkeeping only when a threshold is set
  const size_t seq = (size_t)b * a.kv_heads + kvh;
  const int p0 = split * a.pages_per_split;
  const int p1 = min(p0 + a.pages_per_split, a.pages_per_seq);

  for (int p = p0; p < p1; ++p) {
    if (p * 128 >= seq_len) break;
    const uint8_t* pg = a.cache + a.pm.index((int)seq, a.kv_heads, a.pages_per_seq, p, a.status) * g.bytes;
    const uint32_t* kc = reinterpret_cast<const uint32_t*>(pg + g.off_kcodes);
    const uint32_t* sg = reinterpret_cast<const uint32_t*>(pg + g.off_signs);
    const float* nk = reinterpret_cast<const float*>(pg + g.off_nk);
    const float* gm = reinterpret_cast<const float*>(pg + g.off_gamma);
    const uint32_t* vc = reinterpret_cast<const uint32_t*>(pg + g.off_vcodes);
    const float* nv = reinterpret_cast<const float*>(pg + g.off_nv);
    const int nvalid = min(128, seq_len - p * 128);

    // ---- scores: thread = slot ----
    const int t = tid;
    const bool valid = t < nvalid;
    float n = 0.f, gmm = 0.f;
    if (valid) {
      n = nk[t];
      if (g.m > 0) gmm = gm[t];
    }
    s_nv[t] = valid ? nv[t] : 0.f;
    if (sparse) s_keep[t] = 0;
    for (int hc = 0; hc < G; hc += 4) {
      float am[4] = {0.f, 0.f, 0.f, 0.f}, aq[4] = {0.f, 0.f, 0.f, 0.f};
      if (valid) {
        for (int w = 0; w < KW; ++w) {
          uint32_t planes[kMaxPlanes];
#pragma unroll
          for (int q = 0; q < kMaxPlanes; ++q) planes[q] = q < g.kb ? kc[((size_t)q * 128 + t) * KW + w] : 0u;
          const uint32_t sw = g.m > 0 ? sg[(size_t)t * SW + w] : 0u;
#pragma unroll 4
          for (int bit = 0; bit < 32; ++bit) {
            const int j = coord_of<D>(w, bit);
            int idx = 0;
#pragma unroll
            for (int q = 0; q < kMaxPlanes; ++q) idx |= (int)((planes[q] >> bit) & 1u) << q;
            const float cval = s_ck[idx];
            const bool pos = (sw >> bit) & 1u;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              if (hc + u < G) {
                am[u] = fmaf(s_qr[hc + u][j], cval, am[u]);
                const float qv = s_qs[hc + u][j];
                aq[u] += pos ? qv : -qv;
              }
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (hc + u < G) {
          const float lg = (n * am[u] + gmm * qjl_scale * aq[u]) * inv_sqrt_d;
          s_p[hc + u][t] = valid ? lg : -INFINITY;
          if (valid && a.logits)
            a.logits[((size_t)b * a.q_heads + h0 + hc + u) * a.max_tokens + (size_t)p * 128 + t] = lg;
        }
      }
    }
    __syncthreads();
    // ---- online softmax: warp w handles heads w, w+4, ... ----
    {
      const int warp = tid >> 5, lane = tid & 31;
      for (int hh = warp; hh < G; hh += kDThreads / 32) {
        float mx = -INFINITY;
        for (int i = lane; i < 128; i += 32) mx = fmaxf(mx, s_p[hh][i]);
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
        const float m_old = s_m[hh];
        const float m_new = fmaxf(m_old, mx);
        float sum = 0.f;
        for (int i = lane; i < 128; i += 32) {
          float e = (m_new == -INFINITY) ? 0.f : expf(s_p[hh][i] - m_new);
          sum += e;   // the denominator keeps every position
          if (sparse) {   // Sparse V: the value of a position below the threshold is skipped
            if (e < a.sparse_v) e = 0.f;
            else if (e > 0.f) s_keep[i] = 1;
          }
          s_p[hh][i] = e;
        }
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o2);
        if (lane == 0) {
          const float alpha = (m_old == -INFINITY) ? 0.f : expf(m_old - m_new);
          s_alpha[hh] = alpha;
          s_l[hh] = s_l[hh] * alpha + sum;
          s_m[hh] = m_new;
        }
      }
    }
    __syncthreads();
    // ---- PV in the rotated frame: thread = coordinate ----
#pragma unroll
    for (int u = 0; u < CPT; ++u) {
      const int j = tid + u * kDThreads;
      if (j < D) {
        uint32_t vw[kMaxPlanes][4];
#pragma unroll
        for (int q = 0; q < kMaxPlanes; ++q)
#pragma unroll
          for (int c = 0; c < 4; ++c) vw[q][c] = q < g.vb ? vc[((size_t)q * D + j) * 4 + c] : 0u;
#pragma unroll
        for (int hh = 0; hh < kMaxG; ++hh)
          if (hh < G) o[hh][u] *= s_alpha[hh];
        auto add_slot = [&](int s) {
          int w, bit;
          slot_pos(s, w, bit);
          int idx = 0;
#pragma unroll
          for (int q = 0; q < kMaxPlanes; ++q) idx |= (int)((vw[q][w] >> bit) & 1u) << q;
          const float val = s_nv[s] * s_cv[idx];
#pragma unroll
          for (int hh = 0; hh < kMaxG; ++hh)
            if (hh < G) o[hh][u] = fmaf(s_p[hh][s], val, o[hh][u]);
        };
        if (sparse) {   // positions no head keeps are skipped (uniform over the block)
          for (int s = 0; s < nvalid; ++s)
            if (s_keep[s]) add_slot(s);
        } else {
          for (int s = 0; s < nvalid; ++s) add_slot(s);
        }
      }
    }
    __syncthreads();
  }
  // ---- partials ----
  for (int hh = 0; hh < G; ++hh) {
    float* dst = a.part + (((size_t)b * a.q_heads + h0 + hh) * a.splits + split) * (2 + D);
    if (tid == 0) {
      dst[0] = s_m[hh];
      dst[1] = s_l[hh];
    }
#pragma unroll
    for (int u = 0; u < CPT; ++u) {
      const int j = tid + u * kDThreads;
      if (j < D) dst[2 + j] = o[hh][u];
    }
  }
}

template <int D>
int launch_d(const tq_ctx* c, const float* q, int batch, int q_heads, int kv_heads, const void* cache,
             const int32_t* seq_lens, int max_tokens, float* out, float* logits, void* ws, cudaStream_t st,
             const PageMap& pm) {
  const SplitPlan sp = plan_splits(batch, kv_heads, max_tokens);
  float* qr = static_cast<float*>(ws);
  float* qs = qr + (size_t)batch * q_heads * D;
  float* part = qs + (size_t)batch * q_heads * D;
  prologue_kernel<D><<<dim3(q_heads, batch), 4 * D, 0, st>>>(q, c->d_pit, c->d_st, qr, qs, q_heads, c->m);
  DArgs a;
  a.qr = qr;
  a.qs = qs;
  a.cache = static_cast<const uint8_t*>(cache);
  a.seq_lens = seq_lens;
  a.logits = logits;
  a.part = part;
  a.ck = c->d_ck;
  a.cv = c->d_cv;
  a.status = c->d_status;
  a.q_heads = q_heads;
  a.kv_heads = kv_heads;
  a.group = q_heads / kv_heads;
  a.max_tokens = max_tokens;
  a.pages_per_seq = sp.pages;
  a.pm = pm;
  a.sparse_v = c->sparse_v;
  a.splits = sp.splits;
  a.pages_per_split = sp.pages_per_split;
  a.g = geom_of(c);
  split_kernel<D><<<dim3(sp.splits, kv_heads, batch), kDThreads, 0, st>>>(a);
  launch_combine(c, part, out, batch, q_heads, sp.splits, st);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ECUDA;
}

// ---------------------------------------------------------------- dequantize

// k^ = n Pi^T c_K[idx] (+ gamma sqrt(pi/2)/m S^T (2 sigma - 1) with QJL), v^ = n_v Pi^T c_V[idx];
// one CTA per (page, sequence), one thread per coordinate.
template <int D>
__global__ void __launch_bounds__(D) dequantize_kernel(const uint8_t* __restrict__ cache, int kv_heads, int max_tokens,
                                                       int pages_per_seq, const int32_t* __restrict__ start_pos,
                                                       int n_tokens, const float* __restrict__ pi,
                                                       const float* __restrict__ smat, const float* __restrict__ ck,
                                                       const float* __restrict__ cv, float* __restrict__ k_out,
                                                       float* __restrict__ v_out, int* status, Geom g, PageMap pm) {
  constexpr int KW = D / 32, TILE = D > 128 ? 8 : 16;
  __shared__ float s_uk[TILE][D];   // n_k c_K[idx], rotated frame
  __shared__ float s_uv[TILE][D];   // n_v c_V[idx], rotated frame
  __shared__ float s_sg[TILE][D];   // 2 sigma - 1 (m == D when present)
  __shared__ float s_gam[TILE];
  const int j = threadIdx.x;
  const int seq = blockIdx.y, b = seq / kv_heads;
  const int start = start_pos[b];
  if (start < 0 || start > max_tokens - n_tokens) {
    if (j == 0 && blockIdx.x == 0) atomicOr(status, kFlagBounds);
    return;
  }
  const int page = start / 128 + (int)blockIdx.x;
  const int lo = max(start, page * 128), hi = min(start + n_tokens, page * 128 + 128);
  if (lo >= hi) return;
  const uint8_t* pg = cache + pm.index(seq, kv_heads, pages_per_seq, page, status) * g.bytes;
  const uint32_t* kcodes = reinterpret_cast<const uint32_t*>(pg + g.off_kcodes);
  const uint32_t* signs = reinterpret_cast<const uint32_t*>(pg + g.off_signs);
  const uint32_t* vcodes = reinterpret_cast<const uint32_t*>(pg + g.off_vcodes);
  const float* nk = reinterpret_cast<const float*>(pg + g.off_nk);
  const float* gam = reinterpret_cast<const float*>(pg + g.off_gamma);
  const float* nv = reinterpret_cast<const float*>(pg + g.off_nv);
  int kw, kbit;
  coord_pos<D>(j, kw, kbit);
  const float qc = g.m > 0 ? 1.2533141373155002512f / (float)g.m : 0.f;   // sqrt(pi/2) / m

  for (int t0 = lo; t0 < hi; t0 += TILE) {
    const int nt = min(TILE, hi - t0);
    __syncthreads();   // the previous tile's operands are consumed
    for (int t = 0; t < nt; ++t) {
      const int slot = t0 + t - page * 128;
      int idx = 0;
      for (int q = 0; q < g.kb; ++q) idx |= (int)((kcodes[(q * 128 + slot) * KW + kw] >> kbit) & 1u) << q;
      s_uk[t][j] = nk[slot] * ck[idx];
      s_sg[t][j] = g.m > 0 && ((signs[slot * (g.m / 32) + kw] >> kbit) & 1u) ? 1.f : -1.f;
      int vword, vbit;
      slot_pos(slot, vword, vbit);
      int vidx = 0;
      for (int q = 0; q < g.vb; ++q) vidx |= (int)((vcodes[(q * D + j) * 4 + vword] >> vbit) & 1u) << q;
      s_uv[t][j] = nv[slot] * cv[vidx];
      if (j == 0) s_gam[t] = g.m > 0 ? gam[slot] : 0.f;
    }
    __syncthreads();
    float ak[TILE], av[TILE], aq[TILE];
#pragma unroll
    for (int t = 0; t < TILE; ++t) ak[t] = av[t] = aq[t] = 0.f;
#pragma unroll 4
    for (int k = 0; k < D; ++k) {   // (Pi^T u)_j = sum_k Pi[k][j] u_k
      const float p = pi[(size_t)k * D + j];
#pragma unroll
      for (int t = 0; t < TILE; ++t) {
        ak[t] = fmaf(p, s_uk[t][k], ak[t]);
        av[t] = fmaf(p, s_uv[t][k], av[t]);
      }
    }
    if (g.m > 0) {
#pragma unroll 4
      for (int i = 0; i < D; ++i) {   // (S^T s)_j = sum_i S[i][j] s_i
        const float sv = smat[(size_t)i * D + j];
#pragma unroll
        for (int t = 0; t < TILE; ++t) aq[t] = fmaf(sv, s_sg[t][i], aq[t]);
      }
    }
#pragma unroll
    for (int t = 0; t < TILE; ++t) {
      if (t < nt) {
        const size_t o = ((size_t)seq * n_tokens + (size_t)(t0 + t - start)) * D + j;
        if (k_out) k_out[o] = fmaf(s_gam[t] * qc, aq[t], ak[t]);
        if (v_out) v_out[o] = av[t];
      }
    }
  }
}

template <int D>
int launch_dq(const tq_ctx* c, const void* cache, int batch, int kv_heads, int max_tokens, const int32_t* start_pos,
              int n_tokens, float* k_out, float* v_out, cudaStream_t st, const PageMap& pm) {
  const dim3 grid((unsigned)((n_tokens + 127) / 128 + 1), (unsigned)(batch * kv_heads));
  dequantize_kernel<D><<<grid, D, 0, st>>>(static_cast<const uint8_t*>(cache), kv_heads, max_tokens,
                                           (max_tokens + 127) / 128, start_pos, n_tokens, c->d_pi, c->d_s, c->d_ck,
                                           c->d_cv, k_out, v_out, c->d_status, geom_of(c), pm);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ECUDA;
}

}  // namespace kv2

int prepare_kv2(const tq_ctx* c) {
  auto set = [](const void* fn, size_t bytes) {
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) == cudaSuccess;
  };
  bool ok = true;
  if (c->d == 64) ok = set((const void*)kv2::quantize_kernel<64>, kv2::quant_smem_bytes<64>());
  if (c->d == 128) ok = set((const void*)kv2::quantize_kernel<128>, kv2::quant_smem_bytes<128>());
  if (c->d == 256) ok = set((const void*)kv2::quantize_kernel<256>, kv2::quant_smem_bytes<256>());
  return ok ? TQ_OK : TQ_ECUDA;
}

int launch_quantize_kv2(const tq_ctx* c, const void* k, const void* v, int batch, int kv_heads, int n_tokens,
                        const int32_t* start_pos, void* cache, int max_tokens, const KVLayout& lay, void* stream,
                        const PageMap& pm) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (c->d == 64) return kv2::launch_q<64>(c, k, v, batch, kv_heads, n_tokens, start_pos, cache, max_tokens, st, pm, lay);
  if (c->d == 128) return kv2::launch_q<128>(c, k, v, batch, kv_heads, n_tokens, start_pos, cache, max_tokens, st, pm, lay);
  if (c->d == 256) return kv2::launch_q<256>(c, k, v, batch, kv_heads, n_tokens, start_pos, cache, max_tokens, st, pm, lay);
  return TQ_EUNSUPPORTED;
}

int launch_decode_kv2(const tq_ctx* c, const float* q, int batch, int q_heads, int kv_heads, const void* cache,
                      const int32_t* seq_lens, int max_tokens, float* out, float* logits_out, void* workspace,
                      void* stream, const PageMap& pm) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
#define TQ_D2(DD)                                                                                               \
  if (c->d == DD)                                                                                               \
    return kv2::launch_d<DD>(c, q, batch, q_heads, kv_heads, cache, seq_lens, max_tokens, out, logits_out, workspace, \
                             st, pm);
  TQ_D2(64) TQ_D2(128) TQ_D2(256)
#undef TQ_D2
  return TQ_EUNSUPPORTED;
}

int launch_dequantize_kv2(const tq_ctx* c, const void* cache, int batch, int kv_heads, int max_tokens,
                          const int32_t* start_pos, int n_tokens, float* k_out, float* v_out, void* stream,
                          const PageMap& pm) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (c->d == 64) return kv2::launch_dq<64>(c, cache, batch, kv_heads, max_tokens, start_pos, n_tokens, k_out, v_out, st, pm);
  if (c->d == 128)
    return kv2::launch_dq<128>(c, cache, batch, kv_heads, max_tokens, start_pos, n_tokens, k_out, v_out, st, pm);
  if (c->d == 256)
    return kv2::launch_dq<256>(c, cache, batch, kv_heads, max_tokens, start_pos, n_tokens, k_out, v_out, st, pm);
  return TQ_EUNSUPPORTED;
}

}  // namespace tq
