// tq_quantize_kv, CUDA-core version: one CTA per (page touched, kv head, batch).
//
// [BLOG] "Технология TurboQuant и её применение с локальными LLM", section 1.2:
//   stage 1: y = Pi x (random orthogonal rotation), per-coordinate Lloyd-Max code of y / ||x||
//            with b-1 bits (keys) or b bits (values);
//   stage 2 (keys): r = x - DEQUANT(idx); sign(S r) and ||r||_2 are stored.
// The residual is projected in the rotated frame: S r = (S Pi^T)(Pi r) and
// Pi r = y - n c[idx], so one d x d matrix S' = S Pi^T replaces a second rotation.
//
// Each CTA handles the slots of one page that this call writes (up to 128), in halves of
// 64 rows: load bf16 rows -> fp32 norms -> Y = X Pi^T -> codes, R = Y - n c[idx], gamma
// -> Z = R S'^T -> bit-pack.  Value codes are staged as bytes for the whole page and packed
// at the end, because a value-code word spans 32 slots spread over the page.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "exact.cuh"
#include "layout.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kThreads = 256;
constexpr int kRows = 64;

struct QArgs {
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  int kv_heads, n_tokens, max_tokens, pages_per_seq;
  const int32_t* start_pos;
  uint8_t* cache;
  const float* pit;   // [D][D] Pi^T
  const float* spt;   // [D][M] S'^T
  const float* ck;
  const float* tk;
  const float* cv;
  const float* tv;
  const float* exact;   // exact-decision tables
  int* status;
  PageMap pm;
  KVLayout lay;         // element strides of k and v over (batch, KV head, token)
};

// C[64][N] (row stride N+1) = A[64][D] (row stride D+1) * Bt[D][N]; 256 threads,
// each owns rows ty + 16 i (i < 4) and columns tx*4 + 64 cc + (0..3).
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
    float a[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = A[(ty + 16 * i) * (D + 1) + kk];
#pragma unroll
    for (int cc = 0; cc < NC; ++cc) {
      float4 bv = __ldg(reinterpret_cast<const float4*>(Bt + (size_t)kk * N + tx * 4 + 64 * cc));
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[i][cc][0] = fmaf(a[i], bv.x, acc[i][cc][0]);
        acc[i][cc][1] = fmaf(a[i], bv.y, acc[i][cc][1]);
        acc[i][cc][2] = fmaf(a[i], bv.z, acc[i][cc][2]);
        acc[i][cc][3] = fmaf(a[i], bv.w, acc[i][cc][3]);
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

// Loads up to 64 bf16 rows (slots s0 .. s0+63 of the page) into fp32 smem; rows outside
// [lo, hi) are zero.  Then one warp per row computes the fp32 norm.
template <int D>
__device__ __forceinline__ void load_rows(const __nv_bfloat16* __restrict__ src_seq, int64_t ts, int page, int start,
                                          int s0, int lo, int hi, float* xs, float* nrm) {
  const int tid = threadIdx.x;
  for (int e = tid; e < kRows * (D / 8); e += kThreads) {
    int row = e / (D / 8), ch = e % (D / 8);
    int slot = s0 + row;
    float f[8];
    if (slot >= lo && slot < hi) {
      long tok = (long)page * 128 + slot - start;
      uint4 raw = __ldg(reinterpret_cast<const uint4*>(src_seq + tok * ts) + ch);
      const __nv_bfloat16* hv = reinterpret_cast<const __nv_bfloat16*>(&raw);
#pragma unroll
      for (int u = 0; u < 8; ++u) f[u] = __bfloat162float(hv[u]);
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
      float x = xs[row * (D + 1) + j];
      s = fmaf(x, x, s);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) nrm[row] = sqrtf(s);
  }
  __syncthreads();
}

// idx = #{k : yhat >= t_k}
template <int L>
__device__ __forceinline__ int encode(float yhat, const float* t) {
  int idx = 0;
#pragma unroll
  for (int q = 0; q < L - 1; ++q) idx += (yhat >= t[q]) ? 1 : 0;
  return idx;
}

// Warp-collective: the codes of this warp's coordinates that the fast value put next to a
// boundary, taken again exactly (exact.cuh); returns this thread's (possibly new) code.
template <int D>
__device__ __forceinline__ int resolve_codes(bool near, int idx, int row, int j, const __nv_bfloat16* src_seq,
                                             int64_t ts, int page, int start, int s0, const float* th, const float* tl, int nb,
                                             const exact::Tables& T, int lane) {
  uint32_t ev = __ballot_sync(0xffffffffu, near);
  while (ev) {
    const int L = __ffs(ev) - 1;
    ev &= ev - 1;
    const int rowL = __shfl_sync(0xffffffffu, row, L), jL = __shfl_sync(0xffffffffu, j, L);
    float x[D / 32];
    exact::load_row<D>(src_seq + ((long)page * 128 + s0 + rowL - start) * ts, lane, x);
    const exact::F2 n = exact::norm<D>(x);
    const int r = exact::code<D>(x, n, T.pih, T.pil, jL, th, tl, nb, lane);
    if (lane == L) idx = r;
  }
  return idx;
}

template <int D, int BITS>
__global__ void __launch_bounds__(kThreads) quantize_simt_kernel(QArgs a) {
  using PL = PageLayout<D, BITS>;
  constexpr int BK = PL::BK, BV = PL::BV, LK = 1 << BK, LV = 1 << BV;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  float* xs = reinterpret_cast<float*>(smem_raw);                 // [64][D+1]  X, later Z
  float* ys = xs + kRows * (D + 1);                                // [64][D+1]  Y, later R
  float* nrm = ys + kRows * (D + 1);                               // [64]
  float* gam = nrm + kRows;                                        // [64]
  float* s_ck = gam + kRows;
  float* s_tk = s_ck + LK;
  float* s_cv = s_tk + LK;
  float* s_tv = s_cv + LV;
  float2* s_nk = reinterpret_cast<float2*>(s_tv + LV);              // near tables, one float2 per cell
  float2* s_nv = s_nk + LK;
  uint8_t* kcode = reinterpret_cast<uint8_t*>(s_nv + LV);          // [64][D]
  uint8_t* vcode = kcode + kRows * D;                              // [128][D]

  const int tid = threadIdx.x;
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

  for (int i = tid; i < LK; i += kThreads) s_ck[i] = a.ck[i];
  for (int i = tid; i < LK - 1; i += kThreads) s_tk[i] = a.tk[i];
  for (int i = tid; i < LV; i += kThreads) s_cv[i] = a.cv[i];
  for (int i = tid; i < LV - 1; i += kThreads) s_tv[i] = a.tv[i];
  const exact::Tables T = exact::tables(a.exact, D);
  for (int i = tid; i < 2 * LK; i += kThreads) reinterpret_cast<float*>(s_nk)[i] = T.nkt[i];
  for (int i = tid; i < 2 * LV; i += kThreads) reinterpret_cast<float*>(s_nv)[i] = T.nvt[i];
  const int lane = tid & 31;

  const size_t seq = (size_t)b * a.kv_heads + h;
  uint8_t* pg = a.cache + a.pm.index((int)seq, a.kv_heads, a.pages_per_seq, page, a.status) * PL::bytes;
  uint32_t* g_kc = reinterpret_cast<uint32_t*>(pg + PL::off_kcodes);
  uint32_t* g_sg = reinterpret_cast<uint32_t*>(pg + PL::off_signs);
  float* g_nk = reinterpret_cast<float*>(pg + PL::off_nk);
  float* g_gm = reinterpret_cast<float*>(pg + PL::off_gamma);
  uint32_t* g_vc = reinterpret_cast<uint32_t*>(pg + PL::off_vcodes);
  float* g_nv = reinterpret_cast<float*>(pg + PL::off_nv);
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
      int row = e / D, j = e % D;
      float n = nrm[row];
      float y = ys[row * (D + 1) + j];
      float yh = n > 0.f ? y / n : 0.f;
      int idx = encode<LK>(yh, s_tk);
      const bool near = n > 0.f && fabsf(yh - s_nk[idx].x) > s_nk[idx].y;
      idx = resolve_codes<D>(near, idx, row, j, kseq, a.lay.kt, page, start, s0, T.tkh, T.tkl, LK - 1, T, lane);
      kcode[row * D + j] = (uint8_t)idx;
      ys[row * (D + 1) + j] = y - n * s_ck[idx];                   // r_rot = Pi r
    }
    __syncthreads();
    {
      const int warp = tid >> 5, lane = tid & 31;
      for (int row = warp; row < kRows; row += kThreads / 32) {
        float s = 0.f;
        for (int j = lane; j < D; j += 32) {
          float r = ys[row * (D + 1) + j];
          s = fmaf(r, r, s);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (lane == 0) gam[row] = sqrtf(s);
      }
    }
    gemm64<D, D>(ys, a.spt, xs);                                     // Z = R S'^T
    __syncthreads();
    // projections next to zero: exact sign (stored back into Z as +-1)
    for (int e = tid; e < kRows * D; e += kThreads) {
      const int row = e / D, i = e % D;
      const float z = xs[row * (D + 1) + i];
      const bool near = fabsf(z) < exact::kDeltaSign * gam[row];
      uint32_t ev = __ballot_sync(0xffffffffu, near);
      while (ev) {
        const int L = __ffs(ev) - 1;
        ev &= ev - 1;
        const int rowL = __shfl_sync(0xffffffffu, row, L), iL = __shfl_sync(0xffffffffu, i, L);
        float x[D / 32];
        int codes[D / 32];
        exact::load_row<D>(kseq + ((long)page * 128 + s0 + rowL - start) * a.lay.kt, lane, x);
#pragma unroll
        for (int q = 0; q < D / 32; ++q) codes[q] = kcode[rowL * D + lane * (D / 32) + q];
        const exact::F2 n = exact::norm<D>(x);
        const bool sg = exact::sign<D>(x, n, codes, T.sh, T.sl, T.qh, T.ql, T.ckh, T.ckl, iL, lane);
        if (lane == L) xs[row * (D + 1) + i] = sg ? 1.f : -1.f;
      }
    }
    __syncthreads();
    // bit-pack key codes (BK planes) and signs, one word per thread-iteration
    constexpr int WPR = D / 32;
    for (int e = tid; e < kRows * (BK + 1) * WPR; e += kThreads) {
      int row = e / ((BK + 1) * WPR), rem = e % ((BK + 1) * WPR);
      int plane = rem / WPR, w = rem % WPR;
      int slot = s0 + row;
      if (slot < lo || slot >= hi) continue;
      uint32_t word = 0;
#pragma unroll 8
      for (int bit = 0; bit < 32; ++bit) {
        int j = coord_of<D>(w, bit);
        uint32_t v = plane < BK ? (uint32_t)((kcode[row * D + j] >> plane) & 1)
                                : (uint32_t)(xs[row * (D + 1) + j] >= 0.f);
        word |= v << bit;
      }
      if (plane < BK)
        g_kc[((size_t)plane * 128 + slot) * WPR + w] = word;
      else
        g_sg[(size_t)slot * WPR + w] = word;
    }
    for (int row = tid; row < kRows; row += kThreads) {
      int slot = s0 + row;
      if (slot >= lo && slot < hi) {
        g_nk[slot] = nrm[row];
        g_gm[slot] = gam[row];
      }
    }
    __syncthreads();
    // ---------------- values ----------------
    load_rows<D>(vseq, a.lay.vt, page, start, s0, lo, hi, xs, nrm);
    gemm64<D, D>(xs, a.pit, ys);
    __syncthreads();
    for (int e = tid; e < kRows * D; e += kThreads) {
      int row = e / D, j = e % D;
      float n = nrm[row];
      float yh = n > 0.f ? ys[row * (D + 1) + j] / n : 0.f;
      int idx = encode<LV>(yh, s_tv);
      const bool near = n > 0.f && fabsf(yh - s_nv[idx].x) > s_nv[idx].y;
      idx = resolve_codes<D>(near, idx, row, j, vseq, a.lay.vt, page, start, s0, T.tvh, T.tvl, LV - 1, T, lane);
      vcode[(s0 + row) * D + j] = (uint8_t)idx;
    }
    for (int row = tid; row < kRows; row += kThreads) {
      int slot = s0 + row;
      if (slot >= lo && slot < hi) g_nv[slot] = nrm[row];
    }
    __syncthreads();
  }
  // value-code words: [plane][coord][4], each over 32 slots of the page
  for (int e = tid; e < BV * D * 4; e += kThreads) {
    int plane = e / (D * 4), rem = e % (D * 4), j = rem >> 2, c = rem & 3;
    uint32_t word = 0, mask = 0;
#pragma unroll 8
    for (int bit = 0; bit < 32; ++bit) {
      int slot = slot_of(c, bit);
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
  return (size_t)2 * kRows * (D + 1) * 4 + 2 * kRows * 4 + (32 + 32 + 32 + 32 + 64 + 64) * 4 + (size_t)kRows * D +
         (size_t)128 * D;
}

template <int D, int BITS>
int prepare_q() {
  return cudaFuncSetAttribute(quantize_simt_kernel<D, BITS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)quant_smem_bytes<D>()) == cudaSuccess
             ? TQ_OK
             : TQ_ECUDA;
}

template <int D, int BITS>
int launch_q(const tq_ctx* c, const void* k, const void* v, int batch, int kv_heads, int n_tokens,
             const int32_t* start_pos, void* cache, int max_tokens, cudaStream_t st, const PageMap& pm,
             const KVLayout& lay) {
  constexpr size_t smem = quant_smem_bytes<D>();
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
  dim3 grid((n_tokens + 127) / 128 + 1, kv_heads, batch);
  quantize_simt_kernel<D, BITS><<<grid, kThreads, smem, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ECUDA;
}

}  // namespace
}  // namespace tq

int prepare_quantize_simt(const tq_ctx* c) {
#define TQ_P(DD, BB) \
  if (c->d == DD && c->bits == BB) return tq::prepare_q<DD, BB>();
  TQ_P(64, 2) TQ_P(64, 3) TQ_P(64, 4) TQ_P(64, 5)
  TQ_P(128, 2) TQ_P(128, 3) TQ_P(128, 4) TQ_P(128, 5)
  TQ_P(256, 2) TQ_P(256, 3) TQ_P(256, 4) TQ_P(256, 5)
#undef TQ_P
  return TQ_EUNSUPPORTED;
}

int launch_quantize_simt(const tq_ctx* c, const void* k, const void* v, int batch, int kv_heads,
                         int n_tokens, const int32_t* start_pos, void* cache, int max_tokens,
                         const tq::KVLayout& lay, void* stream, const tq::PageMap& pm) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
#define TQ_Q(DD, BB)                                                                              \
  if (c->d == DD && c->bits == BB)                                                                \
    return tq::launch_q<DD, BB>(c, k, v, batch, kv_heads, n_tokens, start_pos, cache, max_tokens, st, pm, lay);
  TQ_Q(64, 2) TQ_Q(64, 3) TQ_Q(64, 4) TQ_Q(64, 5)
  TQ_Q(128, 2) TQ_Q(128, 3) TQ_Q(128, 4) TQ_Q(128, 5)
  TQ_Q(256, 2) TQ_Q(256, 3) TQ_Q(256, 4) TQ_Q(256, 5)
#undef TQ_Q
  return TQ_EUNSUPPORTED;
}
