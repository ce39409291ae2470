// tq_dequantize_kv: cached vectors rebuilt from their pages in the original frame.
//
// [BLOG] "Технология TurboQuant и её применение с локальными LLM", section 1.2: a vector is
// restored from its codes as n Pi^T c[idx] (stage 1), and for keys the stage-2 sketch adds
// gamma sqrt(pi/2)/m S^T (2 sigma - 1), the unbiased estimate of the residual's inner products.
// This is the explicit reconstruction the decode kernels never materialise; it serves error
// statistics, inspection and tests.  CUDA cores, fp32: one CTA per (page, sequence), one
// thread per coordinate, tokens in tiles so that each matrix element loaded serves a tile.
#include <cuda_runtime.h>

#include <cstdint>

#include "layout.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

template <int D, int BITS>
__global__ void __launch_bounds__(D) dequantize_kernel(const uint8_t* __restrict__ cache, int kv_heads, int max_tokens,
                                                       int pages_per_seq, const int32_t* __restrict__ start_pos,
                                                       int n_tokens, const float* __restrict__ pi,
                                                       const float* __restrict__ smat, const float* __restrict__ ck,
                                                       const float* __restrict__ cv, float* __restrict__ k_out,
                                                       float* __restrict__ v_out, int* status, PageMap pm) {
  using PL = PageLayout<D, BITS>;
  constexpr int M = D, BK = BITS - 1, BV = BITS;
  constexpr int TILE = D > 128 ? 8 : 16;
  __shared__ float s_uk[TILE][D];   // n_k c_K[idx], rotated frame
  __shared__ float s_uv[TILE][D];   // n_v c_V[idx], rotated frame
  __shared__ float s_sg[TILE][M];   // 2 sigma - 1
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
  const uint8_t* pg = cache + pm.index(seq, kv_heads, pages_per_seq, page, status) * PL::bytes;
  const uint32_t* kcodes = reinterpret_cast<const uint32_t*>(pg + PL::off_kcodes);
  const uint32_t* signs = reinterpret_cast<const uint32_t*>(pg + PL::off_signs);
  const uint32_t* vcodes = reinterpret_cast<const uint32_t*>(pg + PL::off_vcodes);
  const float* nk = reinterpret_cast<const float*>(pg + PL::off_nk);
  const float* gam = reinterpret_cast<const float*>(pg + PL::off_gamma);
  const float* nv = reinterpret_cast<const float*>(pg + PL::off_nv);
  int kw, kbit;
  coord_pos<D>(j, kw, kbit);   // coordinate j in a key-code word; sign i = j sits alike (m == d)
  const float qc = 1.2533141373155002512f / (float)M;   // sqrt(pi/2) / m

  for (int t0 = lo; t0 < hi; t0 += TILE) {
    const int nt = min(TILE, hi - t0);
    __syncthreads();   // the previous tile's operands are consumed
    for (int t = 0; t < nt; ++t) {
      const int slot = t0 + t - page * 128;
      int idx = 0;
#pragma unroll
      for (int q = 0; q < BK; ++q) idx |= (int)((kcodes[(q * 128 + slot) * PL::KW + kw] >> kbit) & 1u) << q;
      s_uk[t][j] = nk[slot] * ck[idx];
      s_sg[t][j] = ((signs[slot * PL::SW + kw] >> kbit) & 1u) ? 1.f : -1.f;
      int vword, vbit;
      slot_pos(slot, vword, vbit);
      int vidx = 0;
#pragma unroll
      for (int q = 0; q < BV; ++q) vidx |= (int)((vcodes[(q * D + j) * 4 + vword] >> vbit) & 1u) << q;
      s_uv[t][j] = nv[slot] * cv[vidx];
      if (j == 0) s_gam[t] = gam[slot];
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
#pragma unroll 4
    for (int i = 0; i < M; ++i) {   // (S^T s)_j = sum_i S[i][j] s_i
      const float sv = smat[(size_t)i * D + j];
#pragma unroll
      for (int t = 0; t < TILE; ++t) aq[t] = fmaf(sv, s_sg[t][i], aq[t]);
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

template <int D, int BITS>
int launch_one(const tq_ctx* c, const void* cache, int batch, int kv_heads, int max_tokens, const int32_t* start_pos,
               int n_tokens, float* k_out, float* v_out, cudaStream_t st, const PageMap& pm) {
  const dim3 grid((unsigned)((n_tokens + 127) / 128 + 1), (unsigned)(batch * kv_heads));
  dequantize_kernel<D, BITS><<<grid, D, 0, st>>>(static_cast<const uint8_t*>(cache), kv_heads, max_tokens,
                                                 (max_tokens + 127) / 128, start_pos, n_tokens, c->d_pi, c->d_s,
                                                 c->d_ck, c->d_cv, k_out, v_out, c->d_status, pm);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ECUDA;
}

}  // namespace

int launch_dequantize(const tq_ctx* c, const void* cache, int batch, int kv_heads, int max_tokens,
                      const int32_t* start_pos, int n_tokens, float* k_out, float* v_out, void* stream,
                      const PageMap& pm) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
#define TQ_DQ(DD, BB) \
  if (c->d == DD && c->bits == BB)   \
    return launch_one<DD, BB>(c, cache, batch, kv_heads, max_tokens, start_pos, n_tokens, k_out, v_out, st, pm);
  TQ_DQ(64, 2) TQ_DQ(64, 3) TQ_DQ(64, 4) TQ_DQ(64, 5) TQ_DQ(128, 2) TQ_DQ(128, 3) TQ_DQ(128, 4) TQ_DQ(128, 5)
  TQ_DQ(256, 2) TQ_DQ(256, 3) TQ_DQ(256, 4) TQ_DQ(256, 5)
#undef TQ_DQ
  return TQ_EUNSUPPORTED;
}

}  // namespace tq
