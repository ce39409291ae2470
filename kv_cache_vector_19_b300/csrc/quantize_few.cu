// tq_quantize_kv for calls that write only a few tokens per sequence (decode-time appends):
// one CTA per new (batch, kv head, token) vector pair, one thread per coordinate, fp32.
//
// [BLOG] "Технология TurboQuant и её применение с локальными LLM", section 1.2, for a
// single vector: y = Pi x, Lloyd-Max code of y / ||x|| per coordinate (b-1 bits for the
// key, b for the value); for the key the residual in the rotated frame, Pi r = y - n c[idx],
// is projected by S' = S Pi^T (S r = S' Pi r) and only sign(S r) and ||r|| are kept.
// The page-tile kernels process a whole 128-slot tile per page touched, so a one-token
// append costs as much as a full page; here the two d x d products are matrix-vector
// products against Pi^T and S'^T (L2-resident after the first CTA), and the slot is written
// in place: its key-code, sign and norm words belong to it alone, and its bit of each value
// word (a value word spans 32 slots) is set with an atomic.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "dev_common.cuh"
#include "exact.cuh"
#include "layout.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

// Sum over the CTA's NT threads (every thread gets the total).
template <int NT>
__device__ __forceinline__ float block_sum(float v, float* s_red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();   // s_red free
  if (lane == 0) s_red[warp] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) t += s_red[w];
  return t;
}

template <int D, int BITS>
__global__ void __launch_bounds__(4 * D) quantize_few_kernel(const __nv_bfloat16* __restrict__ k,
                                                         const __nv_bfloat16* __restrict__ v, int kv_heads,
                                                         int n_tokens, int max_tokens, int pages_per_seq,
                                                         const int32_t* __restrict__ start_pos, uint8_t* cache,
                                                         const float* __restrict__ pit, const float* __restrict__ spt,
                                                         const float* __restrict__ ck, const float* __restrict__ tk,
                                                         const float* __restrict__ cv, const float* __restrict__ tv,
                                                         const float* __restrict__ exact_tabs, int* status,
                                                         PageMap pm, KVLayout lay) {
  using PL = PageLayout<D, BITS>;
  constexpr int M = D, BK = BITS - 1, BV = BITS, LK = 1 << BK, LV = 1 << BV;
  constexpr int NT = 4 * D;   // 4 D threads: coordinate j and quarter qp for the per-coordinate steps
  // the two d x d products: thread (cg, pp) sums the KP rows of part pp for the four outputs
  // 4 cg .. 4 cg + 3 with 16-byte loads; the 16 parts are added in shared memory
  constexpr int NC = D / 4, NPART = 16, KP = D / NPART;
  __shared__ float s_xk[D], s_xv[D], s_r[D];
  __shared__ float4 s_pa[NPART][NC], s_pb[NPART][NC];   // partial sums of the parts
  __shared__ float s_red[NT / 32];
  __shared__ uint32_t s_words[BK * PL::KW + PL::SW];   // the slot's key-code and sign words
  __shared__ int s_code[D];                            // the key's codes (exact sign decisions)
  const int j = threadIdx.x % D, qp = threadIdx.x / D;
  const int t = blockIdx.x, seq = blockIdx.y, b = seq / kv_heads;
  const int start = start_pos[b];
  if (start < 0 || start > max_tokens - n_tokens) {
    if (threadIdx.x == 0 && t == 0) atomicOr(status, kFlagBounds);
    return;
  }
  // Every fetch that does not wait for a result starts now, so that the chain below meets
  // one memory latency instead of one per step: S'^T and the near tables into L2 (the
  // projection and the near tests come later), the books into shared memory, and this
  // thread's rows of Pi^T and S'^T (four columns each, 16-byte loads) into registers
  // (head_dim <= 128; at 256 the thread budget is 64 registers and the rows are loaded in the
  // products' loops).
  __shared__ float s_tk[LK], s_tv[LV], s_ck[LK];
  if (threadIdx.x == 0) {
    dev::prefetch_l2(spt, (uint32_t)(D * M * sizeof(float)));
    dev::prefetch_l2(exact_tabs + exact::tables_floats(D) - (6 * 32 + 2 * 64), (6 * 32 + 2 * 64) * sizeof(float));
  }
  if (threadIdx.x < LK - 1) s_tk[threadIdx.x] = tk[threadIdx.x];
  if (threadIdx.x < LV - 1) s_tv[threadIdx.x] = tv[threadIdx.x];
  if (threadIdx.x < LK) s_ck[threadIdx.x] = ck[threadIdx.x];
  constexpr bool kColumnInRegs = D <= 128;
  const int cg = threadIdx.x % NC, pp = threadIdx.x / NC;
  const float4* pit4 = reinterpret_cast<const float4*>(pit);
  const float4* spt4 = reinterpret_cast<const float4*>(spt);
  float4 pcol[kColumnInRegs ? KP : 1], scol[kColumnInRegs ? KP : 1];
  if constexpr (kColumnInRegs) {
#pragma unroll
    for (int kk = 0; kk < KP; ++kk) {
      pcol[kk] = __ldg(pit4 + (size_t)(pp * KP + kk) * NC + cg);   // Pi^T[c][4 cg .. 4 cg + 3]
      scol[kk] = __ldg(spt4 + (size_t)(pp * KP + kk) * (M / 4) + cg);
    }
  }
  const int pos = start + t, page = pos >> 7, slot = pos & 127;
  uint8_t* pg = cache + pm.index(seq, kv_heads, pages_per_seq, page, status) * PL::bytes;
  const int hkv = seq - b * kv_heads;
  const size_t krow = (size_t)(b * lay.kb + hkv * lay.kh + t * lay.kt);   // this token's key row
  const size_t vrow = (size_t)(b * lay.vb + hkv * lay.vh + t * lay.vt);
  float xk = 0.f, xv = 0.f;
  if (qp == 0) {
    xk = __bfloat162float(k[krow + j]);
    xv = __bfloat162float(v[vrow + j]);
    s_xk[j] = xk;
    s_xv[j] = xv;
    if (j < BK * PL::KW + PL::SW) s_words[j] = 0u;
  }
  const float nk = sqrtf(block_sum<NT>(xk * xk, s_red));   // also orders the s_xk / s_xv stores
  const float nv = sqrtf(block_sum<NT>(xv * xv, s_red));
  // y_j = (Pi x)_j = sum_c Pi^T[c][j] x_c
  {
    float4 pa = make_float4(0.f, 0.f, 0.f, 0.f), pb = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int kk = 0; kk < KP; ++kk) {
      const int c = pp * KP + kk;
      float4 p4;
      if constexpr (kColumnInRegs) p4 = pcol[kk];
      else p4 = __ldg(pit4 + (size_t)c * NC + cg);
      const float a = s_xk[c], w = s_xv[c];
      pa = make_float4(fmaf(p4.x, a, pa.x), fmaf(p4.y, a, pa.y), fmaf(p4.z, a, pa.z), fmaf(p4.w, a, pa.w));
      pb = make_float4(fmaf(p4.x, w, pb.x), fmaf(p4.y, w, pb.y), fmaf(p4.z, w, pb.z), fmaf(p4.w, w, pb.w));
    }
    s_pa[pp][cg] = pa;
    s_pb[pp][cg] = pb;
  }
  __syncthreads();
  auto part_sum = [&](const float4 (*sp)[NC]) {   // sum over the parts for coordinate j
    const float* f = reinterpret_cast<const float*>(&sp[0][0]) + j;
    float r = 0.f;
#pragma unroll
    for (int q = 0; q < NPART; ++q) r += f[q * D];
    return r;
  };
  const float yk = part_sum(s_pa);
  const float yv = part_sum(s_pb);
  // Lloyd-Max codes by boundary count (a value on a boundary takes the upper code)
  const float ik = nk > 0.f ? 1.f / nk : 0.f, iv = nv > 0.f ? 1.f / nv : 0.f;
  const float uk = yk * ik, uv = yv * iv;
  int idx = 0, vidx = 0;
#pragma unroll
  for (int q = 0; q < LK - 1; ++q) idx += uk >= s_tk[q] ? 1 : 0;
#pragma unroll
  for (int q = 0; q < LV - 1; ++q) vidx += uv >= s_tv[q] ? 1 : 0;
  // codes next to a boundary are taken again exactly (exact.cuh), each warp for its own 32
  // coordinates (the warps of the four quarters repeat the same decisions)
  const exact::Tables T = exact::tables(exact_tabs, D);
  const int lane = threadIdx.x & 31;
  {
    const bool nk_near = nk > 0.f && fabsf(uk - T.nkt[2 * idx]) > T.nkt[2 * idx + 1];
    const bool nv_near = nv > 0.f && fabsf(uv - T.nvt[2 * vidx]) > T.nvt[2 * vidx + 1];
    uint32_t ev = __ballot_sync(0xffffffffu, nk_near);
    if (ev) {
      float x[D / 32];
      exact::load_row<D>(k + krow, lane, x);
      const exact::F2 n = exact::norm<D>(x);
      while (ev) {
        const int L = __ffs(ev) - 1;
        ev &= ev - 1;
        const int r2 = exact::code<D>(x, n, T.pih, T.pil, __shfl_sync(0xffffffffu, j, L), T.tkh, T.tkl, LK - 1, lane);
        if (lane == L) idx = r2;
      }
    }
    ev = __ballot_sync(0xffffffffu, nv_near);
    if (ev) {
      float x[D / 32];
      exact::load_row<D>(v + vrow, lane, x);
      const exact::F2 n = exact::norm<D>(x);
      while (ev) {
        const int L = __ffs(ev) - 1;
        ev &= ev - 1;
        const int r2 = exact::code<D>(x, n, T.pih, T.pil, __shfl_sync(0xffffffffu, j, L), T.tvh, T.tvl, LV - 1, lane);
        if (lane == L) vidx = r2;
      }
    }
  }
  const float r = yk - nk * s_ck[idx];   // residual in the rotated frame
  if (qp == 0) {
    s_r[j] = r;
    s_code[j] = idx;
  }
  const float gamma = sqrtf(block_sum<NT>(qp == 0 ? r * r : 0.f, s_red));
  // z_i = (S' Pi r)_i = sum_c S'^T[c][i] (Pi r)_c (m == d), by parts as y
  {
    float4 pz = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int kk = 0; kk < KP; ++kk) {
      const int c = pp * KP + kk;
      float4 s4;
      if constexpr (kColumnInRegs) s4 = scol[kk];
      else s4 = __ldg(spt4 + (size_t)c * (M / 4) + cg);
      const float rc = s_r[c];
      pz = make_float4(fmaf(s4.x, rc, pz.x), fmaf(s4.y, rc, pz.y), fmaf(s4.z, rc, pz.z), fmaf(s4.w, rc, pz.w));
    }
    __syncthreads();   // s_pa reads (y) done
    s_pa[pp][cg] = pz;
  }
  __syncthreads();
  const float z = part_sum(s_pa);
  if (qp != 0) return;   // the rest is per coordinate
  // projections next to zero: exact sign
  bool sgn = z >= 0.f;
  {
    uint32_t ev = __ballot_sync(0xffffffffu, fabsf(z) < exact::kDeltaSign * gamma);
    if (ev) {
      float x[D / 32];
      int codes[D / 32];
      exact::load_row<D>(k + krow, lane, x);
#pragma unroll
      for (int q = 0; q < D / 32; ++q) codes[q] = s_code[lane * (D / 32) + q];
      const exact::F2 n = exact::norm<D>(x);
      while (ev) {
        const int L = __ffs(ev) - 1;
        ev &= ev - 1;
        const bool e2 = exact::sign<D>(x, n, codes, T.sh, T.sl, T.qh, T.ql, T.ckh, T.ckl,
                                       __shfl_sync(0xffffffffu, j, L), lane);
        if (lane == L) sgn = e2;
      }
    }
  }
  // the slot's words: coordinate j of each key-code plane and of the sign plane
  int w, bit;
  coord_pos<D>(j, w, bit);
#pragma unroll
  for (int q = 0; q < BK; ++q)
    if ((idx >> q) & 1) atomicOr(&s_words[q * PL::KW + w], 1u << bit);
  if (sgn) atomicOr(&s_words[BK * PL::KW + w], 1u << bit);
  asm volatile("bar.sync 1, %0;" ::"r"(D) : "memory");   // the D remaining threads (warps 0 .. D/32-1)
  uint32_t* kc = reinterpret_cast<uint32_t*>(pg + PL::off_kcodes);
  uint32_t* sg = reinterpret_cast<uint32_t*>(pg + PL::off_signs);
  if (j < BK * PL::KW) kc[((j / PL::KW) * 128 + slot) * PL::KW + (j % PL::KW)] = s_words[j];
  else if (j < BK * PL::KW + PL::SW) sg[slot * PL::SW + (j - BK * PL::KW)] = s_words[j];
  if (j == 0) {
    reinterpret_cast<float*>(pg + PL::off_nk)[slot] = nk;
    reinterpret_cast<float*>(pg + PL::off_gamma)[slot] = gamma;
    reinterpret_cast<float*>(pg + PL::off_nv)[slot] = nv;
  }
  // value code of coordinate j: one bit in each plane's word over this slot's group of 32
  int vw, vb;
  slot_pos(slot, vw, vb);
  uint32_t* vc = reinterpret_cast<uint32_t*>(pg + PL::off_vcodes);
#pragma unroll
  for (int q = 0; q < BV; ++q) {
    uint32_t* word = vc + ((size_t)q * D + j) * 4 + vw;
    if ((vidx >> q) & 1) atomicOr(word, 1u << vb);
    else atomicAnd(word, ~(1u << vb));
  }
}

template <int D, int BITS>
int launch_one(const tq_ctx* c, const void* k, const void* v, int batch, int kv_heads, int n_tokens,
               const int32_t* start_pos, void* cache, int max_tokens, cudaStream_t st, const PageMap& pm,
               const KVLayout& lay) {
  const dim3 grid((unsigned)n_tokens, (unsigned)(batch * kv_heads));
  quantize_few_kernel<D, BITS><<<grid, 4 * D, 0, st>>>(
      static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v), kv_heads, n_tokens, max_tokens,
      (max_tokens + 127) / 128, start_pos, static_cast<uint8_t*>(cache), c->d_pit, c->d_spt, c->d_ck, c->d_tk,
      c->d_cv, c->d_tv, c->d_exact, c->d_status, pm, lay);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ECUDA;
}

}  // namespace

int launch_quantize_few(const tq_ctx* c, const void* k, const void* v, int batch, int kv_heads, int n_tokens,
                        const int32_t* start_pos, void* cache, int max_tokens, const KVLayout& lay, void* stream,
                        const PageMap& pm) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
#define TQ_QF(DD, BB) \
  if (c->d == DD && c->bits == BB) \
    return launch_one<DD, BB>(c, k, v, batch, kv_heads, n_tokens, start_pos, cache, max_tokens, st, pm, lay);
  TQ_QF(64, 2) TQ_QF(64, 3) TQ_QF(64, 4) TQ_QF(64, 5) TQ_QF(128, 2) TQ_QF(128, 3) TQ_QF(128, 4) TQ_QF(128, 5)
  TQ_QF(256, 2) TQ_QF(256, 3) TQ_QF(256, 4) TQ_QF(256, 5)
#undef TQ_QF
  return TQ_EUNSUPPORTED;
}

}  // namespace tq
