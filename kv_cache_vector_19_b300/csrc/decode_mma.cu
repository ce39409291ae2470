// Launch plan, instantiations and the split-merge kernel of the tensor-core decode path.
#include <cuda_runtime.h>

#include "decode_mma.cuh"

namespace tq {

// Balanced split of all pages of all (batch, kv head) sequences over at most `ctas` CTAs:
// every CTA takes `chunk` consecutive pages, which may span sequence boundaries.
bool plan_pages(long ctas, int batch, int kv_heads, int max_tokens, MmaPlan* p) {
  const long pm = (max_tokens + 127) / 128;
  const long total = (long)batch * kv_heads * pm;
  if (total > 0x7fffffffL || total < 1) return false;
  long grid = total < ctas ? total : ctas;
  if (grid < 1) grid = 1;
  long chunk = (total + grid - 1) / grid;
  grid = (total + chunk - 1) / chunk;
  p->pages_per_seq = (int)pm;
  p->total_pages = (int)total;
  p->chunk = (int)chunk;
  p->grid = (int)grid;
  p->slots = (int)((pm - 1) / chunk + 2);
  return true;
}

namespace dmma {

// Merges the partial records of one (query head, batch) and rotates back: out = Pi^T o~ / l.
template <int D>
__global__ void __launch_bounds__(4 * D) combine_kernel(const float* __restrict__ part, const float* __restrict__ pi,
                                                        float* __restrict__ out, int q_heads, int kv_heads, int group,
                                                        int pages_per_seq, int chunk, int slots, int grid) {
  constexpr int KQ = D / 4;
  __shared__ float s_o[D];
  __shared__ float s_r[4][D];
  __shared__ float s_w[512];
  __shared__ float s_norm;
  pdl_wait();   // the decode grid's partial records (at once when launched without the attribute)
  const int hq = blockIdx.x, b = blockIdx.y;
  const size_t row = (size_t)b * q_heads + hq;
  const int seq = b * kv_heads + hq / group, hh = hq % group;
  const int first = (int)(((long)seq * pages_per_seq) / chunk);
  const int last = min(grid - 1, (int)(((long)(seq + 1) * pages_per_seq - 1) / chunk));
  const int n = last - first + 1;
  const int j = threadIdx.x % D, qp = threadIdx.x / D;   // 4 D threads: coordinate, quarter
  auto rec = [&](int s) { return part + (((size_t)seq * slots + s) * group + hh) * (2 + D); };
  if (threadIdx.x == 0) {
    float mx = -INFINITY;
    for (int s = 0; s < n; ++s) mx = fmaxf(mx, rec(s)[0]);
    float l = 0.f;
    for (int s = 0; s < n; ++s) {
      float m = rec(s)[0];
      float w = (m == -INFINITY) ? 0.f : __expf(m - mx);
      s_w[s] = w;
      l += w * rec(s)[1];
    }
    s_norm = l > 0.f ? 1.f / l : 0.f;
  }
  __syncthreads();
  if (qp == 0) {
    float acc = 0.f;
    for (int s = 0; s < n; ++s) {
      float w = s_w[s];
      if (w != 0.f) acc = fmaf(w, rec(s)[2 + j], acc);
    }
    s_o[j] = acc * s_norm;
  }
  __syncthreads();
  // out_j = sum_k Pi[k][j] o~[k], each quarter of k by one quarter of the threads with all of
  // its loads in flight (Pi is usually out of L2 after the cache scan)
  float r = 0.f;
#pragma unroll
  for (int kk = 0; kk < KQ; ++kk) {
    const int k = qp * KQ + kk;
    r = fmaf(pi[(size_t)k * D + j], s_o[k], r);
  }
  s_r[qp][j] = r;
  __syncthreads();
  if (qp == 0) out[row * D + j] = (s_r[0][j] + s_r[1][j]) + (s_r[2][j] + s_r[3][j]);
}

namespace {

template <int D, int BITS, int NGRP>
int prepare_one() {
  using C = Cfg<D, BITS, NGRP>;
  if constexpr (!C::SUPPORTED) {
    return TQ_OK;
  } else {
    const bool ok = cudaFuncSetAttribute(decode_mma_kernel<D, BITS, NGRP, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) == cudaSuccess &&
                    cudaFuncSetAttribute(decode_mma_kernel<D, BITS, NGRP, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) == cudaSuccess;
    return ok ? TQ_OK : TQ_ECUDA;
  }
}

template <int D, int BITS, int NGRP>
bool plan_one(const tq_ctx* c, int batch, int kv_heads, int max_tokens, MmaPlan* p) {
  using C = Cfg<D, BITS, NGRP>;
  if constexpr (!C::SUPPORTED) {
    return false;
  } else {
    return plan_pages((long)c->num_sms * C::MINB, batch, kv_heads, max_tokens, p);
  }
}

template <int D, int BITS, int NGRP>
int launch_one(const tq_ctx* c, const MmaPlan& pl, const float* q, int batch, int q_heads, int kv_heads,
               const void* cache, const int32_t* seq_lens, int max_tokens, float* out, float* logits, void* ws,
               cudaStream_t st, const PageMap& pm) {
  using C = Cfg<D, BITS, NGRP>;
  if constexpr (!C::SUPPORTED) {
    return TQ_EUNSUPPORTED;
  } else {
    float* qr = static_cast<float*>(ws);
    float* qs = qr + (size_t)batch * q_heads * D;
    float* part = qs + (size_t)batch * q_heads * D;
    launch_prologue(c, q, batch, q_heads, qr, qs, st);
    Params a;
    a.qr = qr;
    a.qs = qs;
    a.cache = static_cast<const uint8_t*>(cache);
    a.seq_lens = seq_lens;
    a.logits = logits;
    a.part = part;
    a.alpha_k = c->d_alpha_k;
    a.alpha_v = c->d_alpha_v;
    a.status = c->d_status;
    a.asum_k = c->asum_k;
    a.asum_v = c->asum_v;
    a.batch = batch;
    a.q_heads = q_heads;
    a.kv_heads = kv_heads;
    a.group = q_heads / kv_heads;
    a.max_tokens = max_tokens;
    a.pages_per_seq = pl.pages_per_seq;
    a.chunk = pl.chunk;
    a.slots = pl.slots;
    a.total_pages = pl.total_pages;
    if (pm.table)
      decode_mma_kernel<D, BITS, NGRP, true><<<pl.grid, kThreads, C::SMEM, st>>>(a, pm, c->sparse_v);
    else
      decode_mma_kernel<D, BITS, NGRP, false><<<pl.grid, kThreads, C::SMEM, st>>>(a, pm, c->sparse_v);
    combine_kernel<D><<<dim3(q_heads, batch), 4 * D, 0, st>>>(part, c->d_pi, out, q_heads, kv_heads, a.group,
                                                          pl.pages_per_seq, pl.chunk, pl.slots, pl.grid);
    return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ECUDA;
  }
}

int ngrp_of(int group) { return group <= 4 ? 1 : group <= 8 ? 2 : group <= 16 ? 4 : 0; }

}  // namespace
}  // namespace dmma

#define TQ_FOR_ALL(X)                                                                                     \
  X(64, 2, 1) X(64, 2, 2) X(64, 2, 4) X(64, 3, 1) X(64, 3, 2) X(64, 3, 4) X(64, 4, 1) X(64, 4, 2)           \
  X(64, 4, 4) X(64, 5, 1) X(64, 5, 2) X(64, 5, 4) X(128, 2, 1) X(128, 2, 2) X(128, 2, 4) X(128, 3, 1)        \
  X(128, 3, 2) X(128, 3, 4) X(128, 4, 1) X(128, 4, 2) X(128, 4, 4) X(128, 5, 1) X(128, 5, 2) X(128, 5, 4)    \
  X(256, 2, 1) X(256, 2, 2) X(256, 2, 4) X(256, 3, 1) X(256, 3, 2) X(256, 3, 4) X(256, 4, 1) X(256, 4, 2)    \
  X(256, 4, 4) X(256, 5, 1) X(256, 5, 2) X(256, 5, 4)

int prepare_decode_mma(const tq_ctx* c) {
  int rc = TQ_OK;
#define TQ_P(DD, BB, NG) \
  if (rc == TQ_OK && c->d == DD && c->bits == BB) rc = dmma::prepare_one<DD, BB, NG>();
  TQ_FOR_ALL(TQ_P)
#undef TQ_P
  return rc;
}

bool plan_decode_mma(const tq_ctx* c, int batch, int q_heads, int kv_heads, int max_tokens, MmaPlan* p) {
  if (q_heads % kv_heads != 0) return false;
  const int ng = dmma::ngrp_of(q_heads / kv_heads);
#define TQ_PL(DD, BB, NG) \
  if (c->d == DD && c->bits == BB && ng == NG) return dmma::plan_one<DD, BB, NG>(c, batch, kv_heads, max_tokens, p);
  TQ_FOR_ALL(TQ_PL)
#undef TQ_PL
  return false;
}

int launch_decode_mma(const tq_ctx* c, const MmaPlan& pl, const float* q, int batch, int q_heads, int kv_heads,
                      const void* cache, const int32_t* seq_lens, int max_tokens, float* out, float* logits_out,
                      void* workspace, void* stream, const PageMap& pm) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int ng = dmma::ngrp_of(q_heads / kv_heads);
#define TQ_L(DD, BB, NG)                                                                                    \
  if (c->d == DD && c->bits == BB && ng == NG)                                                              \
    return dmma::launch_one<DD, BB, NG>(c, pl, q, batch, q_heads, kv_heads, cache, seq_lens, max_tokens, out, \
                                        logits_out, workspace, st, pm);
  TQ_FOR_ALL(TQ_L)
#undef TQ_L
  return TQ_EUNSUPPORTED;
}

size_t decode_mma_workspace(const tq_ctx* c, const MmaPlan& pl, int batch, int q_heads, int kv_heads) {
  const size_t rows = (size_t)batch * q_heads;
  const size_t n_seq = (size_t)batch * kv_heads;
  const size_t g = (size_t)(q_heads / kv_heads);
  return (rows * c->d * 2 + n_seq * pl.slots * g * (2 + c->d)) * sizeof(float);
}

}  // namespace tq

// ---------------------------------------------------------------- tcgen05 decode (d = 128)
#include "decode_tc.cuh"

namespace tq {
namespace {

template <int BITS, int GP>
int tc_prepare_one() {
  using C = dtc::Cfg<BITS, GP>;
  if constexpr (!C::SUPPORTED) {
    return TQ_OK;
  } else {
    const bool ok = cudaFuncSetAttribute(dtc::decode_tc_kernel<BITS, GP, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) == cudaSuccess &&
                    cudaFuncSetAttribute(dtc::decode_tc_kernel<BITS, GP, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) == cudaSuccess;
    return ok ? TQ_OK : TQ_ECUDA;
  }
}

int tc_gp(int group) { return group <= 4 ? 4 : group <= 8 ? 8 : group <= 16 ? 16 : 0; }

template <int BITS, int GP>
int tc_launch_one(const tq_ctx* c, const MmaPlan& pl, const float* q, int batch, int q_heads, int kv_heads,
                  const void* cache, const int32_t* seq_lens, int max_tokens, float* out, float* logits, void* ws,
                  cudaStream_t st, const PageMap& pm) {
  using C = dtc::Cfg<BITS, GP>;
  if constexpr (!C::SUPPORTED) {
    return TQ_EUNSUPPORTED;
  } else {
    constexpr int D = 128;
    float* qr = static_cast<float*>(ws);
    float* qs = qr + (size_t)batch * q_heads * D;
    float* part = qs + (size_t)batch * q_heads * D;
    launch_prologue(c, q, batch, q_heads, qr, qs, st);
    dmma::Params a;
    a.qr = qr;
    a.qs = qs;
    a.cache = static_cast<const uint8_t*>(cache);
    a.seq_lens = seq_lens;
    a.logits = logits;
    a.part = part;
    a.alpha_k = c->d_alpha_k;
    a.alpha_v = c->d_alpha_v;
    a.status = c->d_status;
    a.asum_k = c->asum_k;
    a.asum_v = c->asum_v;
    a.batch = batch;
    a.q_heads = q_heads;
    a.kv_heads = kv_heads;
    a.group = q_heads / kv_heads;
    a.max_tokens = max_tokens;
    a.pages_per_seq = pl.pages_per_seq;
    a.chunk = pl.chunk;
    a.slots = pl.slots;
    a.total_pages = pl.total_pages;
    if (pm.table)
      dtc::decode_tc_kernel<BITS, GP, true><<<pl.grid, C::THREADS, C::SMEM, st>>>(a, pm, c->sparse_v);
    else
      dtc::decode_tc_kernel<BITS, GP, false><<<pl.grid, C::THREADS, C::SMEM, st>>>(a, pm, c->sparse_v);
    dmma::combine_kernel<D><<<dim3(q_heads, batch), 4 * D, 0, st>>>(part, c->d_pi, out, q_heads, kv_heads, a.group,
                                                                pl.pages_per_seq, pl.chunk, pl.slots, pl.grid);
    return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ECUDA;
  }
}

}  // namespace

bool decode_tc_supported(const tq_ctx* c, int q_heads, int kv_heads) {
  if (c->d != 128 || q_heads % kv_heads != 0) return false;
  const int gp = tc_gp(q_heads / kv_heads);
  if (gp == 0) return false;
#define TQ_S(BB, GG) \
  if (c->bits == BB && gp == GG) return dtc::Cfg<BB, GG>::SUPPORTED;
  TQ_S(2, 4) TQ_S(2, 8) TQ_S(2, 16) TQ_S(3, 4) TQ_S(3, 8) TQ_S(3, 16)
#undef TQ_S
  return false;
}

bool plan_decode_tc(const tq_ctx* c, int batch, int q_heads, int kv_heads, int max_tokens, MmaPlan* p) {
  return decode_tc_supported(c, q_heads, kv_heads) && plan_pages(c->num_sms, batch, kv_heads, max_tokens, p);
}

bool decode_tc_preferred(const tq_ctx* c, int q_heads, int kv_heads) {
  return decode_tc_supported(c, q_heads, kv_heads);
}

int prepare_decode_tc(const tq_ctx* c) {
  if (c->d != 128) return TQ_OK;
  int rc = TQ_OK;
#define TQ_P(BB, GG) \
  if (rc == TQ_OK && c->bits == BB) rc = tc_prepare_one<BB, GG>();
  TQ_P(2, 4) TQ_P(2, 8) TQ_P(2, 16) TQ_P(3, 4) TQ_P(3, 8) TQ_P(3, 16)
#undef TQ_P
  return rc;
}

int launch_decode_tc(const tq_ctx* c, const MmaPlan& pl, const float* q, int batch, int q_heads, int kv_heads,
                     const void* cache, const int32_t* seq_lens, int max_tokens, float* out, float* logits_out,
                     void* workspace, void* stream, const PageMap& pm) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int gp = tc_gp(q_heads / kv_heads);
#define TQ_L(BB, GG)                                                                                         \
  if (c->bits == BB && gp == GG)                                                                             \
    return tc_launch_one<BB, GG>(c, pl, q, batch, q_heads, kv_heads, cache, seq_lens, max_tokens, out, logits_out, \
                                 workspace, st, pm);
  TQ_L(2, 4) TQ_L(2, 8) TQ_L(2, 16) TQ_L(3, 4) TQ_L(3, 8) TQ_L(3, 16)
#undef TQ_L
  return TQ_EUNSUPPORTED;
}

}  // namespace tq

// ---------------------------------------------------------------- tcgen05 decode, 4-bit operands (d = 128)
#include "decode_f4.cuh"

namespace tq {
namespace {

template <int BITS, int GP, int SPLIT>
int f4_prepare_one() {
  using C = dtf::Cfg<BITS, GP>;
  if constexpr (!C::SUPPORTED) {
    return TQ_OK;
  } else {
    const bool ok = cudaFuncSetAttribute(dtf::decode_f4_kernel<BITS, GP, false, SPLIT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) == cudaSuccess &&
                    cudaFuncSetAttribute(dtf::decode_f4_kernel<BITS, GP, true, SPLIT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM) == cudaSuccess;
    return ok ? TQ_OK : TQ_ECUDA;
  }
}

// Query heads of a KV head per kernel pass (gp, padded) and passes per KV head (split).  With
// 4-bit codes the kernel's tensor memory holds two query heads, so a KV head with 4 or 8 runs as
// 2 or 4 virtual KV heads of two query heads each, which read the same pages; with 2 or 3 bits a
// KV head with 16 query heads runs as 4 virtual KV heads of four.
struct F4Shape {
  int gp, split;
};
F4Shape f4_shape(int bits, int group) {
  if (bits == 4) {
    if (group <= 2) return {2, 1};
    if (group == 4) return {2, 2};
    if (group == 8) return {2, 4};
    return {0, 0};
  }
  if (group == 16) return {4, 4};
  return {group <= 4 ? 4 : group <= 8 ? 8 : 0, 1};
}

template <int BITS, int GP, int SPLIT>
int f4_launch_one(const tq_ctx* c, const MmaPlan& pl, const float* q, int batch, int q_heads, int kv_heads,
                  const void* cache, const int32_t* seq_lens, int max_tokens, float* out, float* logits, void* ws,
                  cudaStream_t st, const PageMap& pm) {
  using C = dtf::Cfg<BITS, GP>;
  if constexpr (!C::SUPPORTED) {
    return TQ_EUNSUPPORTED;
  } else {
    constexpr int D = 128;
    const int kv_virtual = kv_heads * SPLIT;   // the plan is over the virtual KV heads
    float* qr = static_cast<float*>(ws);
    float* qs = qr + (size_t)batch * q_heads * D;
    float* part = qs + (size_t)batch * q_heads * D;
    launch_prologue(c, q, batch, q_heads, qr, qs, st);
    dmma::Params a;
    a.qr = qr;
    a.qs = qs;
    a.cache = static_cast<const uint8_t*>(cache);
    a.seq_lens = seq_lens;
    a.logits = logits;
    a.part = part;
    a.alpha_k = c->d_alpha_k;
    a.alpha_v = c->d_alpha_v;
    a.status = c->d_status;
    a.asum_k = c->asum_k;
    a.asum_v = c->asum_v;
    a.batch = batch;
    a.q_heads = q_heads;
    a.kv_heads = kv_virtual;
    a.group = q_heads / kv_virtual;
    a.max_tokens = max_tokens;
    a.pages_per_seq = pl.pages_per_seq;
    a.chunk = pl.chunk;
    a.slots = pl.slots;
    a.total_pages = pl.total_pages;
    // The decode and the combine are launched with programmatic stream serialization: the
    // decode grid starts its set-up and first page loads while the prologue runs (it reads
    // nothing the prologue writes before its pdl_wait, and the prologue itself starts only
    // after all earlier work), and the combine grid launches as the decode's CTAs finish.
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(pl.grid);
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e =
        pm.table ? cudaLaunchKernelEx(&cfg, dtf::decode_f4_kernel<BITS, GP, true, SPLIT>, a, pm, c->sparse_v)
                 : cudaLaunchKernelEx(&cfg, dtf::decode_f4_kernel<BITS, GP, false, SPLIT>, a, pm, c->sparse_v);
    if (e != cudaSuccess) return TQ_ECUDA;
    cfg.gridDim = dim3(q_heads, batch);
    cfg.blockDim = dim3(4 * D);
    cfg.dynamicSmemBytes = 0;
    e = cudaLaunchKernelEx(&cfg, dmma::combine_kernel<D>, (const float*)part, (const float*)c->d_pi, out, q_heads,
                           kv_virtual, a.group, pl.pages_per_seq, pl.chunk, pl.slots, pl.grid);
    return e == cudaSuccess && cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ECUDA;
  }
}

}  // namespace

bool decode_f4_supported(const tq_ctx* c, int q_heads, int kv_heads) {
  if (c->d != 128 || q_heads % kv_heads != 0) return false;
  const F4Shape sh = f4_shape(c->bits, q_heads / kv_heads);
  if (sh.gp == 0) return false;
#define TQ_S(BB, GG) \
  if (c->bits == BB && sh.gp == GG) return dtf::Cfg<BB, GG>::SUPPORTED;
  TQ_S(2, 4) TQ_S(2, 8) TQ_S(3, 4) TQ_S(3, 8) TQ_S(4, 2)
#undef TQ_S
  return false;
}

bool plan_decode_f4(const tq_ctx* c, int batch, int q_heads, int kv_heads, int max_tokens, MmaPlan* p) {
  if (!decode_f4_supported(c, q_heads, kv_heads)) return false;
  const F4Shape sh = f4_shape(c->bits, q_heads / kv_heads);
  return plan_pages(c->num_sms, batch, kv_heads * sh.split, max_tokens, p);
}

int prepare_decode_f4(const tq_ctx* c) {
  if (c->d != 128) return TQ_OK;
  int rc = TQ_OK;
#define TQ_P(BB, GG, SS) \
  if (rc == TQ_OK && c->bits == BB) rc = f4_prepare_one<BB, GG, SS>();
  TQ_P(2, 4, 1) TQ_P(2, 8, 1) TQ_P(3, 4, 1) TQ_P(3, 8, 1) TQ_P(2, 4, 4) TQ_P(3, 4, 4)
  TQ_P(4, 2, 1) TQ_P(4, 2, 2) TQ_P(4, 2, 4)
#undef TQ_P
  return rc;
}

int launch_decode_f4(const tq_ctx* c, const MmaPlan& pl, const float* q, int batch, int q_heads, int kv_heads,
                     const void* cache, const int32_t* seq_lens, int max_tokens, float* out, float* logits_out,
                     void* workspace, void* stream, const PageMap& pm) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const F4Shape sh = f4_shape(c->bits, q_heads / kv_heads);
#define TQ_L(BB, GG, SS)                                                                                       \
  if (c->bits == BB && sh.gp == GG && sh.split == SS)                                                         \
    return f4_launch_one<BB, GG, SS>(c, pl, q, batch, q_heads, kv_heads, cache, seq_lens, max_tokens, out,   \
                                     logits_out, workspace, st, pm);
  TQ_L(2, 4, 1) TQ_L(2, 8, 1) TQ_L(3, 4, 1) TQ_L(3, 8, 1) TQ_L(2, 4, 4) TQ_L(3, 4, 4)
  TQ_L(4, 2, 1) TQ_L(4, 2, 2) TQ_L(4, 2, 4)
#undef TQ_L
  return TQ_EUNSUPPORTED;
}

}  // namespace tq
