// tq_attn_decode, CUDA-core version (split-T flash-decoding over the compressed pages).
//
// Score of cached key t for query q (rotated frame, q~ = Pi q, q_s = S q):
//   logit_t = ( n_t <q~, c_K[idx_t]> + gamma_t sqrt(pi/2)/m <q_s, 2 sigma_t - 1> ) / sqrt(d)
// ([BLOG] "Технология TurboQuant ...", section 1.2: ||r||_2 is the reconstruction scale of the
// sign sketch; for s ~ N(0, I), E[<s,q> sign<s,r>] = sqrt(2/pi) <q,r> / ||r||, hence sqrt(pi/2).)
// Values are accumulated in the rotated frame, o~ = sum_t p_t n_v,t c_V[idx_t], and rotated
// back once: out = Pi^T o~ / sum_t p_t.
//
// Kernels: prologue (q~, q_s per query head) -> split (one CTA per (split, kv head, batch),
// one thread per token slot of a page, online softmax over its pages) -> combine (LSE merge of
// the splits, then Pi^T).
#include <cuda_runtime.h>

#include <cmath>

#include "layout.cuh"
#include "tq_internal.h"

namespace tq {

SplitPlan plan_splits(int batch, int kv_heads, int max_tokens) {
  SplitPlan p;
  p.pages = (max_tokens + 127) / 128;
  if (p.pages < 1) p.pages = 1;
  long units = (long)batch * kv_heads;
  long target = 2L * 148;                       // about two CTAs per SM
  int splits = (int)((target + units - 1) / units);
  if (splits < 1) splits = 1;
  if (splits > p.pages) splits = p.pages;
  p.pages_per_split = (p.pages + splits - 1) / splits;
  p.splits = (p.pages + p.pages_per_split - 1) / p.pages_per_split;
  return p;
}

namespace {

constexpr int kThreads = 128;
constexpr int kMaxG = 16;

// q~ = Pi q and q_s = S q, one CTA of 4 D threads per (query head, batch).  Thread (c, p)
// sums the D / 16 rows k of part p for the four outputs 4c .. 4c + 3, reading Pi^T and S^T with
// 16-byte loads (the first rows' loads issued before q arrives: the matrices are usually out of
// L2 when a decode starts), and the 16 parts are added in shared memory.
template <int D>
__global__ void __launch_bounds__(4 * D) prologue_kernel(const float* __restrict__ q, const float* __restrict__ pit,
                                                         const float* __restrict__ st, float* __restrict__ qr,
                                                         float* __restrict__ qs, int q_heads) {
  constexpr int NC = D / 4, NP = 16, KP = D / NP, CH = KP < 8 ? KP : 8;   // rows per part, per chunk
  pdl_trigger();   // the decode grid may start its set-up; it waits for q~, q_s at pdl_wait
  __shared__ float sq[D];
  __shared__ float4 s_a[NP][NC], s_s[NP][NC];
  const size_t row = (size_t)blockIdx.y * q_heads + blockIdx.x;
  const int c = threadIdx.x % NC, p = threadIdx.x / NC;
  const float4* pi4 = reinterpret_cast<const float4*>(pit);
  const float4* st4 = reinterpret_cast<const float4*>(st);
  float4 pa[CH], ps[CH];
#pragma unroll
  for (int kk = 0; kk < CH; ++kk) {
    const int k = p * KP + kk;
    pa[kk] = __ldg(pi4 + (size_t)k * NC + c);   // Pi[4c .. 4c+3][k]
    ps[kk] = __ldg(st4 + (size_t)k * NC + c);   // S[4c .. 4c+3][k]
  }
  if (threadIdx.x < D) sq[threadIdx.x] = q[row * D + threadIdx.x];
  __syncthreads();
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f), t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int k0 = 0; k0 < KP; k0 += CH) {
    if (k0 > 0) {
#pragma unroll
      for (int kk = 0; kk < CH; ++kk) {
        const int k = p * KP + k0 + kk;
        pa[kk] = __ldg(pi4 + (size_t)k * NC + c);
        ps[kk] = __ldg(st4 + (size_t)k * NC + c);
      }
    }
#pragma unroll
    for (int kk = 0; kk < CH; ++kk) {
      const float x = sq[p * KP + k0 + kk];
      a.x = fmaf(pa[kk].x, x, a.x);
      a.y = fmaf(pa[kk].y, x, a.y);
      a.z = fmaf(pa[kk].z, x, a.z);
      a.w = fmaf(pa[kk].w, x, a.w);
      t.x = fmaf(ps[kk].x, x, t.x);
      t.y = fmaf(ps[kk].y, x, t.y);
      t.z = fmaf(ps[kk].z, x, t.z);
      t.w = fmaf(ps[kk].w, x, t.w);
    }
  }
  s_a[p][c] = a;
  s_s[p][c] = t;
  __syncthreads();
  if (threadIdx.x < D) {
    const int j = threadIdx.x;
    const float* fa = reinterpret_cast<const float*>(&s_a[0][0]) + j;   // part pp at fa[pp * D]
    const float* fs = reinterpret_cast<const float*>(&s_s[0][0]) + j;
    float r = 0.f, u = 0.f;
#pragma unroll
    for (int pp = 0; pp < NP; ++pp) {
      r += fa[pp * D];
      u += fs[pp * D];
    }
    qr[row * D + j] = r;
    qs[row * D + j] = u;
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
};

// PAGED: pages through the block table (its own instantiation, so that the contiguous kernel
// carries no table code)
template <int D, int BITS, bool PAGED>
__global__ void __launch_bounds__(kThreads) split_kernel(DArgs a) {
  using PL = PageLayout<D, BITS>;
  constexpr int BK = PL::BK, BV = PL::BV, LK = 1 << BK, LV = 1 << BV, KW = PL::KW;
  constexpr int CPT = (D + kThreads - 1) / kThreads;   // coordinates per thread in PV
  __shared__ float s_qr[kMaxG][D];
  __shared__ float s_qs[kMaxG][D];
  __shared__ float s_p[kMaxG][128];
  __shared__ float s_nv[128];
  __shared__ int s_keep[128];   // some head keeps the position's value (Sparse V)
  __shared__ float s_m[kMaxG], s_l[kMaxG], s_alpha[kMaxG];
  __shared__ float s_ck[32], s_cv[32];

  const int tid = threadIdx.x;
  const int split = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int G = a.group;
  int seq_len = a.seq_lens[b];
  if (seq_len > a.max_tokens || seq_len < 0) {
    if (tid == 0 && split == 0 && g == 0) atomicOr(a.status, kFlagBounds);
    seq_len = seq_len < 0 ? 0 : a.max_tokens;
  }
  const int h0 = g * G;
  for (int e = tid; e < G * D; e += kThreads) {
    int hh = e / D, j = e % D;
    size_t row = (size_t)b * a.q_heads + h0 + hh;
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

  const float qjl_scale = 1.2533141373155002512f / (float)PL::M;   // sqrt(pi/2) / m
  const float inv_sqrt_d = 1.0f / sqrtf((float)D);
  const bool sparse = a.sparse_v > 0.f;   // Sparse V bookkeeping only when a threshold is set
  const size_t seq = (size_t)b * a.kv_heads + g;
  const int p0 = split * a.pages_per_split;
  const int p1 = min(p0 + a.pages_per_split, a.pages_per_seq);

  for (int p = p0; p < p1; ++p) {
    if (p * 128 >= seq_len) break;
    const uint8_t* pg;
    if constexpr (PAGED) pg = a.cache + a.pm.index((int)seq, a.kv_heads, a.pages_per_seq, p, a.status) * PL::bytes;
    else pg = a.cache + (seq * a.pages_per_seq + p) * (size_t)PL::bytes;
    const uint32_t* kc = reinterpret_cast<const uint32_t*>(pg + PL::off_kcodes);
    const uint32_t* sg = reinterpret_cast<const uint32_t*>(pg + PL::off_signs);
    const float* nk = reinterpret_cast<const float*>(pg + PL::off_nk);
    const float* gm = reinterpret_cast<const float*>(pg + PL::off_gamma);
    const uint32_t* vc = reinterpret_cast<const uint32_t*>(pg + PL::off_vcodes);
    const float* nv = reinterpret_cast<const float*>(pg + PL::off_nv);
    const int nvalid = min(128, seq_len - p * 128);

    // ---- scores: thread = slot ----
    const int t = tid;
    const bool valid = t < nvalid;
    float n = 0.f, gmm = 0.f;
    if (valid) {
      n = nk[t];
      gmm = gm[t];
    }
    s_nv[t] = valid ? nv[t] : 0.f;
    if (sparse) s_keep[t] = 0;
    for (int hc = 0; hc < G; hc += 4) {
      float am[4] = {0.f, 0.f, 0.f, 0.f}, aq[4] = {0.f, 0.f, 0.f, 0.f};
      if (valid) {
        for (int w = 0; w < KW; ++w) {
          uint32_t planes[BK];
#pragma unroll
          for (int q = 0; q < BK; ++q) planes[q] = kc[((size_t)q * 128 + t) * KW + w];
          uint32_t sw = sg[(size_t)t * KW + w];
#pragma unroll 4
          for (int bit = 0; bit < 32; ++bit) {
            int j = coord_of<D>(w, bit);
            int idx = 0;
#pragma unroll
            for (int q = 0; q < BK; ++q) idx |= ((planes[q] >> bit) & 1u) << q;
            float cval = s_ck[idx];
            bool pos = (sw >> bit) & 1u;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              if (hc + u < G) {
                am[u] = fmaf(s_qr[hc + u][j], cval, am[u]);
                float qv = s_qs[hc + u][j];
                aq[u] += pos ? qv : -qv;
              }
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        if (hc + u < G) {
          float lg = (n * am[u] + gmm * qjl_scale * aq[u]) * inv_sqrt_d;
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
      for (int hh = warp; hh < G; hh += kThreads / 32) {
        float mx = -INFINITY;
        for (int i = lane; i < 128; i += 32) mx = fmaxf(mx, s_p[hh][i]);
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
        float m_old = s_m[hh];
        float m_new = fmaxf(m_old, mx);
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
          float alpha = (m_old == -INFINITY) ? 0.f : expf(m_old - m_new);
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
      const int j = tid + u * kThreads;
      if (j < D) {
        uint32_t vw[BV][4];
#pragma unroll
        for (int q = 0; q < BV; ++q)
#pragma unroll
          for (int c = 0; c < 4; ++c) vw[q][c] = vc[((size_t)q * D + j) * 4 + c];
#pragma unroll
        for (int hh = 0; hh < kMaxG; ++hh)
          if (hh < G) o[hh][u] *= s_alpha[hh];
        auto add_slot = [&](int s) {
          int w, bit;
          slot_pos(s, w, bit);
          int idx = 0;
#pragma unroll
          for (int q = 0; q < BV; ++q) idx |= ((vw[q][w] >> bit) & 1u) << q;
          float val = s_nv[s] * s_cv[idx];
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
      int j = tid + u * kThreads;
      if (j < D) dst[2 + j] = o[hh][u];
    }
  }
}

// Merges the splits of one (query head, batch) and rotates back: out = Pi^T o~ / l.
template <int D>
__global__ void __launch_bounds__(D) combine_kernel(const float* __restrict__ part, const float* __restrict__ pi,
                                                    float* __restrict__ out, int q_heads, int splits) {
  __shared__ float s_o[D];
  __shared__ float s_w[1024];
  __shared__ float s_norm;
  const size_t row = (size_t)blockIdx.y * q_heads + blockIdx.x;
  const float* pr = part + row * splits * (2 + D);
  const int j = threadIdx.x;
  if (j == 0) {
    float mx = -INFINITY;
    for (int s = 0; s < splits; ++s) mx = fmaxf(mx, pr[(size_t)s * (2 + D)]);
    float l = 0.f;
    for (int s = 0; s < splits; ++s) {
      float m = pr[(size_t)s * (2 + D)];
      float w = (m == -INFINITY) ? 0.f : expf(m - mx);
      s_w[s] = w;
      l += w * pr[(size_t)s * (2 + D) + 1];
    }
    s_norm = l > 0.f ? 1.f / l : 0.f;
  }
  __syncthreads();
  float acc = 0.f;
  for (int s = 0; s < splits; ++s) {
    float w = s_w[s];
    if (w != 0.f) acc = fmaf(w, pr[(size_t)s * (2 + D) + 2 + j], acc);
  }
  s_o[j] = acc * s_norm;
  __syncthreads();
  float r = 0.f;
  for (int k = 0; k < D; ++k) r = fmaf(pi[(size_t)k * D + j], s_o[k], r);   // Pi[k][j] o~[k]
  out[row * D + j] = r;
}

template <int D, int BITS>
int launch_d(const tq_ctx* c, const float* q, int batch, int q_heads, int kv_heads, const void* cache,
             const int32_t* seq_lens, int max_tokens, float* out, float* logits, void* ws, cudaStream_t st,
             const PageMap& pm) {
  SplitPlan sp = plan_splits(batch, kv_heads, max_tokens);
  float* qr = static_cast<float*>(ws);
  float* qs = qr + (size_t)batch * q_heads * D;
  float* part = qs + (size_t)batch * q_heads * D;
  prologue_kernel<D><<<dim3(q_heads, batch), 4 * D, 0, st>>>(q, c->d_pit, c->d_st, qr, qs, q_heads);
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
  if (pm.table)
    split_kernel<D, BITS, true><<<dim3(sp.splits, kv_heads, batch), kThreads, 0, st>>>(a);
  else
    split_kernel<D, BITS, false><<<dim3(sp.splits, kv_heads, batch), kThreads, 0, st>>>(a);
  combine_kernel<D><<<dim3(q_heads, batch), D, 0, st>>>(part, c->d_pi, out, q_heads, sp.splits);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ECUDA;
}

}  // namespace

void launch_combine(const tq_ctx* c, const float* part, float* out, int batch, int q_heads, int splits,
                    cudaStream_t st) {
  dim3 grid(q_heads, batch);
  if (c->d == 64) combine_kernel<64><<<grid, 64, 0, st>>>(part, c->d_pi, out, q_heads, splits);
  if (c->d == 128) combine_kernel<128><<<grid, 128, 0, st>>>(part, c->d_pi, out, q_heads, splits);
  if (c->d == 256) combine_kernel<256><<<grid, 256, 0, st>>>(part, c->d_pi, out, q_heads, splits);
}

void launch_prologue(const tq_ctx* c, const float* q, int batch, int q_heads, float* qr, float* qs,
                     cudaStream_t st) {
  dim3 grid(q_heads, batch);
  if (c->d == 64) prologue_kernel<64><<<grid, 4 * 64, 0, st>>>(q, c->d_pit, c->d_st, qr, qs, q_heads);
  if (c->d == 128) prologue_kernel<128><<<grid, 4 * 128, 0, st>>>(q, c->d_pit, c->d_st, qr, qs, q_heads);
  if (c->d == 256) prologue_kernel<256><<<grid, 4 * 256, 0, st>>>(q, c->d_pit, c->d_st, qr, qs, q_heads);
}

}  // namespace tq

int launch_decode_simt(const tq_ctx* c, const float* q, int batch, int q_heads, int kv_heads,
                       const void* cache, const int32_t* seq_lens, int max_tokens, float* out,
                       float* logits_out, void* workspace, void* stream, const tq::PageMap& pm) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
#define TQ_D(DD, BB)                                                                                \
  if (c->d == DD && c->bits == BB)                                                                  \
    return tq::launch_d<DD, BB>(c, q, batch, q_heads, kv_heads, cache, seq_lens, max_tokens, out,  \
                                logits_out, workspace, st, pm);
  TQ_D(64, 2) TQ_D(64, 3) TQ_D(64, 4) TQ_D(64, 5)
  TQ_D(128, 2) TQ_D(128, 3) TQ_D(128, 4) TQ_D(128, 5)
  TQ_D(256, 2) TQ_D(256, 3) TQ_D(256, 4) TQ_D(256, 5)
#undef TQ_D
  return TQ_EUNSUPPORTED;
}
