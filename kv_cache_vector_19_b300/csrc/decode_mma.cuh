// tq_attn_decode on fp8 tensor cores over bit planes (mma.sync m16n8k32, e4m3).
//
// Score of cached key t for query head h ([BLOG] "Технология TurboQuant ...", section 1.2;
// the constant sqrt(pi/2) makes the sign sketch an unbiased inner-product estimate):
//   logit = ( n_t <q~, c_K[idx_t]> + gamma_t sqrt(pi/2)/m <q_s, 2 sigma_t - 1> ) / sqrt(d)
// Values are accumulated in the rotated frame and rotated back once by the combine kernel.
//
// Both inner products run on tensor cores without dequantising codes (see bitplane.h):
// c[idx] = 2 sum_M alpha_M x_M - sum_M alpha_M over XOR planes x_M of the code bits, and a
// plane word turns into four e4m3 operands beta_k + gamma_k * bit with one AND-OR.
//   score:  A = key planes / sign plane (16 tokens x 32 coordinates per fragment),
//           B = query pieces 2 alpha_M q~_j / gamma_k(j) (three e4m3 pieces per value:
//               hi, mid, lo, ~2^-12 relative), N = 4 heads x 3 pieces per head group;
//   values: A = value planes (16 coordinates x 32 tokens), B = softmax weights
//           p_t n_v,t / (N gamma_k(t)) in two e4m3 pieces, N = 4 heads x 2 pieces,
//           one accumulator per value plane, combined with alpha_M at the end.
// The constant parts (beta terms, sum alpha) are removed with per-query and per-head sums.
//
// Work split: the (sequence, page) list of the whole call is cut into equal ranges, one
// per CTA of a grid sized to the SM count; a CTA emits one partial (m, l, o~) record per
// sequence its range touches.  Pages stream through an up-to-8-deep shared-memory ring
// filled by cp.async.bulk (one elected thread, mbarrier completion, bounded waits), with
// L2 prefetches further ahead.  The page loop is software-pipelined: the score MMAs of page
// p run interleaved with the value MMAs of page p-2, then page p-1's softmax weights are
// formed, so one CTA barrier per page hands the weights over.  Softmax keeps a lazy running
// maximum: a page rescales the accumulators only when one of its logits exceeds the running
// maximum by more than kTau (or its largest value norm exceeds the running reference).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "bitplane.h"
#include "dev_common.cuh"
#include "layout.cuh"
#include "tq_internal.h"

namespace tq {
namespace dmma {

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kRingBytes = 120 * 1024;   // page ring budget per CTA
constexpr int kL2Ahead = 12;             // pages prefetched into L2 beyond the ring
constexpr float kTau = 3.0f;          // lazy-maximum threshold (natural-log units)
constexpr float kSB = 2.0f;           // e4m3 range scale of the softmax weights (max 20*8*2 < 448)
constexpr int kRowB = 144;            // bytes per row of the softmax-weight operand (padded)

struct Params {
  const float* qr;          // [B][Hq][D]  Pi q
  const float* qs;          // [B][Hq][D]  S q
  const uint8_t* cache;
  const int32_t* seq_lens;
  float* logits;            // nullable [B][Hq][max_tokens]
  float* part;              // [n_seq][slots][G][2 + D]
  const float* alpha_k;     // [PK] key-book plane coefficients (yhat units)
  const float* alpha_v;     // [PV]
  int* status;
  float asum_k, asum_v;     // sum of the alphas
  int batch, q_heads, kv_heads, group, max_tokens, pages_per_seq, chunk, slots, total_pages;
};

template <int D, int BITS, int NGRP>
struct Cfg {
  using PL = PageLayout<D, BITS>;
  static constexpr int BK = BITS - 1, BV = BITS;
  static constexpr int PK = 1 << (BK - 1);             // key planes (odd XOR monomials)
  static constexpr int PV = 1 << (BV - 1);             // value planes
  static constexpr int NS = PK + 1;                    // score planes: key planes + sign plane
  static constexpr int KB = D / 32;                    // 32-coordinate chunks
  static constexpr int NWS = D >= 128 ? D / 128 : 1;   // words per (token, plane) per thread
  static constexpr int VMW = D >= 128 ? D / 128 : 1;   // value m-tiles per warp
  static constexpr int VKB = D >= 128 ? 4 : 2;         // token chunks per warp (value MMA)
  static constexpr int GP = 4 * NGRP;                  // padded heads per KV head
  static constexpr int BREGS = NS * KB * 4 * NGRP;     // score B-fragment registers
  static constexpr bool BREG = BREGS <= 128;
  static constexpr int OREGS = PV * NGRP * VMW * 4;
  static constexpr int SREGS = NS * NGRP * 2 * 4;       // score accumulators (one set per plane)
  static constexpr int STAGE_BYTES = NGRP * NS * KB * 2 * 32 * 2 * 4;
  static constexpr int MINB = 1;
  static constexpr int KLOOP = KB > VKB ? KB : VKB;    // fused score / value chunk loop
  // shared-memory carve-up
  static constexpr int PAGE = PL::bytes;               // multiple of 128
  static constexpr int NBUF = kRingBytes / PAGE > 8 ? 8 : (kRingBytes / PAGE < 4 ? 4 : kRingBytes / PAGE);
  static constexpr int O_XCHG = D < 128 ? 4 * PV * NGRP * 128 * 4 : 0;   // d=64 accumulator exchange
  static constexpr int RING = NBUF * PAGE > O_XCHG ? NBUF * PAGE : O_XCHG;
  static constexpr int OFF_PAGES = 0;
  static constexpr int OFF_STAGE = OFF_PAGES + RING;
  static constexpr int OFF_BV = OFF_STAGE + STAGE_BYTES;
  static constexpr int BV_BYTES = 2 * NGRP * 8 * kRowB;
  static constexpr int OFF_Q = OFF_BV + BV_BYTES;      // [GP][2][D] f32 query vectors
  static constexpr int OFF_RED = OFF_Q + GP * 2 * D * 4;
  static constexpr int RED_FLOATS = kWarps * GP * 4;
  static constexpr int OFF_HEAD = OFF_RED + RED_FLOATS * 4;   // [GP][8] f32 per-head constants
  static constexpr int OFF_MBAR = OFF_HEAD + GP * 8 * 4;
  static constexpr int OFF_FLAG = OFF_MBAR + NBUF * 8;
  static constexpr int SMEM = OFF_FLAG + 16;
  static constexpr bool SUPPORTED = STAGE_BYTES <= 48 * 1024 && OREGS + SREGS + (BREG ? BREGS : 0) <= 200 &&
                                    OREGS <= 64 && SMEM <= 220 * 1024;
};

using namespace dev;

// ---------------------------------------------------------------- the kernel

template <int D, int BITS, int NGRP, bool PAGED>
__global__ void __launch_bounds__(kThreads, Cfg<D, BITS, NGRP>::MINB) decode_mma_kernel(Params a, PageMap pm, float sparse_v) {
  using C = Cfg<D, BITS, NGRP>;
  using PL = typename C::PL;
  constexpr int NS = C::NS, PK = C::PK, PV = C::PV, KB = C::KB, GP = C::GP, BK = C::BK, BV = C::BV;
  constexpr int NBUF = C::NBUF, VKB = C::VKB, VMW = C::VMW;
  extern __shared__ __align__(128) unsigned char smem[];
  uint8_t* s_pages = smem + C::OFF_PAGES;
  uint32_t* s_stage = reinterpret_cast<uint32_t*>(smem + C::OFF_STAGE);
  uint8_t* s_bv = smem + C::OFF_BV;
  float* s_q = reinterpret_cast<float*>(smem + C::OFF_Q);
  float* s_red = reinterpret_cast<float*>(smem + C::OFF_RED);
  float* s_head = reinterpret_cast<float*>(smem + C::OFF_HEAD);
  uint64_t* s_mbar = reinterpret_cast<uint64_t*>(smem + C::OFF_MBAR);
  volatile int* s_fail = reinterpret_cast<volatile int*>(smem + C::OFF_FLAG);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, tig = lane & 3;
  const int G = a.group, PM = a.pages_per_seq;
  const float inv_sqrt_d = rsqrtf((float)D);
  const float qjl_c = 1.2533141373155002512f / (float)D;   // sqrt(pi/2) / m, m = d

  const int range_lo = blockIdx.x * a.chunk;
  const int range_hi = min(range_lo + a.chunk, a.total_pages);
  if (range_lo >= range_hi) return;

  if (tid == 0) {
    for (int i = 0; i < NBUF; ++i) mbar_init(&s_mbar[i], 1);
    *s_fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  // score operand positions: (2 kb + h) mod 8 for d >= 128; for d = 64 they depend on the
  // lane, so masks and bases are precomputed
  constexpr int KBR = D < 128 ? KB : 1;
  uint32_t smask[KBR][2], sbase[KBR][2];
#pragma unroll
  for (int kb = 0; kb < KBR; ++kb)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      int s = tig * (2 * D / 32) + 2 * kb + h, pos = s & 7;
      smask[kb][h] = 0x01010101u << pos;
      uint32_t base = pos == 3 ? 0x30u : pos == 4 ? 0x28u : pos == 5 ? 0x18u : pos == 6 ? 0x00u : 0x38u;
      sbase[kb][h] = base * 0x01010101u;
    }
  // the softmax weights of token slots 16 w .. 16 w + 15 meet value-code bit position w
  const float v_beta = e4m3_beta(warp), v_gamma = e4m3_gamma(warp), v_igamma = 1.f / e4m3_gamma(warp);

  uint32_t fill_count = 0;     // pages issued so far in this CTA (ring position)
  uint32_t waited = 0;         // fills whose completion this thread has observed
  uint32_t issued = 0;         // fills issued (thread 0)
  bool failed = false;

  // walk the sequences this CTA's range touches
  int gp = range_lo;
  while (gp < range_hi && !failed) {
    const int seq = gp / PM;
    const int seg_lo = gp - seq * PM;
    const int seg_hi = min(range_hi, (seq + 1) * PM) - seq * PM;
    gp = (seq + 1) * PM;
    const int b = seq / a.kv_heads, kvh = seq % a.kv_heads;
    int seq_len = a.seq_lens[b];
    if (seq_len < 0 || seq_len > a.max_tokens) {
      if (tid == 0 && seg_lo == 0) atomicOr(a.status, kFlagBounds);
      seq_len = seq_len < 0 ? 0 : a.max_tokens;
    }
    const int valid_pages = (seq_len + 127) >> 7;
    const int p_lo = seg_lo, p_hi = min(seg_hi, valid_pages);
    const int n_pages = max(0, p_hi - p_lo);
    const int slot = blockIdx.x - (seq * PM) / a.chunk;
    float* rec = a.part + ((size_t)seq * a.slots + slot) * G * (2 + D);
    // page p of this sequence: contiguous, or through the block table (PAGED, a separate
    // instantiation so that the contiguous kernel's address arithmetic stays as it was)
    const uint8_t* seq_base = a.cache + (size_t)seq * PM * PL::bytes;
    auto page_g = [&](int p) -> const uint8_t* {
      if constexpr (PAGED) return a.cache + pm.index(seq, a.kv_heads, PM, p, a.status) * PL::bytes;
      else return seq_base + (size_t)p * PL::bytes;
    };

    __syncthreads();   // the previous segment is fully done with shared memory
    // start streaming this segment's pages while the query operand is built
    const uint32_t fill_base = fill_count;
    if (tid == 0) {
      const int first = min(n_pages, NBUF);
      issued = fill_base + first;
      for (int i = 0; i < first; ++i) {
        const uint32_t slot_i = (fill_base + i) % NBUF;
        fence_proxy_async();
        mbar_expect_tx(&s_mbar[slot_i], PL::bytes);
        bulk_g2s(s_pages + slot_i * C::PAGE, page_g(p_lo + i), PL::bytes, &s_mbar[slot_i]);
      }
      for (int i = NBUF; i < min(n_pages, NBUF + kL2Ahead); ++i)
        prefetch_l2(page_g(p_lo + i), PL::bytes);
    }
    fill_count = fill_base + n_pages;   // every page of the segment is issued and consumed

    // ---- query operand for this KV head: pieces, constants, fragments ----
    for (int e = tid; e < GP * 2 * D; e += kThreads) {
      int hh = e / (2 * D), rem = e % (2 * D), which = rem / D, j = rem % D;
      float v = 0.f;
      if (hh < G) {
        size_t row = (size_t)b * a.q_heads + (size_t)kvh * G + hh;
        v = (which == 0 ? a.qr : a.qs)[row * D + j];
      }
      s_q[e] = v;
    }
    for (int e = tid; e < GP * 8; e += kThreads) s_head[e] = 0.f;
    __syncthreads();
    // per head: max |B| for the MSE planes and for the sign plane -> power-of-two scales
    for (int hh = warp; hh < GP; hh += kWarps) {
      float mk = 0.f, mq = 0.f;
      for (int j = lane; j < D; j += 32) {
        int s = ((j >> 2) & 3) * (2 * D / 32) + 2 * (j >> 5) + ((j >> 4) & 1), pos = s & 7;
        float ig = 1.f / fabsf(e4m3_gamma(pos));
        mk = fmaxf(mk, fabsf(s_q[(hh * 2 + 0) * D + j]) * ig);
        mq = fmaxf(mq, fabsf(s_q[(hh * 2 + 1) * D + j]) * ig);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        mk = fmaxf(mk, __shfl_xor_sync(0xffffffffu, mk, o));
        mq = fmaxf(mq, __shfl_xor_sync(0xffffffffu, mq, o));
      }
      if (lane == 0) {
        float amax = 0.f;
        for (int i = 0; i < PK; ++i) amax = fmaxf(amax, fabsf(a.alpha_k[i]));
        float bk = 2.f * amax * mk, bq = 2.f * mq;
        // largest operand at most 224 (e4m3 max 448), power of two
        float sk = bk > 0.f ? exp2f(floorf(log2f(224.f / bk))) : 1.f;
        float sq = bq > 0.f ? exp2f(floorf(log2f(224.f / bq))) : 1.f;
        s_head[hh * 8 + 0] = sk;
        s_head[hh * 8 + 1] = sq;
      }
    }
    __syncthreads();
    // fragments: lane (g, tig) of every warp holds b0/b1 for n = g, k = 4 tig + e (+16).
    // Column n of tile 0 = (head 4u + n/2, piece n%2); tile 1 = (head 4u + n/2, piece 2 if n even).
    // Stage layout [u][plane][kb][nt][lane][2] u32.
    for (int e = tid; e < NGRP * NS * KB * 2 * 32; e += kThreads) {
      int ln = e & 31, rest = e >> 5;
      int nt = rest % 2;
      rest /= 2;
      int kb = rest % KB;
      rest /= KB;
      int pl = rest % NS, u = rest / NS;
      int gg = ln >> 2, tt = ln & 3;
      int hh = 4 * u + (gg >> 1);
      int piece = nt == 0 ? (gg & 1) : ((gg & 1) ? -1 : 2);
      uint32_t words[2] = {0u, 0u};
      if (hh < G && piece >= 0) {
        float sc = s_head[hh * 8 + (pl < PK ? 0 : 1)];
        float coef = pl < PK ? 2.f * a.alpha_k[pl] : 2.f;
        const float* qv = s_q + (hh * 2 + (pl < PK ? 0 : 1)) * D;
#pragma unroll
        for (int r = 0; r < 2; ++r)
#pragma unroll
          for (int el = 0; el < 4; ++el) {
            int j = 32 * kb + 16 * r + 4 * tt + el;
            int s = ((j >> 2) & 3) * (2 * D / 32) + 2 * (j >> 5) + ((j >> 4) & 1), pos = s & 7;
            float v = coef * qv[j] * sc / e4m3_gamma(pos);
            uint32_t p0, p1, p2;
            split3(v, p0, p1, p2);
            uint32_t byte = piece == 0 ? p0 : piece == 1 ? p1 : p2;
            words[r] |= byte << (8 * el);
          }
      }
      s_stage[e * 2 + 0] = words[0];
      s_stage[e * 2 + 1] = words[1];
    }
    // per-head constants: C = sum over planes and j of beta_k(j) * (hi + mid/16 + lo/256),
    // in scaled units, separately for the MSE planes and the sign plane; sum_j q~_j, sum_i q_s,i.
    for (int hh = warp; hh < GP; hh += kWarps) {
      float cm = 0.f, cq = 0.f, sumk = 0.f, sumq = 0.f;
      if (hh < G) {
        float sk = s_head[hh * 8 + 0], sq = s_head[hh * 8 + 1];
        for (int j = lane; j < D; j += 32) {
          int s = ((j >> 2) & 3) * (2 * D / 32) + 2 * (j >> 5) + ((j >> 4) & 1), pos = s & 7;
          float beta = e4m3_beta(pos), ig = 1.f / e4m3_gamma(pos);
          float qk = s_q[(hh * 2 + 0) * D + j], qq = s_q[(hh * 2 + 1) * D + j];
          sumk += qk;
          sumq += qq;
          for (int pl = 0; pl < PK; ++pl) {
            uint32_t p0, p1, p2;
            split3(2.f * a.alpha_k[pl] * qk * sk * ig, p0, p1, p2);
            cm += beta * split3_val(p0, p1, p2);
          }
          uint32_t p0, p1, p2;
          split3(2.f * qq * sq * ig, p0, p1, p2);
          cq += beta * split3_val(p0, p1, p2);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        cm += __shfl_xor_sync(0xffffffffu, cm, o);
        cq += __shfl_xor_sync(0xffffffffu, cq, o);
        sumk += __shfl_xor_sync(0xffffffffu, sumk, o);
        sumq += __shfl_xor_sync(0xffffffffu, sumq, o);
      }
      if (lane == 0) {
        s_head[hh * 8 + 2] = cm;
        s_head[hh * 8 + 3] = cq;
        s_head[hh * 8 + 4] = sumk;
        s_head[hh * 8 + 5] = sumq;
      }
    }
    __syncthreads();

    uint32_t breg[C::BREG ? NGRP : 1][C::BREG ? NS : 1][C::BREG ? KB : 1][C::BREG ? 2 : 1][2];
    if constexpr (C::BREG) {
#pragma unroll
      for (int u = 0; u < NGRP; ++u)
#pragma unroll
        for (int pl = 0; pl < NS; ++pl)
#pragma unroll
          for (int kb = 0; kb < KB; ++kb)
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
              int e = (((u * NS + pl) * KB + kb) * 2 + nt) * 32 + lane;
              uint2 w = *reinterpret_cast<const uint2*>(&s_stage[e * 2]);
              breg[u][pl][kb][nt][0] = w.x;
              breg[u][pl][kb][nt][1] = w.y;
            }
    }
    // per-thread head constants (heads 4u + tig)
    float inv_sk[NGRP], inv_sq[NGRP], cm[NGRP], cq[NGRP], sumk[NGRP], sumq[NGRP];
#pragma unroll
    for (int u = 0; u < NGRP; ++u) {
      const float* hp = s_head + (4 * u + tig) * 8;
      inv_sk[u] = 1.f / hp[0];
      inv_sq[u] = 1.f / hp[1];
      cm[u] = hp[2];
      cq[u] = hp[3];
      sumk[u] = hp[4];
      sumq[u] = hp[5];
    }

    // ---- running state ----
    float m_run[NGRP], l_part[NGRP], c_part[NGRP], g_part[NGRP];
    float lg_prev[NGRP][2], nv_prev[2] = {0.f, 0.f}, nvpage_prev = 0.f;
#pragma unroll
    for (int u = 0; u < NGRP; ++u) {
      m_run[u] = -INFINITY;
      l_part[u] = c_part[u] = g_part[u] = 0.f;
      lg_prev[u][0] = lg_prev[u][1] = -INFINITY;
    }
    float n_ref = 0.f;                                  // running value-norm reference
    int ovf_prev = 0;                                   // vote of the previous page
    float o[PV][NGRP][VMW][4];
#pragma unroll
    for (int pv = 0; pv < PV; ++pv)
#pragma unroll
      for (int u = 0; u < NGRP; ++u)
#pragma unroll
        for (int mt = 0; mt < VMW; ++mt)
#pragma unroll
          for (int r = 0; r < 4; ++r) o[pv][u][mt][r] = 0.f;

    const int t0 = 16 * warp + g, t1 = t0 + 8;          // score rows of this thread
    const int kb0 = D >= 128 ? 0 : 2 * (warp >> 2);     // first token chunk of the value MMA

    // Software pipeline, one CTA barrier per page.  Iteration it:
    //   score MMAs of page it, interleaved with the value MMAs of page it-2;
    //   rescale (if page it-1 voted for it) and softmax weights of page it-1;
    //   logits and vote of page it; barrier.
    const int n_iter = n_pages > 0 ? n_pages + 2 : 0;
    for (int it = 0; it < n_iter; ++it) {
      const bool do_s = it < n_pages;
      const bool do_v = it >= 2;
      const uint8_t* pg = s_pages + ((fill_base + it) % NBUF) * C::PAGE;
      const uint8_t* pv_pg = s_pages + ((fill_base + it + NBUF - 2) % NBUF) * C::PAGE;   // page it-2
      if (do_s) {
        const uint32_t parity = ((fill_base + it) / NBUF) & 1;
        if (mbar_wait(&s_mbar[(fill_base + it) % NBUF], parity)) {
          waited = fill_base + it + 1;
        } else {
          if (lane == 0) atomicOr(a.status, kFlagTimeout);
          *s_fail = 1;
        }
      }
      // ---------- operands ----------
      float acc[NS][NGRP][2][4];
#pragma unroll
      for (int pl = 0; pl < NS; ++pl)
#pragma unroll
        for (int u = 0; u < NGRP; ++u)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[pl][u][nt][r] = 0.f;
      uint32_t xs[NS][2][C::NWS];            // score plane words (XOR monomials, then signs)
      if (do_s) {
        uint32_t wk[BK][2][C::NWS];
#pragma unroll
        for (int nw = 0; nw < C::NWS; ++nw) {
          const int wi = D >= 128 ? tig * C::NWS + nw : (tig >> 1);
#pragma unroll
          for (int q = 0; q < BK; ++q) {
            const uint32_t* pw = reinterpret_cast<const uint32_t*>(pg + PL::off_kcodes) + (size_t)q * 128 * PL::KW;
            wk[q][0][nw] = pw[t0 * PL::KW + wi];
            wk[q][1][nw] = pw[t1 * PL::KW + wi];
          }
          const uint32_t* ps = reinterpret_cast<const uint32_t*>(pg + PL::off_signs);
          xs[PK][0][nw] = ps[t0 * PL::SW + wi];
          xs[PK][1][nw] = ps[t1 * PL::SW + wi];
        }
#pragma unroll
        for (int pl = 0; pl < PK; ++pl)
#pragma unroll
          for (int tk = 0; tk < 2; ++tk)
#pragma unroll
            for (int nw = 0; nw < C::NWS; ++nw) {
              uint32_t v = 0u;
#pragma unroll
              for (int q = 0; q < BK; ++q)
                if ((mono_mask16(pl) >> q) & 1) v ^= wk[q][tk][nw];
              xs[pl][tk][nw] = v;
            }
      }
      uint32_t xv[PV][VMW][2];               // value plane words (XOR monomials) of page it-2
      uint32_t bfr[NGRP][VKB][2];            // softmax-weight fragments of page it-2
      if (do_v) {
        const uint8_t* bvb = s_bv + (it & 1) * NGRP * 8 * kRowB;    // (it-2) & 1 == it & 1
#pragma unroll
        for (int u = 0; u < NGRP; ++u)
#pragma unroll
          for (int kk = 0; kk < VKB; ++kk) {
            const uint8_t* row = bvb + (u * 8 + g) * kRowB + 32 * (kb0 + kk) + 4 * tig;
            bfr[u][kk][0] = *reinterpret_cast<const uint32_t*>(row);
            bfr[u][kk][1] = *reinterpret_cast<const uint32_t*>(row + 16);
          }
        const uint32_t* pvw = reinterpret_cast<const uint32_t*>(pv_pg + PL::off_vcodes);
#pragma unroll
        for (int mt = 0; mt < VMW; ++mt) {
          const int mtile = D >= 128 ? warp + 8 * mt : (warp & 3);
          const int j0 = 16 * mtile + g, j1 = j0 + 8;
          uint32_t wv[BV][2];
#pragma unroll
          for (int q = 0; q < BV; ++q) {
            wv[q][0] = pvw[((size_t)q * D + j0) * 4 + tig];
            wv[q][1] = pvw[((size_t)q * D + j1) * 4 + tig];
          }
#pragma unroll
          for (int pl = 0; pl < PV; ++pl) {
            uint32_t x0 = 0u, x1 = 0u;
#pragma unroll
            for (int q = 0; q < BV; ++q)
              if ((mono_mask16(pl) >> q) & 1) {
                x0 ^= wv[q][0];
                x1 ^= wv[q][1];
              }
            xv[pl][mt][0] = x0;
            xv[pl][mt][1] = x1;
          }
        }
      }
      // ---------- fused MMA phase: independent chains per plane, interleaved by chunk ----------
#pragma unroll
      for (int kc = 0; kc < C::KLOOP; ++kc) {
        if (do_s && kc < KB) {
          const int kb = kc;
          const int nw = D >= 256 ? (kb >> 2) : 0;
#pragma unroll
          for (int pl = 0; pl < NS; ++pl) {
            uint32_t a0, a1, a2, a3;
            if constexpr (D >= 128) {
              a0 = expand_at(xs[pl][0][nw], 2 * kb);
              a1 = expand_at(xs[pl][1][nw], 2 * kb);
              a2 = expand_at(xs[pl][0][nw], 2 * kb + 1);
              a3 = expand_at(xs[pl][1][nw], 2 * kb + 1);
            } else {
              a0 = expand_rt(xs[pl][0][nw], smask[kb][0], sbase[kb][0]);
              a1 = expand_rt(xs[pl][1][nw], smask[kb][0], sbase[kb][0]);
              a2 = expand_rt(xs[pl][0][nw], smask[kb][1], sbase[kb][1]);
              a3 = expand_rt(xs[pl][1][nw], smask[kb][1], sbase[kb][1]);
            }
#pragma unroll
            for (int u = 0; u < NGRP; ++u)
#pragma unroll
              for (int nt = 0; nt < 2; ++nt) {
                uint32_t b0, b1;
                if constexpr (C::BREG) {
                  b0 = breg[u][pl][kb][nt][0];
                  b1 = breg[u][pl][kb][nt][1];
                } else {
                  int e = (((u * NS + pl) * KB + kb) * 2 + nt) * 32 + lane;
                  uint2 w = *reinterpret_cast<const uint2*>(&s_stage[e * 2]);
                  b0 = w.x;
                  b1 = w.y;
                }
                mma_e4m3(acc[pl][u][nt], a0, a1, a2, a3, b0, b1);
              }
          }
        }
        if (do_v && kc < VKB) {
          const int kb = kb0 + kc;   // token chunk: bit positions 2kb, 2kb+1
#pragma unroll
          for (int mt = 0; mt < VMW; ++mt)
#pragma unroll
            for (int pl = 0; pl < PV; ++pl) {
              const uint32_t a0 = expand_at(xv[pl][mt][0], 2 * kb), a1 = expand_at(xv[pl][mt][1], 2 * kb);
              const uint32_t a2 = expand_at(xv[pl][mt][0], 2 * kb + 1), a3 = expand_at(xv[pl][mt][1], 2 * kb + 1);
#pragma unroll
              for (int u = 0; u < NGRP; ++u) mma_e4m3(o[pl][u][mt], a0, a1, a2, a3, bfr[u][kc][0], bfr[u][kc][1]);
            }
        }
      }
      // ---------- logits of page it (thread owns heads 4u + tig, tokens t0, t1) ----------
      float lg_cur[NGRP][2], nv_cur[2] = {0.f, 0.f}, nvpage_cur = 0.f;
      int ovf = 0;
      if (do_s) {
        const int page = p_lo + it;
        const int nvalid = min(128, seq_len - page * 128);
        const float* nk = reinterpret_cast<const float*>(pg + PL::off_nk);
        const float* gm = reinterpret_cast<const float*>(pg + PL::off_gamma);
        const float* nvp = reinterpret_cast<const float*>(pg + PL::off_nv);
        const bool v0 = t0 < nvalid, v1 = t1 < nvalid;
        const float n0 = v0 ? nk[t0] : 0.f, n1 = v1 ? nk[t1] : 0.f;
        const float g0 = v0 ? gm[t0] : 0.f, g1 = v1 ? gm[t1] : 0.f;
        nv_cur[0] = v0 ? nvp[t0] : 0.f;
        nv_cur[1] = v1 ? nvp[t1] : 0.f;
#pragma unroll
        for (int u = 0; u < NGRP; ++u) {
          const int hh = 4 * u + tig;
          float mse0 = 0.f, mse1 = 0.f;
#pragma unroll
          for (int pl = 0; pl < PK; ++pl) {
            mse0 += acc[pl][u][0][0] + 0.0625f * acc[pl][u][0][1] + 0.00390625f * acc[pl][u][1][0];
            mse1 += acc[pl][u][0][2] + 0.0625f * acc[pl][u][0][3] + 0.00390625f * acc[pl][u][1][2];
          }
          const float qj0 = acc[PK][u][0][0] + 0.0625f * acc[PK][u][0][1] + 0.00390625f * acc[PK][u][1][0];
          const float qj1 = acc[PK][u][0][2] + 0.0625f * acc[PK][u][0][3] + 0.00390625f * acc[PK][u][1][2];
          const float dk0 = (mse0 - cm[u]) * inv_sk[u] - a.asum_k * sumk[u];
          const float dk1 = (mse1 - cm[u]) * inv_sk[u] - a.asum_k * sumk[u];
          const float dq0 = (qj0 - cq[u]) * inv_sq[u] - sumq[u];
          const float dq1 = (qj1 - cq[u]) * inv_sq[u] - sumq[u];
          const float l0 = (n0 * dk0 + g0 * qjl_c * dq0) * inv_sqrt_d;
          const float l1 = (n1 * dk1 + g1 * qjl_c * dq1) * inv_sqrt_d;
          const bool hv = hh < G;
          lg_cur[u][0] = (v0 && hv) ? l0 : -INFINITY;
          lg_cur[u][1] = (v1 && hv) ? l1 : -INFINITY;
          if (a.logits && hv) {
            float* dst =
                a.logits + ((size_t)b * a.q_heads + (size_t)kvh * G + hh) * a.max_tokens + (size_t)page * 128;
            if (v0) dst[t0] = l0;
            if (v1) dst[t1] = l1;
          }
          if (lg_cur[u][0] > m_run[u] + kTau || lg_cur[u][1] > m_run[u] + kTau) ovf = 1;
        }
        // page maximum of the value norms (every warp computes it redundantly)
        float4 n4 = reinterpret_cast<const float4*>(nvp)[lane];
        float m4 = 0.f;
        if (4 * lane + 0 < nvalid) m4 = fmaxf(m4, n4.x);
        if (4 * lane + 1 < nvalid) m4 = fmaxf(m4, n4.y);
        if (4 * lane + 2 < nvalid) m4 = fmaxf(m4, n4.z);
        if (4 * lane + 3 < nvalid) m4 = fmaxf(m4, n4.w);
#pragma unroll
        for (int o2 = 16; o2 > 0; o2 >>= 1) m4 = fmaxf(m4, __shfl_xor_sync(0xffffffffu, m4, o2));
        nvpage_cur = m4;
        if (nvpage_cur > n_ref) ovf = 1;
      } else {
#pragma unroll
        for (int u = 0; u < NGRP; ++u) lg_cur[u][0] = lg_cur[u][1] = -INFINITY;
      }
      // ---------- page it-1: lazy rescale (rare), then its softmax weights ----------
      if (it >= 1 && it - 1 < n_pages) {
        if (ovf_prev) {
#pragma unroll
          for (int u = 0; u < NGRP; ++u) {
            float mx = fmaxf(lg_prev[u][0], lg_prev[u][1]);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            if (g == 0) s_red[(warp * GP + 4 * u + tig)] = mx;
          }
          __syncthreads();
          const float n_new = nvpage_prev > n_ref ? nvpage_prev * 1.25f : n_ref;
#pragma unroll
          for (int u = 0; u < NGRP; ++u) {
            float mx = -INFINITY;
            for (int w2 = 0; w2 < kWarps; ++w2) mx = fmaxf(mx, s_red[w2 * GP + 4 * u + tig]);
            const float m_new = fmaxf(m_run[u], mx);
            const float alpha = (m_run[u] == -INFINITY) ? 0.f : __expf(m_run[u] - m_new);
            const float f = (n_ref > 0.f) ? alpha * (n_ref / n_new) : 0.f;
            l_part[u] *= alpha;
            c_part[u] *= f;
            g_part[u] *= f;
#pragma unroll
            for (int pv = 0; pv < PV; ++pv)
#pragma unroll
              for (int mt = 0; mt < VMW; ++mt)
#pragma unroll
                for (int r = 0; r < 4; ++r) o[pv][u][mt][r] *= f;
            m_run[u] = m_new;
          }
          n_ref = n_new;
          __syncthreads();   // s_red reads done before it is reused
        }
        uint8_t* bvb = s_bv + ((it - 1) & 1) * NGRP * 8 * kRowB;
        const float inv_n = n_ref > 0.f ? 1.f / n_ref : 0.f;
#pragma unroll
        for (int u = 0; u < NGRP; ++u) {
          const float p0 = lg_prev[u][0] == -INFINITY ? 0.f : __expf(lg_prev[u][0] - m_run[u]);
          const float p1 = lg_prev[u][1] == -INFINITY ? 0.f : __expf(lg_prev[u][1] - m_run[u]);
          l_part[u] += p0 + p1;   // the denominator keeps every position
          // Sparse V: a position below the threshold contributes no value
          const float x0 = (p0 < sparse_v ? 0.f : p0) * nv_prev[0] * inv_n * v_igamma * kSB;
          const float x1 = (p1 < sparse_v ? 0.f : p1) * nv_prev[1] * inv_n * v_igamma * kSB;
          const uint32_t hi = cvt_e4m3x2(x1, x0);
          const float2 hf = e4m3x2_to_f2(hi);
          const uint32_t lo = cvt_e4m3x2(16.f * (x1 - hf.y), 16.f * (x0 - hf.x));   // second piece x16
          const float2 lf = e4m3x2_to_f2(lo);
          const float bs = hf.x + hf.y + 0.0625f * (lf.x + lf.y);
          c_part[u] += v_beta * bs;
          g_part[u] += v_gamma * bs;
          uint8_t* r0 = bvb + (u * 8 + 2 * tig) * kRowB;
          uint8_t* r1 = r0 + kRowB;
          r0[t0] = (uint8_t)(hi & 0xFF);
          r0[t1] = (uint8_t)(hi >> 8);
          r1[t0] = (uint8_t)(lo & 0xFF);
          r1[t1] = (uint8_t)(lo >> 8);
        }
      }
      // ---------- barrier: vote of page it; page it-1's weights complete; page it-2 free ----------
      ovf_prev = __syncthreads_or(ovf);
      if (*s_fail) {                 // uniform: written before the barrier
        failed = true;
        break;
      }
#pragma unroll
      for (int u = 0; u < NGRP; ++u) {
        lg_prev[u][0] = lg_cur[u][0];
        lg_prev[u][1] = lg_cur[u][1];
      }
      nv_prev[0] = nv_cur[0];
      nv_prev[1] = nv_cur[1];
      nvpage_prev = nvpage_cur;
      if (tid == 0 && it >= 2) {
        const int nxt = it - 2 + NBUF;
        if (nxt < n_pages) {
          issued = fill_base + nxt + 1;
          const uint32_t slot_i = (fill_base + nxt) % NBUF;
          fence_proxy_async();
          mbar_expect_tx(&s_mbar[slot_i], PL::bytes);
          bulk_g2s(s_pages + slot_i * C::PAGE, page_g(p_lo + nxt), PL::bytes,
                   &s_mbar[slot_i]);
        }
        const int far = nxt + kL2Ahead;
        if (far < n_pages) prefetch_l2(page_g(p_lo + far), PL::bytes);
      }
    }
    if (failed) break;

    // ---------- segment epilogue: reduce per-head sums, write the partial record ----------
    __syncthreads();
#pragma unroll
    for (int u = 0; u < NGRP; ++u) {
      float v3[3] = {l_part[u], c_part[u], g_part[u]};
#pragma unroll
      for (int c = 0; c < 3; ++c) {
        float v = v3[c];
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 16);
        if (g == 0) s_red[(warp * GP + 4 * u + tig) * 3 + c] = v;
      }
    }
    __syncthreads();
    float l_tot[NGRP], c_tot[NGRP], g_tot[NGRP];
#pragma unroll
    for (int u = 0; u < NGRP; ++u) {
      l_tot[u] = c_tot[u] = g_tot[u] = 0.f;
      for (int w2 = 0; w2 < kWarps; ++w2) {
        const float* r = s_red + (w2 * GP + 4 * u + tig) * 3;
        l_tot[u] += r[0];
        c_tot[u] += r[1];
        g_tot[u] += r[2];
      }
    }
    // D = 64: warps w and w + 4 hold partial sums over token halves of the same m-tile
    if constexpr (D < 128) {
      __syncthreads();
      float* s_o = reinterpret_cast<float*>(s_pages);   // the ring is idle here
      if (warp >= 4) {
#pragma unroll
        for (int pv = 0; pv < PV; ++pv)
#pragma unroll
          for (int u = 0; u < NGRP; ++u)
#pragma unroll
            for (int r = 0; r < 4; ++r) s_o[(((warp - 4) * PV + pv) * NGRP + u) * 128 + r * 32 + lane] = o[pv][u][0][r];
      }
      __syncthreads();
      if (warp < 4) {
#pragma unroll
        for (int pv = 0; pv < PV; ++pv)
#pragma unroll
          for (int u = 0; u < NGRP; ++u)
#pragma unroll
            for (int r = 0; r < 4; ++r) o[pv][u][0][r] += s_o[((warp * PV + pv) * NGRP + u) * 128 + r * 32 + lane];
      }
    }
    const bool writer = D >= 128 || warp < 4;
    float alphas_v[PV];
#pragma unroll
    for (int pv = 0; pv < PV; ++pv) alphas_v[pv] = a.alpha_v[pv];
#pragma unroll
    for (int u = 0; u < NGRP; ++u) {
      const int hh = 4 * u + tig;
      if (hh >= G) continue;
      float* rh = rec + (size_t)hh * (2 + D);
      const float scale = n_ref / kSB;
      if (g == 0 && warp == 0) {
        rh[0] = m_run[u];
        rh[1] = l_tot[u];
      }
      if (!writer) continue;
#pragma unroll
      for (int mt = 0; mt < VMW; ++mt) {
        const int mtile = D >= 128 ? warp + 8 * mt : (warp & 3);
        float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
        for (int pv = 0; pv < PV; ++pv) {
          acc0 += alphas_v[pv] * (o[pv][u][mt][0] + 0.0625f * o[pv][u][mt][1] - c_tot[u]);
          acc1 += alphas_v[pv] * (o[pv][u][mt][2] + 0.0625f * o[pv][u][mt][3] - c_tot[u]);
        }
        const float base = a.asum_v * g_tot[u];
        rh[2 + 16 * mtile + g] = scale * (2.f * acc0 - base);
        rh[2 + 16 * mtile + g + 8] = scale * (2.f * acc1 - base);
      }
    }
  }
  // drain: copies still in flight target this CTA's shared memory; wait for them (bounded)
  if (failed && tid == 0) {
    for (uint32_t i = waited; i < issued; ++i) mbar_wait(&s_mbar[i % NBUF], (i / NBUF) & 1);
  }
}

}  // namespace dmma
}  // namespace tq
