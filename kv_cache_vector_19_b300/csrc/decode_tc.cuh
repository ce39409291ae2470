// tq_attn_decode on 5th-generation tensor cores (tcgen05, kind::f8f6f4), head_dim 128.
//
// Same arithmetic as the mma.sync kernel (decode_mma.cuh): the score of a cached key and
// the value accumulation are contractions over bit planes of the codes, each plane word
// turned into e4m3 operands beta_k + gamma_k * bit by one AND-OR (bitplane.h), the per-
// position scales folded into the other operand.  What changes is where the MMAs run:
//   A_s (TMEM, lane = token)      key planes and the sign plane of one page, NS x 128 bytes
//   B_s (smem, K-major)           query pieces: 3 e4m3 pieces per head for the key term and
//                                 3 for the sign term (columns), one row block per plane
//   D_s (TMEM, lane = token)      score partial sums, read back by the token warps
//   A_v (TMEM, lane = coordinate) value planes of one page, PV x 128 bytes
//   B_v (smem, K-major)           softmax weights of the page, 2 e4m3 pieces per head
//   D_v (TMEM, lane = coordinate) one accumulator per value plane, kept across pages
// One thread issues every MMA (12 instructions for the score of a page at b = 3, 16 for
// the values) and the tensor pipe runs them asynchronously; completion is signalled on
// mbarriers by tcgen05.commit.
//
// Warp roles, 8 warps: warps 0-3 ("token warps", TMEM lane = token) read D_s, form logits,
// run the lazy online softmax and write B_v; warps 4-7 ("plane warps", same lane quarters)
// expand the value planes of page p (lane = coordinate) and the key planes of page p+1
// (lane = token) into TMEM.  Per page: one CTA barrier, after which the elected thread
// issues the value MMA of page p and the score MMA of page p+1 and refills the page ring.
#pragma once

#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "bitplane.h"
#include "decode_mma.cuh"
#include "dev_common.cuh"
#include "layout.cuh"
#include "tq_internal.h"

namespace tq {
namespace dtc {

using namespace dev;
using dmma::Params;

constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kL2Ahead = 12;
constexpr float kTau = 3.0f;          // lazy-maximum threshold (natural-log units)
constexpr float kSB = 2.0f;           // e4m3 range scale of the softmax weights

__host__ __device__ constexpr int rnd(int x, int m) { return (x + m - 1) / m * m; }

template <int BITS, int GP>
struct Cfg {
  static constexpr int D = 128;
  using PL = PageLayout<128, BITS>;
  static constexpr int BK = BITS - 1, BV = BITS;
  static constexpr int PK = 1 << (BK - 1), PV = 1 << (BV - 1), NS = PK + 1;
  static constexpr int NHALF = rnd(3 * GP, 8);         // score columns: [key term | sign term]
  static constexpr int NSC = rnd(2 * NHALF, 16);
  static constexpr int NVC = 2 * GP < 16 ? 16 : 2 * GP;  // value columns: 2 pieces per head
  // tensor-memory columns
  static constexpr int TD_S = 0;
  static constexpr int TD_V = rnd(NSC, 32);
  static constexpr int TA_S = TD_V + rnd(PV * NVC, 32);
  static constexpr int TA_V = TA_S + NS * 32;
  static constexpr int TCOLS = TA_V + PV * 32;
  static constexpr int TALLOC = TCOLS <= 256 ? 256 : 512;
  // shared memory
  static constexpr int PAGE = PL::bytes;
  static constexpr int NBUF = (128 * 1024) / PAGE > 8 ? 8 : (128 * 1024) / PAGE;
  static constexpr int BS_BYTES = NSC * NS * 128;
  static constexpr int BV_BYTES = NVC * 128;
  static constexpr int OFF_PAGES = 0;
  static constexpr int OFF_BS = OFF_PAGES + NBUF * PAGE;
  static constexpr int OFF_BV = OFF_BS + BS_BYTES;
  static constexpr int OFF_Q = OFF_BV + BV_BYTES;               // [GP][2][128] f32
  static constexpr int OFF_HEAD = OFF_Q + GP * 2 * 128 * 4;     // [GP][8] f32
  static constexpr int OFF_RED = OFF_HEAD + GP * 8 * 4;         // [4 warps][GP + 1][3] f32
  static constexpr int OFF_F = OFF_RED + 4 * (GP + 1) * 3 * 4;  // [GP] rescale factors, [GP] n_ref
  static constexpr int OFF_MBAR = rnd(OFF_F + (GP + 1) * 4, 8); // full[NBUF], s_done, v_done
  static constexpr int OFF_MISC = OFF_MBAR + (NBUF + 2) * 8;    // tmem base, fail, rescale
  static constexpr int SMEM = OFF_MISC + 16;
  static constexpr bool SUPPORTED = TCOLS <= 512 && SMEM <= 225 * 1024 && NBUF >= 4;
};

// OR-vote / barrier among the four token warps (named barrier 1).
__device__ __forceinline__ int t_vote_or(int pred) {
  int r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.s32 q, %1, 0;\n barrier.cta.red.or.pred p, 1, 128, q;\n selp.s32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"(pred)
      : "memory");
  return r;
}
__device__ __forceinline__ void t_sync() { asm volatile("barrier.cta.sync 1, 128;" ::: "memory"); }

// bit position (0..7) of coordinate or token slot x within its plane word
__host__ __device__ __forceinline__ int kpos_of(int x) { return 2 * (x >> 5) + ((x >> 4) & 1); }
// coordinate / token slot held by byte e of TMEM column (w * 8 + k) of a plane
__host__ __device__ __forceinline__ int slot_of_col(int w, int k, int e) {
  return 32 * (k >> 1) + 16 * (k & 1) + 4 * w + e;
}

template <int BITS, int GP>
__global__ void __launch_bounds__(kThreads, 1) decode_tc_kernel(Params a) {
  using C = Cfg<BITS, GP>;
  using PL = typename C::PL;
  constexpr int D = 128, NS = C::NS, PK = C::PK, PV = C::PV, BK = C::BK, BV = C::BV, NBUF = C::NBUF;
  constexpr int NSC = C::NSC, NVC = C::NVC, NHALF = C::NHALF;
  extern __shared__ __align__(1024) unsigned char smem[];
  uint8_t* s_pages = smem + C::OFF_PAGES;
  uint8_t* s_bs = smem + C::OFF_BS;
  uint8_t* s_bv = smem + C::OFF_BV;
  float* s_q = reinterpret_cast<float*>(smem + C::OFF_Q);
  float* s_head = reinterpret_cast<float*>(smem + C::OFF_HEAD);
  float* s_red = reinterpret_cast<float*>(smem + C::OFF_RED);
  float* s_f = reinterpret_cast<float*>(smem + C::OFF_F);
  uint64_t* s_full = reinterpret_cast<uint64_t*>(smem + C::OFF_MBAR);
  uint64_t* s_sdone = s_full + NBUF;
  uint64_t* s_vdone = s_full + NBUF + 1;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* s_fail = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);
  volatile int* s_rescale = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 8);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool tok = warp < 4;                 // token warps
  const int row = 32 * (warp & 3) + lane;    // TMEM lane of this thread
  const int G = a.group, PM = a.pages_per_seq;
  const float inv_sqrt_d = rsqrtf((float)D);
  const float qjl_c = 1.2533141373155002512f / (float)D;   // sqrt(pi/2) / m, m = d

  const int range_lo = blockIdx.x * a.chunk;
  const int range_hi = min(range_lo + a.chunk, a.total_pages);
  if (range_lo >= range_hi) return;

  if (warp == 0) tmem_alloc(s_tmem, C::TALLOC);
  if (tid == 0) {
    for (int i = 0; i < NBUF + 2; ++i) mbar_init(&s_full[i], 1);
    *s_fail = 0;
    *s_rescale = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);   // this warp's lane quarter

  // softmax-weight operand constants of this token slot (value-plane bit position row >> 4)
  const int vk = row >> 4;
  const float v_beta = e4m3_beta(vk), v_gamma = e4m3_gamma(vk), v_igamma = 1.f / e4m3_gamma(vk);
  constexpr uint32_t idesc_s = make_idesc(0, 0, 128, NSC);
  constexpr uint32_t idesc_v = make_idesc(0, 0, 128, NVC);

  uint32_t fill_count = 0;   // pages issued into the ring (all segments)
  uint32_t waited = 0;       // ring fills this thread has seen complete
  uint32_t issued = 0;       // ring fills issued (thread 0)
  uint32_t n_s = 0, n_v = 0; // MMA groups committed on s_done / v_done (all segments)
  bool failed = false;

  auto fail_now = [&]() {
    if (lane == 0) atomicOr(a.status, kFlagTimeout);
    *s_fail = 1;
  };

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
    const int p_lo = seg_lo, n_pages = max(0, min(seg_hi, valid_pages) - p_lo);
    const int slot = blockIdx.x - (seq * PM) / a.chunk;
    float* rec = a.part + ((size_t)seq * a.slots + slot) * G * (2 + D);
    const uint8_t* seq_base = a.cache + (size_t)seq * PM * PL::bytes;

    __syncthreads();   // previous segment fully done with shared memory
    const uint32_t fill_base = fill_count;
    if (tid == 0) {
      const int first = min(n_pages, NBUF);
      issued = fill_base + first;
      for (int i = 0; i < first; ++i) {
        const uint32_t si = (fill_base + i) % NBUF;
        fence_proxy_async();
        mbar_expect_tx(&s_full[si], PL::bytes);
        bulk_g2s(s_pages + si * C::PAGE, seq_base + (size_t)(p_lo + i) * PL::bytes, PL::bytes, &s_full[si]);
      }
      for (int i = NBUF; i < min(n_pages, NBUF + kL2Ahead); ++i)
        prefetch_l2(seq_base + (size_t)(p_lo + i) * PL::bytes, PL::bytes);
    }
    fill_count = fill_base + n_pages;

    // ---- query operand of this KV head ----
    for (int e = tid; e < GP * 2 * D; e += kThreads) {
      const int hh = e / (2 * D), rem = e % (2 * D), which = rem / D, j = rem % D;
      float v = 0.f;
      if (hh < G) {
        const size_t r = (size_t)b * a.q_heads + (size_t)kvh * G + hh;
        v = (which == 0 ? a.qr : a.qs)[r * D + j];
      }
      s_q[e] = v;
    }
    for (int e = tid; e < GP * 8; e += kThreads) s_head[e] = 0.f;
    __syncthreads();
    for (int hh = warp; hh < GP; hh += kWarps) {   // power-of-two scales: largest operand <= 224
      float mk = 0.f, mq = 0.f;
      for (int j = lane; j < D; j += 32) {
        const float ig = 1.f / fabsf(e4m3_gamma(kpos_of(j)));
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
        const float bk = 2.f * amax * mk, bq = 2.f * mq;
        s_head[hh * 8 + 0] = bk > 0.f ? exp2f(floorf(log2f(224.f / bk))) : 1.f;
        s_head[hh * 8 + 1] = bq > 0.f ? exp2f(floorf(log2f(224.f / bq))) : 1.f;
      }
    }
    __syncthreads();
    // B_s[n][k], K-major canonical: k = plane * 128 + 4 * (8 w + kpos) + e <-> coordinate
    // slot_of_col(w, kpos, e); n = 3 h + piece (key term) or NHALF + 3 h + piece (sign term)
    for (int e4 = tid; e4 < NSC * NS * 32; e4 += kThreads) {
      const int n = e4 / (NS * 32), kw = e4 % (NS * 32);   // kw = 4-byte group index along K
      const int pl = kw / 32, col = kw % 32, w = col >> 3, kp = col & 7;
      int hh = -1, piece = 0;
      if (n < NHALF) {
        if (pl < PK) { hh = n / 3; piece = n % 3; }
      } else if (pl == PK) {
        hh = (n - NHALF) / 3;
        piece = (n - NHALF) % 3;
      }
      uint32_t word = 0u;
      if (hh >= 0 && hh < G) {
        const bool qj = pl == PK;
        const float sc = s_head[hh * 8 + (qj ? 1 : 0)];
        const float coef = qj ? 2.f : 2.f * a.alpha_k[pl];
        const float* qv = s_q + (hh * 2 + (qj ? 1 : 0)) * D;
        const float ig = 1.f / e4m3_gamma(kp);
#pragma unroll
        for (int el = 0; el < 4; ++el) {
          uint32_t p0, p1, p2;
          split3(coef * qv[slot_of_col(w, kp, el)] * sc * ig, p0, p1, p2);
          word |= (piece == 0 ? p0 : piece == 1 ? p1 : p2) << (8 * el);
        }
      }
      *reinterpret_cast<uint32_t*>(s_bs + canon_off(n, 4 * kw, NS * 128)) = word;
    }
    for (int hh = warp; hh < GP; hh += kWarps) {   // constants of the beta terms and plain sums
      float cmv = 0.f, cqv = 0.f, sk = 0.f, sq = 0.f;
      if (hh < G) {
        const float sck = s_head[hh * 8 + 0], scq = s_head[hh * 8 + 1];
        for (int j = lane; j < D; j += 32) {
          const int kp = kpos_of(j);
          const float beta = e4m3_beta(kp), ig = 1.f / e4m3_gamma(kp);
          const float qk = s_q[(hh * 2 + 0) * D + j], qq = s_q[(hh * 2 + 1) * D + j];
          sk += qk;
          sq += qq;
          for (int pl = 0; pl < PK; ++pl) {
            uint32_t p0, p1, p2;
            split3(2.f * a.alpha_k[pl] * qk * sck * ig, p0, p1, p2);
            cmv += beta * split3_val(p0, p1, p2);
          }
          uint32_t p0, p1, p2;
          split3(2.f * qq * scq * ig, p0, p1, p2);
          cqv += beta * split3_val(p0, p1, p2);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        cmv += __shfl_xor_sync(0xffffffffu, cmv, o);
        cqv += __shfl_xor_sync(0xffffffffu, cqv, o);
        sk += __shfl_xor_sync(0xffffffffu, sk, o);
        sq += __shfl_xor_sync(0xffffffffu, sq, o);
      }
      if (lane == 0) {
        s_head[hh * 8 + 2] = cmv;
        s_head[hh * 8 + 3] = cqv;
        s_head[hh * 8 + 4] = sk;
        s_head[hh * 8 + 5] = sq;
      }
    }
    fence_proxy_async();   // B_s is read by the tensor cores
    __syncthreads();

    // ---- running state (token warps; identical in every token thread) ----
    float m_run[GP], l_part[GP], c_part[GP], g_part[GP];
#pragma unroll
    for (int h = 0; h < GP; ++h) {
      m_run[h] = -INFINITY;
      l_part[h] = c_part[h] = g_part[h] = 0.f;
    }
    float n_ref = 0.f;

    auto wait_full = [&](int p) {
      const uint32_t fi = fill_base + p;
      if (mbar_wait(&s_full[fi % NBUF], (fi / NBUF) & 1)) {
        if (fi + 1 > waited) waited = fi + 1;
      } else {
        fail_now();
      }
    };
    // plane warps: key planes and sign plane of token `row` of page p -> A_s
    auto load_keys = [&](int p) {
      const uint8_t* pg = s_pages + ((fill_base + p) % NBUF) * C::PAGE;
      uint4 wk[BK];
#pragma unroll
      for (int q = 0; q < BK; ++q)
        wk[q] = *reinterpret_cast<const uint4*>(pg + PL::off_kcodes + ((size_t)q * 128 + row) * 16);
      const uint4 wsg = *reinterpret_cast<const uint4*>(pg + PL::off_signs + (size_t)row * 16);
#pragma unroll
      for (int pl = 0; pl < NS; ++pl) {
        uint32_t x[4];
        if (pl < PK) {
          x[0] = x[1] = x[2] = x[3] = 0u;
#pragma unroll
          for (int q = 0; q < BK; ++q)
            if ((mono_mask16(pl) >> q) & 1) {
              x[0] ^= wk[q].x;
              x[1] ^= wk[q].y;
              x[2] ^= wk[q].z;
              x[3] ^= wk[q].w;
            }
        } else {
          x[0] = wsg.x;
          x[1] = wsg.y;
          x[2] = wsg.z;
          x[3] = wsg.w;
        }
        uint32_t r[32];
#pragma unroll
        for (int w = 0; w < 4; ++w)
#pragma unroll
          for (int k = 0; k < 8; ++k) r[8 * w + k] = expand_at(x[w], k);
        tmem_st32(tl + C::TA_S + 32 * pl, r);
      }
    };
    // plane warps: value planes of coordinate `row` of page p -> A_v
    auto load_values = [&](int p) {
      const uint8_t* pg = s_pages + ((fill_base + p) % NBUF) * C::PAGE;
      uint4 wv[BV];
#pragma unroll
      for (int q = 0; q < BV; ++q)
        wv[q] = *reinterpret_cast<const uint4*>(pg + PL::off_vcodes + ((size_t)q * D + row) * 16);
#pragma unroll
      for (int pl = 0; pl < PV; ++pl) {
        uint32_t x[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int q = 0; q < BV; ++q)
          if ((mono_mask16(pl) >> q) & 1) {
            x[0] ^= wv[q].x;
            x[1] ^= wv[q].y;
            x[2] ^= wv[q].z;
            x[3] ^= wv[q].w;
          }
        uint32_t r[32];
#pragma unroll
        for (int w = 0; w < 4; ++w)
#pragma unroll
          for (int k = 0; k < 8; ++k) r[8 * w + k] = expand_at(x[w], k);
        tmem_st32(tl + C::TA_V + 32 * pl, r);
      }
    };
    auto issue_score = [&]() {   // elected thread
      tc_fence_after();
#pragma unroll 1
      for (int ks = 0; ks < NS * 4; ++ks) {
        const uint64_t bd = smem_desc(smem_u32(s_bs) + ks * 256, 128, NS * 1024);
        mma_f8_ts(tmem + C::TD_S, tmem + C::TA_S + 8 * ks, bd, idesc_s, ks > 0);
      }
      tc_commit(s_sdone);
    };
    auto issue_values = [&](bool first_page) {   // elected thread
      tc_fence_after();
#pragma unroll 1
      for (int pl = 0; pl < PV; ++pl)
#pragma unroll 1
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t bd = smem_desc(smem_u32(s_bv) + ks * 256, 128, 1024);
          mma_f8_ts(tmem + C::TD_V + pl * NVC, tmem + C::TA_V + 32 * pl + 8 * ks, bd, idesc_v,
                    !(first_page && ks == 0));
        }
      tc_commit(s_vdone);
    };

    if (n_pages > 0) {
      // prologue: plane warps put the keys of page 0 into A_s
      if (!tok) {
        wait_full(0);
        load_keys(0);
        tc_wait_st();
      }
      tc_fence_before();
      __syncthreads();
      if (tid == 0) issue_score();
      ++n_s;

      for (int p = 0; p < n_pages; ++p) {
        const uint8_t* pg = s_pages + ((fill_base + p) % NBUF) * C::PAGE;
        if (tok) {
          // ---------- token warps: logits, lazy softmax, softmax-weight operand ----------
          wait_full(p);
          if (!mbar_wait(s_sdone, (n_s - 1) & 1)) fail_now();
          tc_fence_after();
          float ds[NSC];
#pragma unroll
          for (int c0 = 0; c0 < NSC; c0 += 16) {
            uint32_t r[16];
            tmem_ld16(tl + C::TD_S + c0, r);
            tc_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) ds[c0 + i] = __uint_as_float(r[i]);
          }
          const int nvalid = min(128, seq_len - (p_lo + p) * 128);
          const bool valid = row < nvalid;
          const float nk = valid ? reinterpret_cast<const float*>(pg + PL::off_nk)[row] : 0.f;
          const float gmv = valid ? reinterpret_cast<const float*>(pg + PL::off_gamma)[row] : 0.f;
          const float nvt = valid ? reinterpret_cast<const float*>(pg + PL::off_nv)[row] : 0.f;
          float lg[GP];
          int ovf = nvt > n_ref;
#pragma unroll
          for (int h = 0; h < GP; ++h) {
            const float* hp = s_head + h * 8;
            const float mse = ds[3 * h] + 0.0625f * ds[3 * h + 1] + 0.00390625f * ds[3 * h + 2];
            const float qjl = ds[NHALF + 3 * h] + 0.0625f * ds[NHALF + 3 * h + 1] + 0.00390625f * ds[NHALF + 3 * h + 2];
            const float dk = (mse - hp[2]) / hp[0] - a.asum_k * hp[4];
            const float dq = (qjl - hp[3]) / hp[1] - hp[5];
            const float l = (nk * dk + gmv * qjl_c * dq) * inv_sqrt_d;
            lg[h] = (valid && h < G) ? l : -INFINITY;
            if (a.logits && valid && h < G)
              a.logits[((size_t)b * a.q_heads + (size_t)kvh * G + h) * a.max_tokens + (size_t)(p_lo + p) * 128 + row] = l;
            if (lg[h] > m_run[h] + kTau) ovf = 1;
          }
          if (t_vote_or(ovf)) {
            // exact page maxima over the 128 token threads, new references, rescale factors
#pragma unroll
            for (int h = 0; h <= GP; ++h) {
              float mx = h < GP ? lg[h] : nvt;
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
              if (lane == 0) s_red[warp * (GP + 1) + h] = mx;
            }
            t_sync();
            float nvmax = 0.f;
            for (int w2 = 0; w2 < 4; ++w2) nvmax = fmaxf(nvmax, s_red[w2 * (GP + 1) + GP]);
            const float n_new = nvmax > n_ref ? 1.25f * nvmax : n_ref;
#pragma unroll
            for (int h = 0; h < GP; ++h) {
              float mx = -INFINITY;
              for (int w2 = 0; w2 < 4; ++w2) mx = fmaxf(mx, s_red[w2 * (GP + 1) + h]);
              const float m_new = fmaxf(m_run[h], mx);
              const float alpha = (m_run[h] == -INFINITY) ? 0.f : __expf(m_run[h] - m_new);
              const float f = (n_ref > 0.f) ? alpha * (n_ref / n_new) : 0.f;
              l_part[h] *= alpha;
              c_part[h] *= f;
              g_part[h] *= f;
              if (tid == 0) s_f[h] = f;
              m_run[h] = m_new;
            }
            n_ref = n_new;
            if (tid == 0) *s_rescale = 1;
            t_sync();   // s_red reads done
          } else if (tid == 0) {
            *s_rescale = 0;
          }
          // softmax weights -> two e4m3 pieces per head; the byte for row n = 2h + piece
          const float inv_n = n_ref > 0.f ? 1.f / n_ref : 0.f;
          const float xs = nvt * inv_n * v_igamma * kSB;
          uint32_t wb[NVC / 4];
#pragma unroll
          for (int i = 0; i < NVC / 4; ++i) wb[i] = 0u;
#pragma unroll
          for (int h = 0; h < GP; ++h) {
            const float pr = lg[h] == -INFINITY ? 0.f : __expf(lg[h] - m_run[h]);
            l_part[h] += pr;
            const float x = pr * xs;
            const uint32_t hi = cvt_e4m3x2(0.f, x) & 0xFF;
            const float hf = e4m3x2_to_f2(hi).x;
            const uint32_t lo = cvt_e4m3x2(0.f, 16.f * (x - hf)) & 0xFF;
            const float bsum = hf + 0.0625f * e4m3x2_to_f2(lo).x;
            c_part[h] += v_beta * bsum;
            g_part[h] += v_gamma * bsum;
            wb[(2 * h) >> 2] |= hi << (8 * ((2 * h) & 3));
            wb[(2 * h + 1) >> 2] |= lo << (8 * ((2 * h + 1) & 3));
          }
          // 4 x 4 byte transposes across the 4 lanes holding tokens 4i .. 4i+3: lane e of the
          // group ends up with row 4 r + e, bytes = those 4 tokens
          const int e = lane & 3, base = lane & ~3;
          const int k0 = 32 * ((row >> 2) & 3) + 4 * (row >> 4);   // K byte of token 4i
          // B_v of the previous page is read by its value MMA: wait for it
          if (p > 0 && !mbar_wait(s_vdone, (n_v - 1) & 1)) fail_now();
#pragma unroll
          for (int r4 = 0; r4 < NVC / 4; ++r4) {
            const uint32_t w0 = __shfl_sync(0xffffffffu, wb[r4], base + 0);
            const uint32_t w1 = __shfl_sync(0xffffffffu, wb[r4], base + 1);
            const uint32_t w2 = __shfl_sync(0xffffffffu, wb[r4], base + 2);
            const uint32_t w3 = __shfl_sync(0xffffffffu, wb[r4], base + 3);
            const uint32_t sel = (uint32_t)e | ((uint32_t)(e + 4) << 4);
            const uint32_t t01 = __byte_perm(w0, w1, sel), t23 = __byte_perm(w2, w3, sel);
            const uint32_t outw = __byte_perm(t01, t23, 0x5410);
            *reinterpret_cast<uint32_t*>(s_bv + canon_off(4 * r4 + e, k0, 128)) = outw;
          }
          fence_proxy_async();
        } else {
          // ---------- plane warps: values of page p, keys of page p+1 ----------
          if (p > 0) {
            if (!mbar_wait(s_vdone, (n_v - 1) & 1)) fail_now();   // A_v free
            tc_fence_after();
          }
          load_values(p);
          if (p + 1 < n_pages) {
            wait_full(p + 1);
            if (!mbar_wait(s_sdone, (n_s - 1) & 1)) fail_now();   // A_s free
            tc_fence_after();
            load_keys(p + 1);
          }
          tc_wait_st();
        }
        tc_fence_before();
        __syncthreads();
        if (*s_fail) {
          failed = true;
          break;
        }
        if (*s_rescale && p > 0) {
          // D_v holds pages < p (their MMAs are complete): scale it by the new references
          if (!tok) {
#pragma unroll 1
            for (int c0 = 0; c0 < PV * NVC; c0 += 16) {
              uint32_t r[16];
              tmem_ld16(tl + C::TD_V + c0, r);
              tc_wait_ld();
#pragma unroll
              for (int i = 0; i < 16; ++i) {
                const int h = ((c0 + i) % NVC) >> 1;
                r[i] = __float_as_uint(h < GP ? __uint_as_float(r[i]) * s_f[h] : 0.f);
              }
              tmem_st16(tl + C::TD_V + c0, r);
            }
            tc_wait_st();
          }
          tc_fence_before();
          __syncthreads();
        }
        if (tid == 0) {
          issue_values(p == 0);
          if (p + 1 < n_pages) issue_score();
          // ring slot of page p is free: refill
          const int nxt = p + NBUF;
          if (nxt < n_pages) {
            issued = fill_base + nxt + 1;
            const uint32_t si = (fill_base + nxt) % NBUF;
            fence_proxy_async();
            mbar_expect_tx(&s_full[si], PL::bytes);
            bulk_g2s(s_pages + si * C::PAGE, seq_base + (size_t)(p_lo + nxt) * PL::bytes, PL::bytes, &s_full[si]);
          }
          if (nxt + kL2Ahead < n_pages) prefetch_l2(seq_base + (size_t)(p_lo + nxt + kL2Ahead) * PL::bytes, PL::bytes);
        }
        ++n_v;
        if (p + 1 < n_pages) ++n_s;
      }
    }
    if (failed) break;

    // ---------- segment epilogue ----------
    if (tid == 0) s_f[GP] = n_ref;   // the plane warps need the value-norm reference
    if (tok) {
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        float v3[3] = {l_part[h], c_part[h], g_part[h]};
#pragma unroll
        for (int c = 0; c < 3; ++c) {
          float v = v3[c];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == 0) s_red[(warp * (GP + 1) + h) * 3 + c] = v;
        }
      }
    }
    __syncthreads();
    if (tok && tid < GP && tid < G) {
      float l_tot = 0.f;
      for (int w2 = 0; w2 < 4; ++w2) l_tot += s_red[(w2 * (GP + 1) + tid) * 3];
      float* rh = rec + (size_t)tid * (2 + D);
      rh[0] = m_run[tid];
      rh[1] = l_tot;
    }
    if (!tok) {
      float ov[GP];
#pragma unroll
      for (int h = 0; h < GP; ++h) ov[h] = 0.f;
      if (n_pages > 0) {
        if (!mbar_wait(s_vdone, (n_v - 1) & 1)) fail_now();
        tc_fence_after();
#pragma unroll 1
        for (int pl = 0; pl < PV; ++pl) {
          const float al = a.alpha_v[pl];
#pragma unroll
          for (int c0 = 0; c0 < NVC; c0 += 16) {
            uint32_t r[16];
            tmem_ld16(tl + C::TD_V + pl * NVC + c0, r);
            tc_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
              const int h = (c0 + i) >> 1;
              if (h < GP) ov[h] += al * (__uint_as_float(r[i]) + 0.0625f * __uint_as_float(r[i + 1]));
            }
          }
        }
      }
      const float nref = s_f[GP];
      const float scale = nref > 0.f ? nref / kSB : 0.f;
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        if (h >= G) continue;
        float c_tot = 0.f, g_tot = 0.f;
        for (int w2 = 0; w2 < 4; ++w2) {
          c_tot += s_red[(w2 * (GP + 1) + h) * 3 + 1];
          g_tot += s_red[(w2 * (GP + 1) + h) * 3 + 2];
        }
        float asum = 0.f;
        for (int pl = 0; pl < PV; ++pl) asum += a.alpha_v[pl];
        // o~_j = (n_ref / kSB) [ 2 sum_M alpha_M (D_M - C) - sum alpha G ]
        const float o = scale * (2.f * (ov[h] - asum * c_tot) - a.asum_v * g_tot);
        rec[(size_t)h * (2 + D) + 2 + row] = n_pages > 0 ? o : 0.f;
      }
    }
  }
  // teardown: outstanding copies and MMAs complete (bounded), then free tensor memory
  if (failed && tid == 0) {
    for (uint32_t i = waited; i < issued; ++i) mbar_wait(&s_full[i % NBUF], (i / NBUF) & 1);
    if (n_s > 0) mbar_wait(s_sdone, (n_s - 1) & 1);
    if (n_v > 0) mbar_wait(s_vdone, (n_v - 1) & 1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TALLOC);
  }
}

}  // namespace dtc
}  // namespace tq
