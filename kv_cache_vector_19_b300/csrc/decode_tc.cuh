// tq_attn_decode on 5th-generation tensor cores (tcgen05, kind::f8f6f4), head_dim 128.
//
// Same arithmetic as the mma.sync kernel (decode_mma.cuh): the score of a cached key and
// the value accumulation are contractions over bit planes of the codes, each plane word
// turned into e4m3 operands beta_k + gamma_k * bit by one AND-OR (bitplane.h), the per-
// position scales folded into the other operand.  What changes is where the MMAs run:
//   A_s (smem, K-major, x2)       key planes and the sign plane of one page (row = token),
//                                 NS x 128 bytes per row
//   B_s (smem, K-major)           query pieces: 4 e4m3 pieces per head for the key term and
//                                 4 for the sign term (columns), one row block per plane
//   D_s (TMEM, lane = token, x2)  score partial sums, read back by the token warps
//   A_v (TMEM, lane = coordinate, x2) value planes of one page, PV x 128 bytes
//   B_v (smem, K-major, x2)       softmax weights of the page, 2 e4m3 pieces per head
//   D_v (TMEM, lane = coordinate) one accumulator per value plane, restarted every kFlush pages
//   D_acc (TMEM)                  fp32 running total of the flushed D_v stretches
// Every per-page operand is double-buffered, so each producer / consumer pair has two pages
// in flight and hands over once per page: a hand-off costs a few hundred cycles on B300, and
// chains with one page in flight were what bounded earlier versions of this kernel.
//
// Warp roles, 20 warps, handing work over through mbarriers (no CTA barrier per page):
//   warps 0-3, 16-19  token warps (TMEM lane = token), two sets each owning half of the query
//               heads: read D_s, form logits, run the lazy online softmax, write B_v and, when
//               the running maximum moves or a stretch ends, rescale or flush D_v
//   warps 4-7   key-plane warps (row = token): key XOR planes and the sign plane -> A_s
//   warps 8-11  value-plane warps (lane = coordinate): value XOR planes -> A_v; epilogue
//   warp 12     issues the score MMAs (12 per page at b = 3), warp 13 the value MMAs (16)
//   warps 14-15 wait for the operands of the two issuers; warp 15 also refills the page ring
// A tcgen05.mma of M = 128, K = 32 costs ~46 cycles for any N up to 64 on B300 (two issuing
// threads overlap to ~38): the 28 MMAs of a page (b = 3) are the floor of this kernel.  Inside
// this kernel, beside 16 working warps, each issuer spends ~100-130 cycles per MMA.
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

// Warp numbering: every 4-warp role starts at a multiple of 4 (warp % 4 is the TMEM lane
// quarter a warp may access).  Measured on B300: the order of the 4-warp roles makes no
// difference (within 0.5%); with the issuers and waiters in warps 0-3 instead of 12-15 the
// kernel ran 2-12% slower.
constexpr int kWarpT = 0;             // token warps, first set (4)
constexpr int kWarpK = 4;             // key-plane warps (4)
constexpr int kWarpV = 8;             // value-plane warps (4); epilogue
constexpr int kWarpS = 12;            // issues the score MMAs
constexpr int kWarpM = 13;            // issues the value MMAs
constexpr int kWarpWS = 14;           // waits for the score operands, hands them to kWarpS
constexpr int kWarpWM = 15;           // waits for the value operands, hands them to kWarpM; page ring
constexpr int kWarpT2 = 16;           // token warps, second set (4)
constexpr int kWarpsAll = 20;
static_assert(kWarpT == 0, "the segment's n_ref is stored by thread 0 as the first token thread");
constexpr int kL2Ahead = 12;
constexpr float kTau = 3.0f;          // lazy-maximum threshold (natural-log units)
constexpr float kSB = 2.0f;           // e4m3 range scale of the softmax weights
// The value accumulator D_v restarts every kFlush pages after the token warps add it into
// D_acc in fp32: the tensor core's accumulation rounds at a coarser grain than fp32, and over
// 10^3 pages (the beta offsets of the bit-plane operands keep D_v large) that rounding
// reached 1e-2 of the output; restarted every 32 pages the output stays within ~7e-4.
constexpr int kFlush = 32;
constexpr int kSmemMax = 227 * 1024;

__host__ __device__ constexpr int rnd(int x, int m) { return (x + m - 1) / m * m; }

template <int BITS, int GP>
struct Cfg {
  static constexpr int D = 128;
  using PL = PageLayout<128, BITS>;
  static constexpr int BK = BITS - 1, BV = BITS;
  static constexpr int PK = 1 << (BK - 1), PV = 1 << (BV - 1), NS = PK + 1;
  // token warps: TS = 2 sets of four (one warp per TMEM lane quarter); set s handles the HPT
  // query heads from head s * HPT (set 0 is warps 0-3, set 1 warps 16-19).  Two sets halve
  // each token thread's chain of per-head work on every page, which is the longest chain of
  // the per-page loop.
  static constexpr int TS = 2;
  static constexpr int HPT = GP / TS;
  static constexpr int WARPS = kWarpsAll;
  static constexpr int THREADS = 32 * WARPS;
  static constexpr int NQP = 4;                          // e4m3 pieces per query coordinate
  static constexpr int NHALF = rnd(NQP * GP, 8);       // score columns: [key term | sign term]
  static constexpr int NSC = rnd(2 * NHALF, 16);
  static constexpr int NPW = 2;                           // e4m3 pieces per softmax weight
  static constexpr int NVC = NPW * GP < 16 ? 16 : NPW * GP;  // value columns: hi, lo per head
  // tensor memory: D_s (x2 when it fits), D_v (this stretch of pages), D_acc (fp32 total of
  // the flushed stretches), A_v (x2 when it fits)
  static constexpr int DS_COLS = rnd(NSC, 32);
  static constexpr int DV_COLS = rnd(PV * NVC, 32);
  static constexpr int AV_COLS = PV * 32;
  static constexpr int DSB = 2 * DS_COLS + 2 * DV_COLS + 2 * AV_COLS <= 512 ? 2 : 1;
  static constexpr int AVB = DSB * DS_COLS + 2 * DV_COLS + 2 * AV_COLS <= 512 ? 2 : 1;
  static constexpr int TD_S = 0;
  static constexpr int TD_V = DSB * DS_COLS;
  static constexpr int TD_ACC = TD_V + DV_COLS;
  static constexpr int TA_V = TD_ACC + DV_COLS;
  static constexpr int TCOLS = TA_V + AVB * AV_COLS;
  static constexpr int TALLOC = TCOLS <= 256 ? 256 : 512;
  // shared memory: A_s (key planes, K-major canonical, double-buffered), B_s, B_v (x2), q,
  // per-head constants, reductions, mbarriers, then as many ring pages as fit (<= 8)
  static constexpr int PAGE = PL::bytes;
  static constexpr int AS_BYTES = 128 * NS * 128;                // per buffer
  static constexpr int BS_BYTES = NSC * NS * 128;
  static constexpr int BV_BYTES = NVC * 128;                     // per buffer
  static constexpr int OFF_AS = 0;
  static constexpr int OFF_BS = OFF_AS + 2 * AS_BYTES;
  static constexpr int OFF_BV = OFF_BS + BS_BYTES;
  static constexpr int OFF_Q = OFF_BV + 2 * BV_BYTES;            // [GP][2][128] f32
  static constexpr int OFF_HEAD = OFF_Q + GP * 2 * 128 * 4;      // [GP][8] f32
  static constexpr int OFF_RED = OFF_HEAD + GP * 8 * 4;          // [4 TS token warps][HPT + 1][3] f32
  static constexpr int OFF_F = OFF_RED + 4 * TS * (HPT + 1) * 3 * 4;   // n_ref of the segment
  static constexpr int OFF_MBAR = rnd(OFF_F + 16, 8);
  // full[8], empty[8], as_ready[2], as_free[2], s_fin[2], ds_free[2], av_ready[2], v_fin[2],
  // bv_ready[2], teardown[2]
  static constexpr int NMBAR = 16 + 16;
  static constexpr int OFF_MISC = OFF_MBAR + NMBAR * 8;          // tmem base, fail
  static constexpr int OFF_PAGES = rnd(OFF_MISC + 16, 128);
  static constexpr int NBUF_FIT = (kSmemMax - OFF_PAGES) / PAGE;
  static constexpr int NBUF = NBUF_FIT > 8 ? 8 : NBUF_FIT;
  static constexpr int SMEM = OFF_PAGES + NBUF * PAGE;
  static constexpr bool SUPPORTED = TCOLS <= 512 && SMEM <= kSmemMax && NBUF >= 4;
};

// OR-vote / barrier among the token warps (named barrier 1, NT = 128 or 256 threads).
template <int NT>
__device__ __forceinline__ int t_vote_or(int pred) {
  int r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.s32 q, %1, 0;\n barrier.cta.red.or.pred p, 1, %2, q;\n selp.s32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"(pred), "n"(NT)
      : "memory");
  return r;
}
template <int NT>
__device__ __forceinline__ void t_sync() { asm volatile("barrier.cta.sync 1, %0;" ::"n"(NT) : "memory"); }

// The two MMA-issuing warps never wait on an mbarrier: on B300 a shared-memory access by a
// thread with MMAs in flight (an mbarrier wait included) stalls it for hundreds of cycles,
// while a named barrier does not.  A waiter warp polls the mbarriers (bounded waits) and then
// meets its issuer at a named barrier that both sync, so the two stay in lock step and every
// sync has a partner even after a timeout.  Ids: 1 token-warp sync, 2 score pair, 3 value pair.
constexpr int kNbScore = 2;
constexpr int kNbValue = 3;
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void pair_sync(int id) {
  __syncwarp();
  asm volatile("barrier.cta.sync.aligned %0, 64;" ::"r"(id) : "memory");
}

// bit position (0..7) of coordinate or token slot x within its plane word
__host__ __device__ __forceinline__ int kpos_of(int x) { return 2 * (x >> 5) + ((x >> 4) & 1); }
// coordinate / token slot held by byte e of operand column (w * 8 + k) of a plane
__host__ __device__ __forceinline__ int slot_of_col(int w, int k, int e) {
  return 32 * (k >> 1) + 16 * (k & 1) + 4 * w + e;
}

// xp[pl] for a runtime plane index (predicated selects; keeps the plane loop rolled).
template <int NP>
__device__ __forceinline__ void pick_plane(const uint4 (&xp)[NP], int pl, uint32_t (&x)[4]) {
  uint4 v = xp[0];
#pragma unroll
  for (int i = 1; i < NP; ++i)
    if (pl == i) v = xp[i];
  x[0] = v.x;
  x[1] = v.y;
  x[2] = v.z;
  x[3] = v.w;
}

// One row of a plane: four plane words expanded to the 32 e4m3 operand words (128 bytes).
__device__ __forceinline__ void expand_words(const uint32_t (&x)[4], uint32_t (&r)[32]) {
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int k = 0; k < 8; ++k) r[8 * c + k] = expand_at(x[c], k);
}

template <int BITS, int GP, bool PAGED>
__global__ void __launch_bounds__(Cfg<BITS, GP>::THREADS, 1) decode_tc_kernel(Params a, PageMap pm, float sparse_v) {
  using C = Cfg<BITS, GP>;
  using PL = typename C::PL;
  constexpr int D = 128, NS = C::NS, PK = C::PK, PV = C::PV, BK = C::BK, BV = C::BV, NBUF = C::NBUF;
  constexpr int NSC = C::NSC, NVC = C::NVC, NHALF = C::NHALF, DSB = C::DSB, NPW = C::NPW, AVB = C::AVB;
  constexpr int TS = C::TS, HPT = C::HPT, kThreads = C::THREADS, kWarps = C::WARPS, TNT = 128 * TS;
  // TMEM access widths of the split token warps: this set's score columns, value columns
  constexpr int CKS = 4 * HPT < 16 ? 4 * HPT : 16, CKV = NPW * HPT < 8 ? NPW * HPT : 8;
  extern __shared__ __align__(1024) unsigned char smem[];
  uint8_t* s_pages = smem + C::OFF_PAGES;
  uint8_t* s_as = smem + C::OFF_AS;
  uint8_t* s_bs = smem + C::OFF_BS;
  uint8_t* s_bv = smem + C::OFF_BV;
  float* s_q = reinterpret_cast<float*>(smem + C::OFF_Q);
  float* s_head = reinterpret_cast<float*>(smem + C::OFF_HEAD);
  float* s_red = reinterpret_cast<float*>(smem + C::OFF_RED);
  float* s_f = reinterpret_cast<float*>(smem + C::OFF_F);
  uint64_t* mb = reinterpret_cast<uint64_t*>(smem + C::OFF_MBAR);
  // Every hand-off barrier below exists once per buffer (index = page & 1) and completes once
  // per page of that parity, and every waiter has waited the previous completion: a parity
  // wait can therefore never mistake an older phase for a newer one.
  uint64_t* s_full = mb;            // [8]  page in ring slot landed (+ tx bytes)
  uint64_t* s_empty = mb + 8;       // [8]  page read by every consumer warp (8 + 4 TS)
  uint64_t* as_ready = mb + 16;     // [2]  key planes of the page stored in A_s (4 warps)
  uint64_t* as_free = mb + 18;      // [2]  score MMAs reading that A_s buffer done (commit)
  uint64_t* s_fin = mb + 20;        // [2]  score MMAs into that D_s buffer done (commit)
  uint64_t* ds_free = mb + 22;      // [2]  D_s buffer read by the token warps (4)
  uint64_t* av_ready = mb + 24;     // [2]  value planes stored in that A_v buffer (4 warps)
  uint64_t* v_fin = mb + 26;        // [2]  value MMAs of the page done (commit)
  uint64_t* bv_ready = mb + 28;     // [2]  B_v buffer written, D_v rescaled (4 warps)
  uint64_t* td_bar = mb + 30;       // [2]  teardown drains of the two MMA issuers
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* s_fail = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = 32 * (warp & 3) + lane;    // TMEM lane / operand row of this thread (4-warp roles)
  const int G = a.group, PM = a.pages_per_seq;
  const float inv_sqrt_d = rsqrtf((float)D);
  const float qjl_c = 1.2533141373155002512f / (float)D;   // sqrt(pi/2) / m, m = d

  const int range_lo = blockIdx.x * a.chunk;
  const int range_hi = min(range_lo + a.chunk, a.total_pages);
  if (range_lo >= range_hi) return;

  if (warp == 0) tmem_alloc(s_tmem, C::TALLOC);
  if (tid == 0) {
    for (int i = 0; i < 8; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 8 + 4 * TS);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&as_ready[i], 4);
      mbar_init(&as_free[i], 1);
      mbar_init(&s_fin[i], 1);
      mbar_init(&ds_free[i], 4 * TS);
      mbar_init(&av_ready[i], 4);
      mbar_init(&v_fin[i], 1);
      mbar_init(&bv_ready[i], 4 * TS);
      mbar_init(&td_bar[i], 1);
    }
    *s_fail = 0;
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

  uint32_t pg_base = 0;      // pages (== ring fills) of the previous segments
  uint32_t issued = 0;       // ring fills issued (value-waiter lane)

  auto fail_now = [&]() {
    if (lane == 0) atomicOr(a.status, kFlagTimeout);
    *s_fail = 1;
  };
  // Bounded wait for the k-th completion (0-based) of a barrier.  Once a wait timed out every
  // later wait returns at once: all roles still run their loops to the end, so the paired
  // named-barrier counts stay balanced and the kernel finishes.
  auto wait_k = [&](uint64_t* bar, uint32_t k) {
    if (*s_fail) return;
    if (!mbar_wait(bar, k & 1)) fail_now();
  };

  int gp = range_lo;
  bool s_fail_seen = false;   // read after a CTA barrier, so uniform
  while (gp < range_hi && !s_fail_seen) {
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
    // page p of this sequence: contiguous, or through the block table (PAGED, a separate
    // instantiation so that the contiguous kernel's address arithmetic stays as it was)
    const uint8_t* seq_base = a.cache + (size_t)seq * PM * PL::bytes;
    auto page_g = [&](int p) -> const uint8_t* {
      if constexpr (PAGED) return a.cache + pm.index(seq, a.kv_heads, PM, p, a.status) * PL::bytes;
      else return seq_base + (size_t)p * PL::bytes;
    };
    // ring slot / use of the page with segment index p (ring fills are counted over segments)
    auto ring_slot = [&](int p) { return (pg_base + p) % NBUF; };
    auto ring_use = [&](int p) { return (pg_base + p) / NBUF; };
    auto pg_ptr = [&](int p) { return s_pages + ring_slot(p) * C::PAGE; };

    __syncthreads();   // previous segment fully done
    if (warp == kWarpWM && lane == 0) {
      const int first = min(n_pages, NBUF);
      for (int i = 0; i < first; ++i) {
        const uint32_t si = ring_slot(i);
        fence_proxy_async();
        mbar_expect_tx(&s_full[si], PL::bytes);
        bulk_g2s(s_pages + si * C::PAGE, page_g(p_lo + i), PL::bytes, &s_full[si]);
      }
      issued = pg_base + first;
      for (int i = NBUF; i < min(n_pages, NBUF + kL2Ahead); ++i)
        prefetch_l2(page_g(p_lo + i), PL::bytes);
    }

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
    // both B_v buffers start at zero: the padding rows past 2 GP (N is at least 16) stay zero,
    // the token warps rewrite only the rows of their heads on every page
    for (int e = tid; e < 2 * C::BV_BYTES / 4; e += kThreads) reinterpret_cast<uint32_t*>(s_bv)[e] = 0u;
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
    // slot_of_col(w, kpos, e); n = 4 h + piece (key term) or NHALF + 4 h + piece (sign term)
    for (int e4 = tid; e4 < NSC * NS * 32; e4 += kThreads) {
      const int n = e4 / (NS * 32), kw = e4 % (NS * 32);   // kw = 4-byte group index along K
      const int pl = kw / 32, col = kw % 32, w = col >> 3, kp = col & 7;
      int hh = -1, piece = 0;
      if (n < NHALF) {
        if (pl < PK) { hh = n / 4; piece = n % 4; }
      } else if (pl == PK) {
        hh = (n - NHALF) / 4;
        piece = (n - NHALF) % 4;
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
          uint32_t pc[4];
          split4(coef * qv[slot_of_col(w, kp, el)] * sc * ig, pc);
          word |= (piece == 0 ? pc[0] : piece == 1 ? pc[1] : piece == 2 ? pc[2] : pc[3]) << (8 * el);
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
            uint32_t pc[4];
            split4(2.f * a.alpha_k[pl] * qk * sck * ig, pc);
            cmv += beta * split4_val(pc);
          }
          uint32_t pc[4];
          split4(2.f * qq * scq * ig, pc);
          cqv += beta * split4_val(pc);
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

    // token-warp form of the per-head constants.  From the set-up values s_k, s_q (operand
    // scales), C_k, C_q (beta-term constants), sum q~ and sum q_s:
    //   <q~, c[idx]> = (mse - C_k) / s_k - asum_k sum q~,  <q_s, 2 sigma - 1> = (qjl - C_q) / s_q - sum q_s,
    //   logit = (n_k <q~, c[idx]> + gamma sqrt(pi/2)/m <q_s, 2 sigma - 1>) / sqrt(d)
    //         = n_k (mse ak + bk) + gamma (qjl aq + bq).
    for (int hh = tid; hh < GP; hh += kThreads) {
      float* hp = s_head + hh * 8;
      const float sk = hp[0], sq = hp[1], ck = hp[2], cq = hp[3], sumk = hp[4], sumq = hp[5];
      hp[0] = inv_sqrt_d / sk;
      hp[1] = (-ck / sk - a.asum_k * sumk) * inv_sqrt_d;
      hp[2] = qjl_c * inv_sqrt_d / sq;
      hp[3] = (-cq / sq - sumq) * qjl_c * inv_sqrt_d;
    }
    __syncthreads();



    if (n_pages > 0) {
      if (warp == kWarpWS) {
        // ============ score waiter: A_s(g) stored and D_s buffer free -> meet the score issuer ============
        for (int p = 0; p < n_pages; ++p) {
          const uint32_t g = pg_base + p, x = g & 1;
          wait_k(&as_ready[x], g >> 1);
          if (DSB == 2 && g >= 2) wait_k(&ds_free[x], (g >> 1) - 1);
          if (DSB == 1 && g >= 1) wait_k(&ds_free[(g - 1) & 1], (g - 1) >> 1);
          pair_sync(kNbScore);
        }
      } else if (warp == kWarpS) {
        // ============ score MMAs: D_s[token][column] = A_s[token][plane, coordinate] x B_s ============
        const uint32_t bs = smem_u32(s_bs);
        for (int p = 0; p < n_pages; ++p) {
          const uint32_t g = pg_base + p, x = g & 1, db = DSB == 2 ? x : 0;
          pair_sync(kNbScore);
          if (lane == 0) {
            tc_fence_after();
            const uint32_t as = smem_u32(s_as + x * C::AS_BYTES);
#pragma unroll
            for (int ks = 0; ks < NS * 4; ++ks)
              mma_f8_ss(tmem + C::TD_S + db * C::DS_COLS, smem_desc(as + ks * 256, 128, NS * 1024),
                        smem_desc(bs + ks * 256, 128, NS * 1024), idesc_s, ks > 0);
            tc_commit(&as_free[x]);
            tc_commit(&s_fin[x]);
          }
        }
      } else if (warp == kWarpWM) {
        // ============ value waiter: A_v(g), B_v(g) ready -> meet the value issuer; ring refills ============
        for (int p = 0; p < n_pages; ++p) {
          const uint32_t g = pg_base + p, x = g & 1;
          wait_k(&av_ready[x], g >> 1);
          wait_k(&bv_ready[x], g >> 1);
          pair_sync(kNbValue);
          // every consumer has read page p by now: its slot takes page p + NBUF
          if (lane == 0 && p + NBUF < n_pages) {
            wait_k(&s_empty[ring_slot(p)], ring_use(p));
            const int nxt = p + NBUF;
            const uint32_t si = ring_slot(nxt);
            fence_proxy_async();
            mbar_expect_tx(&s_full[si], PL::bytes);
            bulk_g2s(s_pages + si * C::PAGE, page_g(p_lo + nxt), PL::bytes, &s_full[si]);
            issued = pg_base + nxt + 1;
            if (nxt + kL2Ahead < n_pages)
              prefetch_l2(page_g(p_lo + nxt + kL2Ahead), PL::bytes);
          }
          __syncwarp();
        }
      } else if (warp == kWarpM) {
        // ============ value MMAs: D_v(plane)[coordinate][column] += A_v(plane) x B_v ============
        for (int p = 0; p < n_pages; ++p) {
          const uint32_t g = pg_base + p, x = g & 1;
          pair_sync(kNbValue);
          if (lane == 0) {
            tc_fence_after();
            const uint32_t bva = smem_u32(s_bv + x * C::BV_BYTES);
            const uint32_t av = tmem + C::TA_V + (AVB == 2 ? x : 0) * C::AV_COLS;
            const bool restart = p % kFlush == 0;   // D_v was flushed into D_acc (or the segment starts)
#pragma unroll
            for (int pl = 0; pl < PV; ++pl)
#pragma unroll
              for (int ks = 0; ks < 4; ++ks)
                mma_f8_ts(tmem + C::TD_V + pl * NVC, av + 32 * pl + 8 * ks, smem_desc(bva + ks * 256, 128, 1024),
                          idesc_v, !(restart && ks == 0));
            tc_commit(&v_fin[x]);
          }
        }
      } else if (warp >= kWarpK && warp < kWarpK + 4) {
        // ============ key-plane warps (row = token): XOR planes and the sign plane -> A_s (smem) ============
        for (int p = 0; p < n_pages; ++p) {
          const uint32_t g = pg_base + p, x = g & 1;
          wait_k(&s_full[ring_slot(p)], ring_use(p));
          const uint8_t* pgp = pg_ptr(p);
          uint4 wk[BK + 1];
#pragma unroll
          for (int q = 0; q < BK; ++q)
            wk[q] = *reinterpret_cast<const uint4*>(pgp + PL::off_kcodes + ((size_t)q * 128 + row) * 16);
          wk[BK] = *reinterpret_cast<const uint4*>(pgp + PL::off_signs + (size_t)row * 16);
          __syncwarp();
          if (lane == 0) mbar_arrive(&s_empty[ring_slot(p)]);
          if (g >= 2) wait_k(&as_free[x], (g >> 1) - 1);   // the score MMAs of page g-2 are done
          uint8_t* as = s_as + x * C::AS_BYTES;
          uint4 xk[NS];   // key monomial planes, then the sign plane
          {
            uint4 kp[PK];
            monomial_words<BK + 1, PK>(wk, kp);
#pragma unroll
            for (int i = 0; i < PK; ++i) xk[i] = kp[i];
            xk[PK] = wk[BK];
          }
#pragma unroll 1
          for (int pl = 0; pl < NS; ++pl) {
            uint32_t x[4];
            pick_plane<NS>(xk, pl, x);
            uint32_t r[32];
            expand_words(x, r);
            uint8_t* dst = as + canon_off(row, pl * 128, NS * 128);
#pragma unroll
            for (int j = 0; j < 8; ++j)
              *reinterpret_cast<uint4*>(dst + j * 128) = make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
          }
          fence_proxy_async();   // A_s is read by the tensor cores
          __syncwarp();
          if (lane == 0) mbar_arrive(&as_ready[x]);
        }
      } else if (warp >= kWarpV && warp < kWarpV + 4) {
        // ============ value-plane warps (lane = coordinate): XOR planes -> A_v (tensor memory) ============
        for (int p = 0; p < n_pages; ++p) {
          const uint32_t g = pg_base + p, x = g & 1;
          wait_k(&s_full[ring_slot(p)], ring_use(p));
          const uint8_t* pgp = pg_ptr(p);
          uint4 wv[BV];
#pragma unroll
          for (int q = 0; q < BV; ++q)
            wv[q] = *reinterpret_cast<const uint4*>(pgp + PL::off_vcodes + ((size_t)q * D + row) * 16);
          __syncwarp();
          if (lane == 0) mbar_arrive(&s_empty[ring_slot(p)]);
          if (g >= (uint32_t)AVB) wait_k(&v_fin[(g - AVB) & 1], (g - AVB) >> 1);   // A_v buffer free
          tc_fence_after();
          uint4 xvp[PV];
          monomial_words<BV, PV>(wv, xvp);
#pragma unroll 1
          for (int pl = 0; pl < PV; ++pl) {
            uint32_t xw[4], r[32];
            pick_plane<PV>(xvp, pl, xw);
            expand_words(xw, r);
            tmem_st32(tl + C::TA_V + (AVB == 2 ? x : 0) * C::AV_COLS + 32 * pl, r);
          }
          tc_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&av_ready[x]);
        }
      } else if ((warp >= kWarpT && warp < kWarpT + 4) || (warp >= kWarpT2 && warp < kWarpT2 + 4)) {
        // ============ token warps (lane = token): logits, lazy softmax, weight operand ============
        // set ts of TS handles heads h0 .. h0 + HPT - 1; it owns their D_s columns, their D_v
        // and D_acc columns and their B_v rows, so the sets never write the same word
        const int twarp = (warp >= kWarpT2 && warp < kWarpT2 + 4) ? 4 + (warp - kWarpT2) : warp - kWarpT;   // 0 .. 7
        const int ts = twarp >> 2, h0 = ts * HPT;
        float m_run[HPT], l_part[HPT], c_part[HPT], g_part[HPT];
#pragma unroll
        for (int h = 0; h < HPT; ++h) {
          m_run[h] = -INFINITY;
          l_part[h] = c_part[h] = g_part[h] = 0.f;
        }
        float n_ref = 0.f;
        for (int p = 0; p < n_pages; ++p) {
          const uint32_t g = pg_base + p, x = g & 1, db = DSB == 2 ? x : 0;
          const uint8_t* pgp = pg_ptr(p);
          wait_k(&s_full[ring_slot(p)], ring_use(p));
          const int nvalid = min(128, seq_len - (p_lo + p) * 128);
          const bool valid = row < nvalid;
          const float nk = valid ? reinterpret_cast<const float*>(pgp + PL::off_nk)[row] : 0.f;
          const float gmv = valid ? reinterpret_cast<const float*>(pgp + PL::off_gamma)[row] : 0.f;
          const float nvt = valid ? reinterpret_cast<const float*>(pgp + PL::off_nv)[row] : 0.f;
          __syncwarp();
          if (lane == 0) mbar_arrive(&s_empty[ring_slot(p)]);
          wait_k(&s_fin[x], g >> 1);        // every score MMA of page p is done
          tc_fence_after();
          float dsk[4 * HPT], dsq[4 * HPT];   // this set's key-term and sign-term columns
#pragma unroll
          for (int c0 = 0; c0 < 4 * HPT; c0 += CKS) {
            uint32_t r[CKS], rq[CKS];
            tmem_ldn<CKS>(tl + C::TD_S + db * C::DS_COLS + 4 * h0 + c0, r);
            tmem_ldn<CKS>(tl + C::TD_S + db * C::DS_COLS + NHALF + 4 * h0 + c0, rq);
            tc_wait_ld();
#pragma unroll
            for (int i = 0; i < CKS; ++i) {
              dsk[c0 + i] = __uint_as_float(r[i]);
              dsq[c0 + i] = __uint_as_float(rq[i]);
            }
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&ds_free[x]);
          float lg[HPT];
          int ovf = nvt > n_ref;
#pragma unroll
          for (int h = 0; h < HPT; ++h) {
            const int hg = h0 + h;
            // folded per-head constants (set-up): logit = nk (mse ak + bk) + gamma (qjl aq + bq)
            const float4 hc = *reinterpret_cast<const float4*>(s_head + hg * 8);
            const float* dk = dsk + 4 * h;
            const float* dq = dsq + 4 * h;
            const float mse = fmaf(0.000244140625f, dk[3], fmaf(0.00390625f, dk[2], fmaf(0.0625f, dk[1], dk[0])));
            const float qjl = fmaf(0.000244140625f, dq[3], fmaf(0.00390625f, dq[2], fmaf(0.0625f, dq[1], dq[0])));
            const float l = fmaf(nk, fmaf(mse, hc.x, hc.y), gmv * fmaf(qjl, hc.z, hc.w));
            lg[h] = (valid && hg < G) ? l : -INFINITY;
            if (a.logits && valid && hg < G)
              a.logits[((size_t)b * a.q_heads + (size_t)kvh * G + hg) * a.max_tokens + (size_t)(p_lo + p) * 128 + row] = l;
            if (lg[h] > m_run[h] + kTau) ovf = 1;
          }
          float fh[HPT];
#pragma unroll
          for (int h = 0; h < HPT; ++h) fh[h] = 1.f;
          bool rescale = false;
          if (t_vote_or<TNT>(ovf)) {
#pragma unroll
            for (int h = 0; h <= HPT; ++h) {
              float mx = h < HPT ? lg[h] : nvt;
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
              if (lane == 0) s_red[twarp * (HPT + 1) + h] = mx;
            }
            t_sync<TNT>();
            float nvmax = 0.f;
            for (int w2 = 0; w2 < 4 * TS; ++w2) nvmax = fmaxf(nvmax, s_red[w2 * (HPT + 1) + HPT]);
            const float n_new = nvmax > n_ref ? 1.25f * nvmax : n_ref;
#pragma unroll
            for (int h = 0; h < HPT; ++h) {
              float mx = -INFINITY;
              for (int w2 = 4 * ts; w2 < 4 * ts + 4; ++w2) mx = fmaxf(mx, s_red[w2 * (HPT + 1) + h]);
              const float m_new = fmaxf(m_run[h], mx);
              const float alpha = (m_run[h] == -INFINITY) ? 0.f : __expf(m_run[h] - m_new);
              fh[h] = (n_ref > 0.f) ? alpha * (n_ref / n_new) : 0.f;
              l_part[h] *= alpha;
              c_part[h] *= fh[h];
              g_part[h] *= fh[h];
              m_run[h] = m_new;
            }
            n_ref = n_new;
            rescale = p > 0;
            t_sync<TNT>();   // s_red reads done
          }
          // this set's columns of each plane accumulator: pl NVC + NPW h0 .. + NPW HPT
          if (p == 0) {
            // a new segment: the flushed total starts at zero (the previous epilogue has read it)
            uint32_t z[CKV];
#pragma unroll
            for (int i = 0; i < CKV; ++i) z[i] = 0u;
#pragma unroll 1
            for (int pl = 0; pl < PV; ++pl)
              for (int co = 0; co < NPW * HPT; co += CKV) tmem_stn<CKV>(tl + C::TD_ACC + pl * NVC + NPW * h0 + co, z);
            tc_wait_st();
          }
          const bool flush = p > 0 && p % kFlush == 0;
          if (rescale || flush) {
            // D_v holds exactly the pages of this stretch before p once the value MMAs of page
            // p-1 are done; this warp handles its lane quarter (32 coordinates): on a flush
            // D_acc = (D_acc + D_v) f, otherwise D_acc *= f and D_v *= f (f = 1 without rescale)
            wait_k(&v_fin[(g - 1) & 1], (g - 1) >> 1);
            tc_fence_after();
#pragma unroll 1
            for (int pl = 0; pl < PV; ++pl) {
#pragma unroll
              for (int co = 0; co < NPW * HPT; co += CKV) {
                const uint32_t col = pl * NVC + NPW * h0 + co;
                uint32_t rv[CKV], ra[CKV];
                tmem_ldn<CKV>(tl + C::TD_V + col, rv);
                tmem_ldn<CKV>(tl + C::TD_ACC + col, ra);
                tc_wait_ld();
#pragma unroll
                for (int i = 0; i < CKV; ++i) {
                  const float fv = fh[(co + i) / NPW];
                  const float dv = __uint_as_float(rv[i]), da = __uint_as_float(ra[i]);
                  ra[i] = __float_as_uint(flush ? (da + dv) * fv : da * fv);
                  rv[i] = __float_as_uint(dv * fv);
                }
                tmem_stn<CKV>(tl + C::TD_ACC + col, ra);
                if (!flush) tmem_stn<CKV>(tl + C::TD_V + col, rv);
              }
            }
            tc_wait_st();
          }
          // softmax weights -> two e4m3 pieces per head; the byte for row n = 2 hg + piece
          const float xs = nvt * (n_ref > 0.f ? 1.f / n_ref : 0.f) * v_igamma * kSB;
          uint32_t wb[HPT / 2];
          // two heads per conversion: word h/2 holds rows 2h..2h+3 = [hi(h), lo(h), hi(h+1), lo(h+1)]
#pragma unroll
          for (int h = 0; h < HPT; h += 2) {
            const float p0 = lg[h] == -INFINITY ? 0.f : __expf(lg[h] - m_run[h]);
            const float p1 = lg[h + 1] == -INFINITY ? 0.f : __expf(lg[h + 1] - m_run[h + 1]);
            l_part[h] += p0;   // the denominator keeps every position
            l_part[h + 1] += p1;
            // Sparse V: a position below the threshold contributes no value
            const float x0 = (p0 < sparse_v ? 0.f : p0) * xs, x1 = (p1 < sparse_v ? 0.f : p1) * xs;
            const uint32_t hi2 = cvt_e4m3x2(x1, x0);
            const float2 hf = e4m3x2_to_f2(hi2);
            const uint32_t lo2 = cvt_e4m3x2(16.f * (x1 - hf.y), 16.f * (x0 - hf.x));
            const float2 lf = e4m3x2_to_f2(lo2);
            const float b0 = fmaf(0.0625f, lf.x, hf.x), b1 = fmaf(0.0625f, lf.y, hf.y);
            c_part[h] = fmaf(v_beta, b0, c_part[h]);
            c_part[h + 1] = fmaf(v_beta, b1, c_part[h + 1]);
            g_part[h] = fmaf(v_gamma, b0, g_part[h]);
            g_part[h + 1] = fmaf(v_gamma, b1, g_part[h + 1]);
            wb[h >> 1] = __byte_perm(hi2, lo2, 0x5140);
          }
          // B_v buffer of page p: its previous user, the value MMA of page p-2, must be done
          if (p >= 2) wait_k(&v_fin[g & 1], (g >> 1) - 1);
          uint8_t* bvb = s_bv + (g & 1) * C::BV_BYTES;
          const int e = lane & 3, base = lane & ~3;
          const int k0 = 32 * ((row >> 2) & 3) + 4 * (row >> 4);   // K byte of token 4i
          // this set's words (rows 4 w .. 4 w + 3)
#pragma unroll
          for (int r4 = 0; r4 < HPT / 2; ++r4) {
            const uint32_t wv = wb[r4];
            const uint32_t w0 = __shfl_sync(0xffffffffu, wv, base + 0);
            const uint32_t w1 = __shfl_sync(0xffffffffu, wv, base + 1);
            const uint32_t w2 = __shfl_sync(0xffffffffu, wv, base + 2);
            const uint32_t w3 = __shfl_sync(0xffffffffu, wv, base + 3);
            const uint32_t sel = (uint32_t)e | ((uint32_t)(e + 4) << 4);
            const uint32_t t01 = __byte_perm(w0, w1, sel), t23 = __byte_perm(w2, w3, sel);
            const int word = h0 / 2 + r4;
            *reinterpret_cast<uint32_t*>(bvb + canon_off(4 * word + e, k0, 128)) = __byte_perm(t01, t23, 0x5410);
          }
          fence_proxy_async();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bv_ready[g & 1]);
        }
        // per-head sums of this segment
#pragma unroll
        for (int h = 0; h < HPT; ++h) {
          float v3[3] = {l_part[h], c_part[h], g_part[h]};
#pragma unroll
          for (int c = 0; c < 3; ++c) {
            float v = v3[c];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            if (lane == 0) s_red[(twarp * (HPT + 1) + h) * 3 + c] = v;
          }
        }
        if (tid == 0) s_f[0] = n_ref;   // thread 0: the first token thread (kWarpT == 0)
        // partial record head part (m, l): lane h of the set's first warp for head h0 + h
        t_sync<TNT>();
        if ((twarp & 3) == 0 && lane < HPT && h0 + lane < G) {
          float l_tot = 0.f, mv = 0.f;
          for (int w2 = 4 * ts; w2 < 4 * ts + 4; ++w2) l_tot += s_red[(w2 * (HPT + 1) + lane) * 3];
#pragma unroll
          for (int h = 0; h < HPT; ++h) mv = h == lane ? m_run[h] : mv;
          float* rh = rec + (size_t)(h0 + lane) * (2 + D);
          rh[0] = mv;
          rh[1] = l_tot;
        }
      }
    }
    if (n_pages == 0 && warp == 0 && tid < GP && tid < G) {
      float* rh = rec + (size_t)tid * (2 + D);
      rh[0] = -INFINITY;
      rh[1] = 0.f;
    }
    __syncthreads();   // token sums in s_red
    if (warp >= kWarpV && warp < kWarpV + 4) {
      // ---------- epilogue: o~ = (n_ref / kSB) [ 2 sum_M alpha_M (D_M - C) - sum alpha G ] ----------
      float ov[GP];
#pragma unroll
      for (int h = 0; h < GP; ++h) ov[h] = 0.f;
      if (n_pages > 0) {
        {
          const uint32_t last = pg_base + n_pages - 1;   // the last value MMA is done
          wait_k(&v_fin[last & 1], last >> 1);
        }
        tc_fence_after();
#pragma unroll 1
        for (int pl = 0; pl < PV; ++pl) {
          const float al = a.alpha_v[pl];
          float dv[NVC];
#pragma unroll
          for (int c0 = 0; c0 < NVC; c0 += 16) {
            uint32_t r[16], ra[16];
            tmem_ld16(tl + C::TD_V + pl * NVC + c0, r);
            tmem_ld16(tl + C::TD_ACC + pl * NVC + c0, ra);
            tc_wait_ld();
#pragma unroll
            for (int i = 0; i < 16; ++i) dv[c0 + i] = __uint_as_float(r[i]) + __uint_as_float(ra[i]);
          }
#pragma unroll
          for (int h = 0; h < GP; ++h) ov[h] += al * fmaf(0.0625f, dv[NPW * h + 1], dv[NPW * h]);
        }
      }
      const float nref = n_pages > 0 ? s_f[0] : 0.f;
      const float scale = nref > 0.f ? nref / kSB : 0.f;
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        if (h >= G) continue;
        float c_tot = 0.f, g_tot = 0.f;
        if (n_pages > 0) {
          const int hs = h / HPT, hl = h % HPT;   // the token-warp set that summed head h
          for (int w2 = 4 * hs; w2 < 4 * hs + 4; ++w2) {
            c_tot += s_red[(w2 * (HPT + 1) + hl) * 3 + 1];
            g_tot += s_red[(w2 * (HPT + 1) + hl) * 3 + 2];
          }
        }
        const float o = scale * (2.f * (ov[h] - a.asum_v * c_tot) - a.asum_v * g_tot);
        rec[(size_t)h * (2 + D) + 2 + row] = n_pages > 0 ? o : 0.f;
      }
    }
    pg_base += n_pages;
    tc_fence_before();
    __syncthreads();
    s_fail_seen = *s_fail != 0;
  }
  // teardown after a timeout: the last fill of each ring slot and every MMA the two issuers
  // started complete (bounded waits) before the shared and tensor memory are released
  if (s_fail_seen && lane == 0) {
    if (warp == kWarpWM)
      for (uint32_t i = issued > (uint32_t)NBUF ? issued - NBUF : 0u; i < issued; ++i)
        mbar_wait(&s_full[i % NBUF], (i / NBUF) & 1);
    if (warp == kWarpS || warp == kWarpM) {
      uint64_t* t = &td_bar[warp == kWarpS ? 0 : 1];
      tc_commit(t);
      mbar_wait(t, 0);
    }
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
