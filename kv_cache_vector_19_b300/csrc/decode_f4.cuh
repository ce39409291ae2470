// tq_attn_decode on 5th-generation tensor cores with 4-bit operands (tcgen05 kind::mxf4),
// head_dim 128.
//
// Score of cached key t for query head h ([BLOG] "Технология TurboQuant ...", section 1.2;
// sqrt(pi/2)/m makes the sign sketch an unbiased inner-product estimate):
//   logit = ( n_t <q~, c_K[idx_t]> + gamma_t sqrt(pi/2)/m <q_s, 2 sigma_t - 1> ) / sqrt(d)
// and the output is Pi^T sum_t softmax_t n_v,t c_V[idx_v,t] (values accumulated in the
// rotated frame; the combine kernel rotates back).
//
// Both inner products are contractions over signed bit planes.  A Lloyd-Max book of a
// symmetric density is antisymmetric, so with e_M = prod_{q in M} (1 - 2 b_q) over the odd
// subsets M of the code bits (bitplane.h),
//     c[idx] = - sum_M alpha_M e_M(idx),        2 sigma - 1 = - e_sigma,
// a plane of +-1 entries with no constant part: the tensor core never accumulates a large
// offset that the epilogue would have to cancel.  A plane word becomes four words of e2m1
// operands (+1 = 0x2, -1 = 0xA) with one shift and one AND-OR each (expand_signed4); the
// other operand carries everything else, split into e2m1 "pieces" of power-of-two scale:
//   query  v = -alpha_M q~_j (key planes) or -q_s,j (sign plane): 7 pieces of 3 bits each,
//          ~2^-20 of the largest |v| of the head;
//   weight x_t = p_t n_v,t / n_ref < 2 as a 16-bit fixed-point Y = round(2^15 x): piece k is
//          the bit pair (2k, 2k+1) of Y, and the e2m1 codes 0..3 are exactly 0, 0.5, 1, 1.5,
//          so eight pieces are one bit-spread of Y (no conversions, no serial chain) and the
//          value accumulators hold exact sums of half-integers.
// Each piece is its own MMA column; the token warps sum a head's columns in fp32.
//
// Operands and accumulators (M = 128, K = 64 per MMA, ue8m0 block scales all 1.0):
//   A_s (TMEM, lane = token slot, x2)      key planes + sign plane of one page, 16 columns each
//   B_s (smem, K-major)                    query pieces, columns [key set0|set1|sign set0|set1]
//   D_s (TMEM, lane = token slot, x1/x2)   score columns
//   A_v (TMEM, lane = coordinate, x2)      value planes of one page, 16 columns each
//   B_v (smem, K-major, x2)                softmax-weight pieces of the page, 8 per head
//   D_v (TMEM, lane = coordinate)          one accumulator per value plane, the whole segment
//   (TMEM, lane = token slot, x2)          n_k, gamma, n_v of the page, written by the key-plane
//                                          warps, read by the token warps with the scores
// The token slot of TMEM lane L is tau = (L >> 1) + 64 (L & 1): then the eight slots whose
// weights form one 32-bit word of B_v (the K order of a value-plane word) sit in eight
// consecutive lanes of one warp, and one 8 x 8 nibble transpose builds the word.
//
// MMA issue is what bounds a tcgen05 decode at this size: one issuing thread sustains about
// one MMA per ~60 cycles (any N <= 128, either operand kind), and every extra instruction
// between two MMAs of one thread lengthens that; separate issuing warps add up.  Here three
// warps issue (score; value planes, two halves), each a fully unrolled run of MMAs on
// precomputed descriptors, so a page (b = 3: 6 score + 8 value MMAs) costs each issuer ~4
// MMAs.  Issuers never touch shared memory: a waiter warp polls the mbarriers (bounded
// waits) and releases its issuers through a named barrier.
//
// Warp roles (21 warps with two token-warp sets, 29 with four):
//   0-3, 16-19  token warps (independent sets, each a share of the query heads; further sets
//               at 20-23, 24-27): D_s ->
//               logits, lazy online softmax, D_v rescale when the running maximum moves,
//               weights -> fixed-point pieces -> 8 x 8 nibble transposes -> B_v
//   4-7         key-plane warps: key planes and sign plane -> A_s, token norms -> TMEM
//   8-11        value-plane warps: value planes -> A_v; epilogue
//   12          score-MMA issuer; 13, 14 value-MMA issuers
//   15          score waiter; the last warp value waiter and page ring (cp.async.bulk, L2 prefetch)
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
namespace dtf {

using namespace dev;
using dmma::Params;

constexpr int kWarpT = 0;     // token warps, first set (TMEM lane quarters 0-3)
constexpr int kWarpK = 4;     // key-plane warps
constexpr int kWarpV = 8;     // value-plane warps; epilogue
constexpr int kWarpIS = 12;   // score-MMA issuer
constexpr int kWarpIV0 = 13;  // value-MMA issuer, first half of the planes
constexpr int kWarpIV1 = 14;  // value-MMA issuer, second half
constexpr int kWarpWS = 15;   // score waiter
constexpr int kWarpT2 = 16;   // token warps, further sets (16-19, 20-23, ...), then the value waiter
// Token-warp sets (each a warp per TMEM lane quarter, each owning GP / sets query heads): two
// for up to 4 query heads per KV head, four from 8 on (measured on the long-context shapes:
// G = 4 two sets 248 us, four 254 us; G = 8 two sets 446 us, four 340 us per call).
__host__ __device__ constexpr int token_sets(int gp) { return gp >= 8 ? 4 : (gp < 2 ? gp : 2); }
constexpr int kL2Ahead = 12;  // pages prefetched into L2 beyond the shared-memory ring
constexpr int kRingMax = 8;   // ring slots (as many as fit, at most this; a streaming probe
                              // of this grid runs the whole cache through 4-8 slots at ~5 TB/s)
static_assert(kRingMax + kL2Ahead <= 32, "a paged segment's ring and L2 look-ahead fit two 32-page windows");
// Lazy-maximum threshold (natural-log units): a page rescales the running maximum only when
// one of its logits exceeds it by kTau or a value norm exceeds n_ref, so a weight
// x = p n_v / n_ref stays below e^0.69 = 1.994 and Y = round(2^15 x) fits 16 bits.  The
// resolution is absolute (2^-16), not relative: diffuse attention over a long context is made
// of many small weights whose rounding errors add up, which is what sets the 16 bits.
constexpr float kTau = 0.69f;
constexpr float kWScale = 32768.f;
constexpr int kNQP = 7;       // e2m1 pieces of a query operand
constexpr int kNPW = 8;       // 2-bit pieces of a softmax weight (8 columns per head)
constexpr int kSmemMax = 227 * 1024;
constexpr int kNbVote0 = 1, kNbScore = 2, kNbValue = 3, kNbVote1 = 4;   // named barriers (votes: 1, 4, 5, ..)

__host__ __device__ constexpr int rnd(int x, int m) { return (x + m - 1) / m * m; }

template <int BITS, int GP>
struct Cfg {
  static constexpr int D = 128;
  using PL = PageLayout<128, BITS>;
  static constexpr int BK = BITS - 1, BV = BITS;
  static constexpr int PK = 1 << (BK - 1), PV = 1 << (BV - 1), NS = PK + 1;
  static constexpr int TS = token_sets(GP);          // token-warp sets
  static constexpr int HPT = GP / TS;                  // query heads per token-warp set
  static constexpr int WV = kWarpT2 + 4 * (TS - 1);    // value waiter; page ring
  static constexpr int WARPS = WV + 1;
  static constexpr int THREADS = 32 * WARPS;
  static constexpr int SCOLS = 8 * HPT;                // score columns of one term and set (8 per head)
  static constexpr int NSC = 2 * TS * SCOLS;           // [key: set 0 | set 1 .. | sign: set 0 | set 1 ..]
  static constexpr int VCOLS = 8 * HPT;                // value columns (B_v rows) of one set, 8 per head
  static constexpr int NVC = TS * VCOLS;               // = 8 GP
  // tensor memory
  static constexpr int AS_COLS = NS * 16, AV_COLS = PV * 16, DV_COLS = PV * NVC, SF_COLS = 8, SC_COLS = 8;
  // buffers of D_s, A_s, A_v: two each where tensor memory allows (in that order of priority)
  static constexpr int BASE = DV_COLS + SF_COLS + SC_COLS + NSC + AS_COLS + AV_COLS;
  static constexpr int DSB = BASE + NSC <= 512 ? 2 : 1;
  static constexpr int ASB = BASE + (DSB - 1) * NSC + AS_COLS <= 512 ? 2 : 1;
  static constexpr int AVB = BASE + (DSB - 1) * NSC + (ASB - 1) * AS_COLS + AV_COLS <= 512 ? 2 : 1;
  static constexpr int TD_S = 0;
  static constexpr int TD_V = DSB * NSC;
  static constexpr int TA_S = TD_V + DV_COLS;
  static constexpr int TA_V = TA_S + ASB * AS_COLS;
  static constexpr int TSF = TA_V + AVB * AV_COLS;     // scale factors: A at TSF, B at TSF + 4
  static constexpr int TSC = TSF + SF_COLS;            // token scalars n_k, gamma, n_v (x2, 4 columns each)
  static constexpr int TCOLS = TSC + SC_COLS;
  // shared memory
  static constexpr int PAGE = PL::bytes;
  static constexpr int BS_ROWB = NS * 64;              // bytes per B_s row (NS planes x 128 nibbles)
  static constexpr int BS_BYTES = NSC * BS_ROWB;
  static constexpr int BV_BYTES = NVC * 64;            // per buffer (128 nibbles per row)
  static constexpr int OFF_BS = 0;
  static constexpr int OFF_BV = OFF_BS + BS_BYTES;
  static constexpr int OFF_Q = OFF_BV + 2 * BV_BYTES;         // [GP][2][128] f32: q~, q_s
  static constexpr int OFF_HEAD = OFF_Q + GP * 2 * 128 * 4;   // [GP][4] f32
  static constexpr int OFF_RED = OFF_HEAD + GP * 4 * 4;       // [4 TS token warps][HPT + 1] f32
  static constexpr int OFF_F = OFF_RED + 4 * TS * (HPT + 1) * 4;   // n_ref of each token-warp set
  static constexpr int OFF_MBAR = rnd(OFF_F + 16, 8);
  // full[kRingMax], empty[kRingMax], as_ready[2], as_free[2], s_fin[2], ds_free[2], av_ready[2],
  // v_fin[2], bv_ready[2], teardown[3]
  static constexpr int NMBAR = 2 * kRingMax + 14 + 3;
  static constexpr int OFF_MISC = OFF_MBAR + NMBAR * 8;       // tmem base, fail flag
  static constexpr int OFF_PAGES = rnd(OFF_MISC + 16, 128);
  static constexpr int NBUF_FIT = (kSmemMax - OFF_PAGES) / PAGE;
  static constexpr int NBUF = NBUF_FIT > kRingMax ? kRingMax : NBUF_FIT;
  static constexpr int SMEM = OFF_PAGES + NBUF * PAGE;
  static constexpr bool SUPPORTED = TCOLS <= 512 && NBUF >= 4 && HPT >= 1 && GP % TS == 0 && kNPW <= 8;
};

// OR-vote / barrier among the 128 threads of one token-warp set (named barrier id).
__device__ __forceinline__ int t_vote_or(int id, int pred) {
  int r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.s32 q, %1, 0;\n barrier.cta.red.or.pred p, %2, 128, q;\n selp.s32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"(pred), "r"(id)
      : "memory");
  return r;
}
__device__ __forceinline__ void t_sync(int id) { asm volatile("barrier.cta.sync %0, 128;" ::"r"(id) : "memory"); }
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// a waiter warp and its issuer warp(s) meet at a named barrier (64 or 96 threads)
template <int NT>
__device__ __forceinline__ void group_sync(int id) {
  __syncwarp();
  asm volatile("barrier.cta.sync.aligned %0, %1;" ::"r"(id), "n"(NT) : "memory");
}

// token slot held by TMEM lane L (0..127)
__host__ __device__ __forceinline__ int slot_of_lane(int L) { return (L >> 1) + 64 * (L & 1); }
// coordinate (or token slot) at nibble i of expansion word (c, s) of a plane: a plane word c
// carries element x at bit 2 kb + h + 8 e with x = 32 kb + 16 h + 4 c + e (page format), and
// expand_signed4 puts bit 4 i + s into nibble i of word s
__host__ __device__ __forceinline__ int elem_of_nibble(int c, int s, int i) {
  return 64 * (i & 1) + 16 * s + 4 * c + (i >> 1);
}

// y_0 = v * scale, y_{k+1} = 8 (y_k - e2m1(y_k)): the nibble of piece `piece` of v (|y_0| <= 4)
__device__ __forceinline__ uint32_t piece_nibble(float y, int piece) {
  uint32_t nib = 0u;
  for (int k = 0; k <= piece; ++k) {
    nib = cvt_e2m1x2(0.f, y) & 0xFu;
    y = 8.f * (y - e2m1x2_to_f2(nib).x);
  }
  return nib;
}
// largest power of two s with m * s <= 4 (m > 0), else 1
__device__ __forceinline__ float piece_scale(float m) {
  if (!(m > 0.f)) return 1.f;
  float s = exp2f(floorf(log2f(4.f / m)));
  while (m * s > 4.f) s *= 0.5f;
  while (m * s * 2.f <= 4.f) s *= 2.f;
  return s;
}

// HSPLIT > 1: a.kv_heads counts virtual KV heads, HSPLIT per real one (each with a.group of its
// query heads), and virtual KV head v reads the pages of real KV head v / HSPLIT.
template <int BITS, int GP, bool PAGED, int HSPLIT>
__global__ void __launch_bounds__(Cfg<BITS, GP>::THREADS, 1) decode_f4_kernel(Params a, PageMap pm, float sparse_v) {
  using C = Cfg<BITS, GP>;
  using PL = typename C::PL;
  constexpr int D = 128, NS = C::NS, PK = C::PK, PV = C::PV, BK = C::BK, BV = C::BV, NBUF = C::NBUF;
  constexpr int NSC = C::NSC, NVC = C::NVC, SCOLS = C::SCOLS, VCOLS = C::VCOLS, DSB = C::DSB;
  constexpr int HPT = C::HPT, kThreads = C::THREADS, ASB = C::ASB, AVB = C::AVB, TS = C::TS;
  constexpr int kWarpWV = C::WV, kWarpsAll = C::WARPS;
  extern __shared__ __align__(1024) unsigned char smem[];
  pdl_trigger();   // the combine grid may launch once every CTA of this grid is running
  uint8_t* s_pages = smem + C::OFF_PAGES;
  uint8_t* s_bs = smem + C::OFF_BS;
  uint8_t* s_bv = smem + C::OFF_BV;
  float* s_q = reinterpret_cast<float*>(smem + C::OFF_Q);
  float* s_head = reinterpret_cast<float*>(smem + C::OFF_HEAD);
  float* s_red = reinterpret_cast<float*>(smem + C::OFF_RED);
  float* s_f = reinterpret_cast<float*>(smem + C::OFF_F);
  uint64_t* mb = reinterpret_cast<uint64_t*>(smem + C::OFF_MBAR);
  // Every hand-off barrier exists once per buffer (index = page & 1) and completes once per
  // page of that parity; every waiter has waited for the previous completion, so a parity wait
  // never mistakes an older phase for a newer one.
  uint64_t* s_full = mb;                 // [ring] page in ring slot landed (+ tx bytes)
  uint64_t* s_empty = mb + kRingMax;     // [ring] page read by the key- and value-plane warps (4 + 4)
  uint64_t* as_ready = mb + 2 * kRingMax;  // [2] key planes of the page in A_s (4 warps)
  uint64_t* as_free = as_ready + 2;      // [2]  score MMAs reading that A_s buffer done (commit)
  uint64_t* s_fin = as_ready + 4;        // [2]  score MMAs into that D_s buffer done (commit)
  uint64_t* ds_free = as_ready + 6;      // [2]  D_s buffer read by the token warps (4 TS)
  uint64_t* av_ready = as_ready + 8;     // [2]  value planes in that A_v buffer (4 warps)
  uint64_t* v_fin = as_ready + 10;       // [2]  value MMAs of the page done (commits of 2 issuers)
  uint64_t* bv_ready = as_ready + 12;    // [2]  B_v buffer written, D_v rescaled (4 TS token warps)
  uint64_t* td_bar = as_ready + 14;      // [3]  teardown drains of the three issuers
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* s_fail = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = 32 * (warp & 3) + lane;    // TMEM lane of this thread (4-warp roles)
  const int G = a.group, PM = a.pages_per_seq;
  const float inv_sqrt_d = rsqrtf((float)D);
  const float qjl_c = 1.2533141373155002512f / (float)D;   // sqrt(pi/2) / m, m = d

  const int range_lo = blockIdx.x * a.chunk;
  const int range_hi = min(range_lo + a.chunk, a.total_pages);
  if (range_lo >= range_hi) return;

  if (warp == 0) tmem_alloc(s_tmem, 512);
  if (tid == 0) {
    for (int i = 0; i < NBUF; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], 8);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&as_ready[i], 4);
      mbar_init(&as_free[i], 1);
      mbar_init(&s_fin[i], 1);
      mbar_init(&ds_free[i], 4 * TS);
      mbar_init(&av_ready[i], 4);
      mbar_init(&v_fin[i], 2);
      mbar_init(&bv_ready[i], 4 * TS);
    }
    for (int i = 0; i < 3; ++i) mbar_init(&td_bar[i], 1);
    *s_fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);   // this warp's lane quarter
  if (warp >= kWarpV && warp < kWarpV + 4) {
    // block scale factors: every byte 0x7F (2^0) in all 128 lanes of both regions
    uint32_t r[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) r[i] = 0x7F7F7F7Fu;
    tmem_st8(tl + C::TSF, r);
    tc_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  // key-plane MMAs write the key half of the score columns, sign-plane MMAs the sign half
  constexpr uint32_t idesc_s = make_idesc_mxf4(128, NSC / 2);
  constexpr uint32_t idesc_v = make_idesc_mxf4(128, NVC);
  const uint32_t sfa = tmem + C::TSF, sfb = tmem + C::TSF + 4;

  uint32_t pg_base = 0;      // pages (== ring fills) of the previous segments
  uint32_t issued = 0;       // ring fills issued (value-waiter lane)

  auto fail_now = [&]() {
    if (lane == 0) atomicOr(a.status, kFlagTimeout);
    *s_fail = 1;
  };
  // Bounded wait for the k-th completion (0-based) of a barrier.  Once a wait timed out every
  // later wait returns at once: all roles still run their loops to the end, so the named-
  // barrier counts stay balanced and the kernel finishes.
  auto wait_k = [&](uint64_t* bar, uint32_t k) {
    if (mbar_test_wait(bar, k & 1)) return;
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
    const uint8_t* seq_base = a.cache + (size_t)(seq / HSPLIT) * PM * PL::bytes;
    auto ring_slot = [&](int p) { return (pg_base + p) % NBUF; };
    auto ring_use = [&](int p) { return (pg_base + p) / NBUF; };
    auto pg_ptr = [&](int p) { return s_pages + ring_slot(p) * C::PAGE; };
    // Block pool (PAGED, its own instantiation): the value-waiter warp, which fills the ring,
    // holds the block ids of the segment's pages [32 win, 32 win + 64), one of each window per
    // lane, loaded a window ahead, so that a page address is a shuffle, not a dependent load.
    [[maybe_unused]] const int32_t* trow = nullptr;
    [[maybe_unused]] int win = 0;
    [[maybe_unused]] int32_t blk_a = 0, blk_b = 0;
    auto page_at = [&](int i) -> const uint8_t* {   // page p_lo + i; warp-wide when PAGED
      if constexpr (PAGED) {
        const int32_t x = __shfl_sync(0xffffffffu, blk_a, i & 31);
        const int32_t y = __shfl_sync(0xffffffffu, blk_b, i & 31);
        int blk = i < 32 * (win + 1) ? x : y;
        if ((unsigned)blk >= (unsigned)pm.n_blocks) {   // clamped into the pool, reported
          if (lane == 0) atomicOr(a.status, kFlagBounds);
          blk = blk < 0 ? 0 : pm.n_blocks - 1;
        }
        return a.cache + ((size_t)blk * (a.kv_heads / HSPLIT) + kvh / HSPLIT) * PL::bytes;
      } else {
        return seq_base + (size_t)(p_lo + i) * PL::bytes;
      }
    };

    __syncthreads();   // previous segment fully done
    if constexpr (PAGED) {
      if (warp == kWarpWV) {
        trow = pm.table + (size_t)b * pm.stride + p_lo;
        win = 0;
        blk_a = lane < n_pages ? __ldg(trow + lane) : 0;
        blk_b = 32 + lane < n_pages ? __ldg(trow + 32 + lane) : 0;
        const int first = min(n_pages, NBUF);
        for (int i = 0; i < first; ++i) {
          const uint8_t* src = page_at(i);
          if (lane == 0) {
            const uint32_t si = ring_slot(i);
            fence_proxy_async();
            mbar_expect_tx(&s_full[si], PL::bytes);
            bulk_g2s(s_pages + si * C::PAGE, src, PL::bytes, &s_full[si]);
          }
        }
        if (lane == 0) issued = pg_base + first;
        for (int i = NBUF; i < min(n_pages, NBUF + kL2Ahead); ++i) {
          const uint8_t* src = page_at(i);
          if (lane == 0) prefetch_l2(src, PL::bytes);
        }
      }
    } else {
      if (warp == kWarpWV && lane == 0) {
        const int first = min(n_pages, NBUF);
        for (int i = 0; i < first; ++i) {
          const uint32_t si = ring_slot(i);
          fence_proxy_async();
          mbar_expect_tx(&s_full[si], PL::bytes);
          bulk_g2s(s_pages + si * C::PAGE, page_at(i), PL::bytes, &s_full[si]);
        }
        issued = pg_base + first;
        for (int i = NBUF; i < min(n_pages, NBUF + kL2Ahead); ++i)
          prefetch_l2(page_at(i), PL::bytes);
      }
    }

    // ---- query operand of this KV head ----
    pdl_wait();   // q~ and q_s of the prologue grid (at once after the first segment)
    for (int e = tid; e < GP * 2 * D; e += kThreads) {
      const int hh = e / (2 * D), rem = e % (2 * D), which = rem / D, j = rem % D;
      float v = 0.f;
      if (hh < G) {
        const size_t r = (size_t)b * a.q_heads + (size_t)kvh * G + hh;
        v = (which == 0 ? a.qr : a.qs)[r * D + j];
      }
      s_q[e] = v;
    }
    __syncthreads();
    for (int hh = warp; hh < GP; hh += kWarpsAll) {   // piece scales: largest operand -> (2, 4]
      float mk = 0.f, mq = 0.f;
      for (int j = lane; j < D; j += 32) {
        mk = fmaxf(mk, fabsf(s_q[(hh * 2 + 0) * D + j]));
        mq = fmaxf(mq, fabsf(s_q[(hh * 2 + 1) * D + j]));
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        mk = fmaxf(mk, __shfl_xor_sync(0xffffffffu, mk, o));
        mq = fmaxf(mq, __shfl_xor_sync(0xffffffffu, mq, o));
      }
      if (lane == 0) {
        float amax = 0.f;
        for (int i = 0; i < PK; ++i) amax = fmaxf(amax, fabsf(a.alpha_k[i]));
        s_head[hh * 4 + 0] = piece_scale(amax * mk);
        s_head[hh * 4 + 1] = piece_scale(mq);
      }
    }
    __syncthreads();
    // B_s[n][k]: 32-bit word w of row n holds K positions 8 w .. 8 w + 7 = plane w / 16,
    // expansion word (c, s) = ((w % 16) / 4, w % 4), nibbles i -> element elem_of_nibble(c, s, i)
    for (int e = tid; e < NSC * NS * 16; e += kThreads) {
      const int n = e / (NS * 16), w = e % (NS * 16);
      const int pl = w / 16, c = (w % 16) / 4, s = w % 4;
      const bool sign_term = n >= TS * SCOLS;
      const int set = (n % (TS * SCOLS)) / SCOLS, lc = n % SCOLS;
      const int hh = set * HPT + lc / 8, piece = lc % 8;
      uint32_t word = 0u;
      if (piece < kNQP && hh < G && (sign_term ? pl == PK : pl < PK)) {
        const float sc = s_head[hh * 4 + (sign_term ? 1 : 0)];
        const float coef = sign_term ? -1.f : -a.alpha_k[pl];
        const float* qv = s_q + (hh * 2 + (sign_term ? 1 : 0)) * D;
#pragma unroll
        for (int i = 0; i < 8; ++i) word |= piece_nibble(coef * qv[elem_of_nibble(c, s, i)] * sc, piece) << (4 * i);
      }
      *reinterpret_cast<uint32_t*>(s_bs + canon_off(n, 4 * w, C::BS_ROWB)) = word;
    }
    // token-warp form of the per-head constants:
    //   logit = n_k * (sum_p 8^-p D_key,p) * hk + gamma * (sum_p 8^-p D_sign,p) * hq
    for (int hh = tid; hh < GP; hh += kThreads) {
      float* hp = s_head + hh * 4;
      const float sk = hp[0], sq = hp[1];
      hp[2] = inv_sqrt_d / sk;
      hp[3] = qjl_c * inv_sqrt_d / sq;
    }
    fence_proxy_async();   // B_s is read by the tensor cores
    __syncthreads();

    if (n_pages > 0) {
      if (warp == kWarpWS) {
        // ============ score waiter: A_s(g) stored and a D_s buffer free -> release the score issuer ============
        for (int p = 0; p < n_pages; ++p) {
          const uint32_t g = pg_base + p, x = g & 1;
          wait_k(&as_ready[x], g >> 1);
          if (DSB == 2 && g >= 2) wait_k(&ds_free[x], (g >> 1) - 1);
          if (DSB == 1 && g >= 1) wait_k(&ds_free[(g - 1) & 1], (g - 1) >> 1);
          group_sync<64>(kNbScore);
        }
      } else if (warp == kWarpIS) {
        // ============ score MMAs: D_s[token][column] = A_s[token][planes] x B_s ============
        uint64_t bd[NS * 2];
        const uint32_t bs = smem_u32(s_bs);
        constexpr uint32_t SBO = C::BS_ROWB / 16 * 128;   // bytes per 8-row group of B_s
#pragma unroll
        for (int ks = 0; ks < NS * 2; ++ks)   // the sign half starts at row NSC / 2
          bd[ks] = smem_desc(bs + (ks >= 2 * PK ? (NSC / 2 / 8) * SBO : 0u) + ks * 256, 128, SBO);
        for (int p = 0; p < n_pages; ++p) {
          const uint32_t g = pg_base + p, x = g & 1;
          const uint32_t d = tmem + C::TD_S + (DSB == 2 ? x : 0) * NSC;
          const uint32_t as = tmem + C::TA_S + (ASB == 2 ? x : 0) * C::AS_COLS;
          group_sync<64>(kNbScore);
          if (lane == 0) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < NS * 2; ++ks)
              mma_f4_ts(d + (ks >= 2 * PK ? NSC / 2 : 0), as + 8 * ks, bd[ks], idesc_s, sfa, sfb, ks != 0 && ks != 2 * PK);
            tc_commit(&as_free[x]);
            tc_commit(&s_fin[x]);
          }
        }
      } else if (warp == kWarpWV) {
        // ============ value waiter: A_v(g), B_v(g) ready -> release the value issuers; ring refills ============
        for (int p = 0; p < n_pages; ++p) {
          const uint32_t g = pg_base + p, x = g & 1;
          wait_k(&av_ready[x], g >> 1);
          wait_k(&bv_ready[x], g >> 1);
          group_sync<96>(kNbValue);
          // every consumer has read page p by now: its slot takes page p + NBUF
          if constexpr (PAGED) {
            if (p + NBUF < n_pages) {   // warp-uniform
              const int nxt = p + NBUF;
              if (nxt >= 32 * (win + 1)) {   // slide the window; the next one loads ~20 pages ahead
                blk_a = blk_b;
                ++win;
                const int i = 32 * (win + 1) + lane;
                blk_b = i < n_pages ? __ldg(trow + i) : 0;
              }
              const uint8_t* src = page_at(nxt);
              const uint8_t* far = nxt + kL2Ahead < n_pages ? page_at(nxt + kL2Ahead) : nullptr;
              if (lane == 0) {
                wait_k(&s_empty[ring_slot(p)], ring_use(p));
                const uint32_t si = ring_slot(nxt);
                fence_proxy_async();
                mbar_expect_tx(&s_full[si], PL::bytes);
                bulk_g2s(s_pages + si * C::PAGE, src, PL::bytes, &s_full[si]);
                issued = pg_base + nxt + 1;
                if (far) prefetch_l2(far, PL::bytes);
              }
            }
          } else {
            if (lane == 0 && p + NBUF < n_pages) {
              wait_k(&s_empty[ring_slot(p)], ring_use(p));
              const int nxt = p + NBUF;
              const uint32_t si = ring_slot(nxt);
              fence_proxy_async();
              mbar_expect_tx(&s_full[si], PL::bytes);
              bulk_g2s(s_pages + si * C::PAGE, page_at(nxt), PL::bytes, &s_full[si]);
              issued = pg_base + nxt + 1;
              if (nxt + kL2Ahead < n_pages)
                prefetch_l2(page_at(nxt + kL2Ahead), PL::bytes);
            }
          }
          __syncwarp();
        }
      } else if (warp == kWarpIV0 || warp == kWarpIV1) {
        // ============ value MMAs: D_v(plane)[coordinate][column] += A_v(plane) x B_v ============
        constexpr int HALF = PV / 2;
        const int pl0 = warp == kWarpIV0 ? 0 : HALF;
        const uint32_t bv0 = smem_u32(s_bv);
        uint64_t bd[2][2];
#pragma unroll
        for (int xb = 0; xb < 2; ++xb)
#pragma unroll
          for (int ks = 0; ks < 2; ++ks) bd[xb][ks] = smem_desc(bv0 + xb * C::BV_BYTES + ks * 256, 128, 512);
        for (int p = 0; p < n_pages; ++p) {
          const uint32_t g = pg_base + p, x = g & 1;
          const uint32_t av = tmem + C::TA_V + (AVB == 2 ? x : 0) * C::AV_COLS;
          group_sync<96>(kNbValue);
          if (lane == 0) {
            tc_fence_after();
            const uint32_t first = p == 0 ? 0u : 1u;   // a new segment restarts the accumulators
#pragma unroll
            for (int i = 0; i < HALF; ++i) {
              const int pl = pl0 + i;
              mma_f4_ts(tmem + C::TD_V + pl * NVC, av + 16 * pl, x ? bd[1][0] : bd[0][0], idesc_v, sfa, sfb, first);
              mma_f4_ts(tmem + C::TD_V + pl * NVC, av + 16 * pl + 8, x ? bd[1][1] : bd[0][1], idesc_v, sfa, sfb, 1u);
            }
            tc_commit(&v_fin[x]);
          }
        }
      } else if (warp >= kWarpK && warp < kWarpK + 4) {
        // ============ key-plane warps (TMEM lane = row, token slot slot_of_lane(row)) -> A_s ============
        const int tau = slot_of_lane(row);
        for (int p = 0; p < n_pages; ++p) {
          const uint32_t g = pg_base + p, x = g & 1;
          wait_k(&s_full[ring_slot(p)], ring_use(p));
          const uint8_t* pgp = pg_ptr(p);
          uint4 wk[BK + 1];
#pragma unroll
          for (int q = 0; q < BK; ++q)
            wk[q] = *reinterpret_cast<const uint4*>(pgp + PL::off_kcodes + ((size_t)q * 128 + tau) * 16);
          wk[BK] = *reinterpret_cast<const uint4*>(pgp + PL::off_signs + (size_t)tau * 16);
          uint32_t sc[4];   // n_k, gamma, n_v of this token slot (0 past the sequence end)
          {
            const bool valid = tau < min(128, seq_len - (p_lo + p) * 128);
            sc[0] = valid ? reinterpret_cast<const uint32_t*>(pgp + PL::off_nk)[tau] : 0u;
            sc[1] = valid ? reinterpret_cast<const uint32_t*>(pgp + PL::off_gamma)[tau] : 0u;
            sc[2] = valid ? reinterpret_cast<const uint32_t*>(pgp + PL::off_nv)[tau] : 0u;
            sc[3] = 0u;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&s_empty[ring_slot(p)]);
          uint4 xk[NS];   // key monomial planes, then the sign plane
          {
            uint4 kp[PK];
            monomial_words<BK, PK>(reinterpret_cast<const uint4(&)[BK]>(wk), kp);
#pragma unroll
            for (int i = 0; i < PK; ++i) xk[i] = kp[i];
            xk[PK] = wk[BK];
          }
          if (g >= (uint32_t)ASB) wait_k(&as_free[(g - ASB) & 1], (g - ASB) >> 1);   // A_s buffer free
          if (g >= 2) wait_k(&ds_free[x], (g >> 1) - 1);   // token warps read the scalars of page g-2
          tc_fence_after();
          tmem_st4(tl + C::TSC + 4 * x, sc);
#pragma unroll
          for (int pl = 0; pl < NS; ++pl) {
            uint32_t r[16];
            const uint32_t wv[4] = {xk[pl].x, xk[pl].y, xk[pl].z, xk[pl].w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint32_t o[4];
              expand_signed4(wv[c], o);
#pragma unroll
              for (int s = 0; s < 4; ++s) r[4 * c + s] = o[s];
            }
            tmem_st16(tl + C::TA_S + (ASB == 2 ? x : 0) * C::AS_COLS + 16 * pl, r);
          }
          tc_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&as_ready[x]);
        }
      } else if (warp >= kWarpV && warp < kWarpV + 4) {
        // ============ value-plane warps (TMEM lane = coordinate) -> A_v ============
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
          uint4 xv[PV];
          monomial_words<BV, PV>(wv, xv);
          if (g >= (uint32_t)AVB) wait_k(&v_fin[(g - AVB) & 1], (g - AVB) >> 1);   // A_v buffer free
          tc_fence_after();
#pragma unroll
          for (int pl = 0; pl < PV; ++pl) {
            uint32_t r[16];
            const uint32_t w4[4] = {xv[pl].x, xv[pl].y, xv[pl].z, xv[pl].w};
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              uint32_t o[4];
              expand_signed4(w4[c], o);
#pragma unroll
              for (int s = 0; s < 4; ++s) r[4 * c + s] = o[s];
            }
            tmem_st16(tl + C::TA_V + (AVB == 2 ? x : 0) * C::AV_COLS + 16 * pl, r);
          }
          tc_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&av_ready[x]);
        }
      } else if ((warp >= kWarpT && warp < kWarpT + 4) || (warp >= kWarpT2 && warp < kWarpWV)) {
        // ============ token warps: logits, lazy softmax, weight pieces -> B_v ============
        // set ts handles heads h0 .. h0 + HPT - 1: their D_s columns, D_v columns and B_v rows
        const int twarp = warp >= kWarpT2 ? 4 + (warp - kWarpT2) : warp - kWarpT;   // 0 .. 4 TS - 1
        const int ts = twarp >> 2, h0 = ts * HPT, q4 = warp & 3;
        const int tau = slot_of_lane(row);
        float m_run[HPT], l_part[HPT];
#pragma unroll
        for (int h = 0; h < HPT; ++h) {
          m_run[h] = -INFINITY;
          l_part[h] = 0.f;
        }
        float n_ref = 0.f;
        const int vote_id = ts == 0 ? kNbVote0 : kNbVote1 + ts - 1;
        for (int p = 0; p < n_pages; ++p) {
          const uint32_t g = pg_base + p, x = g & 1;
          const uint32_t db = DSB == 2 ? x : 0;
          const bool valid = tau < min(128, seq_len - (p_lo + p) * 128);
          wait_k(&s_fin[x], g >> 1);        // every score MMA of page p is done
          tc_fence_after();
          // this set's columns: head h at 8 h (key term) and 2 SCOLS + 8 h (sign term), two
          // heads per round of loads
          float lg[HPT];
          float nk, gmv, nvt;
          {
            uint32_t sc[4];
            tmem_ld4(tl + C::TSC + 4 * x, sc);
            tc_wait_ld();
            nk = __uint_as_float(sc[0]);
            gmv = __uint_as_float(sc[1]);
            nvt = __uint_as_float(sc[2]);
          }
          int ovf = nvt > n_ref;
          {
            const uint32_t base = tl + C::TD_S + db * NSC + ts * SCOLS;
            constexpr int HR = HPT < 2 ? HPT : 2;   // heads per round of loads
#pragma unroll
            for (int h2 = 0; h2 < HPT; h2 += HR) {
              uint32_t rk[HR][8], rq[HR][8];
#pragma unroll
              for (int u = 0; u < HR; ++u) {
                tmem_ld8(base + 8 * (h2 + u), rk[u]);
                tmem_ld8(base + TS * SCOLS + 8 * (h2 + u), rq[u]);
              }
              tc_wait_ld();
              if (h2 + HR >= HPT) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&ds_free[x]);
              }
#pragma unroll
              for (int u = 0; u < HR; ++u) {
                const int h = h2 + u, hg = h0 + h;
                const float2 hc = *reinterpret_cast<const float2*>(s_head + hg * 4 + 2);
                float sk = __uint_as_float(rk[u][kNQP - 1]), sq = __uint_as_float(rq[u][kNQP - 1]);
#pragma unroll
                for (int pc = kNQP - 2; pc >= 0; --pc) {
                  sk = fmaf(sk, 0.125f, __uint_as_float(rk[u][pc]));
                  sq = fmaf(sq, 0.125f, __uint_as_float(rq[u][pc]));
                }
                const float l = fmaf(nk * sk, hc.x, gmv * sq * hc.y);
                lg[h] = (valid && hg < G) ? l : -INFINITY;
                if (a.logits && valid && hg < G)
                  a.logits[((size_t)b * a.q_heads + (size_t)kvh * G + hg) * a.max_tokens + (size_t)(p_lo + p) * 128 + tau] = l;
                if (lg[h] > m_run[h] + kTau) ovf = 1;
              }
            }
          }
          float fh[HPT];
#pragma unroll
          for (int h = 0; h < HPT; ++h) fh[h] = 1.f;
          bool rescale = false;
          if (t_vote_or(vote_id, ovf)) {
#pragma unroll
            for (int h = 0; h <= HPT; ++h) {
              float mx = h < HPT ? lg[h] : nvt;
#pragma unroll
              for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
              if (lane == 0) s_red[twarp * (HPT + 1) + h] = mx;
            }
            t_sync(vote_id);
            float nvmax = 0.f;
            for (int w2 = 4 * ts; w2 < 4 * ts + 4; ++w2) nvmax = fmaxf(nvmax, s_red[w2 * (HPT + 1) + HPT]);
            const float n_new = nvmax > n_ref ? 1.25f * nvmax : n_ref;
#pragma unroll
            for (int h = 0; h < HPT; ++h) {
              float mx = -INFINITY;
              for (int w2 = 4 * ts; w2 < 4 * ts + 4; ++w2) mx = fmaxf(mx, s_red[w2 * (HPT + 1) + h]);
              const float m_new = fmaxf(m_run[h], mx);
              const float alpha = (m_run[h] == -INFINITY) ? 0.f : __expf(m_run[h] - m_new);
              fh[h] = (n_ref > 0.f) ? alpha * (n_ref / n_new) : 0.f;
              l_part[h] *= alpha;
              m_run[h] = m_new;
            }
            n_ref = n_new;
            rescale = p > 0;
            t_sync(vote_id);   // s_red reads done
          }
          if (rescale) {
            // D_v holds exactly the pages before p once the value MMAs of page p-1 are done;
            // this warp scales its lane quarter of this set's columns of every plane
            wait_k(&v_fin[(g - 1) & 1], (g - 1) >> 1);
            tc_fence_after();
#pragma unroll 1
            for (int pl = 0; pl < PV; ++pl) {
#pragma unroll
              for (int co = 0; co < VCOLS; co += 8) {
                const uint32_t col = C::TD_V + pl * NVC + ts * VCOLS + co;
                uint32_t rv[8];
                tmem_ld8(tl + col, rv);
                tc_wait_ld();
#pragma unroll
                for (int i = 0; i < 8; ++i) rv[i] = __float_as_uint(__uint_as_float(rv[i]) * fh[co / 8]);
                tmem_st8(tl + col, rv);
              }
            }
            tc_wait_st();
          }
          // softmax weights x = p n_v / n_ref -> Y = round(2^15 x); word h of this lane holds
          // head h0 + h with nibble k = bit pair (2k, 2k+1) of Y
          const float nvr = nvt * (n_ref > 0.f ? __frcp_rn(n_ref) : 0.f);
          uint32_t wb[HPT];
#pragma unroll
          for (int h = 0; h < HPT; ++h) {
            float pw = lg[h] == -INFINITY ? 0.f : __expf(lg[h] - m_run[h]);
            l_part[h] += pw;                   // the denominator keeps every position
            if (pw < sparse_v) pw = 0.f;       // Sparse V: the position's value is skipped
            uint32_t t = min(__float2uint_rn(pw * nvr * kWScale), 65535u);
            t = (t | (t << 8)) & 0x00FF00FFu;
            t = (t | (t << 4)) & 0x0F0F0F0Fu;
            t = (t | (t << 2)) & 0x33333333u;
            wb[h] = t;
          }
          // 8 x 8 nibble transpose among lanes 8c .. 8c + 7: lane 8c + r ends up with row r
          // (piece r) of the head, nibble i taken from lane 8c + i
#pragma unroll
          for (int h = 0; h < HPT; ++h) {
            uint32_t v = wb[h];
            {
              const uint32_t o = __shfl_xor_sync(0xffffffffu, v, 4);
              v = (lane & 4) ? ((o >> 16) | (v & 0xFFFF0000u)) : ((v & 0x0000FFFFu) | (o << 16));
            }
            {
              const uint32_t o = __shfl_xor_sync(0xffffffffu, v, 2);
              v = (lane & 2) ? (((o >> 8) & 0x00FF00FFu) | (v & 0xFF00FF00u)) : ((v & 0x00FF00FFu) | ((o << 8) & 0xFF00FF00u));
            }
            {
              const uint32_t o = __shfl_xor_sync(0xffffffffu, v, 1);
              v = (lane & 1) ? (((o >> 4) & 0x0F0F0F0Fu) | (v & 0xF0F0F0F0u)) : ((v & 0x0F0F0F0Fu) | ((o << 4) & 0xF0F0F0F0u));
            }
            wb[h] = v;
          }
          // B_v buffer of page p: its previous user, the value MMAs of page p-2, must be done
          if (g >= 2) wait_k(&v_fin[x], (g >> 1) - 1);
          uint8_t* bvb = s_bv + x * C::BV_BYTES;
          const int c = lane >> 3, r = lane & 7;
#pragma unroll
          for (int h = 0; h < HPT; ++h) {
            const int n = ts * VCOLS + 8 * h + r;   // head h0 + h, piece r
            *reinterpret_cast<uint32_t*>(bvb + canon_off(n, 16 * c + 4 * q4, 64)) = wb[h];
          }
          fence_proxy_async();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bv_ready[x]);
        }
        // per-head sums of this segment
#pragma unroll
        for (int h = 0; h < HPT; ++h) {
          float v = l_part[h];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
          if (lane == 0) s_red[twarp * (HPT + 1) + h] = v;
        }
        if ((twarp & 3) == 0 && lane == 0) s_f[ts] = n_ref;   // the set's first thread
        t_sync(vote_id);
        if ((twarp & 3) == 0 && lane < HPT && h0 + lane < G) {
          float l_tot = 0.f, mv = 0.f;
          for (int w2 = 4 * ts; w2 < 4 * ts + 4; ++w2) l_tot += s_red[w2 * (HPT + 1) + lane];
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
    __syncthreads();   // n_ref of both sets in s_f
    if (warp >= kWarpV && warp < kWarpV + 4) {
      // ---------- epilogue: o~_j = -(n_ref / 2^14) sum_M alpha_M sum_k 4^k D_v(M)[j][(h, k)] ----------
      float ov[GP];
#pragma unroll
      for (int h = 0; h < GP; ++h) ov[h] = 0.f;
      if (n_pages > 0) {
        {
          const uint32_t last = pg_base + n_pages - 1;   // the last value MMAs are done
          wait_k(&v_fin[last & 1], last >> 1);
        }
        tc_fence_after();
#pragma unroll 1
        for (int pl = 0; pl < PV; ++pl) {
          const float al = a.alpha_v[pl];
#pragma unroll
          for (int h = 0; h < GP; ++h) {   // head h: columns 8 h .. 8 h + kNPW - 1
            uint32_t r[8];
            tmem_ld8(tl + C::TD_V + pl * NVC + 8 * h, r);
            tc_wait_ld();
            float s = __uint_as_float(r[kNPW - 1]);
#pragma unroll
            for (int pc = kNPW - 2; pc >= 0; --pc) s = fmaf(s, 4.f, __uint_as_float(r[pc]));
            ov[h] = fmaf(al, s, ov[h]);
          }
        }
      }
#pragma unroll
      for (int h = 0; h < GP; ++h) {
        if (h >= G) continue;
        const float nref = n_pages > 0 ? s_f[h / HPT] : 0.f;   // n_ref of the set that owns head h
        rec[(size_t)h * (2 + D) + 2 + row] = n_pages > 0 ? -(nref * (2.f / kWScale)) * ov[h] : 0.f;
      }
    }
    pg_base += n_pages;
    tc_fence_before();
    __syncthreads();
    s_fail_seen = *s_fail != 0;
  }
  // teardown after a timeout: the last fill of each ring slot and every MMA the issuers
  // started complete (bounded waits) before the shared and tensor memory are released
  if (s_fail_seen && lane == 0) {
    if (warp == kWarpWV)
      for (uint32_t i = issued > (uint32_t)NBUF ? issued - NBUF : 0u; i < issued; ++i)
        mbar_wait(&s_full[i % NBUF], (i / NBUF) & 1);
    if (warp == kWarpIS || warp == kWarpIV0 || warp == kWarpIV1) {
      uint64_t* t = &td_bar[warp - kWarpIS];
      tc_commit(t);
      mbar_wait(t, 0);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace dtf
}  // namespace tq
