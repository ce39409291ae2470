// Device helpers shared by the decode kernels: bulk copies and mbarriers, e4m3 packing,
// bit-plane operand expansion (see bitplane.h).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "bitplane.h"

namespace tq {
namespace dev {

constexpr uint32_t kSpinLimit = 1u << 26;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

// 1-D bulk copy global -> shared, completing on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

// Non-blocking probe of the phase; on B300 several times cheaper than try_wait when the
// phase has already completed.
__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait: false once kWaitNs of wall time (or kSpinLimit polls) passed without the
// phase completing.  try_wait may suspend the thread for a while, so the bound is on time.
constexpr uint64_t kWaitNs = 2000000000ull;
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_test_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  for (uint32_t i = 1; i < kSpinLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 0 && global_ns() - t0 > kWaitNs) return false;
  }
  return false;
}

__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void mma_e4m3(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Two floats -> two e4m3 bytes (round to nearest even, saturating): low byte = lo_val.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float hi_val, float lo_val) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi_val), "f"(lo_val));
  return r;
}

// Two e4m3 bytes (low byte -> .x) back to floats.
__device__ __forceinline__ float2 e4m3x2_to_f2(uint32_t v) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)v));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

// Word w with its bit k of every byte turned into four e4m3 operands beta_k + gamma_k*bit.
template <int K>
__device__ __forceinline__ uint32_t expand(uint32_t w) {
  return (w & (0x01010101u << K)) | (e4m3_base(K) * 0x01010101u);
}
__device__ __forceinline__ uint32_t expand_rt(uint32_t w, uint32_t mask, uint32_t base) { return (w & mask) | base; }
// expand<K> with K known only after unrolling (the switch folds away).
__device__ __forceinline__ uint32_t expand_at(uint32_t w, int k) {
  switch (k & 7) {
    case 0: return expand<0>(w);
    case 1: return expand<1>(w);
    case 2: return expand<2>(w);
    case 3: return expand<3>(w);
    case 4: return expand<4>(w);
    case 5: return expand<5>(w);
    case 6: return expand<6>(w);
    default: return expand<7>(w);
  }
}

// Three-piece e4m3 split of v: v ~ hi + mid / 16 + lo / 256.  The later pieces are scaled
// up by 2^4 and 2^8 so that they stay in the normal range; they sit in separate MMA
// columns, and the epilogue applies the 2^-4 and 2^-8.
__device__ __forceinline__ void split3(float v, uint32_t& hi, uint32_t& mid, uint32_t& lo) {
  hi = cvt_e4m3x2(0.f, v) & 0xFF;
  float r1 = v - e4m3x2_to_f2(hi).x;
  mid = cvt_e4m3x2(0.f, 16.f * r1) & 0xFF;
  float r2 = r1 - 0.0625f * e4m3x2_to_f2(mid).x;
  lo = cvt_e4m3x2(0.f, 256.f * r2) & 0xFF;
}

// Four-piece split: v ~ p0 + p1 / 16 + p2 / 256 + p3 / 4096 (~2^-16 relative).
__device__ __forceinline__ void split4(float v, uint32_t (&pc)[4]) {
  float r = v;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    pc[k] = cvt_e4m3x2(0.f, r) & 0xFF;
    r = 16.f * (r - e4m3x2_to_f2(pc[k]).x);
  }
}

__device__ __forceinline__ float e4m3_val(uint32_t byte) { return e4m3x2_to_f2(byte).x; }
__device__ __forceinline__ float split3_val(uint32_t hi, uint32_t mid, uint32_t lo) {
  return e4m3_val(hi) + 0.0625f * e4m3_val(mid) + 0.00390625f * e4m3_val(lo);
}
__device__ __forceinline__ float split4_val(const uint32_t (&pc)[4]) {
  return e4m3_val(pc[0]) + 0.0625f * e4m3_val(pc[1]) + 0.00390625f * e4m3_val(pc[2]) +
         0.000244140625f * e4m3_val(pc[3]);
}


// ---------------------------------------------------------------- tcgen05 (5th-gen tensor cores)
// Tensor memory: 128 lanes x 512 columns of 32 bits per SM; address = (lane << 16) | column.
// A warp may access only its lane quarter 32 * (warp % 4) .. + 31.

__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {   // whole warp
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {       // whole warp
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 consecutive columns of this thread's lane <- r[0..31]
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
      "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
      "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
// one column of this thread's lane (call tc_wait_ld before use)
__device__ __forceinline__ uint32_t tmem_ld1(uint32_t taddr) {
  uint32_t r;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(r) : "r"(taddr) : "memory");
  return r;
}
__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(r) : "memory");
}
// r[0..3] <- 4 consecutive columns of this thread's lane (call tc_wait_ld before use)
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t (&r)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t (&r)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
               "r"(r[2]), "r"(r[3])
               : "memory");
}
// r[0..7] <- 8 consecutive columns of this thread's lane (call tc_wait_ld before use)
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr)
               : "memory");
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
// r[0..15] <- 16 consecutive columns of this thread's lane (call tc_wait_ld before use)
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
      "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}
// N = 4, 8 or 16 consecutive columns, chosen at compile time
template <int N>
__device__ __forceinline__ void tmem_ldn(uint32_t taddr, uint32_t (&r)[N]) {
  if constexpr (N == 4) tmem_ld4(taddr, r);
  else if constexpr (N == 8) tmem_ld8(taddr, r);
  else tmem_ld16(taddr, r);
}
template <int N>
__device__ __forceinline__ void tmem_stn(uint32_t taddr, const uint32_t (&r)[N]) {
  if constexpr (N == 4) tmem_st4(taddr, r);
  else if constexpr (N == 8) tmem_st8(taddr, r);
  else tmem_st16(taddr, r);
}

// Shared-memory matrix descriptor, no swizzle, K-major canonical layout: 8-row x 16-byte
// core matrices (128 contiguous bytes); lbo = byte distance between core matrices adjacent
// along K, sbo = byte distance between 8-row groups.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)((lbo >> 4) & 0x3FFF) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) | ((uint64_t)1 << 46);
}
// Byte offset of element (row, kbyte) in that layout with lbo = 128 and rows of kbytes bytes.
__host__ __device__ __forceinline__ uint32_t canon_off(uint32_t row, uint32_t kbyte, uint32_t kbytes) {
  return (row >> 3) * (kbytes / 16) * 128 + (kbyte >> 4) * 128 + (row & 7) * 16 + (kbyte & 15);
}

// Instruction descriptor (kind::f16 / kind::f8f6f4): D format (1 = f32), A/B formats
// (f16 kind: 0 f16, 1 bf16; f8f6f4 kind: 0 e4m3, 1 e5m2), K-major A and B, N >> 3, M >> 4.
__host__ __device__ constexpr uint32_t make_idesc(uint32_t afmt, uint32_t bfmt, uint32_t M, uint32_t N) {
  return (1u << 4) | (afmt << 7) | (bfmt << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T, e4m3 operands, issued by one thread.
__device__ __forceinline__ void mma_f8_ts(uint32_t d_taddr, uint32_t a_taddr, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_taddr),
      "r"(a_taddr), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc]^T, 8-bit operands (kind::f8f6f4), one thread.
__device__ __forceinline__ void mma_f8_ss(uint32_t d_taddr, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_taddr),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc]^T, 16-bit operands, issued by one thread.
__device__ __forceinline__ void mma_f16_ss(uint32_t d_taddr, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_taddr),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc]^T, 16-bit operands (A: 2 elements per column).
__device__ __forceinline__ void mma_f16_ts(uint32_t d_taddr, uint32_t a_taddr, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_taddr),
      "r"(a_taddr), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrives once on `bar` when every tcgen05.mma issued so far by this thread has completed.
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

}  // namespace dev
}  // namespace tq

namespace tq {
namespace dev {

// ---------------------------------------------------------------- 4-bit (e2m1) operands
// Two floats -> two e2m1 nibbles in one byte (round to nearest even, saturating at +-6):
// low nibble = lo_val.  e2m1 values: +-{0, 0.5, 1, 1.5, 2, 3, 4, 6}.
__device__ __forceinline__ uint32_t cvt_e2m1x2(float hi_val, float lo_val) {
  uint16_t r;
  asm("{\n .reg .b8 t;\n cvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n cvt.u16.u8 %0, t;\n}"
      : "=h"(r)
      : "f"(hi_val), "f"(lo_val));
  return r;
}
// Two e2m1 nibbles (low nibble -> .x) back to floats.
__device__ __forceinline__ float2 e2m1x2_to_f2(uint32_t v) {
  uint32_t h2;
  asm("{\n .reg .b8 t;\n cvt.u8.u16 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}" : "=r"(h2) : "h"((uint16_t)v));
  __half2 h = *reinterpret_cast<__half2*>(&h2);
  return __half22float2(h);
}

// Instruction descriptor of kind::mxf4 (block-scaled e2m1 x e2m1 -> f32, K = 64): A and B
// formats e2m1, K-major, N >> 3, ue8m0 scale factors, M >> 4, scale-factor ids 0.
__host__ __device__ constexpr uint32_t make_idesc_mxf4(uint32_t M, uint32_t N) {
  return (1u << 7) | (1u << 10) | ((N >> 3) << 17) | (1u << 23) | ((M >> 4) << 24);
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T, packed e2m1 operands (64 per 32 bytes), one scale
// factor per 32 elements of K from tensor memory (sfa, sfb), issued by one thread.
__device__ __forceinline__ void mma_f4_ts(uint32_t d_taddr, uint32_t a_taddr, uint64_t b_desc, uint32_t idesc,
                                          uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], [%1], %2, %3, [%4], [%5], p;\n}\n" ::"r"(
          d_taddr),
      "r"(a_taddr), "l"(b_desc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}

// The words of every odd-subset ("monomial") plane of a slot row, built once per page with
// the subset masks folded at compile time: xp[pl] = XOR of w[q] over the bits q of subset pl.
template <int NB, int NP>
__device__ __forceinline__ void monomial_words(const uint4 (&w)[NB], uint4 (&xp)[NP]) {
#pragma unroll
  for (int pl = 0; pl < NP; ++pl) {
    uint4 x = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int q = 0; q < NB; ++q)
      if ((mono_mask16(pl) >> q) & 1) {
        x.x ^= w[q].x;
        x.y ^= w[q].y;
        x.z ^= w[q].z;
        x.w ^= w[q].w;
      }
    xp[pl] = x;
  }
}

// A plane word w (32 bits, element k at bit k) as four words of signed e2m1 operands: output
// word s holds, in nibble i, +1 (0x2) if bit 4i + s of w is 0 and -1 (0xA) if it is 1.
__device__ __forceinline__ void expand_signed4(uint32_t w, uint32_t (&o)[4]) {
  o[0] = ((w << 3) & 0x88888888u) | 0x22222222u;
  o[1] = ((w << 2) & 0x88888888u) | 0x22222222u;
  o[2] = ((w << 1) & 0x88888888u) | 0x22222222u;
  o[3] = (w & 0x88888888u) | 0x22222222u;
}

}  // namespace dev
}  // namespace tq
