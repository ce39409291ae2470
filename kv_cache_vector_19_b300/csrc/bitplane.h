// Bit-plane arithmetic shared by the host set-up and the tensor-core decode kernel.
//
// 1. Centroids as affine functions of the code bits.  A code idx of n bits has bits
//    b_q = (idx >> q) & 1 and signs s_q = 2 b_q - 1.  Any function of idx is a sum of
//    products of signs over subsets M of the bits (a Walsh-Hadamard expansion).  A
//    Lloyd-Max book for a symmetric density is antisymmetric, c[L-1-idx] = -c[idx], so only
//    subsets of odd size survive.  For odd |M| the product of signs equals 2 x_M - 1 with
//    x_M the XOR of the bits in M, hence
//        c[idx] = 2 sum_M alpha_M x_M(idx) - sum_M alpha_M,
//        alpha_M = (1/L) sum_idx c[idx] prod_{q in M} s_q(idx).
//    With n bits there are 2^(n-1) odd subsets; mono_mask(i) lists them in increasing order
//    (the list for n bits is a prefix of the list for n+1 bits).
//
// 2. A plane word as four fp8 (e4m3) operands.  For a bit position k of every byte, the
//    e4m3 byte (w & (0x01 << k)) | base_k is an exact e4m3 number beta_k + gamma_k * bit:
//      k      0      1      2      3      4      5       6      7
//      base   0x38   0x38   0x38   0x30   0x28   0x18    0x00   0x38
//      beta   1      1      1      0.5    0.25   0.0625  0      1
//      gamma  0.125  0.25   0.5    0.5    0.75   0.9375  2      -2
//    (0x38 = 1.0; bits 0-2 are mantissa bits over it, bits 3-6 complete an exponent to 1.0
//    or 2.0, bit 7 is the sign).  One AND-OR per 32-bit word yields four operands.
#pragma once

#include <cstdint>

namespace tq {

__host__ __device__ constexpr int popcount_c(int m) { return m == 0 ? 0 : (m & 1) + popcount_c(m >> 1); }

// i-th positive integer with an odd number of set bits (1, 2, 4, 7, 8, 11, 13, 14, ...).
__host__ __device__ constexpr int mono_mask(int i) {
  int m = 1, c = 0;
  while (true) {
    if (popcount_c(m) & 1) {
      if (c == i) return m;
      ++c;
    }
    ++m;
  }
}

// The first 16 values of mono_mask without a loop, so that device code calling it with an
// unrolled loop counter folds to constants.
__host__ __device__ constexpr int mono_mask16(int i) {
  return i == 0 ? 1 : i == 1 ? 2 : i == 2 ? 4 : i == 3 ? 7 : i == 4 ? 8 : i == 5 ? 11 : i == 6 ? 13 : i == 7 ? 14
       : i == 8 ? 16 : i == 9 ? 19 : i == 10 ? 21 : i == 11 ? 22 : i == 12 ? 25 : i == 13 ? 26 : i == 14 ? 28 : 31;
}
static_assert(mono_mask16(3) == mono_mask(3) && mono_mask16(7) == mono_mask(7) && mono_mask16(12) == mono_mask(12) &&
                  mono_mask16(15) == mono_mask(15),
              "odd-popcount table");

__host__ __device__ constexpr uint32_t e4m3_base(int k) {
  return k == 3 ? 0x30u : k == 4 ? 0x28u : k == 5 ? 0x18u : k == 6 ? 0x00u : 0x38u;
}
__host__ __device__ constexpr float e4m3_beta(int k) {
  return k == 3 ? 0.5f : k == 4 ? 0.25f : k == 5 ? 0.0625f : k == 6 ? 0.0f : 1.0f;
}
__host__ __device__ constexpr float e4m3_gamma(int k) {
  return k == 0 ? 0.125f : k == 1 ? 0.25f : k == 2 ? 0.5f : k == 3 ? 0.5f : k == 4 ? 0.75f
       : k == 5 ? 0.9375f : k == 6 ? 2.0f : -2.0f;
}

}  // namespace tq
