// Device-side view of the version-1 compressed page (layout documented in tq.h).
#pragma once

#include <cstdint>

namespace tq {

template <int D, int BITS>
struct PageLayout {
  static constexpr int P = 128;
  static constexpr int M = D;                  // QJL projection size
  static constexpr int BK = BITS - 1;          // key code planes
  static constexpr int BV = BITS;              // value code planes
  static constexpr int KW = D / 32;            // words per slot per key plane
  static constexpr int SW = M / 32;            // sign words per slot
  static constexpr int off_kcodes = 0;
  static constexpr int off_signs = off_kcodes + BK * P * KW * 4;
  static constexpr int off_nk = off_signs + P * SW * 4;
  static constexpr int off_gamma = off_nk + P * 4;
  static constexpr int off_vcodes = off_gamma + P * 4;
  static constexpr int off_nv = off_vcodes + BV * D * 4 * 4;
  static constexpr int bytes = off_nv + P * 4;
};

// Coordinate j of a slot's key-code / sign words -> (word, bit).
template <int DD>
__host__ __device__ inline void coord_pos(int j, int& word, int& bit) {
  int kb = j >> 5, h = (j >> 4) & 1, c = (j >> 2) & 3, e = j & 3;
  int s = c * (2 * (DD / 32)) + 2 * kb + h;
  word = s >> 3;
  bit = (s & 7) + 8 * e;
}

// Inverse of coord_pos: (word, bit) -> coordinate.
template <int DD>
__host__ __device__ inline int coord_of(int word, int bit) {
  int s = word * 8 + (bit & 7), e = bit >> 3;
  int c = s / (2 * (DD / 32)), rem = s % (2 * (DD / 32));
  int kb = rem >> 1, h = rem & 1;
  return 32 * kb + 16 * h + 4 * c + e;
}

// Token slot tau of a coordinate's 4 value-code words -> (word, bit).
__host__ __device__ inline void slot_pos(int tau, int& word, int& bit) {
  int kb = tau >> 5, h = (tau >> 4) & 1, c = (tau >> 2) & 3, e = tau & 3;
  word = c;
  bit = 2 * kb + h + 8 * e;
}

// Inverse of slot_pos.
__host__ __device__ inline int slot_of(int word, int bit) {
  int kb = (bit & 7) >> 1, h = bit & 1, e = bit >> 3;
  return 32 * kb + 16 * h + 4 * word + e;
}

}  // namespace tq
