// tq_ip_topk: the compressed inner-product scan (top-k over the cached keys).
//
// [BLOG] "Технология TurboQuant и её применение с локальными LLM", section 6.4 (research
// directions: vector search, compressing the indexes of RAG systems) and its FAQ (the method
// applies to any high-dimensional vectors).  For a cached key t the estimate of <q, x_t> is the
// decode score times sqrt(d),
//     <q, k^_t> = n_t <Pi q, c_K[idx_t]> + gamma_t sqrt(pi/2)/m <S q, 2 sigma_t - 1>
// (the QJL term only when the keys keep it).  The scan takes the scores from tq_attn_decode's
// logits output (the decode kernel that serves the context), then selects per query head the k
// largest by (score descending, slot ascending) over the order-preserving integer image of the
// fp32 scores.  One pass histograms the top 12 bits and finds the bin that holds the k-th key;
// a second pass gathers every key of that bin or above (fewer than k above it, plus the bin)
// into shared memory, and a bitonic sort of (key, slot) pairs orders them.  When the bin is too
// full for shared memory, a radix select over the remaining 20 bits (three more passes) finds
// the k-th key exactly and only the top k are gathered.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kThreads = 1024;
constexpr int kTopBits = 12;            // bits of the first histogram
constexpr int kBins = 1 << kTopBits;
constexpr int kCap = 4096;              // (key, slot) pairs kept in shared memory
static_assert(kCap >= TQ_TOPK_MAX, "the fallback gathers the top k into the same buffer");

// Order-preserving image of an fp32 value as an unsigned integer (larger value, larger key);
// -0 is taken as +0 so that equal scores make equal keys.
__device__ __forceinline__ uint32_t ordered(float f) {
  const uint32_t u = f == 0.0f ? 0u : __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Sort key of one candidate: larger score first, then lower slot.
__device__ __forceinline__ unsigned long long pair_key(uint32_t u, int t) {
  return ((unsigned long long)u << 32) | (0xFFFFFFFFu - (uint32_t)t);
}

// Calls f(t, ordered(s[t] * scale)) for every t < n, once, spread over the block: a scalar head
// up to the first 16-byte boundary, 16-byte loads (two in flight per thread), a scalar tail.  The
// key is that of the returned estimate, so that estimates equal in fp32 tie.
template <class F>
__device__ __forceinline__ void for_each_key(const float* s, int n, float scale, F&& f) {
  const int tid = threadIdx.x;
  const int head = min(n, (int)(((16u - ((uint32_t)(uintptr_t)s & 15u)) & 15u) >> 2));
  if (tid < head) f(tid, ordered(s[tid] * scale));
  const int nv = (n - head) >> 2;
  const float4* v = reinterpret_cast<const float4*>(s + head);
  auto four = [&](int i, float4 x) {
    const int t = head + 4 * i;
    f(t, ordered(x.x * scale));
    f(t + 1, ordered(x.y * scale));
    f(t + 2, ordered(x.z * scale));
    f(t + 3, ordered(x.w * scale));
  };
  int i = tid;
  for (; i + kThreads < nv; i += 2 * kThreads) {
    const float4 a = v[i], b = v[i + kThreads];
    four(i, a);
    four(i + kThreads, b);
  }
  if (i < nv) four(i, v[i]);
  const int t = head + 4 * nv + tid;
  if (t < n) f(t, ordered(s[t] * scale));
}

// Inclusive prefix sum of one int per thread over the block.
__device__ __forceinline__ int block_incl_scan(int v, int* s_warp) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) s_warp[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const int w = s_warp[lane];
    int y = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int z = __shfl_up_sync(0xffffffffu, y, o);
      if (lane >= o) y += z;
    }
    s_warp[lane] = y - w;
  }
  __syncthreads();
  const int r = s_warp[warp] + x;
  __syncthreads();
  return r;
}

// Exclusive prefix sum of one flag per thread over the block; returns the thread's offset and
// writes the block total.
__device__ __forceinline__ int block_scan(int flag, int* s_warp, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t bal = __ballot_sync(0xffffffffu, flag);
  const int in_warp = __popc(bal & ((1u << lane) - 1u));
  if (lane == 0) s_warp[warp] = __popc(bal);
  __syncthreads();
  if (warp == 0) {
    int v = s_warp[lane];
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    s_warp[lane] = incl - v;
    if (lane == 31) *total = incl;
  }
  __syncthreads();
  const int r = s_warp[warp] + in_warp;
  __syncthreads();
  return r;
}

struct Shared {
  union {
    uint32_t hist[kBins];
    unsigned long long c[kCap];
  } u;
  int warp[32];
  int cnt, total, bin, above, binc;
  uint32_t prefix, mask, remaining;
};

// One CTA per (query head, batch row).
__global__ void __launch_bounds__(kThreads) topk_kernel(const float* __restrict__ logits,
                                                        const int32_t* __restrict__ seq_lens, int q_heads,
                                                        int max_tokens, int k, float scale, int32_t* __restrict__ out_idx,
                                                        float* __restrict__ out_score, int* status) {
  __shared__ Shared sh;
  const int tid = threadIdx.x;
  const size_t row = (size_t)blockIdx.y * q_heads + blockIdx.x;
  int n = seq_lens[blockIdx.y];
  if (n < 0 || n > max_tokens) {
    if (tid == 0 && blockIdx.x == 0) atomicOr(status, kFlagBounds);
    n = n < 0 ? 0 : max_tokens;
  }
  const float* s = logits + row * (size_t)max_tokens;
  const int kk = min(k, n);
  int m = 0;   // candidates in sh.u.c
  if (kk > 0) {
    // ---- histogram of the top 12 bits; the bin of the kk-th key ----
    for (int i = tid; i < kBins; i += kThreads) sh.u.hist[i] = 0u;
    if (tid == 0) sh.cnt = 0;
    __syncthreads();
    for_each_key(s, n, scale, [&](int, uint32_t u) { atomicAdd(&sh.u.hist[u >> (32 - kTopBits)], 1u); });
    __syncthreads();
    {
      constexpr int kPer = kBins / kThreads;   // thread i holds the bins of rank [kPer i, kPer i + kPer) from the top
      const int b0 = kBins - kPer * (tid + 1);
      int own = 0;
#pragma unroll
      for (int j = 0; j < kPer; ++j) own += (int)sh.u.hist[b0 + j];
      const int incl = block_incl_scan(own, sh.warp);
      int cum = incl - own;
      if (cum < kk && incl >= kk) {
        for (int j = kPer - 1; j >= 0; --j) {
          const int h = (int)sh.u.hist[b0 + j];
          if (cum + h >= kk) {
            sh.bin = b0 + j;
            sh.above = cum;
            sh.binc = h;
            break;
          }
          cum += h;
        }
      }
      __syncthreads();
    }
    const uint32_t bin = (uint32_t)sh.bin;
    const int above = sh.above;
    if (above + sh.binc <= kCap) {
      // ---- gather the bin and everything above it ----
      m = above + sh.binc;
      __syncthreads();   // the histogram is dead; its space holds the pairs
      for_each_key(s, n, scale, [&](int t, uint32_t u) {
        if ((u >> (32 - kTopBits)) >= bin) sh.u.c[atomicAdd(&sh.cnt, 1)] = pair_key(u, t);
      });
    } else {
      // ---- radix select of the kk-th key over the remaining 20 bits ----
      if (tid == 0) {
        sh.prefix = bin << (32 - kTopBits);
        sh.mask = ~0u << (32 - kTopBits);
        sh.remaining = (uint32_t)(kk - above);
      }
      for (int pass = 0; pass < 3; ++pass) {
        const int shift = pass == 0 ? 12 : pass == 1 ? 4 : 0;
        const uint32_t dmask = pass == 2 ? 15u : 255u;
        __syncthreads();
        for (int i = tid; i < 256; i += kThreads) sh.u.hist[i] = 0u;
        __syncthreads();
        const uint32_t prefix = sh.prefix, mask = sh.mask;
        for_each_key(s, n, scale, [&](int, uint32_t u) {
          if ((u & mask) == prefix) atomicAdd(&sh.u.hist[(u >> shift) & dmask], 1u);
        });
        __syncthreads();
        if (tid == 0) {
          uint32_t cum = 0u;
          const uint32_t rem = sh.remaining;
          for (int dg = (int)dmask; dg >= 0; --dg) {
            const uint32_t h = sh.u.hist[dg];
            if (cum + h >= rem) {
              sh.remaining = rem - cum;
              sh.prefix = prefix | ((uint32_t)dg << shift);
              sh.mask = mask | (dmask << shift);
              break;
            }
            cum += h;
          }
        }
      }
      __syncthreads();
      const uint32_t K = sh.prefix;
      const int need_eq = (int)sh.remaining;   // keys equal to K that belong to the top kk
      // keys above K (fewer than kk), in any order; then the lowest slots equal to K
      for_each_key(s, n, scale, [&](int t, uint32_t u) {
        if (u > K) sh.u.c[atomicAdd(&sh.cnt, 1)] = pair_key(u, t);
      });
      __syncthreads();
      const int base = sh.cnt;
      int taken = 0;
      for (int t0 = 0; t0 < n && taken < need_eq; t0 += kThreads) {   // uniform loop
        const int t = t0 + tid;
        const int flag = t < n && ordered(s[t] * scale) == K;
        const int off = block_scan(flag, sh.warp, &sh.total);
        if (flag && taken + off < need_eq) sh.u.c[base + taken + off] = pair_key(K, t);
        taken += sh.total;   // read by every thread between the scan's barriers and the next
        __syncthreads();
      }
      m = kk;
    }
  }
  // ---- bitonic sort of the m pairs, descending, over the next power of two ----
  int p2 = 1;
  while (p2 < m) p2 <<= 1;
  __syncthreads();
  for (int i = m + tid; i < p2; i += kThreads) sh.u.c[i] = 0ull;   // padding sorts last
  __syncthreads();
  for (int size = 2; size <= p2; size <<= 1) {
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      for (int i = tid; i < p2; i += kThreads) {
        const int j = i ^ stride;
        if (j > i) {
          const bool desc = (i & size) == 0;
          const unsigned long long a = sh.u.c[i], b = sh.u.c[j];
          if (desc ? a < b : a > b) {
            sh.u.c[i] = b;
            sh.u.c[j] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int i = tid; i < k; i += kThreads) {
    int32_t slot = -1;
    float sc = -INFINITY;
    if (i < kk) {
      slot = (int32_t)(0xFFFFFFFFu - (uint32_t)(sh.u.c[i] & 0xFFFFFFFFull));
      sc = s[slot] * scale;
    }
    out_idx[row * k + i] = slot;
    out_score[row * k + i] = sc;
  }
}

}  // namespace

int launch_topk(const tq_ctx* c, const float* logits, const int32_t* seq_lens, int batch, int q_heads,
                int max_tokens, int k, int32_t* out_idx, float* out_score, void* stream) {
  const float scale = sqrtf((float)c->d);   // logits carry 1/sqrt(d)
  topk_kernel<<<dim3(q_heads, batch), kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      logits, seq_lens, q_heads, max_tokens, k, scale, out_idx, out_score, c->d_status);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ECUDA;
}

}  // namespace tq
