// tq_quantize_kv on 5th-generation tensor cores (tcgen05, kind::f16, fp16 pieces), head_dim 128.
//
// [BLOG] "Технология TurboQuant и её применение с локальными LLM", section 1.2: every key
// and value vector is rotated by the random orthogonal Pi and each rotated coordinate of
// y / ||x|| gets its Lloyd-Max code (b-1 bits for keys, b for values); for keys the residual
// r = x - DEQUANT(idx) is projected by the Gaussian S and only sign(S r) and ||r|| are kept.
// The residual is projected in the rotated frame: S r = S' (Pi r) with S' = S Pi^T and
// Pi r = y - n c[idx].
//
// The three d x d contractions run on tcgen05 with fp32 accumulators in tensor memory.  Every
// K / V row is scaled by a power of two (its largest magnitude into [2^14, 2^15)) and is then
// exact in fp16; 256 Pi, 256 S' and the scaled rotated residual are split into fp16 hi + lo:
//   Y   = X Pi_hi^T + X Pi_lo^T                       (keys and values, 2 x 8 MMAs each)
//   Z   = R_hi S'_hi^T + R_hi S'_lo^T + R_lo S'_hi^T   (keys, 3 x 8 MMAs, R in tensor memory)
// which keeps the rotation within ~2^-20 of ||x||.  A code whose yhat lands within 2^-18 of a
// boundary, or a sign whose projection lands within 2^-14 ||r|| of zero, is taken again in
// double-float arithmetic (exact.cuh) by the warp that owns the row, so the page holds the
// decisions of exact arithmetic.
//
// Persistent CTAs (one per SM): the fp16 operand blob (Pi hi/lo, S' hi/lo, 128 KB) is
// copied into shared memory once; every work item is the slots of one page that the call
// writes, for one (batch, KV head).  Per item: the K and V rows are staged in the no-swizzle
// K-major layout (norms accumulated on the way), the elected thread issues the rotation
// MMAs, warps 0-3 (tensor-memory lane = slot) code the keys and write the residual split
// into tensor memory, warps 4-7 code the values; then the projection MMAs, the sign bits,
// and the bit packing into the page.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include <cuda_fp16.h>

#include "dev_common.cuh"
#include "exact.cuh"
#include "layout.cuh"
#include "tq_internal.h"

namespace tq {
namespace qtc {

using namespace dev;

constexpr int kThreads = 256;
// shared memory
constexpr int OFF_B = 0;                       // Pi_hi, Pi_lo, S'_hi, S'_lo: 4 x 32 KB, canonical
constexpr int B_BYTES = 4 * 128 * 256;
constexpr int OFF_K = OFF_B + B_BYTES;         // K rows (32 KB), later key-code staging unused
constexpr int OFF_V = OFF_K + 128 * 256;       // V rows (32 KB), later value-code staging
constexpr int OFF_NK = OFF_V + 128 * 256;      // [128] f32  ||k|| (stored)
constexpr int OFF_NV = OFF_NK + 512;           // [128] f32  ||v|| (stored)
constexpr int OFF_SK = OFF_NV + 512;           // [128] f32  256 ||2^s k||: yhat = Y / this
constexpr int OFF_SV = OFF_SK + 512;           // [128] f32  256 ||2^s v||
constexpr int OFF_EK = OFF_SV + 512;           // [128] i32  s of each key row
constexpr int OFF_CB = OFF_EK + 512;           // ck[16] tk[16] cv[32] tv[32] nk[32] nv[64] f32
constexpr int OFF_MBAR = OFF_CB + 192 * 4;     // blob, mma
constexpr int OFF_MISC = OFF_MBAR + 16;        // tmem base, fail flag
constexpr int SMEM = OFF_MISC + 16;
// tensor memory columns
constexpr int T_YK = 0, T_YV = 128, T_Z = 256, T_RHI = 384, T_RLO = 448, T_COLS = 512;

struct QArgs {
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  int kv_heads, n_tokens, max_tokens, pages_per_seq, batch, items_per_seq;
  const int32_t* start_pos;
  uint8_t* cache;
  const uint8_t* blob;   // fp16 operand blob, canonical layout
  const float* exact;    // exact-decision tables
  const float* ck;
  const float* tk;
  const float* cv;
  const float* tv;
  int* status;
  PageMap pm;
  KVLayout lay;          // element strides of k and v over (batch, KV head, token)
};

__device__ __forceinline__ float bf16_val(uint32_t bits) { return __uint_as_float(bits << 16); }
// 2^e for e in [-126, 127]
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }
__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }
// largest biased exponent among the 8 bf16 values of a 16-byte chunk
__device__ __forceinline__ uint32_t max_exp8(uint4 w) {
  const uint32_t a = max((w.x >> 7) & 0xFFu, (w.x >> 23) & 0xFFu), b = max((w.y >> 7) & 0xFFu, (w.y >> 23) & 0xFFu);
  const uint32_t c = max((w.z >> 7) & 0xFFu, (w.z >> 23) & 0xFFu), d = max((w.w >> 7) & 0xFFu, (w.w >> 23) & 0xFFu);
  return max(max(a, b), max(c, d));
}
// 8 bf16 values times 2^s as fp16 (exact unless below fp16's normal range), and their sum of
// squares added to acc
__device__ __forceinline__ uint4 scale_to_f16(uint4 w, float f, float& acc) {
  const uint32_t in[4] = {w.x, w.y, w.z, w.w};
  uint32_t out[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float x0 = bf16_val(in[i] & 0xFFFFu) * f, x1 = bf16_val(in[i] >> 16) * f;
    acc = fmaf(x0, x0, fmaf(x1, x1, acc));
    out[i] = h2_bits(__floats2half2_rn(x0, x1));
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}
// scaled residual of one key coordinate (kept as one expression for the fix-up path)
__device__ __forceinline__ float key_resid(float yv, float nk, float c, float g) { return (yv - nk * c) * g; }
// bit of coordinate j inside its key-code / sign word (page layout, head_dim 128)
__device__ __forceinline__ int kbit(int j) { return 2 * (j >> 5) + ((j >> 4) & 1) + 8 * (j & 3); }

template <int BITS>
__global__ void __launch_bounds__(kThreads, 1) quantize_tc_kernel(QArgs a) {
  using PL = PageLayout<128, BITS>;
  constexpr int D = 128, BK = BITS - 1, BV = BITS, LK = 1 << BK, LV = 1 << BV;
  extern __shared__ __align__(1024) unsigned char smem[];
  uint8_t* sB = smem + OFF_B;
  uint8_t* sK = smem + OFF_K;
  uint8_t* sV = smem + OFF_V;
  float* sNk = reinterpret_cast<float*>(smem + OFF_NK);
  float* sNv = reinterpret_cast<float*>(smem + OFF_NV);
  float* sSk = reinterpret_cast<float*>(smem + OFF_SK);
  float* sSv = reinterpret_cast<float*>(smem + OFF_SV);
  int* sEk = reinterpret_cast<int*>(smem + OFF_EK);
  float* s_ck = reinterpret_cast<float*>(smem + OFF_CB);
  float* s_tk = s_ck + 16;
  float* s_cv = s_tk + 16;
  float* s_tv = s_cv + 32;
  const float2* s_nk = reinterpret_cast<const float2*>(s_tv + 32);   // near tables, one float2 per cell
  const float2* s_nv = s_nk + 16;
  const exact::Tables T = exact::tables(a.exact, 128);
  uint64_t* bar_blob = reinterpret_cast<uint64_t*>(smem + OFF_MBAR);
  uint64_t* bar_mma = bar_blob + 1;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  volatile int* s_fail = reinterpret_cast<volatile int*>(smem + OFF_MISC + 4);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row = 32 * (warp & 3) + lane;   // tensor-memory lane = page slot
  const int n_items = a.batch * a.kv_heads * a.items_per_seq;
  if ((int)blockIdx.x >= n_items) return;

  if (warp == 0) tmem_alloc(s_tmem, T_COLS);
  if (tid == 0) {
    mbar_init(bar_blob, 1);
    mbar_init(bar_mma, 1);
    *s_fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  for (int i = tid; i < LK; i += kThreads) s_ck[i] = a.ck[i];
  for (int i = tid; i < LK - 1; i += kThreads) s_tk[i] = a.tk[i];
  for (int i = tid; i < LV; i += kThreads) s_cv[i] = a.cv[i];
  for (int i = tid; i < LV - 1; i += kThreads) s_tv[i] = a.tv[i];
  for (int i = tid; i < 2 * LK; i += kThreads) s_tv[32 + i] = T.nkt[i];
  for (int i = tid; i < 2 * LV; i += kThreads) s_tv[64 + i] = T.nvt[i];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t tl = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
  if (tid == 0) {
    mbar_expect_tx(bar_blob, B_BYTES);
    bulk_g2s(sB, a.blob, B_BYTES, bar_blob);
  }
  if (!mbar_wait(bar_blob, 0)) *s_fail = 1;
  uint32_t n_mma = 0;   // commits on bar_mma so far
  constexpr uint32_t idesc = make_idesc(0, 0, 128, 128);   // f16 x f16 -> f32, M = N = 128
  const uint32_t sB_addr = smem_u32(sB), sK_addr = smem_u32(sK), sV_addr = smem_u32(sV);

  for (int item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int ip = item % a.items_per_seq, seq = item / a.items_per_seq;
    const int b = seq / a.kv_heads;
    const int start = a.start_pos[b];
    if (start < 0 || start > a.max_tokens - a.n_tokens) {   // uniform per item
      if (tid == 0 && ip == 0) atomicOr(a.status, kFlagBounds);
      continue;
    }
    const int page = start / 128 + ip;
    const int lo = max(start, page * 128) - page * 128;
    const int hi = min(start + a.n_tokens, page * 128 + 128) - page * 128;
    if (lo >= hi) continue;
    uint8_t* pg = a.cache + a.pm.index(seq, a.kv_heads, a.pages_per_seq, page, a.status) * PL::bytes;
    const int hkv = seq - b * a.kv_heads;
    const __nv_bfloat16* kseq = a.k + (b * a.lay.kb + hkv * a.lay.kh);   // token i at kseq + i kt
    const __nv_bfloat16* vseq = a.v + (b * a.lay.vb + hkv * a.lay.vh);

    // ---- stage K and V rows (slots outside [lo, hi) are zero); row norms on the way ----
    __syncthreads();   // previous item done with sK / sV
    if (*s_fail) break;   // uniform: a bounded wait gave up
    if (warp == 0) {
      // the rows of this CTA's next item into L2 while this one is processed, when they are one
      // contiguous range (row-by-row prefetches of strided rows cost more than they saved:
      // 6.27 ms against 4.98 ms for a token-major long-context prefill)
      const int nx = item + (int)gridDim.x;
      if (nx < n_items) {
        const int nip = nx % a.items_per_seq, nseq = nx / a.items_per_seq;
        const int nb = nseq / a.kv_heads, nh = nseq - nb * a.kv_heads;
        const int nstart = a.start_pos[nb];
        if (nstart >= 0 && nstart <= a.max_tokens - a.n_tokens) {
          const int npage = nstart / 128 + nip;
          const int nlo = max(nstart, npage * 128), nhi = min(nstart + a.n_tokens, npage * 128 + 128);
          if (nlo < nhi) {
            const __nv_bfloat16* nk = a.k + (nb * a.lay.kb + nh * a.lay.kh + (nlo - nstart) * a.lay.kt);
            const __nv_bfloat16* nv = a.v + (nb * a.lay.vb + nh * a.lay.vh + (nlo - nstart) * a.lay.vt);
            if (a.lay.kt == D && a.lay.vt == D) {
              if (lane == 0) {
                prefetch_l2(nk, (uint32_t)(nhi - nlo) * D * 2);
                prefetch_l2(nv, (uint32_t)(nhi - nlo) * D * 2);
              }
            }
          }
        }
      }
    }
    // 8 operand rows per warp and group; lane (s8, k4) takes 16-byte chunks k4, k4 + 4, ...
    // (a store of the warp covers 8 rows x 64 bytes: conflict free).  K rows are in slot order;
    // V row r holds slot slot_of(r >> 5, r & 31), so that the value coders' ballots are words.
    {
      const int s8 = lane & 7, k4 = lane >> 3;
#pragma unroll 1
      for (int grp = warp; grp < 16; grp += 8) {
        const int r = 8 * grp + s8, vs = slot_of(r >> 5, r & 31);
        const bool kval = r >= lo && r < hi, vval = vs >= lo && vs < hi;
        const uint4* kp = reinterpret_cast<const uint4*>(kseq + ((long)page * 128 + r - start) * a.lay.kt);
        const uint4* vp = reinterpret_cast<const uint4*>(vseq + ((long)page * 128 + vs - start) * a.lay.vt);
        uint4 xk[4], xv[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          xk[q] = kval ? __ldg(kp + k4 + 4 * q) : make_uint4(0u, 0u, 0u, 0u);
          xv[q] = vval ? __ldg(vp + k4 + 4 * q) : make_uint4(0u, 0u, 0u, 0u);
        }
        // the row's scale 2^s: its largest magnitude into [2^14, 2^15)
        uint32_t ek = 0u, ev = 0u;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          ek = max(ek, max_exp8(xk[q]));
          ev = max(ev, max_exp8(xv[q]));
        }
        ek = max(ek, __shfl_xor_sync(0xffffffffu, ek, 8));
        ek = max(ek, __shfl_xor_sync(0xffffffffu, ek, 16));
        ev = max(ev, __shfl_xor_sync(0xffffffffu, ev, 8));
        ev = max(ev, __shfl_xor_sync(0xffffffffu, ev, 16));
        const int sk = min(141 - (int)ek, 126), sv = min(141 - (int)ev, 126);
        float nk2 = 0.f, nv2 = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t off = canon_off(r, 16 * (k4 + 4 * q), 256);
          *reinterpret_cast<uint4*>(sK + off) = scale_to_f16(xk[q], exp2i(sk), nk2);
          *reinterpret_cast<uint4*>(sV + off) = scale_to_f16(xv[q], exp2i(sv), nv2);
        }
        nk2 += __shfl_xor_sync(0xffffffffu, nk2, 8);
        nk2 += __shfl_xor_sync(0xffffffffu, nk2, 16);
        nv2 += __shfl_xor_sync(0xffffffffu, nv2, 8);
        nv2 += __shfl_xor_sync(0xffffffffu, nv2, 16);
        if (k4 == 0) {
          const float rk = sqrtf(nk2), rv = sqrtf(nv2);
          sNk[r] = ldexpf(rk, -sk);   // by slot
          sNv[r] = ldexpf(rv, -sv);   // by V row
          sSk[r] = 256.f * rk;
          sSv[r] = 256.f * rv;
          sEk[r] = sk;
        }
      }
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    // ---- rotation MMAs ----
    if (tid == 0) {
      tc_fence_after();
#pragma unroll 1
      for (int part = 0; part < 2; ++part) {            // Pi_hi, Pi_lo
        const uint32_t bsel = sB_addr + part * 32768;
#pragma unroll 1
        for (int ks = 0; ks < 8; ++ks) {
          const uint64_t bd = smem_desc(bsel + ks * 256, 128, 2048);
          mma_f16_ss(tmem + T_YK, smem_desc(sK_addr + ks * 256, 128, 2048), bd, idesc, part | ks);
          mma_f16_ss(tmem + T_YV, smem_desc(sV_addr + ks * 256, 128, 2048), bd, idesc, part | ks);
        }
      }
      tc_commit(bar_mma);
    }
    ++n_mma;
    if (!mbar_wait(bar_mma, (n_mma - 1) & 1)) *s_fail = 1;
    tc_fence_after();
    const bool valid = row >= lo && row < hi;
    uint32_t kwords[BK][4];   // key-code plane words of this slot
    float gamma2 = 0.f;
    if (warp < 4) {
      // ---------- keys: codes, residual in the rotated frame, fp16 split into tensor memory ----------
#pragma unroll
      for (int q = 0; q < BK; ++q)
#pragma unroll
        for (int w = 0; w < 4; ++w) kwords[q][w] = 0u;
      const float nk = sSk[row];   // Y / nk = yhat
      const float inv = nk > 0.f ? 1.f / nk : 0.f;
      // the residual's fp16 scale: |Y - nk c| <= 2 nk, brought below 2^15
      const int en = (int)((__float_as_uint(nk) >> 23) & 0xFFu) - 127;
      const float g = exp2i(max(-126, min(126, 13 - en)));
      // chunks of 32 coordinates: coordinate c0 + i sits in word (i >> 2) & 3 at bit
      // 2 (c0 >> 5) + ((i >> 4) & 1) + 8 (i & 3)
#pragma unroll 1
      for (int c0 = 0; c0 < 128; c0 += 32) {
        const int kb0 = 2 * (c0 >> 5);
        uint32_t y[32];
        {
          uint32_t t0[16], t1[16];
          tmem_ld16(tl + T_YK + c0, t0);
          tmem_ld16(tl + T_YK + c0 + 16, t1);
          tc_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            y[i] = t0[i];
            y[16 + i] = t1[i];
          }
        }
        uint32_t rh[16], rl[16], near = 0u;
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          float r2[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const float yv = __uint_as_float(y[i + u]);
            const float yh = yv * inv;
            int idx = 0;
#pragma unroll
            for (int t = 0; t < LK - 1; ++t) idx += (yh >= s_tk[t]) ? 1 : 0;
            const float2 cw = s_nk[idx];
            near |= (fabsf(yh - cw.x) > cw.y ? 1u : 0u) << (i + u);
            const int w = ((i + u) >> 2) & 3, bit = kb0 + (((i + u) >> 4) & 1) + 8 * ((i + u) & 3);
#pragma unroll
            for (int q = 0; q < BK; ++q) kwords[q][w] |= (uint32_t)((idx >> q) & 1) << bit;
            r2[u] = key_resid(yv, nk, s_ck[idx], g);
            gamma2 = fmaf(r2[u], r2[u], gamma2);
          }
          const __half2 h = __floats2half2_rn(r2[0], r2[1]);
          rh[i >> 1] = h2_bits(h);
          rl[i >> 1] = h2_bits(__floats2half2_rn(r2[0] - __low2float(h), r2[1] - __high2float(h)));
        }
        tmem_st16(tl + T_RHI + (c0 >> 1), rh);
        tmem_st16(tl + T_RLO + (c0 >> 1), rl);
        if (!(nk > 0.f)) near = 0u;
        uint32_t lanes = __ballot_sync(0xffffffffu, near != 0u);
        if (lanes) {
          // codes next to a boundary: exact decision, then the row's words, residual and gamma
          tc_wait_st();
          while (lanes) {
            const int L = __ffs(lanes) - 1;
            lanes &= lanes - 1;
            uint32_t m = __shfl_sync(0xffffffffu, near, L);
            const __nv_bfloat16* xr = kseq + ((long)page * 128 + 32 * (warp & 3) + L - start) * a.lay.kt;
            while (m) {
              const int j = c0 + __ffs(m) - 1;
              m &= m - 1;
              const int idx2 = exact::code_of_row<128>(xr, T.pih, T.pil, j, T.tkh, T.tkl, LK - 1, lane);
              const uint32_t yj = tmem_ld1(tl + T_YK + j);
              uint32_t hc = tmem_ld1(tl + T_RHI + (j >> 1)), lc = tmem_ld1(tl + T_RLO + (j >> 1));
              tc_wait_ld();
              if (lane == L) {
                const float yv = __uint_as_float(yj), yh = yv * inv;
                int idx = 0;
#pragma unroll
                for (int t = 0; t < LK - 1; ++t) idx += (yh >= s_tk[t]) ? 1 : 0;
                if (idx != idx2) {
                  const int w = (j >> 2) & 3, bit = kbit(j);
#pragma unroll
                  for (int q = 0; q < BK; ++q)
#pragma unroll
                    for (int ww = 0; ww < 4; ++ww)
                      if (ww == w)
                        kwords[q][ww] = (kwords[q][ww] & ~(1u << bit)) | ((uint32_t)((idx2 >> q) & 1) << bit);
                  const float r0 = key_resid(yv, nk, s_ck[idx], g), r1 = key_resid(yv, nk, s_ck[idx2], g);
                  gamma2 = fmaf(r1, r1, fmaf(-r0, r0, gamma2));
                  const __half h = __float2half_rn(r1);
                  const __half l = __float2half_rn(r1 - __half2float(h));
                  const int sh = 16 * (j & 1);
                  hc = (hc & ~(0xFFFFu << sh)) | ((uint32_t)__half_as_ushort(h) << sh);
                  lc = (lc & ~(0xFFFFu << sh)) | ((uint32_t)__half_as_ushort(l) << sh);
                }
              }
              tmem_st1(tl + T_RHI + (j >> 1), hc);
              tmem_st1(tl + T_RLO + (j >> 1), lc);
              tc_wait_st();
            }
          }
        }
      }
      tc_wait_st();
    } else {
      // ---------- values: V row 32 c + lane holds slot slot_of(c, lane), so one ballot per
      // (coordinate, plane) is the page word (plane, coordinate, c); lane i keeps coordinate c0 + i's ----------
      const int c = warp & 3, vrow = 32 * c + lane, slot = slot_of(c, lane);
      const float nv = sSv[vrow];
      const float inv = nv > 0.f ? 1.f / nv : 0.f;
      const bool vvalid = slot >= lo && slot < hi;
      const uint32_t vmask = __ballot_sync(0xffffffffu, vvalid);
      uint32_t* g_vc = reinterpret_cast<uint32_t*>(pg + PL::off_vcodes);
#pragma unroll 1
      for (int c0 = 0; c0 < 128; c0 += 16) {
        uint32_t y[16];
        tmem_ld16(tl + T_YV + c0, y);
        tc_wait_ld();
        uint32_t ib[4] = {0u, 0u, 0u, 0u}, near = 0u;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float yh = __uint_as_float(y[i]) * inv;
          int idx = 0;
#pragma unroll
          for (int t = 0; t < LV - 1; ++t) idx += (yh >= s_tv[t]) ? 1 : 0;
          const float2 cw = s_nv[idx];
          near |= (fabsf(yh - cw.x) > cw.y ? 1u : 0u) << i;
          ib[i >> 2] |= (uint32_t)idx << (8 * (i & 3));
        }
        uint32_t wv[BV];
#pragma unroll
        for (int p = 0; p < BV; ++p) wv[p] = 0u;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const uint32_t idx = (ib[i >> 2] >> (8 * (i & 3))) & 0xFFu;
#pragma unroll
          for (int p = 0; p < BV; ++p) {
            const uint32_t bal = __ballot_sync(0xffffffffu, (idx >> p) & 1u);
            if (lane == i) wv[p] = bal;
          }
        }
        if (!(nv > 0.f)) near = 0u;
        uint32_t lanes = __ballot_sync(0xffffffffu, near != 0u);
        while (lanes) {   // codes next to a boundary: exact decision, into the keeper lane's words
          const int L = __ffs(lanes) - 1;
          lanes &= lanes - 1;
          uint32_t m = __shfl_sync(0xffffffffu, near, L);
          const __nv_bfloat16* xr = vseq + ((long)page * 128 + __shfl_sync(0xffffffffu, slot, L) - start) * a.lay.vt;
          while (m) {
            const int cc = __ffs(m) - 1;
            m &= m - 1;
            const int idx2 = exact::code_of_row<128>(xr, T.pih, T.pil, c0 + cc, T.tvh, T.tvl, LV - 1, lane);
            if (lane == cc) {
#pragma unroll
              for (int p = 0; p < BV; ++p) wv[p] = (wv[p] & ~(1u << L)) | ((uint32_t)((idx2 >> p) & 1) << L);
            }
          }
        }
        if (vmask && lane < 16) {
#pragma unroll
          for (int p = 0; p < BV; ++p) {
            uint32_t* dst = g_vc + ((size_t)p * D + c0 + lane) * 4 + c;
            if (vmask == 0xffffffffu) {
              *dst = wv[p];
            } else {
              atomicAnd(dst, ~vmask);
              atomicOr(dst, wv[p] & vmask);
            }
          }
        }
      }
      if (vvalid) reinterpret_cast<float*>(pg + PL::off_nv)[slot] = sNv[vrow];
    }
    tc_fence_before();
    __syncthreads();
    // ---- projection MMAs: Z = R_hi S'_hi^T + R_hi S'_lo^T + R_lo S'_hi^T ----
    if (tid == 0) {
      tc_fence_after();
#pragma unroll 1
      for (int part = 0; part < 3; ++part) {
        const uint32_t a_col = part == 2 ? T_RLO : T_RHI;
        const uint32_t bsel = sB_addr + (part == 1 ? 3 : 2) * 32768;
#pragma unroll 1
        for (int ks = 0; ks < 8; ++ks)
          mma_f16_ts(tmem + T_Z, tmem + a_col + 8 * ks, smem_desc(bsel + ks * 256, 128, 2048), idesc, part | ks);
      }
      tc_commit(bar_mma);
    }
    ++n_mma;
    if (warp < 4) {
      if (!mbar_wait(bar_mma, (n_mma - 1) & 1)) *s_fail = 1;
      tc_fence_after();
      uint32_t swords[4] = {0u, 0u, 0u, 0u};
      // z = 256 sum_j (g 2^s r_j) S'[i][j]: near zero when within kDeltaSign ||r|| in those units
      const float zthr = exact::kDeltaSign * 256.f * sqrtf(gamma2);
#pragma unroll 1
      for (int c0 = 0; c0 < 128; c0 += 16) {
        uint32_t z[16];
        tmem_ld16(tl + T_Z + c0, z);
        tc_wait_ld();
        uint32_t near = 0u;
#pragma unroll
        for (int i = 0; i < 16; ++i) {   // c0 % 16 == 0: word (i >> 2) & 3
          const float zv = __uint_as_float(z[i]);
          swords[(i >> 2) & 3] |= (zv >= 0.f ? 1u : 0u) << (2 * (c0 >> 5) + ((c0 >> 4) & 1) + 8 * (i & 3));
          near |= (fabsf(zv) < zthr ? 1u : 0u) << i;
        }
        uint32_t lanes = __ballot_sync(0xffffffffu, near != 0u);
        while (lanes) {   // projections next to zero: exact sign
          const int L = __ffs(lanes) - 1;
          lanes &= lanes - 1;
          uint32_t m = __shfl_sync(0xffffffffu, near, L);
          // this lane's 4 codes (coordinates 4 lane + e) of row L: word lane & 3 of each plane
          int codes[4] = {0, 0, 0, 0};
#pragma unroll
          for (int q = 0; q < BK; ++q) {
            const uint32_t w0 = __shfl_sync(0xffffffffu, kwords[q][0], L), w1 = __shfl_sync(0xffffffffu, kwords[q][1], L);
            const uint32_t w2 = __shfl_sync(0xffffffffu, kwords[q][2], L), w3 = __shfl_sync(0xffffffffu, kwords[q][3], L);
            const int w = lane & 3;
            const uint32_t kw = w == 0 ? w0 : w == 1 ? w1 : w == 2 ? w2 : w3;
#pragma unroll
            for (int e = 0; e < 4; ++e) codes[e] |= (int)((kw >> kbit(4 * lane + e)) & 1u) << q;
          }
          const __nv_bfloat16* xr = kseq + ((long)page * 128 + 32 * (warp & 3) + L - start) * a.lay.kt;
          while (m) {
            const int i = c0 + __ffs(m) - 1;
            m &= m - 1;
            const bool sg = exact::sign_of_row<128>(xr, codes, T.sh, T.sl, T.qh, T.ql, T.ckh, T.ckl, i, lane);
            if (lane == L) {
              const int w = (i >> 2) & 3, bit = kbit(i);
#pragma unroll
              for (int ww = 0; ww < 4; ++ww)
                if (ww == w) swords[ww] = (swords[ww] & ~(1u << bit)) | ((sg ? 1u : 0u) << bit);
            }
          }
        }
      }
      if (valid) {
        uint32_t* g_kc = reinterpret_cast<uint32_t*>(pg + PL::off_kcodes);
#pragma unroll
        for (int q = 0; q < BK; ++q)
          *reinterpret_cast<uint4*>(g_kc + ((size_t)q * 128 + row) * 4) =
              make_uint4(kwords[q][0], kwords[q][1], kwords[q][2], kwords[q][3]);
        *reinterpret_cast<uint4*>(pg + PL::off_signs + (size_t)row * 16) =
            make_uint4(swords[0], swords[1], swords[2], swords[3]);
        reinterpret_cast<float*>(pg + PL::off_nk)[row] = sNk[row];
        // gamma = ||g 2^(s+8) r|| / (g 2^(s+8)), g = 2^(13 - exponent of nk)
        const int en = (int)((__float_as_uint(sSk[row]) >> 23) & 0xFFu) - 127;
        reinterpret_cast<float*>(pg + PL::off_gamma)[row] =
            ldexpf(sqrtf(gamma2), -(sEk[row] + 8) - max(-126, min(126, 13 - en)));
      }
    }
  }
  if (*s_fail && tid == 0) {
    atomicOr(a.status, kFlagTimeout);
    mbar_wait(bar_blob, 0);                               // bounded: copies and MMAs in flight
    if (n_mma > 0) mbar_wait(bar_mma, (n_mma - 1) & 1);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, T_COLS);
  }
}

template <int BITS>
int launch(const tq_ctx* c, const void* k, const void* v, int batch, int kv_heads, int n_tokens,
           const int32_t* start_pos, void* cache, int max_tokens, cudaStream_t st, const PageMap& pm,
           const KVLayout& lay) {
  QArgs a;
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.kv_heads = kv_heads;
  a.n_tokens = n_tokens;
  a.max_tokens = max_tokens;
  a.pages_per_seq = (max_tokens + 127) / 128;
  a.batch = batch;
  a.items_per_seq = (n_tokens + 127) / 128 + 1;   // pages a run of n_tokens can touch
  a.start_pos = start_pos;
  a.cache = static_cast<uint8_t*>(cache);
  a.blob = c->d_qblob;
  a.exact = c->d_exact;
  a.ck = c->d_ck;
  a.tk = c->d_tk;
  a.cv = c->d_cv;
  a.tv = c->d_tv;
  a.status = c->d_status;
  a.pm = pm;
  a.lay = lay;
  const long items = (long)batch * kv_heads * a.items_per_seq;
  const int grid = (int)(items < c->num_sms ? items : c->num_sms);
  quantize_tc_kernel<BITS><<<grid, kThreads, SMEM, st>>>(a);
  return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ECUDA;
}

}  // namespace qtc

int prepare_quantize_tc(const tq_ctx* c) {
  if (c->d != 128) return TQ_OK;
  auto set = [](const void* fn) {
    return cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, qtc::SMEM) == cudaSuccess;
  };
  bool okv = true;
  if (c->bits == 2) okv = set((const void*)qtc::quantize_tc_kernel<2>);
  if (c->bits == 3) okv = set((const void*)qtc::quantize_tc_kernel<3>);
  if (c->bits == 4) okv = set((const void*)qtc::quantize_tc_kernel<4>);
  if (c->bits == 5) okv = set((const void*)qtc::quantize_tc_kernel<5>);
  return okv ? TQ_OK : TQ_ECUDA;
}

int launch_quantize_tc(const tq_ctx* c, const void* k, const void* v, int batch, int kv_heads, int n_tokens,
                       const int32_t* start_pos, void* cache, int max_tokens, const KVLayout& lay, void* stream,
                       const PageMap& pm) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (c->d != 128 || !c->d_qblob) return TQ_EUNSUPPORTED;
  switch (c->bits) {
    case 2: return qtc::launch<2>(c, k, v, batch, kv_heads, n_tokens, start_pos, cache, max_tokens, st, pm, lay);
    case 3: return qtc::launch<3>(c, k, v, batch, kv_heads, n_tokens, start_pos, cache, max_tokens, st, pm, lay);
    case 4: return qtc::launch<4>(c, k, v, batch, kv_heads, n_tokens, start_pos, cache, max_tokens, st, pm, lay);
    case 5: return qtc::launch<5>(c, k, v, batch, kv_heads, n_tokens, start_pos, cache, max_tokens, st, pm, lay);
    default: return TQ_EUNSUPPORTED;
  }
}

}  // namespace tq
