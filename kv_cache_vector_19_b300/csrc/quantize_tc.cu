// tq_quantize_kv on 5th-generation tensor cores (tcgen05, kind::f16, bf16), head_dim 128.
//
// [BLOG] "Технология TurboQuant и её применение с локальными LLM", section 1.2: every key
// and value vector is rotated by the random orthogonal Pi and each rotated coordinate of
// y / ||x|| gets its Lloyd-Max code (b-1 bits for keys, b for values); for keys the residual
// r = x - DEQUANT(idx) is projected by the Gaussian S and only sign(S r) and ||r|| are kept.
// The residual is projected in the rotated frame: S r = S' (Pi r) with S' = S Pi^T and
// Pi r = y - n c[idx].
//
// The three d x d contractions run on tcgen05 with fp32 accumulators in tensor memory.  K
// and V are exact in bf16; Pi, S' and the rotated residual are split into bf16 hi + lo:
//   Y   = X Pi_hi^T + X Pi_lo^T                       (keys and values, 2 x 8 MMAs each)
//   Z   = R_hi S'_hi^T + R_hi S'_lo^T + R_lo S'_hi^T   (keys, 3 x 8 MMAs, R in tensor memory)
// which keeps the rotation within ~2^-17 relative, far below what moves a code or a sign
// except at a quantizer boundary.
//
// Persistent CTAs (one per SM): the bf16 operand blob (Pi hi/lo, S' hi/lo, 128 KB) is
// copied into shared memory once; every work item is the slots of one page that the call
// writes, for one (batch, KV head).  Per item: the K and V rows are staged in the no-swizzle
// K-major layout (norms accumulated on the way), the elected thread issues the rotation
// MMAs, warps 0-3 (tensor-memory lane = slot) code the keys and write the residual split
// into tensor memory, warps 4-7 code the values; then the projection MMAs, the sign bits,
// and the bit packing into the page.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "dev_common.cuh"
#include "layout.cuh"
#include "tq_internal.h"

namespace tq {
namespace qtc {

using namespace dev;

constexpr int kThreads = 256;
constexpr int kRowPad = 132;   // bytes per slot row of the value-code staging (bank-conflict free)
// shared memory
constexpr int OFF_B = 0;                       // Pi_hi, Pi_lo, S'_hi, S'_lo: 4 x 32 KB, canonical
constexpr int B_BYTES = 4 * 128 * 256;
constexpr int OFF_K = OFF_B + B_BYTES;         // K rows (32 KB), later key-code staging unused
constexpr int OFF_V = OFF_K + 128 * 256;       // V rows (32 KB), later value-code staging
constexpr int OFF_NK = OFF_V + 128 * 256;      // [128] f32
constexpr int OFF_NV = OFF_NK + 512;           // [128] f32
constexpr int OFF_CB = OFF_NV + 512;           // ck[16] tk[16] cv[32] tv[32] f32
constexpr int OFF_MBAR = OFF_CB + 96 * 4;      // blob, mma
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
  const uint8_t* blob;   // bf16 operand blob, canonical layout
  const float* ck;
  const float* tk;
  const float* cv;
  const float* tv;
  int* status;
};

__device__ __forceinline__ uint32_t bf16_bits(float x) {
  return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x));
}
__device__ __forceinline__ float bf16_val(uint32_t bits) {
  return __bfloat162float(__ushort_as_bfloat16((unsigned short)bits));
}

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
  float* s_ck = reinterpret_cast<float*>(smem + OFF_CB);
  float* s_tk = s_ck + 16;
  float* s_cv = s_tk + 16;
  float* s_tv = s_cv + 32;
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
  constexpr uint32_t idesc = make_idesc(1, 1, 128, 128);   // bf16 x bf16 -> f32, M = N = 128
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
    uint8_t* pg = a.cache + ((size_t)seq * a.pages_per_seq + page) * (size_t)PL::bytes;
    const __nv_bfloat16* kseq = a.k + (size_t)seq * a.n_tokens * D;
    const __nv_bfloat16* vseq = a.v + (size_t)seq * a.n_tokens * D;

    // ---- stage K and V rows (slots outside [lo, hi) are zero); row norms on the way ----
    __syncthreads();   // previous item done with sK / sV
    if (*s_fail) break;   // uniform: a bounded wait gave up
    if (tid == 0) {
      // the rows of this CTA's next item into L2 while this one is processed
      const int nx = item + (int)gridDim.x;
      if (nx < n_items) {
        const int nip = nx % a.items_per_seq, nseq = nx / a.items_per_seq;
        const int nstart = a.start_pos[nseq / a.kv_heads];
        if (nstart >= 0 && nstart <= a.max_tokens - a.n_tokens) {
          const int npage = nstart / 128 + nip;
          const int nlo = max(nstart, npage * 128), nhi = min(nstart + a.n_tokens, npage * 128 + 128);
          if (nlo < nhi) {
            const size_t off = ((size_t)nseq * a.n_tokens + (size_t)(nlo - nstart)) * D;
            prefetch_l2(a.k + off, (uint32_t)(nhi - nlo) * D * 2);
            prefetch_l2(a.v + off, (uint32_t)(nhi - nlo) * D * 2);
          }
        }
      }
    }
#pragma unroll 4
    for (int it = 0; it < 8; ++it) {
      const int c = tid + kThreads * it;   // 16-byte chunk: slot c / 16, chunk c % 16
      const int slot = c >> 4, kc = c & 15;
      uint4 xk = make_uint4(0u, 0u, 0u, 0u), xv = make_uint4(0u, 0u, 0u, 0u);
      if (slot >= lo && slot < hi) {
        const long tok = (long)page * 128 + slot - start;
        xk = __ldg(reinterpret_cast<const uint4*>(kseq + tok * D) + kc);
        xv = __ldg(reinterpret_cast<const uint4*>(vseq + tok * D) + kc);
      }
      const uint32_t off = canon_off(slot, 16 * kc, 256);
      *reinterpret_cast<uint4*>(sK + off) = xk;
      *reinterpret_cast<uint4*>(sV + off) = xv;
      float sk = 0.f, sv = 0.f;
      const uint32_t wk[4] = {xk.x, xk.y, xk.z, xk.w}, wv[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float k0 = bf16_val(wk[i] & 0xFFFF), k1 = bf16_val(wk[i] >> 16);
        const float v0 = bf16_val(wv[i] & 0xFFFF), v1 = bf16_val(wv[i] >> 16);
        sk = fmaf(k0, k0, fmaf(k1, k1, sk));
        sv = fmaf(v0, v0, fmaf(v1, v1, sv));
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) {   // the 16 chunks of a slot are 16 consecutive lanes
        sk += __shfl_xor_sync(0xffffffffu, sk, o);
        sv += __shfl_xor_sync(0xffffffffu, sv, o);
      }
      if (kc == 0) {
        sNk[slot] = sqrtf(sk);
        sNv[slot] = sqrtf(sv);
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
      // ---------- keys: codes, residual in the rotated frame, bf16 split into tensor memory ----------
#pragma unroll
      for (int q = 0; q < BK; ++q)
#pragma unroll
        for (int w = 0; w < 4; ++w) kwords[q][w] = 0u;
      const float n = sNk[row];
      const float inv = n > 0.f ? 1.f / n : 0.f;
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 32) {
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
        uint32_t rh[16], rl[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          float r2[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int j = c0 + i + u;
            const float yv = __uint_as_float(y[i + u]);
            const float yh = yv * inv;
            int idx = 0;
#pragma unroll
            for (int t = 0; t < LK - 1; ++t) idx += (yh >= s_tk[t]) ? 1 : 0;
            // bit position of coordinate j inside its key-code word (layout of the page format)
            const int w = (j >> 2) & 3, bit = 2 * (j >> 5) + ((j >> 4) & 1) + 8 * (j & 3);
#pragma unroll
            for (int q = 0; q < BK; ++q) kwords[q][w] |= (uint32_t)((idx >> q) & 1) << bit;
            r2[u] = yv - n * s_ck[idx];
            gamma2 = fmaf(r2[u], r2[u], gamma2);
          }
          const uint32_t h0 = bf16_bits(r2[0]), h1 = bf16_bits(r2[1]);
          const uint32_t l0 = bf16_bits(r2[0] - bf16_val(h0)), l1 = bf16_bits(r2[1] - bf16_val(h1));
          rh[i >> 1] = h0 | (h1 << 16);
          rl[i >> 1] = l0 | (l1 << 16);
        }
        tmem_st16(tl + T_RHI + (c0 >> 1), rh);
        tmem_st16(tl + T_RLO + (c0 >> 1), rl);
      }
      tc_wait_st();
    } else {
      // ---------- values: codes into the byte staging (slot-major rows, padded) ----------
      const float n = sNv[row];
      const float inv = n > 0.f ? 1.f / n : 0.f;
      uint8_t* dst = sV + row * kRowPad;   // sV's rows were consumed by the MMAs
#pragma unroll 1
      for (int c0 = 0; c0 < 128; c0 += 16) {
        uint32_t y[16];
        tmem_ld16(tl + T_YV + c0, y);
        tc_wait_ld();
        uint32_t packed[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float yh = __uint_as_float(y[i]) * inv;
          int idx = 0;
#pragma unroll
          for (int t = 0; t < LV - 1; ++t) idx += (yh >= s_tv[t]) ? 1 : 0;
          packed[i >> 2] |= (uint32_t)idx << (8 * (i & 3));
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) *reinterpret_cast<uint32_t*>(dst + c0 + 4 * i) = packed[i];
      }
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
#pragma unroll
      for (int c0 = 0; c0 < 128; c0 += 16) {
        uint32_t z[16];
        tmem_ld16(tl + T_Z + c0, z);
        tc_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int j = c0 + i;
          const int w = (j >> 2) & 3, bit = 2 * (j >> 5) + ((j >> 4) & 1) + 8 * (j & 3);
          swords[w] |= (__uint_as_float(z[i]) >= 0.f ? 1u : 0u) << bit;
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
        reinterpret_cast<float*>(pg + PL::off_gamma)[row] = sqrtf(gamma2);
        reinterpret_cast<float*>(pg + PL::off_nv)[row] = sNv[row];
      }
    } else {
      // value-code words [plane][coordinate][4], each over 32 slots of the page; the page
      // layout puts slot tau = 32 kb + 16 h + 4 c + e at word c, bit 2 kb + h + 8 e
      uint32_t* g_vc = reinterpret_cast<uint32_t*>(pg + PL::off_vcodes);
      const int t4 = tid - 128;
#pragma unroll 1
      for (int e = t4; e < BV * D * 4; e += 128) {
        const int plane = e / (D * 4), rem = e % (D * 4), j = rem >> 2, c = rem & 3;
        uint32_t word = 0u, mask = 0u;
#pragma unroll
        for (int bit = 0; bit < 32; ++bit) {
          const int kb = (bit & 7) >> 1, h = bit & 1, el = bit >> 3;
          const int slot = 32 * kb + 16 * h + 4 * c + el;
          if (slot >= lo && slot < hi) {
            mask |= 1u << bit;
            word |= (uint32_t)((sV[slot * kRowPad + j] >> plane) & 1) << bit;
          }
        }
        uint32_t* dst = g_vc + ((size_t)plane * D + j) * 4 + c;
        if (mask == 0xffffffffu) {
          *dst = word;
        } else if (mask != 0u) {
          atomicAnd(dst, ~mask);
          atomicOr(dst, word);
        }
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
           const int32_t* start_pos, void* cache, int max_tokens, cudaStream_t st) {
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
  a.ck = c->d_ck;
  a.tk = c->d_tk;
  a.cv = c->d_cv;
  a.tv = c->d_tv;
  a.status = c->d_status;
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
                       const int32_t* start_pos, void* cache, int max_tokens, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (c->d != 128 || !c->d_qblob) return TQ_EUNSUPPORTED;
  switch (c->bits) {
    case 2: return qtc::launch<2>(c, k, v, batch, kv_heads, n_tokens, start_pos, cache, max_tokens, st);
    case 3: return qtc::launch<3>(c, k, v, batch, kv_heads, n_tokens, start_pos, cache, max_tokens, st);
    case 4: return qtc::launch<4>(c, k, v, batch, kv_heads, n_tokens, start_pos, cache, max_tokens, st);
    case 5: return qtc::launch<5>(c, k, v, batch, kv_heads, n_tokens, start_pos, cache, max_tokens, st);
    default: return TQ_EUNSUPPORTED;
  }
}

}  // namespace tq
