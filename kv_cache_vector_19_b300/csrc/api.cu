// C ABI of the library: context set-up, argument checks, kernel dispatch, status.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <new>
#include <vector>

#include <cuda_fp16.h>

#include "bitplane.h"
#include "exact.cuh"
#include "tq_internal.h"

namespace {

bool supported(int d, int bits, int m) {
  return (d == 64 || d == 128 || d == 256) && bits >= 2 && bits <= 5 && m == d;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int upload(const std::vector<double>& src, float** dst) {
  *dst = nullptr;
  if (src.empty()) return TQ_OK;   // e.g. S for keys without QJL (m = 0)
  std::vector<float> f(src.size());
  for (size_t i = 0; i < src.size(); ++i) f[i] = (float)src[i];
  if (cudaMalloc(reinterpret_cast<void**>(dst), f.size() * sizeof(float)) != cudaSuccess) return TQ_ENOMEM;
  if (cudaMemcpy(*dst, f.data(), f.size() * sizeof(float), cudaMemcpyHostToDevice) != cudaSuccess) return TQ_ECUDA;
  return TQ_OK;
}

// alpha_M = (1/L) sum_idx c[idx] prod_{q in M} (2 bit_q(idx) - 1) over the odd subsets M of
// the code bits, listed by tq::mono_mask (bitplane.h).
std::vector<double> plane_alphas(const std::vector<double>& book, int bits) {
  const int L = 1 << bits, n = 1 << (bits - 1);
  std::vector<double> al(n, 0.0);
  for (int i = 0; i < n; ++i) {
    const int mask = tq::mono_mask(i);
    double acc = 0.0;
    for (int idx = 0; idx < L; ++idx) {
      double sgn = 1.0;
      for (int q = 0; q < bits; ++q)
        if ((mask >> q) & 1) sgn *= ((idx >> q) & 1) ? 1.0 : -1.0;
      acc += book[idx] * sgn;
    }
    al[i] = acc / L;
  }
  return al;
}

uint16_t f16_bits(double x) { return __half_as_ushort(__float2half_rn((float)x)); }
double f16_val(uint16_t h) { return (double)__half2float(__ushort_as_half(h)); }

// fp16 hi/lo operand blob of the tensor-core quantizer (head_dim 128): matrices M[n][k]
// (Pi, then S' = S Pi^T), scaled by 2^8 so that the lo pieces stay clear of fp16's subnormal
// range, split as hi = f16(256 M), lo = f16(256 M - hi), each stored in the no-swizzle K-major
// layout (8-row x 16-byte core matrices, 128 contiguous bytes each; core (n/8, k/8) at
// (n/8) * 2048 + (k/8) * 128).
std::vector<uint8_t> quantizer_blob(const std::vector<double>& pi, const std::vector<double>& sp) {
  const int d = 128;
  std::vector<uint8_t> blob(4 * d * d * 2);
  auto put = [&](int mat, int n, int k, uint16_t v) {
    size_t off = (size_t)mat * d * d * 2 + (size_t)(n >> 3) * 2048 + (size_t)(k >> 3) * 128 + (n & 7) * 16 + (k & 7) * 2;
    blob[off] = (uint8_t)(v & 0xFF);
    blob[off + 1] = (uint8_t)(v >> 8);
  };
  for (int n = 0; n < d; ++n)
    for (int k = 0; k < d; ++k) {
      const double p = 256.0 * pi[(size_t)n * d + k];   // rotation: y_n = sum_k Pi[n][k] x_k
      const double s = 256.0 * sp[(size_t)n * d + k];   // projection: z_n = sum_k S'[n][k] r_k
      const uint16_t ph = f16_bits(p), sh = f16_bits(s);
      put(0, n, k, ph);
      put(1, n, k, f16_bits(p - f16_val(ph)));
      put(2, n, k, sh);
      put(3, n, k, f16_bits(s - f16_val(sh)));
    }
  return blob;
}

// Host image of the exact-decision tables (layout of tq::exact::tables).
std::vector<float> exact_tables(const tq_ctx* c, const std::vector<double>& sp) {
  const int d = c->d;
  const size_t dd = (size_t)d * d;
  std::vector<float> t(tq::exact::tables_floats(d), 0.f);
  auto split = [&](const double* src, size_t n, size_t off_hi, size_t off_lo) {
    for (size_t i = 0; i < n; ++i) {
      const float hi = (float)src[i];
      t[off_hi + i] = hi;
      t[off_lo + i] = (float)(src[i] - (double)hi);
    }
  };
  split(c->pi.data(), dd, 0, dd);
  split(c->s.data(), c->s.size(), 2 * dd, 3 * dd);   // m x d (empty without QJL)
  split(sp.data(), sp.size(), 4 * dd, 5 * dd);
  const size_t b = 6 * dd;
  split(c->tk.data(), c->tk.size(), b, b + 32);
  split(c->tv.data(), c->tv.size(), b + 64, b + 96);
  split(c->ck.data(), c->ck.size(), b + 128, b + 160);
  tq::exact::near_table(c->tk.data(), c->lk, &t[b + 192]);
  tq::exact::near_table(c->tv.data(), c->lv, &t[b + 256]);
  return t;
}

void release(tq_ctx* c) {
  if (!c) return;
  int prev = -1;
  cudaGetDevice(&prev);
  cudaSetDevice(c->device);
  float* bufs[] = {c->d_pi, c->d_pit, c->d_st, c->d_spt, c->d_s, c->d_ck, c->d_tk, c->d_cv, c->d_tv,
                   c->d_alpha_k, c->d_alpha_v, c->d_exact};
  for (float* p : bufs)
    if (p) cudaFree(p);
  if (c->d_status) cudaFree(c->d_status);
  if (c->d_qblob) cudaFree(c->d_qblob);
  if (prev >= 0) cudaSetDevice(prev);
  delete c;
}

// Makes the context's device current for the duration of a call.
struct DeviceGuard {
  int prev = -1, dev;
  explicit DeviceGuard(int d) : dev(d) {
    cudaGetDevice(&prev);
    if (prev != dev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    if (prev >= 0 && prev != dev) cudaSetDevice(prev);
  }
};

}  // namespace

namespace {
// A context of format version 1 (bits > 0: kb = bits - 1 key planes, vb = bits value planes,
// m = d) or version 2 (bits = 0: any kb, vb in [1, 5], m = d or 0).
int create(int d, int bits, int kb, int vb, int m, uint64_t seed, int device, tq_ctx** out) {
  tq_ctx* c = new (std::nothrow) tq_ctx();
  if (!c) return TQ_ENOMEM;
  c->d = d;
  c->bits = bits;
  c->kb = kb;
  c->vb = vb;
  c->m = m;
  c->seed = seed;
  c->device = device;
  c->lk = 1 << kb;
  c->lv = 1 << vb;
  c->page_bytes = (size_t)TQ_PAGE_TOKENS * ((size_t)kb * d / 8 + 4 + (size_t)vb * d / 8 + 4) +
                  (m > 0 ? (size_t)TQ_PAGE_TOKENS * ((size_t)m / 8 + 4) : 0);
  c->pi.resize((size_t)d * d);
  c->s.resize((size_t)m * d);
  c->ck.resize(c->lk);
  c->tk.resize(c->lk - 1);
  c->cv.resize(c->lv);
  c->tv.resize(c->lv - 1);
  tq::haar_rotation(d, seed, c->pi.data());
  tq::gaussian_projection(m, d, seed, c->s.data());
  int rc = tq::lloyd_max(d, c->lk, c->ck.data(), c->tk.data());
  if (rc == TQ_OK) rc = tq::lloyd_max(d, c->lv, c->cv.data(), c->tv.data());
  if (rc != TQ_OK) {
    delete c;
    return rc;
  }
  // derived host matrices: Pi^T, S^T, (S Pi^T)^T
  std::vector<double> pit((size_t)d * d), st((size_t)d * m), spt((size_t)d * m);
  for (int i = 0; i < d; ++i)
    for (int j = 0; j < d; ++j) pit[(size_t)j * d + i] = c->pi[(size_t)i * d + j];
  for (int i = 0; i < m; ++i)
    for (int k = 0; k < d; ++k) st[(size_t)k * m + i] = c->s[(size_t)i * d + k];
  for (int i = 0; i < m; ++i)
    for (int j = 0; j < d; ++j) {
      double acc = 0.0;   // S'[i][j] = sum_k S[i][k] Pi[j][k]
      for (int k = 0; k < d; ++k) acc += c->s[(size_t)i * d + k] * c->pi[(size_t)j * d + k];
      spt[(size_t)j * m + i] = acc;
    }
  {
    DeviceGuard guard(device);
    rc = upload(c->pi, &c->d_pi);
    if (rc == TQ_OK) rc = upload(pit, &c->d_pit);
    if (rc == TQ_OK) rc = upload(st, &c->d_st);
    if (rc == TQ_OK) rc = upload(spt, &c->d_spt);
    if (rc == TQ_OK) rc = upload(c->s, &c->d_s);
    if (rc == TQ_OK) rc = upload(c->ck, &c->d_ck);
    if (rc == TQ_OK) rc = upload(c->tk, &c->d_tk);
    if (rc == TQ_OK) rc = upload(c->cv, &c->d_cv);
    if (rc == TQ_OK) rc = upload(c->tv, &c->d_tv);
    if (rc == TQ_OK && bits > 0) {
      std::vector<double> ak = plane_alphas(c->ck, bits - 1), av = plane_alphas(c->cv, bits);
      for (double x : ak) c->asum_k += (float)x;
      for (double x : av) c->asum_v += (float)x;
      rc = upload(ak, &c->d_alpha_k);
      if (rc == TQ_OK) rc = upload(av, &c->d_alpha_v);
    }
    if (rc == TQ_OK && cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
      rc = TQ_ECUDA;
    if (bits == 0) {
      if (rc == TQ_OK) rc = tq::prepare_kv2(c);
    } else {
      if (rc == TQ_OK) rc = prepare_quantize_simt(c);
      if (rc == TQ_OK) rc = tq::prepare_decode_mma(c);
      if (rc == TQ_OK) rc = tq::prepare_decode_tc(c);
      if (rc == TQ_OK) rc = tq::prepare_decode_f4(c);
    }
    std::vector<double> sp((size_t)m * d);   // S'[i][j] row-major
    for (int i = 0; i < m; ++i)
      for (int j = 0; j < d; ++j) sp[(size_t)i * d + j] = spt[(size_t)j * m + i];
    if (rc == TQ_OK) {
      const std::vector<float> et = exact_tables(c, sp);
      if (cudaMalloc(reinterpret_cast<void**>(&c->d_exact), et.size() * sizeof(float)) != cudaSuccess ||
          cudaMemcpy(c->d_exact, et.data(), et.size() * sizeof(float), cudaMemcpyHostToDevice) != cudaSuccess)
        rc = TQ_ENOMEM;
    }
    if (rc == TQ_OK && d == 128 && bits > 0) {
      std::vector<uint8_t> blob = quantizer_blob(c->pi, sp);
      if (cudaMalloc(reinterpret_cast<void**>(&c->d_qblob), blob.size()) != cudaSuccess ||
          cudaMemcpy(c->d_qblob, blob.data(), blob.size(), cudaMemcpyHostToDevice) != cudaSuccess)
        rc = TQ_ENOMEM;
      if (rc == TQ_OK) rc = tq::prepare_quantize_tc(c);
    }
    if (rc == TQ_OK) {
      if (cudaMalloc(&c->d_status, sizeof(int)) != cudaSuccess ||
          cudaMemset(c->d_status, 0, sizeof(int)) != cudaSuccess)
        rc = TQ_ECUDA;
    }
  }
  if (rc != TQ_OK) {
    release(c);
    return rc;
  }
  // a new context may follow a device reset, which invalidates the no-alloc scratch address
  tq::noalloc_forget_device(device);
  *out = c;
  return TQ_OK;
}
}  // namespace

extern "C" int tq_ctx_create(int d, int bits, int m, uint64_t seed, int device, tq_ctx** out) {
  if (!out) return TQ_EINVAL;
  *out = nullptr;
  if (!supported(d, bits, m)) return TQ_EUNSUPPORTED;
  return create(d, bits, bits - 1, bits, m, seed, device, out);
}

extern "C" int tq_ctx_create_kv(int d, int key_bits, int value_bits, int qjl, uint64_t seed, int device,
                                tq_ctx** out) {
  if (!out) return TQ_EINVAL;
  *out = nullptr;
  if (d != 64 && d != 128 && d != 256) return TQ_EUNSUPPORTED;
  const int kb = qjl ? key_bits - 1 : key_bits;
  if (kb < 1 || kb > 5 || value_bits < 1 || value_bits > 5) return TQ_EUNSUPPORTED;
  if (qjl && key_bits == value_bits)   // the version-1 format, with its tensor-core kernels
    return create(d, key_bits, kb, value_bits, d, seed, device, out);
  return create(d, 0, kb, value_bits, qjl ? d : 0, seed, device, out);
}

extern "C" void tq_ctx_destroy(tq_ctx* ctx) { release(ctx); }

extern "C" size_t tq_page_bytes(const tq_ctx* ctx) { return ctx ? ctx->page_bytes : 0; }

extern "C" size_t tq_cache_bytes(const tq_ctx* ctx, int batch, int kv_heads, int max_tokens) {
  if (!ctx || batch < 1 || kv_heads < 1 || max_tokens < 1) return 0;
  size_t pages = (size_t)(max_tokens + TQ_PAGE_TOKENS - 1) / TQ_PAGE_TOKENS;
  return (size_t)batch * kv_heads * pages * ctx->page_bytes;
}

extern "C" int tq_ctx_get_constants(const tq_ctx* ctx, double* pi, double* s, double* ck, double* tk,
                                    double* cv, double* tv) {
  if (!ctx) return TQ_EINVAL;
  auto cp = [](const std::vector<double>& v, double* dst) {
    if (dst) std::memcpy(dst, v.data(), v.size() * sizeof(double));
  };
  cp(ctx->pi, pi);
  cp(ctx->s, s);
  cp(ctx->ck, ck);
  cp(ctx->tk, tk);
  cp(ctx->cv, cv);
  cp(ctx->tv, tv);
  return TQ_OK;
}

namespace {

int quantize_impl(const tq_ctx* ctx, const void* k, const void* v, int batch, int kv_heads, int n_tokens,
                  const int32_t* start_pos, void* cache, int max_tokens, const tq::PageMap& pm,
                  const int64_t* strides, void* stream) {
  if (!ctx) return TQ_EINVAL;
  if (batch < 1 || kv_heads < 1 || n_tokens < 0 || max_tokens < 1) return TQ_EINVAL;
  if (batch > 65535 || kv_heads > 65535) return TQ_EINVAL;
  if (n_tokens > max_tokens) return TQ_EINVAL;
  if (n_tokens == 0) return TQ_OK;   // nothing to read or write; k and v may be NULL
  if (!k || !v || !start_pos || !cache) return TQ_EINVAL;
  if (!aligned(k, 16) || !aligned(v, 16) || !aligned(cache, 256) || !aligned(start_pos, 4)) return TQ_EINVAL;
  tq::KVLayout lay = tq::contiguous_layout(kv_heads, n_tokens, ctx->d);
  if (strides) {   // multiples of 8 elements keep every token's row on a 16-byte boundary
    for (int i = 0; i < 6; ++i)
      if (strides[i] < 0 || strides[i] % 8 != 0) return TQ_EINVAL;
    lay = tq::KVLayout{strides[0], strides[1], strides[2], strides[3], strides[4], strides[5]};
  }
  DeviceGuard guard(ctx->device);
  if (ctx->bits == 0)
    return tq::launch_quantize_kv2(ctx, k, v, batch, kv_heads, n_tokens, start_pos, cache, max_tokens, lay, stream,
                                   pm);
  if (n_tokens <= tq::kFewTokens)
    return tq::launch_quantize_few(ctx, k, v, batch, kv_heads, n_tokens, start_pos, cache, max_tokens, lay, stream,
                                   pm);
  if (ctx->d == 128)
    return tq::launch_quantize_tc(ctx, k, v, batch, kv_heads, n_tokens, start_pos, cache, max_tokens, lay, stream,
                                  pm);
  return launch_quantize_simt(ctx, k, v, batch, kv_heads, n_tokens, start_pos, cache, max_tokens, lay, stream, pm);
}

// The block-table arguments of the paged entry points: TQ_OK and the page map, or TQ_EINVAL.
int paged_map(const void* pool, int n_blocks, const int32_t* block_table, int max_blocks, tq::PageMap* pm,
              int* max_tokens) {
  if (!pool || !block_table || n_blocks < 1 || max_blocks < 1) return TQ_EINVAL;
  if (max_blocks > INT32_MAX / TQ_PAGE_TOKENS || !aligned(block_table, 4)) return TQ_EINVAL;
  pm->table = block_table;
  pm->stride = max_blocks;
  pm->n_blocks = n_blocks;
  *max_tokens = max_blocks * TQ_PAGE_TOKENS;
  return TQ_OK;
}

}  // namespace

extern "C" int tq_quantize_kv(const tq_ctx* ctx, const void* k, const void* v, int batch, int kv_heads,
                              int n_tokens, const int32_t* start_pos, void* cache, int max_tokens,
                              void* stream) {
  return quantize_impl(ctx, k, v, batch, kv_heads, n_tokens, start_pos, cache, max_tokens, tq::PageMap(), nullptr,
                       stream);
}

extern "C" int tq_quantize_kv_strided(const tq_ctx* ctx, const void* k, const void* v, const int64_t* strides,
                                      int batch, int kv_heads, int n_tokens, const int32_t* start_pos, void* cache,
                                      int max_tokens, void* stream) {
  if (!strides) return TQ_EINVAL;
  return quantize_impl(ctx, k, v, batch, kv_heads, n_tokens, start_pos, cache, max_tokens, tq::PageMap(), strides,
                       stream);
}

extern "C" size_t tq_paged_pool_bytes(const tq_ctx* ctx, int kv_heads, int n_blocks) {
  if (!ctx || kv_heads < 1 || n_blocks < 1) return 0;
  return (size_t)n_blocks * kv_heads * ctx->page_bytes;
}

extern "C" int tq_quantize_kv_paged(const tq_ctx* ctx, const void* k, const void* v, int batch, int kv_heads,
                                    int n_tokens, const int32_t* start_pos, void* pool, int n_blocks,
                                    const int32_t* block_table, int max_blocks, void* stream) {
  tq::PageMap pm;
  int max_tokens = 0;
  const int rc = paged_map(pool, n_blocks, block_table, max_blocks, &pm, &max_tokens);
  if (rc != TQ_OK) return rc;
  return quantize_impl(ctx, k, v, batch, kv_heads, n_tokens, start_pos, pool, max_tokens, pm, nullptr, stream);
}

extern "C" int tq_quantize_kv_paged_strided(const tq_ctx* ctx, const void* k, const void* v, const int64_t* strides,
                                            int batch, int kv_heads, int n_tokens, const int32_t* start_pos,
                                            void* pool, int n_blocks, const int32_t* block_table, int max_blocks,
                                            void* stream) {
  if (!strides) return TQ_EINVAL;
  tq::PageMap pm;
  int max_tokens = 0;
  const int rc = paged_map(pool, n_blocks, block_table, max_blocks, &pm, &max_tokens);
  if (rc != TQ_OK) return rc;
  return quantize_impl(ctx, k, v, batch, kv_heads, n_tokens, start_pos, pool, max_tokens, pm, strides, stream);
}

extern "C" int tq_ctx_set_decode_path(tq_ctx* ctx, int path) {
  if (!ctx) return TQ_EINVAL;
  switch (path) {
    case TQ_DECODE_AUTO:
    case TQ_DECODE_SIMT:
      break;
    case TQ_DECODE_MMA:
      if (ctx->bits == 0 || (ctx->d != 64 && ctx->d != 128 && ctx->d != 256)) return TQ_EUNSUPPORTED;
      break;
    case TQ_DECODE_TC:
      if (ctx->d != 128 || (ctx->bits != 2 && ctx->bits != 3)) return TQ_EUNSUPPORTED;
      break;
    case TQ_DECODE_TC4:
      if (ctx->d != 128 || ctx->bits < 2 || ctx->bits > 4) return TQ_EUNSUPPORTED;
      break;
    default:
      return TQ_EINVAL;
  }
  ctx->decode_path = path;
  return TQ_OK;
}

extern "C" int tq_ctx_set_sparse_v(tq_ctx* ctx, float threshold) {
  if (!ctx || !(threshold >= 0.f && threshold <= 1.f)) return TQ_EINVAL;   // NaN fails too
  ctx->sparse_v = threshold;
  return TQ_OK;
}

namespace {

// Kernel a decode call takes: TQ_DECODE_SIMT / _MMA / _TC, or TQ_EUNSUPPORTED.  The bit-plane
// kernels share one launch plan (mp).
int decode_kernel_for(const tq_ctx* ctx, int batch, int q_heads, int kv_heads, int max_tokens, tq::MmaPlan* mp) {
  tq::MmaPlan pm, pt, pf;
  const bool mma_ok = tq::plan_decode_mma(ctx, batch, q_heads, kv_heads, max_tokens, &pm);
  const bool tc_ok = tq::plan_decode_tc(ctx, batch, q_heads, kv_heads, max_tokens, &pt);
  const bool f4_ok = tq::plan_decode_f4(ctx, batch, q_heads, kv_heads, max_tokens, &pf);
  int kern = TQ_EUNSUPPORTED;
  switch (ctx->decode_path) {
    case TQ_DECODE_SIMT:
      kern = TQ_DECODE_SIMT;
      break;
    case TQ_DECODE_MMA:
      if (mma_ok) kern = TQ_DECODE_MMA;
      break;
    case TQ_DECODE_TC:
      if (tc_ok) kern = TQ_DECODE_TC;
      break;
    case TQ_DECODE_TC4:
      if (f4_ok) kern = TQ_DECODE_TC4;
      break;
    default:
      if (f4_ok) kern = TQ_DECODE_TC4;
      else if (tc_ok && (!mma_ok || tq::decode_tc_preferred(ctx, q_heads, kv_heads))) kern = TQ_DECODE_TC;
      else kern = mma_ok ? TQ_DECODE_MMA : TQ_DECODE_SIMT;
  }
  if (kern == TQ_DECODE_MMA) *mp = pm;
  if (kern == TQ_DECODE_TC) *mp = pt;
  if (kern == TQ_DECODE_TC4) *mp = pf;
  return kern;
}

}  // namespace

extern "C" size_t tq_decode_workspace_bytes(const tq_ctx* ctx, int batch, int q_heads, int kv_heads,
                                            int max_tokens) {
  if (!ctx || batch < 1 || q_heads < 1 || kv_heads < 1 || max_tokens < 1) return 0;
  if (q_heads % kv_heads != 0) return 0;
  tq::MmaPlan mp;
  const int kern = decode_kernel_for(ctx, batch, q_heads, kv_heads, max_tokens, &mp);
  if (kern == TQ_DECODE_MMA || kern == TQ_DECODE_TC || kern == TQ_DECODE_TC4)
    return tq::decode_mma_workspace(ctx, mp, batch, q_heads, kv_heads);
  if (kern != TQ_DECODE_SIMT) return 0;
  tq::SplitPlan sp = tq::plan_splits(batch, kv_heads, max_tokens);
  size_t rows = (size_t)batch * q_heads;
  size_t floats = rows * ctx->d * 2 + rows * sp.splits * (2 + ctx->d);
  return floats * sizeof(float);
}

namespace tq {
// tq_attn_decode's checks of everything but the workspace: TQ_OK or the code it returns.
int check_decode_args(const tq_ctx* ctx, const float* q, int batch, int q_heads, int kv_heads, const void* cache,
                      const int32_t* seq_lens, int max_tokens, const float* out, const float* logits_out) {
  if (!ctx || !q || !cache || !seq_lens || !out) return TQ_EINVAL;
  if (batch < 1 || q_heads < 1 || kv_heads < 1 || max_tokens < 1) return TQ_EINVAL;
  if (batch > 65535 || kv_heads > 65535 || q_heads > 65535) return TQ_EINVAL;
  if (q_heads % kv_heads != 0) return TQ_EINVAL;
  if (q_heads / kv_heads > 16) return TQ_EUNSUPPORTED;
  if (!aligned(q, 16) || !aligned(cache, 256) || !aligned(out, 16) || !aligned(seq_lens, 4) ||
      (logits_out && !aligned(logits_out, 4)))
    return TQ_EINVAL;
  tq::MmaPlan mp;
  const int kern = decode_kernel_for(ctx, batch, q_heads, kv_heads, max_tokens, &mp);
  return kern < 0 ? kern : TQ_OK;
}
}  // namespace tq

namespace {

int decode_impl(const tq_ctx* ctx, const float* q, int batch, int q_heads, int kv_heads, const void* cache,
                const int32_t* seq_lens, int max_tokens, float* out, float* logits_out, void* workspace,
                size_t workspace_bytes, const tq::PageMap& pm, void* stream) {
  const int rc = tq::check_decode_args(ctx, q, batch, q_heads, kv_heads, cache, seq_lens, max_tokens, out, logits_out);
  if (rc != TQ_OK) return rc;
  if (!workspace || !aligned(workspace, 256)) return TQ_EINVAL;
  tq::MmaPlan mp;
  const int kern = decode_kernel_for(ctx, batch, q_heads, kv_heads, max_tokens, &mp);
  if (workspace_bytes < tq_decode_workspace_bytes(ctx, batch, q_heads, kv_heads, max_tokens)) return TQ_ENOMEM;
  DeviceGuard guard(ctx->device);
  if (kern == TQ_DECODE_TC4)
    return tq::launch_decode_f4(ctx, mp, q, batch, q_heads, kv_heads, cache, seq_lens, max_tokens, out, logits_out,
                                workspace, stream, pm);
  if (kern == TQ_DECODE_TC)
    return tq::launch_decode_tc(ctx, mp, q, batch, q_heads, kv_heads, cache, seq_lens, max_tokens, out, logits_out,
                                workspace, stream, pm);
  if (kern == TQ_DECODE_MMA)
    return tq::launch_decode_mma(ctx, mp, q, batch, q_heads, kv_heads, cache, seq_lens, max_tokens, out, logits_out,
                                 workspace, stream, pm);
  if (ctx->bits == 0)
    return tq::launch_decode_kv2(ctx, q, batch, q_heads, kv_heads, cache, seq_lens, max_tokens, out, logits_out,
                                 workspace, stream, pm);
  return launch_decode_simt(ctx, q, batch, q_heads, kv_heads, cache, seq_lens, max_tokens, out, logits_out,
                            workspace, stream, pm);
}

}  // namespace

extern "C" int tq_attn_decode(const tq_ctx* ctx, const float* q, int batch, int q_heads, int kv_heads,
                              const void* cache, const int32_t* seq_lens, int max_tokens, float* out,
                              float* logits_out, void* workspace, size_t workspace_bytes, void* stream) {
  return decode_impl(ctx, q, batch, q_heads, kv_heads, cache, seq_lens, max_tokens, out, logits_out, workspace,
                     workspace_bytes, tq::PageMap(), stream);
}

extern "C" int tq_attn_decode_paged(const tq_ctx* ctx, const float* q, int batch, int q_heads, int kv_heads,
                                    const void* pool, int n_blocks, const int32_t* block_table, int max_blocks,
                                    const int32_t* seq_lens, float* out, float* logits_out, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  tq::PageMap pm;
  int max_tokens = 0;
  const int rc = paged_map(pool, n_blocks, block_table, max_blocks, &pm, &max_tokens);
  if (rc != TQ_OK) return rc;
  return decode_impl(ctx, q, batch, q_heads, kv_heads, pool, seq_lens, max_tokens, out, logits_out, workspace,
                     workspace_bytes, pm, stream);
}

namespace {
size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }
}  // namespace

extern "C" size_t tq_ip_topk_workspace_bytes(const tq_ctx* ctx, int batch, int q_heads, int kv_heads,
                                             int max_tokens) {
  const size_t dw = tq_decode_workspace_bytes(ctx, batch, q_heads, kv_heads, max_tokens);
  if (dw == 0) return 0;
  const size_t rows = (size_t)batch * q_heads;
  return align256(dw) + align256(rows * (size_t)max_tokens * 4) + align256(rows * (size_t)ctx->d * 4);
}

namespace {

int topk_impl(const tq_ctx* ctx, const float* q, int batch, int q_heads, int kv_heads, const void* cache,
              const int32_t* seq_lens, int max_tokens, int k, int32_t* out_idx, float* out_score, void* workspace,
              size_t workspace_bytes, const tq::PageMap& pm, void* stream) {
  if (!ctx || k < 1 || k > TQ_TOPK_MAX || !out_idx || !out_score || !aligned(out_idx, 4) || !aligned(out_score, 4))
    return TQ_EINVAL;
  // the decode's own checks (out stands in for the decode output, which lives in the workspace)
  const int rc0 = tq::check_decode_args(ctx, q, batch, q_heads, kv_heads, cache, seq_lens, max_tokens, out_score,
                                        nullptr);
  if (rc0 != TQ_OK) return rc0;
  if (!workspace || !aligned(workspace, 256)) return TQ_EINVAL;
  const size_t need = tq_ip_topk_workspace_bytes(ctx, batch, q_heads, kv_heads, max_tokens);
  if (need == 0) return TQ_EINVAL;
  if (workspace_bytes < need) return TQ_ENOMEM;
  const size_t dw = tq_decode_workspace_bytes(ctx, batch, q_heads, kv_heads, max_tokens);
  const size_t rows = (size_t)batch * q_heads;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  float* lg = reinterpret_cast<float*>(w + align256(dw));
  float* o = reinterpret_cast<float*>(w + align256(dw) + align256(rows * (size_t)max_tokens * 4));
  const int rc = decode_impl(ctx, q, batch, q_heads, kv_heads, cache, seq_lens, max_tokens, o, lg, w, dw, pm, stream);
  if (rc != TQ_OK) return rc;
  DeviceGuard guard(ctx->device);
  return tq::launch_topk(ctx, lg, seq_lens, batch, q_heads, max_tokens, k, out_idx, out_score, stream);
}

}  // namespace

extern "C" int tq_ip_topk(const tq_ctx* ctx, const float* q, int batch, int q_heads, int kv_heads,
                          const void* cache, const int32_t* seq_lens, int max_tokens, int k, int32_t* out_idx,
                          float* out_score, void* workspace, size_t workspace_bytes, void* stream) {
  return topk_impl(ctx, q, batch, q_heads, kv_heads, cache, seq_lens, max_tokens, k, out_idx, out_score, workspace,
                   workspace_bytes, tq::PageMap(), stream);
}

extern "C" int tq_ip_topk_paged(const tq_ctx* ctx, const float* q, int batch, int q_heads, int kv_heads,
                                const void* pool, int n_blocks, const int32_t* block_table, int max_blocks,
                                const int32_t* seq_lens, int k, int32_t* out_idx, float* out_score, void* workspace,
                                size_t workspace_bytes, void* stream) {
  tq::PageMap pm;
  int max_tokens = 0;
  const int rc = paged_map(pool, n_blocks, block_table, max_blocks, &pm, &max_tokens);
  if (rc != TQ_OK) return rc;
  return topk_impl(ctx, q, batch, q_heads, kv_heads, pool, seq_lens, max_tokens, k, out_idx, out_score, workspace,
                   workspace_bytes, pm, stream);
}

namespace {

int dequantize_impl(const tq_ctx* ctx, const void* cache, int batch, int kv_heads, int max_tokens,
                    const int32_t* start_pos, int n_tokens, float* k_out, float* v_out, const tq::PageMap& pm,
                    void* stream) {
  if (!ctx) return TQ_EINVAL;
  if (batch < 1 || kv_heads < 1 || n_tokens < 0 || max_tokens < 1) return TQ_EINVAL;
  if (batch > 65535 || kv_heads > 65535 || n_tokens > max_tokens) return TQ_EINVAL;
  if (n_tokens == 0 || (!k_out && !v_out)) return TQ_OK;
  if (!cache || !start_pos || !aligned(cache, 256) || !aligned(start_pos, 4)) return TQ_EINVAL;
  if ((k_out && !aligned(k_out, 4)) || (v_out && !aligned(v_out, 4))) return TQ_EINVAL;
  DeviceGuard guard(ctx->device);
  if (ctx->bits == 0)
    return tq::launch_dequantize_kv2(ctx, cache, batch, kv_heads, max_tokens, start_pos, n_tokens, k_out, v_out,
                                     stream, pm);
  return tq::launch_dequantize(ctx, cache, batch, kv_heads, max_tokens, start_pos, n_tokens, k_out, v_out, stream,
                               pm);
}

}  // namespace

extern "C" int tq_dequantize_kv(const tq_ctx* ctx, const void* cache, int batch, int kv_heads, int max_tokens,
                                const int32_t* start_pos, int n_tokens, float* k_out, float* v_out, void* stream) {
  return dequantize_impl(ctx, cache, batch, kv_heads, max_tokens, start_pos, n_tokens, k_out, v_out, tq::PageMap(),
                         stream);
}

extern "C" int tq_dequantize_kv_paged(const tq_ctx* ctx, const void* pool, int n_blocks, const int32_t* block_table,
                                      int max_blocks, int batch, int kv_heads, const int32_t* start_pos,
                                      int n_tokens, float* k_out, float* v_out, void* stream) {
  tq::PageMap pm;
  int max_tokens = 0;
  const int rc = paged_map(pool, n_blocks, block_table, max_blocks, &pm, &max_tokens);
  if (rc != TQ_OK) return rc;
  return dequantize_impl(ctx, pool, batch, kv_heads, max_tokens, start_pos, n_tokens, k_out, v_out, pm, stream);
}

extern "C" int tq_selftest_bounded_wait(const tq_ctx* ctx, void* stream) {
  if (!ctx) return TQ_EINVAL;
  DeviceGuard guard(ctx->device);
  return tq::launch_selftest_wait(ctx, stream);
}

extern "C" int tq_get_device_status(const tq_ctx* ctx, void* stream) {
  if (!ctx) return TQ_EINVAL;
  DeviceGuard guard(ctx->device);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int flags = 0;
  if (cudaStreamSynchronize(st) != cudaSuccess) return TQ_ECUDA;
  if (cudaMemcpy(&flags, ctx->d_status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return TQ_ECUDA;
  if (cudaMemset(ctx->d_status, 0, sizeof(int)) != cudaSuccess) return TQ_ECUDA;
  if (flags & tq::kFlagTimeout) return TQ_ETIMEOUT;
  if (flags & tq::kFlagBounds) return TQ_EBOUNDS;
  return TQ_OK;
}

extern "C" const char* tq_status_string(int status) {
  switch (status) {
    case TQ_OK: return "ok";
    case TQ_EINVAL: return "invalid argument";
    case TQ_EUNSUPPORTED: return "unsupported head dim, bit width, projection size or group size";
    case TQ_ECUDA: return "CUDA runtime error";
    case TQ_ETIMEOUT: return "device-side wait timed out";
    case TQ_EBOUNDS: return "device-side position or length beyond max_tokens";
    case TQ_ENOMEM: return "allocation failed or workspace too small";
    case TQ_ENOTCONV: return "codebook solver did not converge";
    case TQ_ESCRATCH: return "request exceeds the 4 MiB static scratch of tq_attn_decode_noalloc";
    default: return "unknown status";
  }
}
