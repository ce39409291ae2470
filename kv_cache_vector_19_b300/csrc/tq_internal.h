// Internal declarations shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>

#include <cuda_runtime.h>

#include "tq.h"

namespace tq {

void gaussian_stream(uint64_t stream_seed, size_t count, double* out);
void haar_rotation(int d, uint64_t seed, double* pi);
void gaussian_projection(int m, int d, uint64_t seed, double* s);
int lloyd_max(int d, int levels, double* centroids, double* boundaries);

// Sticky device status bits (ORed by kernels into ctx->d_status).
enum : int { kFlagBounds = 1, kFlagTimeout = 2 };

constexpr int kPage = TQ_PAGE_TOKENS;

inline size_t page_bytes(int d, int bits, int m) {
  return (size_t)kPage * ((size_t)(bits - 1) * d / 8 + m / 8 + 8 + (size_t)bits * d / 8 + 4);
}

// Where the pages of a call live.  table == nullptr: the contiguous cache
// [batch][kv_heads][pages_per_seq][page].  Otherwise a pool of blocks, each the kv_heads pages of
// 128 consecutive token slots (page (blk, h) at page index blk * kv_heads + h), and
// table[b * stride + p] the block that holds logical page p of batch row b; a block id outside
// [0, n_blocks) is clamped into it and sets kFlagBounds, so no access leaves the pool.
struct PageMap {
  const int32_t* table = nullptr;
  int stride = 0;
  int n_blocks = 0;
#ifdef __CUDACC__
  // Page index of logical page p of sequence seq = b * kv_heads + h.
  __device__ __forceinline__ size_t index(int seq, int kv_heads, int pages_per_seq, int p, int* status) const {
    if (table == nullptr) return (size_t)seq * pages_per_seq + p;
    const int b = seq / kv_heads, h = seq - b * kv_heads;
    int blk = __ldg(table + (size_t)b * stride + p);
    if ((unsigned)blk >= (unsigned)n_blocks) {
      atomicOr(status, kFlagBounds);
      blk = blk < 0 ? 0 : n_blocks - 1;
    }
    return (size_t)blk * kv_heads + h;
  }
#endif
};

#ifdef __CUDACC__
// Programmatic dependent launch.  pdl_trigger: the next grid of the stream, when launched with
// programmatic stream serialization, may start now (it still waits at its own pdl_wait).
// pdl_wait: blocks until the preceding grid has completed and its memory operations are
// visible; returns at once in a grid launched without the attribute.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
#endif

// Element strides of the bf16 K and V inputs of a quantize call over (batch, KV head, token);
// the d values of one token are contiguous.  The contiguous [batch][kv_heads][n_tokens][d]
// layout is (H T d, T d, d); a prefill projection's [batch][n_tokens][kv_heads][d] is
// (T H d, d, H d).
struct KVLayout {
  int64_t kb, kh, kt, vb, vh, vt;
};
inline KVLayout contiguous_layout(int kv_heads, int n_tokens, int d) {
  const int64_t t = d, h = (int64_t)n_tokens * d, b = (int64_t)kv_heads * n_tokens * d;
  return KVLayout{b, h, t, b, h, t};
}

// Decode split plan shared by the workspace query and the launch.
struct SplitPlan {
  int pages, splits, pages_per_split;
};
SplitPlan plan_splits(int batch, int kv_heads, int max_tokens);

// Tensor-core decode plan: the call's (sequence, page) list cut into `grid` ranges of
// `chunk` pages; every sequence has `slots` partial-record slots.
struct MmaPlan {
  int grid, chunk, slots, pages_per_seq, total_pages;
};

}  // namespace tq

struct tq_ctx {
  int d, bits, m, device;   // bits = 0: format version 2 (kb, vb and m free; m = 0 without QJL)
  int kb = 0, vb = 0;       // key and value code planes
  uint64_t seed;
  int lk, lv;
  size_t page_bytes;
  std::vector<double> pi, s, ck, tk, cv, tv;   // fp64 host copies
  // device constants, fp32
  float* d_pi = nullptr;    // [d][d]  Pi, row-major
  float* d_pit = nullptr;   // [d][d]  Pi^T
  float* d_st = nullptr;    // [d][m]  S^T
  float* d_spt = nullptr;   // [d][m]  (S Pi^T)^T
  float* d_s = nullptr;     // [m][d]  S, row-major
  float* d_ck = nullptr;    // [lk]
  float* d_tk = nullptr;    // [lk-1]
  float* d_cv = nullptr;    // [lv]
  float* d_tv = nullptr;    // [lv-1]
  int* d_status = nullptr;  // sticky flags
  // double-float tables of the exact boundary decisions (exact.cuh: Pi, S, S' as hi + lo,
  // boundaries and key centroids as hi + lo, near tables)
  float* d_exact = nullptr;
  // bit-plane expansion of the books: c[idx] = 2 sum_M alpha_M x_M(idx) - sum_M alpha_M
  float* d_alpha_k = nullptr;   // [2^(bits-2)]
  float* d_alpha_v = nullptr;   // [2^(bits-1)]
  float asum_k = 0.f, asum_v = 0.f;
  int num_sms = 148;
  int decode_path = 0;   // TQ_DECODE_*
  float sparse_v = 0.f;  // Sparse V threshold on p_t = exp(l_t - running max); 0: dense
  // head_dim 128: fp16 B operands of the tensor-core quantizer, no-swizzle K-major layout:
  // 256 Pi as hi, lo and 256 S' as hi, lo (each 128 x 128, 32 KB)
  uint8_t* d_qblob = nullptr;
};

// One-time per-context kernel attributes (dynamic shared memory limits), so that the
// launchers themselves make no configuration calls and can be captured in CUDA graphs.
int prepare_quantize_simt(const tq_ctx* ctx);
namespace tq {
int prepare_quantize_tc(const tq_ctx* c);
int launch_selftest_wait(const tq_ctx* c, void* stream);
int launch_dequantize(const tq_ctx* c, const void* cache, int batch, int kv_heads, int max_tokens,
                      const int32_t* start_pos, int n_tokens, float* k_out, float* v_out, void* stream,
    const PageMap& pm = PageMap());
// Few tokens per sequence (appends): one CTA per new vector pair.
constexpr int kFewTokens = 8;
int launch_quantize_few(const tq_ctx* c, const void* k, const void* v, int batch, int kv_heads, int n_tokens,
                        const int32_t* start_pos, void* cache, int max_tokens, const KVLayout& lay, void* stream,
    const PageMap& pm = PageMap());
int launch_quantize_tc(const tq_ctx* c, const void* k, const void* v, int batch, int kv_heads, int n_tokens,
                       const int32_t* start_pos, void* cache, int max_tokens, const KVLayout& lay, void* stream,
    const PageMap& pm = PageMap());
}  // namespace tq

// Kernel launchers (return TQ_OK or TQ_ECUDA).
int launch_quantize_simt(const tq_ctx* ctx, const void* k, const void* v, int batch, int kv_heads,
                         int n_tokens, const int32_t* start_pos, void* cache, int max_tokens,
                         const tq::KVLayout& lay, void* stream,
    const tq::PageMap& pm = tq::PageMap());
namespace tq {
int prepare_decode_mma(const tq_ctx* c);
bool plan_pages(long ctas, int batch, int kv_heads, int max_tokens, MmaPlan* p);
bool plan_decode_mma(const tq_ctx* c, int batch, int q_heads, int kv_heads, int max_tokens, MmaPlan* p);
bool plan_decode_tc(const tq_ctx* c, int batch, int q_heads, int kv_heads, int max_tokens, MmaPlan* p);
int launch_decode_mma(const tq_ctx* c, const MmaPlan& pl, const float* q, int batch, int q_heads, int kv_heads,
                      const void* cache, const int32_t* seq_lens, int max_tokens, float* out, float* logits_out,
                      void* workspace, void* stream,
    const PageMap& pm = PageMap());
size_t decode_mma_workspace(const tq_ctx* c, const MmaPlan& pl, int batch, int q_heads, int kv_heads);
// tcgen05 decode (head_dim 128, b in {2, 3}, up to 16 query heads per KV head); same plan,
// workspace and partial records as the mma.sync kernel.
bool decode_tc_supported(const tq_ctx* c, int q_heads, int kv_heads);
// whether TQ_DECODE_AUTO takes the tcgen05 kernel over the mma.sync one (by measurement)
bool decode_tc_preferred(const tq_ctx* c, int q_heads, int kv_heads);
int prepare_decode_tc(const tq_ctx* c);
int launch_decode_tc(const tq_ctx* c, const MmaPlan& pl, const float* q, int batch, int q_heads, int kv_heads,
                     const void* cache, const int32_t* seq_lens, int max_tokens, float* out, float* logits_out,
                     void* workspace, void* stream,
    const PageMap& pm = PageMap());
// tcgen05 decode with 4-bit (e2m1) operands: head_dim 128, b in {2, 3}, up to 8 query heads
// per KV head; same plan, workspace and partial records as the mma.sync kernel.
bool decode_f4_supported(const tq_ctx* c, int q_heads, int kv_heads);
bool plan_decode_f4(const tq_ctx* c, int batch, int q_heads, int kv_heads, int max_tokens, MmaPlan* p);
int prepare_decode_f4(const tq_ctx* c);
int launch_decode_f4(const tq_ctx* c, const MmaPlan& pl, const float* q, int batch, int q_heads, int kv_heads,
                     const void* cache, const int32_t* seq_lens, int max_tokens, float* out, float* logits_out,
                     void* workspace, void* stream,
    const PageMap& pm = PageMap());
// tq_attn_decode's argument checks except the workspace (TQ_OK or its error code).
int check_decode_args(const tq_ctx* ctx, const float* q, int batch, int q_heads, int kv_heads, const void* cache,
                      const int32_t* seq_lens, int max_tokens, const float* out, const float* logits_out);
// Drops the no-alloc entry point's cached scratch address of a device (looked up again on the
// next call there).
void noalloc_forget_device(int device);
// q~ = Pi q and q_s = S q for every (batch, query head), fp32.
void launch_prologue(const tq_ctx* c, const float* q, int batch, int q_heads, float* qr, float* qs,
                     cudaStream_t st);
// Split merge and Pi^T of the CUDA-core decode: out = Pi^T o~ / l per (query head, batch).
void launch_combine(const tq_ctx* c, const float* part, float* out, int batch, int q_heads, int splits,
                    cudaStream_t st);
// Top k of each (batch, query head) row of decode logits (scan.cu), scaled back by sqrt(d).
int launch_topk(const tq_ctx* c, const float* logits, const int32_t* seq_lens, int batch, int q_heads,
                int max_tokens, int k, int32_t* out_idx, float* out_score, void* stream);
// Format version 2 (kv2.cu): CUDA-core quantizer, split decode and dequantizer with the plane
// counts and m read from the context.
int prepare_kv2(const tq_ctx* c);
int launch_quantize_kv2(const tq_ctx* c, const void* k, const void* v, int batch, int kv_heads, int n_tokens,
                        const int32_t* start_pos, void* cache, int max_tokens, const KVLayout& lay, void* stream,
    const PageMap& pm = PageMap());
int launch_decode_kv2(const tq_ctx* c, const float* q, int batch, int q_heads, int kv_heads, const void* cache,
                      const int32_t* seq_lens, int max_tokens, float* out, float* logits_out, void* workspace,
                      void* stream,
    const PageMap& pm = PageMap());
int launch_dequantize_kv2(const tq_ctx* c, const void* cache, int batch, int kv_heads, int max_tokens,
                          const int32_t* start_pos, int n_tokens, float* k_out, float* v_out, void* stream,
    const PageMap& pm = PageMap());
}  // namespace tq

int launch_decode_simt(const tq_ctx* ctx, const float* q, int batch, int q_heads, int kv_heads,
                       const void* cache, const int32_t* seq_lens, int max_tokens, float* out,
                       float* logits_out, void* workspace, void* stream,
    const tq::PageMap& pm = tq::PageMap());
