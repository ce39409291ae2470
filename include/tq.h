/*
 * tq.h - C ABI of the TurboQuant compressed KV-cache library for NVIDIA B300 (sm_103a).
 *
 * What the library computes
 * -------------------------
 * Online KV-cache compression as described in
 *   [BLOG]  "Технология TurboQuant и её применение с локальными LLM" (ast-softpro.ru),
 *           section 1.2 "Как работает TurboQuant";
 *   [3BITS] "3 бита вместо 16: разбираем TurboQuant и когда его реально стоит включать"
 *           (kiosknews.app), section "Как работает TurboQuant" and section
 *           "Python + HuggingFace" (quantize returns indices and norms per vector).
 *
 *   key x (d coordinates, bf16):   n = ||x||,  y = Pi x,  idx_j = #{k : y_j / n >= t_k}
 *                                  (Lloyd-Max codebook with 2^(b-1) levels),
 *                                  r = x - n Pi^T c[idx],  gamma = ||r||,
 *                                  sigma_i = [ (S r)_i >= 0 ]  (QJL sign sketch, m = d)
 *   value v (bf16):                n_v = ||v||, idx over a 2^b-level codebook, no QJL.
 *   decode, query q, kv head g = floor(h / G):
 *       logit_t = ( n_t <Pi q, c_K[idx_t]> + gamma_t sqrt(pi/2)/m <S q, 2 sigma_t - 1> ) / sqrt(d)
 *       out     = Pi^T sum_t softmax(logit)_t n_v,t c_V[idx_v,t]
 *
 * Pi is a Haar-random orthogonal d x d matrix (QR of a seeded Gaussian matrix with the
 * signs of R's diagonal moved into Q), S an m x d matrix of i.i.d. N(0,1) entries, both
 * drawn from SplitMix64 + Box-Muller streams seeded with 2*seed and 2*seed+1.  The
 * codebooks are the Lloyd-Max quantizers of the exact density of one coordinate of a
 * uniform unit vector in R^d, (1 - t^2)^((d-3)/2) on [-1, 1]: data-oblivious, computed
 * once per (d, levels) on the host ([3BITS]: the codebook is stored, no calibration).
 *
 * Conventions
 * -----------
 * - Every function returns TQ_OK (0) or a negative TQ_E* code; nothing throws.
 * - Device pointers are plain CUDA device addresses on the context's device; the caller
 *   owns and allocates them (e.g. with PyTorch).  The library owns only the context's
 *   constant buffers (Pi, S, S Pi^T, codebooks, a status word).
 * - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are asynchronous on
 *   that stream and never synchronise the host, except tq_get_device_status.
 * - Supported: d in {64, 128, 256}, bits b in {2, 3, 4, 5}, m == d.
 * - Errors the host cannot see (a start position or sequence length read from device
 *   memory that exceeds max_tokens) make the kernels skip the offending work and set a
 *   sticky flag that tq_get_device_status reports.
 *
 * Compressed cache layout, format version 1
 * -----------------------------------------
 * cache = [batch][kv_head][page][page_bytes], P = TQ_PAGE_TOKENS = 128 token slots per
 * page; token t of a sequence lives in page t / P, slot t % P.  Each page holds six
 * regions, in this order (little-endian u32 words and f32 values):
 *   1. key codes    [b-1 planes][P slots][d/32 words]  plane q carries bit q of each code
 *   2. key signs    [P slots][m/32 words]              bit = sigma_i
 *   3. key norm     [P] f32                             n
 *   4. residual     [P] f32                             gamma
 *   5. value codes  [b planes][d coords][4 words]      plane q carries bit q of each code
 *   6. value norm   [P] f32                             n_v
 * page_bytes = P * ((b-1) d/8 + m/8 + 8 + b d/8 + 4)   (13,824 B at d = 128, b = 3).
 * Key codes and signs: within one slot's words, coordinate j is at
 *     kb = j>>5, h = (j>>4)&1, c = (j>>2)&3, e = j&3, s = c*(2*D/32) + 2*kb + h,
 *     word = s>>3, bit = (s&7) + 8*e          (D = d for codes, m for signs).
 * Value codes: within one coordinate's 4 words, token slot tau is at
 *     kb = tau>>5, h = (tau>>4)&1, c = (tau>>2)&3, e = tau&3, word = c, bit = 2*kb+h+8*e.
 * (These permutations put the bits that one thread of an m16n8k32 tensor-core fragment
 *  needs into one word.)  Slots not yet written hold arbitrary bytes; decode never reads
 *  them as data.
 */
#ifndef TQ_H
#define TQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TQ_FORMAT_VERSION 1
#define TQ_PAGE_TOKENS 128

enum {
  TQ_OK = 0,
  TQ_EINVAL = -1,       /* bad argument (null pointer, negative size, misaligned buffer) */
  TQ_EUNSUPPORTED = -2, /* d, bits, m or group size outside the supported set           */
  TQ_ECUDA = -3,        /* a CUDA runtime call or kernel launch failed                   */
  TQ_ETIMEOUT = -4,     /* a device-side bounded wait gave up (sticky device flag)       */
  TQ_EBOUNDS = -5,      /* device-side position / length beyond max_tokens (sticky flag) */
  TQ_ENOMEM = -6,       /* workspace too small, or a context allocation failed           */
  TQ_ENOTCONV = -7,     /* host codebook solver did not converge                        */
  TQ_ESCRATCH = -8      /* request needs more than the static scratch of                */
                        /* tq_attn_decode_noalloc (4 MiB)                               */
};

typedef struct tq_ctx tq_ctx;

/* Decode kernels (tq_ctx_set_decode_path).  All compute the same attention; they differ in
 * speed and in the configurations they serve. */
enum {
  TQ_DECODE_AUTO = 0, /* fastest kernel that serves the call (the default)                */
  TQ_DECODE_SIMT = 1, /* CUDA cores: every d, bits and group size                          */
  TQ_DECODE_MMA = 2,  /* fp8 mma.sync over bit planes: d in {64,128,256}; how many query   */
                      /* heads per kv head it takes shrinks as d and bits grow (registers) */
  TQ_DECODE_TC = 3,   /* tcgen05 over bit planes, e4m3 operands: d == 128, bits in {2,3},  */
                      /* group size <= 16                                                   */
  TQ_DECODE_TC4 = 4   /* tcgen05 over signed bit planes, block-scaled e2m1 operands        */
                      /* (kind::mxf4): d == 128, bits in {2,3} with group size <= 8 or 16  */
                      /* (four passes of four), bits 4 with group size 1, 2, 4 or 8 (two   */
                      /* query heads per pass)                                             */
};

/* ---- host-only set-up (no GPU needed) ------------------------------------------- */

/* Lloyd-Max codebook for one coordinate of a uniform unit vector in R^d ([BLOG] 1.2,
 * stage 1; [3BITS] "idea two").  d >= 3, 2 <= levels <= 64.  Writes `levels` ascending
 * centroids and `levels-1` interior boundaries (midpoints), fp64, into caller-owned host
 * memory.  The book is exactly antisymmetric, so the middle boundary is 0. */
int tq_make_codebook(int d, int levels, double* centroids, double* boundaries);

/* Haar rotation Pi ([BLOG] 1.2, "random orthogonal rotation"), d x d row-major fp64 into
 * caller-owned host memory; y = Pi x.  1 <= d <= 4096. */
int tq_make_rotation(int d, uint64_t seed, double* pi_out);

/* QJL projection S ([BLOG] 1.2, stage 2, "random Gaussian matrix"), m x d row-major fp64,
 * i.i.d. N(0,1).  1 <= m, d <= 4096. */
int tq_make_projection(int m, int d, uint64_t seed, double* s_out);

/* ---- context -------------------------------------------------------------------- */

/* Builds Pi, S, S Pi^T and both codebooks for (d, bits, m, seed) on the host and copies
 * them to `device`.  Returns TQ_EUNSUPPORTED unless d in {64,128,256}, bits in 2..5 and
 * m == d.  The context is immutable afterwards and may be shared by concurrent calls. */
int tq_ctx_create(int d, int bits, int m, uint64_t seed, int device, tq_ctx** out);

/* Format version 2: separate key and value widths, keys with or without the QJL stage
 * ([3BITS] "Python + HuggingFace": a cache object built with key_bits and value_bits, and a
 * stage-1 quantizer alone returning indices and norms; the same page notes that the llama.cpp
 * forks switch QJL off for keys).  key_bits counts every stored bit of a key coordinate: with
 * qjl != 0 the key book has 2^(key_bits-1) levels plus one sign bit per projected coordinate
 * (m = d); with qjl == 0 it has 2^key_bits levels and the page has no sign and gamma regions.
 * value_bits: value book of 2^value_bits levels.  The page holds the version-1 regions in the
 * same order and bit order with KB = key_bits - (qjl ? 1 : 0) key planes, VB = value_bits value
 * planes and, without QJL, regions 2 (signs) and 4 (gamma) dropped:
 *   page bytes = P (KB d/8 + 4 + VB d/8 + 4) + (qjl ? P (d/8 + 4) : 0).
 * qjl != 0 with key_bits == value_bits is version 1 (tq_ctx_create(d, key_bits, d, ...)).
 * Version-2 contexts quantize, decode (TQ_DECODE_AUTO or _SIMT only) and dequantize on CUDA
 * cores.  TQ_EUNSUPPORTED unless d in {64,128,256}, 1 <= KB <= 5 and 1 <= value_bits <= 5. */
int tq_ctx_create_kv(int d, int key_bits, int value_bits, int qjl, uint64_t seed, int device, tq_ctx** out);
void tq_ctx_destroy(tq_ctx* ctx);

/* Bytes of one page, and of a whole cache [batch][kv_heads][ceil(max_tokens/P)] pages
 * (0 on a bad argument). */
size_t tq_page_bytes(const tq_ctx* ctx);
size_t tq_cache_bytes(const tq_ctx* ctx, int batch, int kv_heads, int max_tokens);

/* Copies the context's fp64 host-side constants into caller buffers (any may be NULL):
 * pi [d*d], s [m*d], key codebook [2^(b-1)] + boundaries [2^(b-1)-1], value codebook
 * [2^b] + boundaries [2^b-1].  Used to cross-check the set-up against an independent
 * implementation. */
int tq_ctx_get_constants(const tq_ctx* ctx, double* pi, double* s, double* ck, double* tk,
                         double* cv, double* tv);

/* Selects the decode kernel of this context (TQ_DECODE_*).  Returns TQ_EINVAL for an
 * unknown value and TQ_EUNSUPPORTED if the kernel cannot serve this context's d and bits;
 * a group size the kernel cannot serve makes tq_attn_decode return TQ_EUNSUPPORTED.  The
 * workspace size depends on the choice, so query tq_decode_workspace_bytes after it.  Not
 * synchronised with decode calls: set it before the context is shared. */
int tq_ctx_set_decode_path(tq_ctx* ctx, int path);

/* ---- hot path ------------------------------------------------------------------- */

/* Quantizes n_tokens new key and value vectors per (batch, kv head) into the cache
 * ([BLOG] 1.2 stages 1 and 2 for keys, stage 1 with b bits for values).
 *   k, v       device bf16 [batch][kv_heads][n_tokens][d], contiguous, 16-byte aligned
 *   start_pos  device int32 [batch]: slot of the first new token of each sequence; token i
 *              goes to slot start_pos[b] + i.  Any alignment is allowed.
 *   cache      device, tq_cache_bytes(ctx, batch, kv_heads, max_tokens) bytes, 256-byte
 *              aligned; only the slots written are modified.
 * If start_pos[b] < 0 or start_pos[b] + n_tokens > max_tokens, sequence b is skipped and
 * the sticky TQ_EBOUNDS flag is set.  Calls that write the same page must be ordered.
 * n_tokens == 0 is a no-op that returns TQ_OK (k, v, start_pos and cache may then be NULL). */
int tq_quantize_kv(const tq_ctx* ctx, const void* k, const void* v, int batch, int kv_heads,
                   int n_tokens, const int32_t* start_pos, void* cache, int max_tokens,
                   void* stream);

/* tq_quantize_kv with the key and value vectors at any strides, so that a prefill writes its
 * projection output straight into the compressed cache without a transpose ([3BITS]: the
 * quantization overhead a prefill pays; [BLOG] 3.5, vLLM).  strides: host int64 [6], in bf16
 * elements: element j of the key of token i of (batch b, kv head h) is
 *   k[b * strides[0] + h * strides[1] + i * strides[2] + j]
 * and likewise v with strides[3..5].  Each stride must be >= 0 and a multiple of 8 (rows stay
 * on 16-byte boundaries); a [batch][n_tokens][kv_heads][d] projection output has
 * (n_tokens kv_heads d, d, kv_heads d).  Otherwise exactly tq_quantize_kv (the contiguous
 * call is strides (kv_heads n_tokens d, n_tokens d, d) twice); NULL strides: TQ_EINVAL. */
int tq_quantize_kv_strided(const tq_ctx* ctx, const void* k, const void* v, const int64_t* strides,
                           int batch, int kv_heads, int n_tokens, const int32_t* start_pos, void* cache,
                           int max_tokens, void* stream);

/* Scratch bytes tq_attn_decode needs for these sizes. */
size_t tq_decode_workspace_bytes(const tq_ctx* ctx, int batch, int q_heads, int kv_heads,
                                 int max_tokens);

/* Decode attention over the compressed cache (one query per head).
 *   q          device fp32 [batch][q_heads][d]
 *   cache      as written by tq_quantize_kv, [batch][kv_heads][pages][page]
 *   seq_lens   device int32 [batch]: attend to slots t < seq_lens[b]; 0 gives a zero row.
 *              A value above max_tokens is clamped and sets the sticky TQ_EBOUNDS flag.
 *   out        device fp32 [batch][q_heads][d]
 *   logits_out NULL, or device fp32 [batch][q_heads][max_tokens]: receives every logit
 *              t < seq_lens[b] (for testing; other entries untouched)
 *   workspace  device scratch of at least tq_decode_workspace_bytes(...) bytes, 256-byte
 *              aligned; its contents need no initialisation.
 * q_heads must be a multiple of kv_heads (query head h reads kv head h / (q_heads/kv_heads)),
 * with at most 16 query heads per kv head. */
int tq_attn_decode(const tq_ctx* ctx, const float* q, int batch, int q_heads, int kv_heads,
                   const void* cache, const int32_t* seq_lens, int max_tokens, float* out,
                   float* logits_out, void* workspace, size_t workspace_bytes, void* stream);

/* tq_attn_decode without a caller-provided workspace, for callers that cannot allocate
 * device memory at decode time (a serving loop whose memory pool is frozen after start-up,
 * a plugin whose host framework forbids cudaMalloc during a request, code that must avoid
 * the synchronisation an allocation can imply).  No counterpart on the pages: this is an
 * interface convenience, the computation is exactly tq_attn_decode's.
 * The scratch is one 4 MiB array in the library's device image (every GPU that loads the
 * library holds it until the process exits); a request whose tq_decode_workspace_bytes
 * exceeds 4 MiB returns TQ_ESCRATCH.  Nothing is allocated: no cudaMalloc, cudaFree or
 * allocating library routine is called.  The scratch needs no initialisation, and it is
 * shared by every call on a device and keeps the last call's contents, so calls that can
 * overlap on the GPU (other streams, other threads) race: order them.  The first call on a
 * device looks up the scratch address (cudaGetSymbolAddress) and must come before any
 * stream capture.  A device reset (cudaDeviceReset) invalidates the looked-up address along with
 * every context on that device; tq_ctx_create on the device makes the next call look it up
 * again.  Arguments and error codes otherwise exactly as tq_attn_decode's. */
int tq_attn_decode_noalloc(const tq_ctx* ctx, const float* q, int batch, int q_heads, int kv_heads,
                           const void* cache, const int32_t* seq_lens, int max_tokens, float* out,
                           float* logits_out, void* stream);

/* Compressed inner-product scan: for every query head, the k cached keys of its KV head with
 * the largest estimated inner product ([BLOG] 6.4, research directions: vector search and the
 * compression of RAG indexes; its FAQ: the method applies to any high-dimensional vectors):
 *   <q, k^_t> = n_t <Pi q, c_K[idx_t]> + gamma_t sqrt(pi/2)/m <S q, 2 sigma_t - 1>
 * (the QJL term only when the keys keep it), i.e. the decode score times sqrt(d).
 *   q, cache, seq_lens, batch, q_heads, kv_heads, max_tokens  as tq_attn_decode (the scores
 *              come from the decode kernel that serves the context)
 *   k          1 .. TQ_TOPK_MAX
 *   out_idx    device int32 [batch][q_heads][k]: slots, by decreasing estimate (the fp32 value
 *              out_score returns), equal estimates by increasing slot; -1 past seq_lens[b]
 *   out_score  device fp32 [batch][q_heads][k]: the estimates (-inf past seq_lens[b])
 *   workspace  device, 256-byte aligned, >= tq_ip_topk_workspace_bytes(...) bytes
 * Errors: tq_attn_decode's, TQ_EINVAL for k or the outputs, TQ_ENOMEM for a short workspace. */
#define TQ_TOPK_MAX 1024
size_t tq_ip_topk_workspace_bytes(const tq_ctx* ctx, int batch, int q_heads, int kv_heads, int max_tokens);
int tq_ip_topk(const tq_ctx* ctx, const float* q, int batch, int q_heads, int kv_heads, const void* cache,
               const int32_t* seq_lens, int max_tokens, int k, int32_t* out_idx, float* out_score, void* workspace,
               size_t workspace_bytes, void* stream);

/* Reconstructs cached vectors in the original frame, from the page contents alone
 * ([BLOG] 1.2: dequantization of stage 1, x~ = n Pi^T c[idx], and the stage-2 estimate of the
 * key residual from its signs; [3BITS] "Python + HuggingFace": dequantize(indices, norms)):
 *   keys    k^ = n_k Pi^T c_K[idx] + gamma sqrt(pi/2)/m S^T (2 sigma - 1)
 *   values  v^ = n_v Pi^T c_V[idx]
 *   cache      as written by tq_quantize_kv
 *   start_pos  device int32 [batch]: slot of the first vector read for each sequence
 *   k_out, v_out  device fp32 [batch][kv_heads][n_tokens][d], either may be NULL (skipped)
 * A sequence whose start_pos[b] < 0 or start_pos[b] + n_tokens > max_tokens is skipped and
 * sets the sticky TQ_EBOUNDS flag.  Not on the decode path (which never materialises k^ or
 * v^): for inspection, error statistics and tests.  CUDA cores, fp32. */
int tq_dequantize_kv(const tq_ctx* ctx, const void* cache, int batch, int kv_heads, int max_tokens,
                     const int32_t* start_pos, int n_tokens, float* k_out, float* v_out, void* stream);

/* Sparse V ([3BITS] llama.cpp section, the format list: positions with low attention weights
 * are skipped during decoding): with p_t = exp(l_t - m), a position whose p_t < threshold
 * contributes no value to the attention output; the softmax denominator still counts every
 * position (the scores are computed either way; the value work is what is skipped).  m is
 * the running maximum of the kernel's pass over the cache (each split its own), which never
 * exceeds the true maximum: a decode keeps every position that the same rule with the true
 * maximum keeps, and possibly more, so its output differs from the rule's definition by at
 * most sum over the definition's skipped t of p_t ||v^_t|| / sum_t p_t.  threshold 0 (the
 * default) is dense attention; 0 <= threshold <= 1, else TQ_EINVAL.  Logits are unaffected.
 * Applies to every later decode call of the context (tq_attn_decode and its _paged and
 * _noalloc forms); tq_ip_topk's estimates do not depend on it. */
int tq_ctx_set_sparse_v(tq_ctx* ctx, float threshold);

/* Paged (block-table) cache: the compressed pages live in a pool of blocks that sequences
 * borrow in any order, the layout of a PagedAttention-style serving engine ([BLOG] 3.5 "Другие
 * инструменты и фреймворки", vLLM: PagedAttention; [3BITS] "vLLM": the TurboQuant attention
 * backend behind --kv-cache-dtype).  The arithmetic, the page format and every kernel are
 * those of the contiguous calls; only where a page lives differs.
 *   pool         device, 256-byte aligned, tq_paged_pool_bytes(ctx, kv_heads, n_blocks) bytes:
 *                n_blocks blocks, each the kv_heads pages (tq_page_bytes each) of 128
 *                consecutive token slots; page (block, h) at byte (block * kv_heads + h) *
 *                tq_page_bytes.  Untouched bytes are never read by a decode that stays
 *                within seq_lens.
 *   block_table  device int32 [batch][max_blocks]: block_table[b][p] = the block holding slots
 *                128 p .. 128 p + 127 of sequence b.  Entries are read only for pages a call
 *                touches.  An entry outside [0, n_blocks) is clamped into the pool and sets
 *                the sticky TQ_EBOUNDS flag; two sequences given the same block share it.
 *   max_blocks   entries per table row; the sequences' capacity is max_blocks * 128 slots and
 *                takes the place of max_tokens in every other argument rule (start_pos,
 *                seq_lens, workspace: tq_decode_workspace_bytes(..., max_blocks * 128)).
 * Otherwise arguments, errors and results exactly as tq_quantize_kv, tq_attn_decode,
 * tq_dequantize_kv and tq_ip_topk with `cache` replaced by (pool, n_blocks, block_table,
 * max_blocks):
 * a paged pool whose table maps (b, p) to block b * max_blocks + p holds the contiguous
 * cache byte for byte when kv_heads == 1, and any table gives bit-identical outputs. */
size_t tq_paged_pool_bytes(const tq_ctx* ctx, int kv_heads, int n_blocks);
int tq_quantize_kv_paged(const tq_ctx* ctx, const void* k, const void* v, int batch, int kv_heads,
                         int n_tokens, const int32_t* start_pos, void* pool, int n_blocks,
                         const int32_t* block_table, int max_blocks, void* stream);
int tq_attn_decode_paged(const tq_ctx* ctx, const float* q, int batch, int q_heads, int kv_heads,
                         const void* pool, int n_blocks, const int32_t* block_table, int max_blocks,
                         const int32_t* seq_lens, float* out, float* logits_out, void* workspace,
                         size_t workspace_bytes, void* stream);
int tq_dequantize_kv_paged(const tq_ctx* ctx, const void* pool, int n_blocks, const int32_t* block_table,
                           int max_blocks, int batch, int kv_heads, const int32_t* start_pos, int n_tokens,
                           float* k_out, float* v_out, void* stream);
/* tq_quantize_kv_paged with strided K / V (strides as tq_quantize_kv_strided). */
int tq_quantize_kv_paged_strided(const tq_ctx* ctx, const void* k, const void* v, const int64_t* strides,
                                 int batch, int kv_heads, int n_tokens, const int32_t* start_pos, void* pool,
                                 int n_blocks, const int32_t* block_table, int max_blocks, void* stream);
/* tq_ip_topk on a paged pool (workspace: tq_ip_topk_workspace_bytes(..., max_blocks * 128)). */
int tq_ip_topk_paged(const tq_ctx* ctx, const float* q, int batch, int q_heads, int kv_heads,
                     const void* pool, int n_blocks, const int32_t* block_table, int max_blocks,
                     const int32_t* seq_lens, int k, int32_t* out_idx, float* out_score, void* workspace,
                     size_t workspace_bytes, void* stream);

/* Self-test of the device-side failure path: launches one thread that waits, with the same
 * bounded wait every kernel uses, on an mbarrier nothing arrives at.  The wait gives up after
 * its limit (2 s), sets the sticky timeout flag and the kernel returns; a following
 * tq_get_device_status reports TQ_ETIMEOUT.  Nothing faults or hangs. */
int tq_selftest_bounded_wait(const tq_ctx* ctx, void* stream);

/* Synchronises `stream`, then returns and clears the sticky device status: TQ_OK,
 * TQ_EBOUNDS or TQ_ETIMEOUT. */
int tq_get_device_status(const tq_ctx* ctx, void* stream);

const char* tq_status_string(int status);

#ifdef __cplusplus
}
#endif
#endif /* TQ_H */
