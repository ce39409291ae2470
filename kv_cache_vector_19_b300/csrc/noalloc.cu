// Decode attention for callers that cannot allocate device memory.
//
// tq_attn_decode needs a scratch workspace (the rotated queries and the per-split partial
// softmax records) that the caller allocates.  Some callers cannot do that at decode time:
// a serving loop whose memory pool is sized and frozen at start-up, an inference plugin
// whose host framework forbids cudaMalloc while a request is in flight, or code that must
// not trigger the device-wide synchronisation an allocation can imply.  For them this file
// keeps one statically sized scratch array in the library's own device image and runs the
// same decode kernels on it.
#include <cuda_runtime.h>

#include <mutex>

#include "tq_internal.h"

namespace {

// Upper bound of the scratch; every GPU that loads the library holds it until the process
// exits.  4 MiB covers, e.g., 4 sequences x 8 KV heads x 32 query heads at 128K tokens.
constexpr size_t kScratchBytes = size_t(4) << 20;
constexpr int kMaxDevices = 64;

// Device-side scratch.  In host code this name is only a stand-in for the symbol, never a
// device address: the address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of g_decode_scratch on `device` (which must be current), looked up once per
// device and again after tq_ctx_create on that device (a device reset reloads the module).
int scratch_address(int device, void** out) {
  if (device < 0 || device >= kMaxDevices) return TQ_EINVAL;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[device]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return TQ_ECUDA;
    g_scratch_addr[device] = p;
  }
  *out = g_scratch_addr[device];
  return TQ_OK;
}

}  // namespace

namespace tq {
void noalloc_forget_device(int device) {
  if (device < 0 || device >= kMaxDevices) return;
  std::lock_guard<std::mutex> lock(g_mu);
  g_scratch_addr[device] = nullptr;
}
}  // namespace tq

extern "C" int tq_attn_decode_noalloc(const tq_ctx* ctx, const float* q, int batch, int q_heads, int kv_heads,
                                      const void* cache, const int32_t* seq_lens, int max_tokens, float* out,
                                      float* logits_out, void* stream) {
  // the same checks and error codes as tq_attn_decode, then the scratch size
  const int chk = tq::check_decode_args(ctx, q, batch, q_heads, kv_heads, cache, seq_lens, max_tokens, out, logits_out);
  if (chk != TQ_OK) return chk;
  const size_t need = tq_decode_workspace_bytes(ctx, batch, q_heads, kv_heads, max_tokens);
  if (need == 0) return TQ_EINVAL;
  if (need > kScratchBytes) return TQ_ESCRATCH;
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) return TQ_ECUDA;
  if (prev != ctx->device && cudaSetDevice(ctx->device) != cudaSuccess) return TQ_ECUDA;
  void* ws = nullptr;
  int rc = scratch_address(ctx->device, &ws);
  if (rc == TQ_OK)
    rc = tq_attn_decode(ctx, q, batch, q_heads, kv_heads, cache, seq_lens, max_tokens, out, logits_out, ws, need,
                        stream);
  if (prev != ctx->device) cudaSetDevice(prev);
  return rc;
}
