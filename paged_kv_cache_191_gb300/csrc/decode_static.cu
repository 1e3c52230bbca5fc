// pa_decode_static_ws: pa_decode for callers that cannot allocate device memory.
//
// Some callers have no way to obtain device scratch when they decode: code
// running as a plugin inside an engine whose allocator owns the whole device
// and offers plugins no scratch hook, or a latency-critical loop in which a
// cudaMalloc/cudaFree pair would add latency and device-wide synchronisation.
// This entry point runs the same kernels as pa_decode, with the split-K
// partials kept in one file-scope device array compiled into the library
// instead of a caller-provided workspace.  It allocates nothing.
//
// - Size: PA_STATIC_WS_BYTES (32 MiB).  Shapes whose workspace
//   (pa_decode_workspace_size) is larger are rejected with PA_ERR_INVALID
//   before anything is launched.
// - Residency: the array is part of the library's device code, so it occupies
//   32 MiB on every device where this entry point has been used, until the
//   process exits.
// - Set-up: the first call made with a device current looks up the array's
//   device address on that device (cudaGetSymbolAddress, once per device,
//   return code checked).  Make that first call before any stream capture.
// - Sharing: every call on a device uses the same array and it keeps the last
//   call's contents.  Nothing in it needs clearing (every partial a call reads
//   was written earlier in the same call), but two calls whose kernels overlap
//   on the GPU race on it: serialise such calls (one stream, or events).
#include <mutex>

#include "pa_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_ws[PA_STATIC_WS_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void* g_static_ws_addr[kMaxDevices] = {};  // device address of g_static_ws, per device

// Device address of the static scratch on the current device (set up once).
pa_status static_ws_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return pa::fail(PA_ERR_CUDA, "pa_decode_static_ws: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return pa::fail(PA_ERR_UNSUPPORTED, "pa_decode_static_ws: device index %d >= %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_static_ws_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_ws);
    if (e != cudaSuccess || !p)
      return pa::fail(PA_ERR_CUDA, "pa_decode_static_ws: cudaGetSymbolAddress failed: %s",
                      cudaGetErrorString(e));
    g_static_ws_addr[dev] = p;
  }
  *out = g_static_ws_addr[dev];
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_static_ws(const void* q, int32_t q_dtype, const void* k_cache,
                                         const void* v_cache, const float* k_scale,
                                         const float* v_scale, const int32_t* block_tables,
                                         int32_t max_blocks_per_seq, const int32_t* context_lens,
                                         int32_t max_context_len, int32_t B, int32_t num_q_heads,
                                         float scale, void* out, int32_t out_dtype,
                                         const pa_cache_desc* desc, int32_t split_tokens,
                                         void* stream) {
  const size_t need =
      pa_decode_workspace_size(B, num_q_heads, max_context_len, desc, split_tokens);
  if (need > PA_STATIC_WS_BYTES)
    return pa::fail(PA_ERR_INVALID,
                    "pa_decode_static_ws: this shape needs %zu bytes of split-K scratch; the "
                    "static array holds %zu (use pa_decode with a caller workspace)",
                    need, static_cast<size_t>(PA_STATIC_WS_BYTES));
  void* ws = nullptr;
  pa_status st = static_ws_address(&ws);
  if (st != PA_OK) return st;
  return pa_decode(q, q_dtype, k_cache, v_cache, k_scale, v_scale, block_tables,
                   max_blocks_per_seq, context_lens, max_context_len, B, num_q_heads, scale, out,
                   out_dtype, desc, ws, PA_STATIC_WS_BYTES, split_tokens, stream);
}
