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
// - Residency: the array is the device code of this file's module, which
//   holds no kernel.  Under lazy module loading (the CUDA default) that
//   module, and so the 32 MiB, is loaded into a context by the first call of
//   this entry point there; with eager loading (CUDA_MODULE_LOADING=EAGER) it
//   is loaded into every context the library's modules are loaded into,
//   whether or not this entry point is ever called.  Either way it stays
//   until the context is destroyed or the process exits.
// - Set-up: the first call made in a context looks up the array's device
//   address there (cudaGetSymbolAddress, return code checked) and caches it
//   under the context's unique id (cuCtxGetId).  A later call in another
//   context -- a second context on the device, or the new primary context
//   after cudaDeviceReset -- looks it up again, so a stale address is never
//   launched.  Make the first call in a context before any stream capture.
// - Sharing: every call in a context uses the same array and it keeps the
//   last call's contents.  Nothing in it needs clearing: every partial a call
//   reads was written earlier in the same call, and the split-K arrival
//   counters count only arrivals tagged with the call's own epoch, so leftover
//   bytes read as no arrivals.  Two calls whose kernels overlap on the GPU
//   race on it: serialise such calls (one stream, or events).
#include <cudaTypedefs.h>

#include <mutex>

#include "pa_internal.h"

namespace pa {

// Unique id of the context current on this thread; false when there is none
// yet (the runtime creates the primary context lazily) or it cannot be read.
bool current_context_id(unsigned long long* id) {
  static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  static PFN_cuCtxGetId_v12000 get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  if (!get_current || !get_id) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
  return get_id(ctx, id) == CUDA_SUCCESS;
}

}  // namespace pa

namespace {

static __device__ __align__(256) unsigned char g_static_ws[PA_STATIC_WS_BYTES];

constexpr int kMaxDevices = 64;

// The array's address as last looked up on a device, and the context it
// belongs to.
struct WsAddr {
  bool valid = false;
  unsigned long long ctx_id = 0;
  void* addr = nullptr;
};
std::mutex g_setup_mu;
WsAddr g_ws[kMaxDevices];

// Device address of the static scratch in the current context.  The cached
// address is reused only while the current context is the one it was looked
// up in; anything else (no context yet, an id that cannot be read, another
// context) looks it up again.
pa_status static_ws_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return pa::fail(PA_ERR_CUDA, "pa_decode_static_ws: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices)
    return pa::fail(PA_ERR_UNSUPPORTED, "pa_decode_static_ws: device index %d >= %d", dev, kMaxDevices);
  unsigned long long id = 0;
  bool have_id = pa::current_context_id(&id);
  std::lock_guard<std::mutex> lock(g_setup_mu);
  WsAddr& c = g_ws[dev];
  if (have_id && c.valid && c.ctx_id == id) {
    *out = c.addr;
    return PA_OK;
  }
  void* p = nullptr;
  e = cudaGetSymbolAddress(&p, g_static_ws);
  if (e != cudaSuccess || !p)
    return pa::fail(PA_ERR_CUDA, "pa_decode_static_ws: cudaGetSymbolAddress failed: %s", cudaGetErrorString(e));
  if (!have_id) have_id = pa::current_context_id(&id);  // the lookup made the primary context current
  c.valid = have_id;
  c.ctx_id = id;
  c.addr = p;
  *out = p;
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
