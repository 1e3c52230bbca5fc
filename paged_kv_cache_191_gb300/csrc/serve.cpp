// One serving iteration, native: the scheduler's decisions become device
// work on one stream with a single host-to-device copy of everything the
// kernels need.
//
// Order on the stream (the decisions require it):
//   H2D of the staged decisions (slots, swap pairs, query offsets, context
//   lengths, block tables);
//   swap-out copies of preempted requests (GPU -> pinned host pool), before
//   any write can reuse the blocks they released;
//   decode items: cache write of the new token fused into paged decode
//   (pa_decode_append), one warp-sized partition per (sequence, kv head);
//   FP8 / INT8 caches carry their per-token scales through every step (the
//   writes store them, attention reads them, swaps move them with the blocks);
//   prompt chunks: pa_cache_write of their tokens, then pa_chunked_prefill
//   (causal inside each chunk);
//   swap-in copies (pinned host pool -> GPU) of requests that run next step.
// The scheduler emits decodes first, so they are a prefix of the items, of
// the query rows and of the slots.
//
// A step is planned (scheduler decisions staged in pinned memory; the caller
// learns how many new tokens the iteration brings, so the model can produce
// exactly their q / K / V) and then launched (device work).  Two pinned
// staging buffers alternate; before refilling one, the host waits for the
// copy that last read it (an event), so the host runs at most one iteration
// ahead of the device.
#include <algorithm>
#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include "pa_internal.h"

struct pa_serve {
  pa_sched* sched = nullptr;
  pa_cache_desc desc{};
  pa_serve_buffers b{};
  int32_t max_batch = 0, max_tokens = 0, cap = 0;
  size_t ws_decode = 0;  // workspace bytes reserved for the decode part (front)
  // staging layout: byte offsets of each field
  size_t o_slots = 0, o_out = 0, o_in = 0, o_qs = 0, o_lens = 0, o_tab = 0, bytes = 0;
  cudaEvent_t copied[2] = {nullptr, nullptr};
  bool used[2] = {false, false};
  int64_t step_no = 0;
  // the planned step waiting for its launch
  bool planned = false;
  int stage = 0;
  int32_t n = 0, n_dec = 0, max_q = 0, n_out = 0, n_in = 0;
  int64_t T = 0;
  // scheduler output arrays when the caller passes none
  std::vector<uint64_t> ids, fin, rec;
  std::vector<int32_t> kinds, starts, lens;
  std::vector<int64_t> slots, sw_out, sw_in;

  ~pa_serve() {
    for (cudaEvent_t e : copied)
      if (e) cudaEventDestroy(e);
  }
};

namespace {

size_t align16(size_t x) { return (x + 15) & ~static_cast<size_t>(15); }

// The model's q / K / V dtype: the cache's for 16-bit caches, F16 or BF16
// for 1-byte caches.
bool input_dtype_ok(int32_t kv_dtype, int32_t in_dtype) {
  if (pa::quantised(kv_dtype)) return in_dtype == PA_DTYPE_F16 || in_dtype == PA_DTYPE_BF16;
  return in_dtype == kv_dtype;
}

struct Layout {
  size_t slots, out, in, qs, lens, tab, bytes;
};

Layout layout(int32_t max_batch, int32_t max_tokens, int32_t num_blocks, int32_t cap) {
  Layout l;
  size_t o = 0;
  l.slots = o;
  o += align16(static_cast<size_t>(max_batch + max_tokens) * 8);
  l.out = o;
  o += align16(static_cast<size_t>(num_blocks) * 16);
  l.in = o;
  o += align16(static_cast<size_t>(num_blocks) * 16);
  l.qs = o;
  o += align16(static_cast<size_t>(max_batch + 1) * 4);
  l.lens = o;
  o += align16(static_cast<size_t>(max_batch) * 4);
  l.tab = o;
  o += align16(static_cast<size_t>(max_batch) * cap * 4);
  l.bytes = o;
  return l;
}

// Workspace of the decode part over every batch size it can see, and of the
// chunk part at the engine's fixed partition size.
void workspace_parts(int32_t max_batch, int32_t max_tokens, int32_t Hq, int32_t max_context,
                     const pa_cache_desc* d, int32_t split, size_t* dec, size_t* pre) {
  *dec = 0;
  for (int32_t B = 1; B <= max_batch; ++B)
    *dec = std::max(*dec, pa_decode_workspace_size(B, Hq, max_context, d, 0));
  *dec = align16(*dec);
  *pre = pa_chunked_prefill_workspace_size(max_tokens, max_batch, Hq, max_tokens, max_context, d, split);
}

}  // namespace

extern "C" {

size_t pa_serve_staging_bytes(const pa_sched* s, int32_t max_context) {
  int32_t mb = 0, mt = 0, nb = 0;
  if (!s || max_context <= 0 || pa_sched_limits(s, &mb, &mt, &nb) != PA_OK) return 0;
  return layout(mb, mt, nb, (max_context + PA_BLOCK_SIZE - 1) / PA_BLOCK_SIZE).bytes;
}

size_t pa_serve_workspace_bytes(const pa_sched* s, int32_t num_q_heads, int32_t max_context,
                                const pa_cache_desc* desc, int32_t split_tokens) {
  int32_t mb = 0, mt = 0, nb = 0;
  if (!s || !desc || split_tokens <= 0 || pa_sched_limits(s, &mb, &mt, &nb) != PA_OK) return 0;
  size_t dec, pre;
  workspace_parts(mb, mt, num_q_heads, max_context, desc, split_tokens, &dec, &pre);
  return dec + pre;
}

pa_status pa_serve_create(pa_sched* s, const pa_cache_desc* desc, const pa_serve_buffers* b, pa_serve** out) {
  if (!out) return pa::fail(PA_ERR_INVALID, "pa_serve_create: out is NULL");
  *out = nullptr;
  if (!s || !desc || !b) return pa::fail(PA_ERR_INVALID, "pa_serve_create: null argument");
  const bool q8 = pa::quantised(desc->kv_dtype);
  if (q8) {
    if (!b->k_scale || !b->v_scale || !pa::aligned16(b->k_scale) || !pa::aligned16(b->v_scale) ||
        (b->host_blocks && (!b->k_host_scale || !b->v_host_scale)))
      return pa::fail(PA_ERR_INVALID, "pa_serve_create: FP8 / INT8 caches need device (and host) scales");
  } else if (b->k_scale || b->v_scale || b->k_host_scale || b->v_host_scale) {
    return pa::fail(PA_ERR_INVALID, "pa_serve_create: scales are only for FP8 / INT8 caches");
  }
  int32_t mb = 0, mt = 0, nb = 0;
  pa_status st = pa_sched_limits(s, &mb, &mt, &nb);
  if (st != PA_OK) return st;
  if (nb != desc->num_blocks) return pa::fail(PA_ERR_INVALID, "pa_serve_create: desc->num_blocks != scheduler pool");
  if (b->max_context <= 0 || b->num_q_heads <= 0 || b->split_tokens <= 0 || b->host_blocks < 0)
    return pa::fail(PA_ERR_INVALID, "pa_serve_create: max_context, num_q_heads, split_tokens must be > 0");
  if (!b->k_cache || !b->v_cache || !b->staging_host || !b->staging_dev || (b->host_blocks && (!b->k_host || !b->v_host)))
    return pa::fail(PA_ERR_INVALID, "pa_serve_create: null buffer");
  pa_serve* e = new (std::nothrow) pa_serve();
  if (!e) return pa::fail(PA_ERR_OOM, "pa_serve_create: host allocation failed");
  e->sched = s;
  e->desc = *desc;
  e->b = *b;
  e->max_batch = mb;
  e->max_tokens = mt;
  e->cap = (b->max_context + PA_BLOCK_SIZE - 1) / PA_BLOCK_SIZE;
  const Layout l = layout(mb, mt, nb, e->cap);
  e->o_slots = l.slots;
  e->o_out = l.out;
  e->o_in = l.in;
  e->o_qs = l.qs;
  e->o_lens = l.lens;
  e->o_tab = l.tab;
  e->bytes = l.bytes;
  size_t dec, pre;
  workspace_parts(mb, mt, b->num_q_heads, e->cap * PA_BLOCK_SIZE, desc, b->split_tokens, &dec, &pre);
  if (b->workspace_bytes < dec + pre || (dec + pre && !b->workspace)) {
    delete e;
    return pa::fail(PA_ERR_INVALID, "pa_serve_create: workspace has %zu bytes, %zu needed", b->workspace_bytes,
                    dec + pre);
  }
  e->ws_decode = dec;
  for (cudaEvent_t& ev : e->copied)
    if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) {
      delete e;
      return pa::fail(PA_ERR_CUDA, "pa_serve_create: cudaEventCreate failed");
    }
  e->ids.resize(mb);
  e->fin.resize(mb);
  e->rec.resize(mb);
  e->kinds.resize(mb);
  e->starts.resize(mb);
  e->lens.resize(mb);
  e->slots.resize(static_cast<size_t>(mb) + mt);
  e->sw_out.resize(2 * static_cast<size_t>(nb));
  e->sw_in.resize(2 * static_cast<size_t>(nb));
  *out = e;
  return pa::ok();
}

void pa_serve_destroy(pa_serve* e) { delete e; }

pa_status pa_serve_plan(pa_serve* e, pa_sched_step_out* d, int64_t* num_tokens) {
  if (!e) return pa::fail(PA_ERR_INVALID, "pa_serve_plan: null handle");
  if (e->planned) return pa::fail(PA_ERR_INVALID, "pa_serve_plan: the previous plan was not launched");
  pa_sched_step_out own;
  if (!d) {
    own.ids = e->ids.data();
    own.kinds = e->kinds.data();
    own.starts = e->starts.data();
    own.lens = e->lens.data();
    own.slots = e->slots.data();
    own.finished = e->fin.data();
    own.recomputed = e->rec.data();
    own.swap_out = e->sw_out.data();
    own.swap_in = e->sw_in.data();
    d = &own;
  }
  const int i = static_cast<int>(e->step_no & 1);
  if (e->used[i] && cudaEventSynchronize(e->copied[i]) != cudaSuccess)
    return pa::fail(PA_ERR_CUDA, "pa_serve_plan: event wait failed");
  pa_status st = pa_sched_step(e->sched, d);
  if (st != PA_OK) return st;
  const int32_t n = d->n_items;
  int32_t n_dec = 0;
  while (n_dec < n && d->kinds[n_dec] == PA_SCHED_DECODE) ++n_dec;
  // ---- stage the decisions ----
  uint8_t* h = static_cast<uint8_t*>(e->b.staging_host) + static_cast<size_t>(i) * e->bytes;
  std::memcpy(h + e->o_slots, d->slots, static_cast<size_t>(d->n_slots) * 8);
  std::memcpy(h + e->o_out, d->swap_out, static_cast<size_t>(d->n_swap_out) * 16);
  std::memcpy(h + e->o_in, d->swap_in, static_cast<size_t>(d->n_swap_in) * 16);
  int32_t* qs = reinterpret_cast<int32_t*>(h + e->o_qs);  // chunk part: offsets from its first row
  qs[0] = 0;
  int32_t max_q = 0;
  for (int32_t k = n_dec; k < n; ++k) {
    qs[k - n_dec + 1] = qs[k - n_dec] + d->lens[k];
    max_q = std::max(max_q, d->lens[k]);
  }
  if (n) {
    st = pa_block_tables(pa_sched_allocator(e->sched), d->ids, n, reinterpret_cast<int32_t*>(h + e->o_tab), e->cap,
                         reinterpret_cast<int32_t*>(h + e->o_lens));
    if (st != PA_OK) return st;
  }
  e->planned = true;
  e->stage = i;
  e->n = n;
  e->n_dec = n_dec;
  e->max_q = max_q;
  e->T = d->n_slots;
  e->n_out = d->n_swap_out;
  e->n_in = d->n_swap_in;
  ++e->step_no;
  if (num_tokens) *num_tokens = d->n_slots;
  return pa::ok();
}

pa_status pa_serve_launch(pa_serve* e, const void* q, const void* k_new, const void* v_new, int32_t in_dtype,
                          void* out, void* stream) {
  if (!e) return pa::fail(PA_ERR_INVALID, "pa_serve_launch: null handle");
  if (!e->planned) return pa::fail(PA_ERR_INVALID, "pa_serve_launch: no planned step");
  if (!input_dtype_ok(e->desc.kv_dtype, in_dtype))
    return pa::fail(PA_ERR_INVALID, "pa_serve_launch: in_dtype must be the cache dtype (F16 / BF16 for FP8 / INT8)");
  if (e->T && (!q || !k_new || !v_new || !out)) return pa::fail(PA_ERR_INVALID, "pa_serve_launch: null argument");
  const pa_serve_buffers& b = e->b;
  const int32_t Hq = b.num_q_heads, Hkv = e->desc.num_kv_heads, D = e->desc.head_dim;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const uint8_t* h = static_cast<const uint8_t*>(b.staging_host) + static_cast<size_t>(e->stage) * e->bytes;
  uint8_t* dv = static_cast<uint8_t*>(b.staging_dev);
  // the plan is consumed whatever happens below
  e->planned = false;
  if (cudaMemcpyAsync(dv, h, e->bytes, cudaMemcpyHostToDevice, cs) != cudaSuccess ||
      cudaEventRecord(e->copied[e->stage], cs) != cudaSuccess)
    return pa::fail(PA_ERR_CUDA, "pa_serve_launch: staging copy failed");
  e->used[e->stage] = true;

  const int64_t* d_slots = reinterpret_cast<const int64_t*>(dv + e->o_slots);
  const int32_t* d_lens = reinterpret_cast<const int32_t*>(dv + e->o_lens);
  const int32_t* d_tab = reinterpret_cast<const int32_t*>(dv + e->o_tab);
  const int32_t max_ctx = e->cap * PA_BLOCK_SIZE;
  const float scale = 1.0f / std::sqrt(static_cast<float>(D));
  const size_t qrow = static_cast<size_t>(Hq) * D * 2, kvrow = static_cast<size_t>(Hkv) * D * 2;
  const int32_t n = e->n, n_dec = e->n_dec;
  pa_status st;
  if (e->n_out) {
    st = pa_swap_blocks(b.k_host, b.v_host, b.k_host_scale, b.v_host_scale, b.host_blocks, b.k_cache, b.v_cache,
                        b.k_scale, b.v_scale, e->desc.num_blocks, reinterpret_cast<const int64_t*>(dv + e->o_out),
                        e->n_out, &e->desc, stream);
    if (st != PA_OK) return st;
  }
  if (n_dec) {
    st = pa_decode_append(k_new, v_new, in_dtype, d_slots, q, in_dtype, b.k_cache, b.v_cache, b.k_scale, b.v_scale, d_tab,
                          e->cap, d_lens, max_ctx, n_dec, Hq, scale, out, in_dtype, &e->desc, b.workspace,
                          e->ws_decode, 0, stream);
    if (st != PA_OK) return st;
  }
  const int64_t Tc = e->T - n_dec;
  if (Tc > 0) {
    const uint8_t* kc = static_cast<const uint8_t*>(k_new) + n_dec * kvrow;
    const uint8_t* vc = static_cast<const uint8_t*>(v_new) + n_dec * kvrow;
    st = pa_cache_write(kc, vc, in_dtype, d_slots + n_dec, Tc, b.k_cache, b.v_cache, b.k_scale, b.v_scale, &e->desc,
                        stream);
    if (st != PA_OK) return st;
    st = pa_chunked_prefill(static_cast<const uint8_t*>(q) + n_dec * qrow, in_dtype,
                            reinterpret_cast<const int32_t*>(dv + e->o_qs), static_cast<int32_t>(Tc), e->max_q,
                            b.k_cache, b.v_cache, b.k_scale, b.v_scale, d_tab + static_cast<size_t>(n_dec) * e->cap,
                            e->cap,
                            d_lens + n_dec, max_ctx, n - n_dec, Hq, scale,
                            static_cast<uint8_t*>(out) + n_dec * qrow, in_dtype, &e->desc,
                            static_cast<uint8_t*>(b.workspace) + e->ws_decode, b.workspace_bytes - e->ws_decode,
                            b.split_tokens, stream);
    if (st != PA_OK) return st;
  }
  if (e->n_in) {
    st = pa_swap_blocks(b.k_cache, b.v_cache, b.k_scale, b.v_scale, e->desc.num_blocks, b.k_host, b.v_host,
                        b.k_host_scale, b.v_host_scale, b.host_blocks, reinterpret_cast<const int64_t*>(dv + e->o_in),
                        e->n_in, &e->desc, stream);
    if (st != PA_OK) return st;
  }
  return pa::ok();
}

pa_status pa_serve_step(pa_serve* e, const void* q, const void* k_new, const void* v_new, int32_t in_dtype,
                        void* out, pa_sched_step_out* d, void* stream) {
  if (!e) return pa::fail(PA_ERR_INVALID, "pa_serve_step: null handle");
  if (!input_dtype_ok(e->desc.kv_dtype, in_dtype))
    return pa::fail(PA_ERR_INVALID, "pa_serve_step: in_dtype must be the cache dtype (F16 / BF16 for FP8 / INT8)");
  pa_status st = pa_serve_plan(e, d, nullptr);
  if (st != PA_OK) return st;
  return pa_serve_launch(e, q, k_new, v_new, in_dtype, out, stream);
}

}  // extern "C"
