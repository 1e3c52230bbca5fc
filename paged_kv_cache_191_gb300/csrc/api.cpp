// C-ABI entry points: host-side validation, then dispatch to the launchers.
// Nothing is enqueued unless every host-visible argument checks out.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <string>

#include <cuda_runtime.h>

#include "pa_internal.h"

#ifndef PA_FUSED_MERGE
#define PA_FUSED_MERGE 1  // split-K partials merged by the decode kernel's last partition
#endif
#ifndef PA_FUSED_MERGE_MAX
#define PA_FUSED_MERGE_MAX 8  // most partitions merged that way
#endif
#ifndef PA_ROUTE_SINGLE16
#define PA_ROUTE_SINGLE16 0  // one-token sequences of a 16-bit multi-token call to the decode kernel
#endif
#ifndef PA_Q8_WARPS
#define PA_Q8_WARPS 4  // warps sharing one partition over a 1-byte cache
#endif

namespace pa {

static thread_local std::string g_last_error;

pa_status fail(pa_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

static pa_status check_desc(const pa_cache_desc* d, const char* fn) {
  if (!d) return fail(PA_ERR_INVALID, "%s: desc is NULL", fn);
  if (d->block_size != PA_BLOCK_SIZE)
    return fail(PA_ERR_UNSUPPORTED, "%s: block_size must be 16", fn);
  if (d->num_blocks <= 0 || d->num_kv_heads <= 0 || d->head_dim <= 0)
    return fail(PA_ERR_INVALID, "%s: num_blocks, num_kv_heads, head_dim must be > 0", fn);
  if (d->kv_dtype != PA_DTYPE_F16 && d->kv_dtype != PA_DTYPE_BF16 && !quantised(d->kv_dtype))
    return fail(PA_ERR_INVALID, "%s: kv_dtype must be F16, BF16, FP8_E4M3 or INT8", fn);
  if (d->head_dim != 64 && d->head_dim != 128)
    return fail(PA_ERR_UNSUPPORTED, "%s: head_dim %d not built (64, 128)", fn, d->head_dim);
  if (quantised(d->kv_dtype) && d->head_dim != 128)
    return fail(PA_ERR_UNSUPPORTED, "%s: FP8 / INT8 caches need head_dim 128", fn);
  return PA_OK;
}

static int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return 148;
  return n;
}

pa_status plan_decode(int32_t B, int32_t Hq, int32_t max_context_len, const pa_cache_desc* d,
                      int32_t split_tokens, DecodePlan* plan) {
  const int64_t nblk_max = max_context_len <= 0 ? 1 : (max_context_len + PA_BLOCK_SIZE - 1) / PA_BLOCK_SIZE;
  int32_t bpp;
  if (split_tokens > 0) {
    if (split_tokens % PA_BLOCK_SIZE || split_tokens > 1024)
      return fail(PA_ERR_INVALID, "split_tokens must be a multiple of 16 in [16, 1024]");
    bpp = split_tokens / PA_BLOCK_SIZE;
  } else {
    // 512-token partitions by default and 1024 for contexts of 8K and more
    // (fewer partials to merge; one-warp CTAs keep the grid fine-grained);
    // shrink them while the grid would give fewer than two partitions per SM.
    const int64_t units = static_cast<int64_t>(B) * d->num_kv_heads;
    const int64_t sms = sm_count();
    bpp = max_context_len >= 8192 ? 64 : 32;
    while (bpp > 4 && units * ((nblk_max + bpp - 1) / bpp) < 2 * sms) bpp /= 2;
  }
  const int64_t parts = (nblk_max + bpp - 1) / bpp;
  if (parts > 65535) return fail(PA_ERR_UNSUPPORTED, "context too long for the partition grid");
  plan->blocks_per_part = bpp;
  plan->max_parts = static_cast<int32_t>(parts);
  // 1-byte codes cost more register-side work per byte (exact conversion of
  // the codes), so four warps share a partition there; 16-bit caches keep
  // one warp per partition (measured best for both).
  plan->item_warps = quantised(d->kv_dtype) ? PA_Q8_WARPS : 1;
  if (parts > 1) {
    const size_t rows = static_cast<size_t>(B) * Hq * parts;
    size_t bytes = rows * d->head_dim * sizeof(float) + 2 * rows * sizeof(float);
    plan->workspace_bytes = (bytes + 255) & ~static_cast<size_t>(255);
  } else {
    plan->workspace_bytes = 0;
  }
  // Splits of at most 8 partitions merge in the decode kernel (one warp merges
  // a pair's partials quickly enough to sit on the grid's critical path):
  // one 8-byte arrival counter per (sequence, kv head) after the partials.
  // Longer merges go to the merge kernel, which spreads them over a warp per
  // query head.
  plan->ticket_offset = 0;
  if (PA_FUSED_MERGE && parts > 1 && parts <= PA_FUSED_MERGE_MAX) {
    plan->ticket_offset = plan->workspace_bytes;
    const size_t tickets = static_cast<size_t>(B) * d->num_kv_heads * 8;
    plan->workspace_bytes += (tickets + 255) & ~static_cast<size_t>(255);
  }
  return PA_OK;
}

bool prefill_routes_short(int32_t max_q_len, int32_t Hq, const pa_cache_desc* d) {
  const int64_t G = Hq / d->num_kv_heads;
  return !quantised(d->kv_dtype) && max_q_len >= 1 && max_q_len <= kShortTokens && max_q_len * G <= 32;
}

pa_status plan_prefill(int32_t T, int32_t B, int32_t Hq, int32_t max_q_len, int32_t max_context_len,
                       const pa_cache_desc* d, int32_t split_tokens, PrefillPlan* plan) {
  const int64_t G = Hq / d->num_kv_heads;
  const int64_t nblk_max = max_context_len <= 0 ? 1 : (max_context_len + PA_BLOCK_SIZE - 1) / PA_BLOCK_SIZE;
  if (split_tokens > 0 && (split_tokens % PA_BLOCK_SIZE || split_tokens > 4096))
    return fail(PA_ERR_INVALID, "split_tokens must be a multiple of 16 in [16, 4096]");
  // the decode kernel's partitions: the call's split up to 1024 tokens, else
  // the library's choice
  const int32_t dsplit = split_tokens > 0 ? std::min<int32_t>(split_tokens, 1024) : 0;
  // Short queries over a 16-bit cache -- decode steps sent through this
  // call, a speculative verification of one or two draft tokens -- would
  // leave most of a 64-row tile empty.  The decode kernel serves them
  // instead: one grid column per (sequence, kv head, query token), the G
  // heads of the token as MMA columns, the columns of one (sequence, kv
  // head) side by side so that their reads of the same K/V tiles meet in L2.
  // Each column streams the tiles again from L2, so the route pays only up
  // to half a tile of rows (32): at 5 tokens x 8 heads the 64-row kernel is
  // as fast, and over 1-byte caches, where every column would convert the
  // codes again, it is faster.
  if (prefill_routes_short(max_q_len, Hq, d)) {
    if (static_cast<int64_t>(B) * max_q_len * d->num_kv_heads > INT32_MAX)
      return fail(PA_ERR_UNSUPPORTED, "too many query rows for one grid");
    pa_status st = plan_decode(B * max_q_len, Hq, max_context_len, d, dsplit, &plan->dec);
    if (st != PA_OK) return st;
    plan->route_short = 1;
    plan->route_single = 0;
    plan->tc = 0;
    plan->row_tiles = 1;
    plan->blocks_per_part = plan->dec.blocks_per_part;
    plan->max_parts = plan->dec.max_parts;
    plan->workspace_bytes = plan->dec.workspace_bytes;
    plan->dec_offset = 0;
    return PA_OK;
  }
  // Rows of one (sequence, kv head) are (query token, head of the group)
  // pairs.  More than 64 of them at head_dim 128 run the tcgen05 kernel
  // (128-row tiles); otherwise the mma.sync kernel (64-row tiles) wastes less
  // of its tile.  Two CTAs per SM either way.
  const int64_t tile_rows = prefill_uses_tc(max_q_len, Hq, d) ? 128 : 64;
  const int64_t tiles = max_q_len <= 0 ? 1 : (static_cast<int64_t>(max_q_len) * G + tile_rows - 1) / tile_rows;
  int64_t bpp;
  if (split_tokens > 0) {
    bpp = split_tokens / PA_BLOCK_SIZE;
  } else {
    // Row tiles that can hold rows: at most one partial tile per sequence
    // beyond the T * G / 64 full ones.  With eight or more such tiles per SM
    // the grid is full without splitting the context (a split costs partial
    // rows written and merged); otherwise 1024-token partitions, halved
    // while the grid would give fewer than four CTAs per SM.
    const int64_t units = d->num_kv_heads * std::min<int64_t>(static_cast<int64_t>(B) * tiles,
                                                             (static_cast<int64_t>(T) * G + tile_rows - 1) / tile_rows + B);
    const int64_t sms = sm_count();
    const int64_t per_sm = 2;  // resident CTAs per SM (both kernels)
    if (units >= 4 * per_sm * sms) {
      bpp = std::max<int64_t>(nblk_max, 1);
    } else {
      bpp = 64;
      while (bpp > 8 && units * ((nblk_max + bpp - 1) / bpp) < 2 * per_sm * sms) bpp /= 2;
    }
  }
  // the tcgen05 kernel stages a partition's block ids in shared memory: at
  // most 1024 blocks (16K tokens) per partition
  if (tile_rows == 128 && bpp > 1024) bpp = 1024;
  const int64_t parts = (nblk_max + bpp - 1) / bpp;
  if (parts > 65535) return fail(PA_ERR_UNSUPPORTED, "context too long for the partition grid");
  if (static_cast<int64_t>(B) * d->num_kv_heads * tiles > INT32_MAX)
    return fail(PA_ERR_UNSUPPORTED, "too many row tiles for one grid");
  plan->tc = tile_rows == 128 ? 1 : 0;
  plan->row_tiles = static_cast<int32_t>(tiles);
  plan->blocks_per_part = static_cast<int32_t>(bpp);
  plan->max_parts = static_cast<int32_t>(parts);
  if (parts > 1) {
    const size_t rows = static_cast<size_t>(T) * Hq * parts;
    size_t bytes = rows * d->head_dim * sizeof(float) + 2 * rows * sizeof(float);
    plan->workspace_bytes = (bytes + 255) & ~static_cast<size_t>(255);
  } else {
    plan->workspace_bytes = 0;
  }
  // A decode step riding in the call would fill one row of a multi-token
  // tile: those one-token sequences go to the decode kernel, whose workspace
  // follows.  It runs on a second stream beside the multi-token grid, whose
  // last wave leaves SMs to it.
  plan->route_single = 1;
  plan->dec_offset = plan->workspace_bytes;
  if (plan->route_single) {
    pa_status st = plan_decode(B, Hq, max_context_len, d, dsplit, &plan->dec);
    if (st != PA_OK) return st;
    plan->workspace_bytes += plan->dec.workspace_bytes;
  }
  return PA_OK;
}

}  // namespace pa

using pa::fail;

extern "C" {

const char* pa_last_error(void) { return pa::g_last_error.c_str(); }

int32_t pa_version(void) { return 100; }

pa_status pa_cache_write(const void* k, const void* v, int32_t in_dtype,
                         const int64_t* slot_mapping, int64_t num_tokens, void* k_cache,
                         void* v_cache, float* k_scale, float* v_scale, const pa_cache_desc* desc,
                         void* stream) {
  pa_status st = pa::check_desc(desc, "pa_cache_write");
  if (st != PA_OK) return st;
  if (num_tokens < 0) return fail(PA_ERR_INVALID, "pa_cache_write: num_tokens < 0");
  if (num_tokens == 0) return PA_OK;
  if (num_tokens > INT32_MAX) return fail(PA_ERR_INVALID, "pa_cache_write: too many tokens");
  if (!k || !v || !slot_mapping || !k_cache || !v_cache)
    return fail(PA_ERR_INVALID, "pa_cache_write: null pointer");
  if (!pa::aligned16(k) || !pa::aligned16(v) || !pa::aligned16(k_cache) || !pa::aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return fail(PA_ERR_INVALID, "pa_cache_write: misaligned pointer");
  const bool q8 = pa::quantised(desc->kv_dtype);
  if (q8) {
    if (in_dtype != PA_DTYPE_F16 && in_dtype != PA_DTYPE_BF16 && in_dtype != PA_DTYPE_F32)
      return fail(PA_ERR_INVALID, "pa_cache_write: FP8 / INT8 cache needs F16, BF16 or F32 input");
    if (!k_scale || !v_scale || !pa::aligned16(k_scale) || !pa::aligned16(v_scale))
      return fail(PA_ERR_INVALID, "pa_cache_write: FP8 / INT8 cache needs 16-byte aligned scales");
  } else {
    if (in_dtype != desc->kv_dtype && in_dtype != PA_DTYPE_F32)
      return fail(PA_ERR_INVALID, "pa_cache_write: in_dtype must equal kv_dtype or be F32");
    if (k_scale || v_scale)
      return fail(PA_ERR_INVALID, "pa_cache_write: scales are only for FP8 / INT8 caches");
  }
  return pa::launch_cache_write(k, v, in_dtype, slot_mapping, num_tokens, k_cache, v_cache,
                                k_scale, v_scale, desc, stream);
}

size_t pa_decode_workspace_size(int32_t B, int32_t num_q_heads, int32_t max_context_len,
                                const pa_cache_desc* desc, int32_t split_tokens) {
  if (pa::check_desc(desc, "pa_decode_workspace_size") != PA_OK || B < 0 || num_q_heads <= 0)
    return 0;
  pa::DecodePlan plan;
  if (pa::plan_decode(B, num_q_heads, max_context_len, desc, split_tokens, &plan) != PA_OK)
    return 0;
  return plan.workspace_bytes;
}

// Kernels a decode call with this plan launches: the main kernel, and the
// merge kernel unless one partition covers the context or the main kernel
// merges its partitions itself.
static int32_t decode_kernels(const pa::DecodePlan& plan) {
  return 1 + (plan.max_parts > 1 && plan.ticket_offset == 0 ? 1 : 0);
}

pa_status pa_decode_plan_info(int32_t B, int32_t num_q_heads, int32_t max_context_len,
                              const pa_cache_desc* desc, int32_t split_tokens, int32_t* partitions,
                              int32_t* blocks_per_partition, int32_t* kernels) {
  pa_status st = pa::check_desc(desc, "pa_decode_plan_info");
  if (st != PA_OK) return st;
  if (B < 0 || num_q_heads <= 0 || max_context_len < 0)
    return fail(PA_ERR_INVALID, "pa_decode_plan_info: B, num_q_heads or max_context_len out of range");
  pa::DecodePlan plan;
  st = pa::plan_decode(B, num_q_heads, max_context_len, desc, split_tokens, &plan);
  if (st != PA_OK) return st;
  if (partitions) *partitions = plan.max_parts;
  if (blocks_per_partition) *blocks_per_partition = plan.blocks_per_part;
  if (kernels) *kernels = decode_kernels(plan);
  return PA_OK;
}

// Whether a batch's decode runs faster over a host-planned list of its live
// partitions (pa_decode_append_segments with one-member groups) than over the
// fixed (sequence, kv head, partition) grid, judged from the context lengths
// the block manager holds on the host.  The fixed grid has B x max_parts
// cells per kv head; a sequence fills ceil(blocks / blocks_per_partition) of
// them and the rest exit at once.  Measured (GB300): with 28 % of the cells
// live (64 sequences, lengths log-uniform in 16..4096) the list is 6 %
// faster; with 62 % (uniform 1..2048) and 75 % (16K..32K) it is as fast or
// slower.  So: the list when fewer than half the cells are live, more than
// one partition, and G <= 8 (a member's query heads are one MMA's columns).
pa_status pa_decode_items_plan(const int32_t* context_lens, int32_t B, int32_t num_q_heads,
                               int32_t max_context_len, const pa_cache_desc* desc, int32_t split_tokens,
                               int32_t* use_items, int32_t* blocks_per_item, int32_t* max_items_per_seq) {
  pa_status st = pa::check_desc(desc, "pa_decode_items_plan");
  if (st != PA_OK) return st;
  if (!context_lens || !use_items || B <= 0 || num_q_heads <= 0 || max_context_len < 0)
    return fail(PA_ERR_INVALID, "pa_decode_items_plan: null pointer, B, num_q_heads or max_context_len out of range");
  pa::DecodePlan plan;
  st = pa::plan_decode(B, num_q_heads, max_context_len, desc, split_tokens, &plan);
  if (st != PA_OK) return st;
  const int64_t bpp = plan.blocks_per_part;
  int64_t live = 0;
  for (int32_t b = 0; b < B; ++b) {
    const int32_t L = context_lens[b];
    if (L < 0 || L > max_context_len)
      return fail(PA_ERR_INVALID, "pa_decode_items_plan: context length %d of sequence %d outside 0..%d", L, b,
                  max_context_len);
    live += ((L + PA_BLOCK_SIZE - 1) / PA_BLOCK_SIZE + bpp - 1) / bpp;
  }
  const int64_t cells = static_cast<int64_t>(B) * plan.max_parts;
  const int64_t G = num_q_heads / desc->num_kv_heads;
  *use_items = plan.max_parts > 1 && G <= 8 && 2 * live < cells && plan.max_parts <= 65535 ? 1 : 0;
  if (blocks_per_item) *blocks_per_item = static_cast<int32_t>(std::min<int64_t>(bpp, 64));
  if (max_items_per_seq) {
    const int64_t nblk_max = (max_context_len + PA_BLOCK_SIZE - 1) / PA_BLOCK_SIZE;
    *max_items_per_seq = static_cast<int32_t>(std::max<int64_t>(1, (nblk_max + bpp - 1) / bpp));
  }
  return PA_OK;
}

// Shared-prefix groups of a grouped decode call (none: n_groups == 0).
struct Groups {
  const int32_t* start = nullptr;
  const int32_t* prefix = nullptr;
  int32_t n = 0, max_size = 0, max_prefix = 0;
  // segment items instead of prefixes (pa_decode_append_segments)
  const int32_t* items = nullptr;
  int32_t n_items = 0, max_items = 0;
};

// The segment grid: one CTA per (item, kv head); each member's partials
// take max_items slots (the items of its group); a merge kernel follows.
static pa_status plan_segments(int32_t B, int32_t Hq, const pa_cache_desc* d, const Groups& gr,
                               pa::DecodePlan* plan) {
  if (gr.n <= 0 || gr.n > B || gr.max_size <= 0 || gr.max_size > 8 || gr.n_items < 0 || gr.n_items > 65535 ||
      gr.max_items <= 0 || gr.max_items > 65535)
    return fail(PA_ERR_INVALID, "pa_decode_append_segments: n_groups, max_group_size, n_items or max_group_items "
                                "out of range");
  if (static_cast<int64_t>(gr.max_size) * (Hq / d->num_kv_heads) > 8)
    return fail(PA_ERR_UNSUPPORTED, "pa_decode_append_segments: max_group_size * G above 8 query columns");
  plan->ticket_offset = 0;  // merged by decode_reduce_segments
  plan->pre_parts = plan->tail_parts = 0;
  plan->max_parts = gr.max_items;
  const size_t rows = static_cast<size_t>(B) * Hq * gr.max_items;
  const size_t bytes = rows * d->head_dim * sizeof(float) + 2 * rows * sizeof(float);
  plan->workspace_bytes = (bytes + 255) & ~static_cast<size_t>(255);
  return PA_OK;
}

// The grouped grid's partition counts on top of the plain plan: prefix
// partitions of the longest allowed shared prefix, tail partitions of the
// longest context; every member's rows are partials.
static pa_status plan_grouped(int32_t B, int32_t Hq, int32_t max_context_len, const pa_cache_desc* d,
                              const Groups& gr, pa::DecodePlan* plan) {
  if (gr.n <= 0 || gr.n > B || gr.max_size <= 0 || gr.max_size > B || gr.max_prefix < 0)
    return fail(PA_ERR_INVALID, "pa_decode_append_grouped: n_groups, max_group_size or max_prefix_blocks out of range");
  if (static_cast<int64_t>(gr.max_size) * (Hq / d->num_kv_heads) > 8)
    return fail(PA_ERR_UNSUPPORTED, "pa_decode_append_grouped: max_group_size * G above 8 query columns");
  const int64_t nblk_max = max_context_len <= 0 ? 1 : (max_context_len + PA_BLOCK_SIZE - 1) / PA_BLOCK_SIZE;
  const int64_t bpp = plan->blocks_per_part;
  const int64_t pre = (std::min<int64_t>(gr.max_prefix, nblk_max) + bpp - 1) / bpp;
  const int64_t tail = (nblk_max + bpp - 1) / bpp;
  if (pre + static_cast<int64_t>(gr.max_size) * tail > 65535 ||
      static_cast<int64_t>(gr.n) * d->num_kv_heads * gr.max_size > (int64_t{1} << 31) - 1)
    return fail(PA_ERR_UNSUPPORTED, "pa_decode_append_grouped: grid too large");
  plan->ticket_offset = 0;  // groups merge in decode_reduce_grouped
  plan->pre_parts = static_cast<int32_t>(pre);
  plan->tail_parts = static_cast<int32_t>(tail);
  plan->max_parts = static_cast<int32_t>(pre + tail);
  const size_t rows = static_cast<size_t>(B) * Hq * plan->max_parts;
  const size_t bytes = rows * d->head_dim * sizeof(float) + 2 * rows * sizeof(float);
  plan->workspace_bytes = (bytes + 255) & ~static_cast<size_t>(255);
  return PA_OK;
}

static pa_status decode_impl(const void* q, int32_t q_dtype, const void* k_cache, const void* v_cache,
                             const float* k_scale, const float* v_scale, const int32_t* block_tables,
                             int32_t max_blocks_per_seq, const int32_t* context_lens,
                             int32_t max_context_len, int32_t B, int32_t num_q_heads, float scale,
                             void* out, int32_t out_dtype, const pa_cache_desc* desc, void* workspace,
                             size_t workspace_bytes, int32_t split_tokens, void* stream,
                             const void* k_new, const void* v_new, int32_t new_dtype,
                             const int64_t* slot_mapping, const Groups& gr = Groups()) {
  pa_status st = pa::check_desc(desc, "pa_decode");
  if (st != PA_OK) return st;
  if (B < 0 || num_q_heads <= 0 || max_blocks_per_seq <= 0 || max_context_len < 0)
    return fail(PA_ERR_INVALID, "pa_decode: B, num_q_heads, max_blocks_per_seq, max_context_len out of range");
  if (num_q_heads % desc->num_kv_heads)
    return fail(PA_ERR_INVALID, "pa_decode: num_q_heads must be a multiple of num_kv_heads");
  if (num_q_heads / desc->num_kv_heads > PA_MAX_GROUP)
    return fail(PA_ERR_UNSUPPORTED, "pa_decode: more than %d query heads per kv head", PA_MAX_GROUP);
  if (!std::isfinite(scale)) return fail(PA_ERR_INVALID, "pa_decode: scale is not finite");
  const bool q8 = pa::quantised(desc->kv_dtype);
  if (q8) {
    if (q_dtype != PA_DTYPE_F16 && q_dtype != PA_DTYPE_BF16)
      return fail(PA_ERR_INVALID, "pa_decode: q_dtype must be F16 or BF16 for an FP8 / INT8 cache");
    if (!k_scale || !v_scale || !pa::aligned16(k_scale) || !pa::aligned16(v_scale))
      return fail(PA_ERR_INVALID, "pa_decode: FP8 / INT8 cache needs 16-byte aligned scales");
  } else {
    if (q_dtype != desc->kv_dtype)
      return fail(PA_ERR_INVALID, "pa_decode: q_dtype must equal kv_dtype");
    if (k_scale || v_scale) return fail(PA_ERR_INVALID, "pa_decode: scales are only for FP8 / INT8 caches");
  }
  if (out_dtype != q_dtype && out_dtype != PA_DTYPE_F32)
    return fail(PA_ERR_INVALID, "pa_decode: out_dtype must be q_dtype or F32");
  if (B == 0) return PA_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out)
    return fail(PA_ERR_INVALID, "pa_decode: null pointer");
  if (!pa::aligned16(q) || !pa::aligned16(k_cache) || !pa::aligned16(v_cache) ||
      !pa::aligned16(out) || (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
      (reinterpret_cast<uintptr_t>(context_lens) & 3u))
    return fail(PA_ERR_INVALID, "pa_decode: misaligned pointer");
  pa::DecodePlan plan;
  st = pa::plan_decode(B, num_q_heads, max_context_len, desc, split_tokens, &plan);
  if (st != PA_OK) return st;
  if (gr.n > 0 && gr.max_items > 0) {
    if (!gr.start || (gr.n_items > 0 && !gr.items) || (reinterpret_cast<uintptr_t>(gr.start) & 3u) ||
        (reinterpret_cast<uintptr_t>(gr.items) & 15u))
      return fail(PA_ERR_INVALID, "pa_decode_append_segments: group_start / items NULL or misaligned");
    st = plan_segments(B, num_q_heads, desc, gr, &plan);
    if (st != PA_OK) return st;
  } else if (gr.n > 0) {
    if (!gr.start || !gr.prefix || (reinterpret_cast<uintptr_t>(gr.start) & 3u) ||
        (reinterpret_cast<uintptr_t>(gr.prefix) & 3u))
      return fail(PA_ERR_INVALID, "pa_decode_append_grouped: group_start / prefix_blocks NULL or misaligned");
    st = plan_grouped(B, num_q_heads, max_context_len, desc, gr, &plan);
    if (st != PA_OK) return st;
  }
  if (plan.workspace_bytes) {
    if (!workspace || !pa::aligned16(workspace))
      return fail(PA_ERR_INVALID, "pa_decode: workspace NULL or misaligned (%zu bytes needed)",
                  plan.workspace_bytes);
    if (workspace_bytes < plan.workspace_bytes)
      return fail(PA_ERR_INVALID, "pa_decode: workspace has %zu bytes, %zu needed", workspace_bytes,
                  plan.workspace_bytes);
  }
  pa::DecodeLaunch a;
  a.q = q;
  a.q_dtype = q_dtype;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.block_tables = block_tables;
  a.max_blocks = max_blocks_per_seq;
  a.context_lens = context_lens;
  a.max_context_len = max_context_len;
  a.B = B;
  a.Hq = num_q_heads;
  a.Hkv = desc->num_kv_heads;
  a.D = desc->head_dim;
  a.num_blocks = desc->num_blocks;
  a.kv_dtype = desc->kv_dtype;
  a.scale = scale;
  a.out = out;
  a.out_dtype = out_dtype;
  a.workspace = workspace;
  a.plan = plan;
  if (slot_mapping) {
    if (!k_new || !v_new) return fail(PA_ERR_INVALID, "pa_decode_append: k_new / v_new is NULL");
    if (!pa::aligned16(k_new) || !pa::aligned16(v_new) || (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
      return fail(PA_ERR_INVALID, "pa_decode_append: misaligned pointer");
    if (q8 ? (new_dtype != PA_DTYPE_F16 && new_dtype != PA_DTYPE_BF16 && new_dtype != PA_DTYPE_F32)
            : (new_dtype != desc->kv_dtype && new_dtype != PA_DTYPE_F32))
      return fail(PA_ERR_INVALID, "pa_decode_append: new_dtype does not match the cache");
    a.k_new = k_new;
    a.v_new = v_new;
    a.slot_mapping = slot_mapping;
    a.new_dtype = new_dtype;
  }
  a.group_start = gr.start;
  a.prefix_blocks = gr.prefix;
  a.n_groups = gr.n;
  a.max_members = gr.max_size;
  a.segments = gr.max_items > 0 ? 1 : 0;
  a.seg_items = gr.items;
  a.n_seg_items = gr.n_items;
  return pa::launch_decode(a, stream);
}

pa_status pa_decode(const void* q, int32_t q_dtype, const void* k_cache, const void* v_cache,
                    const float* k_scale, const float* v_scale, const int32_t* block_tables,
                    int32_t max_blocks_per_seq, const int32_t* context_lens,
                    int32_t max_context_len, int32_t B, int32_t num_q_heads, float scale,
                    void* out, int32_t out_dtype, const pa_cache_desc* desc, void* workspace,
                    size_t workspace_bytes, int32_t split_tokens, void* stream) {
  return decode_impl(q, q_dtype, k_cache, v_cache, k_scale, v_scale, block_tables, max_blocks_per_seq,
                     context_lens, max_context_len, B, num_q_heads, scale, out, out_dtype, desc, workspace,
                     workspace_bytes, split_tokens, stream, nullptr, nullptr, 0, nullptr);
}

pa_status pa_decode_append(const void* k_new, const void* v_new, int32_t new_dtype,
                           const int64_t* slot_mapping, const void* q, int32_t q_dtype, void* k_cache,
                           void* v_cache, float* k_scale, float* v_scale, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* context_lens,
                           int32_t max_context_len, int32_t B, int32_t num_q_heads, float scale,
                           void* out, int32_t out_dtype, const pa_cache_desc* desc, void* workspace,
                           size_t workspace_bytes, int32_t split_tokens, void* stream) {
  if (!slot_mapping) return fail(PA_ERR_INVALID, "pa_decode_append: slot_mapping is NULL");
  return decode_impl(q, q_dtype, k_cache, v_cache, k_scale, v_scale, block_tables, max_blocks_per_seq,
                     context_lens, max_context_len, B, num_q_heads, scale, out, out_dtype, desc, workspace,
                     workspace_bytes, split_tokens, stream, k_new, v_new, new_dtype, slot_mapping);
}

size_t pa_decode_grouped_workspace_size(int32_t B, int32_t num_q_heads, int32_t max_context_len,
                                        int32_t n_groups, int32_t max_group_size, int32_t max_prefix_blocks,
                                        const pa_cache_desc* desc, int32_t split_tokens) {
  if (pa::check_desc(desc, "pa_decode_grouped_workspace_size") != PA_OK || B <= 0 || num_q_heads <= 0 ||
      num_q_heads % desc->num_kv_heads)
    return 0;
  pa::DecodePlan plan;
  if (pa::plan_decode(B, num_q_heads, max_context_len, desc, split_tokens, &plan) != PA_OK) return 0;
  Groups gr;
  gr.n = n_groups;
  gr.max_size = max_group_size;
  gr.max_prefix = max_prefix_blocks;
  if (plan_grouped(B, num_q_heads, max_context_len, desc, gr, &plan) != PA_OK) return 0;
  return plan.workspace_bytes;
}

pa_status pa_decode_append_grouped(const void* k_new, const void* v_new, int32_t new_dtype,
                                   const int64_t* slot_mapping, const void* q, int32_t q_dtype, void* k_cache,
                                   void* v_cache, float* k_scale, float* v_scale, const int32_t* block_tables,
                                   int32_t max_blocks_per_seq, const int32_t* context_lens,
                                   int32_t max_context_len, int32_t B, int32_t num_q_heads, float scale,
                                   const int32_t* group_start, const int32_t* prefix_blocks, int32_t n_groups,
                                   int32_t max_group_size, int32_t max_prefix_blocks, void* out,
                                   int32_t out_dtype, const pa_cache_desc* desc, void* workspace,
                                   size_t workspace_bytes, int32_t split_tokens, void* stream) {
  if (!slot_mapping) return fail(PA_ERR_INVALID, "pa_decode_append_grouped: slot_mapping is NULL");
  if (B <= 0) return B == 0 ? PA_OK : fail(PA_ERR_INVALID, "pa_decode_append_grouped: B < 0");
  Groups gr;
  gr.start = group_start;
  gr.prefix = prefix_blocks;
  gr.n = n_groups;
  gr.max_size = max_group_size;
  gr.max_prefix = max_prefix_blocks;
  if (n_groups <= 0) return fail(PA_ERR_INVALID, "pa_decode_append_grouped: n_groups must be > 0");
  return decode_impl(q, q_dtype, k_cache, v_cache, k_scale, v_scale, block_tables, max_blocks_per_seq,
                     context_lens, max_context_len, B, num_q_heads, scale, out, out_dtype, desc, workspace,
                     workspace_bytes, split_tokens, stream, k_new, v_new, new_dtype, slot_mapping, gr);
}

size_t pa_decode_segments_workspace_size(int32_t B, int32_t num_q_heads, int32_t n_groups, int32_t max_group_size,
                                         int32_t max_group_items, const pa_cache_desc* desc) {
  if (pa::check_desc(desc, "pa_decode_segments_workspace_size") != PA_OK || B <= 0 || num_q_heads <= 0 ||
      num_q_heads % desc->num_kv_heads)
    return 0;
  pa::DecodePlan plan;
  if (pa::plan_decode(B, num_q_heads, 0, desc, 0, &plan) != PA_OK) return 0;
  Groups gr;
  gr.n = n_groups;
  gr.max_size = max_group_size;
  gr.max_items = max_group_items;
  if (plan_segments(B, num_q_heads, desc, gr, &plan) != PA_OK) return 0;
  return plan.workspace_bytes;
}

pa_status pa_decode_append_segments(const void* k_new, const void* v_new, int32_t new_dtype,
                                    const int64_t* slot_mapping, const void* q, int32_t q_dtype, void* k_cache,
                                    void* v_cache, float* k_scale, float* v_scale, const int32_t* block_tables,
                                    int32_t max_blocks_per_seq, const int32_t* context_lens,
                                    int32_t max_context_len, int32_t B, int32_t num_q_heads, float scale,
                                    const int32_t* group_start, int32_t n_groups, int32_t max_group_size,
                                    const int32_t* items, int32_t n_items, int32_t max_group_items, void* out,
                                    int32_t out_dtype,
                                    const pa_cache_desc* desc, void* workspace, size_t workspace_bytes,
                                    void* stream) {
  if (!slot_mapping) return fail(PA_ERR_INVALID, "pa_decode_append_segments: slot_mapping is NULL");
  if (B <= 0) return B == 0 ? PA_OK : fail(PA_ERR_INVALID, "pa_decode_append_segments: B < 0");
  if (n_groups <= 0 || max_group_items <= 0)
    return fail(PA_ERR_INVALID, "pa_decode_append_segments: n_groups and max_group_items must be > 0");
  Groups gr;
  gr.start = group_start;
  gr.n = n_groups;
  gr.max_size = max_group_size;
  gr.items = items;
  gr.n_items = n_items;
  gr.max_items = max_group_items;
  return decode_impl(q, q_dtype, k_cache, v_cache, k_scale, v_scale, block_tables, max_blocks_per_seq,
                     context_lens, max_context_len, B, num_q_heads, scale, out, out_dtype, desc, workspace,
                     workspace_bytes, 0, stream, k_new, v_new, new_dtype, slot_mapping, gr);
}

static pa_status check_prefill(int32_t T, int32_t B, int32_t num_q_heads, int32_t max_q_len,
                               int32_t max_context_len, const pa_cache_desc* desc) {
  pa_status st = pa::check_desc(desc, "pa_chunked_prefill");
  if (st != PA_OK) return st;
  if (T < 0 || B < 0 || num_q_heads <= 0 || max_q_len < 0 || max_context_len < 0)
    return fail(PA_ERR_INVALID, "pa_chunked_prefill: negative size or num_q_heads <= 0");
  if (T > 0 && max_q_len == 0) return fail(PA_ERR_INVALID, "pa_chunked_prefill: max_q_len is 0 with tokens");
  if (max_q_len > 65535) return fail(PA_ERR_UNSUPPORTED, "pa_chunked_prefill: max_q_len above 65535");
  if (num_q_heads % desc->num_kv_heads)
    return fail(PA_ERR_INVALID, "pa_chunked_prefill: num_q_heads must be a multiple of num_kv_heads");
  if (num_q_heads / desc->num_kv_heads > PA_MAX_GROUP)
    return fail(PA_ERR_UNSUPPORTED, "pa_chunked_prefill: more than %d query heads per kv head", PA_MAX_GROUP);
  return PA_OK;
}

pa_status pa_chunked_prefill_plan_info(int32_t num_tokens, int32_t B, int32_t num_q_heads, int32_t max_q_len,
                                       int32_t max_context_len, const pa_cache_desc* desc, int32_t split_tokens,
                                       int32_t* tensor_cores, int32_t* partitions,
                                       int32_t* blocks_per_partition, int32_t* kernels) {
  pa_status st = check_prefill(num_tokens, B, num_q_heads, max_q_len, max_context_len, desc);
  if (st != PA_OK) return st;
  pa::PrefillPlan plan;
  st = pa::plan_prefill(num_tokens, B, num_q_heads, max_q_len, max_context_len, desc, split_tokens, &plan);
  if (st != PA_OK) return st;
  if (tensor_cores) *tensor_cores = plan.tc;
  if (partitions) *partitions = plan.max_parts;
  if (blocks_per_partition) *blocks_per_partition = plan.blocks_per_part;
  if (kernels) {
    if (plan.route_short) {
      *kernels = decode_kernels(plan.dec);
    } else {
      const int32_t multi = max_q_len > 1 || !plan.route_single ? 1 + (plan.max_parts > 1 ? 1 : 0) : 0;
      *kernels = multi + (plan.route_single ? decode_kernels(plan.dec) : 0);
    }
  }
  return PA_OK;
}

size_t pa_chunked_prefill_workspace_size(int32_t num_tokens, int32_t B, int32_t num_q_heads,
                                         int32_t max_q_len, int32_t max_context_len,
                                         const pa_cache_desc* desc, int32_t split_tokens) {
  if (check_prefill(num_tokens, B, num_q_heads, max_q_len, max_context_len, desc) != PA_OK) return 0;
  pa::PrefillPlan plan;
  if (pa::plan_prefill(num_tokens, B, num_q_heads, max_q_len, max_context_len, desc, split_tokens, &plan) !=
      PA_OK)
    return 0;
  // A call with fewer query tokens per sequence may take the decode route,
  // whose workspace grows with B x tokens instead of num_tokens: cover those
  // plans too, so the size holds for every call up to these bounds.
  size_t bytes = plan.workspace_bytes;
  for (int32_t q = 1; q < max_q_len && q <= pa::kShortTokens; ++q) {
    if (!pa::prefill_routes_short(q, num_q_heads, desc)) continue;
    pa::PrefillPlan p2;
    if (pa::plan_prefill(num_tokens, B, num_q_heads, q, max_context_len, desc, split_tokens, &p2) == PA_OK)
      bytes = std::max(bytes, p2.workspace_bytes);
  }
  return bytes;
}

pa_status pa_chunked_prefill(const void* q, int32_t q_dtype, const int32_t* q_start, int32_t num_tokens,
                             int32_t max_q_len, const void* k_cache, const void* v_cache,
                             const float* k_scale, const float* v_scale,
                             const int32_t* block_tables, int32_t max_blocks_per_seq,
                             const int32_t* context_lens, int32_t max_context_len, int32_t B,
                             int32_t num_q_heads, float scale, void* out, int32_t out_dtype,
                             const pa_cache_desc* desc, void* workspace, size_t workspace_bytes,
                             int32_t split_tokens, void* stream) {
  pa_status st = check_prefill(num_tokens, B, num_q_heads, max_q_len, max_context_len, desc);
  if (st != PA_OK) return st;
  if (max_blocks_per_seq <= 0) return fail(PA_ERR_INVALID, "pa_chunked_prefill: max_blocks_per_seq <= 0");
  if (!std::isfinite(scale)) return fail(PA_ERR_INVALID, "pa_chunked_prefill: scale is not finite");
  const bool q8 = pa::quantised(desc->kv_dtype);
  if (q8) {
    if (q_dtype != PA_DTYPE_F16 && q_dtype != PA_DTYPE_BF16)
      return fail(PA_ERR_INVALID, "pa_chunked_prefill: q_dtype must be F16 or BF16 for an FP8 / INT8 cache");
    if (!k_scale || !v_scale || !pa::aligned16(k_scale) || !pa::aligned16(v_scale))
      return fail(PA_ERR_INVALID, "pa_chunked_prefill: FP8 / INT8 cache needs 16-byte aligned scales");
  } else {
    if (q_dtype != desc->kv_dtype)
      return fail(PA_ERR_INVALID, "pa_chunked_prefill: q_dtype must equal kv_dtype");
    if (k_scale || v_scale)
      return fail(PA_ERR_INVALID, "pa_chunked_prefill: scales are only for FP8 / INT8 caches");
  }
  if (out_dtype != q_dtype && out_dtype != PA_DTYPE_F32)
    return fail(PA_ERR_INVALID, "pa_chunked_prefill: out_dtype must be q_dtype or F32");
  if (B == 0 || num_tokens == 0) return PA_OK;
  if (!q || !q_start || !k_cache || !v_cache || !block_tables || !context_lens || !out)
    return fail(PA_ERR_INVALID, "pa_chunked_prefill: null pointer");
  if (!pa::aligned16(q) || !pa::aligned16(k_cache) || !pa::aligned16(v_cache) || !pa::aligned16(out) ||
      (reinterpret_cast<uintptr_t>(q_start) & 3u) || (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
      (reinterpret_cast<uintptr_t>(context_lens) & 3u))
    return fail(PA_ERR_INVALID, "pa_chunked_prefill: misaligned pointer");
  pa::PrefillPlan plan;
  st = pa::plan_prefill(num_tokens, B, num_q_heads, max_q_len, max_context_len, desc, split_tokens, &plan);
  if (st != PA_OK) return st;
  if (plan.workspace_bytes) {
    if (!workspace || !pa::aligned16(workspace))
      return fail(PA_ERR_INVALID, "pa_chunked_prefill: workspace NULL or misaligned (%zu bytes needed)",
                  plan.workspace_bytes);
    if (workspace_bytes < plan.workspace_bytes)
      return fail(PA_ERR_INVALID, "pa_chunked_prefill: workspace has %zu bytes, %zu needed", workspace_bytes,
                  plan.workspace_bytes);
  }
  pa::PrefillLaunch a;
  a.q = q;
  a.q_dtype = q_dtype;
  a.q_start = q_start;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.block_tables = block_tables;
  a.max_blocks = max_blocks_per_seq;
  a.context_lens = context_lens;
  a.max_context_len = max_context_len;
  a.max_q_len = max_q_len;
  a.B = B;
  a.T = num_tokens;
  a.Hq = num_q_heads;
  a.Hkv = desc->num_kv_heads;
  a.D = desc->head_dim;
  a.num_blocks = desc->num_blocks;
  a.kv_dtype = desc->kv_dtype;
  a.scale = scale;
  a.out = out;
  a.out_dtype = out_dtype;
  a.workspace = workspace;
  a.plan = plan;
  return pa::launch_prefill(a, stream);
}

pa_status pa_copy_blocks(void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                         const int64_t* pairs, int64_t num_pairs, const pa_cache_desc* desc,
                         void* stream) {
  pa_status st = pa::check_desc(desc, "pa_copy_blocks");
  if (st != PA_OK) return st;
  if (num_pairs < 0) return fail(PA_ERR_INVALID, "pa_copy_blocks: num_pairs < 0");
  if (num_pairs == 0) return PA_OK;
  if (num_pairs > 65535) return fail(PA_ERR_INVALID, "pa_copy_blocks: at most 65535 pairs per call");
  if (!k_cache || !v_cache || !pairs) return fail(PA_ERR_INVALID, "pa_copy_blocks: null pointer");
  if (!pa::aligned16(k_cache) || !pa::aligned16(v_cache) || (reinterpret_cast<uintptr_t>(pairs) & 7u))
    return fail(PA_ERR_INVALID, "pa_copy_blocks: misaligned pointer");
  const bool q8 = pa::quantised(desc->kv_dtype);
  if (q8 && (!k_scale || !v_scale))
    return fail(PA_ERR_INVALID, "pa_copy_blocks: FP8 / INT8 cache needs scales");
  if (!q8 && (k_scale || v_scale))
    return fail(PA_ERR_INVALID, "pa_copy_blocks: scales are only for FP8 / INT8 caches");
  return pa::launch_copy_blocks(k_cache, v_cache, k_scale, v_scale, pairs, num_pairs, desc, stream);
}

pa_status pa_swap_blocks(void* dst_k, void* dst_v, float* dst_k_scale, float* dst_v_scale,
                         int32_t dst_num_blocks, const void* src_k, const void* src_v,
                         const float* src_k_scale, const float* src_v_scale, int32_t src_num_blocks,
                         const int64_t* pairs, int64_t num_pairs, const pa_cache_desc* desc,
                         void* stream) {
  pa_status st = pa::check_desc(desc, "pa_swap_blocks");
  if (st != PA_OK) return st;
  if (num_pairs < 0) return fail(PA_ERR_INVALID, "pa_swap_blocks: num_pairs < 0");
  if (num_pairs == 0) return PA_OK;
  if (num_pairs > 65535) return fail(PA_ERR_INVALID, "pa_swap_blocks: at most 65535 pairs per call");
  if (dst_num_blocks <= 0 || src_num_blocks <= 0)
    return fail(PA_ERR_INVALID, "pa_swap_blocks: pool sizes must be > 0");
  if (!dst_k || !dst_v || !src_k || !src_v || !pairs)
    return fail(PA_ERR_INVALID, "pa_swap_blocks: null pointer");
  if (!pa::aligned16(dst_k) || !pa::aligned16(dst_v) || !pa::aligned16(src_k) || !pa::aligned16(src_v) ||
      (reinterpret_cast<uintptr_t>(pairs) & 7u))
    return fail(PA_ERR_INVALID, "pa_swap_blocks: misaligned pointer");
  const bool q8 = pa::quantised(desc->kv_dtype);
  if (q8 != (dst_k_scale && dst_v_scale && src_k_scale && src_v_scale))
    return fail(PA_ERR_INVALID, "pa_swap_blocks: FP8 / INT8 pools need all four scale arrays, others none");
  if (!q8 && (dst_k_scale || dst_v_scale || src_k_scale || src_v_scale))
    return fail(PA_ERR_INVALID, "pa_swap_blocks: scales are only for FP8 / INT8 pools");
  return pa::launch_swap_blocks(dst_k, dst_v, dst_k_scale, dst_v_scale, dst_num_blocks, src_k, src_v,
                                src_k_scale, src_v_scale, src_num_blocks, pairs, num_pairs, desc, stream);
}

pa_status pa_device_errors(uint32_t* flags, int32_t clear) {
  if (!flags) return fail(PA_ERR_INVALID, "pa_device_errors: flags is NULL");
  uint32_t a = 0, b = 0, c = 0;
  pa_status st = pa::read_errors_decode(&a, clear != 0);
  if (st != PA_OK) return st;
  st = pa::read_errors_cache_ops(&b, clear != 0);
  if (st != PA_OK) return st;
  st = pa::read_errors_prefill(&c, clear != 0);
  if (st != PA_OK) return st;
  *flags = a | b | c;
  return PA_OK;
}

}  // extern "C"
