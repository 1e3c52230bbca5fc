// Internal host-side declarations shared by the C-ABI layer and the kernels.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <utility>

#include <cuda_runtime.h>

#include "../../include/pagedkv.h"

namespace pa {

// Record `msg` as the calling thread's last error and return `st`.
pa_status fail(pa_status st, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
inline pa_status ok() { return PA_OK; }

// Element size in bytes of a pa_dtype (0 for an unknown value).
inline int dtype_bytes(int32_t dt) {
  switch (dt) {
    case PA_DTYPE_F16:
    case PA_DTYPE_BF16: return 2;
    case PA_DTYPE_FP8_E4M3:
    case PA_DTYPE_INT8: return 1;
    case PA_DTYPE_F32: return 4;
    default: return 0;
  }
}

// Caches of 1-byte codes with per-token scale rows (FP8 E4M3, INT8).
inline bool quantised(int32_t dt) { return dt == PA_DTYPE_FP8_E4M3 || dt == PA_DTYPE_INT8; }

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Split-K plan for one pa_decode shape (pure function of its arguments and
// the device's SM count).
struct DecodePlan {
  int32_t blocks_per_part;  // 16-token blocks per partition
  int32_t max_parts;        // partitions of the longest allowed context
  size_t workspace_bytes;   // 0 when max_parts == 1
  int32_t item_warps;       // warps sharing one partition (1, 2 or 4)
  // shared-prefix groups: grid rows of prefix partitions and of tail
  // partitions per member (max_parts = pre_parts + tail_parts); 0 otherwise
  int32_t pre_parts = 0, tail_parts = 0;
  // plain grid with max_parts > 1: the split-K partials are merged inside the
  // decode kernel by the last partition of each (sequence, kv head) to
  // finish; their arrival counters start at this byte of the workspace
  // (0: no counters, a merge kernel runs instead)
  size_t ticket_offset = 0;
};
pa_status plan_decode(int32_t B, int32_t num_q_heads, int32_t max_context_len,
                      const pa_cache_desc* desc, int32_t split_tokens, DecodePlan* plan);

// Arguments of the decode launch after host validation.
struct DecodeLaunch {
  const void* q;
  int32_t q_dtype;
  const void* k_cache;
  const void* v_cache;
  const float* k_scale;
  const float* v_scale;
  const int32_t* block_tables;
  int32_t max_blocks;
  const int32_t* context_lens;
  int32_t max_context_len;
  int32_t B, Hq, Hkv, D, num_blocks, kv_dtype;
  float scale;
  void* out;
  int32_t out_dtype;
  void* workspace;
  DecodePlan plan;
  // fused cache write of this step's token (pa_decode_append), else null
  const void* k_new = nullptr;
  const void* v_new = nullptr;
  const int64_t* slot_mapping = nullptr;
  int32_t new_dtype = 0;
  // shared-prefix groups (pa_decode_append_grouped), else n_groups == 0
  const int32_t* group_start = nullptr;
  const int32_t* prefix_blocks = nullptr;
  int32_t n_groups = 0, max_members = 0;
  // segments of groups (pa_decode_append_segments): int32 [n_seg_items][4]
  // items
  int32_t segments = 0;
  const int32_t* seg_items = nullptr;
  int32_t n_seg_items = 0;
  // rows of a multi-token call (pa_chunked_prefill): sequence b's n_b query
  // tokens are rows q_start[b] .. of q_rows, one grid column per token up to
  // q_tokens; longer sequences are skipped (left to the multi-token kernel)
  // unless q_report, when they are flagged as out of range
  const int32_t* q_start = nullptr;
  int32_t q_rows = 0;
  int32_t q_tokens = 1;
  int32_t q_report = 0;
};
pa_status launch_decode(const DecodeLaunch& a, void* stream);

// Split-K plan for one pa_chunked_prefill shape.
struct PrefillPlan {
  int32_t tc;               // 1: tcgen05 kernel with 128-row tiles; 0: mma.sync, 64-row tiles
  int32_t row_tiles;        // row tiles per (sequence, kv head) for max_q_len
  int32_t blocks_per_part;  // 16-token blocks per partition
  int32_t max_parts;        // partitions of the longest allowed context
  size_t workspace_bytes;   // 0 when max_parts == 1 and no one-token routing
  // one-token sequences of the call go to the decode kernel (on a side
  // stream when the call also has longer ones), with plan dec, its
  // workspace at byte dec_offset
  int32_t route_single = 0;
  // short queries over a 16-bit cache (at most kShortTokens per sequence and
  // 32 rows per kv head): the decode kernel serves the whole call, one grid
  // column per query token (plan dec for B x max_q_len rows, workspace at
  // byte 0)
  int32_t route_short = 0;
  DecodePlan dec;
  size_t dec_offset = 0;
};
constexpr int32_t kShortTokens = 8;
// Whether pa_chunked_prefill runs its tcgen05 kernel (128-row tiles) for
// this shape: head_dim 128 and more than 64 rows per (sequence, kv head).
// 1-byte caches too: their codes are converted to 16-bit in shared memory.
#ifndef PA_TC_MIN_ROWS
#define PA_TC_MIN_ROWS 64
#endif
inline bool prefill_uses_tc(int32_t max_q_len, int32_t num_q_heads, const pa_cache_desc* d) {
  return d->head_dim == 128 &&
         static_cast<int64_t>(max_q_len) * (num_q_heads / d->num_kv_heads) > PA_TC_MIN_ROWS;
}
// Whether pa_chunked_prefill sends the whole call to the decode kernel: a
// 16-bit cache, at most kShortTokens query tokens per sequence and 32 rows
// per kv head.
bool prefill_routes_short(int32_t max_q_len, int32_t num_q_heads, const pa_cache_desc* d);
pa_status plan_prefill(int32_t num_tokens, int32_t B, int32_t num_q_heads, int32_t max_q_len,
                       int32_t max_context_len, const pa_cache_desc* desc, int32_t split_tokens,
                       PrefillPlan* plan);

struct PrefillLaunch {
  const void* q;
  int32_t q_dtype;
  const int32_t* q_start;
  const void* k_cache;
  const void* v_cache;
  const float* k_scale;  // FP8 / INT8 caches, else null
  const float* v_scale;
  const int32_t* block_tables;
  int32_t max_blocks;
  const int32_t* context_lens;
  int32_t max_context_len, max_q_len;
  int32_t B, T, Hq, Hkv, D, num_blocks, kv_dtype;
  float scale;
  void* out;
  int32_t out_dtype;
  void* workspace;
  PrefillPlan plan;
};
pa_status launch_prefill(const PrefillLaunch& a, void* stream);

pa_status launch_cache_write(const void* k, const void* v, int32_t in_dtype,
                             const int64_t* slots, int64_t T, void* k_cache, void* v_cache,
                             float* k_scale, float* v_scale, const pa_cache_desc* d,
                             void* stream);

pa_status launch_copy_blocks(void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                             const int64_t* pairs, int64_t n, const pa_cache_desc* d,
                             void* stream);

pa_status launch_swap_blocks(void* dk, void* dv, float* dks, float* dvs, int32_t dnb, const void* sk,
                             const void* sv, const float* sks, const float* svs, int32_t snb,
                             const int64_t* pairs, int64_t n, const pa_cache_desc* d, void* stream);

// Launch `kernel` on `stream` as a programmatic dependent of the previous
// kernel in the stream: it may be scheduled while that kernel drains, and
// must call griddepcontrol.wait before touching memory the predecessor wrote.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Unique id of the CUDA context current on this thread (cuCtxGetId); false
// when there is none yet or it cannot be read.
bool current_context_id(unsigned long long* id);

// Per-translation-unit device error words, OR-ed by pa_device_errors.
pa_status read_errors_decode(uint32_t* flags, bool clear);
pa_status read_errors_cache_ops(uint32_t* flags, bool clear);
pa_status read_errors_prefill(uint32_t* flags, bool clear);

}  // namespace pa
