/*
 * pagedkv.h -- C ABI of libpagedkv.so: paged-KV attention for GB300 (sm_103a)
 * -- decode (plain, fused with the cache write, grouped over shared
 * prefixes), multi-token chunks, cache write, block copy and swap -- plus the
 * host-side block manager, the continuous-batching scheduler and the serving
 * iteration that drive it.
 *
 * Sources, cited by page title and section:
 *   [LLM-INF] "LLM推理引擎深度实战：从PagedAttention到分布式推理部署" (ybb.press)
 *             2.2 paging with 16-token pages, per-request page tables,
 *                 on-demand allocation, copy-on-write via refcounts;
 *             2.3 the attention kernel resolves the page table itself and
 *                 gathers scattered K/V, transparent to the model;
 *             5.3 FP8 (and INT8) KV cache with per-token or per-channel scales;
 *             3.1 continuous (iteration-level) batching;
 *             3.2 preemption by swapping to host memory or dropping;
 *             3.3 first-come-first-served scheduling;
 *             6.1 speculative decoding: the target model verifies the draft
 *                 tokens in one pass.
 *   [KV-CB]   "大模型推理引擎优化：KV Cache 与连续批处理" (devpress.csdn.net)
 *             2.2 16-token blocks;
 *             三   the block manager: block table, free list, refcount,
 *                 allocate / append / free / utilisation; the continuous
 *                 batching scheduler;
 *             4.1 chunked prefill: prompt chunks run beside decode steps;
 *             4.2 copy-on-write when a shared block is written.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Block size is fixed at PA_BLOCK_SIZE = 16 tokens.
 * - A KV cache is two device arrays k_cache, v_cache, each laid out
 *   [num_blocks][num_kv_heads][16][head_dim] in kv_dtype, so one (block,
 *   kv head) tile of 16 tokens is contiguous.  FP8 caches hold E4M3 codes and
 *   INT8 caches symmetric int8 codes; both carry two float32 arrays k_scale,
 *   v_scale laid out [num_blocks][16]: one scale per stored token, shared by
 *   all of that token's heads and dims.
 * - "slot" s addresses block s / 16, row s % 16.
 * - Ownership: the caller owns and allocates every device buffer (queues,
 *   tables, caches, outputs, workspace).  The library never allocates device
 *   memory, never synchronises the stream it is given, and keeps no pointer
 *   after a call returns.
 * - Streams: device work is enqueued on `stream` (a cudaStream_t passed as
 *   void*; NULL = legacy default stream) in call order.
 * - Errors: every call returns a pa_status.  Host arguments are validated
 *   before anything is enqueued, so a call that returns an error launched
 *   nothing.  pa_last_error() gives a message for the calling thread's last
 *   failed call.  Values that live on the device (slots, block ids, context
 *   lengths) cannot be checked on the host: the kernels bounds-check them,
 *   replace the offending access (a bad block id reads block 0) and set a bit in
 *   a per-device error word, read with pa_device_errors().  No kernel traps.
 * - Device pointers must be 16-byte aligned.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PA_BLOCK_SIZE 16
#define PA_MAX_GROUP 8      /* query heads per kv head supported by pa_decode */

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID = 1,      /* bad argument (null, shape, alignment, range) */
  PA_ERR_OOM = 2,          /* block manager: not enough free blocks */
  PA_ERR_NOT_FOUND = 3,    /* block manager: unknown sequence id */
  PA_ERR_UNSUPPORTED = 4,  /* valid but not built (head_dim, dtype, group) */
  PA_ERR_CUDA = 5          /* a CUDA runtime call or launch failed */
} pa_status;

typedef enum {
  PA_DTYPE_F16 = 0,
  PA_DTYPE_BF16 = 1,
  PA_DTYPE_FP8_E4M3 = 2,   /* OCP E4M3 codes + per-token float32 scales */
  PA_DTYPE_F32 = 3,
  PA_DTYPE_INT8 = 4        /* symmetric int8 codes + per-token float32 scales */
} pa_dtype;

/* Bits of the per-device error word (pa_device_errors). */
#define PA_DEVERR_SLOT_RANGE   0x1u  /* cache write: slot >= num_blocks*16 */
#define PA_DEVERR_BLOCK_RANGE  0x2u  /* decode/copy: block id outside the pool */
#define PA_DEVERR_CONTEXT_LEN  0x4u  /* decode: length < 0 or above a stated bound */
#define PA_DEVERR_TIMEOUT      0x8u  /* a bounded barrier wait gave up */
#define PA_DEVERR_QUERY_RANGE  0x10u /* chunked prefill: q_start out of order or range */
#define PA_DEVERR_GROUP        0x20u /* grouped decode: bad group bounds, or members' shared blocks differ */

/* Shape of a paged KV cache. */
typedef struct {
  int32_t num_blocks;    /* physical blocks in the pool, > 0 */
  int32_t num_kv_heads;  /* Hkv, > 0 */
  int32_t head_dim;      /* D: 64 or 128 (FP8 / INT8: 128) */
  int32_t block_size;    /* must be PA_BLOCK_SIZE */
  int32_t kv_dtype;      /* pa_dtype: F16, BF16, FP8_E4M3 or INT8 */
} pa_cache_desc;

/* Message for the calling thread's last failed call ("" if none). */
const char* pa_last_error(void);

/* ABI version of this header (major * 100 + minor). */
int32_t pa_version(void);

/*
 * pa_cache_write -- store this step's K/V rows in their slots.
 * [LLM-INF] 2.2 (pages exist only for generated tokens), [KV-CB] 三 (append).
 *
 * k, v         device, [num_tokens][num_kv_heads][head_dim] in in_dtype
 *              (F16, BF16 or F32).  For F16/BF16 caches in_dtype must equal
 *              kv_dtype or be F32 (rounded to nearest even); the copy of a
 *              same-dtype row is exact.
 * slot_mapping device int64 [num_tokens]; slot < 0 skips the row (padding).
 *              Slots must be distinct; a slot >= num_blocks*16 is skipped and
 *              flagged PA_DEVERR_SLOT_RANGE.
 * k_scale, v_scale  FP8 / INT8 caches only (else NULL): device float32
 *              [num_blocks][16].  Rows are quantised per token: amax =
 *              max|x| over all heads and dims of the token.  FP8: scale =
 *              amax/448 (float32 RN division; 1 when amax = 0), code =
 *              E4M3(x/scale) with round-to-nearest-even and saturation to
 *              +-448.  INT8: scale = amax/127 (1 when amax = 0), code =
 *              x/scale rounded half to even and clamped to [-127, 127].
 */
pa_status pa_cache_write(const void* k, const void* v, int32_t in_dtype,
                         const int64_t* slot_mapping, int64_t num_tokens,
                         void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                         const pa_cache_desc* desc, void* stream);

/*
 * pa_decode_workspace_size -- bytes of device workspace pa_decode needs for
 * the same (B, num_q_heads, max_context_len, desc, split_tokens).  0 when a
 * single partition covers max_context_len (no split-K pass).
 */
size_t pa_decode_workspace_size(int32_t B, int32_t num_q_heads, int32_t max_context_len,
                                const pa_cache_desc* desc, int32_t split_tokens);

/*
 * pa_decode_plan_info -- the split pa_decode / pa_decode_append would use for
 * the same arguments, for callers that size, log or profile their steps (host
 * only; nothing is launched).  partitions: partitions of the longest allowed
 * context; blocks_per_partition: 16-token blocks per partition; kernels:
 * kernels one call launches (1 when one partition covers the context or the
 * decode kernel merges the partitions itself -- at most 8 of them; 2 when a
 * merge kernel follows).  Any output pointer may be NULL.  PA_ERR_INVALID /
 * PA_ERR_UNSUPPORTED as pa_decode would return for the shape.
 */
pa_status pa_decode_plan_info(int32_t B, int32_t num_q_heads, int32_t max_context_len,
                              const pa_cache_desc* desc, int32_t split_tokens,
                              int32_t* partitions, int32_t* blocks_per_partition, int32_t* kernels);

/*
 * pa_decode -- one decode step of paged attention.
 * [LLM-INF] 2.3: the kernel translates logical token t of sequence b into
 * physical block block_tables[b][t/16], row t%16, and gathers K/V from there.
 * For every sequence b < B and query head h (kv head g = h / G, G =
 * num_q_heads / num_kv_heads, contiguous groups):
 *     out[b][h] = sum_t softmax_t(scale * q[b][h] . K_t) V_t,  t < context_lens[b]
 * context_lens[b] = 0 gives a zero row.
 *
 * q            device [B][num_q_heads][head_dim] in q_dtype.  For F16/BF16
 *              caches q_dtype must equal kv_dtype; for FP8 / INT8 caches F16
 *              or BF16.
 * k_scale, v_scale  FP8 / INT8 caches only (else NULL), as in pa_cache_write.
 * block_tables device int32 [B][max_blocks_per_seq]; entries past
 *              ceil(context_lens[b]/16) are never read.
 * context_lens device int32 [B]; each must be <= max_context_len and
 *              <= max_blocks_per_seq*16 (else clamped and flagged).
 * max_context_len host upper bound on context_lens, sizes the split.
 * out          device [B][num_q_heads][head_dim] in out_dtype (q_dtype or F32).
 * workspace    device, >= pa_decode_workspace_size(...) bytes, 16-byte
 *              aligned; may be NULL when that size is 0.  Contents are
 *              scratch: overwritten by the call, meaningless afterwards.
 * split_tokens tokens per split-K partition (multiple of 16, 16..1024), or 0
 *              to let the library choose from the shape and the SM count.
 *
 * Work: one CTA per (sequence, kv head, partition); all G query heads of a
 * kv head share every K/V tile load.  When a context splits into at most 8
 * partitions, the last partition of each (sequence, kv head) to finish
 * merges them inside the same kernel (arrival counters in the workspace,
 * stamped per launch, so their prior contents never matter); longer splits
 * are merged by a second kernel.  pa_decode_plan_info reports the split.
 *
 * Determinism: work is mapped statically; the arrival counter only decides
 * which CTA merges, and the merge sums the partitions in a fixed order, so
 * the same inputs, shape and split_tokens give bit-identical outputs on
 * every run, whatever the physical block ids the tables name.
 */
pa_status pa_decode(const void* q, int32_t q_dtype,
                    const void* k_cache, const void* v_cache,
                    const float* k_scale, const float* v_scale,
                    const int32_t* block_tables, int32_t max_blocks_per_seq,
                    const int32_t* context_lens, int32_t max_context_len,
                    int32_t B, int32_t num_q_heads, float scale,
                    void* out, int32_t out_dtype,
                    const pa_cache_desc* desc,
                    void* workspace, size_t workspace_bytes,
                    int32_t split_tokens, void* stream);

/*
 * pa_decode_append -- pa_cache_write of this step's tokens fused into
 * pa_decode: sequence b's new token (row b of k_new, v_new [B][Hkv][head_dim]
 * in new_dtype) is stored at slot_mapping[b] (< 0: none), then attention runs
 * as in pa_decode.  Results, cache contents and FP8 / INT8 scales are identical to
 * the two calls in sequence; the store is done inside the decode launch by the
 * work item that reads that block, before it reads it.  Requires the
 * block-manager invariant that slot_mapping[b] is the slot of sequence b's
 * last token (position context_lens[b] - 1 of its table).  Other arguments
 * and errors as in pa_cache_write and pa_decode.
 */
pa_status pa_decode_append(const void* k_new, const void* v_new, int32_t new_dtype,
                           const int64_t* slot_mapping,
                           const void* q, int32_t q_dtype,
                           void* k_cache, void* v_cache,
                           float* k_scale, float* v_scale,
                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* context_lens, int32_t max_context_len,
                           int32_t B, int32_t num_q_heads, float scale,
                           void* out, int32_t out_dtype,
                           const pa_cache_desc* desc,
                           void* workspace, size_t workspace_bytes,
                           int32_t split_tokens, void* stream);

/*
 * pa_decode_grouped_workspace_size -- bytes of device workspace
 * pa_decode_append_grouped needs for the same arguments (0 on an invalid
 * argument).
 */
size_t pa_decode_grouped_workspace_size(int32_t B, int32_t num_q_heads, int32_t max_context_len,
                                        int32_t n_groups, int32_t max_group_size, int32_t max_prefix_blocks,
                                        const pa_cache_desc* desc, int32_t split_tokens);

/*
 * pa_decode_append_grouped -- pa_decode_append for a batch whose sequences
 * come in groups sharing the leading blocks of their tables: the beams or
 * samples of one prompt after fork, which share those blocks by reference
 * count and copy on write ([LLM-INF] 2.2, [KV-CB] 4.2).  It computes what
 * pa_decode_append computes.  Results differ only by rounding, because the
 * partitions differ: the float32 summation order and the 16-bit rounding of the
 * softmax weights against each partition's running max.  What changes is how
 * the shared blocks are read.  One work item per (group, kv head,
 * partition of the shared prefix) loads each shared K/V tile once and scores
 * it against the queries of every member of the group; pa_decode_append reads
 * the tile once per member.  The members' private tails run as ordinary
 * partitions, and a merge kernel combines each member's prefix and tail
 * partitions.
 *
 * group_start   device int32 [n_groups + 1].  Group k is sequences
 *               group_start[k] .. group_start[k+1] - 1, with group_start[0] = 0
 *               and group_start[n_groups] = B.  Every group is non-empty and at
 *               most max_group_size long; a sequence in no group is a group of
 *               one.  Bad bounds skip the group and set PA_DEVERR_GROUP.
 * prefix_blocks device int32 [n_groups]: the number of leading table entries
 *               every member of group k has in common.  The kernel shares
 *               E_k = min(prefix_blocks[k], (L_m - 1) / 16 over the members'
 *               lengths L_m) blocks, so a shared block never holds a member's
 *               last token, where the fused write lands.  Members whose table
 *               entries differ within those blocks set PA_DEVERR_GROUP, and
 *               their rows are then unspecified.
 * n_groups      number of groups (1 .. B).
 * max_group_size host bound on group sizes, with
 *               max_group_size * num_q_heads / num_kv_heads <= 8.
 * max_prefix_blocks host bound on prefix_blocks; it sizes the grid.
 * workspace     device, >= pa_decode_grouped_workspace_size bytes.
 * Other arguments and errors as pa_decode_append.
 */
pa_status pa_decode_append_grouped(const void* k_new, const void* v_new, int32_t new_dtype,
                                   const int64_t* slot_mapping, const void* q, int32_t q_dtype,
                                   void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                                   const int32_t* block_tables, int32_t max_blocks_per_seq,
                                   const int32_t* context_lens, int32_t max_context_len,
                                   int32_t B, int32_t num_q_heads, float scale,
                                   const int32_t* group_start, const int32_t* prefix_blocks,
                                   int32_t n_groups, int32_t max_group_size, int32_t max_prefix_blocks,
                                   void* out, int32_t out_dtype, const pa_cache_desc* desc,
                                   void* workspace, size_t workspace_bytes,
                                   int32_t split_tokens, void* stream);

/*
 * pa_decode_append_segments -- pa_decode_append for groups whose members
 * share blocks in any pattern, not only a common prefix: after beam search
 * reselects, sibling beams hold their parent's blocks, so the members' tables
 * form a tree ([LLM-INF] 2.2 copy on write, [KV-CB] 4.2).  The caller lists
 * the segments: runs of table positions whose blocks a subset of a group's
 * members all hold (pa_table_segments computes them from the block
 * tables).  Each item reads its blocks once and scores them against the
 * queries of every member it lists; a merge kernel combines each member's
 * items.  It computes what pa_decode_append computes, up to rounding (the
 * partitions differ), reading each block of the batch once.  A batch without
 * shared blocks is B one-member groups: its items are then the sequences'
 * live partitions (pa_decode_items_plan says when that beats the fixed grid).
 *
 * group_start   device int32 [n_groups + 1], as for pa_decode_append_grouped;
 *               the groups cover sequences 0 .. B-1.
 * items         device int32 [n_items][4], 16-byte aligned, in any order (the
 *               order they are dispatched in: longest first balances best):
 *               {group k, member list, first block j0, nb | nm << 8 |
 *               slot << 16}.  The nm (1..8) members are indices within group
 *               k, 4 bits each, the first one's table row is read; every
 *               listed member holds the same blocks at table positions j0 ..
 *               j0 + nb - 1 (nb 1..64).  An item of several members lies
 *               before each member's last block (where the fused write
 *               lands).  Every position below a member's block count is in
 *               exactly one item listing it.  slot (< max_group_items) is the
 *               item's partial slot: the items listing one member have
 *               distinct slots.
 * n_items       host: rows of items (0 .. 65535; 0: every row is zero).
 * max_group_items host bound on slots (1..65535); it sizes the workspace
 *               (pa_decode_segments_workspace_size).
 * An item with bad fields is skipped and sets PA_DEVERR_GROUP (its members'
 * rows are then unspecified), as do members whose blocks differ.  Other
 * arguments and errors as pa_decode_append_grouped.
 */
pa_status pa_decode_append_segments(const void* k_new, const void* v_new, int32_t new_dtype,
                                    const int64_t* slot_mapping, const void* q, int32_t q_dtype,
                                    void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                                    const int32_t* block_tables, int32_t max_blocks_per_seq,
                                    const int32_t* context_lens, int32_t max_context_len,
                                    int32_t B, int32_t num_q_heads, float scale,
                                    const int32_t* group_start, int32_t n_groups, int32_t max_group_size,
                                    const int32_t* items, int32_t n_items, int32_t max_group_items, void* out,
                                    int32_t out_dtype,
                                    const pa_cache_desc* desc, void* workspace, size_t workspace_bytes,
                                    void* stream);

/*
 * pa_table_segments -- the items of pa_decode_append_segments from the block
 * tables (host only; nothing is launched).  Per group and table position j,
 * the members whose tables hold the same block at j form a class, except that
 * at and after a member's last block (the block its next token is written
 * to) the member is alone; a segment is a maximal run of positions over which
 * a member's class stays the same.  Each segment is listed once, by its lowest
 * member, cut into items of at most blocks_per_item blocks; a group's items
 * take slots 0, 1, ... in the order (lowest member, first position), and the
 * list is sorted longest first (ties in that order, groups in turn).
 *
 * block_tables  host int32 [n_sequences][max_blocks].
 * context_lens  host int32, 0 .. max_blocks * 16.
 * group_start   host int32 [n_groups + 1]; groups of 0 .. 8 members.
 * items         host int32 [max_items][4] out, the layout of
 *               pa_decode_append_segments; *n_items out; *max_slots out (the
 *               most items of one group), may be NULL.
 * PA_ERR_INVALID on a bad argument or more than max_items items (at most the
 * members' blocks summed are ever needed).
 */
pa_status pa_table_segments(const int32_t* block_tables, int32_t max_blocks, const int32_t* context_lens,
                            const int32_t* group_start, int32_t n_groups, int32_t blocks_per_item,
                            int32_t* items, int32_t max_items, int32_t* n_items, int32_t* max_slots);

/*
 * pa_decode_segments_workspace_size -- bytes of device workspace
 * pa_decode_append_segments needs: the split-K partials of B sequences x
 * num_q_heads x max_group_items (0 on an invalid argument).
 */
size_t pa_decode_segments_workspace_size(int32_t B, int32_t num_q_heads, int32_t n_groups,
                                         int32_t max_group_size, int32_t max_group_items,
                                         const pa_cache_desc* desc);

/*
 * pa_decode_items_plan -- whether a batch without shared blocks decodes
 * faster as a host-planned list of its live partitions than over
 * pa_decode_append's fixed grid (host only; nothing is launched).  The fixed
 * grid gives every sequence max_parts partitions per kv head (a block table
 * maps only the blocks below a sequence's length, [LLM-INF] 2.2), and the
 * cells past a short sequence's end exit at once;
 * with skewed lengths most cells are empty.  The list is B one-member groups
 * (group_start = 0, 1, ..., B) for pa_decode_append_segments, whose items
 * pa_table_segments cuts from each sequence's length -- the same partitions,
 * none empty.
 *
 * context_lens  host int32 [B], 0 .. max_context_len: this step's lengths.
 * Other inputs as pa_decode_plan_info.
 * *use_items    out: 1 when fewer than half of the fixed grid's cells hold
 *               blocks, the split has more than one partition and G <= 8
 *               (measured on GB300: 28 % live cells, 6 % faster; 62 % and
 *               75 %, as fast or slower); else 0.
 * *blocks_per_item out (may be NULL): the plan's partition length, for
 *               pa_table_segments.
 * *max_items_per_seq out (may be NULL): partitions of the longest allowed
 *               context: max_group_items of the call and of its workspace.
 * PA_ERR_INVALID on a null pointer or a length out of range; errors of
 * pa_decode_plan_info otherwise.
 */
pa_status pa_decode_items_plan(const int32_t* context_lens, int32_t B, int32_t num_q_heads,
                               int32_t max_context_len, const pa_cache_desc* desc, int32_t split_tokens,
                               int32_t* use_items, int32_t* blocks_per_item, int32_t* max_items_per_seq);

/*
 * pa_chunked_prefill_workspace_size -- bytes of device workspace
 * pa_chunked_prefill needs for the same arguments, and for a call with a
 * smaller max_q_len that the decode kernel serves (its split-K partials grow
 * with B * max_q_len rather than num_tokens); 0 when one partition covers
 * max_context_len and nothing goes to the decode kernel (or on an invalid
 * argument).
 */
size_t pa_chunked_prefill_workspace_size(int32_t num_tokens, int32_t B, int32_t num_q_heads,
                                         int32_t max_q_len, int32_t max_context_len,
                                         const pa_cache_desc* desc, int32_t split_tokens);

/*
 * pa_chunked_prefill_plan_info -- what pa_chunked_prefill would launch for
 * the same arguments (host only).  tensor_cores: 1 for the tcgen05 kernel
 * (128-row tiles), 0 for the mma.sync kernel (64-row tiles); partitions and
 * blocks_per_partition of the multi-token kernel; kernels: kernels one call
 * launches at most (over a 1-byte cache the one-token sequences first go
 * through the decode kernel, and a call with max_q_len 1 launches only
 * those).  Any output pointer may be NULL.
 */
pa_status pa_chunked_prefill_plan_info(int32_t num_tokens, int32_t B, int32_t num_q_heads,
                                       int32_t max_q_len, int32_t max_context_len,
                                       const pa_cache_desc* desc, int32_t split_tokens,
                                       int32_t* tensor_cores, int32_t* partitions,
                                       int32_t* blocks_per_partition, int32_t* kernels);

/*
 * pa_chunked_prefill -- paged attention for several query tokens per
 * sequence: a prompt chunk whose prefill runs beside decode steps ([KV-CB]
 * 4.1), or the gamma + 1 tokens a target model checks in one pass when
 * verifying a draft ([LLM-INF] 6.1).  Decode steps may ride in the same
 * call as one-token chunks.
 *
 * The n_b = q_start[b+1] - q_start[b] query tokens of sequence b are the
 * last n_b of its context_lens[b] = L_b tokens; their K/V must already be in
 * the cache (pa_cache_write first).  Query token i (0 <= i < n_b) is at
 * position L_b - n_b + i and attends, causally, to keys 0 .. L_b - n_b + i:
 *     out[q_start[b]+i][h] = sum_t softmax_t(scale * q[q_start[b]+i][h] . K_t) V_t,
 *                            t <= L_b - n_b + i,  kv head g = h / G.
 * A token with no key (n_b > L_b, flagged PA_DEVERR_CONTEXT_LEN) gets a
 * zero row.  n_b = 0 is allowed.
 *
 * q            device [num_tokens][num_q_heads][head_dim] in q_dtype, the
 *              sequences' tokens packed in order.  q_dtype equals kv_dtype for
 *              F16 / BF16 caches; for FP8_E4M3 / INT8 caches it is F16 or BF16
 *              (codes are converted to it exactly; head_dim 128).
 * k_scale, v_scale  FP8 / INT8 caches: device float [num_blocks][16] per-token
 *              scales as pa_cache_write stores them (16-byte aligned); NULL
 *              for F16 / BF16 caches.
 * q_start      device int32 [B + 1], q_start[0] = 0, nondecreasing,
 *              q_start[B] <= num_tokens, each n_b <= max_q_len (else that
 *              sequence is skipped and PA_DEVERR_QUERY_RANGE is set).
 * max_q_len    host upper bound on n_b (<= 65535), sizes the grid.
 * block_tables, context_lens, max_context_len, scale, desc, workspace,
 * split_tokens  as pa_decode (split_tokens up to 4096 here).
 * out          device [num_tokens][num_q_heads][head_dim] in out_dtype
 *              (q_dtype or F32); rows of tokens outside every sequence's range
 *              are not written.
 *
 * Work: one CTA per (sequence, kv head, 64-row tile of (token, head) rows,
 * partition); K/V tiles of a partition are loaded once per CTA by TMA and
 * shared by its four compute warps; partitions are merged by a second
 * kernel when a row's keys span more than one.  At head_dim 128 with more
 * than 64 rows per kv head the tiles are 128 rows on tcgen05 (FP8 / INT8
 * codes are converted to 16-bit in shared memory on the way to the tensor
 * cores).  The sequences with one query token (the decode steps riding in
 * the call) are served by the decode kernel, whose workspace follows the
 * multi-token kernel's, on a second stream of the calling thread that the
 * call forks from `stream` and joins back to it (the multi-token grid's last
 * wave leaves SMs to the decode rows); a call whose max_q_len is 1 launches
 * only the decode kernel, on `stream`.  Over a 16-bit cache a call with
 * max_q_len <= 8 and max_q_len * num_q_heads / num_kv_heads <= 32 runs
 * entirely in the decode kernel, one CTA per (sequence, kv head, query
 * token, partition), the columns of one (sequence, kv head) neighbours so
 * that their K/V reads meet in L2; malformed sequences are flagged as
 * above.  pa_chunked_prefill_plan_info reports what a call launches.
 */
pa_status pa_chunked_prefill(const void* q, int32_t q_dtype, const int32_t* q_start,
                             int32_t num_tokens, int32_t max_q_len,
                             const void* k_cache, const void* v_cache,
                             const float* k_scale, const float* v_scale,
                             const int32_t* block_tables, int32_t max_blocks_per_seq,
                             const int32_t* context_lens, int32_t max_context_len,
                             int32_t B, int32_t num_q_heads, float scale,
                             void* out, int32_t out_dtype, const pa_cache_desc* desc,
                             void* workspace, size_t workspace_bytes,
                             int32_t split_tokens, void* stream);

/*
 * pa_decode_static_ws -- pa_decode that allocates nothing.  The pages have no
 * counterpart: this entry point exists for callers of this library that
 * cannot allocate device memory when they decode -- code running as a plugin
 * inside an engine whose allocator owns the whole device and offers no
 * scratch hook, or a latency-critical loop where cudaMalloc/cudaFree would add
 * latency and device-wide synchronisation.
 *
 * Arguments and results are those of pa_decode without workspace /
 * workspace_bytes: the split-K partials live in one static device array of
 * PA_STATIC_WS_BYTES compiled into the library.  The caller still passes
 * inputs and outputs.
 * - A shape whose pa_decode_workspace_size exceeds PA_STATIC_WS_BYTES returns
 *   PA_ERR_INVALID and launches nothing.
 * - The first call made in a context looks the array's address up there
 *   (one cudaGetSymbolAddress) and caches it under the context's unique id,
 *   so a call in another context -- a second context on the device, or the
 *   new primary context after cudaDeviceReset -- looks it up again.  Make the
 *   first call in a context before any stream capture.
 * - Residency: with lazy module loading (the CUDA default) the array takes
 *   PA_STATIC_WS_BYTES of device memory in a context from the first call of
 *   this entry point there; with CUDA_MODULE_LOADING=EAGER in every context
 *   the library's device code is loaded into, whether or not this entry point
 *   is ever called.  It stays until the context is destroyed or the process
 *   exits.
 * - All calls on a device share the array, which keeps the last call's
 *   contents; calls whose kernels overlap on the GPU race on it, so
 *   serialise them (one stream, or events).
 * - No cudaMalloc, cudaFree or allocating library routine is called.
 */
#define PA_STATIC_WS_BYTES (32u * 1024u * 1024u)
pa_status pa_decode_static_ws(const void* q, int32_t q_dtype,
                              const void* k_cache, const void* v_cache,
                              const float* k_scale, const float* v_scale,
                              const int32_t* block_tables, int32_t max_blocks_per_seq,
                              const int32_t* context_lens, int32_t max_context_len,
                              int32_t B, int32_t num_q_heads, float scale,
                              void* out, int32_t out_dtype,
                              const pa_cache_desc* desc,
                              int32_t split_tokens, void* stream);

/*
 * pa_copy_blocks -- copy-on-write block copies.
 * [LLM-INF] 2.2 and [KV-CB] 4.2: before a shared block is written, its
 * contents are copied to a private block.  For each pair (src, dst) in
 * `pairs` (device int64 [num_pairs][2]) the whole K block, V block and, for
 * FP8 / INT8 caches, both 16-entry scale rows are copied.  No dst may repeat or appear as a
 * src (the block manager never emits such pairs); ids outside the pool are
 * skipped and flagged PA_DEVERR_BLOCK_RANGE.
 */
pa_status pa_copy_blocks(void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                         const int64_t* pairs, int64_t num_pairs,
                         const pa_cache_desc* desc, void* stream);

/*
 * pa_swap_blocks -- move whole blocks between two pools of the same shape,
 * for preemption and resume: a request's pages go to CPU memory when the GPU
 * runs short and come back when it is scheduled again ([LLM-INF] 3.2).
 * Each pool is laid out like a cache, k and v [num_blocks][Hkv][16][D] (+ FP8 /
 * INT8 scale rows [num_blocks][16]); either may be device memory or page-locked
 * host memory that the device addresses directly (cudaHostAlloc /
 * cudaHostRegister under unified addressing, e.g. torch pin_memory()).
 * pairs: device-accessible int64 [num_pairs][2], (src block of the src pool,
 * dst block of the dst pool); no dst may repeat.  desc gives Hkv, head_dim,
 * block_size and kv_dtype (its num_blocks is not used).  One kernel launch
 * (a gather, not one copy per block); ids outside a pool are skipped and
 * flagged PA_DEVERR_BLOCK_RANGE.
 */
pa_status pa_swap_blocks(void* dst_k, void* dst_v, float* dst_k_scale, float* dst_v_scale,
                         int32_t dst_num_blocks,
                         const void* src_k, const void* src_v,
                         const float* src_k_scale, const float* src_v_scale,
                         int32_t src_num_blocks,
                         const int64_t* pairs, int64_t num_pairs,
                         const pa_cache_desc* desc, void* stream);

/*
 * pa_device_errors -- read (and optionally clear) the current device's error
 * word (PA_DEVERR_* bits).  Synchronises the device.
 */
pa_status pa_device_errors(uint32_t* flags, int32_t clear);

/* ------------------------------------------------------------------------
 * Host block manager ([KV-CB] 三; copy-on-write per [LLM-INF] 2.2).
 * Single-threaded: a handle must not be used by two threads at once.
 * Free list is FIFO: allocation takes from the front, release appends at the
 * back, a table is released in logical order.  Every mutating call is
 * all-or-nothing: on error the state is unchanged.
 * ------------------------------------------------------------------------ */
typedef struct pa_alloc pa_alloc;

/* num_blocks > 0; block_size must be 16; free_order (host int64
 * [num_blocks], a permutation of 0..num_blocks-1) sets the initial free-list
 * order, NULL = ascending. */
pa_status pa_alloc_create(int32_t num_blocks, int32_t block_size,
                          const int64_t* free_order, pa_alloc** out);
void pa_alloc_destroy(pa_alloc* a);

/* New sequence holding num_tokens tokens: takes ceil(num_tokens/16) blocks.
 * PA_ERR_INVALID if seq_id exists, PA_ERR_OOM if too few blocks are free. */
pa_status pa_alloc_seq(pa_alloc* a, uint64_t seq_id, int64_t num_tokens);

/* Reserve the slot of the sequence's next token; returns slot = block*16 +
 * row.  If the last block is full a fresh block is appended.  If the last
 * block is partial and shared (refcount > 1) the sequence first moves to a
 * fresh block: *cow_src, *cow_dst name the copy the caller must perform
 * (pa_copy_blocks) before writing; otherwise both are -1. */
pa_status pa_append_slot(pa_alloc* a, uint64_t seq_id, int64_t* slot,
                         int64_t* cow_src, int64_t* cow_dst);

/* Batched pa_append_slot over n distinct sequences, in order, all or
 * nothing.  slots: host int64 [n]; cow_pairs: host int64 [n][2] receives the
 * copies (src, dst) packed at the front; *n_cow their number. */
pa_status pa_append_slots(pa_alloc* a, const uint64_t* seq_ids, int32_t n,
                          int64_t* slots, int64_t* cow_pairs, int32_t* n_cow);

/* Append n tokens to a sequence at once (n successive pa_append_slot): all
 * or nothing.  slots (optional, host int64 [n]) receives their slots; only the
 * first token can need a copy-on-write, reported in *cow_src, *cow_dst (else
 * -1, -1).  Used to grow a sequence by a prompt chunk. */
pa_status pa_append_tokens(pa_alloc* a, uint64_t seq_id, int64_t n, int64_t* slots,
                           int64_t* cow_src, int64_t* cow_dst);

/* child shares every block of parent (refcount + 1 each); same token count. */
pa_status pa_fork(pa_alloc* a, uint64_t parent, uint64_t child);

/* n forks parents[i] -> children[i] in order, all or nothing (a child may
 * serve as a later parent).  Beam search reselects beams this way. */
pa_status pa_fork_seqs(pa_alloc* a, const uint64_t* parents, const uint64_t* children,
                       int32_t n);

/* Release n distinct sequences in order, all or nothing. */
pa_status pa_free_seqs(pa_alloc* a, const uint64_t* ids, int32_t n);

/* Beam reselection in place: sequence ids[i] takes over the table and token
 * count of ids[parent_idx[i]] (0 <= parent_idx[i] < n).  Equivalent to forking
 * every ids[parent_idx[i]] into a new sequence, then releasing the n old
 * sequences in order, then renaming the forks to ids[i]; shared blocks keep
 * refcounts, so the next pa_append_slots copies a shared partial block
 * ([LLM-INF] 2.2 copy-on-write for beam search).  All or nothing. */
pa_status pa_reselect(pa_alloc* a, const uint64_t* ids, const int32_t* parent_idx, int32_t n);

/* Release a sequence: refcount - 1 per block, freed at 0. */
pa_status pa_free_seq(pa_alloc* a, uint64_t seq_id);

/* Copy one table (cap entries max) and its token count. */
pa_status pa_block_table(const pa_alloc* a, uint64_t seq_id, int32_t* out, int32_t cap,
                         int32_t* n_blocks, int64_t* n_tokens);

/* Tables of n sequences as a host int32 [n][cap] array padded with -1, and
 * their token counts as int32 [n] (the decode kernel's context_lens). */
pa_status pa_block_tables(const pa_alloc* a, const uint64_t* seq_ids, int32_t n,
                          int32_t* tables, int32_t cap, int32_t* context_lens);

/* Pool statistics; refcounts (optional, int32 [num_blocks]) receives every
 * block's refcount.  Utilisation = (total - free) / total ([KV-CB] 三). */
pa_status pa_alloc_stats(const pa_alloc* a, int32_t* total, int32_t* free_blocks,
                         int32_t* refcounts);

/* Free list front to back (cap entries max); *n = its full length. */
pa_status pa_free_list(const pa_alloc* a, int32_t* out, int32_t cap, int32_t* n);

/* ---------------------------------------------------------------------------
 * Continuous-batching scheduler ([LLM-INF] 3.1-3.3, [KV-CB] 三 and 4.1).
 * Host only.  It owns a block manager of num_blocks GPU blocks and a host
 * swap pool of host_blocks blocks, and decides every iteration which
 * requests run and which tokens they bring:
 *   1. requests that produced their last output in the previous step retire
 *      (their blocks are released);
 *   2. every decoding request gets one slot; while the free blocks do not
 *      cover them, a running request is preempted: the one holding the most
 *      blocks (later arrival on a tie) is swapped to the host pool if it
 *      fits there, else the one holding the fewest (later arrival on a tie)
 *      is dropped and goes back to the waiting queue to start over;
 *   3. running requests continue their prompt in chunks bounded by the token
 *      budget left (max_tokens minus the decodes) and the blocks they can get;
 *   4. swapped requests come back in arrival order while their blocks fit
 *      and the batch (max_batch) has room; they run from the next step;
 *   5. waiting requests are admitted in arrival order with a first chunk
 *      while the batch has room, budget is left and the chunk's blocks fit
 *      (each admission lowers the free count); admission stops at the first
 *      request that does not fit;
 *   6. if nothing could run while requests are running, one is preempted.
 * A request preempted in a step comes back in a later one at the earliest.
 * The step that prefills a prompt's last token yields its first output;
 * every later step appends the previous output's K/V and yields the next;
 * after max_new_tokens outputs the request retires at the next step.
 * ------------------------------------------------------------------------- */
typedef struct pa_sched pa_sched;

#define PA_SCHED_PREFILL 0
#define PA_SCHED_DECODE  1

/* One step's decisions.  Arrays are caller-owned and must hold at least:
 * ids, kinds, starts, lens, finished, recomputed: max_batch entries;
 * slots: max_batch + max_tokens; swap_out, swap_in: 2 * num_blocks. */
typedef struct {
  int32_t   n_items;      /* requests that run this step, in batch order */
  uint64_t* ids;
  int32_t*  kinds;        /* PA_SCHED_PREFILL (a prompt chunk) or PA_SCHED_DECODE */
  int32_t*  starts;       /* position of the item's first new token */
  int32_t*  lens;         /* new tokens of the item (1 for a decode) */
  int64_t   n_slots;      /* sum of lens */
  int64_t*  slots;        /* cache slots of the new tokens, items in order */
  int32_t   n_finished;
  uint64_t* finished;     /* retired at the start of this step */
  int32_t   n_swap_out;
  int64_t*  swap_out;     /* [n][2] (GPU block, host block): copy before this step's writes */
  int32_t   n_swap_in;
  int64_t*  swap_in;      /* [n][2] (host block, GPU block): copy before the next step */
  int32_t   n_recomputed;
  uint64_t* recomputed;   /* dropped back to the waiting queue */
} pa_sched_step_out;

/* free_order: host int64 permutation of the GPU pool, or NULL for 0..n-1;
 * max_batch, max_tokens > 0; host_blocks >= 0 (0 = preempt by recompute). */
pa_status pa_sched_create(int32_t num_blocks, const int64_t* free_order, int32_t max_batch,
                          int32_t max_tokens, int32_t host_blocks, pa_sched** out);
void pa_sched_destroy(pa_sched* s);
/* Queue a request.  PA_ERR_INVALID for an id in use, a prompt or output
 * length < 1, or ceil((prompt_len + max_new_tokens) / 16) > num_blocks. */
pa_status pa_sched_add(pa_sched* s, uint64_t id, int32_t prompt_len, int32_t max_new_tokens);
pa_status pa_sched_step(pa_sched* s, pa_sched_step_out* out);
/* The scheduler's block manager, for pa_block_tables on the running ids
 * (read only: the scheduler is its only writer). */
const pa_alloc* pa_sched_allocator(const pa_sched* s);
pa_status pa_sched_stats(const pa_sched* s, int32_t* n_waiting, int32_t* n_running, int32_t* n_swapped,
                         int32_t* free_blocks, int32_t* free_host_blocks);
/* The limits the scheduler was created with. */
pa_status pa_sched_limits(const pa_sched* s, int32_t* max_batch, int32_t* max_tokens, int32_t* num_blocks);

/* ---------------------------------------------------------------------------
 * Serving iteration engine: one scheduler step turned into device work on one
 * stream -- one host-to-device copy of the staged decisions; swap-out copies
 * (GPU -> host pool) of preempted requests; the decode items' cache write
 * fused into pa_decode; pa_cache_write + pa_chunked_prefill for the prompt
 * chunks; swap-in copies (host pool -> GPU) of requests that run next step.
 * F16 / BF16 caches, or FP8_E4M3 / INT8 caches with per-token scales (the
 * model's q / K / V then in F16 or BF16).  Every buffer is caller-owned.
 * ------------------------------------------------------------------------- */
typedef struct pa_serve pa_serve;

typedef struct {
  void*   k_cache;          /* device pools of the scheduler's num_blocks blocks */
  void*   v_cache;
  void*   k_host;           /* pinned host swap pools [host_blocks][Hkv][16][D] (NULL if 0) */
  void*   v_host;
  int32_t host_blocks;      /* as given to pa_sched_create */
  int32_t num_q_heads;
  int32_t max_context;      /* bound on a request's prompt + outputs (tokens) */
  int32_t split_tokens;     /* partition size of the chunk kernel (> 0, multiple of 16) */
  void*   staging_host;     /* pinned, 2 * pa_serve_staging_bytes() bytes, 16-byte aligned */
  void*   staging_dev;      /* device, pa_serve_staging_bytes() bytes, 16-byte aligned */
  void*   workspace;        /* device, >= pa_serve_workspace_bytes() bytes (may be NULL if 0) */
  size_t  workspace_bytes;
  float*  k_scale;          /* FP8 / INT8 caches: device per-token scales [num_blocks][16], */
  float*  v_scale;          /*   16-byte aligned; NULL for F16 / BF16 caches */
  float*  k_host_scale;     /* FP8 / INT8 caches with host_blocks > 0: pinned [host_blocks][16] */
  float*  v_host_scale;
} pa_serve_buffers;

size_t pa_serve_staging_bytes(const pa_sched* s, int32_t max_context);
size_t pa_serve_workspace_bytes(const pa_sched* s, int32_t num_q_heads, int32_t max_context,
                                const pa_cache_desc* desc, int32_t split_tokens);
/* The engine keeps pointers to s and to the buffers until destroyed. */
pa_status pa_serve_create(pa_sched* s, const pa_cache_desc* desc, const pa_serve_buffers* bufs,
                          pa_serve** out);
void pa_serve_destroy(pa_serve* e);
/* Plan the next iteration: run the scheduler step and stage its decisions
 * (host only; waits for the staging copy of two iterations before).
 * decisions: arrays as for pa_sched_step, or NULL to keep them internal;
 * *num_tokens (if not NULL) = T, the new tokens the iteration brings.  A plan
 * must be launched before the next one is made. */
pa_status pa_serve_plan(pa_serve* e, pa_sched_step_out* decisions, int64_t* num_tokens);
/* Launch the planned iteration on `stream`: q: device [>= T][num_q_heads][D],
 * k_new / v_new: device [>= T][Hkv][D], all in_dtype (the cache dtype; F16
 * or BF16 for FP8 / INT8 caches),
 * row t for the t-th new token (items in order; decodes come first); out:
 * device [>= T][num_q_heads][D] in in_dtype. */
pa_status pa_serve_launch(pa_serve* e, const void* q, const void* k_new, const void* v_new, int32_t in_dtype,
                          void* out, void* stream);
/* pa_serve_plan followed by pa_serve_launch.
 * One iteration.  q: device [>= T][num_q_heads][D], k_new / v_new: device
 * [>= T][Hkv][D], all in_dtype (the cache dtype; F16 or BF16 for FP8 / INT8
 * caches), row t for the t-th new
 * token of the step (items in order; decodes come first); out: device
 * [>= T][num_q_heads][D] in in_dtype.  decisions: arrays as for
 * pa_sched_step, or NULL to keep them internal.  Blocks the host only to
 * wait for the staging copy of two steps before. */
pa_status pa_serve_step(pa_serve* e, const void* q, const void* k_new, const void* v_new, int32_t in_dtype,
                        void* out, pa_sched_step_out* decisions, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* PAGEDKV_H */
