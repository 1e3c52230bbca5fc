// Paged decode attention for sm_103a.
//
// What it computes ("LLM推理引擎深度实战：从PagedAttention到分布式推理部署",
// section 2.3): for each sequence and query head, softmax(scale q.K^T).V over
// the sequence's context, where the kernel itself maps logical token t to
// physical block block_tables[b][t/16], row t%16, and gathers the scattered
// K/V tiles from there.
//
// Design (GB300):
// * Work item = (sequence b, kv head g, partition p of `bpp` 16-token
//   blocks), one single-warp CTA per item (grid: b*Hkv + g, p).  All G query
//   heads of kv head g share every K/V tile, so K/V bytes are read from HBM
//   once per step.  Small one-warp CTAs keep many independent load streams per
//   SM (six or more), which is what hides HBM latency here; an item needs no
//   block-wide barrier and no cross-warp merge, and an empty grid cell (a
//   partition past a short sequence's end) costs one warp launch.
// * The warp streams its item's (block, kv head) tiles -- 16 rows x D,
//   contiguous -- through a ring of shared-memory stages with TMA
//   (cp.async.bulk.tensor, 128-byte swizzle) completed by mbarriers.  As soon
//   as a tile's fragments are in registers the stage is refilled with the
//   tile NS blocks ahead.
// * Scores on tensor cores, transposed: S^T[16 tokens x 8 heads] =
//   K_tile[16 x D] . Q^T[D x 8] with mma.m16n8k16 (A = K from ldmatrix,
//   B = Q from registers; G < 8 pads N with zero heads).  Online softmax in
//   fp32 (exp2, log2e folded into the scale), then O^T[D x 8] += V^T[D x 16] .
//   P^T[16 x 8] with A = V via ldmatrix.trans and B = P^T from the score
//   fragment by movmatrix.  bf16 P is carried as hi + lo bf16 parts (rounding
//   error ~2^-17).
// * FP8 E4M3 and INT8 caches (1-byte codes): codes are converted exactly to
//   f16/bf16 in registers; the per-token K scale multiplies the score, the
//   per-token V scale multiplies p before the PV product.
// * A one-partition sequence is written directly; otherwise the partition
//   writes (o, m, l) and decode_reduce merges the partitions with log-sum-exp
//   weights, launched as a programmatic dependent (triggered once every item
//   has started, so its CTAs are resident when the last items finish).
// * Shared prefixes (pa_decode_append_grouped; "LLM推理引擎深度实战" 2.2 and
//   "大模型推理引擎优化：KV Cache 与连续批处理" 4.2 share blocks by refcount): the
//   beams of one prompt hold the same blocks for the prompt.  A prefix item
//   reads each shared tile once and scores it against the queries of every
//   member of the group, as extra MMA columns (members x G <= 8).  Members'
//   tails are ordinary items, and decode_reduce_grouped merges each member's
//   prefix and tail partitions.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "device_common.cuh"
#include "kv_map.h"
#include "pa_internal.h"

namespace pa {
namespace {

__device__ uint32_t g_decode_err;

#ifndef PA_RING_KB
#define PA_RING_KB 16  // two 8 KB stages for 16-bit D=128: ~12 CTAs per SM
#endif
constexpr int kRingBytes = PA_RING_KB * 1024;  // K/V stage ring of one warp-CTA
constexpr int kMaxDevices = 64;
#ifndef PA_MERGE_SPEC
#define PA_MERGE_SPEC 1  // the merge kernel loads its first 32 partial rows with the length
#endif
#ifndef PA_EARLY_ISSUE
#define PA_EARLY_ISSUE 1
#endif
#ifndef PA_P_ASC
#define PA_P_ASC 0
#endif

struct DecodeArgs {
  const void* q;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const float* k_scale;
  const float* v_scale;
  void* out;
  float* part_o;
  float* part_m;
  float* part_l;
  int32_t B, Hq, Hkv, G, max_blocks, num_blocks, max_context_len;
  int32_t bpp, max_parts;
  float scale_log2;
  int32_t out_f32;
  // fused cache write (pa_decode_append): sequence b's new token, row b of
  // k_new / v_new [B][Hkv][D] in new_dtype, goes to slot_mapping[b] first
  const void* k_new;
  const void* v_new;
  void* k_cache_w;  // the caches, for the fused row store
  void* v_cache_w;
  const int64_t* slot_mapping;
  float* k_scale_w;  // FP8 / INT8 scales, writable views of k_scale / v_scale
  float* v_scale_w;
  int32_t new_dtype;
  int32_t fuse_write;
  // shared-prefix groups (pa_decode_append_grouped), else n_groups == 0:
  // group k = sequences group_start[k] .. group_start[k+1]-1 sharing their
  // first prefix_blocks[k] blocks
  const int32_t* group_start;
  const int32_t* prefix_blocks;
  int32_t n_groups, max_members;
  int32_t pre_parts, tail_parts;  // grid rows: shared-prefix partitions, tail partitions
  // segments of groups (pa_decode_append_segments), else null: item i =
  // {group k, member list (4 bits per member index within the group, nm of
  // them), first block j0, nb | nm << 8 | slot << 16}; its partials are
  // partial slot `slot` of each of its members
  const int4* seg_items;
  int32_t n_seg_items;
  // in-kernel split-K merge (plain grid): one arrival counter per (sequence,
  // kv head), stamped with this launch's epoch
  unsigned long long* tickets;
  uint32_t epoch;
  // rows of a multi-token call (else null): sequence b brings the n_b =
  // q_start[b+1] - q_start[b] query tokens q_start[b] .. of q_rows, the last
  // n_b of its context; token t attends causally to the first L_b - n_b + 1 + t
  // keys and is served by the grid column (b, g, t), t < q_tokens.  Sequences
  // with n_b > q_tokens are left to the multi-token kernel (with q_tokens = 1,
  // the one-token sequences only), unless q_report: then the decode kernel
  // serves the whole call and flags them as the multi-token kernel would.
  const int32_t* q_start;
  int32_t q_rows, q_tokens, q_report;
};

// A group's usable shared prefix: whole blocks every member has before the
// block of its last token (so the fused write never lands in a shared
// block), at most the caller's prefix_blocks.  Lane m < members holds member
// m's clamped length in `Lm`; every lane gets the result.
__device__ __forceinline__ int group_prefix(int pre, int members, int Lm, int lane) {
  int e = lane < members ? (Lm > 0 ? (Lm - 1) >> 4 : 0) : 0x7fffffff;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) e = min(e, __shfl_xor_sync(0xffffffffu, e, o));
  return max(0, min(pre, e));
}

// Element i (of a contiguous row) of a K/V input in f16, bf16 or f32, as float.
__device__ __forceinline__ float load_in(const void* p, size_t i, int dt) {
  if (dt == PA_DTYPE_F32) return static_cast<const float*>(p)[i];
  if (dt == PA_DTYPE_F16) return __half2float(static_cast<const __half*>(p)[i]);
  return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
}

// One warp stores kv head g's row of this step's new token (K and V) into
// the cache slot, exactly as pa_cache_write does: a same-dtype copy, a
// round-to-nearest-even conversion from f32, or for FP8 / INT8 the per-token
// amax / scale / code encoding over all Hkv*D values of the token.  Every kv
// head's warp recomputes the token's amax and stores the (identical) scale:
// its own later read of the scale row must not depend on another CTA.
template <typename KT, int D>
__device__ __forceinline__ void write_new_row(const DecodeArgs& a, KT* kc, KT* vc, int b, int g,
                                              int64_t slot, int lane) {
  constexpr bool Q8 = sizeof(KT) == 1;  // 1-byte codes: E4M3 or INT8
  const int64_t blk = slot / 16, off = slot % 16;
  const size_t dst = ((static_cast<size_t>(blk) * a.Hkv + g) * 16 + off) * D;
#pragma unroll
  for (int which = 0; which < 2; ++which) {
    const void* src = which ? a.v_new : a.k_new;
    KT* cache = which ? vc : kc;
    const size_t row = (static_cast<size_t>(b) * a.Hkv + g) * D;
    if constexpr (Q8) {
      float amax = 0.f;
      const size_t tok = static_cast<size_t>(b) * a.Hkv * D;
      for (int i = lane; i < a.Hkv * D; i += 32) amax = fmaxf(amax, fabsf(load_in(src, tok + i, a.new_dtype)));
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
      constexpr bool INT8 = std::is_same<KT, int8_t>::value;
      const float scale = amax > 0.f ? __fdiv_rn(amax, INT8 ? 127.0f : 448.0f) : 1.0f;
      for (int d = lane; d < D; d += 32) {
        const float x = __fdiv_rn(load_in(src, row + d, a.new_dtype), scale);
        if constexpr (INT8)
          cache[dst + d] = static_cast<KT>(max(-127, min(127, __float2int_rn(x))));
        else
          cache[dst + d] = static_cast<KT>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
      }
      if (lane == 0) (which ? a.v_scale_w : a.k_scale_w)[slot] = scale;
    } else {
      for (int d = lane; d < D; d += 32) {
        if (a.new_dtype == PA_DTYPE_F32) {
          const float x = static_cast<const float*>(src)[row + d];
          if constexpr (std::is_same<KT, __half>::value)
            cache[dst + d] = __float2half_rn(x);
          else
            cache[dst + d] = __float2bfloat16_rn(x);
        } else {
          cache[dst + d] = static_cast<const KT*>(src)[row + d];
        }
      }
    }
  }
}

template <typename KT, int D, int RING_BYTES = kRingBytes>
struct Tile {
  static constexpr int ROWB = D * static_cast<int>(sizeof(KT));  // bytes per token row
  static constexpr int BYTES = 16 * ROWB;                          // one (block, head) tile
  static constexpr int NBOX = ROWB / 128;                          // 128-byte swizzle boxes
  static constexpr int BOXE = 128 / static_cast<int>(sizeof(KT));  // elements per box row
  // a tile two 128-byte swizzle spans wide is fetched as one 5-D box
  // (d_lo, row, d_hi, head, block): one TMA issue per tile instead of two
  static constexpr bool ONE_BOX = NBOX == 2;
  static constexpr int NS = RING_BYTES / (2 * BYTES);             // K+V stages per warp
  static constexpr int RING = NS * 2 * BYTES;                      // one warp's ring
  // shared memory of a W-warp CTA: rings [W], code scales [W][NS][32] f32,
  // full barriers [W][NS]
  static constexpr int off_sc(int W) { return W * RING; }
  static constexpr int off_bar(int W) { return off_sc(W) + W * NS * 128; }
  static constexpr int smem(int W) { return 1024 + off_bar(W) + W * NS * 8; }
  static_assert(ROWB % 128 == 0, "rows must be whole 128-byte swizzle spans");
  static_assert(NS >= 2, "stage ring too small");
  static_assert(RING >= (8 * D + 16) * 4, "a warp's ring must hold its merge state");
};

// Byte offset of 16-byte chunk `c` of row `r` inside a swizzled tile.
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return static_cast<uint32_t>((c >> 3) * 2048 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Clamp a context length to the bounds the launch can serve; flag violations.
__device__ __forceinline__ int checked_len(const DecodeArgs& a, int b, bool report) {
  int L = a.context_lens[b];
  const int cap = min(a.max_context_len, a.max_blocks * 16);
  if (L < 0 || L > cap) {
    if (report) atomicOr(&g_decode_err, PA_DEVERR_CONTEXT_LEN);
    L = max(0, min(L, cap));
  }
  return L;
}

template <typename QT>
__device__ __forceinline__ void store_out(const DecodeArgs& a, size_t idx, float v) {
  if (a.out_f32)
    static_cast<float*>(a.out)[idx] = v;
  else if constexpr (std::is_same<QT, __half>::value)
    static_cast<__half*>(a.out)[idx] = __float2half_rn(v);
  else
    static_cast<__nv_bfloat16*>(a.out)[idx] = __float2bfloat16_rn(v);
}

// ---- in-kernel split-K merge ------------------------------------------------------
// The partitions of one (sequence b, kv head g) end at different times.  Each
// writes its partial (o, m, l), makes it visible device-wide and takes a
// ticket on the pair's arrival counter; the last to arrive merges all of
// them into the G output rows at once.  The merges of early-finishing
// sequences overlap the rest of the grid, and no second kernel has to wait
// for the whole grid to end.  A counter holds {epoch, arrivals}: a launch
// counts only arrivals stamped with its own epoch, so whatever the workspace
// held before (another launch's counts, uninitialised bytes) reads as zero,
// and the last arrival puts the counter back to {epoch, 0}.

// Thread 0's ticket: true if this partition is the pair's last to arrive.
__device__ __forceinline__ bool take_ticket(const DecodeArgs& a, int b, int g, int np) {
  unsigned long long* t = a.tickets + static_cast<size_t>(b) * a.Hkv + g;
  unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(t);
  uint32_t cnt = 0;
  for (int it = 0; it < 65536; ++it) {  // bounded: at most np CTAs ever race here
    cnt = static_cast<uint32_t>(old >> 32) == a.epoch ? static_cast<uint32_t>(old) : 0u;
    const unsigned long long want = (static_cast<unsigned long long>(a.epoch) << 32) | (cnt + 1u);
    const unsigned long long prev = atomicCAS(t, old, want);
    if (prev == old) return cnt + 1u == static_cast<uint32_t>(np);
    old = prev;
  }
  atomicOr(&g_decode_err, PA_DEVERR_TIMEOUT);
  return false;
}

// One warp merges the np partitions of (b, g) into the G output rows of the
// kv head: out = sum_p w_p o_p with w_p = exp2(m_p - M) / sum_q exp2(m_q - M) l_q.
// Partials written by other CTAs are read at L2 (ld.global.cg).  `sw` is
// G * np floats of this warp's idle shared memory.  np <= 64.
template <typename QT, int D>
__device__ __forceinline__ void merge_pair(const DecodeArgs& a, int b, int g, int np, int lane, float* sw,
                                           int64_t oshift) {
  constexpr unsigned FULL = 0xffffffffu;
  constexpr int V = D / 32;  // dims per lane
  const size_t head0 = static_cast<size_t>(b) * a.Hq + static_cast<size_t>(g) * a.G;
  {  // weights: 4 lanes per head (c = lane / 4), partitions p = lane % 4, +4, ...
    const int c = lane >> 2, sub = lane & 3;
    const bool on = c < a.G;
    const size_t row = (head0 + (on ? c : 0)) * a.max_parts;
    float mv[16], lv[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int p = sub + 4 * i;
      const bool ok = on && p < np;
      mv[i] = ok ? __ldcg(a.part_m + row + p) : -INFINITY;
      lv[i] = ok ? __ldcg(a.part_l + row + p) : 0.f;
    }
    float M = -INFINITY;
#pragma unroll
    for (int i = 0; i < 16; ++i) M = fmaxf(M, mv[i]);
    M = fmaxf(M, __shfl_xor_sync(FULL, M, 1));
    M = fmaxf(M, __shfl_xor_sync(FULL, M, 2));
    float ls = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) ls += dev::ex2(mv[i] - M) * lv[i];  // exp2(-inf) = 0 past np
    ls += __shfl_xor_sync(FULL, ls, 1);
    ls += __shfl_xor_sync(FULL, ls, 2);
    const float inv = 1.f / ls;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int p = sub + 4 * i;
      if (on && p < np) sw[c * np + p] = dev::ex2(mv[i] - M) * inv;
    }
  }
  __syncwarp();
  float acc[PA_MAX_GROUP][V];
#pragma unroll
  for (int c = 0; c < PA_MAX_GROUP; ++c)
#pragma unroll
    for (int v = 0; v < V; ++v) acc[c][v] = 0.f;
  for (int p0 = 0; p0 < np; p0 += 4) {  // four partitions of every head in flight
    float x[4][PA_MAX_GROUP][V];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int c = 0; c < PA_MAX_GROUP; ++c) {
        const bool ok = c < a.G && p0 + i < np;
        const float* src = a.part_o + ((head0 + (ok ? c : 0)) * a.max_parts + p0 + i) * D + lane * V;
        if constexpr (V == 4) {
          const float4 t = ok ? __ldcg(reinterpret_cast<const float4*>(src)) : make_float4(0.f, 0.f, 0.f, 0.f);
          x[i][c][0] = t.x; x[i][c][1] = t.y; x[i][c][2] = t.z; x[i][c][3] = t.w;
        } else {
          const float2 t = ok ? __ldcg(reinterpret_cast<const float2*>(src)) : make_float2(0.f, 0.f);
          x[i][c][0] = t.x; x[i][c][1] = t.y;
        }
      }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int c = 0; c < PA_MAX_GROUP; ++c) {
        if (c < a.G && p0 + i < np) {
          const float w = sw[c * np + p0 + i];
#pragma unroll
          for (int v = 0; v < V; ++v) acc[c][v] += w * x[i][c][v];
        }
      }
  }
#pragma unroll
  for (int c = 0; c < PA_MAX_GROUP; ++c)
    if (c < a.G)
#pragma unroll
      for (int v = 0; v < V; ++v)
        store_out<QT>(a, static_cast<size_t>(static_cast<int64_t>((head0 + c) * D + lane * V + v) + oshift), acc[c][v]);
  if (lane == 0)  // ready for the next launch with this epoch (a replayed graph)
    a.tickets[static_cast<size_t>(b) * a.Hkv + g] = static_cast<unsigned long long>(a.epoch) << 32;
}

template <typename KT, typename QT, int D, int W>
__global__ void __launch_bounds__(32 * W)
    decode_main(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                const DecodeArgs a) {
  using TL = Tile<KT, D>;
  constexpr int NS = TL::NS;
  constexpr bool Q8 = sizeof(KT) == 1;  // 1-byte codes: E4M3 or INT8
  constexpr int KSTEPS = D / 16;
  constexpr int MT = D / 16;
  constexpr uint32_t STAGE_TX = 2 * TL::BYTES + (Q8 ? 128 : 0);
  constexpr bool SPLIT_P = std::is_same<QT, __nv_bfloat16>::value;
  constexpr unsigned FULL = 0xffffffffu;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = dev::smem_addr(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (sbase - raw);
  // Each warp of the CTA owns a ring, scales and barriers, and takes blocks
  // wid, wid + W, wid + 2W, ... of the item.
  const int wid = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
  const uint32_t tiles = sbase + wid * TL::RING;
  float* s_scale = reinterpret_cast<float*>(base + TL::off_sc(W)) + wid * NS * 32;
  const uint32_t bar_full = sbase + TL::off_bar(W) + wid * NS * 8;
  // Partitions are dispatched last-first (blockIdx.y = 0 is the last
  // partition): the long sequences' full partitions start early and the
  // short sequences' single small partitions fill in around them, which
  // approximates longest-first scheduling of the items.
  // Work item.  Plain grid: (sequence b, kv head g, partition p), the G
  // query heads of (b, g) as MMA columns.  Grouped grid (shared prefixes):
  // row y < pre_parts is partition pre_parts-1-y of group k's shared prefix,
  // whose columns are the G heads of every member (members x G <= 8), read
  // through member 0's table; the other rows are partitions of one member's
  // tail (blocks after the prefix).  Column c is query head g*G + c % G of
  // sequence seq0 + c / G (segment items: seq0 + member c / G of the item's
  // member list).
  int b, g, p;       // table owner (and fused-write sequence), kv head, partition of its rows
  int seq0, ncols;   // query columns
  uint32_t mlist = 0x76543210u;  // column c reads sequence seq0 + member c / G of this list (4 bits each)
  int qb = -1;       // query / output row of sequence seq0 (seq0 unless the call maps rows)
  int pseq;          // row base of this item's split-K partials and arrival counter
  int j0, L, nb;     // first block, owner's length, blocks of this item
  bool direct;       // one partition covers the rows: write the output itself
  bool write_new;    // this item reads the owner's last block (fused write)
  const int r = lane >> 2, q4 = lane & 3;
  uint32_t qf[KSTEPS][2];
  int t0, t1;        // block ids j0 + lane, j0 + 32 + lane
  auto load_q = [&]() {
    const int c = r < ncols ? r : 0;
    const int cm = static_cast<int>((mlist >> (4 * (c / a.G))) & 15u);
    const QT* qrow = static_cast<const QT*>(a.q) +
                     (static_cast<size_t>((qb >= 0 ? qb : seq0) + cm) * a.Hq + g * a.G + c % a.G) * D;
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
      if (r < ncols) {
        if constexpr (Q8) {  // permuted k order matching the register-converted K fragment
          const uint2 w = *reinterpret_cast<const uint2*>(qrow + 32 * q4 + 4 * kk);
          qf[kk][0] = w.x;
          qf[kk][1] = w.y;
        } else {
          qf[kk][0] = *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 2 * q4);
          qf[kk][1] = *reinterpret_cast<const uint32_t*>(qrow + 16 * kk + 8 + 2 * q4);
        }
      } else {
        qf[kk][0] = qf[kk][1] = 0u;
      }
    }
  };
  auto zero_rows = [&](int bz) {  // empty context: zero rows of (bz, g)
    const size_t ob = qb >= 0 && bz == seq0 ? qb : bz;
    for (int i = lane; i < a.G * D; i += 32)
      store_out<QT>(a, (ob * a.Hq + g * a.G + i / D) * D + i % D, 0.f);
  };

  // Launched as a dependent of the preceding kernel (normally the cache
  // write): everything below may read what it wrote.
  dev::grid_dependency_wait();
  if (a.seg_items) {
    // segment item: nb blocks from j0 that the nm listed members of group k
    // all hold (the owner's table row is read); every block is before each
    // listed member's last one, except in a one-member item
    const int4 it = a.seg_items[blockIdx.y];
    g = static_cast<int>(blockIdx.x);
    const int k = it.x;
    mlist = static_cast<uint32_t>(it.y);
    j0 = it.z;
    nb = it.w & 0xff;
    const int nm = (it.w >> 8) & 0xff;
    p = (it.w >> 16) & 0xffff;  // the item's partial slot
    const bool lane0 = lane == 0 && g == 0;
    if (k < 0 || k >= a.n_groups) {
      if (lane0) atomicOr(&g_decode_err, PA_DEVERR_GROUP);
      return;
    }
    const int gs0 = a.group_start[k], members = a.group_start[k + 1] - gs0;
    bool bad = gs0 < 0 || members <= 0 || gs0 + members > a.B || nm < 1 || nm > members || nm * a.G > 8 ||
               nb < 1 || nb > 64 || j0 < 0 || p >= a.max_parts;
    const int mi = lane < nm ? static_cast<int>((mlist >> (4 * lane)) & 15u) : 0;
    bad = bad || __any_sync(FULL, lane < nm && mi >= members);
    if (bad) {
      if (lane0) atomicOr(&g_decode_err, PA_DEVERR_GROUP);
      return;
    }
    seq0 = gs0;
    pseq = gs0;
    b = gs0 + static_cast<int>(mlist & 15u);  // the owner: the first listed member
    ncols = nm * a.G;
    const int Lm = lane < nm ? checked_len(a, gs0 + mi, false) : 0;
    L = __shfl_sync(FULL, Lm, 0);
    const int nblk = (L + 15) >> 4;
    direct = false;
    write_new = nm == 1 && j0 + nb == nblk;
    // a multi-member item must lie before every member's last block (that
    // block takes this step's token and is the member's own)
    const int lastb = (Lm - 1) >> 4;
    if ((nm > 1 && __any_sync(FULL, lane < nm && j0 + nb > lastb)) || j0 + nb > nblk) {
      if (lane0) atomicOr(&g_decode_err, PA_DEVERR_GROUP);
      return;
    }
    const int32_t* row = a.block_tables + static_cast<size_t>(b) * a.max_blocks + j0;
    t0 = lane < nb ? row[lane] : 0;
    t1 = lane + 32 < nb ? row[lane + 32] : 0;
    load_q();
    // every listed member must hold the same blocks here
    bool differ = false;
    for (int m = 1; m < nm; ++m) {
      const int sm = gs0 + static_cast<int>((mlist >> (4 * m)) & 15u);
      const int32_t* rm = a.block_tables + static_cast<size_t>(sm) * a.max_blocks + j0;
      differ |= (lane < nb && rm[lane] != t0) || (lane + 32 < nb && rm[lane + 32] != t1);
    }
    if (__any_sync(FULL, differ) && lane == 0) atomicOr(&g_decode_err, PA_DEVERR_GROUP);
  } else if (a.n_groups == 0) {
    // grid column (b, g, t): the q_tokens query tokens of (b, g) are
    // neighbours, so their reads of the same K/V tiles meet in L2
    const int tq = a.q_tokens;
    const int bg = static_cast<int>(blockIdx.x) / tq, t = static_cast<int>(blockIdx.x) - bg * tq;
    b = bg / a.Hkv;
    g = bg - b * a.Hkv;
    p = PA_P_ASC ? static_cast<int>(blockIdx.y) : static_cast<int>(gridDim.y) - 1 - static_cast<int>(blockIdx.y);
    seq0 = b;
    pseq = b;
    ncols = a.G;
    j0 = p * a.bpp;
    // The length, this partition's block ids (one or two per lane, read up to
    // the partition size and the row end before the length is known) and Q
    // are independent loads, so they share one memory round trip.
    const int32_t* row = a.block_tables + static_cast<size_t>(b) * a.max_blocks + j0;
    const int row_left = a.max_blocks - j0;
    t0 = (lane < a.bpp && lane < row_left) ? row[lane] : 0;
    t1 = (lane + 32 < a.bpp && lane + 32 < row_left) ? row[lane + 32] : 0;
    const bool report = lane == 0 && g == 0 && p == 0 && t == 0;
    int n = 1;
    if (a.q_start) {  // rows of a multi-token call
      const int s0 = a.q_start[b];
      n = a.q_start[b + 1] - s0;
      if (s0 < 0 || n < 0 || n > tq || s0 > a.q_rows - n) {
        if (a.q_report && report) atomicOr(&g_decode_err, PA_DEVERR_QUERY_RANGE);
        return;
      }
      if (t >= n) return;
      qb = s0 + t;
      pseq = b * tq + t;
    }
    load_q();
    L = checked_len(a, b, lane == 0 && p == 0 && t == 0);
    if (a.q_start) {
      // more query tokens than context: the early tokens have no keys
      if (n > L && a.q_report && report) atomicOr(&g_decode_err, PA_DEVERR_CONTEXT_LEN);
      L = max(0, L - n + 1 + t);  // causal: the keys up to this token's position
    }
    const int nblk = (L + 15) >> 4;
    if (j0 >= nblk) {
      if (p == 0) zero_rows(b);
      return;
    }
    nb = min(a.bpp, nblk - j0);
    direct = (nblk + a.bpp - 1) / a.bpp == 1;
    write_new = j0 + nb == nblk;
  } else {
    const int k = blockIdx.x / a.Hkv, y = static_cast<int>(blockIdx.y);
    g = blockIdx.x - k * a.Hkv;
    const int gs0 = a.group_start[k], gs1 = a.group_start[k + 1], pre = a.prefix_blocks[k];
    const int members = gs1 - gs0;
    if (gs0 < 0 || members <= 0 || gs1 > a.B || members > a.max_members) {
      if (lane == 0 && g == 0 && y == 0) atomicOr(&g_decode_err, PA_DEVERR_GROUP);
      return;
    }
    const int Lm = lane < members ? checked_len(a, gs0 + lane, g == 0 && y == a.pre_parts) : 0;
    const int E = group_prefix(pre, members, Lm, lane);
    if (y < a.pre_parts) {  // shared prefix
      p = a.pre_parts - 1 - y;
      j0 = p * a.bpp;
      if (j0 >= E) return;
      nb = min(a.bpp, E - j0);
      b = gs0;
      seq0 = gs0;
      pseq = gs0;
      ncols = members * a.G;
      L = __shfl_sync(FULL, Lm, 0);
      direct = false;
      write_new = false;
      const int32_t* row = a.block_tables + static_cast<size_t>(b) * a.max_blocks + j0;
      t0 = lane < nb ? row[lane] : 0;
      t1 = lane + 32 < nb ? row[lane + 32] : 0;
      load_q();
      // every member must hold the same blocks here
      bool differ = false;
      for (int m = 1; m < members; ++m) {
        const int32_t* rm = a.block_tables + static_cast<size_t>(gs0 + m) * a.max_blocks + j0;
        differ |= (lane < nb && rm[lane] != t0) || (lane + 32 < nb && rm[lane + 32] != t1);
      }
      if (__any_sync(FULL, differ) && lane == 0) atomicOr(&g_decode_err, PA_DEVERR_GROUP);
    } else {  // one member's tail
      const int t = y - a.pre_parts;
      const int m = t % a.max_members, pt = a.tail_parts - 1 - t / a.max_members;
      if (m >= members) return;
      b = gs0 + m;
      seq0 = b;
      pseq = b;
      ncols = a.G;
      L = __shfl_sync(FULL, Lm, m);
      const int nblk = (L + 15) >> 4, pp = (E + a.bpp - 1) / a.bpp;
      j0 = E + pt * a.bpp;
      if (j0 >= nblk) {
        if (pt == 0 && L == 0) zero_rows(b);
        return;
      }
      nb = min(a.bpp, nblk - j0);
      p = pp + pt;
      direct = pp + (nblk - E + a.bpp - 1) / a.bpp == 1;
      write_new = j0 + nb == nblk;
      const int32_t* row = a.block_tables + static_cast<size_t>(b) * a.max_blocks + j0;
      t0 = lane < nb ? row[lane] : 0;
      t1 = lane + 32 < nb ? row[lane + 32] : 0;
      load_q();
    }
  }
  // output rows are query rows: shifted when the call maps sequences to rows
  const int64_t oshift = qb >= 0 ? static_cast<int64_t>(qb - pseq) * a.Hq * D : 0;
  const bool bad = (lane < nb && (t0 < 0 || t0 >= a.num_blocks)) ||
                   (lane + 32 < nb && (t1 < 0 || t1 >= a.num_blocks));
  if (bad) {
    atomicOr(&g_decode_err, PA_DEVERR_BLOCK_RANGE);  // read a valid block instead; flagged
    if (t0 < 0 || t0 >= a.num_blocks) t0 = 0;
    if (t1 < 0 || t1 >= a.num_blocks) t1 = 0;
  }
  // This partition holds the sequence's last token: store the new row of kv
  // head g before the tile holding it is read, and make the stores visible to
  // the TMA (async proxy) reads that follow.  When that tile is not among the
  // ring's first fills (one warp, more blocks than stages), the first tiles
  // are requested before the store, so the store does not delay them.
  const bool defer_write = W == 1 && PA_EARLY_ISSUE && nb > NS;
  auto fused_write = [&]() {
    const int64_t slot = a.slot_mapping[b];
    if (slot >= static_cast<int64_t>(a.num_blocks) * 16) {
      if (lane == 0) atomicOr(&g_decode_err, PA_DEVERR_SLOT_RANGE);
    } else if (slot >= 0) {
      write_new_row<KT, D>(a, static_cast<KT*>(const_cast<void*>(a.k_cache_w)),
                           static_cast<KT*>(const_cast<void*>(a.v_cache_w)), b, g, slot, lane);
      asm volatile("fence.proxy.async.global;" ::: "memory");
    }
  };
  if (a.fuse_write && write_new && wid == 0 && !defer_write) fused_write();
  if (lane == 0) {
    dev::prefetch_tensormap(&tmK);
    dev::prefetch_tensormap(&tmV);
    for (int s = 0; s < NS; ++s) dev::mbar_init(bar_full + 8 * s, 1);
    dev::fence_barrier_init();
  }
  if constexpr (W > 1)
    __syncthreads();  // the fused row store (warp 0) precedes every warp's reads
  else
    __syncwarp();
  if (lane == 0) asm volatile("fence.proxy.async.global;" ::: "memory");

  auto block_id = [&](int j) { return __shfl_sync(FULL, j < 32 ? t0 : t1, j & 31); };
  auto issue = [&](int pb, int s) {  // lane 0 only
    const uint32_t bar = bar_full + 8 * s;
    const uint32_t kdst = tiles + s * 2 * TL::BYTES, vdst = kdst + TL::BYTES;
    dev::mbar_arrive_expect_tx(bar, STAGE_TX);
    if constexpr (TL::ONE_BOX) {
      dev::tma_load_5d(kdst, &tmK, bar, 0, 0, 0, g, pb);
      dev::tma_load_5d(vdst, &tmV, bar, 0, 0, 0, g, pb);
    } else {
#pragma unroll
      for (int bx = 0; bx < TL::NBOX; ++bx) {
        dev::tma_load_3d(kdst + bx * 2048, &tmK, bar, bx * TL::BOXE, g * 16, pb);
        dev::tma_load_3d(vdst + bx * 2048, &tmV, bar, bx * TL::BOXE, g * 16, pb);
      }
    }
    if constexpr (Q8) {
      dev::bulk_load(dev::smem_addr(s_scale + s * 32), a.k_scale + static_cast<size_t>(pb) * 16, 64, bar);
      dev::bulk_load(dev::smem_addr(s_scale + s * 32 + 16), a.v_scale + static_cast<size_t>(pb) * 16, 64, bar);
    }
  };
#pragma unroll
  for (int i = 0; i < NS; ++i) {
    const int j = wid + i * W;
    const int pb = block_id(min(j, 63));
    if (j < nb && lane == 0) issue(pb, i);
  }
  if (a.fuse_write && write_new && defer_write) {
    fused_write();  // before any refill: the last block is requested by a refill
    __syncwarp();
  }
  // Every CTA of this grid has started once all of them pass here, so the
  // merge kernel may be scheduled now: its CTAs become resident as slots
  // free up and wait (griddepcontrol.wait) for this grid's completion
  // instead of being launched after it.
  dev::grid_launch_dependents();
  float o[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const float sl2 = a.scale_log2;

  for (int i = 0;; ++i) {
    const int j = wid + i * W;  // this warp's i-th block of the item
    if (j >= nb) break;
    const int s = i % NS;
    const int next_pb = block_id(min(j + NS * W, 63));  // block id of the refill (all lanes shuffle)
    if (!dev::mbar_wait_bounded(bar_full + 8 * s, (i / NS) & 1)) {
      if (lane == 0) atomicOr(&g_decode_err, PA_DEVERR_TIMEOUT);
      // let this warp's other copies in flight land (bounded), then stop
      for (int i2 = i + 1; i2 < i + NS && wid + i2 * W < nb; ++i2)
        dev::mbar_wait_bounded(bar_full + 8 * (i2 % NS), (i2 / NS) & 1, 100000000ull);
      break;
    }
    const uint32_t kb = tiles + s * 2 * TL::BYTES, vb = kb + TL::BYTES;
    const int nvalid = min(16, L - (j0 + j) * 16);

    // ---- K and V fragments -> registers, then refill the stage ---------------
    uint32_t kf[KSTEPS][4], vf[MT][4];
    float c_r = sl2, c_r8 = sl2, vs_r = 1.f, vs_r8 = 1.f;
    if constexpr (Q8) {
      const uint4 x0 = dev::lds128(kb + swz(r, 2 * q4));
      const uint4 x1 = dev::lds128(kb + swz(r, 2 * q4 + 1));
      const uint4 y0 = dev::lds128(kb + swz(r + 8, 2 * q4));
      const uint4 y1 = dev::lds128(kb + swz(r + 8, 2 * q4 + 1));
      const int tt = 2 * q4;
      uint4 X = dev::lds128(vb + swz(tt, r));
      uint4 Y = dev::lds128(vb + swz(tt + 1, r));
      uint4 Z = dev::lds128(vb + swz(tt + 8, r));
      uint4 Wq = dev::lds128(vb + swz(tt + 9, r));
      c_r *= s_scale[s * 32 + r];
      c_r8 *= s_scale[s * 32 + r + 8];
      vs_r = r < nvalid ? s_scale[s * 32 + 16 + r] : 0.f;  // a stale scale past the context may be NaN
      vs_r8 = r + 8 < nvalid ? s_scale[s * 32 + 16 + r + 8] : 0.f;
      if (nvalid < 16) {  // rows past the context: weight 0, and their stale bytes must not be NaN codes
        if (tt >= nvalid) X = make_uint4(0, 0, 0, 0);
        if (tt + 1 >= nvalid) Y = make_uint4(0, 0, 0, 0);
        if (tt + 8 >= nvalid) Z = make_uint4(0, 0, 0, 0);
        if (tt + 9 >= nvalid) Wq = make_uint4(0, 0, 0, 0);
      }
      const uint32_t wr[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      const uint32_t wr8[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
      for (int kk = 0; kk < KSTEPS; ++kk) {
        kf[kk][0] = wr[kk];
        kf[kk][1] = wr8[kk];
      }
      const uint32_t xw[4] = {X.x, X.y, X.z, X.w}, yw[4] = {Y.x, Y.y, Y.z, Y.w};
      const uint32_t zw[4] = {Z.x, Z.y, Z.z, Z.w}, ww[4] = {Wq.x, Wq.y, Wq.z, Wq.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        vf[i][0] = xw[i];
        vf[i][1] = yw[i];
        vf[i][2] = zw[i];
        vf[i][3] = ww[i];
      }
    } else {
      const int krow = (lane & 7) + ((lane >> 3) & 1) * 8;
      const int vrow = (lane & 7) + (lane >> 4) * 8;
#pragma unroll
      for (int kk = 0; kk < KSTEPS; ++kk) dev::ldmatrix_x4(kf[kk], kb + swz(krow, 2 * kk + (lane >> 4)));
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) dev::ldmatrix_x4_trans(vf[mt], vb + swz(vrow, 2 * mt + ((lane >> 3) & 1)));
      if (nvalid < 16) {
        // V rows past the context get weight 0, but 0 * NaN is NaN: clear the
        // halves of tokens >= nvalid (a0/a1: tokens 2q4, 2q4+1; a2/a3: +8)
        const int t0 = 2 * q4;
        const uint32_t m0 = (t0 < nvalid ? 0xFFFFu : 0u) | (t0 + 1 < nvalid ? 0xFFFF0000u : 0u);
        const uint32_t m8 = (t0 + 8 < nvalid ? 0xFFFFu : 0u) | (t0 + 9 < nvalid ? 0xFFFF0000u : 0u);
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          vf[mt][0] &= m0;
          vf[mt][1] &= m0;
          vf[mt][2] &= m8;
          vf[mt][3] &= m8;
        }
      }
    }
    __syncwarp();
    if (lane == 0 && j + NS * W < nb) {
      dev::fence_proxy_async_smem();
      issue(next_pb, s);
    }

    // ---- S^T = K . Q^T -----------------------------------------------------
    float sacc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
      uint32_t af[4];
      if constexpr (Q8) {
        dev::code8x4_to<KT, QT>(kf[kk][0], af[0], af[2]);
        dev::code8x4_to<KT, QT>(kf[kk][1], af[1], af[3]);
      } else {
        af[0] = kf[kk][0];
        af[1] = kf[kk][1];
        af[2] = kf[kk][2];
        af[3] = kf[kk][3];
      }
      dev::Mma<QT>::run(sacc, af, qf[kk][0], qf[kk][1]);
    }

    // ---- online softmax over this block's 16 tokens ---------------------------
    const bool v_r = r < nvalid, v_r8 = r + 8 < nvalid;
    const float x0 = v_r ? sacc[0] * c_r : -INFINITY;
    const float x1 = v_r ? sacc[1] * c_r : -INFINITY;
    const float x2 = v_r8 ? sacc[2] * c_r8 : -INFINITY;
    const float x3 = v_r8 ? sacc[3] * c_r8 : -INFINITY;
    float bm0 = fmaxf(x0, x2), bm1 = fmaxf(x1, x3);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      bm0 = fmaxf(bm0, __shfl_xor_sync(FULL, bm0, off));
      bm1 = fmaxf(bm1, __shfl_xor_sync(FULL, bm1, off));
    }
    // The reference max of each head moves only when a tile's max exceeds it
    // by more than 8 (log2 units; one warp vote moves every head at once).
    // Otherwise the weights exp2(x - m) stay <= 2^8 against the old reference
    // and O and l keep their scale, so most tiles skip the rescale.  The
    // first tile always moves it (m = -inf).
    float al0 = 1.f, al1 = 1.f;
    if (__any_sync(FULL, bm0 > m0 + 8.f || bm1 > m1 + 8.f)) {
      const float mn0 = fmaxf(m0, bm0), mn1 = fmaxf(m1, bm1);
      al0 = dev::ex2(m0 - mn0);
      al1 = dev::ex2(m1 - mn1);
      m0 = mn0;
      m1 = mn1;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        o[mt][0] *= al0;
        o[mt][1] *= al1;
        o[mt][2] *= al0;
        o[mt][3] *= al1;
      }
    }
    float p0 = dev::ex2(x0 - m0), p1 = dev::ex2(x1 - m1), p2 = dev::ex2(x2 - m0), p3 = dev::ex2(x3 - m1);

    uint32_t ph_r, ph_r8, pl_r = 0, pl_r8 = 0;
    if constexpr (Q8) {
      l0 = l0 * al0 + (p0 + p2);
      l1 = l1 * al1 + (p1 + p3);
      p0 *= vs_r;
      p1 *= vs_r;
      p2 *= vs_r8;
      p3 *= vs_r8;
    }
    ph_r = dev::pack2<QT>(p0, p1);
    ph_r8 = dev::pack2<QT>(p2, p3);
    if constexpr (SPLIT_P) {
      const float2 h_r = dev::unpack2<QT>(ph_r), h_r8 = dev::unpack2<QT>(ph_r8);
      pl_r = dev::pack2<QT>(p0 - h_r.x, p1 - h_r.y);
      pl_r8 = dev::pack2<QT>(p2 - h_r8.x, p3 - h_r8.y);
      if constexpr (!Q8) {
        l0 = l0 * al0 + (p0 + p2);
        l1 = l1 * al1 + (p1 + p3);
      }
    } else if constexpr (!Q8) {
      // normalise with the rounded weights actually used in the PV product
      const float2 h_r = dev::unpack2<QT>(ph_r), h_r8 = dev::unpack2<QT>(ph_r8);
      l0 = l0 * al0 + (h_r.x + h_r8.x);
      l1 = l1 * al1 + (h_r.y + h_r8.y);
    }
    const uint32_t bh0 = dev::movmatrix_trans(ph_r), bh1 = dev::movmatrix_trans(ph_r8);
    uint32_t bl0 = 0, bl1 = 0;
    if constexpr (SPLIT_P) {
      bl0 = dev::movmatrix_trans(pl_r);
      bl1 = dev::movmatrix_trans(pl_r8);
    }

    // ---- O^T += V^T . P^T ------------------------------------------------------
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      uint32_t af[4];
      if constexpr (Q8) {
        const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
        const uint32_t xy = dev::prmt(vf[mt >> 1][0], vf[mt >> 1][1], sel);
        const uint32_t zv = dev::prmt(vf[mt >> 1][2], vf[mt >> 1][3], sel);
        dev::code8x4_to<KT, QT>(xy, af[0], af[1]);
        dev::code8x4_to<KT, QT>(zv, af[2], af[3]);
      } else {
        af[0] = vf[mt][0];
        af[1] = vf[mt][1];
        af[2] = vf[mt][2];
        af[3] = vf[mt][3];
      }
      dev::Mma<QT>::run(o[mt], af, bh0, bh1);
      if constexpr (SPLIT_P) dev::Mma<QT>::run(o[mt], af, bl0, bl1);
    }
  }

  // ---- output: this item's (o, m, l) or, for one partition, o / l -----------------
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(FULL, l0, off);
    l1 += __shfl_xor_sync(FULL, l1, off);
  }
  const int hA = 2 * q4, hB = 2 * q4 + 1;
  if constexpr (W > 1) {
    // Merge the W warps' softmax states through their (now idle) rings.
    float* ow = reinterpret_cast<float*>(base + wid * TL::RING);  // [8][D], then m[8], l[8]
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      int d_r, d_r8;
      if constexpr (Q8) {
        d_r = 16 * r + 2 * mt;
        d_r8 = d_r + 1;
      } else {
        d_r = 16 * mt + r;
        d_r8 = d_r + 8;
      }
      ow[hA * D + d_r] = o[mt][0];
      ow[hB * D + d_r] = o[mt][1];
      ow[hA * D + d_r8] = o[mt][2];
      ow[hB * D + d_r8] = o[mt][3];
    }
    if (lane < 4) {
      ow[8 * D + hA] = m0;
      ow[8 * D + hB] = m1;
      ow[8 * D + 8 + hA] = l0;
      ow[8 * D + 8 + hB] = l1;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < ncols * D; idx += 32 * W) {
      const int h = idx / D, d = idx - h * D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < W; ++w)
        M = fmaxf(M, reinterpret_cast<const float*>(base + w * TL::RING)[8 * D + h]);
      float acc = 0.f, ls = 0.f;
#pragma unroll
      for (int w = 0; w < W; ++w) {
        const float* ov = reinterpret_cast<const float*>(base + w * TL::RING);
        const float f = dev::ex2(ov[8 * D + h] - M);  // 0 for a warp without blocks
        acc += f * ov[h * D + d];
        ls += f * ov[8 * D + 8 + h];
      }
      const size_t head =
          static_cast<size_t>(pseq + static_cast<int>((mlist >> (4 * (h / a.G))) & 15u)) * a.Hq + g * a.G + h % a.G;
      if (direct) {
        store_out<QT>(a, static_cast<size_t>(static_cast<int64_t>(head * D + d) + oshift), acc / ls);
      } else {
        const size_t rowp = head * a.max_parts + p;
        a.part_o[rowp * D + d] = acc;
        if (d == 0) {
          a.part_m[rowp] = M;
          a.part_l[rowp] = ls;
        }
      }
    }
    if (!direct && a.tickets) {
      __shared__ int s_last;
      const int np = (((L + 15) >> 4) + a.bpp - 1) / a.bpp;
      __threadfence();  // this CTA's partial is visible before its ticket
      __syncthreads();  // every warp is done with the rings
      if (threadIdx.x == 0) s_last = take_ticket(a, pseq, g, np);
      __syncthreads();
      if (s_last && wid == 0) {
        __threadfence();  // the other partitions' partials, published before their tickets
        merge_pair<QT, D>(a, pseq, g, np, lane, reinterpret_cast<float*>(base), oshift);
      }
    }
    return;
  }
  const bool okA = hA < ncols, okB = hB < ncols;
  const int mA = static_cast<int>((mlist >> (4 * (hA / a.G))) & 15u), mB = static_cast<int>((mlist >> (4 * (hB / a.G))) & 15u);
  const size_t headA = static_cast<size_t>(pseq + mA) * a.Hq + g * a.G + hA % a.G;
  const size_t headB = static_cast<size_t>(pseq + mB) * a.Hq + g * a.G + hB % a.G;
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) {
    int d_r, d_r8;
    if constexpr (Q8) {
      d_r = 16 * r + 2 * mt;
      d_r8 = d_r + 1;
    } else {
      d_r = 16 * mt + r;
      d_r8 = d_r + 8;
    }
    if (direct) {
      const int64_t oA = static_cast<int64_t>(headA * D) + oshift, oB = static_cast<int64_t>(headB * D) + oshift;
      if (okA) {
        store_out<QT>(a, static_cast<size_t>(oA + d_r), o[mt][0] / l0);
        store_out<QT>(a, static_cast<size_t>(oA + d_r8), o[mt][2] / l0);
      }
      if (okB) {
        store_out<QT>(a, static_cast<size_t>(oB + d_r), o[mt][1] / l1);
        store_out<QT>(a, static_cast<size_t>(oB + d_r8), o[mt][3] / l1);
      }
    } else {
      const size_t rowA = headA * a.max_parts + p, rowB = headB * a.max_parts + p;
      if (okA) {
        a.part_o[rowA * D + d_r] = o[mt][0];
        a.part_o[rowA * D + d_r8] = o[mt][2];
      }
      if (okB) {
        a.part_o[rowB * D + d_r] = o[mt][1];
        a.part_o[rowB * D + d_r8] = o[mt][3];
      }
    }
  }
  if (!direct && lane < 4) {
    if (okA) {
      a.part_m[headA * a.max_parts + p] = m0;
      a.part_l[headA * a.max_parts + p] = l0;
    }
    if (okB) {
      a.part_m[headB * a.max_parts + p] = m1;
      a.part_l[headB * a.max_parts + p] = l1;
    }
  }
  if (!direct && a.tickets) {
    const int np = (((L + 15) >> 4) + a.bpp - 1) / a.bpp;
    __threadfence();  // this warp's partial is visible before its ticket
    __syncwarp();
    const bool last = __shfl_sync(FULL, lane == 0 ? take_ticket(a, pseq, g, np) : false, 0);
    if (last) {
      __threadfence();  // the other partitions' partials, published before their tickets
      merge_pair<QT, D>(a, pseq, g, np, lane, reinterpret_cast<float*>(base), oshift);
    }
  }
}

// Merge n partition rows of one query head (rows row0 .. row0 + n - 1) with
// log-sum-exp weights into output row `orow`.  Partitions are taken 32 at a
// time: lane i holds partition i's (m, l), so the chunk's weights are known
// after one round trip; every lane then reads its D/32 dims of the chunk's
// partial rows 16 partitions at a time, all loads of a batch in flight
// together.  Chunks merge online (running max).  `mv`, `lv` are the first
// chunk's (m, l) as the caller loaded them; lanes past n are reset here, so
// stale scratch never enters a sum.
template <typename QT, int D>
__device__ __forceinline__ void merge_rows(const DecodeArgs& a, size_t row0, int n, float mv, float lv,
                                           size_t orow, int lane) {
  constexpr unsigned FULL = 0xffffffffu;
  constexpr int CH = 32;      // partitions per chunk (one per lane)
  constexpr int RB = 16;      // partial rows per load batch
  constexpr int V = D / 32;   // dims per lane (4 or 2)
  const float* po = a.part_o + row0 * D + lane * V;
  float M = -INFINITY, ls = 0.f, acc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = 0.f;
  for (int c0 = 0; c0 < n; c0 += CH) {
    const int cn = min(CH, n - c0);
    if (c0 > 0) {
      mv = lane < cn ? a.part_m[row0 + c0 + lane] : -INFINITY;
      lv = lane < cn ? a.part_l[row0 + c0 + lane] : 0.f;
    }
    if (lane >= cn) {
      mv = -INFINITY;
      lv = 0.f;
    }
    float cm = mv;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) cm = fmaxf(cm, __shfl_xor_sync(FULL, cm, off));
    const float nm = fmaxf(M, cm);
    const float rescale = dev::ex2(M - nm);  // 0 on the first chunk
    M = nm;
    const float w = dev::ex2(mv - nm);       // this lane's partition weight
    float wl = w * lv;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) wl += __shfl_xor_sync(FULL, wl, off);
    ls = ls * rescale + wl;
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] *= rescale;
    for (int i0 = 0; i0 < cn; i0 += RB) {
      float x[RB][V];
#pragma unroll
      for (int i = 0; i < RB; ++i) {
        if (i0 + i < cn) {
          if constexpr (V == 4) {
            const float4 t = *reinterpret_cast<const float4*>(po + static_cast<size_t>(c0 + i0 + i) * D);
            x[i][0] = t.x; x[i][1] = t.y; x[i][2] = t.z; x[i][3] = t.w;
          } else {
            const float2 t = *reinterpret_cast<const float2*>(po + static_cast<size_t>(c0 + i0 + i) * D);
            x[i][0] = t.x; x[i][1] = t.y;
          }
        }
      }
#pragma unroll
      for (int i = 0; i < RB; ++i) {
        const float wi = __shfl_sync(FULL, w, (i0 + i) & 31);
        if (i0 + i < cn) {
#pragma unroll
          for (int v = 0; v < V; ++v) acc[v] += wi * x[i][v];
        }
      }
    }
  }
#pragma unroll
  for (int v = 0; v < V; ++v) store_out<QT>(a, orow * D + lane * V + v, acc[v] / ls);
}

// Merge the partitions of each (sequence, query head).  One warp per query
// head and 32 dims, G warps per CTA (grid: sequence and kv head -- and query
// token when the call maps rows -- by D / 32 dim slices).  Partitions are
// taken 32 at a time, lane p holding partition p's (m, l) and every lane
// reading its dim of all 32 partial rows, so one round trip brings a chunk:
// the first chunk's loads go out together with the context length (the
// workspace holds max_parts rows, and rows past the split are masked before
// use: they may hold stale bytes).  Chunks merge online (running max).
template <typename QT, int D>
__global__ void __launch_bounds__(32 * PA_MAX_GROUP) decode_reduce(const DecodeArgs a) {
  constexpr unsigned FULL = 0xffffffffu;
  constexpr int CH = 32;  // partitions per chunk: one per lane
  const int tq = a.q_tokens;
  const int bg = static_cast<int>(blockIdx.x) / tq, t = static_cast<int>(blockIdx.x) - bg * tq;
  const int b = bg / a.Hkv, g = bg - b * a.Hkv;
  const int h = g * a.G + static_cast<int>(threadIdx.x >> 5), lane = threadIdx.x & 31;
  const int d = static_cast<int>(blockIdx.y) * 32 + lane;  // this lane's dim
  dev::grid_dependency_wait();  // partials of decode_main are complete and visible
  int ob = b, pseq = b, n = 1;
  if (a.q_start) {  // rows of a multi-token call: as decode_main maps them
    const int s0 = a.q_start[b];
    n = a.q_start[b + 1] - s0;
    if (s0 < 0 || n < 0 || n > tq || s0 > a.q_rows - n || t >= n) return;
    ob = s0 + t;
    pseq = b * tq + t;
  }
  const size_t row0 = (static_cast<size_t>(pseq) * a.Hq + h) * a.max_parts;
  const int pre = min(CH, a.max_parts);
  float mv = lane < pre ? __ldcg(a.part_m + row0 + lane) : -INFINITY;
  float lv = lane < pre ? __ldcg(a.part_l + row0 + lane) : 0.f;
  float x[CH];
  if (PA_MERGE_SPEC) {
#pragma unroll
    for (int p = 0; p < CH; ++p) x[p] = p < pre ? __ldcg(a.part_o + (row0 + p) * D + d) : 0.f;
  }
  int L = checked_len(a, b, false);
  if (a.q_start) L = max(0, L - n + 1 + t);
  const int nblk = (L + 15) >> 4;
  const int nparts = (nblk + a.bpp - 1) / a.bpp;
  if (nparts <= 1) return;  // written by decode_main (zero rows included)
  float M = -INFINITY, ls = 0.f, acc = 0.f;
  for (int c0 = 0; c0 < nparts; c0 += CH) {
    const int cn = min(CH, nparts - c0);
    if (c0 > 0) {
      mv = lane < cn ? __ldcg(a.part_m + row0 + c0 + lane) : -INFINITY;
      lv = lane < cn ? __ldcg(a.part_l + row0 + c0 + lane) : 0.f;
    }
    if (c0 > 0 || !PA_MERGE_SPEC) {
#pragma unroll
      for (int p = 0; p < CH; ++p) x[p] = p < cn ? __ldcg(a.part_o + (row0 + c0 + p) * D + d) : 0.f;
    }
    if (lane >= cn) {
      mv = -INFINITY;
      lv = 0.f;
    }
#pragma unroll
    for (int p = 0; p < CH; ++p)
      if (p >= cn) x[p] = 0.f;  // rows past the split: stale, never weighed
    float cm = mv;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) cm = fmaxf(cm, __shfl_xor_sync(FULL, cm, off));
    const float nm = fmaxf(M, cm);
    const float rescale = dev::ex2(M - nm);  // 0 on the first chunk
    M = nm;
    const float w = lane < cn ? dev::ex2(mv - nm) : 0.f;  // this lane's partition weight
    float wl = w * lv;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) wl += __shfl_xor_sync(FULL, wl, off);
    ls = ls * rescale + wl;
    acc *= rescale;
#pragma unroll
    for (int p = 0; p < CH; ++p) acc += __shfl_sync(FULL, w, p) * x[p];
  }
  store_out<QT>(a, (static_cast<size_t>(ob) * a.Hq + h) * D + d, acc / ls);
}

// The grouped form: one CTA per (group k, member m, kv head g).  A member's
// partitions are its shared-prefix partitions (written by the group's
// prefix items) followed by its tail partitions.
template <typename QT, int D>
__global__ void __launch_bounds__(32 * PA_MAX_GROUP) decode_reduce_grouped(const DecodeArgs a) {
  const int g = blockIdx.x % a.Hkv, km = blockIdx.x / a.Hkv;
  const int m = km % a.max_members, k = km / a.max_members;
  const int h = g * a.G + static_cast<int>(threadIdx.x >> 5), lane = threadIdx.x & 31;
  dev::grid_dependency_wait();  // partials of decode_main are complete and visible
  const int gs0 = a.group_start[k], gs1 = a.group_start[k + 1], pre = a.prefix_blocks[k];
  const int members = gs1 - gs0;
  if (gs0 < 0 || members <= 0 || gs1 > a.B || members > a.max_members || m >= members) return;
  const int Lm = lane < members ? checked_len(a, gs0 + lane, false) : 0;
  const int E = group_prefix(pre, members, Lm, lane);
  const int b = gs0 + m, L = __shfl_sync(0xffffffffu, Lm, m);
  const int nblk = (L + 15) >> 4;
  if (nblk == 0) return;  // zero rows written by decode_main
  const int nparts = (E + a.bpp - 1) / a.bpp + (nblk - E + a.bpp - 1) / a.bpp;
  if (nparts <= 1) return;
  const size_t row0 = (static_cast<size_t>(b) * a.Hq + h) * a.max_parts;
  const float mv = lane < nparts ? a.part_m[row0 + lane] : -INFINITY;
  const float lv = lane < nparts ? a.part_l[row0 + lane] : 0.f;
  merge_rows<QT, D>(a, row0, nparts, mv, lv, static_cast<size_t>(b) * a.Hq + h, lane);
}

// The segment form: one CTA per (sequence b, kv head g), a warp per query
// head.  Sequence b is member m of group k; its partials are the slots of the
// items that list it.  The items are the caller's input, so each warp finds
// those slots before the decode kernel's partials are complete (it is
// launched early as a programmatic dependent): lane j ends up holding the
// j-th one.  After the wait the partials merge with log-sum-exp weights in
// item order, in one round trip when there are at most 32 (else chunk by
// chunk).  A member no item lists gets zero rows.
template <typename QT, int D>
__global__ void __launch_bounds__(32 * PA_MAX_GROUP) decode_reduce_segments(const DecodeArgs a) {
  constexpr unsigned FULL = 0xffffffffu;
  constexpr int V = D / 32;
  const int b = static_cast<int>(blockIdx.x) / a.Hkv, g = static_cast<int>(blockIdx.x) - b * a.Hkv;
  const int h = g * a.G + static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
  if (a.group_start[0] > b || a.group_start[a.n_groups] <= b) return;  // in no group: not served
  int lo = 0, hi = a.n_groups;  // the group k with group_start[k] <= b < group_start[k + 1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (a.group_start[mid] <= b) lo = mid; else hi = mid;
  }
  const int m = b - a.group_start[lo];
  // item i (lane i of a chunk) lists member m: its slot, else -1
  auto slot_of = [&](int i) {
    if (i >= a.n_seg_items) return -1;
    const int4 it = a.seg_items[i];
    const int nm = (it.w >> 8) & 0xff, slot = (it.w >> 16) & 0xffff;
    if (it.x != lo || slot >= a.max_parts) return -1;
    for (int j = 0; j < nm && j < 8; ++j)
      if (static_cast<int>((static_cast<uint32_t>(it.y) >> (4 * j)) & 15u) == m) return slot;
    return -1;
  };
  int mine = -1, count = 0;
  for (int c0 = 0; c0 < a.n_seg_items; c0 += 32) {
    const int s = slot_of(c0 + lane);
    const unsigned vm = __ballot_sync(FULL, s >= 0);
    const int k = lane - count;  // this lane takes the chunk's k-th listed slot
    const bool take = k >= 0 && k < __popc(vm);
    const int got = __shfl_sync(FULL, s, take ? static_cast<int>(__fns(vm, 0, k + 1)) : lane);
    if (take) mine = got;
    count += __popc(vm);
  }
  dev::grid_dependency_wait();  // partials of decode_main are complete and visible
  const size_t row0 = (static_cast<size_t>(b) * a.Hq + h) * a.max_parts;
  const float* po = a.part_o + row0 * D + lane * V;
  float M = -INFINITY, ls = 0.f, acc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = 0.f;
  const int chunks = count <= 32 ? 1 : (a.n_seg_items + 31) / 32;
  for (int c = 0; c < chunks && count > 0; ++c) {
    const int slot = count <= 32 ? mine : slot_of(32 * c + lane);
    const bool valid = slot >= 0;
    const float mv = valid ? __ldcg(a.part_m + row0 + slot) : -INFINITY;
    const float lv = valid ? __ldcg(a.part_l + row0 + slot) : 0.f;
    float cm = mv;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) cm = fmaxf(cm, __shfl_xor_sync(FULL, cm, off));
    const float nm_ = fmaxf(M, cm);
    if (nm_ == -INFINITY) continue;  // nothing of this member so far
    const float rescale = dev::ex2(M - nm_);  // 0 on its first partials
    M = nm_;
    const float w = valid ? dev::ex2(mv - nm_) : 0.f;
    float wl = w * lv;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) wl += __shfl_xor_sync(FULL, wl, off);
    ls = ls * rescale + wl;
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] *= rescale;
    const unsigned vm = __ballot_sync(FULL, valid);
    for (int q0 = 0; q0 < 32; q0 += 8) {  // valid rows 8 lanes at a time, their loads in flight together
      if (!((vm >> q0) & 0xffu)) continue;
      float x[8][V];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int sj = __shfl_sync(FULL, slot, q0 + j);
        if ((vm >> (q0 + j)) & 1u) {
          const float* src = po + static_cast<size_t>(sj) * D;
          if constexpr (V == 4) {
            const float4 t = __ldcg(reinterpret_cast<const float4*>(src));
            x[j][0] = t.x; x[j][1] = t.y; x[j][2] = t.z; x[j][3] = t.w;
          } else {
            const float2 t = __ldcg(reinterpret_cast<const float2*>(src));
            x[j][0] = t.x; x[j][1] = t.y;
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float wj = __shfl_sync(FULL, w, q0 + j);
        if ((vm >> (q0 + j)) & 1u) {
#pragma unroll
          for (int v = 0; v < V; ++v) acc[v] += wj * x[j][v];
        }
      }
    }
  }
  const float inv = ls > 0.f ? 1.f / ls : 0.f;
#pragma unroll
  for (int v = 0; v < V; ++v) store_out<QT>(a, (static_cast<size_t>(b) * a.Hq + h) * D + lane * V + v, acc[v] * inv);
}

// ---- host side -------------------------------------------------------------------
template <typename KT, int D>
pa_status make_map(CUtensorMap* m, const void* cache, int Hkv, int num_blocks, CUtensorMapDataType dt) {
  using TL = Tile<KT, D>;
  static_assert(TL::ONE_BOX == (TL::ROWB == 256), "the 5-D box covers exactly two swizzle spans");
  return make_kv_map(m, cache, Hkv, num_blocks, TL::ROWB, static_cast<int>(sizeof(KT)), dt, "pa_decode");
}

// A fresh stamp for each launch's arrival counters (never 0 or all ones, the
// values zeroed and 0xFF-filled memory would show).
uint32_t next_epoch() {
  static std::atomic<uint32_t> counter{0};
  uint32_t v;
  do {
    v = counter.fetch_add(1u, std::memory_order_relaxed) + 1u;
  } while (v == 0u || v == 0xFFFFFFFFu);
  return v;
}

template <typename KT, typename QT, int D>
pa_status launch_t(const DecodeLaunch& l, CUtensorMapDataType dt, cudaStream_t stream) {
  using TL = Tile<KT, D>;
  CUtensorMap tmK, tmV;
  pa_status st = make_map<KT, D>(&tmK, l.k_cache, l.Hkv, l.num_blocks, dt);
  if (st != PA_OK) return st;
  st = make_map<KT, D>(&tmV, l.v_cache, l.Hkv, l.num_blocks, dt);
  if (st != PA_OK) return st;

  DecodeArgs a;
  a.q = l.q;
  a.block_tables = l.block_tables;
  a.context_lens = l.context_lens;
  a.k_scale = l.k_scale;
  a.v_scale = l.v_scale;
  a.out = l.out;
  const int tq = l.q_start ? l.q_tokens : 1;  // grid columns per (sequence, kv head)
  const size_t rows = static_cast<size_t>(l.B) * tq * l.Hq * l.plan.max_parts;
  // partials: a split, or segment items (whose rows are always partials)
  a.part_o = l.plan.max_parts > 1 || l.segments ? static_cast<float*>(l.workspace) : nullptr;
  a.part_m = a.part_o ? a.part_o + rows * D : nullptr;
  a.part_l = a.part_m ? a.part_m + rows : nullptr;
  a.B = l.B;
  a.Hq = l.Hq;
  a.Hkv = l.Hkv;
  a.G = l.Hq / l.Hkv;
  a.max_blocks = l.max_blocks;
  a.num_blocks = l.num_blocks;
  a.max_context_len = l.max_context_len;
  a.bpp = l.plan.blocks_per_part;
  a.max_parts = l.plan.max_parts;
  a.scale_log2 = l.scale * 1.4426950408889634f;
  a.out_f32 = l.out_dtype == PA_DTYPE_F32;
  a.k_new = l.k_new;
  a.v_new = l.v_new;
  a.slot_mapping = l.slot_mapping;
  a.k_cache_w = const_cast<void*>(l.k_cache);
  a.v_cache_w = const_cast<void*>(l.v_cache);
  a.k_scale_w = const_cast<float*>(l.k_scale);
  a.v_scale_w = const_cast<float*>(l.v_scale);
  a.new_dtype = l.new_dtype;
  a.fuse_write = l.slot_mapping != nullptr;
  a.group_start = l.group_start;
  a.prefix_blocks = l.prefix_blocks;
  a.n_groups = l.n_groups;
  a.max_members = l.max_members;
  a.pre_parts = l.plan.pre_parts;
  a.tail_parts = l.plan.tail_parts;
  a.seg_items = l.segments ? reinterpret_cast<const int4*>(l.seg_items) : nullptr;
  a.n_seg_items = l.n_seg_items;
  a.q_start = l.q_start;
  a.q_rows = l.q_rows;
  a.q_tokens = tq;
  a.q_report = l.q_start ? l.q_report : 0;
  a.tickets = nullptr;
  a.epoch = 0;
  if (l.plan.ticket_offset) {  // after the partials: the arrival counters
    a.tickets = reinterpret_cast<unsigned long long*>(static_cast<uint8_t*>(l.workspace) + l.plan.ticket_offset);
    a.epoch = next_epoch();
  }

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(PA_ERR_CUDA, "pa_decode: no CUDA device");
  if (dev >= kMaxDevices) return fail(PA_ERR_UNSUPPORTED, "pa_decode: device index %d", dev);
  static std::once_flag once[kMaxDevices];  // raise the smem limit once per device
  static cudaError_t setup_err[kMaxDevices];
  std::call_once(once[dev], [dev] {
    cudaError_t e = cudaFuncSetAttribute(decode_main<KT, QT, D, 1>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, TL::smem(1));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(decode_main<KT, QT, D, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               TL::smem(2));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(decode_main<KT, QT, D, 4>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               TL::smem(4));
    setup_err[dev] = e;
  });
  if (setup_err[dev] != cudaSuccess)
    return fail(PA_ERR_CUDA, "pa_decode: %s", cudaGetErrorString(setup_err[dev]));

  if (l.segments) {
    // one CTA per (segment item, kv head), then the merge of each member's items
    cudaError_t e = cudaSuccess;
    if (l.n_seg_items > 0) {
      // kv heads fastest: the items (listed longest first) are dispatched in order
      const dim3 sgrid(static_cast<unsigned>(l.Hkv), static_cast<unsigned>(l.n_seg_items));
      const int W = l.plan.item_warps;
      if (W == 4)
        e = launch_dependent(decode_main<KT, QT, D, 4>, sgrid, dim3(128), TL::smem(4), stream, tmK, tmV, a);
      else if (W == 2)
        e = launch_dependent(decode_main<KT, QT, D, 2>, sgrid, dim3(64), TL::smem(2), stream, tmK, tmV, a);
      else
        e = launch_dependent(decode_main<KT, QT, D, 1>, sgrid, dim3(32), TL::smem(1), stream, tmK, tmV, a);
    }
    if (e == cudaSuccess)
      e = launch_dependent(decode_reduce_segments<QT, D>, dim3(static_cast<unsigned>(l.B * l.Hkv)),
                           dim3(static_cast<unsigned>(32 * a.G)), 0, stream, a);
    if (e == cudaSuccess) e = cudaGetLastError();
    if (e != cudaSuccess) return fail(PA_ERR_CUDA, "pa_decode launch: %s", cudaGetErrorString(e));
    return PA_OK;
  }
  const bool grouped = l.n_groups > 0;
  const dim3 grid = grouped ? dim3(static_cast<unsigned>(l.n_groups * l.Hkv),
                                   static_cast<unsigned>(l.plan.pre_parts + l.max_members * l.plan.tail_parts))
                            : dim3(static_cast<unsigned>(l.B * l.Hkv * tq), static_cast<unsigned>(l.plan.max_parts));
  const int W = l.plan.item_warps;
  cudaError_t e;
  if (W == 4)
    e = launch_dependent(decode_main<KT, QT, D, 4>, grid, dim3(128), TL::smem(4), stream, tmK, tmV, a);
  else if (W == 2)
    e = launch_dependent(decode_main<KT, QT, D, 2>, grid, dim3(64), TL::smem(2), stream, tmK, tmV, a);
  else
    e = launch_dependent(decode_main<KT, QT, D, 1>, grid, dim3(32), TL::smem(1), stream, tmK, tmV, a);
  if (e == cudaSuccess && grouped)
    e = launch_dependent(decode_reduce_grouped<QT, D>,
                         dim3(static_cast<unsigned>(l.n_groups * l.max_members * l.Hkv)),
                         dim3(static_cast<unsigned>(32 * a.G)), 0, stream, a);
  else if (e == cudaSuccess && l.plan.max_parts > 1 && !a.tickets)
    e = launch_dependent(decode_reduce<QT, D>, dim3(static_cast<unsigned>(l.B * l.Hkv * tq), D / 32),
                         dim3(static_cast<unsigned>(32 * a.G)), 0, stream, a);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "pa_decode launch: %s", cudaGetErrorString(e));
  return PA_OK;
}

}  // namespace

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

pa_status make_kv_map(CUtensorMap* m, const void* cache, int Hkv, int num_blocks, int row_bytes,
                      int elem_bytes, CUtensorMapDataType dt, const char* what, bool one_box) {
  auto fn = encode_fn();
  if (!fn) return fail(PA_ERR_CUDA, "%s: cuTensorMapEncodeTiled unavailable", what);
  if (row_bytes != 128 && row_bytes != 256) return fail(PA_ERR_UNSUPPORTED, "%s: row of %d bytes", what, row_bytes);
  const cuuint64_t boxe = static_cast<cuuint64_t>(128 / elem_bytes);  // elements per 128-byte span
  const cuuint64_t rowb = static_cast<cuuint64_t>(row_bytes);
  CUresult r;
  if (row_bytes == 256 && one_box) {
    const cuuint64_t dims[5] = {boxe, 16, 2, static_cast<cuuint64_t>(Hkv), static_cast<cuuint64_t>(num_blocks)};
    const cuuint64_t strides[4] = {rowb, 128, rowb * 16, rowb * 16 * Hkv};
    const cuuint32_t box[5] = {static_cast<cuuint32_t>(boxe), 16, 2, 1, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    r = fn(m, dt, 5, const_cast<void*>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    const cuuint64_t dims[3] = {rowb / elem_bytes, static_cast<cuuint64_t>(16) * Hkv,
                                static_cast<cuuint64_t>(num_blocks)};
    const cuuint64_t strides[2] = {rowb, rowb * 16 * Hkv};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(boxe), 16, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    r = fn(m, dt, 3, const_cast<void*>(cache), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "%s: tensor map encode failed (%d)", what, static_cast<int>(r));
  return PA_OK;
}

pa_status launch_decode(const DecodeLaunch& l, void* stream_ptr) {
  cudaStream_t st = static_cast<cudaStream_t>(stream_ptr);
  if (l.kv_dtype == PA_DTYPE_F16) {
    if (l.D == 64) return launch_t<__half, __half, 64>(l, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, st);
    return launch_t<__half, __half, 128>(l, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, st);
  }
  if (l.kv_dtype == PA_DTYPE_BF16) {
    if (l.D == 64) return launch_t<__nv_bfloat16, __nv_bfloat16, 64>(l, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, st);
    return launch_t<__nv_bfloat16, __nv_bfloat16, 128>(l, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, st);
  }
  // 1-byte codes (E4M3 as uint8_t, INT8 as int8_t), head_dim 128 (checked by
  // the caller); the tensor map moves raw bytes either way
  if (l.kv_dtype == PA_DTYPE_INT8) {
    if (l.q_dtype == PA_DTYPE_F16) return launch_t<int8_t, __half, 128>(l, CU_TENSOR_MAP_DATA_TYPE_UINT8, st);
    return launch_t<int8_t, __nv_bfloat16, 128>(l, CU_TENSOR_MAP_DATA_TYPE_UINT8, st);
  }
  if (l.q_dtype == PA_DTYPE_F16) return launch_t<uint8_t, __half, 128>(l, CU_TENSOR_MAP_DATA_TYPE_UINT8, st);
  return launch_t<uint8_t, __nv_bfloat16, 128>(l, CU_TENSOR_MAP_DATA_TYPE_UINT8, st);
}

pa_status read_errors_decode(uint32_t* flags, bool clear) {
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_decode_err, sizeof(v));
  if (e == cudaSuccess && clear) {
    const uint32_t z = 0;
    e = cudaMemcpyToSymbol(g_decode_err, &z, sizeof(z));
  }
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "pa_device_errors: %s", cudaGetErrorString(e));
  *flags = v;
  return PA_OK;
}

}  // namespace pa
