// Paged attention for several query tokens per sequence (chunked prefill,
// speculative verification) for sm_103a.
//
// What it computes ("大模型推理引擎优化：KV Cache 与连续批处理", section 4.1:
// a long prompt is split into chunks that run beside decode steps;
// "LLM推理引擎深度实战：从PagedAttention到分布式推理部署", section 6.1: the large
// model checks the draft's tokens in one pass): sequence b brings n_b query
// tokens, the last n_b of its L_b-token context (their K/V already written to
// the cache).  Query token i sits at position L_b - n_b + i and attends to
// keys 0 .. L_b - n_b + i through the sequence's block table -- the causal
// mask, so a prompt run chunk by chunk gives the rows of one pass.
//
// Design (GB300):
// * The query rows of one (sequence b, kv head g) are the pairs (token i,
//   head h of the group), row = i * G + h, so every row of a tile reads the
//   same K/V.  A CTA takes 64 rows (four consumer warps x 16 rows) and one
//   partition of the context: grid (b * Hkv + g) * QT + row tile, partition.
//   Row tiles of one (b, g) are adjacent in the grid, so their K/V reads of
//   the same partition meet in L2 and HBM serves each tile once.
// * A fifth warp produces: it streams the partition's (block, kv head) K and
//   V tiles (4 KB each at D = 128, 16-bit) into a ring of stages with TMA
//   (128-byte swizzle) and refills a stage when every consumer warp has
//   released it (full / empty mbarrier pairs, all waits bounded).
// * Consumers run flash-attention style on tensor cores (mma.m16n8k16, fp32
//   accumulate): S[16 rows x 16 tokens] = Q[16 x D] . K^T with Q held in
//   registers and K via ldmatrix, a causal / length mask per (row, token),
//   online softmax in fp32 (exp2, log2 e folded into the scale), then
//   O[16 x D] += P[16 x 16] . V with P taken straight from the score
//   registers and V via ldmatrix.trans.  bf16 P is carried as hi + lo bf16
//   parts (rounding error ~2^-17), f16 P once, normalised by the rounded
//   weights.
// * FP8 E4M3 and INT8 caches (1-byte codes, head_dim 128; this kernel
//   only): the stage also carries the block's 16 K and 16 V per-token scales
//   (two bulk copies on the same barrier).  Codes are converted exactly to
//   the query's 16-bit type in registers.  For Q . K^T the head dimension is
//   visited in a permuted order (lane q4 takes dims 32 q4 .. 32 q4 + 31, four
//   per k-step, Q loaded the same way), so a lane reads 32 contiguous bytes of
//   a key row; the K scale multiplies the score.  For P . V a lane reads one
//   32-bit word (4 dims) of each of its four token rows and byte-permutes
//   them into the B fragments of four column tiles, so the output columns
//   come out permuted (undone at the store); the V scale multiplies p.
// * A row whose keys fit one partition is written directly; otherwise each
//   partition writes (o, m, l) and prefill_reduce merges them with
//   log-sum-exp weights, launched as a programmatic dependent.
#include <cudaTypedefs.h>

#include <mutex>

#include "device_common.cuh"
#include "kv_map.h"
#include "pa_internal.h"

namespace pa {
namespace {

__device__ uint32_t g_prefill_err;

constexpr int kConsumers = 4;                   // consumer warps, 16 rows each
constexpr int kRows = 16 * kConsumers;          // query rows per CTA
constexpr int kThreads = 32 * (kConsumers + 1);  // + the producer warp
constexpr int kRingBytes = 64 * 1024;           // K/V stages of one CTA
#ifndef PA_PREFILL_MINB
#define PA_PREFILL_MINB 2  // resident CTAs per SM the register budget is cut for
#endif
constexpr int kMaxDevices = 64;
constexpr unsigned FULL = 0xffffffffu;

struct PrefillArgs {
  const void* q;
  const int32_t* q_start;
  const int32_t* block_tables;
  const int32_t* context_lens;
  void* out;
  float* part_o;
  float* part_m;
  float* part_l;
  int32_t B, T, Hq, Hkv, G, max_blocks, num_blocks, max_context_len, max_q_len;
  int32_t QT;  // row tiles per (sequence, kv head): ceil(max_q_len * G / tile rows)
  int32_t bpp, max_parts;
  float scale_log2;
  int32_t out_f32;
  const float* k_scale;  // FP8 / INT8 caches: [num_blocks][16] per-token scales
  const float* v_scale;
  int32_t skip_single;   // sequences with one query token are served by the decode kernel
};

// Shared memory of prefill_main: the K/V stage ring, full and empty
// barriers, and for 1-byte codes each stage's 16 K and 16 V scales.
template <typename KT, int D>
struct PTile {
  static constexpr bool Q8 = sizeof(KT) == 1;
  static constexpr int ROWB = D * static_cast<int>(sizeof(KT));  // bytes per token row
  static constexpr int TB = 16 * ROWB;                             // one (block, head) tile
  static constexpr int NS = kRingBytes / (2 * TB);                 // K+V stages
  static constexpr int SCALES = Q8 ? NS * 128 : 0;
  static constexpr int SMEM = 1024 + NS * 2 * TB + NS * 16 + SCALES;
  static_assert(ROWB == 128 || ROWB == 256, "rows of one or two 128-byte swizzle spans");
  static_assert(NS >= 2, "stage ring too small");
};

// Byte offset of 16-byte chunk `c` of row `r` inside a swizzled tile laid
// out as [c / 8][16 rows][128 bytes].
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return static_cast<uint32_t>((c >> 3) * 2048 + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// The sequence's query range and context length, clamped to what the
// launch can serve; violations are flagged once per sequence.
struct SeqView {
  int qs, n, L;
};
__device__ __forceinline__ SeqView seq_view(const PrefillArgs& a, int b, bool report) {
  SeqView v;
  v.qs = a.q_start[b];
  v.n = a.q_start[b + 1] - v.qs;
  v.L = a.context_lens[b];
  if (v.qs < 0 || v.n < 0 || v.n > a.max_q_len || v.qs > a.T - v.n) {
    if (report) atomicOr(&g_prefill_err, PA_DEVERR_QUERY_RANGE);
    v.qs = 0;
    v.n = 0;
  }
  const int cap = min(a.max_context_len, a.max_blocks * 16);
  if (v.L < 0 || v.L > cap) {
    if (report) atomicOr(&g_prefill_err, PA_DEVERR_CONTEXT_LEN);
    v.L = max(0, min(v.L, cap));
  }
  if (v.n > v.L && report) atomicOr(&g_prefill_err, PA_DEVERR_CONTEXT_LEN);  // early tokens get no keys
  if (a.skip_single && v.n == 1) v.n = 0;  // its row is the decode kernel's
  return v;
}

template <typename T>
__device__ __forceinline__ void store_pair(const PrefillArgs& a, size_t idx, float x, float y) {
  if (a.out_f32)
    *reinterpret_cast<float2*>(static_cast<float*>(a.out) + idx) = make_float2(x, y);
  else
    *reinterpret_cast<uint32_t*>(static_cast<T*>(a.out) + idx) = dev::pack2<T>(x, y);
}

template <typename KT, typename T, int D>
__global__ void __launch_bounds__(kThreads, PA_PREFILL_MINB)
    prefill_main(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 const PrefillArgs a) {
  using TL = PTile<KT, D>;
  constexpr bool Q8 = TL::Q8;
  static_assert(!Q8 || D == 128, "1-byte codes at head_dim 128");
  constexpr int NS = TL::NS;
  constexpr int KSTEPS = D / 16;
  constexpr int DT = D / 8;  // 8-wide column tiles of O
  constexpr bool SPLIT_P = std::is_same<T, __nv_bfloat16>::value;
  constexpr uint32_t STAGE_TX = 2 * TL::TB + (Q8 ? 128 : 0);

  extern __shared__ uint8_t smem_raw[];
  const uint32_t ring = (dev::smem_addr(smem_raw) + 1023u) & ~1023u;
  const uint32_t bar_full = ring + NS * 2 * TL::TB, bar_empty = bar_full + NS * 8;
  const uint32_t scales = bar_empty + NS * 8;  // Q8: stage s holds K scales [16], V scales [16]
  const float* s_scale = reinterpret_cast<const float*>(smem_raw + (scales - dev::smem_addr(smem_raw)));

  const int wid = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
  const int qt = static_cast<int>(blockIdx.x) % a.QT, bg = static_cast<int>(blockIdx.x) / a.QT;
  const int b = bg / a.Hkv, g = bg - b * a.Hkv;
  // last partition first: long rows' early partitions start early and short
  // work fills in around them (as in the decode kernel)
  const int p = static_cast<int>(gridDim.y) - 1 - static_cast<int>(blockIdx.y);

  dev::grid_dependency_wait();  // the cache write before this kernel is visible
  const SeqView sv = seq_view(a, b, g == 0 && qt == 0 && p == 0 && threadIdx.x == 0);
  const int nrows = sv.n * a.G;
  const int R0 = qt * kRows;
  if (R0 >= nrows) return;
  const int shift = sv.L - sv.n;  // position of query token i is shift + i
  const int j0 = p * a.bpp;
  // key blocks this CTA needs (its last row sees the most keys)
  const int pos_cta = shift + (min(R0 + kRows, nrows) - 1) / a.G;
  const int nb = min(a.bpp, (pos_cta + 16) / 16 - j0);  // <= 0 when pos_cta < 16 * j0

  // rows of warp w: [R0 + 16w, R0 + 16w + 16) within nrows; the warp takes
  // part when it has a row with at least one key in this partition
  auto warp_last_pos = [&](int w) { return shift + (min(R0 + 16 * w + 16, nrows) - 1) / a.G; };
  auto warp_active = [&](int w) { return R0 + 16 * w < nrows && warp_last_pos(w) >= 16 * j0; };
  int n_active = 0;
#pragma unroll
  for (int w = 0; w < kConsumers; ++w) n_active += warp_active(w) ? 1 : 0;

  if (nb <= 0 || n_active == 0) {
    // Nothing to read.  Partition 0 still owns the output of rows without
    // keys (a sequence with more query tokens than context): zero rows.
    if (p == 0 && wid < kConsumers) {
      const int row0 = R0 + 16 * wid;
      for (int k = lane; k < 16 * D; k += 32) {
        const int rr = row0 + k / D;
        if (rr < nrows && shift + rr / a.G < 0) {
          const size_t head = static_cast<size_t>(sv.qs + rr / a.G) * a.Hq + g * a.G + rr % a.G;
          if (a.out_f32)
            static_cast<float*>(a.out)[head * D + k % D] = 0.f;
          else
            static_cast<uint16_t*>(a.out)[head * D + k % D] = 0;  // +0 in f16 and in bf16
        }
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < NS; ++s) {
      dev::mbar_init(bar_full + 8 * s, 1);
      dev::mbar_init(bar_empty + 8 * s, static_cast<uint32_t>(n_active));
    }
    dev::fence_barrier_init();
  }
  __syncthreads();

  if (wid == kConsumers) {
    // ---- producer warp: block ids 32 at a time, lane 0 issues the copies ----
    const int32_t* row = a.block_tables + static_cast<size_t>(b) * a.max_blocks + j0;
    int issued = 0;
    bool ok = true;
    if (lane == 0) {
      dev::prefetch_tensormap(&tmK);
      dev::prefetch_tensormap(&tmV);
    }
    for (int c = 0; c < nb && ok; c += 32) {
      int id = c + lane < nb ? row[c + lane] : 0;
      if (id < 0 || id >= a.num_blocks) {
        atomicOr(&g_prefill_err, PA_DEVERR_BLOCK_RANGE);  // read block 0 instead; flagged
        id = 0;
      }
      const int cnt = min(32, nb - c);
      for (int k = 0; k < cnt; ++k) {
        const int pb = __shfl_sync(FULL, id, k);
        if (lane == 0 && ok) {
          const int i = c + k, s = i % NS;
          if (i >= NS && !dev::mbar_wait_bounded(bar_empty + 8 * s, ((i / NS) - 1) & 1)) {
            atomicOr(&g_prefill_err, PA_DEVERR_TIMEOUT);
            ok = false;
          } else {
            // consumers' reads of this stage precede the refill's writes
            dev::fence_proxy_async_smem();
            const uint32_t bar = bar_full + 8 * s, kdst = ring + s * 2 * TL::TB, vdst = kdst + TL::TB;
            dev::mbar_arrive_expect_tx(bar, STAGE_TX);
            if constexpr (TL::ROWB == 256) {
              dev::tma_load_5d(kdst, &tmK, bar, 0, 0, 0, g, pb);
              dev::tma_load_5d(vdst, &tmV, bar, 0, 0, 0, g, pb);
            } else {
              dev::tma_load_3d(kdst, &tmK, bar, 0, g * 16, pb);
              dev::tma_load_3d(vdst, &tmV, bar, 0, g * 16, pb);
            }
            if constexpr (Q8) {
              dev::bulk_load(scales + s * 128, a.k_scale + static_cast<size_t>(pb) * 16, 64, bar);
              dev::bulk_load(scales + s * 128 + 64, a.v_scale + static_cast<size_t>(pb) * 16, 64, bar);
            }
            issued = i + 1;
          }
        }
        ok = __shfl_sync(FULL, ok ? 1 : 0, 0) != 0;
      }
    }
    // no copy may still be landing when the CTA exits
    if (lane == 0)
      for (int i = max(0, issued - NS); i < issued; ++i)
        dev::mbar_wait_bounded(bar_full + 8 * (i % NS), (i / NS) & 1, 100000000ull);
    return;
  }

  // ---- consumer warp ----------------------------------------------------------------
  dev::grid_launch_dependents();
  const int row0 = R0 + 16 * wid;
  const int r = lane >> 2, q4 = lane & 3;
  const int rowA = row0 + r, rowB = rowA + 8;
  const bool hasA = rowA < nrows, hasB = rowB < nrows;
  const int posA = hasA ? shift + rowA / a.G : -1;
  const int posB = hasB ? shift + rowB / a.G : -1;
  const size_t headA = hasA ? static_cast<size_t>(sv.qs + rowA / a.G) * a.Hq + g * a.G + rowA % a.G : 0;
  const size_t headB = hasB ? static_cast<size_t>(sv.qs + rowB / a.G) * a.Hq + g * a.G + rowB % a.G : 0;
  const bool active = warp_active(wid);
  const int last_pos = row0 < nrows ? warp_last_pos(wid) : -1;

  float o[DT][4];
#pragma unroll
  for (int t = 0; t < DT; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
  float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;

  if (active) {
    // Q rows as the A operand (row = query row, k = head dim)
    uint32_t qf[KSTEPS][4];
    {
      const T* qa = static_cast<const T*>(a.q) + headA * D;
      const T* qb = static_cast<const T*>(a.q) + headB * D;
#pragma unroll
      for (int kk = 0; kk < KSTEPS; ++kk) {
        if constexpr (Q8) {  // permuted head dims: lane q4 takes 32 q4 + 4 kk .. + 3
          const uint2 wa = hasA ? *reinterpret_cast<const uint2*>(qa + 32 * q4 + 4 * kk) : make_uint2(0u, 0u);
          const uint2 wb = hasB ? *reinterpret_cast<const uint2*>(qb + 32 * q4 + 4 * kk) : make_uint2(0u, 0u);
          qf[kk][0] = wa.x;
          qf[kk][1] = wb.x;
          qf[kk][2] = wa.y;
          qf[kk][3] = wb.y;
        } else {
          const int c = 16 * kk + 2 * q4;
          qf[kk][0] = hasA ? *reinterpret_cast<const uint32_t*>(qa + c) : 0u;
          qf[kk][1] = hasB ? *reinterpret_cast<const uint32_t*>(qb + c) : 0u;
          qf[kk][2] = hasA ? *reinterpret_cast<const uint32_t*>(qa + c + 8) : 0u;
          qf[kk][3] = hasB ? *reinterpret_cast<const uint32_t*>(qb + c + 8) : 0u;
        }
      }
    }
    const float sl2 = a.scale_log2;
    const int krow = (lane & 7) + (lane >> 4) * 8, kcol = (lane >> 3) & 1;
    const int vrow = (lane & 7) + ((lane >> 3) & 1) * 8, vcol = lane >> 4;

    for (int i = 0; i < nb; ++i) {
      const int s = i % NS;
      if (!dev::mbar_wait_bounded(bar_full + 8 * s, (i / NS) & 1)) {
        if (lane == 0) atomicOr(&g_prefill_err, PA_DEVERR_TIMEOUT);
        break;
      }
      const int tok0 = (j0 + i) * 16;
      if (tok0 <= last_pos) {
        // The block holding the context's end (its rows past the end may
        // hold stale bytes, NaN included) runs a copy of the body that masks
        // them out of P . V; every other block runs the copy without masks.
        auto block = [&](auto tail_c) {
          constexpr bool TAIL = decltype(tail_c)::value;
          const uint32_t kb = ring + s * 2 * TL::TB, vb = kb + TL::TB;
          // ---- S = Q . K^T over this block's 16 tokens (two 8-token tiles) -----
          // even and odd k-steps accumulate separately: four independent MMA
          // chains instead of two, summed once
          float sc[2][4], sd[2][4];
#pragma unroll
          for (int k = 0; k < 4; ++k) sc[0][k] = sc[1][k] = sd[0][k] = sd[1][k] = 0.f;
          if constexpr (Q8) {
            // key rows r (tile 0) and r + 8 (tile 1): bytes 32 q4 .. 32 q4 + 31
            const uint4 x0 = dev::lds128(kb + swz(r, 2 * q4)), x1 = dev::lds128(kb + swz(r, 2 * q4 + 1));
            const uint4 y0 = dev::lds128(kb + swz(r + 8, 2 * q4)), y1 = dev::lds128(kb + swz(r + 8, 2 * q4 + 1));
            const uint32_t wx[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
            const uint32_t wy[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
              float(&acc0)[4] = (kk & 1) ? sd[0] : sc[0];
              float(&acc1)[4] = (kk & 1) ? sd[1] : sc[1];
              uint32_t bx0, bx1, by0, by1;
              dev::code8x4_to<KT, T>(wx[kk], bx0, bx1);
              dev::code8x4_to<KT, T>(wy[kk], by0, by1);
              dev::Mma<T>::run(acc0, qf[kk], bx0, bx1);
              dev::Mma<T>::run(acc1, qf[kk], by0, by1);
            }
          } else {
#pragma unroll
            for (int kk = 0; kk < KSTEPS; ++kk) {
              uint32_t kf[4];
              dev::ldmatrix_x4(kf, kb + swz(krow, 2 * kk + kcol));
              float(&acc0)[4] = (kk & 1) ? sd[0] : sc[0];
              float(&acc1)[4] = (kk & 1) ? sd[1] : sc[1];
              dev::Mma<T>::run(acc0, qf[kk], kf[0], kf[1]);
              dev::Mma<T>::run(acc1, qf[kk], kf[2], kf[3]);
            }
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            sc[0][k] += sd[0][k];
            sc[1][k] += sd[1][k];
          }
          // ---- causal / length mask, online softmax ------------------------------
          float x[2][4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int t = tok0 + nt * 8 + 2 * q4 + e;
              const float c = Q8 ? sl2 * s_scale[s * 32 + nt * 8 + 2 * q4 + e] : sl2;  // K scale of token t
              x[nt][e] = t <= posA ? sc[nt][e] * c : -INFINITY;
              x[nt][2 + e] = t <= posB ? sc[nt][2 + e] * c : -INFINITY;
            }
          float bA = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
          float bB = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
          bA = fmaxf(bA, __shfl_xor_sync(FULL, bA, 1));
          bB = fmaxf(bB, __shfl_xor_sync(FULL, bB, 1));
          bA = fmaxf(bA, __shfl_xor_sync(FULL, bA, 2));
          bB = fmaxf(bB, __shfl_xor_sync(FULL, bB, 2));
          const float nA = fmaxf(mA, bA), nB = fmaxf(mB, bB);
          // a row without any key so far keeps m = -inf; its weights are 0
          const float zA = nA == -INFINITY ? 0.f : nA, zB = nB == -INFINITY ? 0.f : nB;
          const float alA = exp2f(mA - zA), alB = exp2f(mB - zB);
          mA = nA;
          mB = nB;
          float pv[2][4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            pv[nt][0] = exp2f(x[nt][0] - zA);
            pv[nt][1] = exp2f(x[nt][1] - zA);
            pv[nt][2] = exp2f(x[nt][2] - zB);
            pv[nt][3] = exp2f(x[nt][3] - zB);
          }
          if constexpr (Q8) {
            // l sums the weights; V's per-token scale rides on p (0 past the
            // context, where a stale scale may be NaN)
            lA = lA * alA + (pv[0][0] + pv[0][1] + pv[1][0] + pv[1][1]);
            lB = lB * alB + (pv[0][2] + pv[0][3] + pv[1][2] + pv[1][3]);
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
              for (int e = 0; e < 2; ++e) {
                const int tt = nt * 8 + 2 * q4 + e;
                const float vs = tok0 + tt < sv.L ? s_scale[s * 32 + 16 + tt] : 0.f;
                pv[nt][e] *= vs;
                pv[nt][2 + e] *= vs;
              }
          }
          // P as the A operand: rows r / r + 8, tokens 2q4.. of each 8-token tile
          uint32_t ph[4], pl[4] = {0u, 0u, 0u, 0u};
          ph[0] = dev::pack2<T>(pv[0][0], pv[0][1]);
          ph[1] = dev::pack2<T>(pv[0][2], pv[0][3]);
          ph[2] = dev::pack2<T>(pv[1][0], pv[1][1]);
          ph[3] = dev::pack2<T>(pv[1][2], pv[1][3]);
          if constexpr (SPLIT_P) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float2 h = dev::unpack2<T>(ph[k]);
              const int nt = k >> 1, e = (k & 1) * 2;
              pl[k] = dev::pack2<T>(pv[nt][e] - h.x, pv[nt][e + 1] - h.y);
            }
            if constexpr (!Q8) {
              lA = lA * alA + (pv[0][0] + pv[0][1] + pv[1][0] + pv[1][1]);
              lB = lB * alB + (pv[0][2] + pv[0][3] + pv[1][2] + pv[1][3]);
            }
          } else if constexpr (!Q8) {
            // normalise with the rounded weights the PV product uses
            const float2 h0 = dev::unpack2<T>(ph[0]), h1 = dev::unpack2<T>(ph[1]);
            const float2 h2 = dev::unpack2<T>(ph[2]), h3 = dev::unpack2<T>(ph[3]);
            lA = lA * alA + (h0.x + h0.y + h2.x + h2.y);
            lB = lB * alB + (h1.x + h1.y + h3.x + h3.y);
          }
          // ---- O = O * alpha + P . V ---------------------------------------------
          // V rows past the context get weight 0, but 0 * NaN is NaN: masks for
          // the halves of tokens past it (b0b1: tokens 2q4, 2q4+1; b2b3: +8)
          uint32_t m0 = 0xFFFFFFFFu, m8 = 0xFFFFFFFFu;
          uint32_t m0x = 0xFFFFFFFFu, m0y = 0xFFFFFFFFu, m8x = 0xFFFFFFFFu, m8y = 0xFFFFFFFFu;  // 1-byte rows
          if constexpr (TAIL) {
            const int t0 = tok0 + 2 * q4;
            m0 = (t0 < sv.L ? 0xFFFFu : 0u) | (t0 + 1 < sv.L ? 0xFFFF0000u : 0u);
            m8 = (t0 + 8 < sv.L ? 0xFFFFu : 0u) | (t0 + 9 < sv.L ? 0xFFFF0000u : 0u);
            m0x = t0 < sv.L ? 0xFFFFFFFFu : 0u;
            m0y = t0 + 1 < sv.L ? 0xFFFFFFFFu : 0u;
            m8x = t0 + 8 < sv.L ? 0xFFFFFFFFu : 0u;
            m8y = t0 + 9 < sv.L ? 0xFFFFFFFFu : 0u;
          }
          if constexpr (Q8) {
            // Column tile 4 mm + c holds, in this lane's column slot, dim
            // 4 (r + 8 mm) + c: one word at that offset from each of the lane's
            // token rows 2q4, 2q4+1 (first B register) and 2q4+8, 2q4+9 (second)
#pragma unroll
            for (int mm = 0; mm < 4; ++mm) {
              const uint32_t off = 4u * static_cast<uint32_t>(r & 3);
              const int ch = (r >> 2) + 2 * mm;
              uint32_t X = dev::lds32(vb + swz(2 * q4, ch) + off), Y = dev::lds32(vb + swz(2 * q4 + 1, ch) + off);
              uint32_t Z = dev::lds32(vb + swz(2 * q4 + 8, ch) + off), W = dev::lds32(vb + swz(2 * q4 + 9, ch) + off);
              if constexpr (TAIL) {
                X &= m0x;
                Y &= m0y;
                Z &= m8x;
                W &= m8y;
              }
#pragma unroll
              for (int cp = 0; cp < 2; ++cp) {  // dims c = 2 cp, 2 cp + 1
                const uint32_t sel = cp ? 0x7362u : 0x5140u;
                const uint32_t xy = dev::prmt(X, Y, sel), zw = dev::prmt(Z, W, sel);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const int ct = 4 * mm + 2 * cp + h;
                  const uint32_t b0 = dev::code8x2_to<KT, T>(static_cast<uint16_t>(h ? xy >> 16 : xy & 0xffffu));
                  const uint32_t b1 = dev::code8x2_to<KT, T>(static_cast<uint16_t>(h ? zw >> 16 : zw & 0xffffu));
                  float* oo = o[ct];
                  oo[0] *= alA;
                  oo[1] *= alA;
                  oo[2] *= alB;
                  oo[3] *= alB;
                  dev::Mma<T>::run(o[ct], ph, b0, b1);
                  if constexpr (SPLIT_P) dev::Mma<T>::run(o[ct], pl, b0, b1);
                }
              }
            }
          } else {
#pragma unroll
            for (int t2 = 0; t2 < D / 16; ++t2) {
              uint32_t vf[4];
              dev::ldmatrix_x4_trans(vf, vb + swz(vrow, 2 * t2 + vcol));
              if constexpr (TAIL) {
                vf[0] &= m0;
                vf[1] &= m8;
                vf[2] &= m0;
                vf[3] &= m8;
              }
#pragma unroll
              for (int h = 0; h < 2; ++h) {
                float* oo = o[2 * t2 + h];
                oo[0] *= alA;
                oo[1] *= alA;
                oo[2] *= alB;
                oo[3] *= alB;
                dev::Mma<T>::run(o[2 * t2 + h], ph, vf[2 * h], vf[2 * h + 1]);
                if constexpr (SPLIT_P) dev::Mma<T>::run(o[2 * t2 + h], pl, vf[2 * h], vf[2 * h + 1]);
              }
            }
          }
        };
        if (tok0 + 16 > sv.L)
          block(std::true_type{});
        else
          block(std::false_type{});
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * s);  // stage s may be refilled
    }
    lA += __shfl_xor_sync(FULL, lA, 1);
    lB += __shfl_xor_sync(FULL, lB, 1);
    lA += __shfl_xor_sync(FULL, lA, 2);
    lB += __shfl_xor_sync(FULL, lB, 2);
  }

  // ---- output --------------------------------------------------------------------------
  // Row with position pos needs ceil(ceil((pos + 1) / 16) / bpp) partitions:
  // one -> written here as o / l (partition 0); more -> partial (o, m, l).
  auto parts_of = [&](int pos) { return ((pos + 16) / 16 + a.bpp - 1) / a.bpp; };
  // pair t (0 .. DT-1) of this lane's row values: its first output dim and
  // the two values.  16-bit: column tile t, dims 8 t + 2 q4 (+1).  1-byte
  // codes: tile 4 mm + c holds dim 32 mm + 8 q4 + 4 e + c in slot e, so pair
  // t = 4 mm + jp is dims 32 mm + 8 q4 + 2 jp (+1).
  auto pair_dim = [&](int t) { return Q8 ? 32 * (t >> 2) + 8 * q4 + 2 * (t & 3) : 8 * t + 2 * q4; };
  auto pair_val = [&](int t, int half) {
    if constexpr (Q8) {
      const int c0 = 4 * (t >> 2) + 2 * (t & 1), e = 2 * half + ((t >> 1) & 1);
      return make_float2(o[c0][e], o[c0 + 1][e]);
    } else {
      return make_float2(o[t][2 * half], o[t][2 * half + 1]);
    }
  };
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const bool has = half ? hasB : hasA;
    const int pos = half ? posB : posA;
    const size_t head = half ? headB : headA;
    const float l = half ? lB : lA, m = half ? mB : mA;
    if (!has) continue;
    if (pos < 0) {  // no keys at all: a zero row, from partition 0
      if (p == 0)
#pragma unroll
        for (int t = 0; t < DT; ++t) store_pair<T>(a, head * D + 8 * t + 2 * q4, 0.f, 0.f);
      continue;
    }
    const int np = parts_of(pos);
    if (p >= np) continue;
    if (np == 1) {
      const float inv = 1.f / l;
#pragma unroll
      for (int t = 0; t < DT; ++t) {
        const float2 v = pair_val(t, half);
        store_pair<T>(a, head * D + pair_dim(t), v.x * inv, v.y * inv);
      }
    } else {
      const size_t prow = head * a.max_parts + p;
      float* po = a.part_o + prow * D;
#pragma unroll
      for (int t = 0; t < DT; ++t) *reinterpret_cast<float2*>(po + pair_dim(t)) = pair_val(t, half);
      if (q4 == 0) {
        a.part_m[prow] = m;
        a.part_l[prow] = l;
      }
    }
  }
}

// Merge the partitions of each (query token, head) row whose keys span more
// than one partition: log-sum-exp weights, partitions taken 16 at a time
// (lane i holds partition i's (m, l); each lane holds D/32 dims of the
// partial rows).  One warp per row, kReduceRows rows per CTA; a row finds
// its sequence by binary search over q_start.
constexpr int kReduceRows = 8;

template <typename T, int D>
__global__ void __launch_bounds__(32 * kReduceRows) prefill_reduce(const PrefillArgs a) {
  constexpr int CH = 16;
  constexpr int V = D / 32;
  const int lane = static_cast<int>(threadIdx.x & 31);
  const int64_t row = static_cast<int64_t>(blockIdx.x) * kReduceRows + (threadIdx.x >> 5);
  dev::grid_dependency_wait();  // partials of prefill_main are complete and visible
  if (row >= static_cast<int64_t>(a.T) * a.Hq) return;
  const int t = static_cast<int>(row / a.Hq), h = static_cast<int>(row - static_cast<int64_t>(t) * a.Hq);
  // sequence b with q_start[b] <= t < q_start[b + 1] (last such b; empty sequences skipped)
  int lo = 0, hi = a.B;  // invariant: q_start[lo] <= t, answer in [lo, hi)
  if (a.q_start[0] > t) return;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (a.q_start[mid] <= t) lo = mid; else hi = mid;
  }
  const int b = lo;
  const SeqView sv = seq_view(a, b, false);
  const int i = t - sv.qs;
  if (i < 0 || i >= sv.n) return;  // a token outside every (valid) sequence
  const int pos = sv.L - sv.n + i;
  if (pos < 0) return;
  const int nparts = ((pos + 16) / 16 + a.bpp - 1) / a.bpp;
  if (nparts <= 1) return;  // written by prefill_main
  const size_t head = static_cast<size_t>(t) * a.Hq + h;
  const size_t row0 = head * a.max_parts;
  const float* po = a.part_o + row0 * D + lane * V;
  float M = -INFINITY, ls = 0.f, acc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = 0.f;
  for (int c0 = 0; c0 < nparts; c0 += CH) {
    const int n = min(CH, nparts - c0);
    const float mv = lane < n ? a.part_m[row0 + c0 + lane] : -INFINITY;
    const float lv = lane < n ? a.part_l[row0 + c0 + lane] : 0.f;
    float cm = mv;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) cm = fmaxf(cm, __shfl_xor_sync(FULL, cm, off));
    const float nm = fmaxf(M, cm);
    const float rescale = exp2f(M - nm);  // 0 on the first chunk
    M = nm;
    const float w = lane < n ? exp2f(mv - nm) : 0.f;
    float wl = w * lv;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) wl += __shfl_xor_sync(FULL, wl, off);
    ls = ls * rescale + wl;
#pragma unroll
    for (int v = 0; v < V; ++v) acc[v] *= rescale;
    for (int k = 0; k < n; ++k) {
      const float wk = __shfl_sync(FULL, w, k);
      const float* src = po + static_cast<size_t>(c0 + k) * D;
#pragma unroll
      for (int v = 0; v < V; ++v) acc[v] += wk * src[v];
    }
  }
  const float inv = 1.f / ls;
#pragma unroll
  for (int v = 0; v < V; v += 2) store_pair<T>(a, head * D + lane * V + v, acc[v] * inv, acc[v + 1] * inv);
}

// ---- tensor-core (tcgen05) kernel for head_dim 128 ------------------------------------
// Same work decomposition as prefill_main with 128-row tiles, two CTAs per SM:
//   warp 0      TMA producer: 64-key chunks (4 blocks) of K and V into two
//               32 KB stages laid out [d half][64 keys][128 B] (128-byte
//               swizzle), so a chunk is one UMMA operand;
//   warp 1      allocates 256 TMEM columns (S0 | S1 | O) and issues, from one
//               thread, S(c) = Q . K(c)^T (M 128, N 64, K 128, both operands
//               K-major in shared memory) into S buffer c % 2, and
//               O += P(c) . V(c) (M 128, N 128, K 64) with P read from TMEM
//               and V as an MN-major operand in shared memory;
//   warps 2..5  the softmax warpgroup: thread r owns query row r = TMEM lane r;
//               reads S(c), masks it (causal, partition end), keeps a
//               reference max per row that moves only when the chunk max
//               exceeds it by more than 2^8 (then O and l are rescaled in
//               TMEM), and writes P = exp2(s - ref) back over S(c) as 16-bit
//               pairs (bf16 as hi + lo halves of the buffer); at the end it
//               reads O and writes the row.
// S(c + 1) is issued before O += P(c) V(c) waits for P(c), so scores of the
// next chunk are computed while the softmax works.  MMA completion is
// signalled with tcgen05.commit on mbarriers; all waits are bounded; TMEM is
// released on every path.
namespace tcg {
constexpr int kRows = 128;
constexpr int kKeys = 64;
#ifndef PA_TC_STAGES
#define PA_TC_STAGES 2
#endif
constexpr int kStages = PA_TC_STAGES;
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 256;
constexpr float kRescale = 8.f;
constexpr int kMaxIds = 1024;  // blocks of one partition (the plan keeps partitions within this)

struct Smem {  // byte offsets from the 1024-aligned base
  static constexpr int Q = 0;                                  // [2][128][128 B]
  static constexpr int K0 = 32768;                             // K ring: [stage][2][64][128 B]
  static constexpr int V0 = K0 + kStages * 16384;              // V ring, same layout
  static constexpr int HALF = 16384;                           // one K or V chunk
  static constexpr int IDS = V0 + kStages * 16384;             // the partition's block ids [kMaxIds]
  static constexpr int KSC = IDS + kMaxIds * 4;                 // 1-byte caches: K scales of 4 chunks [4][64]
  static constexpr int VSC = KSC + 4 * 64 * 4;                  // and V scales [4][64] f32
  static constexpr int BAR = VSC + 4 * 64 * 4;
  static constexpr int NBAR = 6 * kStages + 8;
  static constexpr int TSLOT = BAR + NBAR * 8;
  static constexpr int SMEM = TSLOT + 16 + 1024;
};

// tcgen05 shared-memory descriptor: 128-byte swizzle, version 1.
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((addr >> 4) & 0x3FFFu) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}
// Instruction descriptor of kind::f16, f32 accumulate, M = 128.
template <typename T>
__device__ __forceinline__ uint32_t idesc(int N, bool b_mn_major) {
  const uint32_t ab = std::is_same<T, __nv_bfloat16>::value ? 1u : 0u;
  return (1u << 4) | (ab << 7) | (ab << 10) | (static_cast<uint32_t>(b_mn_major) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(kRows >> 4) << 24);
}
// D (TMEM) (+)= A (shared memory descriptor) . B (shared memory descriptor)
__device__ __forceinline__ void mma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(id), "r"(acc));
}
// D (TMEM) (+)= A (TMEM: lane = row, 16-bit pairs along K) . B (shared memory descriptor)
__device__ __forceinline__ void mma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t id, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a), "l"(b), "r"(id), "r"(acc));
}
__device__ __forceinline__ void commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// 2^x with one MUFU operation (flushes denormal results to zero; the
// arguments here are <= 8 and a flushed weight is below 2^-126).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
#ifndef PA_TC_SPIN
#define PA_TC_SPIN 0
#endif
// Bounded wait polled with plain try_wait (no suspend-time hint): these
// handoffs sit on the per-chunk critical path.
__device__ __forceinline__ bool wait_spin(uint32_t bar, uint32_t parity, uint64_t limit_ns = 2000000000ull) {
  if (dev::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = dev::global_timer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (dev::mbar_try_wait(bar, parity)) return true;
    if (dev::global_timer_ns() - t0 > limit_ns) return false;
  }
}
// A bounded wait whose outcome is the same in every lane (lane 0's), so the
// warp-collective tcgen05 instructions that follow stay converged.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity) {
  const bool ok = PA_TC_SPIN ? wait_spin(bar, parity) : dev::mbar_wait_bounded(bar, parity);
  return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}
}  // namespace tcg

template <typename KT, typename T>
__global__ void __launch_bounds__(tcg::kThreads, 2)
    prefill_tc(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
               const PrefillArgs a) {
  using namespace tcg;
  using L = Smem;
  constexpr int D = 128;
  constexpr bool SPLIT = std::is_same<T, __nv_bfloat16>::value;
  constexpr bool Q8 = sizeof(KT) == 1;  // 1-byte codes (E4M3 / INT8) converted to T on the way in
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = dev::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gb = smem_raw + (base - raw);

  const int wid = static_cast<int>(threadIdx.x >> 5), lane = static_cast<int>(threadIdx.x & 31);
  const int qt = static_cast<int>(blockIdx.x) % a.QT, bg = static_cast<int>(blockIdx.x) / a.QT;
  const int b = bg / a.Hkv, g = bg - b * a.Hkv;
  const int p = static_cast<int>(gridDim.y) - 1 - static_cast<int>(blockIdx.y);

  dev::grid_dependency_wait();
  const SeqView sv = seq_view(a, b, g == 0 && qt == 0 && p == 0 && threadIdx.x == 0);
  const int nrows = sv.n * a.G;
  const int R0 = qt * tcg::kRows;
  if (R0 >= nrows) return;
  const int shift = sv.L - sv.n;
  const int j0 = p * a.bpp;
  const int pos_cta = shift + (min(R0 + tcg::kRows, nrows) - 1) / a.G;
  const int nb = min(a.bpp, (pos_cta + 16) / 16 - j0);
  // this thread's row (softmax warps 2..5; TMEM lane 32 * (warp % 4) + lane)
  const int r = 32 * (wid & 3) + lane;
  const int rr = R0 + r;
  const bool has = wid >= 2 && rr < nrows;
  const int pos = has ? shift + rr / a.G : -1;
  const size_t head = has ? static_cast<size_t>(sv.qs + rr / a.G) * a.Hq + g * a.G + rr % a.G : 0;
  if (nb <= 0) {  // no key in this partition; partition 0 owns the zero rows of tokens without keys
    if (p == 0 && has && pos < 0)
      for (int d = 0; d < D; d += 2) store_pair<T>(a, head * D + d, 0.f, 0.f);
    return;
  }
  const int nc = (min(nb, kMaxIds) + 3) / 4;                 // 64-key chunks
  const int kend = min(sv.L, (j0 + min(nb, kMaxIds)) * 16);  // keys past this are masked (V rows zeroed)

  // K(c) is released when S(c) completes, V(c) when O += P(c) V(c) does, so
  // the producer runs up to two chunks ahead on K independently of V
  const uint32_t bar = base + L::BAR;
  auto kfull = [&](int s) { return bar + 8 * s; };
  auto kempty = [&](int s) { return bar + 8 * (kStages + s); };
  auto vfull = [&](int s) { return bar + 8 * (2 * kStages + s); };
  auto vempty = [&](int s) { return bar + 8 * (3 * kStages + s); };
  const uint32_t qfull = bar + 8 * (4 * kStages);
  auto sfull = [&](int i) { return bar + 8 * (4 * kStages + 1 + i); };  // S(c) in TMEM
  auto pfull = [&](int i) { return bar + 8 * (4 * kStages + 3 + i); };  // P(c) in TMEM (over S(c))
  auto pfree = [&](int i) { return bar + 8 * (4 * kStages + 5 + i); };  // O += P(c) V(c) complete
  const uint32_t mdone = bar + 8 * (4 * kStages + 7);
  auto kcode = [&](int s) { return bar + 8 * (4 * kStages + 8 + s); };            // 1-byte codes landed
  auto vcode = [&](int s) { return bar + 8 * (5 * kStages + 8 + s); };
  auto kstage = [&](int s) { return base + L::K0 + s * L::HALF; };
  auto vstage = [&](int s) { return base + L::V0 + s * L::HALF; };

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      dev::mbar_init(kfull(s), 1);
      dev::mbar_init(kempty(s), 1);
      dev::mbar_init(vfull(s), 1);
      dev::mbar_init(vempty(s), 1);
      dev::mbar_init(kcode(s), 1);
      dev::mbar_init(vcode(s), 1);
    }
    dev::mbar_init(qfull, 4);
    for (int i = 0; i < 2; ++i) {
      dev::mbar_init(sfull(i), 1);
      dev::mbar_init(pfull(i), 4);
      dev::mbar_init(pfree(i), 1);
    }
    dev::mbar_init(mdone, 1);
    dev::fence_barrier_init();
  }
  if (wid == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(base + L::TSLOT),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(gb + L::TSLOT);

  // 1-byte codes -> T in place: the codes of a chunk (upper half of its
  // stage, 4 blocks of 16 rows x 128 B, 128-byte swizzled) are read into
  // registers by the whole warp, then the stage is rewritten as 16-bit values
  // (exact) in the 128-byte-swizzled K-major layout the UMMA descriptors read.
  auto convert = [&](uint32_t stage) {  // every lane: 16 chunks of 16 codes
    uint8_t* st = gb + (stage - base);
    uint4 w[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int i = lane + 32 * j, k = i >> 7, t = (i >> 3) & 15, c16 = i & 7;
      w[j] = *reinterpret_cast<const uint4*>(st + 8192 + k * 2048 + t * 128 + ((c16 ^ (t & 7)) << 4));
    }
    __syncwarp();  // every code is in registers before the stage is rewritten
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int i = lane + 32 * j, k = i >> 7, t = (i >> 3) & 15, c16 = i & 7;
      const int kr = 16 * k + t, cc = 2 * (c16 & 3);
      uint32_t f[8];
      dev::code8x4_to<KT, T>(w[j].x, f[0], f[1]);
      dev::code8x4_to<KT, T>(w[j].y, f[2], f[3]);
      dev::code8x4_to<KT, T>(w[j].z, f[4], f[5]);
      dev::code8x4_to<KT, T>(w[j].w, f[6], f[7]);
      uint8_t* row = st + (c16 >> 2) * 8192 + kr * 128;
      *reinterpret_cast<uint4*>(row + ((cc ^ (kr & 7)) << 4)) = make_uint4(f[0], f[1], f[2], f[3]);
      *reinterpret_cast<uint4*>(row + (((cc + 1) ^ (kr & 7)) << 4)) = make_uint4(f[4], f[5], f[6], f[7]);
    }
    dev::fence_proxy_async_smem();  // the rewritten stage is read by the tensor cores
    __syncwarp();
  };
  if (wid == 0) {
    // ---- producer: the warp stages the partition's block ids in shared memory
    // (coalesced, checked), then lane 0 polls both rings and issues whichever
    // is free ----------------------------------------------------------------------
    int32_t* ids = reinterpret_cast<int32_t*>(gb + L::IDS);
    {
      const int32_t* row = a.block_tables + static_cast<size_t>(b) * a.max_blocks + j0;
      const int n_ids = min(nb, kMaxIds);
      bool bad = nb > kMaxIds;
      for (int i = lane; i < n_ids; i += 32) {
        int v = row[i];
        if (v < 0 || v >= a.num_blocks) {
          bad = true;
          v = 0;  // read block 0 instead; flagged
        }
        ids[i] = v;
      }
      if (__any_sync(FULL, bad) && lane == 0) atomicOr(&g_prefill_err, PA_DEVERR_BLOCK_RANGE);
      __syncwarp();
    }
    if constexpr (Q8) {
      // 1-byte codes.  Lane 0 requests a chunk's codes into the upper half of
      // a free stage; a K request also brings the chunk's 64 K and 64 V
      // per-token scales into slot c % 4 of the scale rings.  When a K chunk's
      // codes have landed the warp converts it and arrives on the full
      // barrier; V chunks are converted by the MMA warp just before their
      // product.  A scale slot is reused by the K request of chunk c + 4,
      // which waits for S(c + 2), which waits for the softmax of chunk c.
      if (lane == 0) {
        dev::prefetch_tensormap(&tmK);
        dev::prefetch_tensormap(&tmV);
      }
      const int last = min(nb, kMaxIds) - 1;
      auto request = [&](const CUtensorMap* m, uint32_t stage, uint32_t cb, int c, bool scales) {  // lane 0
        dev::mbar_arrive_expect_tx(cb, 8192 + (scales ? 512 : 0));
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int pb = ids[min(4 * c + k, last)];
          dev::tma_load_3d(stage + 8192 + k * 2048, m, cb, 0, g * 16, pb);
          if (scales) {
            dev::bulk_load(base + L::KSC + (c & 3) * 256 + 64 * k, a.k_scale + static_cast<size_t>(pb) * 16, 64, cb);
            dev::bulk_load(base + L::VSC + (c & 3) * 256 + 64 * k, a.v_scale + static_cast<size_t>(pb) * 16, 64, cb);
          }
        }
      };
      int ik = 0, iv = 0, ck = 0;  // chunks requested (K, V), K chunks converted
      bool ok = true;
      uint64_t t0 = dev::global_timer_ns();
      while (ok && (iv < nc || ck < nc)) {
        int act = 0;
        if (lane == 0) {
          if (ik < nc && (ik < kStages || dev::mbar_test(kempty(ik % kStages), ((ik / kStages) - 1) & 1))) act |= 1;
          if (iv < ik && (iv < kStages || dev::mbar_test(vempty(iv % kStages), ((iv / kStages) - 1) & 1))) act |= 2;
          if (ck < ik && dev::mbar_test(kcode(ck % kStages), (ck / kStages) & 1)) act |= 4;
        }
        act = __shfl_sync(FULL, act, 0);
        if (act & 1) {
          if (lane == 0) request(&tmK, kstage(ik % kStages), kcode(ik % kStages), ik, true);
          ++ik;
        }
        if (act & 2) {
          if (lane == 0) request(&tmV, vstage(iv % kStages), vcode(iv % kStages), iv, false);
          ++iv;
        }
        if (act & 4) {
          convert(kstage(ck % kStages));
          if (lane == 0) mbar_arrive(kfull(ck % kStages));
          ++ck;
        }
        if (act) {
          t0 = dev::global_timer_ns();
        } else if (dev::global_timer_ns() - t0 > 2000000000ull) {
          if (lane == 0) atomicOr(&g_prefill_err, PA_DEVERR_TIMEOUT);
          ok = false;
        }
      }
      // no copy may still be landing when the CTA exits (the last V chunks'
      // phases have normally completed already: the MMA warp waited for them)
      if (lane == 0) {
        for (int i = ck; i < ik; ++i) dev::mbar_wait_bounded(kcode(i % kStages), (i / kStages) & 1, 100000000ull);
        for (int i = max(0, iv - kStages); i < iv; ++i)
          dev::mbar_wait_bounded(vcode(i % kStages), (i / kStages) & 1, 100000000ull);
      }
    } else if (lane == 0) {
      dev::prefetch_tensormap(&tmK);
      dev::prefetch_tensormap(&tmV);
      const int last = min(nb, kMaxIds) - 1;
      int ck = 0, cv = 0;
      bool ok = true;
      uint64_t t0 = dev::global_timer_ns();
      // chunk c's blocks 4c .. 4c + 3; padding past the partition repeats its last block (masked)
      auto load = [&](const CUtensorMap* m, uint32_t dst, uint32_t bar_full, int c) {
        dev::mbar_arrive_expect_tx(bar_full, L::HALF);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int pb = ids[min(4 * c + k, last)];
#pragma unroll
          for (int h = 0; h < 2; ++h) dev::tma_load_3d(dst + h * 8192 + k * 2048, m, bar_full, h * 64, g * 16, pb);
        }
      };
      while (ok && cv < nc) {
        bool progressed = false;
        if (ck < nc && (ck < kStages || dev::mbar_test(kempty(ck % kStages), ((ck / kStages) - 1) & 1))) {
          load(&tmK, kstage(ck % kStages), kfull(ck % kStages), ck);
          ++ck;
          progressed = true;
        }
        if (cv < ck && (cv < kStages || dev::mbar_test(vempty(cv % kStages), ((cv / kStages) - 1) & 1))) {
          load(&tmV, vstage(cv % kStages), vfull(cv % kStages), cv);
          ++cv;
          progressed = true;
        }
        if (progressed) {
          t0 = dev::global_timer_ns();
        } else if (dev::global_timer_ns() - t0 > 2000000000ull) {
          atomicOr(&g_prefill_err, PA_DEVERR_TIMEOUT);
          ok = false;
        }
      }
      // no copy may still be landing when the CTA exits
      for (int i = max(0, ck - kStages); i < ck; ++i)
        dev::mbar_wait_bounded(kfull(i % kStages), (i / kStages) & 1, 100000000ull);
      for (int i = max(0, cv - kStages); i < cv; ++i)
        dev::mbar_wait_bounded(vfull(i % kStages), (i / kStages) & 1, 100000000ull);
    }
    __syncwarp();
  } else if (wid == 1) {
    // ---- MMA issuer -----------------------------------------------------------------------
    const uint32_t id_s = idesc<T>(kKeys, false), id_o = idesc<T>(D, true);
    bool ok = wait_warp(qfull, 0);
    // The warp polls (lane 0 tests, the warp follows) and issues whichever is
    // ready: S(cs) = Q . K(cs)^T once K(cs) has landed and S buffer cs % 2 is
    // free (O += P(cs - 2) V(cs - 2) done), or O += P(cp) V(cp) once the
    // softmax has written P(cp) and V(cp) has landed.
    int cs = 0, cp = 0;
    uint64_t t0 = dev::global_timer_ns();
    while (ok && cp < nc) {
      bool progressed = false;
      int go = 0;
      if (lane == 0 && cs < nc && cs <= cp + 1 && dev::mbar_test(kfull(cs % kStages), (cs / kStages) & 1) &&
          (cs < 2 || dev::mbar_test(pfree(cs & 1), ((cs >> 1) - 1) & 1)))
        go = 1;
      if (__shfl_sync(FULL, go, 0)) {
        fence_after();
        if (lane == 0) {
          const uint32_t kd = kstage(cs % kStages);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ss(tmem + 64 * (cs & 1), sdesc(base + L::Q + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                   sdesc(kd + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024), id_s, kk > 0 ? 1u : 0u);
          commit(sfull(cs & 1));
          commit(kempty(cs % kStages));
        }
        __syncwarp();
        ++cs;
        progressed = true;
      }
      go = 0;
      if (lane == 0 && cp < cs && dev::mbar_test(pfull(cp & 1), (cp >> 1) & 1) &&
          dev::mbar_test(Q8 ? vcode(cp % kStages) : vfull(cp % kStages), (cp / kStages) & 1))
        go = 1;
      if (__shfl_sync(FULL, go, 0)) {
        fence_after();
        const int sv_ = cp % kStages;
        // 1-byte codes: V(cp) -> 16-bit in place, here (converting earlier
        // delays the S products that keep the tensor pipe busy)
        if constexpr (Q8) convert(vstage(sv_));
        const int key0 = (j0 + 4 * cp) * 16;
        const int first_bad = max(0, min(kKeys, kend - key0));  // V rows from here on are zeroed
        if (first_bad < kKeys) {
          uint8_t* v = gb + (vstage(sv_) - base);
          for (int i = first_bad * 16 + lane; i < kKeys * 16; i += 32) {  // (row, 16-B chunk) pairs
            const int kr = i >> 4, ch = i & 15;
            *reinterpret_cast<uint4*>(v + (ch >> 3) * 8192 + kr * 128 + ((ch & 7) << 4)) = make_uint4(0, 0, 0, 0);
          }
          dev::fence_proxy_async_smem();
          __syncwarp();
        }
        if (lane == 0) {
          const uint32_t pt = tmem + 64 * (cp & 1), vd = vstage(sv_);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            const uint64_t bv = sdesc(vd + kk * 2048, 8192, 1024);
            mma_ts(tmem + 128, pt + 8 * kk, bv, id_o, (cp > 0 || kk > 0) ? 1u : 0u);
            if constexpr (SPLIT) mma_ts(tmem + 128, pt + 32 + 8 * kk, bv, id_o, 1u);
          }
          commit(pfree(cp & 1));
          commit(vempty(sv_));
        }
        __syncwarp();
        ++cp;
        progressed = true;
      }
      if (progressed) {
        t0 = dev::global_timer_ns();
      } else if (dev::global_timer_ns() - t0 > 2000000000ull) {
        ok = false;
      }
    }
    if (!ok && lane == 0) atomicOr(&g_prefill_err, PA_DEVERR_TIMEOUT);
    // every MMA issued has completed before TMEM is released
    if (lane == 0) commit(mdone);
    __syncwarp();
    dev::mbar_wait_bounded(mdone, 0, 100000000ull);
  } else {
    // ---- softmax warpgroup ------------------------------------------------------------------
    {  // Q row -> shared memory (zeros for padding rows), K-major, 128-byte swizzle
      const uint4* qrow = reinterpret_cast<const uint4*>(static_cast<const T*>(a.q) + head * D);
#pragma unroll
      for (int ch = 0; ch < 16; ++ch) {
        const uint4 v = has ? qrow[ch] : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(gb + L::Q + (ch >> 3) * 16384 + r * 128 + (((ch & 7) ^ (r & 7)) << 4)) = v;
      }
      dev::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(qfull);
    }
    const uint32_t trow = tmem + (static_cast<uint32_t>(32 * (wid & 3)) << 16);
    const float sl2 = a.scale_log2;
    float ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int c = 0; c < nc; ++c) {
      if (!wait_warp(sfull(c & 1), (c >> 1) & 1)) {
        ok = false;
        break;
      }
      fence_after();
      const uint32_t sb = trow + 64 * (c & 1);
      float x[kKeys];
      {
        uint32_t u[32], v[32];
        ld32(sb, u);
        ld32(sb + 32, v);
        wait_ld();
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          x[j] = __uint_as_float(u[j]);
          x[32 + j] = __uint_as_float(v[j]);
        }
      }
      // raw scores; the scale (> 0) is applied to the max and folded into
      // the exponent's FFMA below
      const int key0 = (j0 + 4 * c) * 16;
      // 1-byte caches: the chunk's per-token K and V scales (slot c % 4)
      const float* ksc = reinterpret_cast<const float*>(gb + L::KSC + (c & 3) * 256);
      const float* vsc = reinterpret_cast<const float*>(gb + L::VSC + (c & 3) * 256);
      float cm[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) cm[k] = -INFINITY;
      if (key0 + kKeys - 1 <= pos && key0 + kKeys <= kend) {  // every key of the chunk is visible
#pragma unroll
        for (int j = 0; j < kKeys; ++j) {
          if constexpr (Q8) x[j] *= ksc[j];
          cm[j & 7] = fmaxf(cm[j & 7], x[j]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < kKeys; ++j) {
          const int t = key0 + j;
          // a masked key's stale scale may be NaN: it never multiplies
          x[j] = (t <= pos && t < kend) ? (Q8 ? x[j] * ksc[j] : x[j]) : -INFINITY;
          cm[j & 7] = fmaxf(cm[j & 7], x[j]);
        }
      }
      const float cmax = fmaxf(fmaxf(fmaxf(cm[0], cm[1]), fmaxf(cm[2], cm[3])),
                               fmaxf(fmaxf(cm[4], cm[5]), fmaxf(cm[6], cm[7]))) * sl2;
      // move the reference when the chunk max outgrows it; O and l follow
      const bool move = cmax > ref + kRescale;
      if (__any_sync(FULL, move && ref != -INFINITY)) {
        if (!wait_warp(pfree((c - 1) & 1), ((c - 1) >> 1) & 1)) {  // O += P(c-1) V(c-1) done
          ok = false;
          break;
        }
        fence_after();
        const float alpha = (move && ref != -INFINITY) ? ex2(ref - cmax) : 1.f;
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
          uint32_t u[32];
          ld32(trow + 128 + 32 * q, u);
          wait_ld();
#pragma unroll
          for (int j = 0; j < 32; ++j) u[j] = __float_as_uint(__uint_as_float(u[j]) * alpha);
          st32(trow + 128 + 32 * q, u);
        }
        wait_st();
        l *= alpha;
      }
      if (move) ref = cmax;
      // P over S(c): 16-bit pairs, bf16 as hi (columns 0..31) and lo (32..63)
      uint32_t hi[32], lo[32];
      float ls[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) ls[k] = 0.f;
      // p = 2^(s * scale * log2 e - ref); a row without keys so far keeps
      // ref = -inf and gets p = 0 (its masked scores are -inf too)
      const float nref = ref == -INFINITY ? 0.f : -ref;
#pragma unroll
      for (int j = 0; j < kKeys; j += 2) {
        const float p0 = ex2(fmaf(x[j], sl2, nref));
        const float p1 = ex2(fmaf(x[j + 1], sl2, nref));
        if constexpr (Q8) {
          // the product takes p * v_scale (the V codes carry no scale); l sums p.
          // A masked key has p = 0 exactly and a possibly stale (NaN) scale.
          const float q0 = p0 == 0.f ? 0.f : p0 * vsc[j], q1 = p1 == 0.f ? 0.f : p1 * vsc[j + 1];
          hi[j >> 1] = dev::pack2<T>(q0, q1);
          if constexpr (SPLIT) {
            const float2 h = dev::unpack2<T>(hi[j >> 1]);
            lo[j >> 1] = dev::pack2<T>(q0 - h.x, q1 - h.y);
          }
          ls[(j >> 1) & 7] += p0 + p1;
        } else {
          hi[j >> 1] = dev::pack2<T>(p0, p1);
          const float2 h = dev::unpack2<T>(hi[j >> 1]);
          if constexpr (SPLIT) {
            lo[j >> 1] = dev::pack2<T>(p0 - h.x, p1 - h.y);
            ls[(j >> 1) & 7] += p0 + p1;
          } else {
            ls[(j >> 1) & 7] += h.x + h.y;  // normalise with the rounded weights the product uses
          }
        }
      }
      l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
      st32(sb, hi);
      if constexpr (SPLIT) st32(sb + 32, lo);
      wait_st();
      fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(pfull(c & 1));
    }
    dev::grid_launch_dependents();
    if (!ok && lane == 0) atomicOr(&g_prefill_err, PA_DEVERR_TIMEOUT);
    // ---- epilogue: O row -> output, partial, zero row or nothing ----
    if (ok && wait_warp(pfree((nc - 1) & 1), ((nc - 1) >> 1) & 1)) {
      fence_after();
      const int np = pos < 0 ? 0 : ((pos + 16) / 16 + a.bpp - 1) / a.bpp;
      const bool direct = has && pos >= 0 && np == 1 && p == 0;  // later partitions hold it without keys
      const bool partial = has && pos >= 0 && np > 1 && p < np;
      const bool zero = has && pos < 0 && p == 0;
      const float inv = direct ? 1.f / l : 1.f;
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        uint32_t u[32];
        ld32(trow + 128 + 32 * q, u);
        wait_ld();
        if (direct || zero) {
#pragma unroll
          for (int j = 0; j < 32; j += 2)
            store_pair<T>(a, head * D + 32 * q + j, zero ? 0.f : __uint_as_float(u[j]) * inv,
                          zero ? 0.f : __uint_as_float(u[j + 1]) * inv);
        } else if (partial) {
          float* po = a.part_o + (head * a.max_parts + p) * D + 32 * q;
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            *reinterpret_cast<float4*>(po + j) = make_float4(__uint_as_float(u[j]), __uint_as_float(u[j + 1]),
                                                             __uint_as_float(u[j + 2]), __uint_as_float(u[j + 3]));
        }
      }
      if (partial) {
        a.part_m[head * a.max_parts + p] = ref;
        a.part_l[head * a.max_parts + p] = l;
      }
    } else if (lane == 0) {
      atomicOr(&g_prefill_err, PA_DEVERR_TIMEOUT);
    }
  }
  fence_before();
  __syncthreads();
  if (wid == 1) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

#ifndef PA_FORK_SINGLE
#define PA_FORK_SINGLE 1
#endif

// A second stream of the calling thread in the current context, with the
// events that fork it from and join it back to the caller's stream.  The
// decode kernel for the one-token sequences of a call runs there, beside the
// multi-token kernel: SMs left idle by the multi-token grid (its last wave)
// stream the decode rows meanwhile.  Created on first use per thread and
// device, and again when the context changed (a device reset); never freed.
struct SideStream {
  unsigned long long ctx = 0;
  cudaStream_t s = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

pa_status side_stream(int dev, SideStream** out) {
  thread_local SideStream sides[kMaxDevices];
  SideStream& sd = sides[dev];
  unsigned long long ctx = 0;
  if (!current_context_id(&ctx)) return fail(PA_ERR_CUDA, "pa_chunked_prefill: no current CUDA context");
  if (!sd.s || sd.ctx != ctx) {
    cudaError_t e = cudaStreamCreateWithFlags(&sd.s, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming);
    if (e != cudaSuccess) {
      sd.s = nullptr;
      return fail(PA_ERR_CUDA, "pa_chunked_prefill: side stream: %s", cudaGetErrorString(e));
    }
    sd.ctx = ctx;
  }
  *out = &sd;
  return PA_OK;
}

// The decode kernel's launch for the rows of a multi-token call it serves:
// every sequence (q_tokens = max_q_len, out-of-range sequences flagged), or
// only the one-token sequences (q_tokens = 1, the rest left to the
// multi-token kernel).
DecodeLaunch rows_to_decode(const PrefillLaunch& l, int32_t q_tokens, int32_t q_report) {
  DecodeLaunch d;
  d.q = l.q;
  d.q_dtype = l.q_dtype;
  d.k_cache = l.k_cache;
  d.v_cache = l.v_cache;
  d.k_scale = l.k_scale;
  d.v_scale = l.v_scale;
  d.block_tables = l.block_tables;
  d.max_blocks = l.max_blocks;
  d.context_lens = l.context_lens;
  d.max_context_len = l.max_context_len;
  d.B = l.B;
  d.Hq = l.Hq;
  d.Hkv = l.Hkv;
  d.D = l.D;
  d.num_blocks = l.num_blocks;
  d.kv_dtype = l.kv_dtype;
  d.scale = l.scale;
  d.out = l.out;
  d.out_dtype = l.out_dtype;
  d.workspace = static_cast<uint8_t*>(l.workspace) + l.plan.dec_offset;
  d.plan = l.plan.dec;
  d.q_start = l.q_start;
  d.q_rows = l.T;
  d.q_tokens = q_tokens;
  d.q_report = q_report;
  return d;
}

template <typename KT, typename T, int D>
pa_status launch_t(const PrefillLaunch& l, CUtensorMapDataType dt, cudaStream_t stream) {
  using TL = PTile<KT, D>;
  if (l.plan.route_short) return launch_decode(rows_to_decode(l, l.max_q_len, 1), stream);
  // tcgen05 kernel (128-row tiles; 1-byte codes converted to T in shared
  // memory) or mma.sync kernel (64-row tiles), as planned
  const bool TC = D == 128 && l.plan.tc;
  constexpr int EB = static_cast<int>(sizeof(KT));
  CUtensorMap tmK, tmV;
  pa_status st = make_kv_map(&tmK, l.k_cache, l.Hkv, l.num_blocks, TL::ROWB, EB, dt, "pa_chunked_prefill", !TC);
  if (st != PA_OK) return st;
  st = make_kv_map(&tmV, l.v_cache, l.Hkv, l.num_blocks, TL::ROWB, EB, dt, "pa_chunked_prefill", !TC);
  if (st != PA_OK) return st;

  PrefillArgs a;
  a.q = l.q;
  a.q_start = l.q_start;
  a.block_tables = l.block_tables;
  a.context_lens = l.context_lens;
  a.out = l.out;
  const size_t rows = static_cast<size_t>(l.T) * l.Hq * l.plan.max_parts;
  a.part_o = l.plan.max_parts > 1 ? static_cast<float*>(l.workspace) : nullptr;
  a.part_m = a.part_o ? a.part_o + rows * D : nullptr;
  a.part_l = a.part_m ? a.part_m + rows : nullptr;
  a.B = l.B;
  a.T = l.T;
  a.Hq = l.Hq;
  a.Hkv = l.Hkv;
  a.G = l.Hq / l.Hkv;
  a.max_blocks = l.max_blocks;
  a.num_blocks = l.num_blocks;
  a.max_context_len = l.max_context_len;
  a.max_q_len = l.max_q_len;
  a.QT = l.plan.row_tiles;
  a.bpp = l.plan.blocks_per_part;
  a.max_parts = l.plan.max_parts;
  a.scale_log2 = l.scale * 1.4426950408889634f;
  a.out_f32 = l.out_dtype == PA_DTYPE_F32;
  a.k_scale = l.k_scale;
  a.v_scale = l.v_scale;
  a.skip_single = l.plan.route_single;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(PA_ERR_CUDA, "pa_chunked_prefill: no CUDA device");
  if (dev >= kMaxDevices) return fail(PA_ERR_UNSUPPORTED, "pa_chunked_prefill: device index %d", dev);
  // One-token sequences (decode steps riding in the call) go to the decode
  // kernel: a one-row tile would waste the multi-token kernel's CTA.  With
  // multi-token sequences as well, that launch goes on the side stream,
  // forked here (after what the caller enqueued before the call) and joined
  // back after the multi-token kernel.
  SideStream* side = nullptr;
  if (l.plan.route_single) {
    if (l.max_q_len <= 1) return launch_decode(rows_to_decode(l, 1, 0), stream);
    if (PA_FORK_SINGLE) {
      pa_status ss = side_stream(dev, &side);
      if (ss != PA_OK) return ss;
      cudaError_t e = cudaEventRecord(side->fork, stream);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(side->s, side->fork, 0);
      if (e != cudaSuccess) return fail(PA_ERR_CUDA, "pa_chunked_prefill: fork: %s", cudaGetErrorString(e));
    } else {
      pa_status ds = launch_decode(rows_to_decode(l, 1, 0), stream);
      if (ds != PA_OK) return ds;
    }
  }
  static std::once_flag once[kMaxDevices];
  static cudaError_t setup_err[kMaxDevices];
  using TS = tcg::Smem;
  std::call_once(once[dev], [dev] {
    cudaError_t e =
        cudaFuncSetAttribute(prefill_main<KT, T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, TL::SMEM);
    if constexpr (D == 128)
      if (e == cudaSuccess)
        e = cudaFuncSetAttribute(prefill_tc<KT, T>, cudaFuncAttributeMaxDynamicSharedMemorySize, TS::SMEM);
    setup_err[dev] = e;
  });
  if (setup_err[dev] != cudaSuccess)
    return fail(PA_ERR_CUDA, "pa_chunked_prefill: %s", cudaGetErrorString(setup_err[dev]));

  const dim3 grid(static_cast<unsigned>(l.B * l.Hkv * l.plan.row_tiles), static_cast<unsigned>(l.plan.max_parts));
  cudaError_t e;
  if constexpr (D == 128) {
    if (TC)
      e = launch_dependent(prefill_tc<KT, T>, grid, dim3(tcg::kThreads), TS::SMEM, stream, tmK, tmV, a);
    else
      e = launch_dependent(prefill_main<KT, T, D>, grid, dim3(kThreads), TL::SMEM, stream, tmK, tmV, a);
  } else {
    e = launch_dependent(prefill_main<KT, T, D>, grid, dim3(kThreads), TL::SMEM, stream, tmK, tmV, a);
  }
  if (e == cudaSuccess && l.plan.max_parts > 1)
    e = launch_dependent(prefill_reduce<T, D>,
                         dim3(static_cast<unsigned>((static_cast<int64_t>(l.T) * l.Hq + kReduceRows - 1) / kReduceRows)),
                         dim3(32 * kReduceRows), 0, stream, a);
  if (e == cudaSuccess) e = cudaGetLastError();
  pa_status ds = PA_OK;
  if (side) {  // the decode rows on the side stream, then the join (also after a failed launch)
    if (e == cudaSuccess) ds = launch_decode(rows_to_decode(l, 1, 0), side->s);
    cudaError_t j = cudaEventRecord(side->join, side->s);
    if (j == cudaSuccess) j = cudaStreamWaitEvent(stream, side->join, 0);
    if (j != cudaSuccess && e == cudaSuccess) e = j;
  }
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "pa_chunked_prefill launch: %s", cudaGetErrorString(e));
  return ds;
}

}  // namespace

pa_status launch_prefill(const PrefillLaunch& l, void* stream_ptr) {
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
  // the caller), read as the query's 16-bit type; the map moves raw bytes
  const bool f16 = l.q_dtype == PA_DTYPE_F16;
  if (l.kv_dtype == PA_DTYPE_INT8)
    return f16 ? launch_t<int8_t, __half, 128>(l, CU_TENSOR_MAP_DATA_TYPE_UINT8, st)
               : launch_t<int8_t, __nv_bfloat16, 128>(l, CU_TENSOR_MAP_DATA_TYPE_UINT8, st);
  return f16 ? launch_t<uint8_t, __half, 128>(l, CU_TENSOR_MAP_DATA_TYPE_UINT8, st)
             : launch_t<uint8_t, __nv_bfloat16, 128>(l, CU_TENSOR_MAP_DATA_TYPE_UINT8, st);
}

pa_status read_errors_prefill(uint32_t* flags, bool clear) {
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_prefill_err, sizeof(v));
  if (e == cudaSuccess && clear) {
    const uint32_t z = 0;
    e = cudaMemcpyToSymbol(g_prefill_err, &z, sizeof(z));
  }
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "pa_device_errors: %s", cudaGetErrorString(e));
  *flags = v;
  return PA_OK;
}

}  // namespace pa
