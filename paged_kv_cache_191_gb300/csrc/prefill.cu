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
  int32_t QT;  // row tiles per (sequence, kv head): ceil(max_q_len * G / 64)
  int32_t bpp, max_parts;
  float scale_log2;
  int32_t out_f32;
};

template <int D>
struct PTile {
  static constexpr int ROWB = 2 * D;                       // bytes per token row
  static constexpr int TB = 16 * ROWB;                     // one (block, head) tile
  static constexpr int NS = kRingBytes / (2 * TB);         // K+V stages
  static constexpr int SMEM = 1024 + NS * 2 * TB + NS * 16;
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
  return v;
}

template <typename T>
__device__ __forceinline__ void store_pair(const PrefillArgs& a, size_t idx, float x, float y) {
  if (a.out_f32)
    *reinterpret_cast<float2*>(static_cast<float*>(a.out) + idx) = make_float2(x, y);
  else
    *reinterpret_cast<uint32_t*>(static_cast<T*>(a.out) + idx) = dev::pack2<T>(x, y);
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, PA_PREFILL_MINB)
    prefill_main(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 const PrefillArgs a) {
  using TL = PTile<D>;
  constexpr int NS = TL::NS;
  constexpr int KSTEPS = D / 16;
  constexpr int DT = D / 8;  // 8-wide column tiles of O
  constexpr bool SPLIT_P = std::is_same<T, __nv_bfloat16>::value;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t ring = (dev::smem_addr(smem_raw) + 1023u) & ~1023u;
  const uint32_t bar_full = ring + NS * 2 * TL::TB, bar_empty = bar_full + NS * 8;

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
            dev::mbar_arrive_expect_tx(bar, 2 * TL::TB);
            if constexpr (TL::ROWB == 256) {
              dev::tma_load_5d(kdst, &tmK, bar, 0, 0, 0, g, pb);
              dev::tma_load_5d(vdst, &tmV, bar, 0, 0, 0, g, pb);
            } else {
              dev::tma_load_3d(kdst, &tmK, bar, 0, g * 16, pb);
              dev::tma_load_3d(vdst, &tmV, bar, 0, g * 16, pb);
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
        const int c = 16 * kk + 2 * q4;
        qf[kk][0] = hasA ? *reinterpret_cast<const uint32_t*>(qa + c) : 0u;
        qf[kk][1] = hasB ? *reinterpret_cast<const uint32_t*>(qb + c) : 0u;
        qf[kk][2] = hasA ? *reinterpret_cast<const uint32_t*>(qa + c + 8) : 0u;
        qf[kk][3] = hasB ? *reinterpret_cast<const uint32_t*>(qb + c + 8) : 0u;
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
        const uint32_t kb = ring + s * 2 * TL::TB, vb = kb + TL::TB;
        // ---- S = Q . K^T over this block's 16 tokens (two 8-token tiles) -----
        // even and odd k-steps accumulate separately: four independent MMA
        // chains instead of two, summed once
        float sc[2][4], sd[2][4];
#pragma unroll
        for (int k = 0; k < 4; ++k) sc[0][k] = sc[1][k] = sd[0][k] = sd[1][k] = 0.f;
#pragma unroll
        for (int kk = 0; kk < KSTEPS; ++kk) {
          uint32_t kf[4];
          dev::ldmatrix_x4(kf, kb + swz(krow, 2 * kk + kcol));
          float(&acc0)[4] = (kk & 1) ? sd[0] : sc[0];
          float(&acc1)[4] = (kk & 1) ? sd[1] : sc[1];
          dev::Mma<T>::run(acc0, qf[kk], kf[0], kf[1]);
          dev::Mma<T>::run(acc1, qf[kk], kf[2], kf[3]);
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
            x[nt][e] = t <= posA ? sc[nt][e] * sl2 : -INFINITY;
            x[nt][2 + e] = t <= posB ? sc[nt][2 + e] * sl2 : -INFINITY;
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
          lA = lA * alA + (pv[0][0] + pv[0][1] + pv[1][0] + pv[1][1]);
          lB = lB * alB + (pv[0][2] + pv[0][3] + pv[1][2] + pv[1][3]);
        } else {
          // normalise with the rounded weights the PV product uses
          const float2 h0 = dev::unpack2<T>(ph[0]), h1 = dev::unpack2<T>(ph[1]);
          const float2 h2 = dev::unpack2<T>(ph[2]), h3 = dev::unpack2<T>(ph[3]);
          lA = lA * alA + (h0.x + h0.y + h2.x + h2.y);
          lB = lB * alB + (h1.x + h1.y + h3.x + h3.y);
        }
        // ---- O = O * alpha + P . V ---------------------------------------------
#pragma unroll
        for (int t2 = 0; t2 < D / 16; ++t2) {
          uint32_t vf[4];
          dev::ldmatrix_x4_trans(vf, vb + swz(vrow, 2 * t2 + vcol));
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
      for (int t = 0; t < DT; ++t)
        store_pair<T>(a, head * D + 8 * t + 2 * q4, o[t][2 * half] * inv, o[t][2 * half + 1] * inv);
    } else {
      const size_t prow = head * a.max_parts + p;
      float* po = a.part_o + prow * D;
#pragma unroll
      for (int t = 0; t < DT; ++t)
        *reinterpret_cast<float2*>(po + 8 * t + 2 * q4) = make_float2(o[t][2 * half], o[t][2 * half + 1]);
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

template <typename T, int D>
pa_status launch_t(const PrefillLaunch& l, CUtensorMapDataType dt, cudaStream_t stream) {
  using TL = PTile<D>;
  CUtensorMap tmK, tmV;
  pa_status st = make_kv_map(&tmK, l.k_cache, l.Hkv, l.num_blocks, TL::ROWB, 2, dt, "pa_chunked_prefill");
  if (st != PA_OK) return st;
  st = make_kv_map(&tmV, l.v_cache, l.Hkv, l.num_blocks, TL::ROWB, 2, dt, "pa_chunked_prefill");
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

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(PA_ERR_CUDA, "pa_chunked_prefill: no CUDA device");
  if (dev >= kMaxDevices) return fail(PA_ERR_UNSUPPORTED, "pa_chunked_prefill: device index %d", dev);
  static std::once_flag once[kMaxDevices];
  static cudaError_t setup_err[kMaxDevices];
  std::call_once(once[dev], [dev] {
    setup_err[dev] =
        cudaFuncSetAttribute(prefill_main<T, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, TL::SMEM);
  });
  if (setup_err[dev] != cudaSuccess)
    return fail(PA_ERR_CUDA, "pa_chunked_prefill: %s", cudaGetErrorString(setup_err[dev]));

  const dim3 grid(static_cast<unsigned>(l.B * l.Hkv * l.plan.row_tiles), static_cast<unsigned>(l.plan.max_parts));
  cudaError_t e = launch_dependent(prefill_main<T, D>, grid, dim3(kThreads), TL::SMEM, stream, tmK, tmV, a);
  if (e == cudaSuccess && l.plan.max_parts > 1)
    e = launch_dependent(prefill_reduce<T, D>,
                         dim3(static_cast<unsigned>((static_cast<int64_t>(l.T) * l.Hq + kReduceRows - 1) / kReduceRows)),
                         dim3(32 * kReduceRows), 0, stream, a);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "pa_chunked_prefill launch: %s", cudaGetErrorString(e));
  return PA_OK;
}

}  // namespace

pa_status launch_prefill(const PrefillLaunch& l, void* stream_ptr) {
  cudaStream_t st = static_cast<cudaStream_t>(stream_ptr);
  if (l.kv_dtype == PA_DTYPE_F16) {
    if (l.D == 64) return launch_t<__half, 64>(l, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, st);
    return launch_t<__half, 128>(l, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, st);
  }
  if (l.D == 64) return launch_t<__nv_bfloat16, 64>(l, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, st);
  return launch_t<__nv_bfloat16, 128>(l, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, st);
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
