// Paged decode attention for sm_103a.
//
// What it computes ("LLM推理引擎深度实战：从PagedAttention到分布式推理部署",
// section 2.3): for each sequence and query head, softmax(scale q.K^T).V over
// the sequence's context, where the kernel itself maps logical token t to
// physical block block_tables[b][t/16], row t%16, and gathers the scattered
// K/V tiles from there.
//
// Design (GB300):
// * Work unit = one CTA per (sequence b, kv head g, partition p of
//   `bpp` 16-token blocks).  All G query heads of kv head g share every K/V
//   tile, so K/V bytes are read from HBM exactly once per step.
// * Each (block, kv head) tile is 16 rows x D contiguous elements.  It is
//   fetched by TMA (cp.async.bulk.tensor, 128-byte swizzle) into a per-warp
//   ring of shared-memory stages completed by mbarriers; each of the 4 warps
//   owns blocks w, w+4, w+8, ... of the partition and refills its own stages,
//   so warps never wait on one another inside the loop.
// * Scores on tensor cores, transposed: S^T[16 tokens x 8 heads] =
//   K_tile[16 x D] . Q^T[D x 8] with mma.m16n8k16 (A = K from ldmatrix,
//   B = Q from registers; G < 8 pads the N dimension with zero heads).
//   Online softmax in fp32 (exp2 with log2e folded into the scale), then
//   O^T[D x 8] += V^T[D x 16] . P^T[16 x 8] with A = V via ldmatrix.trans and
//   B = P^T obtained from the score fragment by movmatrix.  bf16 P is split
//   into hi + lo bf16 parts so its rounding error stays ~2^-17.
// * FP8 E4M3 caches: codes are converted exactly to f16/bf16 in registers;
//   the per-token K scale multiplies the score, the per-token V scale
//   multiplies p before the PV product.
// * Partitions of one (b, g) are merged by decode_reduce with the usual
//   log-sum-exp weights; a single-partition sequence is written directly.
#include <cudaTypedefs.h>

#include <mutex>

#include "device_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

__device__ uint32_t g_decode_err;

constexpr int kNW = 4;   // warps per CTA
constexpr int kNSW = 2;  // pipeline stages per warp
constexpr int kNS = kNW * kNSW;
constexpr int kMaxBpp = 64;

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
};

template <typename KT, int D>
struct Tile {
  static constexpr int ROWB = D * static_cast<int>(sizeof(KT));  // bytes per token row
  static constexpr int BYTES = 16 * ROWB;                          // one (block, head) tile
  static constexpr int NBOX = ROWB / 128;                          // 128-byte swizzle boxes
  static constexpr int BOXE = 128 / static_cast<int>(sizeof(KT));  // elements per box row
  static constexpr int SMEM = 1024 + kNS * 2 * BYTES + kNS * 128 + kNS * 8 + kMaxBpp * 4;
  static_assert(ROWB % 128 == 0, "rows must be whole 128-byte swizzle spans");
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
  else if constexpr (sizeof(QT) == 2) {
    if constexpr (std::is_same<QT, __half>::value)
      static_cast<__half*>(a.out)[idx] = __float2half_rn(v);
    else
      static_cast<__nv_bfloat16*>(a.out)[idx] = __float2bfloat16_rn(v);
  }
}

template <typename KT, typename QT, int D>
__global__ void __launch_bounds__(kNW * 32)
    decode_main(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                const DecodeArgs a) {
  using TL = Tile<KT, D>;
  constexpr bool FP8 = sizeof(KT) == 1;
  constexpr int KSTEPS = D / 16;
  constexpr int MT = D / 16;
  constexpr uint32_t STAGE_TX = 2 * TL::BYTES + (FP8 ? 128 : 0);
  constexpr bool SPLIT_P = std::is_same<QT, __nv_bfloat16>::value;
  constexpr unsigned FULL = 0xffffffffu;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = dev::smem_addr(smem_raw);
  const uint32_t tiles = (raw + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (tiles - raw);
  float* s_scale = reinterpret_cast<float*>(base + kNS * 2 * TL::BYTES);  // [kNS][32]
  uint64_t* s_bar = reinterpret_cast<uint64_t*>(base + kNS * 2 * TL::BYTES + kNS * 128);
  int32_t* s_tab = reinterpret_cast<int32_t*>(s_bar + kNS);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.x / a.Hkv, g = blockIdx.x - b * a.Hkv, p = blockIdx.y;

  // Launched as a dependent of the preceding kernel (normally the cache
  // write): everything below may read what it wrote.
  dev::grid_dependency_wait();
  const int L = checked_len(a, b, threadIdx.x == 0 && p == 0);
  const int nblk = (L + 15) >> 4;
  const int j0 = p * a.bpp;
  if (j0 >= nblk) {
    if (p == 0)  // empty context: zero rows
      for (int i = threadIdx.x; i < a.G * D; i += blockDim.x)
        store_out<QT>(a, (static_cast<size_t>(b) * a.Hq + g * a.G + i / D) * D + i % D, 0.f);
    return;
  }
  const int nb = min(a.bpp, nblk - j0);
  const int nparts = (nblk + a.bpp - 1) / a.bpp;

  // Block ids of this partition -> shared memory (one coalesced read).
  for (int i = threadIdx.x; i < nb; i += blockDim.x) {
    int pb = a.block_tables[static_cast<size_t>(b) * a.max_blocks + j0 + i];
    if (pb < 0 || pb >= a.num_blocks) {
      atomicOr(&g_decode_err, PA_DEVERR_BLOCK_RANGE);
      pb = 0;  // read a valid block instead; the result is flagged
    }
    s_tab[i] = pb;
  }
  if (threadIdx.x == 0) {
    dev::prefetch_tensormap(&tmK);
    dev::prefetch_tensormap(&tmV);
    for (int s = 0; s < kNS; ++s) dev::mbar_init(dev::smem_addr(&s_bar[s]), 1);
    dev::fence_barrier_init();
  }
  __syncthreads();

  auto issue = [&](int jj, int s) {
    const int pb = s_tab[jj];
    const uint32_t bar = dev::smem_addr(&s_bar[s]);
    const uint32_t kdst = tiles + s * 2 * TL::BYTES, vdst = kdst + TL::BYTES;
    dev::mbar_arrive_expect_tx(bar, STAGE_TX);
#pragma unroll
    for (int bx = 0; bx < TL::NBOX; ++bx) {
      dev::tma_load_3d(kdst + bx * 2048, &tmK, bar, bx * TL::BOXE, g * 16, pb);
      dev::tma_load_3d(vdst + bx * 2048, &tmV, bar, bx * TL::BOXE, g * 16, pb);
    }
    if constexpr (FP8) {
      dev::bulk_load(dev::smem_addr(s_scale + s * 32), a.k_scale + static_cast<size_t>(pb) * 16, 64, bar);
      dev::bulk_load(dev::smem_addr(s_scale + s * 32 + 16), a.v_scale + static_cast<size_t>(pb) * 16, 64,
                     bar);
    }
  };
  if (lane == 0) {
#pragma unroll
    for (int i = 0; i < kNSW; ++i) {
      const int jj = warp + i * kNW;
      if (jj < nb) issue(jj, warp * kNSW + i);
    }
  }

  // Q as the B operand (k = head dim, n = query head of the group).
  const int r = lane >> 2, q4 = lane & 3;
  uint32_t qf[KSTEPS][2];
  {
    const int n = r;
    const QT* qrow = static_cast<const QT*>(a.q) + (static_cast<size_t>(b) * a.Hq + g * a.G + n) * D;
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
      if (n < a.G) {
        if constexpr (FP8) {
          // permuted k order matching the register-converted K fragment
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
  }

  float o[MT][4];
#pragma unroll
  for (int mt = 0; mt < MT; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const float sl2 = a.scale_log2;

  for (int i = 0;; ++i) {
    const int jj = warp + i * kNW;
    if (jj >= nb) break;
    const int s = warp * kNSW + (i % kNSW);
    if (!dev::mbar_wait_bounded(dev::smem_addr(&s_bar[s]), (i / kNSW) & 1)) {
      if (lane == 0) atomicOr(&g_decode_err, PA_DEVERR_TIMEOUT);
      // drain this warp's other copies in flight (bounded), then stop
      for (int i2 = i + 1; i2 < i + kNSW; ++i2) {
        const int j2 = warp + i2 * kNW;
        if (j2 < nb)
          dev::mbar_wait_bounded(dev::smem_addr(&s_bar[warp * kNSW + (i2 % kNSW)]), (i2 / kNSW) & 1,
                                 100000000ull);
      }
      break;
    }
    const uint32_t kb = tiles + s * 2 * TL::BYTES, vb = kb + TL::BYTES;
    const int nvalid = min(16, L - (j0 + jj) * 16);

    // ---- S^T = K . Q^T -----------------------------------------------------
    float sacc[4] = {0.f, 0.f, 0.f, 0.f};
    if constexpr (FP8) {
      const uint4 x0 = dev::lds128(kb + swz(r, 2 * q4));
      const uint4 x1 = dev::lds128(kb + swz(r, 2 * q4 + 1));
      const uint4 y0 = dev::lds128(kb + swz(r + 8, 2 * q4));
      const uint4 y1 = dev::lds128(kb + swz(r + 8, 2 * q4 + 1));
      const uint32_t wr[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
      const uint32_t wr8[8] = {y0.x, y0.y, y0.z, y0.w, y1.x, y1.y, y1.z, y1.w};
#pragma unroll
      for (int kk = 0; kk < KSTEPS; ++kk) {
        uint32_t af[4];
        af[0] = dev::e4m3x2_to<QT>(static_cast<uint16_t>(wr[kk] & 0xffffu));
        af[1] = dev::e4m3x2_to<QT>(static_cast<uint16_t>(wr8[kk] & 0xffffu));
        af[2] = dev::e4m3x2_to<QT>(static_cast<uint16_t>(wr[kk] >> 16));
        af[3] = dev::e4m3x2_to<QT>(static_cast<uint16_t>(wr8[kk] >> 16));
        dev::Mma<QT>::run(sacc, af, qf[kk][0], qf[kk][1]);
      }
    } else {
      const int krow = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
      for (int kk = 0; kk < KSTEPS; ++kk) {
        uint32_t af[4];
        dev::ldmatrix_x4(af, kb + swz(krow, 2 * kk + (lane >> 4)));
        dev::Mma<QT>::run(sacc, af, qf[kk][0], qf[kk][1]);
      }
    }

    // ---- online softmax over this block's 16 tokens ---------------------------
    float c_r = sl2, c_r8 = sl2;
    if constexpr (FP8) {
      c_r *= s_scale[s * 32 + r];
      c_r8 *= s_scale[s * 32 + r + 8];
    }
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
    const float mn0 = fmaxf(m0, bm0), mn1 = fmaxf(m1, bm1);
    const float al0 = exp2f(m0 - mn0), al1 = exp2f(m1 - mn1);
    m0 = mn0;
    m1 = mn1;
    float p0 = exp2f(x0 - mn0), p1 = exp2f(x1 - mn1), p2 = exp2f(x2 - mn0), p3 = exp2f(x3 - mn1);

    uint32_t ph_r, ph_r8, pl_r = 0, pl_r8 = 0;
    if constexpr (FP8) {
      l0 = l0 * al0 + (p0 + p2);
      l1 = l1 * al1 + (p1 + p3);
      const float vs_r = s_scale[s * 32 + 16 + r], vs_r8 = s_scale[s * 32 + 16 + r + 8];
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
      if constexpr (!FP8) {
        l0 = l0 * al0 + (p0 + p2);
        l1 = l1 * al1 + (p1 + p3);
      }
    } else if constexpr (!FP8) {
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
      o[mt][0] *= al0;
      o[mt][1] *= al1;
      o[mt][2] *= al0;
      o[mt][3] *= al1;
    }
    if constexpr (FP8) {
      const int t0 = 2 * q4;
      const uint4 X = dev::lds128(vb + swz(t0, r));
      const uint4 Y = dev::lds128(vb + swz(t0 + 1, r));
      const uint4 Z = dev::lds128(vb + swz(t0 + 8, r));
      const uint4 W = dev::lds128(vb + swz(t0 + 9, r));
      const uint32_t xw[4] = {X.x, X.y, X.z, X.w}, yw[4] = {Y.x, Y.y, Y.z, Y.w};
      const uint32_t zw[4] = {Z.x, Z.y, Z.z, Z.w}, ww[4] = {W.x, W.y, W.z, W.w};
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
        const uint32_t xy = dev::prmt(xw[mt >> 1], yw[mt >> 1], sel);
        const uint32_t zv = dev::prmt(zw[mt >> 1], ww[mt >> 1], sel);
        uint32_t af[4];
        af[0] = dev::e4m3x2_to<QT>(static_cast<uint16_t>(xy & 0xffffu));
        af[1] = dev::e4m3x2_to<QT>(static_cast<uint16_t>(xy >> 16));
        af[2] = dev::e4m3x2_to<QT>(static_cast<uint16_t>(zv & 0xffffu));
        af[3] = dev::e4m3x2_to<QT>(static_cast<uint16_t>(zv >> 16));
        dev::Mma<QT>::run(o[mt], af, bh0, bh1);
        if constexpr (SPLIT_P) dev::Mma<QT>::run(o[mt], af, bl0, bl1);
      }
    } else {
      const int vrow = (lane & 7) + (lane >> 4) * 8;
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        uint32_t af[4];
        dev::ldmatrix_x4_trans(af, vb + swz(vrow, 2 * mt + ((lane >> 3) & 1)));
        dev::Mma<QT>::run(o[mt], af, bh0, bh1);
        if constexpr (SPLIT_P) dev::Mma<QT>::run(o[mt], af, bl0, bl1);
      }
    }

    __syncwarp();
    if (lane == 0) {
      const int jn = jj + kNSW * kNW;
      if (jn < nb) {
        dev::fence_proxy_async_smem();
        issue(jn, s);
      }
    }
  }

  // ---- merge the warps' partial softmax states ----------------------------------
  dev::grid_launch_dependents();  // the merge kernel may start being scheduled
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    l0 += __shfl_xor_sync(FULL, l0, off);
    l1 += __shfl_xor_sync(FULL, l1, off);
  }
  __syncthreads();  // every stage consumed: tile memory is free
  float* s_o = reinterpret_cast<float*>(base);  // [kNW][8][D]
  float* s_m = s_o + kNW * 8 * D;                // [kNW][8]
  float* s_l = s_m + kNW * 8;
  {
    const int hA = 2 * q4, hB = 2 * q4 + 1;
    float* ow = s_o + warp * 8 * D;
#pragma unroll
    for (int mt = 0; mt < MT; ++mt) {
      int d_r, d_r8;
      if constexpr (FP8) {
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
      s_m[warp * 8 + hA] = m0;
      s_m[warp * 8 + hB] = m1;
      s_l[warp * 8 + hA] = l0;
      s_l[warp * 8 + hB] = l1;
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < a.G * D; idx += blockDim.x) {
    const int h = idx / D, d = idx - h * D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kNW; ++w) M = fmaxf(M, s_m[w * 8 + h]);
    float acc = 0.f, ls = 0.f;
#pragma unroll
    for (int w = 0; w < kNW; ++w) {
      const float f = exp2f(s_m[w * 8 + h] - M);
      acc += f * s_o[(w * 8 + h) * D + d];
      ls += f * s_l[w * 8 + h];
    }
    const size_t head = static_cast<size_t>(b) * a.Hq + g * a.G + h;
    if (nparts == 1) {
      store_out<QT>(a, head * D + d, acc / ls);
    } else {
      const size_t row = head * a.max_parts + p;
      a.part_o[row * D + d] = acc;
      if (d == 0) {
        a.part_m[row] = M;
        a.part_l[row] = ls;
      }
    }
  }
}

// Merge the partitions of one (sequence, query head): log-sum-exp weights.
template <typename QT, int D>
__global__ void __launch_bounds__(D) decode_reduce(const DecodeArgs a) {
  const int h = blockIdx.x, b = blockIdx.y, d = threadIdx.x;
  dev::grid_dependency_wait();  // partials of decode_main are complete and visible
  const int L = checked_len(a, b, false);
  const int nblk = (L + 15) >> 4;
  const int nparts = (nblk + a.bpp - 1) / a.bpp;
  if (nparts <= 1) return;
  const size_t row0 = (static_cast<size_t>(b) * a.Hq + h) * a.max_parts;
  float M = -INFINITY;
  for (int p = 0; p < nparts; ++p) M = fmaxf(M, a.part_m[row0 + p]);
  float acc = 0.f, ls = 0.f;
  for (int p = 0; p < nparts; ++p) {
    const float f = exp2f(a.part_m[row0 + p] - M);
    acc += f * a.part_o[(row0 + p) * D + d];
    ls += f * a.part_l[row0 + p];
  }
  store_out<QT>(a, (static_cast<size_t>(b) * a.Hq + h) * D + d, acc / ls);
}

// ---- host side -------------------------------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// Tensor map over a cache viewed as [num_blocks][Hkv*16 rows][D], box = one
// 128-byte span of 16 rows (one kv head of one block), 128-byte swizzle.
template <typename KT, int D>
pa_status make_map(CUtensorMap* m, const void* cache, int Hkv, int num_blocks, CUtensorMapDataType dt) {
  using TL = Tile<KT, D>;
  auto fn = encode_fn();
  if (!fn) return fail(PA_ERR_CUDA, "pa_decode: cuTensorMapEncodeTiled unavailable");
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(16) * Hkv,
                              static_cast<cuuint64_t>(num_blocks)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(TL::ROWB),
                                 static_cast<cuuint64_t>(TL::ROWB) * 16 * Hkv};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(TL::BOXE), 16, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, dt, 3, const_cast<void*>(cache), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(PA_ERR_CUDA, "pa_decode: tensor map encode failed (%d)", static_cast<int>(r));
  return PA_OK;
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
  const size_t rows = static_cast<size_t>(l.B) * l.Hq * l.plan.max_parts;
  a.part_o = l.plan.max_parts > 1 ? static_cast<float*>(l.workspace) : nullptr;
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

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return fail(PA_ERR_CUDA, "pa_decode: no CUDA device");
  static std::once_flag attr_once[64];
  cudaError_t attr_err = cudaSuccess;
  auto set_attr = [&] {
    attr_err = cudaFuncSetAttribute(decode_main<KT, QT, D>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, TL::SMEM);
  };
  if (dev < 64)
    std::call_once(attr_once[dev], set_attr);
  else
    set_attr();
  if (attr_err != cudaSuccess) return fail(PA_ERR_CUDA, "pa_decode: %s", cudaGetErrorString(attr_err));

  const dim3 grid(static_cast<unsigned>(l.B * l.Hkv), static_cast<unsigned>(l.plan.max_parts));
  cudaError_t e = launch_dependent(decode_main<KT, QT, D>, grid, dim3(kNW * 32), TL::SMEM, stream,
                                   tmK, tmV, a);
  if (e == cudaSuccess && l.plan.max_parts > 1)
    e = launch_dependent(decode_reduce<QT, D>,
                         dim3(static_cast<unsigned>(l.Hq), static_cast<unsigned>(l.B)), dim3(D), 0,
                         stream, a);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "pa_decode launch: %s", cudaGetErrorString(e));
  return PA_OK;
}

}  // namespace

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
  // FP8 E4M3 codes, head_dim 128 (checked by the caller)
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
