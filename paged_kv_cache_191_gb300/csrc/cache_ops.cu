// Cache write, copy-on-write block copy and block swap for sm_103a.
//
// Cache write ("LLM推理引擎深度实战：从PagedAttention到分布式推理部署", 2.2:
// physical pages hold only generated tokens; "大模型推理引擎优化：KV Cache 与
// 连续批处理", 三: append reserves the slot): token i's K/V rows go to block
// slot/16, row slot%16 of every kv head.  Both kernels are HBM-bound byte
// movers: 16-byte vector loads and stores, one CTA per token (write) or per
// (pair, chunk) (copy).
//
// FP8 E4M3 and INT8 caches ("LLM推理引擎深度实战" 5.3): one float32 scale per
// token per tensor, scale = amax/448 (E4M3) or amax/127 (INT8) by IEEE
// division, code = RNE-satfinite E4M3, or round-to-nearest-even INT8, of
// x/scale (IEEE division), so the codes are a deterministic function of the
// input bits.
//
// Block copy ("LLM推理引擎深度实战" 2.2 copy-on-write; "大模型推理引擎优化" 4.2):
// whole K and V blocks (and their scale rows) are copied src -> dst.  Block
// swap ("LLM推理引擎深度实战" 3.2, preemption by moving a request's pages to CPU
// memory and back) is the same copy between two pools, one of them in
// page-locked host memory that the kernel addresses directly.
#include "device_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

__device__ uint32_t g_cache_err;

constexpr int kWriteThreads = 256;

// 8 consecutive input values as float, from f16 / bf16 / f32 storage.
template <int IN>
__device__ __forceinline__ void load8(const void* base, size_t idx, float (&x)[8]) {
  if constexpr (IN == PA_DTYPE_F32) {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + idx);
    const float4 a = p[0], b = p[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  } else {
    const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + idx);
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 f;
      if constexpr (IN == PA_DTYPE_F16)
        f = dev::unpack2<__half>(w[i]);
      else
        f = dev::unpack2<__nv_bfloat16>(w[i]);
      x[2 * i] = f.x;
      x[2 * i + 1] = f.y;
    }
  }
}

// 16-bit cache: copy (same dtype, exact) or round from f32.
template <int IN, int KV>
__global__ void __launch_bounds__(kWriteThreads)
    cache_write_16(const void* __restrict__ k, const void* __restrict__ v,
                   const int64_t* __restrict__ slots, void* __restrict__ kc, void* __restrict__ vc,
                   int Hkv, int D, int num_blocks) {
  dev::grid_dependency_wait();
  dev::grid_launch_dependents();  // a dependent decode waits for our completion itself
  const int t = blockIdx.x;
  const int64_t slot = slots[t];
  if (slot < 0) return;
  if (slot >= static_cast<int64_t>(num_blocks) * PA_BLOCK_SIZE) {
    if (threadIdx.x == 0) atomicOr(&g_cache_err, PA_DEVERR_SLOT_RANGE);
    return;
  }
  const int64_t blk = slot / PA_BLOCK_SIZE, off = slot % PA_BLOCK_SIZE;
  const int vpr = D / 8;  // 8-element vectors per head row
  const int nvec = Hkv * vpr;
  for (int i = threadIdx.x; i < 2 * nvec; i += blockDim.x) {
    const bool isv = i >= nvec;
    const int j = isv ? i - nvec : i;
    const int h = j / vpr, c = j - h * vpr;
    const size_t src = (static_cast<size_t>(t) * Hkv + h) * D + c * 8;
    const size_t dst = ((static_cast<size_t>(blk) * Hkv + h) * PA_BLOCK_SIZE + off) * D + c * 8;
    uint4 out;
    if constexpr (IN == KV) {
      out = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(isv ? v : k) + src);
    } else {
      float x[8];
      load8<IN>(isv ? v : k, src, x);
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if constexpr (KV == PA_DTYPE_F16)
          w[e] = dev::pack2<__half>(x[2 * e], x[2 * e + 1]);
        else
          w[e] = dev::pack2<__nv_bfloat16>(x[2 * e], x[2 * e + 1]);
      }
      out = make_uint4(w[0], w[1], w[2], w[3]);
    }
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(isv ? vc : kc) + dst) = out;
  }
}

__device__ __forceinline__ float block_max(float x, float* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) red[w] = x;
  __syncthreads();
  if (threadIdx.x < 32) {
    float y = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) y = fmaxf(y, __shfl_xor_sync(0xffffffffu, y, off));
    if (threadIdx.x == 0) red[32] = y;
  }
  __syncthreads();
  return red[32];
}

// One code of a quantised cache from a float already divided by the scale:
// E4M3 round-to-nearest-even saturating to finite, or INT8 round-to-nearest-
// even (the scale makes |x| <= 127 up to its own rounding; clamped).
template <bool INT8>
__device__ __forceinline__ uint32_t encode_q8(float x) {
  if constexpr (INT8)
    return static_cast<uint32_t>(static_cast<uint8_t>(static_cast<int8_t>(max(-127, min(127, __float2int_rn(x))))));
  else
    return __nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}

// Quantised cache (E4M3 or INT8): per-token amax -> scale -> codes, for K then V.
template <int IN, bool INT8>
__global__ void __launch_bounds__(kWriteThreads)
    cache_write_q8(const void* __restrict__ k, const void* __restrict__ v,
                    const int64_t* __restrict__ slots, uint8_t* __restrict__ kc,
                    uint8_t* __restrict__ vc, float* __restrict__ ks, float* __restrict__ vs,
                    int Hkv, int D, int num_blocks) {
  __shared__ float red[33];
  dev::grid_dependency_wait();
  dev::grid_launch_dependents();
  const int t = blockIdx.x;
  const int64_t slot = slots[t];
  if (slot < 0) return;
  if (slot >= static_cast<int64_t>(num_blocks) * PA_BLOCK_SIZE) {
    if (threadIdx.x == 0) atomicOr(&g_cache_err, PA_DEVERR_SLOT_RANGE);
    return;
  }
  const int64_t blk = slot / PA_BLOCK_SIZE, off = slot % PA_BLOCK_SIZE;
  const int vpr = D / 8;
  const int nvec = Hkv * vpr;
#pragma unroll 1
  for (int which = 0; which < 2; ++which) {
    const void* src = which ? v : k;
    uint8_t* cache = which ? vc : kc;
    float amax = 0.f;
    for (int j = threadIdx.x; j < nvec; j += blockDim.x) {
      float x[8];
      load8<IN>(src, static_cast<size_t>(t) * Hkv * D + static_cast<size_t>(j) * 8, x);
#pragma unroll
      for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(x[e]));
    }
    amax = block_max(amax, red);
    const float scale = amax > 0.f ? __fdiv_rn(amax, INT8 ? 127.0f : 448.0f) : 1.0f;
    for (int j = threadIdx.x; j < nvec; j += blockDim.x) {
      const int h = j / vpr, c = j - h * vpr;
      float x[8];
      load8<IN>(src, (static_cast<size_t>(t) * Hkv + h) * D + c * 8, x);
      uint32_t lo = 0, hi = 0;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t code = encode_q8<INT8>(__fdiv_rn(x[e], scale));
        if (e < 4)
          lo |= code << (8 * e);
        else
          hi |= code << (8 * (e - 4));
      }
      const size_t dst = ((static_cast<size_t>(blk) * Hkv + h) * PA_BLOCK_SIZE + off) * D + c * 8;
      *reinterpret_cast<uint2*>(cache + dst) = make_uint2(lo, hi);
    }
    if (threadIdx.x == 0) (which ? vs : ks)[slot] = scale;
    __syncthreads();  // `red` is reused by the next tensor
  }
}

constexpr int kCopyThreads = 256;
constexpr int kCopyChunk = 16384;  // bytes of one block copied by one CTA

// A pool of whole blocks: K, V (and FP8 scales) laid out like a cache.
struct BlockPool {
  uint8_t* k;
  uint8_t* v;
  float* ks;  // [num_blocks][16] or null
  float* vs;
  int num_blocks;
};

// Copy block pairs[i] = (src, dst) from pool `from` to pool `to` (the same
// pool for copy-on-write, a pinned host pool for swapping).  One CTA per
// (pair, 16 KB chunk); ids outside either pool are skipped and flagged.
__global__ void __launch_bounds__(kCopyThreads)
    copy_blocks_kernel(BlockPool to, BlockPool from, const int64_t* __restrict__ pairs,
                       size_t block_bytes) {
  const int64_t src = pairs[2 * blockIdx.x], dst = pairs[2 * blockIdx.x + 1];
  if (src < 0 || src >= from.num_blocks || dst < 0 || dst >= to.num_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0) atomicOr(&g_cache_err, PA_DEVERR_BLOCK_RANGE);
    return;
  }
  const size_t begin = static_cast<size_t>(blockIdx.y) * kCopyChunk;
  const size_t end = min(begin + kCopyChunk, block_bytes);
  const uint4* ksrc = reinterpret_cast<const uint4*>(from.k + src * block_bytes);
  const uint4* vsrc = reinterpret_cast<const uint4*>(from.v + src * block_bytes);
  uint4* kdst = reinterpret_cast<uint4*>(to.k + dst * block_bytes);
  uint4* vdst = reinterpret_cast<uint4*>(to.v + dst * block_bytes);
  for (size_t i = begin / 16 + threadIdx.x; i < end / 16; i += blockDim.x) {
    const uint4 a = ksrc[i], b = vsrc[i];
    kdst[i] = a;
    vdst[i] = b;
  }
  if (from.ks && blockIdx.y == 0 && threadIdx.x < PA_BLOCK_SIZE) {
    to.ks[dst * PA_BLOCK_SIZE + threadIdx.x] = from.ks[src * PA_BLOCK_SIZE + threadIdx.x];
    to.vs[dst * PA_BLOCK_SIZE + threadIdx.x] = from.vs[src * PA_BLOCK_SIZE + threadIdx.x];
  }
}

template <int IN>
void launch_q8(const void* k, const void* v, const int64_t* s, int64_t T, void* kc, void* vc,
               float* ks, float* vs, const pa_cache_desc* d, cudaStream_t st) {
  auto kernel = d->kv_dtype == PA_DTYPE_INT8 ? cache_write_q8<IN, true> : cache_write_q8<IN, false>;
  kernel<<<static_cast<unsigned>(T), kWriteThreads, 0, st>>>(
      k, v, s, static_cast<uint8_t*>(kc), static_cast<uint8_t*>(vc), ks, vs, d->num_kv_heads,
      d->head_dim, d->num_blocks);
}

}  // namespace

pa_status launch_cache_write(const void* k, const void* v, int32_t in_dtype, const int64_t* slots,
                             int64_t T, void* kc, void* vc, float* ks, float* vs,
                             const pa_cache_desc* d, void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const unsigned grid = static_cast<unsigned>(T);
  const int H = d->num_kv_heads, D = d->head_dim, N = d->num_blocks;
  switch (d->kv_dtype) {
    case PA_DTYPE_F16:
      if (in_dtype == PA_DTYPE_F16)
        cache_write_16<PA_DTYPE_F16, PA_DTYPE_F16><<<grid, kWriteThreads, 0, st>>>(k, v, slots, kc, vc, H, D, N);
      else
        cache_write_16<PA_DTYPE_F32, PA_DTYPE_F16><<<grid, kWriteThreads, 0, st>>>(k, v, slots, kc, vc, H, D, N);
      break;
    case PA_DTYPE_BF16:
      if (in_dtype == PA_DTYPE_BF16)
        cache_write_16<PA_DTYPE_BF16, PA_DTYPE_BF16><<<grid, kWriteThreads, 0, st>>>(k, v, slots, kc, vc, H, D, N);
      else
        cache_write_16<PA_DTYPE_F32, PA_DTYPE_BF16><<<grid, kWriteThreads, 0, st>>>(k, v, slots, kc, vc, H, D, N);
      break;
    default:
      if (in_dtype == PA_DTYPE_F16)
        launch_q8<PA_DTYPE_F16>(k, v, slots, T, kc, vc, ks, vs, d, st);
      else if (in_dtype == PA_DTYPE_BF16)
        launch_q8<PA_DTYPE_BF16>(k, v, slots, T, kc, vc, ks, vs, d, st);
      else
        launch_q8<PA_DTYPE_F32>(k, v, slots, T, kc, vc, ks, vs, d, st);
      break;
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "pa_cache_write launch: %s", cudaGetErrorString(e));
  return PA_OK;
}

static pa_status launch_pool_copy(const BlockPool& to, const BlockPool& from, const int64_t* pairs,
                                  int64_t n, const pa_cache_desc* d, void* stream, const char* what) {
  const size_t block_bytes = static_cast<size_t>(d->num_kv_heads) * PA_BLOCK_SIZE * d->head_dim *
                             dtype_bytes(d->kv_dtype);
  const unsigned chunks = static_cast<unsigned>((block_bytes + kCopyChunk - 1) / kCopyChunk);
  copy_blocks_kernel<<<dim3(static_cast<unsigned>(n), chunks), kCopyThreads, 0,
                       static_cast<cudaStream_t>(stream)>>>(to, from, pairs, block_bytes);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "%s launch: %s", what, cudaGetErrorString(e));
  return PA_OK;
}

pa_status launch_copy_blocks(void* kc, void* vc, float* ks, float* vs, const int64_t* pairs,
                             int64_t n, const pa_cache_desc* d, void* stream) {
  const BlockPool pool{static_cast<uint8_t*>(kc), static_cast<uint8_t*>(vc), ks, vs, d->num_blocks};
  return launch_pool_copy(pool, pool, pairs, n, d, stream, "pa_copy_blocks");
}

pa_status launch_swap_blocks(void* dk, void* dv, float* dks, float* dvs, int32_t dnb, const void* sk,
                             const void* sv, const float* sks, const float* svs, int32_t snb,
                             const int64_t* pairs, int64_t n, const pa_cache_desc* d, void* stream) {
  const BlockPool to{static_cast<uint8_t*>(dk), static_cast<uint8_t*>(dv), dks, dvs, dnb};
  const BlockPool from{static_cast<uint8_t*>(const_cast<void*>(sk)), static_cast<uint8_t*>(const_cast<void*>(sv)),
                       const_cast<float*>(sks), const_cast<float*>(svs), snb};
  return launch_pool_copy(to, from, pairs, n, d, stream, "pa_swap_blocks");
}

pa_status read_errors_cache_ops(uint32_t* flags, bool clear) {
  uint32_t v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_cache_err, sizeof(v));
  if (e == cudaSuccess && clear) {
    const uint32_t z = 0;
    e = cudaMemcpyToSymbol(g_cache_err, &z, sizeof(z));
  }
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "pa_device_errors: %s", cudaGetErrorString(e));
  *flags = v;
  return PA_OK;
}

}  // namespace pa
