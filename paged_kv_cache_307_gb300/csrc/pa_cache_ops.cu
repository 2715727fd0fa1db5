// pa_cache_ops.cu — KV append (reshape_and_cache) and copy-on-write block copy.
//
// Both are pure data movement, bound by HBM bandwidth, and must be byte-exact:
//  * append: "19.2 KV Cache 系统化管理" §19.2.3 (a token's K/V written into a
//    slot of a physical block; slot from the block-table append) and Fig 19-6
//    (decode appends into the partly filled last block);
//  * copy: the same page's Fig 19-8 (copy-on-write: a new block receives the
//    old block's contents before the table is remapped) and "LLM 推理引擎的
//    内存管理与调度…" §四.
//
//  * fp8 append: the same write, with each token's K vector and V vector
//    quantised on their own ("19.2 KV Cache 系统化管理" §19.2.4, per-token
//    scaling): scale = amax/448, codes = e4m3(x * (448/amax)), rounded to
//    nearest even with saturation, all in fp32.
//
// Layout: each token's K (or V) row for all heads, [Hkv, D], is contiguous in
// both the source [T, Hkv, D] and the pool [NB, bs, Hkv, D]; a whole block is
// contiguous too.  So both kernels are 16-byte vector copies of contiguous
// spans: one CTA per (token, K|V) for the append, one CTA per (pair, K|V,
// span) for the block copy.  Loads use the non-coherent path with no L1
// allocation (each byte is read once); several 16-byte loads are in flight
// per thread before the stores.
#include "pa_common.cuh"

namespace pa {
namespace {

__device__ unsigned g_status_cache;

constexpr int kCopyThreads = 256;
constexpr int kUnroll = 4;

// Copy `chunks` 16-byte chunks from src to dst with the whole CTA.
__device__ __forceinline__ void cta_copy16(unsigned char* __restrict__ dst,
                                           const unsigned char* __restrict__ src, int chunks) {
  int c = threadIdx.x;
  for (; c + (kUnroll - 1) * kCopyThreads < chunks; c += kUnroll * kCopyThreads) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = ld_nc_v4(src + (size_t)(c + u * kCopyThreads) * 16);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) st_v4(dst + (size_t)(c + u * kCopyThreads) * 16, v[u]);
  }
  for (; c < chunks; c += kCopyThreads) st_v4(dst + (size_t)c * 16, ld_nc_v4(src + (size_t)c * 16));
}

// grid: (num_tokens, 2).  blockIdx.y selects K (0) or V (1).
__global__ void __launch_bounds__(kCopyThreads)
reshape_and_cache_kernel(const unsigned char* __restrict__ key, const unsigned char* __restrict__ value,
                         const int64_t* __restrict__ slot_mapping,
                         unsigned char* __restrict__ k_cache, unsigned char* __restrict__ v_cache,
                         long long num_slots, int row_bytes) {
  const int t = blockIdx.x;
  const long long slot = slot_mapping[t];
  if (slot < 0) return;                       // padding
  if (slot >= num_slots) {
    if (threadIdx.x == 0 && blockIdx.y == 0) atomicOr(&g_status_cache, PA_DEV_BAD_SLOT);
    return;
  }
  const unsigned char* src = (blockIdx.y == 0 ? key : value) + (size_t)t * row_bytes;
  unsigned char* dst = (blockIdx.y == 0 ? k_cache : v_cache) + (size_t)slot * row_bytes;
  cta_copy16(dst, src, row_bytes / 16);
}

// grid: (num_tokens, 2).  Quantise token t's K (y = 0) or V (y = 1) row of
// n = Hkv*D elements of type T into e4m3 codes plus one fp32 scale.
template <typename T>
__global__ void __launch_bounds__(kCopyThreads)
reshape_and_cache_fp8_kernel(const T* __restrict__ key, const T* __restrict__ value,
                             const int64_t* __restrict__ slot_mapping, uint8_t* __restrict__ k_cache,
                             uint8_t* __restrict__ v_cache, float* __restrict__ k_scale, float* __restrict__ v_scale,
                             long long num_slots, int n) {
  using E = Elem<T>;
  constexpr int EPC = E::kPerChunk;   // elements per 16-byte chunk
  __shared__ float red[kCopyThreads / 32];
  const int t = blockIdx.x;
  const long long slot = slot_mapping[t];
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (threadIdx.x == 0 && blockIdx.y == 0) atomicOr(&g_status_cache, PA_DEV_BAD_SLOT);
    return;
  }
  const unsigned char* src = reinterpret_cast<const unsigned char*>(blockIdx.y == 0 ? key : value) +
                             (size_t)t * n * sizeof(T);
  uint8_t* dst = (blockIdx.y == 0 ? k_cache : v_cache) + (size_t)slot * n;
  const int chunks = n / EPC;
  float amax = 0.f;
  for (int c = threadIdx.x; c < chunks; c += kCopyThreads) {
    float f[EPC];
    E::unpack(ld_nc_v4(src + (size_t)c * 16), f);
#pragma unroll
    for (int e = 0; e < EPC; ++e) amax = fmaxf(amax, fabsf(f[e]));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = red[0];
#pragma unroll
  for (int w = 1; w < kCopyThreads / 32; ++w) amax = fmaxf(amax, red[w]);
  const float inv = amax > 0.f ? __fdiv_rn(448.f, amax) : 0.f;
  for (int c = threadIdx.x; c < chunks; c += kCopyThreads) {
    float f[EPC];
    E::unpack(ld_nc_v4(src + (size_t)c * 16), f);
    uint32_t w[EPC / 4];
#pragma unroll
    for (int i = 0; i < EPC / 4; ++i) {
      uint32_t v = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t code = amax > 0.f ? (uint32_t)__nv_cvt_float_to_fp8(__fmul_rn(f[4 * i + e], inv),
                                                                           __NV_SATFINITE, __NV_E4M3)
                                         : 0u;
        v |= code << (8 * e);
      }
      w[i] = v;
    }
    if constexpr (EPC == 8) {
      *reinterpret_cast<uint2*>(dst + (size_t)c * EPC) = make_uint2(w[0], w[1]);
    } else {
      *reinterpret_cast<uint32_t*>(dst + (size_t)c * EPC) = w[0];
    }
  }
  if (threadIdx.x == 0) (blockIdx.y == 0 ? k_scale : v_scale)[slot] = amax > 0.f ? __fdiv_rn(amax, 448.f) : 0.f;
}

// grid: (num_pairs, 2, spans).  Each CTA copies one span of one block.
__global__ void __launch_bounds__(kCopyThreads)
copy_blocks_kernel(unsigned char* __restrict__ k_cache, unsigned char* __restrict__ v_cache,
                   const int64_t* __restrict__ pairs, long long num_blocks,
                   long long block_bytes, int span_bytes) {
  const long long src = pairs[2 * (size_t)blockIdx.x];
  const long long dst = pairs[2 * (size_t)blockIdx.x + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) atomicOr(&g_status_cache, PA_DEV_BAD_BLOCK);
    return;
  }
  if (src == dst) return;     // a block copied onto itself is unchanged (and would alias the restrict operands)
  unsigned char* base = blockIdx.y == 0 ? k_cache : v_cache;
  const long long off = (long long)blockIdx.z * span_bytes;
  const long long n = block_bytes - off < span_bytes ? block_bytes - off : span_bytes;
  cta_copy16(base + dst * block_bytes + off, base + src * block_bytes + off, (int)(n / 16));
}

// Coherent 16-byte copy (the source may be page-locked host memory).
__device__ __forceinline__ void cta_copy16_coherent(unsigned char* __restrict__ dst,
                                                    const unsigned char* __restrict__ src, int chunks) {
  int c = threadIdx.x;
  for (; c + (kUnroll - 1) * kCopyThreads < chunks; c += kUnroll * kCopyThreads) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) v[u] = *reinterpret_cast<const uint4*>(src + (size_t)(c + u * kCopyThreads) * 16);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) st_v4(dst + (size_t)(c + u * kCopyThreads) * 16, v[u]);
  }
  for (; c < chunks; c += kCopyThreads)
    st_v4(dst + (size_t)c * 16, *reinterpret_cast<const uint4*>(src + (size_t)c * 16));
}

// grid: (num_pairs, 2, spans).  Block pairs[i,1] of the destination pool
// becomes a copy of block pairs[i,0] of the source pool.
__global__ void __launch_bounds__(kCopyThreads)
swap_blocks_kernel(unsigned char* __restrict__ dst_k, unsigned char* __restrict__ dst_v,
                   const unsigned char* __restrict__ src_k, const unsigned char* __restrict__ src_v,
                   const int64_t* __restrict__ pairs, long long src_blocks, long long dst_blocks,
                   long long block_bytes, int span_bytes) {
  const long long src = pairs[2 * (size_t)blockIdx.x];
  const long long dst = pairs[2 * (size_t)blockIdx.x + 1];
  if (src < 0 || src >= src_blocks || dst < 0 || dst >= dst_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) atomicOr(&g_status_cache, PA_DEV_BAD_BLOCK);
    return;
  }
  const long long off = (long long)blockIdx.z * span_bytes;
  const long long n = block_bytes - off < span_bytes ? block_bytes - off : span_bytes;
  unsigned char* d = (blockIdx.y == 0 ? dst_k : dst_v) + dst * block_bytes + off;
  const unsigned char* s = (blockIdx.y == 0 ? src_k : src_v) + src * block_bytes + off;
  cta_copy16_coherent(d, s, (int)(n / 16));
}

}  // namespace

// Block copies move whole blocks as 16-byte chunks: any shape whose block is
// a whole number of chunks (this includes the [NB, bs, 1, 1] fp32 scale rows
// of an e4m3 pool).
static bool copyable_block(int block_size, int heads, int dim, pa_dtype dt) {
  if (!supported_block_size(block_size) || heads <= 0 || dim <= 0) return false;
  const long long bytes = (long long)block_size * heads * dim * elem_bytes(dt);
  return bytes % 16 == 0 && bytes <= (1ll << 30);
}

unsigned fetch_status_cache_ops() {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_status_cache, sizeof(v)) != cudaSuccess) return 0xffffffffu;
  if (v && cudaMemcpyToSymbol(g_status_cache, &zero, sizeof(zero)) != cudaSuccess) return 0xffffffffu;
  return v;
}

}  // namespace pa

using namespace pa;

extern "C" int pa_reshape_and_cache(const void* key, const void* value, const int64_t* slot_mapping,
                                    int num_tokens, void* k_cache, void* v_cache, int num_blocks,
                                    int block_size, int num_kv_heads, int head_dim, pa_dtype dtype,
                                    void* stream) {
  if (dtype != PA_F32 && dtype != PA_BF16) return PA_ERR_DTYPE;
  if (num_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0 || !supported_head_dim(head_dim) ||
      !supported_block_size(block_size))
    return PA_ERR_SHAPE;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !slot_mapping || !k_cache || !v_cache) return PA_ERR_NULL;
  if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_ALIGN;
  const int row_bytes = num_kv_heads * head_dim * elem_bytes(dtype);
  dim3 grid((unsigned)num_tokens, 2);
  reshape_and_cache_kernel<<<grid, kCopyThreads, 0, (cudaStream_t)stream>>>(
      (const unsigned char*)key, (const unsigned char*)value, slot_mapping, (unsigned char*)k_cache,
      (unsigned char*)v_cache, (long long)num_blocks * block_size, row_bytes);
  return ck(cudaGetLastError(), "launch reshape_and_cache_kernel") ? PA_OK : PA_ERR_CUDA;
}

extern "C" int pa_copy_blocks(void* k_cache, void* v_cache, const int64_t* pairs, int num_pairs,
                              int num_blocks, int block_size, int num_kv_heads, int head_dim,
                              pa_dtype dtype, void* stream) {
  if (dtype != PA_F32 && dtype != PA_BF16 && dtype != PA_FP8_E4M3) return PA_ERR_DTYPE;
  if (num_pairs < 0 || num_blocks <= 0 || !copyable_block(block_size, num_kv_heads, head_dim, dtype))
    return PA_ERR_SHAPE;
  if (num_pairs == 0) return PA_OK;
  if (!k_cache || !v_cache || !pairs) return PA_ERR_NULL;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_ALIGN;
  const long long block_bytes = (long long)block_size * num_kv_heads * head_dim * elem_bytes(dtype);
  const int span = 32 * 1024;
  const unsigned spans = (unsigned)((block_bytes + span - 1) / span);
  dim3 grid((unsigned)num_pairs, 2, spans);
  copy_blocks_kernel<<<grid, kCopyThreads, 0, (cudaStream_t)stream>>>(
      (unsigned char*)k_cache, (unsigned char*)v_cache, pairs, num_blocks, block_bytes, span);
  return ck(cudaGetLastError(), "launch copy_blocks_kernel") ? PA_OK : PA_ERR_CUDA;
}

extern "C" int pa_swap_blocks(void* dst_k, void* dst_v, int dst_num_blocks, const void* src_k, const void* src_v,
                              int src_num_blocks, const int64_t* pairs, int num_pairs, int block_size,
                              int num_kv_heads, int head_dim, pa_dtype dtype, void* stream) {
  if (dtype != PA_F32 && dtype != PA_BF16 && dtype != PA_FP8_E4M3) return PA_ERR_DTYPE;
  if (num_pairs < 0 || dst_num_blocks <= 0 || src_num_blocks <= 0 ||
      !copyable_block(block_size, num_kv_heads, head_dim, dtype))
    return PA_ERR_SHAPE;
  if (num_pairs == 0) return PA_OK;
  if (!dst_k || !dst_v || !src_k || !src_v || !pairs) return PA_ERR_NULL;
  if (!aligned16(dst_k) || !aligned16(dst_v) || !aligned16(src_k) || !aligned16(src_v)) return PA_ERR_ALIGN;
  const long long block_bytes = (long long)block_size * num_kv_heads * head_dim * elem_bytes(dtype);
  const int span = 32 * 1024;
  const unsigned spans = (unsigned)((block_bytes + span - 1) / span);
  dim3 grid((unsigned)num_pairs, 2, spans);
  swap_blocks_kernel<<<grid, kCopyThreads, 0, (cudaStream_t)stream>>>(
      (unsigned char*)dst_k, (unsigned char*)dst_v, (const unsigned char*)src_k, (const unsigned char*)src_v, pairs,
      src_num_blocks, dst_num_blocks, block_bytes, span);
  return ck(cudaGetLastError(), "launch swap_blocks_kernel") ? PA_OK : PA_ERR_CUDA;
}

extern "C" int pa_reshape_and_cache_fp8(const void* key, const void* value, const int64_t* slot_mapping,
                                        int num_tokens, void* k_cache, void* v_cache, float* k_scale,
                                        float* v_scale, int num_blocks, int block_size, int num_kv_heads,
                                        int head_dim, pa_dtype src_dtype, void* stream) {
  if (src_dtype != PA_F32 && src_dtype != PA_BF16) return PA_ERR_DTYPE;
  if (num_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0 || !supported_head_dim(head_dim) ||
      !supported_block_size(block_size))
    return PA_ERR_SHAPE;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !slot_mapping || !k_cache || !v_cache || !k_scale || !v_scale) return PA_ERR_NULL;
  if (!aligned16(key) || !aligned16(value) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_scale) ||
      !aligned16(v_scale))
    return PA_ERR_ALIGN;
  const int n = num_kv_heads * head_dim;
  dim3 grid((unsigned)num_tokens, 2);
  const long long slots = (long long)num_blocks * block_size;
  if (src_dtype == PA_BF16)
    reshape_and_cache_fp8_kernel<__nv_bfloat16><<<grid, kCopyThreads, 0, (cudaStream_t)stream>>>(
        (const __nv_bfloat16*)key, (const __nv_bfloat16*)value, slot_mapping, (uint8_t*)k_cache,
        (uint8_t*)v_cache, k_scale, v_scale, slots, n);
  else
    reshape_and_cache_fp8_kernel<float><<<grid, kCopyThreads, 0, (cudaStream_t)stream>>>(
        (const float*)key, (const float*)value, slot_mapping, (uint8_t*)k_cache, (uint8_t*)v_cache, k_scale,
        v_scale, slots, n);
  return ck(cudaGetLastError(), "launch reshape_and_cache_fp8_kernel") ? PA_OK : PA_ERR_CUDA;
}
