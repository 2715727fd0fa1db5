// pa_decode.cu — host side of paged decode attention (pa_decode,
// pa_decode_fp8, pa_decode_noalloc) and the f32/bf16-pool kernel instances.
//
// The kernels themselves (what they compute and how) are in
// pa_decode_kernel.cuh; the e4m3-pool instances are compiled in
// pa_decode_fp8.cu.  This file picks the variant for the arguments (CUDA-core
// or tensor-core path, KV heads per work item, query heads per item), builds
// the tensor maps of the K/V pools (cached per pool), sizes the stage rings
// and the persistent grid from the occupancy, and launches the decode kernel
// and, when any sequence spans several partitions, the merge kernel.
#include "pa_decode_kernel.cuh"

#include <mutex>
#include <map>
#include <tuple>
#include <stdio.h>

namespace pa {
namespace {

// ------------------------------------------------------------------ host side

// Launch-shape parameters of the CUDA-core path (compile-time defaults).
#ifndef PA_FFMA_STAGE_BUDGET
#define PA_FFMA_STAGE_BUDGET 65536    // bytes of K/V stages per CTA
#endif
#ifndef PA_MAX_STAGES_PER_GROUP
#define PA_MAX_STAGES_PER_GROUP 4
#endif
#ifndef PA_MHA_HEADS_PER_ITEM
#define PA_MHA_HEADS_PER_ITEM 1       // bf16 pools, head_dim 128, one query head per KV head
#endif

// CUDA-core variant: KT is the pool's element type, HG KV heads per item.
template <typename T, typename KT, int D, int GT, int HG = 1>
Launch pick3() {
  return {reinterpret_cast<const void*>(&decode_kernel<T, KT, D, GT, false, HG>),
          reinterpret_cast<const void*>(&merge_kernel<T, D>)};
}

// Tensor-core GQA variant: bf16, head_dim 64 or 128, GT query heads per KV head.
template <int D, int GT>
Launch pick_mma_hg(int hg) {
  const void* merge = reinterpret_cast<const void*>(&merge_kernel<__nv_bfloat16, D>);
  using B16 = __nv_bfloat16;
  if (hg == 4) return {reinterpret_cast<const void*>(&decode_kernel<B16, B16, D, GT, true, 4>), merge};
  if (hg == 2) return {reinterpret_cast<const void*>(&decode_kernel<B16, B16, D, GT, true, 2>), merge};
  return {reinterpret_cast<const void*>(&decode_kernel<B16, B16, D, GT, true, 1>), merge};
}

template <int D>
Launch pick_mma(int gt, int hg) {
  if (gt == 16) return pick_mma_hg<D, 16>(hg);
  if (gt == 8) return pick_mma_hg<D, 8>(hg);
  if (gt == 4) return pick_mma_hg<D, 4>(hg);
  return pick_mma_hg<D, 2>(hg);
}

template <typename T, typename KT, int D>
Launch pick2(int gt, int hg) {
  if (gt == 4) return pick3<T, KT, D, 4>();
  if (gt == 2) return pick3<T, KT, D, 2>();
  if constexpr (PA_MHA_HEADS_PER_ITEM > 1 && D == 128 && sizeof(T) == 2)
    if (hg == PA_MHA_HEADS_PER_ITEM) return pick3<T, KT, D, 1, PA_MHA_HEADS_PER_ITEM>();
  return pick3<T, KT, D, 1>();
}

template <typename T, typename KT>
Launch pick1(int d, int gt, int hg) {
  if (d == 32) return pick2<T, KT, 32>(gt, hg);
  if (d == 64) return pick2<T, KT, 64>(gt, hg);
  return pick2<T, KT, 128>(gt, hg);
}

struct KernelInfo {
  int occupancy = 0;
};

std::mutex g_mu;
std::map<std::tuple<const void*, int, size_t>, KernelInfo> g_kinfo;  // (kernel, device, smem)

struct MapKey {
  const void* base;
  int dt, nb, bs, h, d, dev, swz, boxh;
  bool operator<(const MapKey& o) const {
    return std::tie(base, dt, nb, bs, h, d, dev, swz, boxh) <
           std::tie(o.base, o.dt, o.nb, o.bs, o.h, o.d, o.dev, o.swz, o.boxh);
  }
};
std::map<MapKey, CUtensorMap> g_maps;

// swz = false: box {D, boxh heads, bs, 1 block}, no swizzle (CUDA-core path).
// swz = true: box {64, 1 head, bs, 1 block}, 128-byte swizzle (tensor-core path).
bool get_map(CUtensorMap* out, const void* base, pa_dtype dt, int nb, int bs, int h, int d, int dev, bool swz,
             int boxh) {
  MapKey key{base, (int)dt, nb, bs, h, d, dev, swz ? 1 : 0, swz ? 1 : boxh};
  std::lock_guard<std::mutex> lk(g_mu);
  auto f = g_maps.find(key);
  if (f != g_maps.end()) {
    *out = f->second;
    return true;
  }
  bool ok;
  if (swz) {
    const uint64_t e = (uint64_t)elem_bytes(dt);
    const uint64_t dims[4] = {(uint64_t)d, (uint64_t)h, (uint64_t)bs, (uint64_t)nb};
    const uint64_t str[3] = {d * e, (uint64_t)h * d * e, (uint64_t)bs * h * d * e};
    const uint32_t box[4] = {(uint32_t)(128 / e), 1, (uint32_t)bs, 1};   // one 128-byte row span
    ok = encode_map(out, base, dt, 4, dims, str, box, true);
  } else {
    const uint64_t e = (uint64_t)elem_bytes(dt);
    const uint64_t dims[4] = {(uint64_t)d, (uint64_t)h, (uint64_t)bs, (uint64_t)nb};
    const uint64_t str[3] = {d * e, (uint64_t)h * d * e, (uint64_t)bs * h * d * e};
    const uint32_t box[4] = {(uint32_t)d, (uint32_t)boxh, (uint32_t)bs, 1};
    ok = encode_map(out, base, dt, 4, dims, str, box, false);
  }
  if (!ok) return false;
  if (g_maps.size() > 64) g_maps.clear();
  g_maps[key] = *out;
  return true;
}

int occupancy_for(const void* kernel, size_t smem, int dev) {
  std::lock_guard<std::mutex> lk(g_mu);
  auto key = std::make_tuple(kernel, dev, smem);
  auto f = g_kinfo.find(key);
  if (f != g_kinfo.end()) return f->second.occupancy;
  // The dynamic shared-memory limit is a property of the kernel function, so
  // raise it once to the device's opt-in maximum (never per launch size).
  if (!raise_smem_limit(kernel, dev)) return 0;
  int occ = 0;
  if (!ck(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kThreads, smem),
          "cudaOccupancyMaxActiveBlocksPerMultiprocessor"))
    return 0;
  g_kinfo[key] = KernelInfo{occ};
  return occ;
}

// KV heads per work item for e4m3 pools: one TMA box and one pair of scale
// copies then serve several heads, so the single producer thread moves more
// bytes per instruction (an e4m3 tile is half a bf16 one).
#ifndef PA_FP8_HEADS_PER_ITEM
#define PA_FP8_HEADS_PER_ITEM 2
#endif
int fp8_heads_per_item(int num_kv_heads) {
  int hg = PA_FP8_HEADS_PER_ITEM > 2 ? 2 : PA_FP8_HEADS_PER_ITEM;   // instances: 1 or 2
  while (hg > 1 && num_kv_heads % hg) hg >>= 1;
  return hg;
}

// Automatic split.  MHA: 256 tokens over 16-bit pools (finer items balance
// the persistent grid better than 512: c2 +0.5 %, c3 +1.3 %) and 512 over
// e4m3 pools, where an item's fixed costs (table read, lane and warp merges,
// the partial's write) weigh on half the bytes (c2 over e4m3: +7 %).  GQA:
// items already cover several query heads per K/V read, and long partitions
// (2048 tokens) measured best while the batch alone gives the grid enough
// items; a batch with fewer unsplit items than three per CTA of the grid
// (two CTAs on each of GB300's 152 SMs) is cut finer, to about sixteen items
// per SM at the table's capacity (the lengths themselves are on the device),
// between 256 and 2048 tokens.  On 256 requests over contexts U[128, 2048]
// the 2048-token split left a third of the SM time idle in the grid's tail;
// 256 tokens were 1.28x faster.
constexpr long long kGridCtas = 2 * 152;
int resolve_partition(int max_blocks, int bs, int partition_size, int G, bool fp8, int num_seqs,
                      int num_kv_heads) {
  const int max_ctx = max_blocks * bs;
  if (partition_size < 0) return max_ctx;
  int P = partition_size;
  if (P <= 0) {
    if (G < 2) {
      P = fp8 ? 512 : 256;
    } else {
      const long long items = (long long)num_seqs * ((num_kv_heads + 3) / 4);   // one partition each
      P = 2048;
      if (items < 3 * kGridCtas) {
        const long long want = (long long)max_ctx * items / (8 * kGridCtas);
        P = 256;
        while (P < 2048 && 2LL * P <= want) P *= 2;
      }
    }
  }
  if (P >= max_ctx) P = max_ctx;
  return P;
}

// Clears the decode kernel's item counter.  The decode kernel is its
// programmatic dependent on eager calls: its CTAs become resident and build
// their tables while this runs, and wait for it on the device before their
// first fetch.
__global__ void __launch_bounds__(32) decode_reset_kernel(int32_t* next) {
  asm volatile("griddepcontrol.launch_dependents;");
  if (threadIdx.x == 0) *next = 0;
}

// A launch that may begin before the previous kernel on the stream has
// completed (programmatic stream serialisation), on eager calls only; under
// stream capture, or where the attribute is refused, a plain launch.
cudaError_t launch_dependent(const void* kernel, dim3 grid, dim3 block, void** args, size_t smem,
                             cudaStream_t stream) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) == cudaSuccess && cap == cudaStreamCaptureStatusNone) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelExC(&cfg, kernel, args) == cudaSuccess) return cudaSuccess;
    (void)cudaGetLastError();
  }
  return cudaLaunchKernel(kernel, grid, block, args, smem, stream);
}

}  // namespace

unsigned fetch_status_decode() {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_status_decode, sizeof(v)) != cudaSuccess) return 0xffffffffu;
  if (v && cudaMemcpyToSymbol(g_status_decode, &zero, sizeof(zero)) != cudaSuccess) return 0xffffffffu;
  return v;
}

}  // namespace pa

using namespace pa;

static int partition_size_impl(bool fp8, int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                              int max_blocks_per_seq, int block_size, int partition_size) {
  (void)head_dim;
  if (num_seqs < 0 || max_blocks_per_seq <= 0 || !supported_block_size(block_size)) return PA_ERR_SHAPE;
  if (partition_size > 0 && partition_size % block_size) return PA_ERR_SHAPE;
  if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads) return PA_ERR_SHAPE;
  return resolve_partition(max_blocks_per_seq, block_size, partition_size, num_heads / num_kv_heads, fp8, num_seqs,
                           num_kv_heads);
}

extern "C" int pa_decode_partition_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                        int max_blocks_per_seq, int block_size, int partition_size) {
  return partition_size_impl(false, num_seqs, num_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size,
                             partition_size);
}

extern "C" int pa_decode_fp8_partition_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                            int max_blocks_per_seq, int block_size, int partition_size) {
  return partition_size_impl(true, num_seqs, num_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size,
                             partition_size);
}

extern "C" size_t pa_decode_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                           int max_blocks_per_seq, int block_size, int partition_size) {
  const int P = pa_decode_partition_size(num_seqs, num_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                         block_size, partition_size);
  if (P <= 0 || num_seqs <= 0 || num_heads <= 0) return 0;
  const long long max_ctx = (long long)max_blocks_per_seq * block_size;
  const long long max_parts = (max_ctx + P - 1) / P;
  if (max_parts <= 1) return 0;
  const long long rows = (long long)num_seqs * num_heads * max_parts;
  const long long ml = ((rows * 2 * 4) + 255) / 256 * 256;
  return (size_t)(ml + rows * head_dim * 4 + 256);     // + the work-item counter
}

// Shared by pa_decode and pa_decode_fp8: dtype is the query/output type,
// kv the pool's (dtype itself, or PA_FP8_E4M3 with per-token scales).
static int decode_impl(void* out, const void* query, const void* k_cache, const void* v_cache,
                       const float* k_scale, const float* v_scale, const int32_t* block_tables,
                       int max_blocks_per_seq, const int32_t* context_lens, int num_seqs, int num_heads,
                       int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
                       int partition_size, void* workspace, size_t workspace_bytes, pa_dtype dtype, pa_dtype kv,
                       void* stream) {
  if (dtype != PA_F32 && dtype != PA_BF16) return PA_ERR_DTYPE;
  if (kv != dtype && !(kv == PA_FP8_E4M3 && dtype == PA_BF16)) return PA_ERR_DTYPE;
  const bool fp8 = kv == PA_FP8_E4M3;
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads ||
      !supported_head_dim(head_dim) || !supported_block_size(block_size) || num_blocks <= 0 ||
      max_blocks_per_seq <= 0)
    return PA_ERR_SHAPE;
  if (partition_size > 0 && partition_size % block_size) return PA_ERR_SHAPE;
  if (num_seqs == 0) return PA_OK;
  if (!out || !query || !k_cache || !v_cache || !block_tables || !context_lens) return PA_ERR_NULL;
  if (fp8 && (!k_scale || !v_scale)) return PA_ERR_NULL;
  if (!aligned16(out) || !aligned16(query) || !aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_ALIGN;
  if (fp8 && (!aligned16(k_scale) || !aligned16(v_scale))) return PA_ERR_ALIGN;

  const int P = resolve_partition(max_blocks_per_seq, block_size, partition_size, num_heads / num_kv_heads,
                                  kv == PA_FP8_E4M3, num_seqs, num_kv_heads);
  const long long max_ctx = (long long)max_blocks_per_seq * block_size;
  const int max_parts = (int)((max_ctx + P - 1) / P);
  const size_t need = pa_decode_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim,
                                                max_blocks_per_seq, block_size, partition_size);
  if (need && (!workspace || workspace_bytes < need)) return PA_ERR_WORKSPACE;

  int dev = 0;
  if (!ck(cudaGetDevice(&dev), "cudaGetDevice")) return PA_ERR_CUDA;
  CUtensorMap mapK, mapV;
  const int G = num_heads / num_kv_heads;
  // Tensor cores over the query group when it is a real contraction (G >= 2).
  const bool use_mma = ((kv == PA_BF16 && (head_dim == 64 || head_dim == 128)) ||
                        (kv == PA_FP8_E4M3 && head_dim == 128)) &&
                       G >= 2 && (G & (G - 1)) == 0 && block_size >= 8;
  // KV heads per work item: 4 on the tensor-core path (one warp per head,
  // the four heads' tiles loaded back to back); 1 on the CUDA-core path,
  // where a warp ring per head measured faster for MHA.
  const bool mha_hg = kv == PA_BF16 && head_dim == 128 && G == 1 && PA_MHA_HEADS_PER_ITEM > 1 &&
                      num_kv_heads % PA_MHA_HEADS_PER_ITEM == 0;
// KV heads per item on the e4m3 tensor-core path (2 measured fastest).
#ifndef PA_FP8_MMA_HG
#define PA_FP8_MMA_HG 2
#endif
  const int hg_mma = fp8 ? PA_FP8_MMA_HG : 4;
  const int HG = use_mma ? (num_kv_heads % hg_mma == 0 ? hg_mma : num_kv_heads % 2 == 0 ? 2 : 1)
                 : fp8    ? fp8_heads_per_item(num_kv_heads)
                 : mha_hg ? PA_MHA_HEADS_PER_ITEM
                          : 1;
  if (!get_map(&mapK, k_cache, kv, num_blocks, block_size, num_kv_heads, head_dim, dev, use_mma, HG) ||
      !get_map(&mapV, v_cache, kv, num_blocks, block_size, num_kv_heads, head_dim, dev, use_mma, HG)) {
    note_host_error("cuTensorMapEncodeTiled failed for the K/V pool");
    return PA_ERR_CUDA;
  }

  const int GT = use_mma ? (G < 16 ? G : 16) : (G % 4 == 0) ? 4 : (G % 2 == 0) ? 2 : 1;

  DecodeParams prm;
  prm.out = out;
  prm.q = query;
  prm.block_tables = block_tables;
  prm.context_lens = context_lens;
  const long long rows = (long long)num_seqs * num_heads * max_parts;
  prm.ws_ml = need ? static_cast<float*>(workspace) : nullptr;
  prm.ws_o = need ? reinterpret_cast<float*>(static_cast<char*>(workspace) + ((rows * 8) + 255) / 256 * 256)
                  : nullptr;
  // the work-item counter: the workspace's last 256 bytes
  prm.ws_next = need ? reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + need - 256) : nullptr;
  prm.B = num_seqs;
  prm.Hq = num_heads;
  prm.Hkv = num_kv_heads;
  prm.G = G;
  prm.nsub = G / GT;
  prm.max_blocks = max_blocks_per_seq;
  prm.bs = block_size;
  prm.num_blocks = num_blocks;
  prm.part_tokens = P;
  // largest-first order (partial last partitions at the end) for long
  // partitions only: on c2 (256 tokens) it measured 3.5 % slower, the short
  // items' fixed costs meeting at the end of the launch; at 512 tokens and
  // above it gained (c2 over e4m3 +6.6 %, c4 +0.8 %)
  prm.lpt = P >= 512 ? 1 : 0;
  prm.max_parts = max_parts;
  prm.HG = HG;
  prm.n_hg = num_kv_heads / prm.HG;
  prm.WPH = kConsumerWarps / prm.HG;
  prm.n_virtual = (long long)max_parts * prm.nsub * prm.n_hg * num_seqs;
  prm.dense = num_seqs <= kDenseMaxSeqs ? 1 : 0;
  prm.qscale = scale * kLog2e;
  prm.k_scale = fp8 ? k_scale : nullptr;
  prm.v_scale = fp8 ? v_scale : nullptr;
  prm.tile_bytes = (uint32_t)(block_size * head_dim * elem_bytes(kv));
  // K/V stages per CTA: ~96 KB on the tensor-core path (one ring shared by
  // the four head warps), ~64 KB on the CUDA-core path (a ring per warp);
  // 1..4 stages per warp group.  A shared ring keeps at least 2 stages, and
  // when its stages are so large that one CTA fills the SM anyway, 3.
  const int budget = use_mma ? 98304 : PA_FFMA_STAGE_BUDGET;
  int spg = (int)(budget / (2 * prm.tile_bytes * kConsumerWarps));
  spg = spg < 1 ? 1 : (spg > PA_MAX_STAGES_PER_GROUP ? PA_MAX_STAGES_PER_GROUP : spg);
  while (!use_mma && (spg & (spg - 1))) spg &= spg - 1;   // CUDA-core path: a power of two
  // e4m3 tensor-core path: three stages per group, so that three CTAs fit on
  // an SM beside the dense tables of up to 1024 sequences (four stages of
  // 8 KB left room for two at 256 sequences)
  if (use_mma && kv == PA_FP8_E4M3 && spg > 3) spg = 3;
  if (prm.WPH == 1) {
    const size_t stage = 2 * (size_t)prm.HG * prm.tile_bytes;
    if (spg < 2) spg = 2;
    if ((size_t)spg * stage > 102400 && 3 * stage <= 200 * 1024) spg = 3;
  }
  prm.spg = spg;
  prm.spg_shift = (spg & (spg - 1)) ? -1 : (spg == 1 ? 0 : spg == 2 ? 1 : spg == 4 ? 2 : 3);
  const int S = spg * prm.WPH;

  const Launch L = fp8               ? pick_decode_fp8(head_dim, GT, prm.HG, use_mma)
                   : use_mma         ? (head_dim == 64 ? pick_mma<64>(GT, prm.HG) : pick_mma<128>(GT, prm.HG))
                   : dtype == PA_F32 ? pick1<float, float>(head_dim, GT, prm.HG)
                                     : pick1<__nv_bfloat16, __nv_bfloat16>(head_dim, GT, prm.HG);
  const size_t smem = 2 * (size_t)S * prm.HG * prm.tile_bytes + (fp8 ? 2 * (size_t)S * block_size * 4 : 0) +
                      (size_t)kConsumerWarps * GT * (head_dim + 2) * sizeof(float) +
                      2 * (size_t)S * sizeof(uint64_t) + 2 * kItemQ * sizeof(uint64_t) + 16 +
                      (kItemQ + 4) * sizeof(int) +
                      (prm.dense ? 4 * (3 * (size_t)num_seqs + 1 + kThreads / 32) : 0) + kSmemAlign;
  const int occ = occupancy_for(L.kernel, smem, dev);
  if (occ <= 0) return PA_ERR_CUDA;
  long long grid = (long long)occ * device_sm_count();
  if (grid > prm.n_virtual) grid = prm.n_virtual;

  void* args[] = {&mapK, &mapV, &prm};
  if (prm.ws_next && prm.dense) {
    // items handed out at run time from the counter in the workspace
    void* rargs[] = {&prm.ws_next};
    if (!ck(cudaLaunchKernel(reinterpret_cast<const void*>(&decode_reset_kernel), dim3(1), dim3(32), rargs, 0,
                             (cudaStream_t)stream),
            "cudaLaunchKernel(decode_reset_kernel)"))
      return PA_ERR_CUDA;
    if (!ck(launch_dependent(L.kernel, dim3((unsigned)grid), dim3(kThreads), args, smem, (cudaStream_t)stream),
            "cudaLaunchKernel(decode_kernel)"))
      return PA_ERR_CUDA;
  } else if (!ck(cudaLaunchKernel(L.kernel, dim3((unsigned)grid), dim3(kThreads), args, smem,
                                  (cudaStream_t)stream),
                 "cudaLaunchKernel(decode_kernel)")) {
    return PA_ERR_CUDA;
  }
  if (max_parts > 1) {
    const long long warps = (long long)num_seqs * num_heads;
    const unsigned blocks = (unsigned)((warps * 32 + 255) / 256);
    void* margs[] = {&prm};
    // eager calls: the merge as a programmatic dependent of the decode kernel,
    // so its CTAs are resident when the decode grid completes (c2 +0.9 %)
    if (!ck(launch_after(L.merge, dim3(blocks), dim3(256), margs, (cudaStream_t)stream),
            "cudaLaunchKernel(merge_kernel)"))
      return PA_ERR_CUDA;
  }
  return PA_OK;
}

extern "C" int pa_decode(void* out, const void* query, const void* k_cache, const void* v_cache,
                         const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                         int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                         int num_blocks, float scale, int partition_size, void* workspace,
                         size_t workspace_bytes, pa_dtype dtype, void* stream) {
  return decode_impl(out, query, k_cache, v_cache, nullptr, nullptr, block_tables, max_blocks_per_seq,
                     context_lens, num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                     partition_size, workspace, workspace_bytes, dtype, dtype, stream);
}

extern "C" int pa_decode_fp8(void* out, const void* query, const void* k_cache, const void* v_cache,
                             const float* k_scale, const float* v_scale, const int32_t* block_tables,
                             int max_blocks_per_seq, const int32_t* context_lens, int num_seqs, int num_heads,
                             int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
                             int partition_size, void* workspace, size_t workspace_bytes, pa_dtype dtype,
                             void* stream) {
  return decode_impl(out, query, k_cache, v_cache, k_scale, v_scale, block_tables, max_blocks_per_seq,
                     context_lens, num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                     partition_size, workspace, workspace_bytes, dtype, PA_FP8_E4M3, stream);
}

// ---------------------------------------------------------------------------
// Allocation-free decode.
//
// Some callers cannot allocate device memory when they call in: a plug-in
// hosted by an engine that owns every device allocation through its own pool
// (and budgets it up front), or a latency-critical path that cannot afford an
// allocation call that may synchronise the device.  pa_decode_noalloc serves
// them by using a scratch array compiled into this library as the split-K
// workspace.  Every device that loads the library holds the array until the
// process exits.  The array is shared by every call on a device: calls whose
// GPU work overlaps in time (for instance on two streams) race on it, so they
// must be ordered.  Nothing in it needs to start at zero: every value a call
// reads was written earlier by the same call.
namespace pa {
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)PA_NOALLOC_SCRATCH_BYTES;
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {};
void* g_scratch_ctx[64] = {};

// The driver's current context (cuCtxGetCurrent through the runtime's
// driver entry point); null if it cannot be read.
void* current_context() {
  using Fn = int (*)(void**);
  static Fn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return (Fn) nullptr;
    return reinterpret_cast<Fn>(p);
  }();
  void* ctx = nullptr;
  if (!fn || fn(&ctx) != 0) return nullptr;
  return ctx;
}

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address has to come
// from cudaGetSymbolAddress, with that device current.  It is looked up on
// the first call on a device and again whenever the device's context has
// changed since (a cudaDeviceReset() reloads the module at a new address).
void* scratch_address(int dev) {
  if (dev < 0 || dev >= 64) {
    note_host_error("pa_decode_noalloc: device ordinals of 64 and above are not supported");
    return nullptr;
  }
  void* ctx = current_context();
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev] || ctx != g_scratch_ctx[dev]) {
    void* ptr = nullptr;
    if (!ck(cudaGetSymbolAddress(&ptr, g_noalloc_scratch), "cudaGetSymbolAddress(no-alloc scratch)"))
      return nullptr;
    g_scratch_ptr[dev] = ptr;
    g_scratch_ctx[dev] = ctx;
  }
  return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace pa

extern "C" int pa_decode_noalloc(void* out, const void* query, const void* k_cache, const void* v_cache,
                                 const int32_t* block_tables, int max_blocks_per_seq,
                                 const int32_t* context_lens, int num_seqs, int num_heads, int num_kv_heads,
                                 int head_dim, int block_size, int num_blocks, float scale,
                                 int partition_size, pa_dtype dtype, void* stream) {
  const size_t need = pa_decode_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                                block_size, partition_size);
  if (need > pa::kNoAllocScratchBytes) {
    char msg[160];
    snprintf(msg, sizeof(msg), "pa_decode_noalloc: these sizes need %zu bytes of scratch; the built-in array "
             "holds %zu", need, pa::kNoAllocScratchBytes);
    pa::note_host_error(msg);
    return PA_ERR_WORKSPACE;
  }
  int dev = 0;
  if (!pa::ck(cudaGetDevice(&dev), "cudaGetDevice")) return PA_ERR_CUDA;
  void* scratch = pa::scratch_address(dev);
  if (!scratch) return PA_ERR_CUDA;
  return pa_decode(out, query, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                   num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, partition_size, scratch,
                   pa::kNoAllocScratchBytes, dtype, stream);
}
