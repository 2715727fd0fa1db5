// pa_decode_fp8.cu — decode kernel instances for e4m3 K/V pools with
// per-token scales ("19.2 KV Cache 系统化管理" §19.2.4: each token's K and V
// vectors quantised on their own, FP8 at one byte per element).
//
// The kernel is the one in pa_decode_kernel.cuh with KT = e4m3 codes: the
// producer adds the block's two scale rows (bs fp32 values each) to every
// stage with two bulk copies on the same mbarrier, and the consumers multiply
// each token's score by its K scale and its softmax weight by its V scale.
// Queries and output are bf16; arithmetic is fp32.  Compiled on its own so
// the instances build in parallel with the f32/bf16 ones.
#include "pa_decode_kernel.cuh"

namespace pa {
namespace {

using B16 = __nv_bfloat16;

// CUDA-core instances: 1 or 2 KV heads per item.
template <int D, int GT>
Launch pick_hg(int hg) {
  const void* merge = reinterpret_cast<const void*>(&merge_kernel<B16, D>);
  if (hg == 2) return {reinterpret_cast<const void*>(&decode_kernel<B16, fp8e4m3, D, GT, false, 2>), merge};
  return {reinterpret_cast<const void*>(&decode_kernel<B16, fp8e4m3, D, GT, false, 1>), merge};
}

template <int D>
Launch pick_gt(int gt, int hg) {
  if (gt == 4) return pick_hg<D, 4>(hg);
  if (gt == 2) return pick_hg<D, 2>(hg);
  return pick_hg<D, 1>(hg);
}

// Tensor-core instances (head_dim 128): GT query heads per KV head, HG KV heads per item.
template <int GT>
Launch pick_mma_hg(int hg) {
  const void* merge = reinterpret_cast<const void*>(&merge_kernel<B16, 128>);
  if (hg == 4) return {reinterpret_cast<const void*>(&decode_kernel<B16, fp8e4m3, 128, GT, true, 4>), merge};
  if (hg == 2) return {reinterpret_cast<const void*>(&decode_kernel<B16, fp8e4m3, 128, GT, true, 2>), merge};
  return {reinterpret_cast<const void*>(&decode_kernel<B16, fp8e4m3, 128, GT, true, 1>), merge};
}

}  // namespace

Launch pick_decode_fp8(int head_dim, int gt, int hg, bool mma) {
  if (mma) {
    if (gt == 16) return pick_mma_hg<16>(hg);
    if (gt == 8) return pick_mma_hg<8>(hg);
    if (gt == 4) return pick_mma_hg<4>(hg);
    return pick_mma_hg<2>(hg);
  }
  if (head_dim == 32) return pick_gt<32>(gt, hg);
  if (head_dim == 64) return pick_gt<64>(gt, hg);
  return pick_gt<128>(gt, hg);
}

unsigned fetch_status_decode_fp8() {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_status_decode, sizeof(v)) != cudaSuccess) return 0xffffffffu;
  if (v && cudaMemcpyToSymbol(g_status_decode, &zero, sizeof(zero)) != cudaSuccess) return 0xffffffffu;
  return v;
}

}  // namespace pa
