// pa_decode.cu — paged decode attention (GQA, split-K) and its merge kernel.
//
// What it computes ("19.2 KV Cache 系统化管理" §19.2.3 and Fig 19-5; "LLM 推理
// 引擎的内存管理与调度…" §三): for each sequence b and query head h, attention of
// q[b,h] over the sequence's K/V, which sit in fixed-size physical blocks named
// by the block table; only the valid slots of the last block count; the
// softmax is accumulated block by block with a running maximum, a running sum
// of exponentials and a rescaled output, normalised at the end.
//
// How (GB300):
//  * Work item = (sequence, KV head, query-head subgroup, partition of P
//    tokens).  A persistent grid (resident CTAs x SMs) strides over the item
//    space; the sequence index is innermost so CTAs running side by side read
//    the same blocks when sequences share a prompt.
//  * Each CTA = 1 producer warp + kConsumerWarps consumer warps.  The producer
//    reads the item's block-table entries with one coalesced warp load, then
//    issues, per block, two TMA tensor loads (box {D, 1 head, bs, 1 block} of
//    the [NB, bs, Hkv, D] pool) for K and V into a ring of shared-memory
//    stages, completing on an mbarrier with transaction bytes.  A block id
//    outside the pool is flagged and replaced by block 0, so no copy leaves
//    the pool.
//  * Consumer warps take the item's blocks round-robin, and each warp owns its
//    own ring of SPW stages which it consumes strictly in order (a ring shared
//    by several round-robin consumers lets a warp wait on a stage two phases
//    ahead, where a parity wait matches the stale phase).  Inside a warp, LPT
//    lanes share one token (each lane owns two 16-byte chunks of head_dim), so
//    one warp covers TPW tokens per pass with conflict-free 16-byte shared
//    loads.  Each lane group keeps its own online-softmax state (m, l, o) for
//    its tokens; group, warp and partition states are merged by log-sum-exp at
//    the end, which is exact up to rounding (the update is associative).
//  * Scores are computed in the base-2 domain (q pre-multiplied by
//    scale*log2 e), with exp2f.  The K/V rows are read once from HBM and used
//    for all GT query heads of the subgroup (GQA) straight from registers.
//  * A sequence whose context fits one partition is normalised and written
//    directly; longer ones write (m, l, unnormalised o) per partition to the
//    workspace, and merge_kernel combines them.
//  * Waits are bounded (2 s).  A wait that runs out sets PA_DEV_TIMEOUT and an
//    abort flag; every role then skips the remaining work while still passing
//    the CTA's barriers, and the producer waits (bounded) for the TMA loads it
//    issued before the CTA exits.
#include "pa_common.cuh"

#include <mutex>
#include <map>
#include <tuple>
#include <stdio.h>

namespace pa {
namespace {

__device__ unsigned g_status_decode;

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kSmemAlign = 1024;

struct DecodeParams {
  void* out;
  const void* q;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float* ws_ml;       // [B*Hq*max_parts][2]   (m in log2 units, l)
  float* ws_o;        // [B*Hq*max_parts][D]   unnormalised output
  int B, Hq, Hkv, G, nsub;
  int max_blocks, bs, num_blocks;
  int part_tokens, max_parts;
  long long n_virtual;
  float qscale;       // scale * log2(e)
  int HG;             // KV heads per work item (one consumer warp each when HG = 4)
  int n_hg;           // Hkv / HG
  int WPH;            // warp groups: kConsumerWarps / HG (warps sharing one head)
  int spg;            // shared-memory stages per warp group
  uint32_t tile_bytes;  // one head's K (or V) tile of one block: bs * D * elem
};

struct Item {
  int b, kvh0, sg, part, t1, jb, je;
  bool split;
};

// m16n8k16 bf16 tensor-core product with fp32 accumulation (per warp).
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr) : "memory");
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr) : "memory");
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ bool decode_item(const DecodeParams& p, long long v, Item& it) {
  it.b = (int)(v % p.B);
  long long r = v / p.B;
  it.kvh0 = (int)(r % p.n_hg) * p.HG;
  r /= p.n_hg;
  it.sg = (int)(r % p.nsub);
  it.part = (int)(r / p.nsub);
  int L = __ldg(&p.context_lens[it.b]);
  const int Lmax = p.max_blocks * p.bs;
  if (L < 0 || L > Lmax) L = L < 0 ? 0 : Lmax;   // flagged by the consumer
  const int nparts = L > 0 ? (L + p.part_tokens - 1) / p.part_tokens : 1;
  if (it.part >= nparts) return false;
  const int t0 = it.part * p.part_tokens;
  it.t1 = min(L, t0 + p.part_tokens);
  it.jb = t0 / p.bs;
  it.je = (it.t1 + p.bs - 1) / p.bs;
  if (it.je < it.jb) it.je = it.jb;
  it.split = nparts > 1;
  return true;
}

template <typename T, int D, int GT, bool MMA, int HG>
__global__ void __launch_bounds__(kThreads)
decode_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
              const DecodeParams p) {
  using E = Elem<T>;
  constexpr int CHUNKS = D * E::kBytes / 16;   // 16-byte chunks per token row
  constexpr int LPT = CHUNKS / 2;              // lanes per token
  constexpr int TPW = 32 / LPT;                // tokens per warp pass
  constexpr int EPC = E::kPerChunk;            // elements per chunk
  constexpr int DPL = 2 * EPC;                 // head dims per lane
  constexpr int NS = TPW >= 16 ? 1 : 16 / TPW; // tokens per lane group per softmax step
  constexpr int ROW = D * E::kBytes;
  constexpr int NCW = kConsumerWarps;
  static_assert(LPT >= 1 && LPT <= 32 && (32 % LPT) == 0, "lane split");

  constexpr int WPH = kConsumerWarps / HG;               // warp groups (warps sharing a head)
  static_assert(HG == 1 || HG == 2 || HG == 4, "KV heads per item");
  const int S = p.spg * WPH;                             // stages in total
  const uint32_t stage_bytes = (uint32_t)HG * p.tile_bytes;  // K (or V) of one block, HG heads
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // TMA destinations must be 128-byte aligned: align the base explicitly
  // (the host reserves kSmemAlign bytes of slack).
  unsigned char* smem = smem_raw + ((kSmemAlign - (smem_u32(smem_raw) & (kSmemAlign - 1))) & (kSmemAlign - 1));
  unsigned char* tilesK = smem;
  unsigned char* tilesV = smem + (size_t)S * stage_bytes;
  float* mbuf = reinterpret_cast<float*>(tilesV + (size_t)S * stage_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(mbuf + NCW * GT * (D + 2));
  uint64_t* empty = full + S;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + S);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], HG);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // An item covers HG KV heads.  Consumer warp w works on head w % HG of
  // the item, in warp group w / HG; block i of the item goes to group
  // i % WPH (WPH = NCW / HG), and every warp of that group reads its own head
  // from the same stage.  Each group owns SPW stages which all its warps
  // consume strictly in order, so every stage has one producer and one set of
  // consumers that walk its phases in order and a parity wait can never match
  // a stale phase.  u = the group's running block count (same arithmetic in
  // every role); stage = g*SPW + u % SPW.  The HG heads of a block are loaded
  // back to back, so the DRAM sees neighbouring rows of the pool together.
  const int SPW = p.spg;

  if (warp == NCW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&mapK);
      prefetch_tensormap(&mapV);
    }
    const uint64_t pol = policy_evict_first();
    // base[g] = warp group g's running block count, issued[g] = loads issued
    // into its stages (WPH is a compile-time constant, so the group
    // arithmetic below is shifts and selects).
    uint32_t base[NCW], issued[NCW];
#pragma unroll
    for (int w = 0; w < NCW; ++w) base[w] = issued[w] = 0;
    for (long long v = blockIdx.x; v < p.n_virtual; v += gridDim.x) {
      Item item;
      if (!decode_item(p, v, item)) continue;
      const int32_t* row = p.block_tables + (size_t)item.b * p.max_blocks;
      const int nblk = item.je - item.jb;
      for (int j0 = 0; j0 < nblk; j0 += 32) {
        const int n = min(32, nblk - j0);
        int blk = 0;
        if (lane < n) {
          blk = __ldg(&row[item.jb + j0 + lane]);
          if ((unsigned)blk >= (unsigned)p.num_blocks) {
            atomicOr(&g_status_decode, PA_DEV_BAD_BLOCK);
            blk = 0;    // keep every copy inside the pool
          }
        }
        for (int i = 0; i < n; ++i) {
          const int bi = __shfl_sync(0xffffffffu, blk, i);
          const int w = (j0 + i) % WPH;
          uint32_t u = 0;
#pragma unroll
          for (int k = 0; k < WPH; ++k)
            if (k == w) u = base[k] + (uint32_t)((j0 + i) / WPH);
          const int st = w * SPW + (int)(u % SPW);
          const uint32_t ph = (u / SPW) & 1u;
          constexpr int HALVES = MMA ? D / 64 : 1;
          constexpr int NOPS = MMA ? 2 * HG * HALVES : 2;   // TMA loads per block
          int go = 0;
          if (lane == 0 && !*abort_flag) {
            if (!mbar_wait(&empty[st], ph ^ 1u)) {
              atomicOr(&g_status_decode, PA_DEV_TIMEOUT);
              *abort_flag = 1;
            } else {
              mbar_arrive_expect_tx(&full[st], 2u * stage_bytes);
              go = 1;
              if constexpr (NOPS == 2) {
                // one box {D, HG heads, bs, 1} each for K and V: smem [bs][HG][D]
                tma_load_4d(tilesK + (size_t)st * stage_bytes, &mapK, &full[st], 0, item.kvh0, 0, bi, pol);
                tma_load_4d(tilesV + (size_t)st * stage_bytes, &mapV, &full[st], 0, item.kvh0, 0, bi, pol);
              }
            }
          }
          if constexpr (NOPS > 2) {
            // tensor-core path: many 128-byte-swizzled 64-column halves per
            // block, issued by one warp instruction: lane l takes K (l even)
            // or V (l odd) of head l/2/HALVES, half l/2%HALVES
            if (__shfl_sync(0xffffffffu, go, 0) && lane < NOPS) {
              const int rest = lane >> 1;
              const int hl = rest / HALVES, hh = rest % HALVES;
              const size_t off = (size_t)st * stage_bytes + (size_t)hl * p.tile_bytes + (size_t)hh * p.bs * 128;
              unsigned char* dst = ((lane & 1) ? tilesV : tilesK) + off;
              tma_load_4d(dst, (lane & 1) ? &mapV : &mapK, &full[st], hh * 64, item.kvh0 + hl, 0, bi, pol);
            }
          }
          if (lane == 0 && go) {
#pragma unroll
            for (int k = 0; k < WPH; ++k)
              if (k == w) issued[k] = u + 1;
          }
        }
      }
#pragma unroll
      for (int w = 0; w < WPH; ++w) base[w] += nblk > w ? (uint32_t)((nblk - w + WPH - 1) / WPH) : 0u;
    }
    // Never leave the CTA with TMA writes into its shared memory in flight:
    // wait (bounded) for the last SPW loads issued into each group's stages.
    if (lane == 0) {
#pragma unroll
      for (int w = 0; w < WPH; ++w) {
        const uint32_t first = issued[w] > (uint32_t)SPW ? issued[w] - SPW : 0u;
        for (uint32_t u = first; u < issued[w]; ++u)
          mbar_wait(&full[w * SPW + (int)(u % SPW)], (u / SPW) & 1u);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int grp = lane / LPT;     // token slot within a warp pass
  const int li = lane % LPT;      // chunk owner within the token row
  const int c0 = li, c1 = li + LPT;
  const int ctid = threadIdx.x;   // 0 .. NCW*32-1
  uint32_t wcount = 0;            // blocks this warp's group has consumed so far
  const int hl = warp % HG;       // the item's KV head this warp works on
  const int gw = warp / HG;       // this warp's group

  for (long long v = blockIdx.x; v < p.n_virtual; v += gridDim.x) {
    Item item;
    if (!decode_item(p, v, item)) continue;
    if (ctid == 0 && item.kvh0 == 0 && item.sg == 0 && item.part == 0) {
      const int L = __ldg(&p.context_lens[item.b]);
      if (L < 0 || L > p.max_blocks * p.bs) atomicOr(&g_status_decode, PA_DEV_BAD_LEN);
    }
    const int h0 = (item.kvh0 + hl) * p.G + item.sg * GT;

    if constexpr (MMA) {
      // Query heads h0..h0+GT-1 are the M rows of m16n8k16 (rows >= GT are
      // zero); K rows are the N columns of S = Q K^T, and P (bf16) times V
      // accumulates O[16 x D] in registers.  Lane (g = lane/4, tq = lane%4)
      // holds rows g and g+8.  K/V tiles sit in shared memory as 128-byte-
      // swizzled 64-column halves, so ldmatrix reads are conflict-free.
      constexpr int KS = D / 16;
      constexpr int NT = D / 8;
      const int g = lane >> 2, tq = lane & 3;
      const bool r0v = g < GT, r1v = g + 8 < GT;
      const uint32_t* q0p = reinterpret_cast<const uint32_t*>(
          static_cast<const unsigned char*>(p.q) + ((size_t)item.b * p.Hq + h0 + (r0v ? g : 0)) * ROW);
      const uint32_t* q1p = reinterpret_cast<const uint32_t*>(
          static_cast<const unsigned char*>(p.q) + ((size_t)item.b * p.Hq + h0 + (r1v ? g + 8 : 0)) * ROW);
      uint32_t qa[KS][4];
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        qa[kk][0] = r0v ? __ldg(q0p + kk * 8 + tq) : 0u;
        qa[kk][1] = r1v ? __ldg(q1p + kk * 8 + tq) : 0u;
        qa[kk][2] = r0v ? __ldg(q0p + kk * 8 + 4 + tq) : 0u;
        qa[kk][3] = r1v ? __ldg(q1p + kk * 8 + 4 + tq) : 0u;
      }
      float O[NT][4];
#pragma unroll
      for (int n = 0; n < NT; ++n) O[n][0] = O[n][1] = O[n][2] = O[n][3] = 0.f;
      float mr[2] = {-INFINITY, -INFINITY}, lr[2] = {0.f, 0.f};
      const uint32_t half_bytes = (uint32_t)p.bs * 128u;

      const int nblk = item.je - item.jb;
      for (int i = gw; i < nblk; i += WPH, ++wcount) {
        const int st = gw * SPW + (int)(wcount % SPW);
        const uint32_t ph = (wcount / SPW) & 1u;
        bool live = __shfl_sync(0xffffffffu, *abort_flag, 0) == 0;
        if (live) {
          const bool late = !mbar_wait(&full[st], ph);
          if (__any_sync(0xffffffffu, late)) {
            live = false;
            if (lane == 0) {
              atomicOr(&g_status_decode, PA_DEV_TIMEOUT);
              *abort_flag = 1;
            }
          }
        }
        if (live) {
          const int valid = min(p.bs, item.t1 - (item.jb + i) * p.bs);
          unsigned char* vt_ptr = tilesV + (size_t)st * stage_bytes + (size_t)hl * p.tile_bytes;
          const uint32_t kt = smem_u32(tilesK + (size_t)st * stage_bytes + (size_t)hl * p.tile_bytes);
          const uint32_t vt = smem_u32(vt_ptr);
          if (valid < p.bs) {
            // slots past the context may hold anything; P is 0 there, but
            // 0 * NaN is NaN inside the product, so clear those V rows
            for (int idx = lane; idx < (p.bs - valid) * (D / 8); idx += 32) {
              const int t = valid + idx / (D / 8), c = idx % (D / 8);
              *reinterpret_cast<uint4*>(vt_ptr + (c >> 3) * half_bytes + t * 128 + (c & 7) * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
          for (int tb = 0; tb < valid; tb += 16) {
            float S[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            {
              const int tt = min(tb + (lane & 7) + ((lane >> 4) << 3), p.bs - 1);
#pragma unroll
              for (int kk = 0; kk < KS; ++kk) {
                const int c = 2 * kk + ((lane >> 3) & 1);
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kt + (c >> 3) * half_bytes + tt * 128 + (((c & 7) ^ (tt & 7)) << 4), b0, b1, b2, b3);
                mma_bf16_16816(S[0], qa[kk], b0, b1);
                mma_bf16_16816(S[1], qa[kk], b2, b3);
              }
            }
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int t = tb + n * 8 + 2 * tq + (e & 1);
                S[n][e] = t < valid ? S[n][e] * p.qscale : -INFINITY;
                mx[e >> 1] = fmaxf(mx[e >> 1], S[n][e]);
              }
            float alpha[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
              mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
              mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
              const float mn = fmaxf(mr[r], mx[r]);
              alpha[r] = mn == -INFINITY ? 1.f : exp2f(mr[r] - mn);
              mr[r] = mn;
              lr[r] *= alpha[r];
            }
            if (alpha[0] != 1.f || alpha[1] != 1.f) {
#pragma unroll
              for (int n = 0; n < NT; ++n) {
                O[n][0] *= alpha[0];
                O[n][1] *= alpha[0];
                O[n][2] *= alpha[1];
                O[n][3] *= alpha[1];
              }
            }
            float pv[2][4];
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float m_ = mr[e >> 1];
                pv[n][e] = (S[n][e] == -INFINITY) ? 0.f : exp2f(S[n][e] - m_);
                lr[e >> 1] += pv[n][e];
              }
            const uint32_t pa[4] = {pack_bf16(pv[0][0], pv[0][1]), pack_bf16(pv[0][2], pv[0][3]),
                                    pack_bf16(pv[1][0], pv[1][1]), pack_bf16(pv[1][2], pv[1][3])};
            {
              const int tt = min(tb + (lane & 7) + (((lane >> 3) & 1) << 3), p.bs - 1);
#pragma unroll
              for (int j = 0; j < D / 16; ++j) {
                const int c = 2 * j + (lane >> 4);
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vt + (c >> 3) * half_bytes + tt * 128 + (((c & 7) ^ (tt & 7)) << 4), b0, b1, b2, b3);
                mma_bf16_16816(O[2 * j], pa, b0, b1);
                mma_bf16_16816(O[2 * j + 1], pa, b2, b3);
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
      }
      // the row sums are split over the 4 lanes of a row group
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        lr[r] += __shfl_xor_sync(0xffffffffu, lr[r], 1);
        lr[r] += __shfl_xor_sync(0xffffffffu, lr[r], 2);
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int h = g + 8 * r;
        if (h < GT) {
          float* dst = mbuf + (warp * GT + h) * (D + 2);
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            dst[n * 8 + 2 * tq] = O[n][2 * r];
            dst[n * 8 + 2 * tq + 1] = O[n][2 * r + 1];
          }
          if (tq == 0) {
            dst[D] = mr[r];
            dst[D + 1] = lr[r];
          }
        }
      }
    } else {
      float q[GT][DPL];
  #pragma unroll
      for (int h = 0; h < GT; ++h) {
        const unsigned char* qrow =
            static_cast<const unsigned char*>(p.q) + ((size_t)item.b * p.Hq + h0 + h) * ROW;
        float f[EPC];
        E::unpack(__ldg(reinterpret_cast<const uint4*>(qrow + c0 * 16)), f);
  #pragma unroll
        for (int e = 0; e < EPC; ++e) q[h][e] = f[e] * p.qscale;
        E::unpack(__ldg(reinterpret_cast<const uint4*>(qrow + c1 * 16)), f);
  #pragma unroll
        for (int e = 0; e < EPC; ++e) q[h][EPC + e] = f[e] * p.qscale;
      }
      float m[GT], l[GT], o[GT][DPL];
  #pragma unroll
      for (int h = 0; h < GT; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
  #pragma unroll
        for (int d = 0; d < DPL; ++d) o[h][d] = 0.f;
      }

      const int nblk = item.je - item.jb;
      for (int i = gw; i < nblk; i += WPH, ++wcount) {
        const int st = gw * SPW + (int)(wcount % SPW);
        const uint32_t ph = (wcount / SPW) & 1u;
        bool live = __shfl_sync(0xffffffffu, *abort_flag, 0) == 0;
        if (live) {
          const bool late = !mbar_wait(&full[st], ph);
          if (__any_sync(0xffffffffu, late)) {
            live = false;
            if (lane == 0) {
              atomicOr(&g_status_decode, PA_DEV_TIMEOUT);
              *abort_flag = 1;
            }
          }
        }
        if (live) {
          const int valid = min(p.bs, item.t1 - (item.jb + i) * p.bs);
          // stage layout [bs][HG][D]: token t of head hl at (t*HG + hl) * ROW
          const unsigned char* kt = tilesK + (size_t)st * stage_bytes + (size_t)hl * ROW;
          const unsigned char* vt = tilesV + (size_t)st * stage_bytes + (size_t)hl * ROW;
          for (int tb = 0; tb < valid; tb += TPW * NS) {
            float s[NS][GT];
  #pragma unroll
            for (int k = 0; k < NS; ++k) {
              const int t = tb + k * TPW + grp;
              const bool ok = t < valid;
              float part[GT];
  #pragma unroll
              for (int h = 0; h < GT; ++h) part[h] = 0.f;
              if (ok) {
                float kf[DPL];
                E::unpack(*reinterpret_cast<const uint4*>(kt + t * (HG * ROW) + c0 * 16), kf);
                E::unpack(*reinterpret_cast<const uint4*>(kt + t * (HG * ROW) + c1 * 16), kf + EPC);
  #pragma unroll
                for (int h = 0; h < GT; ++h)
  #pragma unroll
                  for (int d = 0; d < DPL; ++d) part[h] = fmaf(q[h][d], kf[d], part[h]);
              }
  #pragma unroll
              for (int h = 0; h < GT; ++h) {
  #pragma unroll
                for (int off = LPT / 2; off > 0; off >>= 1)
                  part[h] += __shfl_xor_sync(0xffffffffu, part[h], off);
                s[k][h] = ok ? part[h] : -INFINITY;
              }
            }
  #pragma unroll
            for (int h = 0; h < GT; ++h) {
              float mx = m[h];
  #pragma unroll
              for (int k = 0; k < NS; ++k) mx = fmaxf(mx, s[k][h]);
              const float alpha = mx == -INFINITY ? 1.f : exp2f(m[h] - mx);
              m[h] = mx;
              l[h] *= alpha;
  #pragma unroll
              for (int d = 0; d < DPL; ++d) o[h][d] *= alpha;
            }
  #pragma unroll
            for (int k = 0; k < NS; ++k) {
              const int t = tb + k * TPW + grp;
              if (t < valid) {
                float vf[DPL];
                E::unpack(*reinterpret_cast<const uint4*>(vt + t * (HG * ROW) + c0 * 16), vf);
                E::unpack(*reinterpret_cast<const uint4*>(vt + t * (HG * ROW) + c1 * 16), vf + EPC);
  #pragma unroll
                for (int h = 0; h < GT; ++h) {
                  const float pk = exp2f(s[k][h] - m[h]);
                  l[h] += pk;
  #pragma unroll
                  for (int d = 0; d < DPL; ++d) o[h][d] = fmaf(pk, vf[d], o[h][d]);
                }
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
      }

      // merge the lane groups of this warp (lanes with equal li own equal dims)
  #pragma unroll
      for (int off = LPT; off < 32; off <<= 1) {
  #pragma unroll
        for (int h = 0; h < GT; ++h) {
          const float m2 = __shfl_xor_sync(0xffffffffu, m[h], off);
          const float l2 = __shfl_xor_sync(0xffffffffu, l[h], off);
          const float M = fmaxf(m[h], m2);
          const float a = m[h] == -INFINITY ? 0.f : exp2f(m[h] - M);
          const float b = m2 == -INFINITY ? 0.f : exp2f(m2 - M);
          l[h] = a * l[h] + b * l2;
  #pragma unroll
          for (int d = 0; d < DPL; ++d) {
            const float o2 = __shfl_xor_sync(0xffffffffu, o[h][d], off);
            o[h][d] = a * o[h][d] + b * o2;
          }
          m[h] = M;
        }
      }
      if (grp == 0) {
  #pragma unroll
        for (int h = 0; h < GT; ++h) {
          float* dst = mbuf + (warp * GT + h) * (D + 2);
  #pragma unroll
          for (int e = 0; e < EPC; ++e) {
            dst[c0 * EPC + e] = o[h][e];
            dst[c1 * EPC + e] = o[h][EPC + e];
          }
          if (li == 0) {
            dst[D] = m[h];
            dst[D + 1] = l[h];
          }
        }
      }
    }
    named_sync(1, NCW * 32);

    // merge the warp groups (warps gw*HG + hl share head hl) and write
    for (int idx = ctid; idx < HG * GT * D; idx += NCW * 32) {
      const int hh = idx / (GT * D), h = (idx / D) % GT, d = idx % D;
      float M = -INFINITY;
#pragma unroll
      for (int g = 0; g < WPH; ++g) M = fmaxf(M, mbuf[((g * HG + hh) * GT + h) * (D + 2) + D]);
      float num = 0.f, den = 0.f;
      if (M != -INFINITY) {
#pragma unroll
        for (int g = 0; g < WPH; ++g) {
          const float* src = mbuf + ((g * HG + hh) * GT + h) * (D + 2);
          const float a = src[D] == -INFINITY ? 0.f : exp2f(src[D] - M);
          num = fmaf(a, src[d], num);
          den = fmaf(a, src[D + 1], den);
        }
      }
      const size_t bh = (size_t)item.b * p.Hq + (size_t)(item.kvh0 + hh) * p.G + item.sg * GT + h;
      if (!item.split) {
        E::store1(static_cast<T*>(p.out) + bh * D + d, den > 0.f ? num / den : 0.f);
      } else {
        const size_t slot = bh * p.max_parts + item.part;
        p.ws_o[slot * D + d] = num;
        if (d == 0) {
          p.ws_ml[slot * 2] = M;
          p.ws_ml[slot * 2 + 1] = den;
        }
      }
    }
    named_sync(1, NCW * 32);
  }
}

// One warp per (sequence, query head) with more than one partition.
template <typename T, int D>
__global__ void __launch_bounds__(256)
merge_kernel(const DecodeParams p) {
  using E = Elem<T>;
  constexpr int PER = D / 32;
  const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= (long long)p.B * p.Hq) return;
  const int b = (int)(gw / p.Hq);
  int L = __ldg(&p.context_lens[b]);
  const int Lmax = p.max_blocks * p.bs;
  if (L < 0 || L > Lmax) L = L < 0 ? 0 : Lmax;
  const int nparts = L > 0 ? (L + p.part_tokens - 1) / p.part_tokens : 1;
  if (nparts <= 1) return;
  const size_t base = (size_t)gw * p.max_parts;
  float M = -INFINITY;
  for (int i = lane; i < nparts; i += 32) M = fmaxf(M, p.ws_ml[(base + i) * 2]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float den = 0.f;
  for (int i = lane; i < nparts; i += 32) {
    const float mi = p.ws_ml[(base + i) * 2];
    if (mi != -INFINITY) den += exp2f(mi - M) * p.ws_ml[(base + i) * 2 + 1];
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
  float acc[PER];
#pragma unroll
  for (int k = 0; k < PER; ++k) acc[k] = 0.f;
  for (int i = 0; i < nparts; ++i) {
    const float mi = p.ws_ml[(base + i) * 2];
    const float w = mi == -INFINITY ? 0.f : exp2f(mi - M);
    const float* oi = p.ws_o + (base + i) * D;
#pragma unroll
    for (int k = 0; k < PER; ++k) acc[k] = fmaf(w, oi[lane + 32 * k], acc[k]);
  }
  T* out = static_cast<T*>(p.out) + (size_t)gw * D;
#pragma unroll
  for (int k = 0; k < PER; ++k) E::store1(out + lane + 32 * k, den > 0.f ? acc[k] / den : 0.f);
}

// ------------------------------------------------------------------ host side

struct Launch {
  const void* kernel;
  const void* merge;
};

template <typename T, int D, int GT>
Launch pick3(int hg) {
  const void* merge = reinterpret_cast<const void*>(&merge_kernel<T, D>);
  if (hg == 4) return {reinterpret_cast<const void*>(&decode_kernel<T, D, GT, false, 4>), merge};
  return {reinterpret_cast<const void*>(&decode_kernel<T, D, GT, false, 1>), merge};
}

// Tensor-core GQA variant: bf16, head_dim 64 or 128, GT query heads per KV head.
template <int D, int GT>
Launch pick_mma_hg(int hg) {
  const void* merge = reinterpret_cast<const void*>(&merge_kernel<__nv_bfloat16, D>);
  if (hg == 4) return {reinterpret_cast<const void*>(&decode_kernel<__nv_bfloat16, D, GT, true, 4>), merge};
  if (hg == 2) return {reinterpret_cast<const void*>(&decode_kernel<__nv_bfloat16, D, GT, true, 2>), merge};
  return {reinterpret_cast<const void*>(&decode_kernel<__nv_bfloat16, D, GT, true, 1>), merge};
}

template <int D>
Launch pick_mma(int gt, int hg) {
  if (gt == 16) return pick_mma_hg<D, 16>(hg);
  if (gt == 8) return pick_mma_hg<D, 8>(hg);
  if (gt == 4) return pick_mma_hg<D, 4>(hg);
  return pick_mma_hg<D, 2>(hg);
}

template <typename T, int D>
Launch pick2(int gt, int hg) {
  if (gt == 4) return pick3<T, D, 4>(hg);
  if (gt == 2) return pick3<T, D, 2>(hg);
  return pick3<T, D, 1>(hg);
}

template <typename T>
Launch pick1(int d, int gt, int hg) {
  if (d == 32) return pick2<T, 32>(gt, hg);
  if (d == 64) return pick2<T, 64>(gt, hg);
  return pick2<T, 128>(gt, hg);
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
    const uint32_t box[4] = {64, 1, (uint32_t)bs, 1};
    ok = encode_map(out, base, dt == PA_F32, 4, dims, str, box, true);
  } else {
    const uint64_t e = (uint64_t)elem_bytes(dt);
    const uint64_t dims[4] = {(uint64_t)d, (uint64_t)h, (uint64_t)bs, (uint64_t)nb};
    const uint64_t str[3] = {d * e, (uint64_t)h * d * e, (uint64_t)bs * h * d * e};
    const uint32_t box[4] = {(uint32_t)d, (uint32_t)boxh, (uint32_t)bs, 1};
    ok = encode_map(out, base, dt == PA_F32, 4, dims, str, box, false);
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

// Automatic split: 512-token partitions for MHA (G = 1), 2048 for GQA, whose
// items already cover several query heads per K/V read.
int resolve_partition(int max_blocks, int bs, int partition_size, int G) {
  const int max_ctx = max_blocks * bs;
  if (partition_size < 0) return max_ctx;
  int P = partition_size > 0 ? partition_size : (G >= 2 ? 2048 : 512);
  if (P >= max_ctx) P = max_ctx;
  return P;
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

extern "C" int pa_decode_partition_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                        int max_blocks_per_seq, int block_size, int partition_size) {
  (void)num_seqs; (void)head_dim;
  if (max_blocks_per_seq <= 0 || !supported_block_size(block_size)) return PA_ERR_SHAPE;
  if (partition_size > 0 && partition_size % block_size) return PA_ERR_SHAPE;
  if (num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads) return PA_ERR_SHAPE;
  return resolve_partition(max_blocks_per_seq, block_size, partition_size, num_heads / num_kv_heads);
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
  return (size_t)(ml + rows * head_dim * 4);
}

extern "C" int pa_decode(void* out, const void* query, const void* k_cache, const void* v_cache,
                         const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                         int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size,
                         int num_blocks, float scale, int partition_size, void* workspace,
                         size_t workspace_bytes, pa_dtype dtype, void* stream) {
  if (dtype != PA_F32 && dtype != PA_BF16) return PA_ERR_DTYPE;
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads ||
      !supported_head_dim(head_dim) || !supported_block_size(block_size) || num_blocks <= 0 ||
      max_blocks_per_seq <= 0)
    return PA_ERR_SHAPE;
  if (partition_size > 0 && partition_size % block_size) return PA_ERR_SHAPE;
  if (num_seqs == 0) return PA_OK;
  if (!out || !query || !k_cache || !v_cache || !block_tables || !context_lens) return PA_ERR_NULL;
  if (!aligned16(out) || !aligned16(query) || !aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_ALIGN;

  const int P = resolve_partition(max_blocks_per_seq, block_size, partition_size, num_heads / num_kv_heads);
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
  const bool use_mma = dtype == PA_BF16 && (head_dim == 64 || head_dim == 128) && G >= 2 && (G & (G - 1)) == 0 &&
                       block_size >= 8;
  // KV heads per work item: 4 on the tensor-core path (one warp per head,
  // the four heads' tiles loaded back to back); 1 on the CUDA-core path,
  // where a warp ring per head measured faster for MHA.
  const int HG = use_mma ? (num_kv_heads % 4 == 0 ? 4 : num_kv_heads % 2 == 0 ? 2 : 1) : 1;
  if (!get_map(&mapK, k_cache, dtype, num_blocks, block_size, num_kv_heads, head_dim, dev, use_mma, HG) ||
      !get_map(&mapV, v_cache, dtype, num_blocks, block_size, num_kv_heads, head_dim, dev, use_mma, HG)) {
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
  prm.B = num_seqs;
  prm.Hq = num_heads;
  prm.Hkv = num_kv_heads;
  prm.G = G;
  prm.nsub = G / GT;
  prm.max_blocks = max_blocks_per_seq;
  prm.bs = block_size;
  prm.num_blocks = num_blocks;
  prm.part_tokens = P;
  prm.max_parts = max_parts;
  prm.HG = HG;
  prm.n_hg = num_kv_heads / prm.HG;
  prm.WPH = kConsumerWarps / prm.HG;
  prm.n_virtual = (long long)max_parts * prm.nsub * prm.n_hg * num_seqs;
  prm.qscale = scale * kLog2e;
  prm.tile_bytes = (uint32_t)(block_size * head_dim * elem_bytes(dtype));
  // K/V stages per CTA: ~96 KB on the tensor-core path (one ring shared by
  // the four head warps), ~64 KB on the CUDA-core path (a ring per warp);
  // 1..4 stages per warp group.  A shared ring keeps at least 2 stages, and
  // when its stages are so large that one CTA fills the SM anyway, 3.
  const int budget = use_mma ? 98304 : 65536;
  int spg = (int)(budget / (2 * prm.tile_bytes * kConsumerWarps));
  spg = spg < 1 ? 1 : (spg > 4 ? 4 : spg);
  if (prm.WPH == 1) {
    const size_t stage = 2 * (size_t)prm.HG * prm.tile_bytes;
    if (spg < 2) spg = 2;
    if ((size_t)spg * stage > 102400 && 3 * stage <= 200 * 1024) spg = 3;
  }
  prm.spg = spg;
  const int S = spg * prm.WPH;

  const Launch L = use_mma ? (head_dim == 64 ? pick_mma<64>(GT, prm.HG) : pick_mma<128>(GT, prm.HG))
                   : dtype == PA_F32 ? pick1<float>(head_dim, GT, prm.HG)
                                     : pick1<__nv_bfloat16>(head_dim, GT, prm.HG);
  const size_t smem = 2 * (size_t)S * prm.HG * prm.tile_bytes +
                      (size_t)kConsumerWarps * GT * (head_dim + 2) * sizeof(float) +
                      2 * (size_t)S * sizeof(uint64_t) + 16 + kSmemAlign;
  const int occ = occupancy_for(L.kernel, smem, dev);
  if (occ <= 0) return PA_ERR_CUDA;
  long long grid = (long long)occ * device_sm_count();
  if (grid > prm.n_virtual) grid = prm.n_virtual;

  void* args[] = {&mapK, &mapV, &prm};
  if (!ck(cudaLaunchKernel(L.kernel, dim3((unsigned)grid), dim3(kThreads), args, smem, (cudaStream_t)stream),
          "cudaLaunchKernel(decode_kernel)"))
    return PA_ERR_CUDA;
  if (max_parts > 1) {
    const long long warps = (long long)num_seqs * num_heads;
    const unsigned blocks = (unsigned)((warps * 32 + 255) / 256);
    void* margs[] = {&prm};
    if (!ck(cudaLaunchKernel(L.merge, dim3(blocks), dim3(256), margs, 0, (cudaStream_t)stream),
            "cudaLaunchKernel(merge_kernel)"))
      return PA_ERR_CUDA;
  }
  return PA_OK;
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

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address has to come
// from cudaGetSymbolAddress, once per device, with that device current.
void* scratch_address(int dev) {
  if (dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    if (!ck(cudaGetSymbolAddress(&ptr, g_noalloc_scratch), "cudaGetSymbolAddress(no-alloc scratch)"))
      return nullptr;
    g_scratch_ptr[dev] = ptr;
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
