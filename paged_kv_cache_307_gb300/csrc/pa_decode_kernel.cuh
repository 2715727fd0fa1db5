// pa_decode_kernel.cuh — the paged decode attention kernel and its merge kernel,
// shared by the translation units that instantiate them (pa_decode.cu: f32 and
// bf16 pools; pa_decode_fp8.cu: e4m3 pools).  Each including unit gets its own
// copy of the kernels and its own sticky status word (internal linkage).
//
// What it computes ("19.2 KV Cache 系统化管理" §19.2.3 and Fig 19-5; "LLM 推理
// 引擎的内存管理与调度…" §三): for each sequence b and query head h, attention of
// q[b,h] over the sequence's K/V, which sit in fixed-size physical blocks named
// by the block table; only the valid slots of the last block count; the
// softmax is accumulated block by block with a running maximum, a running sum
// of exponentials and a rescaled output, normalised at the end.
//
// How (GB300):
//  * Work item = (sequence, partition of P tokens, group of HG KV heads,
//    query-head subgroup).  A persistent grid (resident CTAs x SMs) strides
//    over the items.  With up to kDenseMaxSeqs sequences every CTA first
//    builds the clamped lengths and the prefix sum of partitions per sequence
//    in shared memory and numbers only the real items, sequence by sequence
//    (the HG-group / subgroup index innermost), so each CTA gets the same
//    number of items up to one; beyond that a sparse index over max_parts
//    partitions is used.
//  * Each CTA = 1 producer warp + kConsumerWarps consumer warps.  The producer
//    reads an item's block-table entries with one coalesced warp load, then
//    per block arms a stage's mbarrier (lane 0) and issues the block's TMA
//    tensor loads from parallel lanes: one box {D, HG heads, bs, 1 block} each
//    for K and V on the CUDA-core path, 128-byte-swizzled 128-byte column
//    spans on the tensor-core paths, plus the two scale rows of an e4m3 pool
//    (untiled bulk copies).  A block id outside the pool is flagged and
//    replaced by block 0, so no copy leaves the pool.
//  * Consumer warp w works on head w % HG of the item in warp group w / HG;
//    block i of an item goes to group i % (kConsumerWarps / HG), and every
//    group owns its own ring of SPW stages, consumed strictly in order by all
//    its warps (a ring shared by round-robin consumers lets a warp wait on a
//    stage two phases ahead, where a parity wait matches the stale phase).
//  * Consumers, by pool and group size:
//      - CUDA cores (MHA, fp32, e4m3 MHA, odd groups): LPT lanes share one
//        token, each owning one or two 16-byte chunks of head_dim; scores in
//        the base-2 domain (q pre-multiplied by scale*log2 e), exp2f, one
//        online-softmax state per lane group; on 16/32-bit pools the dot
//        products and the P V update run on packed fp32 pairs (f32x2);
//      - tensor cores, tokens in M (bf16 and e4m3, groups of up to 8):
//        S^T = K Q^T with the 16 tokens of a k-step as the M rows and the
//        heads as N = 8, P^T transposed in registers (movmatrix) into the B
//        operand of O^T = V^T P;
//      - tensor cores, query rows in M (groups of 16): S = Q K^T with the
//        query group as the M rows of m16n8k16.
//    e4m3 codes are converted exactly (cvt.rn.f16x2.e4m3x2); the per-token K
//    scale multiplies the score and the V scale the softmax weight.  Lane
//    groups, warp groups and partitions are merged by log-sum-exp, exact up to
//    rounding (the update is associative).
//  * A sequence whose context fits one partition is normalised and written
//    directly; longer ones write (m, l, unnormalised o) per partition to the
//    workspace, and merge_kernel combines them (on eager calls it is launched
//    as a programmatic dependent: its CTAs may be resident before this grid
//    completes, and it waits for it with griddepcontrol.wait).
//  * Waits are bounded (2 s).  A wait that runs out sets PA_DEV_TIMEOUT and an
//    abort flag; every role then skips the remaining work while still passing
//    the CTA's barriers, and the producer waits (bounded) for the TMA loads it
//    issued before the CTA exits.
#pragma once

#include "pa_common.cuh"
#include "pa_mma.cuh"

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
  int dense;          // 1: enumerate only real items through a per-CTA prefix table (B <= kDenseMaxSeqs)
  float qscale;       // scale * log2(e)
  const float* k_scale;  // e4m3 pools: per-token K scales [num_blocks * bs]; else null
  const float* v_scale;  // e4m3 pools: per-token V scales
  int HG;             // KV heads per work item (one consumer warp each when HG = 4)
  int n_hg;           // Hkv / HG
  int WPH;            // warp groups: kConsumerWarps / HG (warps sharing one head)
  int spg;            // shared-memory stages per warp group
  int spg_shift;      // log2(spg) when spg is a power of two, else -1
  uint32_t tile_bytes;  // one head's K (or V) tile of one block: bs * D * elem
  int32_t* ws_next;     // item counter in the workspace, zero at launch; null: items by static striding
  int lpt;              // dense order: partial last partitions after all full ones, largest first
};

struct Item {
  int b, kvh0, sg, part, t1, jb, je;
  bool split;
};

// Sequences up to which items are enumerated densely: each CTA keeps the
// clamped lengths and the prefix sum of partitions per sequence in shared
// memory (8 bytes per sequence).
constexpr int kDenseMaxSeqs = 1024;

// Items handed out at run time (a workspace holds the counter and the
// enumeration is dense): the producer passes each item index to the consumer
// warps through a queue of kItemQ slots in shared memory.
constexpr int kItemQ = 4;

__device__ __forceinline__ void finish_item(const DecodeParams& p, int L, int nparts, Item& it) {
  const int t0 = it.part * p.part_tokens;
  it.t1 = min(L, t0 + p.part_tokens);
  it.jb = t0 / p.bs;
  it.je = (it.t1 + p.bs - 1) / p.bs;
  if (it.je < it.jb) it.je = it.jb;
  it.split = nparts > 1;
}

// Dense enumeration order, with lpt: every sequence's full partitions first
// (sequence by sequence), then each sequence's partial last partition,
// largest first (a stable counting sort on the remainder in kRemBuckets
// buckets), so the items handed out last are the shortest; without: every
// sequence's partitions in order, sequence by sequence (short partitions:
// their fixed per-item cost then stays spread among long items instead of
// meeting at the end of the launch).  The n_hg * nsub items of a
// (sequence, partition) unit are consecutive.
constexpr int kRemBuckets = 64;

// Bucket of a sequence's partial last partition (-1: it has none): larger
// remainders first, an empty sequence (its one empty unit) last.
__device__ __forceinline__ int rem_bucket(int L, int P) {
  const int rem = L - (L / P) * P;
  if (L > 0 && rem == 0) return -1;
  return kRemBuckets - 1 - min(kRemBuckets - 1, (int)((long long)rem * kRemBuckets / P));
}

// Dense item i -> (sequence, partition, KV-head group, query subgroup).
// pre[b]: the units of the sequences before b in the first class (their
// full partitions with lpt, all their partitions without; pre[B] = NF);
// perm: with lpt, the sequences with a partial last partition in the order
// above.
__device__ __forceinline__ void dense_item(const DecodeParams& p, const int* pre, const int* perm, const int* Ls,
                                           int i, Item& it) {
  const int nper = p.n_hg * p.nsub;
  const int u = i / nper;
  const int r = i - u * nper;
  it.kvh0 = (r % p.n_hg) * p.HG;
  it.sg = r / p.n_hg;
  const int NF = pre[p.B];
  if (u < NF) {
    int lo = 0, hi = p.B - 1;       // the last sequence whose first full unit is <= u
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= u) lo = mid;
      else hi = mid - 1;
    }
    it.b = lo;
    it.part = u - pre[lo];
  } else {
    it.b = perm[u - NF];
    it.part = Ls[it.b] / p.part_tokens;
  }
  const int L = Ls[it.b];
  finish_item(p, L, L > 0 ? (L + p.part_tokens - 1) / p.part_tokens : 1, it);
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
  finish_item(p, L, nparts, it);
  return true;
}

// T: query/output element type; KT: K/V pool element type (T itself, or
// e4m3 codes with a per-token scale for K and for V).
// e4m3 tensor-core instances are held to three CTAs per SM (at most 136
// registers): their per-block conversion work needs the extra warps to hide
// latency (20 % faster on the grouped-query workload than two CTAs per SM).
// Groups of 16 (query rows in M, 64 accumulator registers) get two, which
// they fill without spilling.
#ifndef PA_FP8_MMA_MIN_BLOCKS
#define PA_FP8_MMA_MIN_BLOCKS 3
#endif
template <typename T, typename KT, int D, int GT, bool MMA, int HG>
__global__ void __launch_bounds__(kThreads, (MMA && sizeof(KT) == 1) ? (GT <= 8 ? PA_FP8_MMA_MIN_BLOCKS : 2) : 1)
decode_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
              const DecodeParams p) {
  using E = Elem<T>;                           // queries and output
  using EK = Elem<KT>;                         // K/V pool
  constexpr bool SCALED = EK::kBytes == 1;     // e4m3 codes with per-token scales
  constexpr int CHUNKS = D * EK::kBytes / 16;  // 16-byte chunks per token row
  // chunks per lane: two, except for e4m3 with several query heads, where
  // two chunks (32 dims) per lane would need 2*GT*32 registers for q and o
  constexpr int CPL = (SCALED && GT > 1) ? 1 : 2;
  constexpr int LPT = CHUNKS / CPL;            // lanes per token
  constexpr int TPW = 32 / LPT;                // tokens per warp pass
  constexpr int EPC = EK::kPerChunk;           // elements per chunk
  constexpr int DPL = CPL * EPC;               // head dims per lane
  constexpr int NS = TPW >= 16 ? 1 : 16 / TPW; // tokens per lane group per softmax step
  constexpr int ROW = D * EK::kBytes;          // one head's K (or V) row
  constexpr int QROW = D * E::kBytes;          // one head's query (or output) row
  constexpr int QPC = EPC / E::kPerChunk;      // query 16-byte loads per K/V chunk
  constexpr int NCW = kConsumerWarps;
  static_assert(LPT >= 1 && LPT <= 32 && (32 % LPT) == 0, "lane split");
  static_assert(QPC >= 1 && EPC % E::kPerChunk == 0, "query chunking");
  static_assert(!(SCALED && MMA) || D == 128, "e4m3 tensor-core path: head_dim 128");

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
  // e4m3 pools: each stage also holds the block's bs K scales and bs V scales
  float* sclK = reinterpret_cast<float*>(tilesV + (size_t)S * stage_bytes);
  float* sclV = sclK + (SCALED ? S * p.bs : 0);
  float* mbuf = sclV + (SCALED ? S * p.bs : 0);
  uint64_t* full = reinterpret_cast<uint64_t*>(mbuf + NCW * GT * (D + 2));
  uint64_t* empty = full + S;
  uint64_t* qfull = empty + S;                  // [kItemQ] item queue: index written
  uint64_t* qempty = qfull + kItemQ;            // [kItemQ] item queue: index taken by the consumers
  volatile int* abort_flag = reinterpret_cast<volatile int*>(qempty + kItemQ);
  int* qid = const_cast<int*>(abort_flag) + 4;  // [kItemQ], then the index the consumers work on
  // dense enumeration: partition prefix [B+1], clamped lengths [B], warp sums
  int* pre = qid + kItemQ + 4;
  int* Ls = pre + (p.dense ? p.B + 1 : 0);
  int* perm = Ls + (p.dense ? p.B : 0);          // [B] partial last partitions, largest first
  int* wsum = perm + (p.dense ? p.B : 0);
  // [kRemBuckets * NW + 1] per (bucket, warp) counts while the tables are
  // built: scratch in the K stages, which no copy fills before then
  int* hist = reinterpret_cast<int*>(tilesK);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // the merge kernel (a programmatic dependent on eager calls) may be
  // scheduled now; it waits for this grid's completion before reading
  asm volatile("griddepcontrol.launch_dependents;");

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], HG);
    }
    for (int q = 0; q < kItemQ; ++q) {
      mbar_init(&qfull[q], 1);
      mbar_init(&qempty[q], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  long long n_items = p.n_virtual;
  if (p.dense) {
    // Every CTA builds the same tables: each thread takes a contiguous run
    // of sequences, then a block-wide exclusive scan of the run totals (full
    // partitions per sequence); then a stable counting sort of the
    // sequences with a partial last partition, each warp counting and then
    // placing a contiguous range of sequences (no atomics: every CTA gets the
    // same permutation).
    constexpr int NW = kThreads / 32;
    const int Lmax = p.max_blocks * p.bs;
    const int P = p.part_tokens;
    for (int i = threadIdx.x; i <= kRemBuckets * NW; i += kThreads) hist[i] = 0;
    const int per = (p.B + kThreads - 1) / kThreads;
    const int b0 = min(p.B, (int)threadIdx.x * per), b1 = min(p.B, b0 + per);
    int sum = 0;
    for (int b = b0; b < b1; ++b) {
      int L = __ldg(&p.context_lens[b]);
      if (L < 0 || L > Lmax) L = L < 0 ? 0 : Lmax;   // flagged by the consumer
      Ls[b] = L;
      sum += p.lpt ? L / P : (L > 0 ? (L + P - 1) / P : 1);
    }
    int incl = sum;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    int run = incl - sum;
    for (int w = 0; w < warp; ++w) run += wsum[w];
    for (int b = b0; b < b1; ++b) {
      pre[b] = run;
      run += p.lpt ? Ls[b] / P : (Ls[b] > 0 ? (Ls[b] + P - 1) / P : 1);
    }
    if (threadIdx.x == kThreads - 1) pre[p.B] = run;
    // counts per (bucket, warp) over each warp's range
    const int chunk = (p.B + NW - 1) / NW;
    const int r0 = warp * chunk, r1 = p.lpt ? min(p.B, r0 + chunk) : r0;
    for (int base = r0; base < r1; base += 32) {
      const int b = base + lane;
      const int d = b < r1 ? rem_bucket(Ls[b], P) : -1;
      const unsigned m = __match_any_sync(0xffffffffu, d);
      if (d >= 0 && (m & ((1u << lane) - 1u)) == 0) hist[d * NW + warp] += __popc(m);
      __syncwarp();
    }
    __syncthreads();
    // exclusive scan of the counts (bucket-major, then warp): warp 0
    if (p.lpt && warp == 0) {
      int carry = 0;
      for (int i0 = 0; i0 < kRemBuckets * NW; i0 += 32) {
        const int c = i0 + lane < kRemBuckets * NW ? hist[i0 + lane] : 0;
        int x = c;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, x, off);
          if (lane >= off) x += y;
        }
        if (i0 + lane < kRemBuckets * NW) hist[i0 + lane] = carry + x - c;
        carry += __shfl_sync(0xffffffffu, x, 31);
      }
      if (lane == 0) hist[kRemBuckets * NW] = carry;
    }
    __syncthreads();
    const int nR = hist[kRemBuckets * NW];
    for (int base = r0; base < r1; base += 32) {
      const int b = base + lane;
      const int d = b < r1 ? rem_bucket(Ls[b], P) : -1;
      const unsigned m = __match_any_sync(0xffffffffu, d);
      const int rank = __popc(m & ((1u << lane) - 1u));
      int pos = 0;
      if (d >= 0) pos = hist[d * NW + warp] + rank;
      __syncwarp();
      if (d >= 0) {
        perm[pos] = b;
        if (rank == 0) hist[d * NW + warp] += __popc(m);
      }
      __syncwarp();
    }
    // order these generic writes to the stage memory before the TMA copies
    // that will overwrite it
    fence_proxy_async_smem();
    __syncthreads();
    n_items = (long long)(pre[p.B] + nR) * p.n_hg * p.nsub;
  } else {
    __syncthreads();
  }
  // Run-time items: each CTA's producer takes the next index from the
  // counter when it gets to it (the counter is cleared by the kernel launched
  // just before this one, which this grid may overlap on eager calls: wait
  // for it before the first fetch).
  const bool dyn = p.ws_next != nullptr && p.dense;

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
  // Running block count u of a group -> (stage within the group's ring,
  // phase parity).  Shifts when the ring depth is a power of two: a runtime
  // division here costs a noticeable share of the producer's per-block work.
  const int spw_shift = p.spg_shift;
  auto ring = [SPW, spw_shift](uint32_t u, uint32_t& ph) -> int {
    if (spw_shift >= 0) {
      ph = (u >> spw_shift) & 1u;
      return (int)(u & (uint32_t)(SPW - 1));
    }
    ph = (u / (uint32_t)SPW) & 1u;
    return (int)(u % (uint32_t)SPW);
  };

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
    int pend = 0, kq = 0;
    if (dyn) {
      asm volatile("griddepcontrol.wait;" ::: "memory");
      if (lane == 0) pend = atomicAdd(p.ws_next, 1);
    }
    for (long long v = blockIdx.x;; v += gridDim.x) {
      if (dyn) {
        // hand the next index (-1: none left) to the consumers; the one
        // after it is fetched while this item's loads go out
        const int q = kq % kItemQ;
        int nv = -1;
        if (lane == 0) {
          if (!*abort_flag && mbar_wait(&qempty[q], ((uint32_t)(kq / kItemQ) & 1u) ^ 1u)) {
            nv = pend < n_items ? pend : -1;
            if (nv >= 0) pend = atomicAdd(p.ws_next, 1);
            qid[q] = nv;
            mbar_arrive(&qfull[q]);
          } else if (!*abort_flag) {
            atomicOr(&g_status_decode, PA_DEV_TIMEOUT);
            *abort_flag = 1;
          }
        }
        ++kq;
        v = __shfl_sync(0xffffffffu, nv, 0);
        if (v < 0) break;
      } else if (v >= n_items) {
        break;
      }
      Item item;
      if (p.dense) dense_item(p, pre, perm, Ls, (int)v, item);
      else if (!decode_item(p, v, item)) continue;
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
          uint32_t ph;
          const int st = w * SPW + ring(u, ph);
          constexpr int HALVES = MMA ? D * EK::kBytes / 128 : 1;   // 128-byte swizzled column spans
          constexpr int NOPS = MMA ? 2 * HG * HALVES : 2;   // TMA loads per block
          int go = 0;
          if (lane == 0 && !*abort_flag) {
            if (!mbar_wait(&empty[st], ph ^ 1u)) {
              atomicOr(&g_status_decode, PA_DEV_TIMEOUT);
              *abort_flag = 1;
            } else {
              mbar_arrive_expect_tx(&full[st], 2u * stage_bytes + (SCALED ? 8u * (uint32_t)p.bs : 0u));
              go = 1;
            }
          }
          // The block's copies are issued by parallel lanes in one warp
          // instruction once lane 0 has armed the stage (one thread issuing
          // them in series is slower).
          if (__shfl_sync(0xffffffffu, go, 0)) {
            if constexpr (NOPS == 2) {
              // one box {D, HG heads, bs, 1} each for K (lane 0) and V
              // (lane 1): smem [bs][HG][D]; e4m3 pools also move the block's
              // two scale rows (bs fp32 values each) from lanes 2 and 3
              if (lane < 2)
                tma_load_4d((lane ? tilesV : tilesK) + (size_t)st * stage_bytes, lane ? &mapV : &mapK, &full[st],
                            0, item.kvh0, 0, bi, pol);
              if constexpr (SCALED) {
                if (lane == 2 || lane == 3)
                  bulk_load((lane == 2 ? sclK : sclV) + st * p.bs,
                            (lane == 2 ? p.k_scale : p.v_scale) + (size_t)bi * p.bs, 4u * p.bs, &full[st], pol);
              }
            } else if (lane < NOPS) {
              // tensor-core path: many 128-byte-swizzled column spans per
              // block (64 bf16 or 128 e4m3 columns): lane l takes K (l even)
              // or V (l odd) of head l/2/HALVES, span l/2%HALVES
              const int rest = lane >> 1;
              const int hl = rest / HALVES, hh = rest % HALVES;
              const size_t off = (size_t)st * stage_bytes + (size_t)hl * p.tile_bytes + (size_t)hh * p.bs * 128;
              unsigned char* dst = ((lane & 1) ? tilesV : tilesK) + off;
              tma_load_4d(dst, (lane & 1) ? &mapV : &mapK, &full[st], hh * (128 / EK::kBytes), item.kvh0 + hl, 0,
                          bi, pol);
            } else if (SCALED && (lane == NOPS || lane == NOPS + 1)) {
              const bool vs = lane == NOPS + 1;
              bulk_load((vs ? sclV : sclK) + st * p.bs, (vs ? p.v_scale : p.k_scale) + (size_t)bi * p.bs, 4u * p.bs,
                        &full[st], pol);
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
  // this lane owns chunks li + j*LPT of each row, j < CPL
  const int ctid = threadIdx.x;   // 0 .. NCW*32-1
  uint32_t wcount = 0;            // blocks this warp's group has consumed so far
  const int hl = warp % HG;       // the item's KV head this warp works on
  const int gw = warp / HG;       // this warp's group

  int kq = 0;
  volatile int* cur = qid + kItemQ;   // the index every consumer warp works on next
  for (long long v = blockIdx.x;; v += gridDim.x) {
    if (dyn) {
      // Consumer warp 0 takes the producer's next index (-1: none left, or
      // the pipeline aborted) and every consumer warp reads it after a
      // barrier, so all of them walk the same items and meet at the same
      // per-item barriers.
      if (warp == 0) {
        const int q = kq % kItemQ;
        int nv = -1;
        if (__shfl_sync(0xffffffffu, *abort_flag, 0) == 0) {
          const bool late = !mbar_wait(&qfull[q], (uint32_t)(kq / kItemQ) & 1u);
          if (__any_sync(0xffffffffu, late)) {
            if (lane == 0) {
              atomicOr(&g_status_decode, PA_DEV_TIMEOUT);
              *abort_flag = 1;
            }
          } else {
            nv = qid[q];
          }
        }
        __syncwarp();
        if (lane == 0) {
          *cur = nv;
          if (nv >= 0 || *abort_flag == 0) mbar_arrive(&qempty[q]);
        }
      }
      ++kq;
      named_sync(2, NCW * 32);
      v = *cur;
      if (v < 0) break;
    } else if (v >= n_items) {
      break;
    }
    Item item;
    if (p.dense) dense_item(p, pre, perm, Ls, (int)v, item);
    else if (!decode_item(p, v, item)) continue;
    if (ctid == 0 && item.kvh0 == 0 && item.sg == 0 && item.part == 0) {
      const int L = __ldg(&p.context_lens[item.b]);
      if (L < 0 || L > p.max_blocks * p.bs) atomicOr(&g_status_decode, PA_DEV_BAD_LEN);
    }
    const int h0 = (item.kvh0 + hl) * p.G + item.sg * GT;

    if constexpr (MMA && SCALED && GT <= 8) {
      // e4m3 pool, query group of at most 8 heads: tokens in the M rows.
      // S^T = K Q^T with the 16 tokens of a k-step as M and the query heads
      // as N (8 columns), then O^T = V^T P with head dims as M and heads as N:
      //  * K codes come through ldmatrix as byte pairs (a lane gets dims
      //    4tq..4tq+3 of a 16-dim chunk of one token) and form the A
      //    fragment; the k-step's reduction index is permuted the same way
      //    in the Q^T fragment (slots 2tq,2tq+1 <-> dims 4tq,4tq+1; slots
      //    2tq+8,2tq+9 <-> dims 4tq+2,4tq+3);
      //  * V codes come through ldmatrix.trans; one byte permute splits a
      //    lane's codes into even-dim and odd-dim pairs, so each 16-dim chunk
      //    is one M tile whose rows g and g+8 are dims 2g and 2g+1;
      //  * P^T (tokens x heads, the S^T accumulator) becomes the B operand
      //    through an in-register 8x8 transpose (movmatrix);
      //  * Q, the K and V scales and the f16 range of P are handled as on
      //    the query-rows-in-M path (power-of-two Q scaling, per-token K
      //    scale on the scores, V scale relative to a running power-of-two
      //    reference on P).
      constexpr int KS = D / 16;       // k-steps of S^T
      constexpr int MT = D / 16;       // M tiles of O^T (16 dims each)
      const int g = lane >> 2, tq = lane & 3;
      const bool hv = g < GT;          // this lane's Q^T column (head g) is a real head
      const uint2* qp = reinterpret_cast<const uint2*>(
          static_cast<const unsigned char*>(p.q) + ((size_t)item.b * p.Hq + h0 + (hv ? g : 0)) * QROW);
      uint2 qraw[KS];
      float qmax = 0.f;
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        qraw[kk] = hv ? __ldg(qp + kk * 4 + tq) : make_uint2(0u, 0u);    // dims 16kk+4tq .. +3
        qmax = fmaxf(qmax, fmaxf(fmaxf(fabsf(bf16lo(qraw[kk].x)), fabsf(bf16hi(qraw[kk].x))),
                                 fmaxf(fabsf(bf16lo(qraw[kk].y)), fabsf(bf16hi(qraw[kk].y)))));
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, off));
      int qe = 0;
      if (qmax > 0.f) qe = max(-100, min(100, ilogbf(qmax) - 14));
      const float qdown = ldexpf(1.f, -qe);
      uint32_t qb[KS][2];
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        qb[kk][0] = pack_f16(bf16lo(qraw[kk].x) * qdown, bf16hi(qraw[kk].x) * qdown);
        qb[kk][1] = pack_f16(bf16lo(qraw[kk].y) * qdown, bf16hi(qraw[kk].y) * qdown);
      }
      const float sfac = p.qscale * ldexpf(1.f, qe);
      float OT[MT][4];               // rows: dims 16c+2g (0,1) and 16c+2g+1 (2,3); columns: heads 2tq, 2tq+1
#pragma unroll
      for (int c = 0; c < MT; ++c) OT[c][0] = OT[c][1] = OT[c][2] = OT[c][3] = 0.f;
      float mh[2] = {-INFINITY, -INFINITY}, lh[2] = {0.f, 0.f};   // heads 2tq, 2tq+1 (partial l per lane)
      int rexp = -1000;

      const int nblk = item.je - item.jb;
      for (int i = gw; i < nblk; i += WPH, ++wcount) {
        uint32_t ph;
        const int st = gw * SPW + ring(wcount, ph);
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
          const float* sk = sclK + st * p.bs;
          const float* sv = sclV + st * p.bs;
          if (valid < p.bs) {
            for (int idx = lane; idx < (p.bs - valid) * 8; idx += 32)
              *reinterpret_cast<uint4*>(vt_ptr + (valid + idx / 8) * 128 + (idx % 8) * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
            fence_proxy_async_smem();
            __syncwarp();
          }
          float vmax = 0.f;
          for (int t = lane; t < valid; t += 32) vmax = fmaxf(vmax, sv[t]);
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, off));
          if (vmax > 0.f) {
            const int ve = ilogbf(vmax) + 1;
            if (ve > rexp) {
              if (rexp > -1000) {
                const float f = ldexpf(1.f, rexp - ve);
#pragma unroll
                for (int c = 0; c < MT; ++c) {
                  OT[c][0] *= f;
                  OT[c][1] *= f;
                  OT[c][2] *= f;
                  OT[c][3] *= f;
                }
              }
              rexp = ve;
            }
          }
          const float vdown = rexp > -1000 ? ldexpf(1.f, -rexp) : 0.f;
          for (int tb = 0; tb < valid; tb += 16) {
            // S^T: rows tokens tb+g, tb+g+8; columns heads 2tq, 2tq+1
            float St[4] = {0.f, 0.f, 0.f, 0.f};
            {
              // lanes 0-7: tokens tb..+7, chunk 2kp; 8-15: tokens tb+8..+15,
              // chunk 2kp; 16-31: the same for chunk 2kp+1
              const int tt = min(tb + (lane & 7) + (((lane >> 3) & 1) << 3), p.bs - 1);
#pragma unroll
              for (int kp = 0; kp < KS / 2; ++kp) {
                const int c = 2 * kp + (lane >> 4);
                uint32_t r0, r1, r2, r3;
                ldsm_x4(kt + tt * 128 + ((c ^ (tt & 7)) << 4), r0, r1, r2, r3);
                uint32_t a[2][4];
                e4m3x4_to_f16x2x2(r0, a[0][0], a[0][2]);    // tokens 0-7: dims 4tq..+1, 4tq+2..+3
                e4m3x4_to_f16x2x2(r1, a[0][1], a[0][3]);    // tokens 8-15
                e4m3x4_to_f16x2x2(r2, a[1][0], a[1][2]);
                e4m3x4_to_f16x2x2(r3, a[1][1], a[1][3]);
                mma_f16_16816(St, a[0], qb[2 * kp][0], qb[2 * kp][1]);
                mma_f16_16816(St, a[1], qb[2 * kp + 1][0], qb[2 * kp + 1][1]);
              }
            }
            const int t0 = tb + g, t1 = tb + g + 8;
            const bool ok0 = t0 < valid, ok1 = t1 < valid;
            const float f0 = ok0 ? sfac * sk[t0] : 0.f, f1 = ok1 ? sfac * sk[t1] : 0.f;
            St[0] = ok0 ? St[0] * f0 : -INFINITY;
            St[1] = ok0 ? St[1] * f0 : -INFINITY;
            St[2] = ok1 ? St[2] * f1 : -INFINITY;
            St[3] = ok1 ? St[3] * f1 : -INFINITY;
            float alpha[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              float mx = fmaxf(St[e], St[2 + e]);
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
              const float mn = fmaxf(mh[e], mx);
              alpha[e] = mn == -INFINITY ? 1.f : exp2f(mh[e] - mn);
              mh[e] = mn;
              lh[e] *= alpha[e];
            }
            if (alpha[0] != 1.f || alpha[1] != 1.f) {
#pragma unroll
              for (int c = 0; c < MT; ++c) {
                OT[c][0] *= alpha[0];
                OT[c][1] *= alpha[1];
                OT[c][2] *= alpha[0];
                OT[c][3] *= alpha[1];
              }
            }
            const float vs0 = ok0 ? sv[t0] * vdown : 0.f, vs1 = ok1 ? sv[t1] * vdown : 0.f;
            float pw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float pk = St[e] == -INFINITY ? 0.f : exp2f(St[e] - mh[e & 1]);
              lh[e & 1] += pk;
              pw[e] = pk * (e < 2 ? vs0 : vs1);
            }
            // P^T as the B operand: transpose the two 8x8 (tokens x heads) halves
            const uint32_t b0 = movmatrix_t(pack_f16(pw[0], pw[1]));   // tokens 0-7
            const uint32_t b1 = movmatrix_t(pack_f16(pw[2], pw[3]));   // tokens 8-15
            {
              // ldmatrix.trans: lanes 0-7 tokens tb..+7, 8-15 tokens tb+8..+15
              // (chunk 2j); lanes 16-31 the same for chunk 2j+1
              const int tt = min(tb + (lane & 7) + (((lane >> 3) & 1) << 3), p.bs - 1);
#pragma unroll
              for (int j = 0; j < D / 32; ++j) {
                const int c = 2 * j + (lane >> 4);
                uint32_t r0, r1, r2, r3;
                ldsm_x4_t(vt + tt * 128 + ((c ^ (tt & 7)) << 4), r0, r1, r2, r3);
                uint32_t a0[4], a1[4];   // {even dims tokens 0-7, odd dims tokens 0-7, even 8-15, odd 8-15}
                e4m3x4_to_f16x2x2(__byte_perm(r0, 0u, 0x3120), a0[0], a0[1]);
                e4m3x4_to_f16x2x2(__byte_perm(r1, 0u, 0x3120), a0[2], a0[3]);
                e4m3x4_to_f16x2x2(__byte_perm(r2, 0u, 0x3120), a1[0], a1[1]);
                e4m3x4_to_f16x2x2(__byte_perm(r3, 0u, 0x3120), a1[2], a1[3]);
                mma_f16_16816(OT[2 * j], a0, b0, b1);
                mma_f16_16816(OT[2 * j + 1], a1, b0, b1);
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
      }
      // the row sums are split over the 8 lanes sharing tq
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        lh[e] += __shfl_xor_sync(0xffffffffu, lh[e], 4);
        lh[e] += __shfl_xor_sync(0xffffffffu, lh[e], 8);
        lh[e] += __shfl_xor_sync(0xffffffffu, lh[e], 16);
      }
      const float vup = rexp > -1000 ? ldexpf(1.f, rexp) : 0.f;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int h = 2 * tq + e;
        if (h < GT) {
          float* dst = mbuf + (warp * GT + h) * (D + 2);
#pragma unroll
          for (int c = 0; c < MT; ++c) {
            dst[16 * c + 2 * g] = OT[c][e] * vup;
            dst[16 * c + 2 * g + 1] = OT[c][2 + e] * vup;
          }
          if (g == 0) {
            dst[D] = mh[e];
            dst[D + 1] = lh[e];
          }
        }
      }
    } else if constexpr (MMA && SCALED) {
      // e4m3 pool on tensor cores (f16 m16n8k16, fp32 accumulation), the
      // query group in the M rows as on the bf16 path.  Differences:
      //  * K codes are read with ldmatrix as byte pairs: a lane gets 4
      //    consecutive codes (head dims 4tq..4tq+3 of a 16-dim chunk) of one
      //    token, converted exactly to two f16x2 values.  The reduction
      //    index of each k-step is permuted the same way in the Q fragment
      //    (slots 2tq,2tq+1 <-> dims 4tq,4tq+1; slots 2tq+8,2tq+9 <-> dims
      //    4tq+2,4tq+3), which leaves Q K^T unchanged.
      //  * Q is converted to f16 after a per-item power-of-two scaling that
      //    puts its largest magnitude in [2^14, 2^15), so the conversion is
      //    exact for every value within 2^-28 of that maximum; the scores
      //    get the inverse power of two with the softmax scale, and each
      //    token's K scale.
      //  * V codes are read with ldmatrix.trans as byte pairs; one byte
      //    permute splits a lane's 4 codes into its even-dim and odd-dim
      //    pairs, so each 16-dim chunk gives two n-tiles (even dims, odd
      //    dims) of the output.
      //  * P carries the token's V scale relative to a running power-of-two
      //    reference 2^rexp (the largest V scale seen, rounded up), so the
      //    f16 P stays in [0, 1]; O is rescaled when the reference grows and
      //    multiplied back by 2^rexp at the end.  The softmax sum uses the
      //    unscaled weights.
      constexpr int KS = D / 16;       // k-steps of Q K^T
      constexpr int NT = D / 8;        // output n-tiles (two per 16-dim chunk)
      const int g = lane >> 2, tq = lane & 3;
      const bool r0v = g < GT, r1v = g + 8 < GT;
      const uint2* q0p = reinterpret_cast<const uint2*>(
          static_cast<const unsigned char*>(p.q) + ((size_t)item.b * p.Hq + h0 + (r0v ? g : 0)) * QROW);
      const uint2* q1p = reinterpret_cast<const uint2*>(
          static_cast<const unsigned char*>(p.q) + ((size_t)item.b * p.Hq + h0 + (r1v ? g + 8 : 0)) * QROW);
      uint2 qraw[KS][2];
      float qmax = 0.f;
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        qraw[kk][0] = r0v ? __ldg(q0p + kk * 4 + tq) : make_uint2(0u, 0u);   // dims 16kk+4tq .. +3
        qraw[kk][1] = r1v ? __ldg(q1p + kk * 4 + tq) : make_uint2(0u, 0u);
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          qmax = fmaxf(qmax, fmaxf(fabsf(bf16lo(qraw[kk][r].x)), fabsf(bf16hi(qraw[kk][r].x))));
          qmax = fmaxf(qmax, fmaxf(fabsf(bf16lo(qraw[kk][r].y)), fabsf(bf16hi(qraw[kk][r].y))));
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, off));
      // 2^qe >= qmax / 2^15, so |q| * 2^-qe <= 2^15 < 65504
      int qe = 0;
      if (qmax > 0.f) qe = max(-100, min(100, ilogbf(qmax) - 14));
      const float qdown = ldexpf(1.f, -qe);
      uint32_t qa[KS][4];
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        qa[kk][0] = pack_f16(bf16lo(qraw[kk][0].x) * qdown, bf16hi(qraw[kk][0].x) * qdown);
        qa[kk][1] = pack_f16(bf16lo(qraw[kk][1].x) * qdown, bf16hi(qraw[kk][1].x) * qdown);
        qa[kk][2] = pack_f16(bf16lo(qraw[kk][0].y) * qdown, bf16hi(qraw[kk][0].y) * qdown);
        qa[kk][3] = pack_f16(bf16lo(qraw[kk][1].y) * qdown, bf16hi(qraw[kk][1].y) * qdown);
      }
      const float sfac = p.qscale * ldexpf(1.f, qe);
      float O[NT][4];
#pragma unroll
      for (int n = 0; n < NT; ++n) O[n][0] = O[n][1] = O[n][2] = O[n][3] = 0.f;
      float mr[2] = {-INFINITY, -INFINITY}, lr[2] = {0.f, 0.f};
      int rexp = -1000;                // V-scale reference exponent (none yet)

      const int nblk = item.je - item.jb;
      for (int i = gw; i < nblk; i += WPH, ++wcount) {
        uint32_t ph;
        const int st = gw * SPW + ring(wcount, ph);
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
          const float* sk = sclK + st * p.bs;
          const float* sv = sclV + st * p.bs;
          if (valid < p.bs) {
            // slots past the context may hold anything (NaN codes): clear
            // those V rows (P is 0 there, but 0 * NaN would be NaN)
            for (int idx = lane; idx < (p.bs - valid) * 8; idx += 32)
              *reinterpret_cast<uint4*>(vt_ptr + (valid + idx / 8) * 128 + (idx % 8) * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
            fence_proxy_async_smem();
            __syncwarp();
          }
          // V-scale reference for this block (valid tokens only)
          float vmax = 0.f;
          for (int t = lane; t < valid; t += 32) vmax = fmaxf(vmax, sv[t]);
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, off));
          if (vmax > 0.f) {
            const int ve = ilogbf(vmax) + 1;          // 2^ve > vmax
            if (ve > rexp) {
              if (rexp > -1000) {
                const float f = ldexpf(1.f, rexp - ve);
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                  O[n][0] *= f;
                  O[n][1] *= f;
                  O[n][2] *= f;
                  O[n][3] *= f;
                }
              }
              rexp = ve;
            }
          }
          const float vdown = rexp > -1000 ? ldexpf(1.f, -rexp) : 0.f;
          for (int tb = 0; tb < valid; tb += 16) {
            float S[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
            {
              // lanes 0-7: tokens tb..+7, chunk 2kp; 8-15: same tokens,
              // chunk 2kp+1; 16-31: tokens tb+8..+15, chunks 2kp, 2kp+1
              const int tt = min(tb + (lane & 7) + ((lane >> 4) << 3), p.bs - 1);
#pragma unroll
              for (int kp = 0; kp < KS / 2; ++kp) {
                const int c = 2 * kp + ((lane >> 3) & 1);
                uint32_t r0, r1, r2, r3;
                ldsm_x4(kt + tt * 128 + ((c ^ (tt & 7)) << 4), r0, r1, r2, r3);
                uint32_t b[4][2];
                e4m3x4_to_f16x2x2(r0, b[0][0], b[0][1]);
                e4m3x4_to_f16x2x2(r1, b[1][0], b[1][1]);
                e4m3x4_to_f16x2x2(r2, b[2][0], b[2][1]);
                e4m3x4_to_f16x2x2(r3, b[3][0], b[3][1]);
                mma_f16_16816(S[0], qa[2 * kp], b[0][0], b[0][1]);
                mma_f16_16816(S[0], qa[2 * kp + 1], b[1][0], b[1][1]);
                mma_f16_16816(S[1], qa[2 * kp], b[2][0], b[2][1]);
                mma_f16_16816(S[1], qa[2 * kp + 1], b[3][0], b[3][1]);
              }
            }
            float mx[2] = {-INFINITY, -INFINITY};
            float vsc[2][2];
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const int t = tb + n * 8 + 2 * tq + (e & 1);
                const bool ok = t < valid;
                S[n][e] = ok ? S[n][e] * (sfac * sk[t]) : -INFINITY;
                if (e < 2) vsc[n][e] = ok ? sv[t] * vdown : 0.f;
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
            float pw[2][4];
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float pk = (S[n][e] == -INFINITY) ? 0.f : exp2f(S[n][e] - mr[e >> 1]);
                lr[e >> 1] += pk;
                pw[n][e] = pk * vsc[n][e & 1];
              }
            const uint32_t pa[4] = {pack_f16(pw[0][0], pw[0][1]), pack_f16(pw[0][2], pw[0][3]),
                                    pack_f16(pw[1][0], pw[1][1]), pack_f16(pw[1][2], pw[1][3])};
            {
              // ldmatrix.trans: lanes 0-7 tokens tb..+7, 8-15 tokens tb+8..+15
              // (chunk 2j); lanes 16-31 the same for chunk 2j+1.  A lane gets
              // codes (token 2tq: dims 2g, 2g+1; token 2tq+1: dims 2g, 2g+1).
              const int tt = min(tb + (lane & 7) + (((lane >> 3) & 1) << 3), p.bs - 1);
#pragma unroll
              for (int j = 0; j < D / 32; ++j) {
                const int c = 2 * j + (lane >> 4);
                uint32_t r0, r1, r2, r3;
                ldsm_x4_t(vt + tt * 128 + ((c ^ (tt & 7)) << 4), r0, r1, r2, r3);
                // bytes [b0 b2 | b1 b3]: even-dim pair low, odd-dim pair high
                uint32_t ev[4], od[4];   // even-dim / odd-dim f16x2 pairs of r0..r3
                e4m3x4_to_f16x2x2(__byte_perm(r0, 0u, 0x3120), ev[0], od[0]);
                e4m3x4_to_f16x2x2(__byte_perm(r1, 0u, 0x3120), ev[1], od[1]);
                e4m3x4_to_f16x2x2(__byte_perm(r2, 0u, 0x3120), ev[2], od[2]);
                e4m3x4_to_f16x2x2(__byte_perm(r3, 0u, 0x3120), ev[3], od[3]);
                mma_f16_16816(O[4 * j + 0], pa, ev[0], ev[1]);
                mma_f16_16816(O[4 * j + 1], pa, od[0], od[1]);
                mma_f16_16816(O[4 * j + 2], pa, ev[2], ev[3]);
                mma_f16_16816(O[4 * j + 3], pa, od[2], od[3]);
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
      }
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        lr[r] += __shfl_xor_sync(0xffffffffu, lr[r], 1);
        lr[r] += __shfl_xor_sync(0xffffffffu, lr[r], 2);
      }
      const float vup = rexp > -1000 ? ldexpf(1.f, rexp) : 0.f;
#pragma unroll
      for (int r = 0; r < 2; ++r) {
        const int h = g + 8 * r;
        if (h < GT) {
          float* dst = mbuf + (warp * GT + h) * (D + 2);
          // n-tile nt = 2*chunk + parity holds dims 16*chunk + 2*col + parity
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            const int d0 = 16 * (n >> 1) + 4 * tq + (n & 1);
            dst[d0] = O[n][2 * r] * vup;
            dst[d0 + 2] = O[n][2 * r + 1] * vup;
          }
          if (tq == 0) {
            dst[D] = mr[r];
            dst[D + 1] = lr[r];
          }
        }
      }
    } else if constexpr (MMA && GT <= 8) {
      // bf16 pool, query group of at most 8 heads: tokens in the M rows.
      // S^T = K Q^T (M = 16 tokens, N = 8 heads) with K rows straight from
      // ldmatrix as the A fragment; O^T = V^T P (M = 16 head dims, N = heads)
      // with V^T from ldmatrix.trans and P^T turned into the B operand by an
      // in-register 8x8 transpose.  Half the MMAs of the query-rows-in-M
      // formulation for groups of up to 8, and O^T in 32 registers.
      constexpr int KS = D / 16;       // k-steps of S^T
      constexpr int MT = D / 16;       // M tiles of O^T
      const int g = lane >> 2, tq = lane & 3;
      const bool hv = g < GT;
      const uint32_t* qp = reinterpret_cast<const uint32_t*>(
          static_cast<const unsigned char*>(p.q) + ((size_t)item.b * p.Hq + h0 + (hv ? g : 0)) * QROW);
      uint32_t qb[KS][2];             // Q^T B fragment: head g, dims 16kk+2tq..+1 and 16kk+2tq+8..+9
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        qb[kk][0] = hv ? __ldg(qp + kk * 8 + tq) : 0u;
        qb[kk][1] = hv ? __ldg(qp + kk * 8 + 4 + tq) : 0u;
      }
      float OT[MT][4];               // rows: dims 16m+g (0,1) and 16m+8+g (2,3); columns: heads 2tq, 2tq+1
#pragma unroll
      for (int m = 0; m < MT; ++m) OT[m][0] = OT[m][1] = OT[m][2] = OT[m][3] = 0.f;
      float mh[2] = {-INFINITY, -INFINITY}, lh[2] = {0.f, 0.f};
      const uint32_t half_bytes = (uint32_t)p.bs * 128u;

      const int nblk = item.je - item.jb;
      for (int i = gw; i < nblk; i += WPH, ++wcount) {
        uint32_t ph;
        const int st = gw * SPW + ring(wcount, ph);
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
            // slots past the context may hold anything: clear those V rows
            for (int idx = lane; idx < (p.bs - valid) * (D / 8); idx += 32) {
              const int t = valid + idx / (D / 8), c = idx % (D / 8);
              *reinterpret_cast<uint4*>(vt_ptr + (c >> 3) * half_bytes + t * 128 + (c & 7) * 16) =
                  make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
          for (int tb = 0; tb < valid; tb += 16) {
            float St[4] = {0.f, 0.f, 0.f, 0.f};
            {
              // lanes 0-7: tokens tb..+7, chunk 2kk; 8-15: tokens tb+8..+15,
              // chunk 2kk; 16-31: the same for chunk 2kk+1 (8 dims per chunk)
              const int tt = min(tb + (lane & 7) + (((lane >> 3) & 1) << 3), p.bs - 1);
#pragma unroll
              for (int kk = 0; kk < KS; ++kk) {
                const int c = 2 * kk + (lane >> 4);
                uint32_t a[4];
                ldsm_x4(kt + (c >> 3) * half_bytes + tt * 128 + (((c & 7) ^ (tt & 7)) << 4), a[0], a[1], a[2], a[3]);
                mma_bf16_16816(St, a, qb[kk][0], qb[kk][1]);
              }
            }
            const int t0 = tb + g, t1 = tb + g + 8;
            const bool ok0 = t0 < valid, ok1 = t1 < valid;
            St[0] = ok0 ? St[0] * p.qscale : -INFINITY;
            St[1] = ok0 ? St[1] * p.qscale : -INFINITY;
            St[2] = ok1 ? St[2] * p.qscale : -INFINITY;
            St[3] = ok1 ? St[3] * p.qscale : -INFINITY;
            float alpha[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              float mx = fmaxf(St[e], St[2 + e]);
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
              mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
              const float mn = fmaxf(mh[e], mx);
              alpha[e] = mn == -INFINITY ? 1.f : exp2f(mh[e] - mn);
              mh[e] = mn;
              lh[e] *= alpha[e];
            }
            if (alpha[0] != 1.f || alpha[1] != 1.f) {
#pragma unroll
              for (int m = 0; m < MT; ++m) {
                OT[m][0] *= alpha[0];
                OT[m][1] *= alpha[1];
                OT[m][2] *= alpha[0];
                OT[m][3] *= alpha[1];
              }
            }
            float pw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              pw[e] = St[e] == -INFINITY ? 0.f : exp2f(St[e] - mh[e & 1]);
              lh[e & 1] += pw[e];
            }
            const uint32_t b0 = movmatrix_t(pack_bf16(pw[0], pw[1]));   // tokens 0-7
            const uint32_t b1 = movmatrix_t(pack_bf16(pw[2], pw[3]));   // tokens 8-15
            {
              // ldmatrix.trans: lanes 0-7 tokens tb..+7 chunk 2m; 8-15 the
              // same tokens, chunk 2m+1; 16-31 tokens tb+8..+15, chunks 2m, 2m+1
              const int tt = min(tb + (lane & 7) + ((lane >> 4) << 3), p.bs - 1);
#pragma unroll
              for (int m = 0; m < MT; ++m) {
                const int c = 2 * m + ((lane >> 3) & 1);
                uint32_t a[4];
                ldsm_x4_t(vt + (c >> 3) * half_bytes + tt * 128 + (((c & 7) ^ (tt & 7)) << 4), a[0], a[1], a[2],
                          a[3]);
                mma_bf16_16816(OT[m], a, b0, b1);
              }
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        lh[e] += __shfl_xor_sync(0xffffffffu, lh[e], 4);
        lh[e] += __shfl_xor_sync(0xffffffffu, lh[e], 8);
        lh[e] += __shfl_xor_sync(0xffffffffu, lh[e], 16);
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int h = 2 * tq + e;
        if (h < GT) {
          float* dst = mbuf + (warp * GT + h) * (D + 2);
#pragma unroll
          for (int m = 0; m < MT; ++m) {
            dst[16 * m + g] = OT[m][e];
            dst[16 * m + 8 + g] = OT[m][2 + e];
          }
          if (g == 0) {
            dst[D] = mh[e];
            dst[D + 1] = lh[e];
          }
        }
      }
    } else if constexpr (MMA) {
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
          static_cast<const unsigned char*>(p.q) + ((size_t)item.b * p.Hq + h0 + (r0v ? g : 0)) * QROW);
      const uint32_t* q1p = reinterpret_cast<const uint32_t*>(
          static_cast<const unsigned char*>(p.q) + ((size_t)item.b * p.Hq + h0 + (r1v ? g + 8 : 0)) * QROW);
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
        uint32_t ph;
        const int st = gw * SPW + ring(wcount, ph);
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
            static_cast<const unsigned char*>(p.q) + ((size_t)item.b * p.Hq + h0 + h) * QROW;
        // this lane's head dims: its CPL K/V chunks, EPC dims each
  #pragma unroll
        for (int hf = 0; hf < CPL; ++hf) {
  #pragma unroll
          for (int j = 0; j < QPC; ++j) {
            float f[E::kPerChunk];
            const int d0 = (li + hf * LPT) * EPC + j * E::kPerChunk;
            E::unpack(__ldg(reinterpret_cast<const uint4*>(qrow + (size_t)d0 * E::kBytes)), f);
  #pragma unroll
            for (int e = 0; e < E::kPerChunk; ++e) q[h][hf * EPC + j * E::kPerChunk + e] = f[e] * p.qscale;
          }
        }
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
        uint32_t ph;
        const int st = gw * SPW + ring(wcount, ph);
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
  #pragma unroll
                for (int hf = 0; hf < CPL; ++hf)
                  EK::unpack(*reinterpret_cast<const uint4*>(kt + t * (HG * ROW) + (li + hf * LPT) * 16),
                             kf + hf * EPC);
  #pragma unroll
                for (int h = 0; h < GT; ++h) {
                  if constexpr (SCALED) {
                    // e4m3: scalar FMAs (the widened codes do not pair up in
                    // registers: the packed form measured 15 % slower)
  #pragma unroll
                    for (int d = 0; d < DPL; ++d) part[h] = fmaf(q[h][d], kf[d], part[h]);
                  } else {
                    // two interleaved partial sums on packed fp32 pairs
                    uint64_t acc = f2pack(0.f, 0.f);
  #pragma unroll
                    for (int d = 0; d < DPL; d += 2)
                      acc = ffma2(f2pack(q[h][d], q[h][d + 1]), f2pack(kf[d], kf[d + 1]), acc);
                    float a0, a1;
                    f2unpack(acc, a0, a1);
                    part[h] = a0 + a1;
                  }
                }
              }
              // e4m3: the token's K scale multiplies its whole score
              float ksc = 1.f;
              if constexpr (SCALED) ksc = ok ? sclK[st * p.bs + t] : 0.f;
  #pragma unroll
              for (int h = 0; h < GT; ++h) {
  #pragma unroll
                for (int off = LPT / 2; off > 0; off >>= 1)
                  part[h] += __shfl_xor_sync(0xffffffffu, part[h], off);
                s[k][h] = ok ? part[h] * ksc : -INFINITY;
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
              if constexpr (SCALED) {
  #pragma unroll
                for (int d = 0; d < DPL; ++d) o[h][d] *= alpha;
              } else {
                const uint64_t al2 = f2pack(alpha, alpha);
  #pragma unroll
                for (int d = 0; d < DPL; d += 2) {
                  const uint64_t o2 = fmul2(f2pack(o[h][d], o[h][d + 1]), al2);
                  f2unpack(o2, o[h][d], o[h][d + 1]);
                }
              }
            }
  #pragma unroll
            for (int k = 0; k < NS; ++k) {
              const int t = tb + k * TPW + grp;
              if (t < valid) {
                float vf[DPL];
  #pragma unroll
                for (int hf = 0; hf < CPL; ++hf)
                  EK::unpack(*reinterpret_cast<const uint4*>(vt + t * (HG * ROW) + (li + hf * LPT) * 16),
                             vf + hf * EPC);
                // e4m3: the token's V scale rides on its softmax weight
                float vsc = 1.f;
                if constexpr (SCALED) vsc = sclV[st * p.bs + t];
  #pragma unroll
                for (int h = 0; h < GT; ++h) {
                  const float pk = exp2f(s[k][h] - m[h]);
                  l[h] += pk;
                  const float pw = SCALED ? pk * vsc : pk;
                  if constexpr (SCALED) {
  #pragma unroll
                    for (int d = 0; d < DPL; ++d) o[h][d] = fmaf(pw, vf[d], o[h][d]);
                  } else {
                    const uint64_t pw2 = f2pack(pw, pw);
  #pragma unroll
                    for (int d = 0; d < DPL; d += 2) {
                      const uint64_t o2 = ffma2(pw2, f2pack(vf[d], vf[d + 1]), f2pack(o[h][d], o[h][d + 1]));
                      f2unpack(o2, o[h][d], o[h][d + 1]);
                    }
                  }
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
  #pragma unroll
            for (int hf = 0; hf < CPL; ++hf) dst[(li + hf * LPT) * EPC + e] = o[h][hf * EPC + e];
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

// One warp per (sequence, query head) with more than one partition:
// out = sum_i 2^(m_i - M) o_i / sum_i 2^(m_i - M) l_i with M = max_i m_i.
// Lane i < 32 computes partition i's weight (broadcast by shuffle); each
// partition's row of o is read as one vector of D/32 floats per lane.
template <typename T, int D>
__global__ void __launch_bounds__(256)
merge_kernel(const DecodeParams p) {
  using E = Elem<T>;
  constexpr int VPL = D / 32;                 // dims per lane: 4, 2 or 1
  const long long gw = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (gw >= (long long)p.B * p.Hq) return;
  const int b = (int)(gw / p.Hq);
  int L = __ldg(&p.context_lens[b]);
  const int Lmax = p.max_blocks * p.bs;
  if (L < 0 || L > Lmax) L = L < 0 ? 0 : Lmax;
  const int nparts = L > 0 ? (L + p.part_tokens - 1) / p.part_tokens : 1;
  if (nparts <= 1) return;
  // launched as a programmatic dependent of the decode kernel (eager calls):
  // the partials are read only once that grid has completed and its writes
  // are visible; a plain launch passes straight through
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const size_t base = (size_t)gw * p.max_parts;
  float M = -INFINITY;
  for (int i = lane; i < nparts; i += 32) M = fmaxf(M, p.ws_ml[(base + i) * 2]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float den = 0.f;
  float acc[VPL];
#pragma unroll
  for (int k = 0; k < VPL; ++k) acc[k] = 0.f;
  for (int i0 = 0; i0 < nparts; i0 += 32) {
    const int i = i0 + lane;
    float w = 0.f;
    if (i < nparts) {
      const float mi = p.ws_ml[(base + i) * 2];
      w = mi == -INFINITY ? 0.f : exp2f(mi - M);
      den = fmaf(w, p.ws_ml[(base + i) * 2 + 1], den);
    }
    const int cnt = min(32, nparts - i0);
    const float* o = p.ws_o + (base + i0) * D + lane * VPL;
#pragma unroll 4
    for (int k = 0; k < cnt; ++k) {
      const float wk = __shfl_sync(0xffffffffu, w, k);
      if constexpr (VPL == 4) {
        const float4 v = *reinterpret_cast<const float4*>(o + (size_t)k * D);
        acc[0] = fmaf(wk, v.x, acc[0]);
        acc[1] = fmaf(wk, v.y, acc[1]);
        acc[2] = fmaf(wk, v.z, acc[2]);
        acc[3] = fmaf(wk, v.w, acc[3]);
      } else if constexpr (VPL == 2) {
        const float2 v = *reinterpret_cast<const float2*>(o + (size_t)k * D);
        acc[0] = fmaf(wk, v.x, acc[0]);
        acc[1] = fmaf(wk, v.y, acc[1]);
      } else {
        acc[0] = fmaf(wk, o[(size_t)k * D], acc[0]);
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
  const float inv = den > 0.f ? 1.f / den : 0.f;
  T* out = static_cast<T*>(p.out) + (size_t)gw * D + lane * VPL;
#pragma unroll
  for (int k = 0; k < VPL; ++k) E::store1(out + k, acc[k] * inv);
}

}  // namespace

// A decode kernel and the merge kernel that goes with it.
struct Launch {
  const void* kernel;
  const void* merge;
};

// e4m3-pool instances (pa_decode_fp8.cu): bf16 queries, hg KV heads per
// work item, tensor cores (head_dim 128, gt a power of two >= 2) or CUDA cores.
Launch pick_decode_fp8(int head_dim, int gt, int hg, bool mma);

}  // namespace pa
