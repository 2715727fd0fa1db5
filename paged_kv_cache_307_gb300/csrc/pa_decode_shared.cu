// pa_decode_shared.cu — paged decode attention for batches whose sequences
// share prompt blocks (pa_decode_shared).
//
// What it computes: the result of pa_decode.  Samples drawn from one prompt
// (parallel sampling, beam search, a common system prompt) point their block
// tables at the same physical blocks for the prompt, each block carrying a
// reference count ("19.2 KV Cache 系统化管理" §19.2.2 Fig 19-8 and §19.2.5;
// "LLM 推理引擎的内存管理与调度…" §四).  The caller names those groups: the
// sequences group_start[g] .. group_start[g+1]-1 hold the same first
// shared_blocks[g] block-table entries.  Attention over the shared tokens is
// then one dense product for the whole group: every query row of every
// member reads the same K/V rows.  The online softmax of §19.2.3 is
// associative, so each member's result is the log-sum-exp combination of
// its state over the shared blocks and its state over its own tail.
//
// How (GB300):
//  * Work item = either a SHARED item (group, partition of the shared
//    blocks, KV heads, row chunk) whose rows are (member, query head) pairs
//    of the group, or a TAIL item (sequence, partition of its own tokens
//    after the shared blocks, four KV heads) whose rows are the sequence's
//    query heads.  A shared block is read from HBM once for every row of the
//    group instead of once per member.
//  * Every CTA builds, in shared memory, the clamped lengths, the per-group
//    shared length S_g = min(shared_blocks[g], floor(L_b / bs) over the
//    members) and prefix sums of items in three classes, handed out in this
//    order: tail items larger than a full shared item, the shared items
//    (512-token partitions by default), the other tail items; the tail
//    items of each class go largest first (a stable counting sort of the
//    sequences on their tail length), so the last items to start are the
//    shortest and the CTAs finish close together.  A persistent
//    grid takes items at run time from a counter in the workspace (cleared
//    by a one-thread kernel launched just before, whose programmatic
//    dependent the decode kernel is on eager calls: its CTAs build their
//    tables while the clear runs and wait for it on the device before the
//    first fetch): the producer fetches the next index while
//    the current item's loads go out and passes each index to the consumer
//    warps through a four-slot queue in shared memory, so a CTA that
//    finishes early takes the next item instead of idling.
//  * One producer warp per CTA fills a ring of stages by TMA; a stage holds
//    four (block, KV head) tiles of K and V (128-byte-swizzled 64-column
//    spans): four heads of one block, or two heads of two blocks.
//  * Four consumer warps run tensor-core products with the block's tokens as
//    the M rows (S^T = K Q^T, m16n8k16, then O^T = V^T P with P^T
//    transposed in registers by movmatrix): each warp owns 8 or 16 query
//    rows (one or two n-tiles) of one KV head.  Groups of up to 16 rows per
//    head: one warp per head, four heads per stage.  Groups of 17..32 rows:
//    two warps per head (16 rows each), two heads of two blocks per stage.
//    Larger groups are split into chunks of 32 rows.  Tails: one warp per
//    head, the sequence's G query heads as the columns.
//  * A warp owns whole rows over all of an item's tokens, so no merge
//    between warps.  A row whose sequence has one partition in all writes
//    its normalised output; otherwise it writes (max, sum, unnormalised
//    output) to its partition's slot of the workspace and a merge kernel
//    combines the slots (on eager calls launched as a programmatic dependent
//    that waits for this grid on the device).
//  * Waits are bounded (2 s) as in pa_decode: a wait that runs out sets
//    PA_DEV_TIMEOUT, the CTA skips its remaining work and waits (bounded) for
//    its own TMA loads before it exits.
#include "pa_common.cuh"
#include "pa_mma.cuh"

#include <map>
#include <mutex>
#include <tuple>

namespace pa {
namespace {

__device__ unsigned g_status_shared;

constexpr int kSW = 4;                       // consumer warps
constexpr int kST = (kSW + 1) * 32;          // threads per CTA
constexpr int kTiles = 4;                    // (block, KV head) tiles per stage
constexpr int kSMaxSeqs = 1024;              // sequences per call on this path
constexpr int kSMaxGroups = 1024;            // groups per call on this path
constexpr float kLog2eS = 1.4426950408889634f;
constexpr uint32_t kAlign = 1024;
constexpr int kQ = 4;                        // item queue slots (producer -> consumers)
constexpr int kKH = 32;                      // tail-size buckets per class (big tails, others)
constexpr int kLB = 8;                       // lengths loaded per thread per round of global loads

struct SParams {
  void* out;
  const void* q;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* group_start;
  const int32_t* shared_blocks;
  float* ws_ml;                 // [B*Hq*max_parts][2]  (m in log2 units, l)
  float* ws_o;                  // [B*Hq*max_parts][D]
  int32_t* ws_parts;            // [B] partitions of each sequence (shared + tail)
  int32_t* ws_next;             // item counter, zero at launch (cleared by shared_reset_kernel)
  int B, Hq, Hkv, G, ng;
  int max_blocks, bs, num_blocks;
  int ps_blocks;                // shared partition, blocks
  int pt_tokens;                // tail partition, tokens (a multiple of bs)
  int max_parts;
  int nstage;
  uint32_t tile_bytes;          // one (block, head) tile of K (or V): bs * D * 2
  float qscale;                 // scale * log2(e)
  int bs_shift;                 // log2(bs)
  int ginv;                     // ceil(2^16 / G): row r (< 1024 G) of a group -> member (r * ginv) >> 16
};

// Shared-memory tables every CTA builds (ngE = effective number of groups).
struct Tables {
  int* Ls;      // [B]      clamped context lengths
  int* perm;    // [B]      sequences with tail items, largest item first
  int* preT;    // [B+1]    prefix of tail items over perm's order
  int* preS;    // [ngE+1]  prefix of shared items per group
  int* Sg;      // [ngE]    shared blocks used per group
  int* gsm;     // [ngE+1]  group boundaries
  unsigned char* one;   // [B] 1: the sequence has one partition in all (its rows store the output)
  int ngE;
  int nT;       // sequences in perm
  int nB, nS;   // tail items of the big tails (perm's first ones), shared items
};

struct SItem {
  int s0;          // first sequence of the rows (the group's first member / the tail's sequence)
  int R;           // rows of this item (<= 32)
  int row0;        // first row of this chunk within the group's rows
  int kvh0;        // first KV head
  int bps;         // blocks per stage (1 or 2); heads per stage = 4 / bps
  int nt;          // n-tiles (8 rows each) per warp
  int wh;          // warps per head
  int jb, je, t1;  // blocks [jb, je) of row s0's table; tokens end at t1
  int slot;        // partition slot of this item in each row's sequence
  int shared;      // 1: shared item
  int S;           // the group's shared blocks
  int s1;          // end of the group's sequences (shared items)
};

__device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Partitions of sequence b: shared ones (if its group shares) then tail
// ones; a sequence with nothing to read still has one (it writes zeros).
__device__ __forceinline__ void seq_parts(const SParams& p, int S, int L, int& nsp, int& ntp) {
  nsp = S > 0 ? ceil_div(S, p.ps_blocks) : 0;
  const int tail = L - S * p.bs;
  ntp = tail > 0 ? ceil_div(tail, p.pt_tokens) : (nsp == 0 ? 1 : 0);
}

// Items of one shared partition of a group with R rows per KV head.
__device__ __forceinline__ int shared_items_per_part(const SParams& p, int R) {
  if (R <= 16) return ceil_div(p.Hkv, 4);
  return ceil_div(R, 32) * ceil_div(p.Hkv, 2);
}

// Block-wide exclusive scan of arr[0..n) in place (NTH threads, all of the
// block); arr[n] = total.
template <int NTH>
__device__ void block_scan(int* arr, int n, int* wsum) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int per = (n + NTH - 1) / NTH;
  const int i0 = min(n, (int)threadIdx.x * per), i1 = min(n, i0 + per);
  int sum = 0;
  for (int i = i0; i < i1; ++i) sum += arr[i];
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
  for (int i = i0; i < i1; ++i) {
    const int c = arr[i];
    arr[i] = run;
    run += c;
  }
  if (threadIdx.x == NTH - 1) arr[n] = run;
  __syncthreads();
}

// Two block-wide exclusive scans at once (a[0..na), b[0..nb)), in place,
// with a[na] and b[nb] the totals; wsum holds 16 ints.
template <int NTH>
__device__ void block_scan2(int* a, int na, int* b, int nb, int* wsum) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pa = (na + NTH - 1) / NTH, pb = (nb + NTH - 1) / NTH;
  const int a0 = min(na, (int)threadIdx.x * pa), a1 = min(na, a0 + pa);
  const int b0 = min(nb, (int)threadIdx.x * pb), b1 = min(nb, b0 + pb);
  int sa = 0, sb = 0;
  for (int i = a0; i < a1; ++i) sa += a[i];
  for (int i = b0; i < b1; ++i) sb += b[i];
  int ia = sa, ib = sb;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int ya = __shfl_up_sync(0xffffffffu, ia, off);
    const int yb = __shfl_up_sync(0xffffffffu, ib, off);
    if (lane >= off) ia += ya, ib += yb;
  }
  if (lane == 31) wsum[warp] = ia, wsum[8 + warp] = ib;
  __syncthreads();
  int ra = ia - sa, rb = ib - sb;
  for (int w = 0; w < warp; ++w) ra += wsum[w], rb += wsum[8 + w];
  for (int i = a0; i < a1; ++i) {
    const int c = a[i];
    a[i] = ra;
    ra += c;
  }
  for (int i = b0; i < b1; ++i) {
    const int c = b[i];
    b[i] = rb;
    rb += c;
  }
  if (threadIdx.x == NTH - 1) a[na] = ra, b[nb] = rb;
  __syncthreads();
}

// Items of one shared partition of a group with R rows per KV head, and of
// one tail partition (KV heads grouped as the stages hold them).
__device__ __forceinline__ int part_items(const SParams& p, int R, bool shared) {
  return shared ? shared_items_per_part(p, R) : ceil_div(p.Hkv, 4);
}

// Every CTA builds the same tables (all NTH threads take part): the clamped
// lengths, the group descriptor (checked: non-decreasing from 0 to B,
// otherwise every sequence is its own group and PA_DEV_BAD_GROUP is set), the
// shared blocks used per group, the partitions of every sequence (written to
// the workspace by CTA 0 for the merge), item counts and their prefix sums.
// Tail items are ordered by size, largest first (a stable counting sort of
// the sequences on the size of their largest tail item, in kKH buckets per
// class), so the items handed out last are the shortest.  tmp: scratch of
// 3 * B + 2 * kKH * NTH / 32 + 1 ints (the stage ring, unused until the
// first load).  Returns the number of items.
template <int NTH>
__device__ int build_tables(const SParams& p, Tables& t, int* wsum, int* tmp) {
  constexpr int NW = NTH / 32;
  constexpr int NK = 2 * kKH;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Lmax = p.max_blocks * p.bs;
  int* key = tmp;                 // [B] bucket of each sequence (-1: no tail item)
  int* nit = tmp + p.B;           // [B] tail items of each sequence
  int* gid = tmp + 2 * p.B;       // [B] group of each sequence
  int* hist = tmp + 3 * p.B;      // [NK * NW + 1] per (bucket, warp) counts, then offsets
  for (int i = threadIdx.x; i <= NK * NW; i += NTH) hist[i] = 0;
  // One round of global loads for the lengths and the descriptor: each
  // thread issues all of its loads before storing any.
  const int nld = max(p.B, p.ng + 1);
  for (int i0 = 0; i0 < nld; i0 += kLB * NTH) {
    int lv[kLB], gv[kLB], sv[kLB];
#pragma unroll
    for (int k = 0; k < kLB; ++k) {
      const int i = i0 + k * NTH + threadIdx.x;
      lv[k] = i < p.B ? __ldg(&p.context_lens[i]) : 0;
      gv[k] = i <= p.ng ? __ldg(&p.group_start[i]) : 0;
      sv[k] = i < p.ng ? __ldg(&p.shared_blocks[i]) : 0;
    }
#pragma unroll
    for (int k = 0; k < kLB; ++k) {
      const int i = i0 + k * NTH + threadIdx.x;
      if (i < p.B) {
        int L = lv[k];
        if (L < 0 || L > Lmax) {
          if (blockIdx.x == 0) atomicOr(&g_status_shared, PA_DEV_BAD_LEN);
          L = L < 0 ? 0 : Lmax;
        }
        t.Ls[i] = L;
      }
      if (i <= p.ng) t.gsm[i] = gv[k];
      if (i < p.ng) t.Sg[i] = sv[k];
    }
  }
  __syncthreads();
  bool ok = true;
  for (int g = threadIdx.x; g < p.ng; g += NTH) {
    const int a = t.gsm[g], c = t.gsm[g + 1];
    if (a > c || a < 0 || c > p.B) ok = false;
  }
  if (threadIdx.x == 0 && (t.gsm[0] != 0 || t.gsm[p.ng] != p.B)) ok = false;
  const bool valid = __syncthreads_and(ok) != 0;
  if (!valid) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(&g_status_shared, PA_DEV_BAD_GROUP);
    for (int g = threadIdx.x; g <= p.B; g += NTH) t.gsm[g] = g;
    __syncthreads();
  }
  t.ngE = valid ? p.ng : p.B;
  // Items are handed out in three classes, the larger first, so the last
  // ones to start are short: tail items larger than a full shared item
  // (shared_items_per_part's usual two KV heads x ps_blocks blocks), the
  // shared items, then the other tail items.
  const int ipt = part_items(p, p.G, false);
  const int big_tokens = p.ps_blocks * p.bs * 2 / 4;   // a tail item covers 4 KV heads
  const int chunk = (p.B + NW - 1) / NW;               // sequences per warp in the placement pass
  for (int g = threadIdx.x; g < t.ngE; g += NTH) {
    const int s0 = t.gsm[g], s1 = t.gsm[g + 1];
    int S = 0;
    if (valid && s1 - s0 >= 2) {
      S = min(max(t.Sg[g], 0), p.max_blocks);
      for (int b = s0; b < s1; ++b) S = min(S, t.Ls[b] >> p.bs_shift);
    }
    t.Sg[g] = S;
    const int nspg = S > 0 ? ceil_div(S, p.ps_blocks) : 0;
    t.preS[g] = nspg * part_items(p, (s1 - s0) * p.G, true);
    for (int b = s0; b < s1; ++b) gid[b] = g;
  }
  __syncthreads();
  // per-sequence pass by the warp that places the sequence later: its
  // (bucket, warp) counts need no atomics
  const int b0 = warp * chunk, b1 = min(p.B, b0 + chunk);
  for (int base = b0; base < b1; base += 32) {
    const int b = base + lane;
    int d = -1;
    if (b < b1) {
      const int S = t.Sg[gid[b]];
      int nsp, ntp;
      seq_parts(p, S, t.Ls[b], nsp, ntp);
      const int first = min(max(t.Ls[b] - S * p.bs, 0), p.pt_tokens);   // tokens of its largest tail item
      const int kb = min((first + p.bs - 1) >> p.bs_shift, kKH - 1);
      d = ntp > 0 ? (first > big_tokens ? 0 : kKH) + (kKH - 1 - kb) : -1;
      nit[b] = ntp * ipt;
      key[b] = d;
      t.one[b] = nsp + ntp == 1;
      if (blockIdx.x == 0) p.ws_parts[b] = nsp + ntp;
    }
    const unsigned m = __match_any_sync(0xffffffffu, d);
    if (d >= 0 && (m & ((1u << lane) - 1u)) == 0) hist[d * NW + warp] += __popc(m);
    __syncwarp();
  }
  __syncthreads();
  block_scan2<NTH>(hist, NK * NW, t.preS, t.ngE, wsum);
  const int nT = hist[NK * NW];
  const int nbig = hist[kKH * NW];       // sequences in the big-tail buckets
  __syncthreads();
  // placement: warp w walks its sequences in order, so equal buckets keep
  // sequence order and every CTA computes the same permutation
  for (int base = b0; base < b1; base += 32) {
    const int b = base + lane;
    const int d = b < b1 ? key[b] : -1;
    const unsigned m = __match_any_sync(0xffffffffu, d);
    const int rank = __popc(m & ((1u << lane) - 1u));
    int pos = 0;
    if (d >= 0) pos = hist[d * NW + warp] + rank;
    __syncwarp();
    if (d >= 0) {
      t.perm[pos] = b;
      t.preT[pos] = nit[b];
      if (rank == 0) hist[d * NW + warp] += __popc(m);
    }
    __syncwarp();
  }
  __syncthreads();
  block_scan<NTH>(t.preT, nT, wsum);
  t.nT = nT;
  t.nB = t.preT[nbig];
  t.nS = t.preS[t.ngE];
  // the scratch is the stage ring: order these generic writes before the
  // TMA loads that will overwrite it
  fence_proxy_async_smem();
  __syncthreads();
  return t.preT[nT] + t.nS;
}

// Largest index i in [0, n) with a[i] <= x (a non-decreasing, a[0] <= x):
// over a prefix of item counts, the entry that holds item x.
__device__ __forceinline__ int last_le(const int* a, int n, int x) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a[mid] <= x) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Item i -> its description (every role computes the same): big tail
// items [0, nB), shared items [nB, nB + nS), the other tail items after.
__device__ __forceinline__ void s_item(const SParams& p, const Tables& t, int i, SItem& it) {
  int g, r, b = 0, rr = 0;
  const bool shared = i >= t.nB && i < t.nB + t.nS;
  if (shared) {
    r = i - t.nB;
    g = last_le(t.preS, t.ngE, r);      // the group holding shared item r
    r -= t.preS[g];
  } else {
    const int k = i < t.nB ? i : i - t.nS;
    const int j = last_le(t.preT, t.nT, k);   // the sequence holding tail item k
    b = t.perm[j];
    rr = k - t.preT[j];
    g = last_le(t.gsm, t.ngE, b);       // its group
    r = 0;
  }
  const int s0 = t.gsm[g], s1 = t.gsm[g + 1];
  const int S = t.Sg[g];
  it.S = S;
  if (shared) {
    const int R = (s1 - s0) * p.G;
    int nhg, chunks;
    if (R <= 16) {
      it.nt = R <= 8 ? 1 : 2;
      it.wh = 1;
      it.bps = 1;
      nhg = ceil_div(p.Hkv, 4);
      chunks = 1;
    } else {
      it.nt = 2;
      it.wh = 2;
      it.bps = 2;
      nhg = ceil_div(p.Hkv, 2);
      chunks = ceil_div(R, 32);
    }
    const int per = nhg * chunks;
    const int part = r / per, k = r - part * per;
    const int chunk = k / nhg;
    it.kvh0 = (k - chunk * nhg) * (4 / it.bps);
    it.row0 = chunk * 32;
    it.R = min(32, R - it.row0);
    it.s0 = s0;
    it.jb = part * p.ps_blocks;
    it.je = min(S, it.jb + p.ps_blocks);
    it.t1 = it.je * p.bs;
    it.slot = part;
    it.shared = 1;
    it.s1 = s1;
  } else {
    (void)r;
    const int nhg = ceil_div(p.Hkv, 4);
    const int part = rr / nhg;
    it.kvh0 = (rr - part * nhg) * 4;
    const int T0 = S * p.bs + part * p.pt_tokens;
    const int L = t.Ls[b];
    it.t1 = max(T0, min(L, T0 + p.pt_tokens));
    it.jb = T0 >> p.bs_shift;
    it.je = (it.t1 + p.bs - 1) >> p.bs_shift;
    int nsp, ntp;
    seq_parts(p, S, L, nsp, ntp);
    it.slot = nsp + part;
    it.s0 = b;
    it.R = p.G;
    it.row0 = 0;
    it.nt = 1;
    it.wh = 1;
    it.bps = 1;
    it.shared = 0;
    it.s1 = b + 1;
  }
}

// 2^x by the MUFU instruction (flush-to-zero; 2^-inf = +0).
__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The exponent reference of a column moves only when a score exceeds it by
// more than 2^kTau (base-2 units), so most steps need neither the
// cross-lane maximum nor a rescale of the accumulators; weights stay below
// 2^kTau, far inside fp32 and bf16 range.  Any reference gives the same
// normalised result (the online softmax is exact for any choice of m).
constexpr float kTau = 8.f;

// Two 16-token chunks per online-softmax step (1) or one (0; measured faster:
// the pair's extra registers spill at the two-CTA-per-SM budget).
#ifndef PA_SHARED_PAIR
#define PA_SHARED_PAIR 0
#endif

// KB chunks of up to 16 tokens each (one online-softmax step over all of
// them) for NT n-tiles of 8 query rows: S^T = K Q^T with the chunk's tokens as
// the M rows, the column reference check, then O^T += V^T P.  Chunk k: K and
// V tiles at kt[k], vt[k] (128-byte-swizzled 64-column spans of bs rows),
// tokens tb[k] .. tb[k]+15 of the tile, the first valid[k] - tb[k] of them
// real (FULL: all 16).  When fewer than four accumulation chains would run
// (KB * NT < 4), the k-steps alternate between two accumulators so that
// consecutive MMAs do not wait on each other.
template <int D, int NT, int KB, bool FULL>
__device__ __forceinline__ void step_chunks(const uint32_t (&kt)[KB], const uint32_t (&vt)[KB], const int (&tb)[KB],
                                            const int (&valid)[KB], int bs, uint32_t half_bytes, float qscale,
                                            const uint32_t (&qb)[NT][D / 16][2], float (&OT)[D / 16][NT][4],
                                            float (&mh)[NT][2], float (&lh)[NT][2]) {
  constexpr int KS = D / 16;
  constexpr int MT = D / 16;
  constexpr bool SPLIT = KB * NT < 4;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  float St[KB][NT][4];
  float Su[KB][NT][4];            // odd k-steps when SPLIT
#pragma unroll
  for (int k = 0; k < KB; ++k)
#pragma unroll
    for (int n = 0; n < NT; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) St[k][n][e] = Su[k][n][e] = 0.f;
  {
    // K rows as the A fragment: lanes 0-7 tokens tb..+7, chunk 2kk; 8-15
    // tokens tb+8..+15, chunk 2kk; 16-31 the same for chunk 2kk+1.  Tokens
    // tb[k] + r share the swizzle phase of tb[0] + r (tb is a multiple of 16).
    uint32_t krow[KB];
#pragma unroll
    for (int k = 0; k < KB; ++k) {
      const int tt = min(tb[k] + (lane & 7) + (((lane >> 3) & 1) << 3), bs - 1);
      krow[k] = kt[k] + tt * 128;
    }
    const int tsw = (min(tb[0] + (lane & 7) + (((lane >> 3) & 1) << 3), bs - 1)) & 7;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      const int c = 2 * kk + (lane >> 4);
#pragma unroll
      for (int k = 0; k < KB; ++k) {
        uint32_t a[4];
        ldsm_x4(krow[k] + (c >> 3) * half_bytes + (((c & 7) ^ tsw) << 4), a[0], a[1], a[2], a[3]);
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          if (SPLIT && (kk & 1)) mma_bf16_16816(Su[k][n], a, qb[n][kk][0], qb[n][kk][1]);
          else mma_bf16_16816(St[k][n], a, qb[n][kk][0], qb[n][kk][1]);
        }
      }
    }
  }
  uint32_t pb[KB][NT][2];
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    float lmax[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int k = 0; k < KB; ++k) {
      const bool ok0 = FULL || tb[k] + g < valid[k], ok1 = FULL || tb[k] + g + 8 < valid[k];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float v = (SPLIT ? St[k][n][e] + Su[k][n][e] : St[k][n][e]) * qscale;
        St[k][n][e] = FULL ? v : ((e < 2 ? ok0 : ok1) ? v : -INFINITY);
      }
      lmax[0] = fmaxf(lmax[0], fmaxf(St[k][n][0], St[k][n][2]));
      lmax[1] = fmaxf(lmax[1], fmaxf(St[k][n][1], St[k][n][3]));
    }
    const bool need = lmax[0] > mh[n][0] + kTau || lmax[1] > mh[n][1] + kTau;
    if (__any_sync(0xffffffffu, need)) {
      float alpha[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float m_ = lmax[e];
        m_ = fmaxf(m_, __shfl_xor_sync(0xffffffffu, m_, 4));
        m_ = fmaxf(m_, __shfl_xor_sync(0xffffffffu, m_, 8));
        m_ = fmaxf(m_, __shfl_xor_sync(0xffffffffu, m_, 16));
        alpha[e] = 1.f;
        if (m_ > mh[n][e] + kTau) {
          alpha[e] = ex2f(mh[n][e] - m_);        // 0 when there was no reference yet
          mh[n][e] = m_;
          lh[n][e] *= alpha[e];
        }
      }
      if (alpha[0] != 1.f || alpha[1] != 1.f) {
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          OT[m][n][0] *= alpha[0];
          OT[m][n][1] *= alpha[1];
          OT[m][n][2] *= alpha[0];
          OT[m][n][3] *= alpha[1];
        }
      }
    }
    // a column with no reference yet has seen only masked tokens: its
    // weights are 2^-inf = 0 against any finite reference
    const float r0 = mh[n][0] == -INFINITY ? 0.f : mh[n][0];
    const float r1 = mh[n][1] == -INFINITY ? 0.f : mh[n][1];
#pragma unroll
    for (int k = 0; k < KB; ++k) {
      float pw[4];
      pw[0] = ex2f(St[k][n][0] - r0);
      pw[1] = ex2f(St[k][n][1] - r1);
      pw[2] = ex2f(St[k][n][2] - r0);
      pw[3] = ex2f(St[k][n][3] - r1);
      lh[n][0] += pw[0] + pw[2];
      lh[n][1] += pw[1] + pw[3];
      pb[k][n][0] = movmatrix_t(pack_bf16(pw[0], pw[1]));   // tokens 0-7 of the chunk
      pb[k][n][1] = movmatrix_t(pack_bf16(pw[2], pw[3]));   // tokens 8-15
    }
  }
  {
    // V^T as the A fragment (ldmatrix.trans): lanes 0-7 tokens tb..+7 chunk
    // 2m; 8-15 the same tokens, chunk 2m+1; 16-31 tokens tb+8..+15, chunks
    // 2m, 2m+1
    uint32_t vrow[KB];
#pragma unroll
    for (int k = 0; k < KB; ++k) {
      const int tt = min(tb[k] + (lane & 7) + ((lane >> 4) << 3), bs - 1);
      vrow[k] = vt[k] + tt * 128;
    }
    const int tsw = (min(tb[0] + (lane & 7) + ((lane >> 4) << 3), bs - 1)) & 7;
#pragma unroll
    for (int m = 0; m < MT; ++m) {
      const int c = 2 * m + ((lane >> 3) & 1);
#pragma unroll
      for (int k = 0; k < KB; ++k) {
        uint32_t a[4];
        ldsm_x4_t(vrow[k] + (c >> 3) * half_bytes + (((c & 7) ^ tsw) << 4), a[0], a[1], a[2], a[3]);
#pragma unroll
        for (int n = 0; n < NT; ++n) mma_bf16_16816(OT[m][n], a, pb[k][n][0], pb[k][n][1]);
      }
    }
  }
}

// One consumer warp's share of an item: NT n-tiles (8 query rows each) of
// KV head kvh0 + hd over the tiles hd*bps .. hd*bps+bps-1 of every stage.
template <int D, int NT>
__device__ __forceinline__ void run_rows(const SParams& p, const Tables& t, const SItem& it, int hd, int rbase,
                                         bool active, unsigned char* tilesK, unsigned char* tilesV,
                                         uint64_t* full, uint64_t* empty, volatile int* abort_flag,
                                         int& st_idx, uint32_t& st_ph) {
  constexpr int KS = D / 16;     // k-steps of S^T
  constexpr int MT = D / 16;     // M tiles of O^T
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2, tq = lane & 3;
  const int kvh = it.kvh0 + hd;

  // this lane's Q^T column g of each n-tile: row rbase + 8n + g
  uint32_t qb[NT][KS][2];
#pragma unroll
  for (int n = 0; n < NT; ++n) {
    const int rho = rbase + 8 * n + g;
    const bool ok = active && rho < it.R;
    const int gr = it.row0 + rho;
    const int mem = ok ? (gr * p.ginv) >> 16 : 0;
    const int seq = it.s0 + mem;
    const int qh = kvh * p.G + (ok ? gr - mem * p.G : 0);
    const uint32_t* qp = reinterpret_cast<const uint32_t*>(
        static_cast<const unsigned char*>(p.q) + ((size_t)seq * p.Hq + (ok ? qh : 0)) * (D * 2));
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      qb[n][kk][0] = ok ? __ldg(qp + kk * 8 + tq) : 0u;
      qb[n][kk][1] = ok ? __ldg(qp + kk * 8 + 4 + tq) : 0u;
    }
  }
  float OT[MT][NT][4];
#pragma unroll
  for (int m = 0; m < MT; ++m)
#pragma unroll
    for (int n = 0; n < NT; ++n) OT[m][n][0] = OT[m][n][1] = OT[m][n][2] = OT[m][n][3] = 0.f;
  float mh[NT][2], lh[NT][2];
#pragma unroll
  for (int n = 0; n < NT; ++n) mh[n][0] = mh[n][1] = -INFINITY, lh[n][0] = lh[n][1] = 0.f;
  const uint32_t half_bytes = (uint32_t)p.bs * 128u;
  const int cpt = (p.bs + 15) >> 4;     // 16-token chunks per full tile

  const int nstages = ceil_div(it.je - it.jb, it.bps);
  for (int s = 0; s < nstages; ++s) {
    const int st = st_idx;
    const uint32_t ph = st_ph;
    if (++st_idx == p.nstage) {
      st_idx = 0;
      st_ph ^= 1u;
    }
    bool live = __shfl_sync(0xffffffffu, *abort_flag, 0) == 0;
    if (live) {
      const bool late = !mbar_wait(&full[st], ph);
      if (__any_sync(0xffffffffu, late)) {
        live = false;
        if (lane == 0) {
          atomicOr(&g_status_shared, PA_DEV_TIMEOUT);
          *abort_flag = 1;
        }
      }
    }
    if (live && active) {
      const int j0 = it.jb + s * it.bps;
      const int ntile = min(it.bps, it.je - j0);
      const int tile0 = st * kTiles + hd * it.bps;
      // slots past the context may hold anything; P is 0 there, but 0 * NaN
      // is NaN inside the product, so clear those V rows.  Only a tail
      // item's last tile can be partial, and it has one reader.
      const int vlast = min(p.bs, it.t1 - (j0 + ntile - 1) * p.bs);
      if (vlast < p.bs) {
        unsigned char* vt_ptr = tilesV + (size_t)(tile0 + ntile - 1) * p.tile_bytes;
        for (int idx = lane; idx < (p.bs - vlast) * (D / 8); idx += 32) {
          const int tk = vlast + idx / (D / 8), c = idx % (D / 8);
          *reinterpret_cast<uint4*>(vt_ptr + (c >> 3) * half_bytes + tk * 128 + (c & 7) * 16) =
              make_uint4(0u, 0u, 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
      }
      // the stage's chunks of 16 tokens, two per online-softmax step
      const int nch = (ntile - 1) * cpt + ((vlast + 15) >> 4);
      const uint32_t kbase = smem_u32(tilesK + (size_t)tile0 * p.tile_bytes);
      const uint32_t vbase = smem_u32(tilesV + (size_t)tile0 * p.tile_bytes);
      int ci = 0;
      for (; PA_SHARED_PAIR && ci + 1 < nch; ci += 2) {
        uint32_t kt[2], vt[2];
        int tb[2], vd[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          const int kb = (ci + k) / cpt;
          tb[k] = ((ci + k) - kb * cpt) * 16;
          vd[k] = kb == ntile - 1 ? vlast : p.bs;
          kt[k] = kbase + (uint32_t)kb * p.tile_bytes;
          vt[k] = vbase + (uint32_t)kb * p.tile_bytes;
        }
        if (tb[0] + 16 <= vd[0] && tb[1] + 16 <= vd[1])
          step_chunks<D, NT, 2, true>(kt, vt, tb, vd, p.bs, half_bytes, p.qscale, qb, OT, mh, lh);
        else
          step_chunks<D, NT, 2, false>(kt, vt, tb, vd, p.bs, half_bytes, p.qscale, qb, OT, mh, lh);
      }
      for (; ci < nch; ++ci) {
        const int kb = ci / cpt;
        uint32_t kt[1] = {kbase + (uint32_t)kb * p.tile_bytes}, vt[1] = {vbase + (uint32_t)kb * p.tile_bytes};
        int tb[1] = {(ci - kb * cpt) * 16}, vd[1] = {kb == ntile - 1 ? vlast : p.bs};
        if (tb[0] + 16 <= vd[0])
          step_chunks<D, NT, 1, true>(kt, vt, tb, vd, p.bs, half_bytes, p.qscale, qb, OT, mh, lh);
        else
          step_chunks<D, NT, 1, false>(kt, vt, tb, vd, p.bs, half_bytes, p.qscale, qb, OT, mh, lh);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[st]);
  }
  if (!active) return;

  // the column sums are split over the 8 lanes sharing tq
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      lh[n][e] += __shfl_xor_sync(0xffffffffu, lh[n][e], 4);
      lh[n][e] += __shfl_xor_sync(0xffffffffu, lh[n][e], 8);
      lh[n][e] += __shfl_xor_sync(0xffffffffu, lh[n][e], 16);
    }
#pragma unroll
  for (int n = 0; n < NT; ++n)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int rho = rbase + 8 * n + 2 * tq + e;
      if (rho >= it.R) continue;
      const int gr = it.row0 + rho;
      const int mem = (gr * p.ginv) >> 16;
      const int seq = it.s0 + mem;
      const int qh = kvh * p.G + gr - mem * p.G;
      const size_t bh = (size_t)seq * p.Hq + qh;
      if (t.one[seq]) {
        const float inv = lh[n][e] > 0.f ? 1.f / lh[n][e] : 0.f;
        __nv_bfloat16* o = static_cast<__nv_bfloat16*>(p.out) + bh * D;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          o[16 * m + g] = __float2bfloat16_rn(OT[m][n][e] * inv);
          o[16 * m + 8 + g] = __float2bfloat16_rn(OT[m][n][2 + e] * inv);
        }
      } else {
        const size_t slot = bh * p.max_parts + it.slot;
        float* o = p.ws_o + slot * D;
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          o[16 * m + g] = OT[m][n][e];
          o[16 * m + 8 + g] = OT[m][n][2 + e];
        }
        if (g == 0) {
          p.ws_ml[slot * 2] = mh[n][e];
          p.ws_ml[slot * 2 + 1] = lh[n][e];
        }
      }
    }
}

template <int D>
__global__ void __launch_bounds__(kST, 2)
shared_decode_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
                     const SParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((kAlign - (smem_u32(smem_raw) & (kAlign - 1))) & (kAlign - 1));
  const uint32_t stage_bytes = kTiles * p.tile_bytes;
  unsigned char* tilesK = smem;
  unsigned char* tilesV = smem + (size_t)p.nstage * stage_bytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(tilesV + (size_t)p.nstage * stage_bytes);
  uint64_t* empty = full + p.nstage;
  uint64_t* qfull = empty + p.nstage;                 // [kQ] item queue: index written
  uint64_t* qempty = qfull + kQ;                      // [kQ] item queue: index read by every consumer
  volatile int* abort_flag = reinterpret_cast<volatile int*>(qempty + kQ);
  int* qid = const_cast<int*>(abort_flag) + 4;        // [kQ]
  SItem* qit = reinterpret_cast<SItem*>(qid + kQ);    // [kQ] the items behind qid
  int* wsum = reinterpret_cast<int*>(qit + kQ);       // [16]
  const int ngMax = max(p.ng, p.B);
  Tables t;
  t.Ls = wsum + 16;
  t.perm = t.Ls + p.B;
  t.preT = t.perm + p.B;
  t.gsm = t.preT + p.B + 1;
  t.preS = t.gsm + ngMax + 1;
  t.Sg = t.preS + ngMax + 1;
  t.one = reinterpret_cast<unsigned char*>(t.Sg + ngMax);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the merge kernel (a programmatic dependent on eager calls) may be
  // scheduled now; it waits for this grid's completion before reading
  asm volatile("griddepcontrol.launch_dependents;");
  if (threadIdx.x == 0) {
    for (int s = 0; s < p.nstage; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kSW);
    }
    for (int q = 0; q < kQ; ++q) {
      mbar_init(&qfull[q], 1);
      mbar_init(&qempty[q], kSW);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }

  const int n_items = build_tables<kST>(p, t, wsum, reinterpret_cast<int*>(tilesK));
  // the item counter is cleared by the kernel launched just before this one
  // (this grid may start early on eager calls): wait for it before fetching
  asm volatile("griddepcontrol.wait;" ::: "memory");
  int pend = 0;
  if (warp == kSW && lane == 0) pend = atomicAdd(p.ws_next, 1);

  if (warp == kSW) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&mapK);
      prefetch_tensormap(&mapV);
    }
    const uint64_t pol = policy_evict_first();
    constexpr int HALVES = D * 2 / 128;            // 128-byte column spans per row
    constexpr int OPS = kTiles * 2 * HALVES;       // TMA loads per full stage
    int st_idx = 0;
    uint32_t st_ph = 0;
    uint32_t ucount = 0;                           // stages walked so far
    uint32_t armed_end = 0;                        // 1 + index of the last stage armed
    // Items are taken from the launch-wide counter as this CTA gets to them
    // (the next index is fetched while the current item's loads go out) and
    // passed to the consumers through a queue of kQ slots.
    for (int kq = 0;; ++kq) {
      const int q = kq % kQ;
      // the item is described once here and handed to the consumers with
      // its index
      const int v = __shfl_sync(0xffffffffu, pend < n_items ? pend : -1, 0);
      SItem it;
      if (v >= 0) s_item(p, t, v, it);
      if (lane == 0) {
        if (!*abort_flag && mbar_wait(&qempty[q], ((uint32_t)(kq / kQ) & 1u) ^ 1u)) {
          if (v >= 0) {
            pend = atomicAdd(p.ws_next, 1);
            qit[q] = it;
          }
          qid[q] = v;
          mbar_arrive(&qfull[q]);
        } else if (!*abort_flag) {
          atomicOr(&g_status_shared, PA_DEV_TIMEOUT);
          *abort_flag = 1;
        }
      }
      if (v < 0 || __shfl_sync(0xffffffffu, *abort_flag, 0)) break;
      const int32_t* row = p.block_tables + (size_t)it.s0 * p.max_blocks;
      const int nblk = it.je - it.jb;
      const int nh = 4 / it.bps;
      // A shared item checks that every member's row names the shared blocks
      // it reads through the first member's row (once per group partition).
      const bool check = it.shared && it.kvh0 == 0 && it.row0 == 0;
      for (int j0 = 0; j0 < nblk; j0 += 32) {
        const int n = min(32, nblk - j0);
        int blk = 0;
        if (lane < n) {
          blk = __ldg(&row[it.jb + j0 + lane]);
          if ((unsigned)blk >= (unsigned)p.num_blocks) {
            atomicOr(&g_status_shared, PA_DEV_BAD_BLOCK);
            blk = 0;    // keep every copy inside the pool
          }
        }
        if (check) {
          bool same = true;
          if (lane < n)
            for (int b = it.s0 + 1; b < it.s1; ++b)
              same &= __ldg(&p.block_tables[(size_t)b * p.max_blocks + it.jb + j0 + lane]) ==
                      __ldg(&row[it.jb + j0 + lane]);
          if (!__all_sync(0xffffffffu, same) && lane == 0) atomicOr(&g_status_shared, PA_DEV_BAD_GROUP);
        }
        // stages of this 32-block window: bps blocks each
        for (int i = 0; i < n; i += it.bps) {
          const int st = st_idx;
          const uint32_t ph = st_ph;
          const uint32_t u = ucount++;
          if (++st_idx == p.nstage) {
            st_idx = 0;
            st_ph ^= 1u;
          }
          const int nb = min(it.bps, n - i);        // blocks in this stage
          const int heads = min(nh, p.Hkv - it.kvh0);
          int go = 0;
          if (lane == 0 && !*abort_flag) {
            if (!mbar_wait(&empty[st], ph ^ 1u)) {
              atomicOr(&g_status_shared, PA_DEV_TIMEOUT);
              *abort_flag = 1;
            } else {
              mbar_arrive_expect_tx(&full[st], (uint32_t)(2 * nb * heads) * p.tile_bytes);
              go = 1;
            }
          }
          if (__shfl_sync(0xffffffffu, go, 0)) {
            armed_end = u + 1;
            // lane l: tile l / (2*HALVES), K (even op) or V (odd op), span
            const int tile = lane / (2 * HALVES);
            const int op = lane % (2 * HALVES);
            const int kv = op & 1, hh = op >> 1;
            const int hd = tile / it.bps, kb = tile % it.bps;
            const int bi = __shfl_sync(0xffffffffu, blk, min(i + kb, 31));
            if (lane < OPS && hd < heads && kb < nb) {
              unsigned char* dst = (kv ? tilesV : tilesK) + (size_t)(st * kTiles + tile) * p.tile_bytes +
                                   (size_t)hh * p.bs * 128;
              tma_load_4d(dst, kv ? &mapV : &mapK, &full[st], hh * 64, it.kvh0 + hd, 0, bi, pol);
            }
          }
        }
      }
    }
    // Never leave the CTA with TMA writes into its shared memory in flight:
    // wait (bounded) for the last stages armed.
    if (lane == 0) {
      const uint32_t first = armed_end > (uint32_t)p.nstage ? armed_end - p.nstage : 0u;
      for (uint32_t u = first; u < armed_end; ++u)
        mbar_wait(&full[u % p.nstage], (u / p.nstage) & 1u);
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  int st_idx = 0;
  uint32_t st_ph = 0;
  for (int kq = 0;; ++kq) {
    const int q = kq % kQ;
    bool live = __shfl_sync(0xffffffffu, *abort_flag, 0) == 0;
    if (live) {
      const bool late = !mbar_wait(&qfull[q], (uint32_t)(kq / kQ) & 1u);
      if (__any_sync(0xffffffffu, late)) {
        live = false;
        if (lane == 0) {
          atomicOr(&g_status_shared, PA_DEV_TIMEOUT);
          *abort_flag = 1;
        }
      }
    }
    const int v = live ? qid[q] : -1;
    SItem it;
    if (v >= 0) it = qit[q];
    __syncwarp();
    if (live && lane == 0) mbar_arrive(&qempty[q]);
    if (v < 0) break;
    const int hd = warp / it.wh;
    const int rbase = (warp % it.wh) * 8 * it.nt;
    const bool active = hd < 4 / it.bps && it.kvh0 + hd < p.Hkv && rbase < it.R;
    if (it.nt == 1)
      run_rows<D, 1>(p, t, it, hd, rbase, active, tilesK, tilesV, full, empty, abort_flag, st_idx, st_ph);
    else
      run_rows<D, 2>(p, t, it, hd, rbase, active, tilesK, tilesV, full, empty, abort_flag, st_idx, st_ph);
  }
}

// The merge: out = sum_i 2^(m_i - M) o_i / sum_i 2^(m_i - M) l_i over a
// (sequence, query head) row's partials in slot order, M = max_i m_i.  One
// warp takes kMR rows; every load those rows need for their first kMP
// partials (the sequence's partition count, the (m, l) pairs, the rows of o)
// is issued before any is used, so the warp waits for one round trip to L2;
// partials past kMP (long private tails) follow in a loop.  Lane l holds dims
// l*D/32 .. l*D/32 + D/32 - 1.
constexpr int kMR = 4;
constexpr int kMP = 2;

template <int VPL>
__device__ __forceinline__ void ld_cg(const float* src, float (&v)[VPL]) {
  if constexpr (VPL == 4) {
    const float4 t = __ldcg(reinterpret_cast<const float4*>(src));
    v[0] = t.x, v[1] = t.y, v[2] = t.z, v[3] = t.w;
  } else {
    const float2 t = __ldcg(reinterpret_cast<const float2*>(src));
    v[0] = t.x, v[1] = t.y;
  }
}

// 128-thread blocks: one fits beside the decode kernel's two CTAs on an SM
// (registers), so on eager calls some are resident before the decode grid
// completes.
constexpr int kMergeThreads = 128;

template <int D>
__global__ void __launch_bounds__(kMergeThreads) shared_merge_kernel(const SParams p) {
  constexpr int VPL = D / 32;
  const long long nrows = (long long)p.B * p.Hq;
  const long long r0 = (((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * kMR;
  const int lane = threadIdx.x & 31;
  if (r0 >= nrows) return;
  // a programmatic dependent of the decode kernel on eager calls: the
  // partition counts and partials are read once that grid has completed
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int sp = min(kMP, p.max_parts);
  int np[kMR];
  float2 ml[kMR];          // lane i < sp: partial i's (m, l)
  float ov[kMR][kMP][VPL];
#pragma unroll
  for (int r = 0; r < kMR; ++r) {
    const bool ok = r0 + r < nrows;
    const long long row = ok ? r0 + r : r0;
    const size_t base = (size_t)row * p.max_parts;
    np[r] = ok ? __ldcg(&p.ws_parts[row / p.Hq]) : 0;
    ml[r] = lane < sp ? __ldcg(reinterpret_cast<const float2*>(p.ws_ml) + base + lane) : make_float2(-INFINITY, 0.f);
#pragma unroll
    for (int i = 0; i < kMP; ++i) {
      if (i < sp) {
        ld_cg<VPL>(p.ws_o + (base + i) * D + lane * VPL, ov[r][i]);
      } else {
#pragma unroll
        for (int k = 0; k < VPL; ++k) ov[r][i][k] = 0.f;
      }
    }
  }
#pragma unroll
  for (int r = 0; r < kMR; ++r) {
    const int n = np[r];
    if (n <= 1) continue;
    const size_t base = (size_t)(r0 + r) * p.max_parts;
    float M = -INFINITY;
#pragma unroll
    for (int i = 0; i < kMP; ++i) {
      const float mi = __shfl_sync(0xffffffffu, ml[r].x, i);
      if (i < n) M = fmaxf(M, mi);
    }
    if (n > kMP) {
      for (int i = kMP + lane; i < n; i += 32) M = fmaxf(M, __ldcg(&p.ws_ml[(base + i) * 2]));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    }
    float den = 0.f, acc[VPL];
#pragma unroll
    for (int k = 0; k < VPL; ++k) acc[k] = 0.f;
#pragma unroll
    for (int i = 0; i < kMP; ++i) {
      const float mi = __shfl_sync(0xffffffffu, ml[r].x, i);
      const float li = __shfl_sync(0xffffffffu, ml[r].y, i);
      if (i < n) {
        const float w = mi == -INFINITY ? 0.f : exp2f(mi - M);
        den = fmaf(w, li, den);
#pragma unroll
        for (int k = 0; k < VPL; ++k) acc[k] = fmaf(w, ov[r][i][k], acc[k]);
      }
    }
    for (int i = kMP; i < n; ++i) {
      const float2 mli = __ldcg(reinterpret_cast<const float2*>(p.ws_ml) + base + i);
      float v[VPL];
      ld_cg<VPL>(p.ws_o + (base + i) * D + lane * VPL, v);
      const float w = mli.x == -INFINITY ? 0.f : exp2f(mli.x - M);
      den = fmaf(w, mli.y, den);
#pragma unroll
      for (int k = 0; k < VPL; ++k) acc[k] = fmaf(w, v[k], acc[k]);
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + (size_t)(r0 + r) * D + lane * VPL;
    if constexpr (VPL == 4) {
      uint2 v;
      v.x = pack_bf16(acc[0] * inv, acc[1] * inv);
      v.y = pack_bf16(acc[2] * inv, acc[3] * inv);
      *reinterpret_cast<uint2*>(out) = v;
    } else {
      *reinterpret_cast<uint32_t*>(out) = pack_bf16(acc[0] * inv, acc[1] * inv);
    }
  }
}

// Clears the launch's item counter.  The decode kernel is its programmatic
// dependent on eager calls: its CTAs become resident and build their tables
// while this runs, and wait for it on the device before their first fetch.
__global__ void __launch_bounds__(32) shared_reset_kernel(int32_t* next) {
  asm volatile("griddepcontrol.launch_dependents;");
  if (threadIdx.x == 0) *next = 0;
}

// ------------------------------------------------------------------ host side

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

std::mutex g_smu;
std::map<std::tuple<const void*, int, int, int, int, int>, CUtensorMap> g_smaps;   // (base, nb, bs, h, d, dev)
std::map<std::tuple<const void*, int, size_t>, int> g_socc;                          // (kernel, dev, smem)

bool shared_map(CUtensorMap* out, const void* base, int nb, int bs, int h, int d, int dev) {
  const auto key = std::make_tuple(base, nb, bs, h, d, dev);
  std::lock_guard<std::mutex> lk(g_smu);
  auto f = g_smaps.find(key);
  if (f != g_smaps.end()) {
    *out = f->second;
    return true;
  }
  const uint64_t dims[4] = {(uint64_t)d, (uint64_t)h, (uint64_t)bs, (uint64_t)nb};
  const uint64_t str[3] = {(uint64_t)d * 2, (uint64_t)h * d * 2, (uint64_t)bs * h * d * 2};
  const uint32_t box[4] = {64, 1, (uint32_t)bs, 1};   // one 128-byte row span of one head
  if (!encode_map(out, base, PA_BF16, 4, dims, str, box, true)) return false;
  if (g_smaps.size() > 64) g_smaps.clear();
  g_smaps[key] = *out;
  return true;
}

int shared_occupancy(const void* kernel, size_t smem, int dev) {
  std::lock_guard<std::mutex> lk(g_smu);
  const auto key = std::make_tuple(kernel, dev, smem);
  auto f = g_socc.find(key);
  if (f != g_socc.end()) return f->second;
  if (!raise_smem_limit(kernel, dev)) return 0;
  int occ = 0;
  if (!ck(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kST, smem),
          "cudaOccupancyMaxActiveBlocksPerMultiprocessor"))
    return 0;
  g_socc[key] = occ;
  return occ;
}

// Automatic shared partition: the largest of 1024, 512, 256 and 128 tokens
// whose shared items, counted as if every group shared its whole longest
// context, number at least half of a grid of two CTAs on each of 152 SMs
// (host arithmetic only, like pa_decode's partition rule).  With tail items
// handed out largest first, long shared items balance against the tails
// and cost fewer items and partials, until a single shared item is a large
// share of a CTA's work.  c5-shaped batches (1024-token prompts, 8 samples,
// ms per call): 64 prompts 0.1073 at 1024 tokens, 0.1168 at 512; 32 prompts
// 0.0841 at 1024, 0.0718 at 512; 16 prompts 0.0709 at 1024, 0.0552 at 512,
// 0.0564 at 256; 8 prompts 0.0473 at 512, 0.0398 at 256, 0.0456 at 128.
constexpr int kSharedRefCtas = 2 * 152;

struct SharedPlan {
  int ps_blocks, pt_tokens, max_parts;
  size_t ml_bytes, o_bytes, parts_bytes;
};

bool shared_eligible(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int block_size, int num_groups,
                     pa_dtype dtype) {
  const int G = num_kv_heads > 0 ? num_heads / num_kv_heads : 0;
  return dtype == PA_BF16 && (head_dim == 64 || head_dim == 128) && block_size >= 8 && G >= 1 && G <= 8 &&
         num_seqs <= kSMaxSeqs && num_groups >= 1 && num_groups <= kSMaxGroups;
}

SharedPlan shared_plan(int num_seqs, int num_heads, int num_kv_heads, int head_dim, int max_blocks, int block_size,
                       int partition_size, int num_groups) {
  SharedPlan pl;
  const int max_ctx = max_blocks * block_size;
  const int G = num_heads / num_kv_heads;
  if (partition_size < 0) {
    pl.ps_blocks = max_blocks;
    pl.pt_tokens = max_ctx;
  } else if (partition_size > 0) {
    pl.ps_blocks = partition_size / block_size;
    pl.pt_tokens = partition_size;
  } else {
    const int ng = num_groups > 0 ? num_groups : 1;
    const int R = (num_seqs + ng - 1) / ng * G;                     // rows of an average group
    const int ipp = R <= 16 ? (num_kv_heads + 3) / 4 : (R + 31) / 32 * ((num_kv_heads + 1) / 2);
    int pst = 128;
    for (int cand = 1024; cand >= 128; cand >>= 1)
      if ((long long)ng * ipp * (max_ctx / cand) >= kSharedRefCtas / 2) {
        pst = cand;
        break;
      }
    pl.ps_blocks = pst / block_size > 0 ? pst / block_size : 1;
    pl.pt_tokens = pa_decode_partition_size(num_seqs, num_heads, num_kv_heads, head_dim, max_blocks, block_size, 0);
  }
  if (pl.pt_tokens > max_ctx) pl.pt_tokens = max_ctx;
  if (pl.ps_blocks > max_blocks) pl.ps_blocks = max_blocks;
  const int minp = pl.ps_blocks * block_size < pl.pt_tokens ? pl.ps_blocks * block_size : pl.pt_tokens;
  // a sequence has at most ceil(x / Ps) + ceil((max_ctx - x) / Pt) partitions
  pl.max_parts = (max_ctx + minp - 1) / minp + 1;
  const size_t rows = (size_t)num_seqs * num_heads * pl.max_parts;
  pl.parts_bytes = ((size_t)(num_seqs + 1) * 4 + 255) / 256 * 256;   // + the item counter
  pl.ml_bytes = (rows * 8 + 255) / 256 * 256;
  pl.o_bytes = rows * head_dim * 4;
  return pl;
}

}  // namespace

unsigned fetch_status_shared() {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_status_shared, sizeof(v)) != cudaSuccess) return 0xffffffffu;
  if (v && cudaMemcpyToSymbol(g_status_shared, &zero, sizeof(zero)) != cudaSuccess) return 0xffffffffu;
  return v;
}

}  // namespace pa

using namespace pa;

extern "C" size_t pa_decode_shared_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                                   int max_blocks_per_seq, int block_size, int partition_size,
                                                   int num_groups) {
  const size_t plain = pa_decode_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                                 block_size, partition_size);
  if (num_seqs <= 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads ||
      max_blocks_per_seq <= 0 || !supported_block_size(block_size) ||
      (partition_size > 0 && partition_size % block_size))
    return plain;
  if (!shared_eligible(num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_groups, PA_BF16)) return plain;
  const SharedPlan pl =
      shared_plan(num_seqs, num_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size, partition_size,
                  num_groups);
  const size_t need = pl.parts_bytes + pl.ml_bytes + pl.o_bytes;
  return need > plain ? need : plain;
}

extern "C" int pa_decode_shared(void* out, const void* query, const void* k_cache, const void* v_cache,
                                const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
                                int num_seqs, const int32_t* group_start, const int32_t* shared_blocks,
                                int num_groups, int num_heads, int num_kv_heads, int head_dim, int block_size,
                                int num_blocks, float scale, int partition_size, void* workspace,
                                size_t workspace_bytes, pa_dtype dtype, void* stream) {
  if (dtype != PA_F32 && dtype != PA_BF16) return PA_ERR_DTYPE;
  if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads ||
      !supported_head_dim(head_dim) || !supported_block_size(block_size) || num_blocks <= 0 ||
      max_blocks_per_seq <= 0 || num_groups < 0)
    return PA_ERR_SHAPE;
  if (partition_size > 0 && partition_size % block_size) return PA_ERR_SHAPE;
  if (num_seqs == 0) return PA_OK;
  if (num_groups > 0 && (!group_start || !shared_blocks)) return PA_ERR_NULL;
  if (!shared_eligible(num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_groups, dtype))
    return pa_decode(out, query, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
                     num_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, partition_size, workspace,
                     workspace_bytes, dtype, stream);
  if (!out || !query || !k_cache || !v_cache || !block_tables || !context_lens) return PA_ERR_NULL;
  if (!aligned16(out) || !aligned16(query) || !aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_ALIGN;
  const SharedPlan pl =
      shared_plan(num_seqs, num_heads, num_kv_heads, head_dim, max_blocks_per_seq, block_size, partition_size,
                  num_groups);
  const size_t need = pa_decode_shared_workspace_bytes(num_seqs, num_heads, num_kv_heads, head_dim,
                                                       max_blocks_per_seq, block_size, partition_size, num_groups);
  if (!workspace || workspace_bytes < need) return PA_ERR_WORKSPACE;
  if (!aligned16(workspace)) return PA_ERR_ALIGN;

  int dev = 0;
  if (!ck(cudaGetDevice(&dev), "cudaGetDevice")) return PA_ERR_CUDA;
  CUtensorMap mapK, mapV;
  if (!shared_map(&mapK, k_cache, num_blocks, block_size, num_kv_heads, head_dim, dev) ||
      !shared_map(&mapV, v_cache, num_blocks, block_size, num_kv_heads, head_dim, dev)) {
    note_host_error("cuTensorMapEncodeTiled failed for the K/V pool");
    return PA_ERR_CUDA;
  }

  SParams prm;
  prm.out = out;
  prm.q = query;
  prm.block_tables = block_tables;
  prm.context_lens = context_lens;
  prm.group_start = group_start;
  prm.shared_blocks = shared_blocks;
  char* ws = static_cast<char*>(workspace);
  prm.ws_parts = reinterpret_cast<int32_t*>(ws);
  prm.ws_next = prm.ws_parts + num_seqs;
  prm.ws_ml = reinterpret_cast<float*>(ws + pl.parts_bytes);
  prm.ws_o = reinterpret_cast<float*>(ws + pl.parts_bytes + pl.ml_bytes);
  prm.B = num_seqs;
  prm.Hq = num_heads;
  prm.Hkv = num_kv_heads;
  prm.G = num_heads / num_kv_heads;
  prm.ng = num_groups;
  prm.max_blocks = max_blocks_per_seq;
  prm.bs = block_size;
  prm.num_blocks = num_blocks;
  prm.ps_blocks = pl.ps_blocks;
  prm.pt_tokens = pl.pt_tokens;
  prm.max_parts = pl.max_parts;
  prm.tile_bytes = (uint32_t)(block_size * head_dim * 2);
  prm.qscale = scale * kLog2eS;
  prm.bs_shift = block_size == 4 ? 2 : block_size == 8 ? 3 : block_size == 16 ? 4 : 5;
  prm.ginv = (65536 + prm.G - 1) / prm.G;

  // Stages of four tiles: as many as fit beside
  // the tables for two CTAs per SM (2..6), or, when a stage is so large that
  // two do not fit, one CTA per SM with up to 3.
  // shared memory: stages (K and V tiles), their two mbarriers each, the
  // item queue's 2 x kQ mbarriers, the abort flag (16 bytes), qid[kQ], then
  // the queue's items qit[kQ], then the tables: wsum[16], Ls[B], perm[B],
  // preT[B+1], gsm[ngMax+1], preS[ngMax+1], Sg[ngMax], one[B] (bytes)
  const size_t stage = 2 * (size_t)kTiles * prm.tile_bytes;
  const size_t ngMax = (size_t)(num_groups > num_seqs ? num_groups : num_seqs);
  const size_t tables = 2 * kQ * sizeof(uint64_t) + 16 + 4 * (size_t)kQ + kQ * sizeof(SItem) +
                        4 * (16 + 3 * (size_t)num_seqs + 1 + 3 * ngMax + 2) + ((size_t)num_seqs + 3) / 4 * 4;
  const size_t per_cta = (227 * 1024) / 2 - 1024;
  int ns = (int)((per_cta - tables - kAlign) / (stage + 16));
  if (ns >= 2) {
    if (ns > 6) ns = 6;
  } else {
    ns = (int)((227 * 1024 - tables - kAlign) / (stage + 16));
    if (ns > 3) ns = 3;
    if (ns < 1) return PA_ERR_SHAPE;
  }
  // the table build's scratch lives in the stage ring until the first load
  if ((3 * (size_t)num_seqs + 2 * kKH * (kST / 32) + 1) * 4 > (size_t)ns * stage) return PA_ERR_SHAPE;
  prm.nstage = ns;
  const size_t smem = (size_t)ns * (stage + 2 * sizeof(uint64_t)) + tables + kAlign;

  const void* kern = head_dim == 64 ? reinterpret_cast<const void*>(&shared_decode_kernel<64>)
                                    : reinterpret_cast<const void*>(&shared_decode_kernel<128>);
  const void* merge = head_dim == 64 ? reinterpret_cast<const void*>(&shared_merge_kernel<64>)
                                     : reinterpret_cast<const void*>(&shared_merge_kernel<128>);
  const int occ = shared_occupancy(kern, smem, dev);
  if (occ <= 0) return PA_ERR_CUDA;
  const unsigned grid = (unsigned)(occ * device_sm_count());
  void* rargs[] = {&prm.ws_next};
  if (!ck(cudaLaunchKernel(reinterpret_cast<const void*>(&shared_reset_kernel), dim3(1), dim3(32), rargs, 0,
                           (cudaStream_t)stream),
          "cudaLaunchKernel(shared_reset_kernel)"))
    return PA_ERR_CUDA;
  void* args[] = {&mapK, &mapV, &prm};
  if (!ck(launch_dependent(kern, dim3(grid), dim3(kST), args, smem, (cudaStream_t)stream),
          "cudaLaunchKernel(shared_decode_kernel)"))
    return PA_ERR_CUDA;
  const long long warps = ((long long)num_seqs * num_heads + kMR - 1) / kMR;
  const unsigned blocks = (unsigned)((warps * 32 + kMergeThreads - 1) / kMergeThreads);
  void* margs[] = {&prm};
  if (!ck(launch_after(merge, dim3(blocks), dim3(kMergeThreads), margs, (cudaStream_t)stream),
          "cudaLaunchKernel(shared_merge_kernel)"))
    return PA_ERR_CUDA;
  return PA_OK;
}
