// pa_prefill.cu — causal chunked-prefill query tile over the paged KV cache,
// on the 5th-generation tensor cores (tcgen05.mma, accumulators in TMEM).
//
// What it computes ("LLM 推理引擎的内存管理与调度…" §8.1, chunked prefill; the
// block-table addressing of its §三 and of "19.2 KV Cache 系统化管理"
// §19.2.3): the last Tq tokens of each sequence's context are the query tile;
// query i sits at position p = L - Tq + i and attends with softmax to the
// keys at positions 0..p of its paged context.  Rows with p < 0 are zeros.
//
// How (GB300), one CTA per (query tile, sequence, KV head):
//  * Rows = 128 (query position, head) pairs that share one KV head: QP =
//    128/G positions x G query heads (GQA packing), so every K/V tile is
//    loaded once for all G heads.  D = 128.
//  * Warp 0 (TMA, K): the Q tile (two 64-column halves, 128-byte swizzle)
//    once, then per 64-key tile the K rows of its physical blocks (box {64,
//    1 head, bs, 1 block} per half) into a 2-stage ring; warp 6 (TMA, V)
//    loads the V rows the same way into a ring of its own.  Lane 0 arms a
//    stage's mbarrier and the tile's loads are issued by parallel lanes (one
//    warp instruction), since one thread issuing them in series was slow.
//    A K stage is free once S of its tile is done, a V stage only after P V.
//  * Warp 1 (MMA): allocates 256 TMEM columns (S buffers at columns 0 and 64,
//    O at 128..255) and issues S_{j+1} = Q K_{j+1}^T (M = 128, N = 64,
//    K = 128: 8 tcgen05.mma) before waiting for P_j, so the next tile's
//    scores are computed while the softmax works on this one; then
//    O += P_j V_j with P read from TMEM (the .kind::f16 form whose A operand
//    is in tensor memory; V is an MN-major shared-memory operand).  Each
//    group of MMAs completes on an mbarrier through tcgen05.commit; MMAs and
//    commits execute in issue order, which is what makes reusing an S
//    buffer (and the P written over it) safe two tiles later.
//  * Warps 2-5 (softmax): one thread per row loads its 64 scores from TMEM
//    once (tcgen05.ld 32x32b) and keeps them in registers, applies the causal
//    mask (diagonal tile only) and scale (base 2), keeps a running max and
//    sum, and writes P = exp2(s - m) (fp32 exponentials) back as packed
//    bf16 over the first 32 columns of the same S buffer (tcgen05.st); at the
//    end it reads O back and divides by the sum.  A full tile's bf16 rows are
//    staged in the Q buffer (free once the last S product has completed) and
//    written by two TMA tile stores; a ragged tile's rows past the
//    sequence's queries belong to the next sequence, so each thread stores
//    its own row there.
//  * 98 KB of shared memory and 224 threads per CTA: two CTAs per SM, so one
//    CTA's softmax overlaps the other's MMAs.
//  * The running max used as the exponent reference only moves when a new
//    maximum exceeds it by more than 2^8; then the row's O is rescaled in
//    TMEM (after the previous P V has completed).  The sum and O always share
//    the same reference, so the final quotient is exact up to rounding.
//  * V rows at keys >= L (the unfilled tail of the last block, or blocks not
//    loaded) are zeroed in shared memory before P V reads them: those slots
//    may hold anything, and 0 * NaN would poison the product.
//  * Every wait is bounded (2 s); a timeout sets PA_DEV_TIMEOUT, the roles
//    wind down, outstanding TMA loads and MMAs are drained, TMEM is freed.
#include "pa_tc.cuh"

namespace pa {
namespace {

__device__ unsigned g_status_prefill;

constexpr int kThreads = 224;          // 7 warps: K loads, MMA, 4 softmax, V loads
constexpr int kRows = 128;             // query rows per tile
constexpr int kKT = 64;                // keys per tile
constexpr int kD = 128;
constexpr uint32_t kQHalf = 16384;     // 128 rows x 64 columns of bf16
constexpr uint32_t kKVHalf = 8192;     // 64 keys x 64 columns of bf16
constexpr uint32_t kOffQ = 0;          // Q: 2 halves x 16 KB
constexpr uint32_t kOffK = 32768;      // K: 2 stages x (2 halves x 8 KB)
constexpr uint32_t kOffV = 65536;      // V: 2 stages x (2 halves x 8 KB)
constexpr uint32_t kOffBar = 98304;
constexpr uint32_t kOffTab = kOffBar + 256;  // ragged batches: tile prefix [B+1] + 8 warp sums
constexpr uint32_t kSmemBytes = kOffTab + 1024;          // + alignment slack (fixed query count)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;   // log2 units
// TMEM columns: S buffers at 0 and 64 (fp32, 64 keys each; P overwrites the
// first 32 columns of its own S buffer as packed bf16), O at 128..255.
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColO = 128;

struct PrefillParams {
  void* out;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const int32_t* query_start;   // ragged batch: [B+1] cumulative query counts; null: Tq each
  int B, Tq, Hq, Hkv, G, QP, n_qt;
  int rows;                     // ragged batch: total query rows
  int max_blocks, bs, num_blocks;
  float qscale;
};

// Ragged batches up to this many sequences: each CTA keeps the prefix of
// query tiles per sequence in shared memory (4 bytes per sequence).
constexpr int kVarlenMaxSeqs = 2048;

// Key tile j uses K/V stage j & 1 and S/P buffer j & 1; each has its own
// barriers.  tcgen05 operations from the MMA thread execute in issue order
// and a commit arrives only when every earlier one has completed, so P_j can
// live in S buffer j & 1 until S_{j+2} (issued after P_j V_j) overwrites it,
// and an S_j completion also proves that P_{j-2} V_{j-2} has completed.
struct Bars {
  uint64_t q, full_k[2], full_v[2], empty_k[2], empty_v[2], s[2], p[2], pv[2], drain;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= kOffTab - kOffBar, "barrier block overlaps the tile table");

// 2^x in fp32 by the MUFU instruction (flush-to-zero; 2^-inf = +0).
__device__ __forceinline__ float ex2_f32(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// max(a, b, c) in one instruction (the three-input form of max.f32).
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Query rows of sequence i in a ragged batch, or -1 when its pair of
// starts is decreasing or leaves [0, rows] (flagged; the sequence is skipped).
__device__ __forceinline__ int seq_queries(const PrefillParams& p, int i) {
  const int a = __ldg(&p.query_start[i]), b = __ldg(&p.query_start[i + 1]);
  return (a >= 0 && b >= a && b <= p.rows) ? b - a : -1;
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
  if (*abort_flag) return false;
  if (mbar_wait(bar, parity)) return true;
  atomicOr(&g_status_prefill, PA_DEV_TIMEOUT);
  *abort_flag = 1;
  return false;
}

__global__ void __launch_bounds__(kThreads, 2)
prefill_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapK,
               const __grid_constant__ CUtensorMap mapV, const __grid_constant__ CUtensorMap mapO,
               const PrefillParams p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  Bars* bars = reinterpret_cast<Bars*>(smem + kOffBar);
  volatile int* abort_flag = &bars->abort;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---------------------------------------------------------------- work item
  // Fixed count: (sequence, KV head, query tile), the longest tile first.  Ragged batch (query_start given): the tiles of all
  // sequences numbered sequence by sequence through a prefix table built by
  // every CTA; CTAs past the last tile have nothing to do.
  int b, kvh, qt, nq, qrow0;
  if (p.query_start == nullptr) {
    // the query tiles of one (sequence, KV head) are neighbours in launch
    // order, so the CTAs running together share K/V in L2 (9 % faster than
    // taking the longest tile of every sequence first)
    const int grp = (int)(blockIdx.x / p.n_qt);
    qt = p.n_qt - 1 - (int)(blockIdx.x % p.n_qt);
    b = grp / p.Hkv;
    kvh = grp % p.Hkv;
    nq = p.Tq;
    qrow0 = b * p.Tq;
  } else {
    int* tpre = reinterpret_cast<int*>(smem + kOffTab);         // [B+1] tile prefix
    int* wsum = tpre + p.B + 1;
    const int per = (p.B + kThreads - 1) / kThreads;
    const int b0 = min(p.B, (int)threadIdx.x * per), b1 = min(p.B, b0 + per);
    int sum = 0;
    for (int i = b0; i < b1; ++i) {
      const int n = seq_queries(p, i);
      if (n < 0 && blockIdx.x == 0) atomicOr(&g_status_prefill, PA_DEV_BAD_LEN);
      sum += n > 0 ? (n + p.QP - 1) / p.QP : 0;
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
    for (int i = b0; i < b1; ++i) {
      tpre[i] = run;
      const int n = seq_queries(p, i);
      run += n > 0 ? (n + p.QP - 1) / p.QP : 0;
    }
    if (threadIdx.x == kThreads - 1) tpre[p.B] = run;
    __syncthreads();
    const int t = (int)(blockIdx.x / p.Hkv);
    kvh = (int)(blockIdx.x % p.Hkv);
    if (t >= tpre[p.B]) return;                     // no tile: nothing allocated yet
    int lo = 0, hi = p.B - 1;                       // the sequence holding tile t
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tpre[mid] <= t) lo = mid;
      else hi = mid - 1;
    }
    b = lo;
    const int ntb = tpre[b + 1] - tpre[b];
    qt = ntb - 1 - (t - tpre[b]);                   // the sequence's longest tile first
    qrow0 = __ldg(&p.query_start[b]);
    nq = seq_queries(p, b);                         // > 0: b holds a tile (bad pairs hold none)
  }
  const int q0 = qt * p.QP;
  int L = __ldg(&p.context_lens[b]);
  const int Lmax = p.max_blocks * p.bs;
  if (L < 0 || L > Lmax) {
    if (threadIdx.x == 0 && qt == p.n_qt - 1 && kvh == 0) atomicOr(&g_status_prefill, PA_DEV_BAD_LEN);
    L = L < 0 ? 0 : Lmax;
  }
  const int pos0 = L - nq + q0;                   // position of the tile's first query
  const int kend = min(L, pos0 + p.QP);           // keys this tile needs: [0, kend)
  const int nt = kend > 0 ? (kend + kKT - 1) / kKT : 0;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q, 1);
    for (int s2 = 0; s2 < 2; ++s2) {
      mbar_init(&bars->full_k[s2], 1);
      mbar_init(&bars->full_v[s2], 1);
      mbar_init(&bars->empty_k[s2], 1);
      mbar_init(&bars->empty_v[s2], 1);
      mbar_init(&bars->s[s2], 1);
      mbar_init(&bars->p[s2], 128);
      mbar_init(&bars->pv[s2], 1);
    }
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
    if (nt > 0) {
      // Q goes out at once (this thread is also the K producer's lane 0):
      // its latency overlaps the TMEM allocation and the CTA barrier.
      // Q as [rows, Hq, D]: rows past the sequence's queries (a ragged tile)
      // belong to the next sequence or are zero-filled past the end; their
      // scores are computed and never written.
      prefetch_tensormap(&mapQ);
      prefetch_tensormap(&mapK);
      mbar_arrive_expect_tx(&bars->q, 2 * kQHalf);
      const uint64_t pol = policy_evict_first();
      tma_load_4d(smem + kOffQ, &mapQ, &bars->q, 0, kvh * p.G, qrow0 + q0, 0, pol);
      tma_load_4d(smem + kOffQ + kQHalf, &mapQ, &bars->q, 64, kvh * p.G, qrow0 + q0, 0, pol);
    }
  }
  // the producers' first block-table entries, read before the CTA barrier
  int blk_first = 0;
  if ((warp == 0 || warp == 6) && nt > 0 && lane < min(kKT / p.bs, (L + p.bs - 1) / p.bs))
    blk_first = __ldg(&p.block_tables[(size_t)b * p.max_blocks + lane]);
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  const uint32_t tO = tmem + kColO;

  if (warp == 0 || warp == 6) {
    // ------------------------------------------------------------ TMA producers
    // Warp 0 loads Q once and then K; warp 6 loads V.  K of tile t can be
    // reloaded once S_{t-2} has completed, V only after P_{t-2} V_{t-2}: with
    // one producer per operand neither waits behind the other's stage.
    const bool is_k = warp == 0;
    int issued_q = 0, issued = 0;
    if (nt > 0) {
      if (lane == 0 && !is_k) prefetch_tensormap(&mapV);
      issued_q = is_k ? 1 : 0;                    // Q went out with the barriers (above)
      const uint64_t pol = policy_evict_last();   // K/V tiles are re-read by other query tiles
      const int32_t* row = p.block_tables + (size_t)b * p.max_blocks;
      const int nbt = kKT / p.bs;
      const uint32_t rows_bytes = (uint32_t)p.bs * 128u;    // one half-box
      uint64_t* full = is_k ? bars->full_k : bars->full_v;
      uint64_t* empty = is_k ? bars->empty_k : bars->empty_v;
      const CUtensorMap* map = is_k ? &mapK : &mapV;
      unsigned char* base = smem + (is_k ? kOffK : kOffV);
      for (int t = 0; t < nt; ++t) {
        const int st = t & 1;
        const uint32_t u = (uint32_t)(t >> 1);
        const int k0 = t * kKT;
        const int nvalid = min(nbt, (L - k0 + p.bs - 1) / p.bs);
        int blk = 0;
        if (lane < nvalid) {
          blk = t == 0 ? blk_first : __ldg(&row[k0 / p.bs + lane]);
          if ((unsigned)blk >= (unsigned)p.num_blocks) {
            if (is_k) atomicOr(&g_status_prefill, PA_DEV_BAD_BLOCK);
            blk = 0;
          }
        }
        bool ok = true;
        if (lane == 0) ok = wait_or_abort(&empty[st], (u & 1u) ^ 1u, abort_flag);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        if (lane == 0) mbar_arrive_expect_tx(&full[st], (uint32_t)nvalid * 2u * rows_bytes);
        __syncwarp();
        // lane jj loads block jj of the tile: one warp instruction per operand half
        if (lane < nvalid) {
          unsigned char* dst = base + st * 2 * kKVHalf + lane * rows_bytes;
          tma_load_4d(dst, map, &full[st], 0, kvh, 0, blk, pol);
          tma_load_4d(dst + kKVHalf, map, &full[st], 64, kvh, 0, blk, pol);
        }
        issued = t + 1;
      }
    }
    // drain: no TMA write may land after the CTA exits
    if (lane == 0) {
      if (issued_q) mbar_wait(&bars->q, 0);
      for (int j = max(0, issued - 2); j < issued; ++j) mbar_wait(&(is_k ? bars->full_k : bars->full_v)[j & 1], (uint32_t)(j >> 1) & 1u);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // S_{j+1} = Q K_{j+1}^T is issued before O += P_j V_j, so the tensor core
    // computes the next scores while the softmax warps work on the current ones.
    if (lane == 0 && nt > 0) {
      constexpr uint32_t idS = idesc_bf16_f32(kRows, kKT, false, false);
      constexpr uint32_t idO = idesc_bf16_f32(kRows, kD, false, true);
      auto issue_s = [&](int j) {
        const uint32_t kb = sbase + kOffK + (j & 1) * 2 * kKVHalf;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          umma_bf16(tmem + (j & 1) * kKT,
                    sdesc_sw128(sbase + kOffQ + (uint32_t)(kk >> 2) * kQHalf + (uint32_t)(kk & 3) * 32u, 16, 1024),
                    sdesc_sw128(kb + (uint32_t)(kk >> 2) * kKVHalf + (uint32_t)(kk & 3) * 32u, 16, 1024), idS,
                    kk > 0 ? 1u : 0u);
        }
        umma_commit(&bars->s[j & 1]);
        umma_commit(&bars->empty_k[j & 1]);    // K_j's stage is free once S_j is done
      };
      if (wait_or_abort(&bars->q, 0, abort_flag) && wait_or_abort(&bars->full_k[0], 0, abort_flag)) {
        tc_fence_after();
        issue_s(0);
        for (int j = 0; j < nt; ++j) {
          const int st = j & 1;
          const uint32_t ph = (uint32_t)(j >> 1) & 1u;
          if (j + 1 < nt) {
            if (!wait_or_abort(&bars->full_k[(j + 1) & 1], (uint32_t)((j + 1) >> 1) & 1u, abort_flag)) break;
            tc_fence_after();
            issue_s(j + 1);
          }
          if (!wait_or_abort(&bars->p[st], ph, abort_flag)) break;
          if (!wait_or_abort(&bars->full_v[st], ph, abort_flag)) break;
          tc_fence_after();
          const uint32_t vb = sbase + kOffV + st * 2 * kKVHalf;
#pragma unroll
          for (int kk = 0; kk < kKT / 16; ++kk) {
            // A = P (bf16 pairs in S buffer st, 8 columns per 16 keys); B = V rows kk*16.., MN-major
            umma_bf16_ts(tO, tmem + st * kKT + kk * 8, sdesc_sw128(vb + (uint32_t)kk * 2048u, kKVHalf, 1024), idO,
                         (j > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(&bars->pv[st]);
          umma_commit(&bars->empty_v[st]);
        }
      }
      // drain: every MMA issued so far has completed before TMEM is freed
      umma_commit(&bars->drain);
      mbar_wait(&bars->drain, 0);
    }
  } else {
    // ------------------------------------------------------------ softmax + epilogue
    const int quarter = warp & 3;                 // TMEM lane quarter of this warp
    const int r = quarter * 32 + lane;            // tile row
    const int qi = r / p.G, hh = r % p.G;
    const int pos = pos0 + qi;
    const bool row_out = (q0 + qi) < nq;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    float m_ref = -INFINITY, lsum = 0.f;
    bool live = true;

    for (int j = 0; j < nt && live; ++j) {
      const int st = j & 1;
      const uint32_t ph = (uint32_t)(j >> 1) & 1u;
      const int k0 = j * kKT;
      bool ok = wait_or_abort(&bars->s[st], ph, abort_flag);
      if (!__all_sync(0xffffffffu, ok)) { live = false; break; }
      tc_fence_after();
      // The row's 64 raw scores (the causal mask only bites on tiles
      // reaching past this row) and their maximum.  Eight independent
      // partial maxima keep the dependency chains short.
      const bool full_tile = k0 + kKT - 1 <= pos;
      float mx8[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx8[i] = -INFINITY;
      uint32_t v[2][32];
      tmem_ld32(tmem + st * kKT + lane_off, v[0]);
      tmem_ld32(tmem + st * kKT + 32 + lane_off, v[1]);
      tmem_ld_wait();
      if (!full_tile) {
#pragma unroll
        for (int c = 0; c < kKT; ++c)
          if (k0 + c > pos) v[c >> 5][c & 31] = __float_as_uint(-INFINITY);
      }
#pragma unroll
      for (int c = 0; c < kKT; c += 2)
        mx8[(c >> 1) & 7] = fmax3(mx8[(c >> 1) & 7], __uint_as_float(v[c >> 5][c & 31]),
                                  __uint_as_float(v[c >> 5][(c + 1) & 31]));
      float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7]));
      mx *= p.qscale;                                     // scale > 0 (checked by the host)
      const bool need = mx > m_ref + kRescaleThreshold;   // false while mx is -inf
      const float alpha = need ? exp2f(m_ref - mx) : 1.f; // m_ref = -inf gives 0
      if (need) m_ref = mx;
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        // O must hold P_{j-1} V_{j-1} before it is rescaled
        ok = wait_or_abort(&bars->pv[(j - 1) & 1], (uint32_t)((j - 1) >> 1) & 1u, abort_flag);
        if (!__all_sync(0xffffffffu, ok)) { live = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {         // 16 columns at a time: the scores stay live
          uint32_t w[16];
          tmem_ld16(tO + lane_off + c * 16, w);
          tmem_ld_wait();
#pragma unroll
          for (int i = 0; i < 16; ++i) w[i] = __float_as_uint(__uint_as_float(w[i]) * alpha);
          tmem_st16(tO + lane_off + c * 16, w);
        }
        tmem_st_wait();
      }
      lsum *= alpha;
      // V rows at keys >= L hold no context: zero them once the tile has landed
      if (r < kKT && k0 + r >= L) {
        ok = wait_or_abort(&bars->full_v[st], ph, abort_flag);
        if (ok) {
          uint4 z = make_uint4(0, 0, 0, 0);
          unsigned char* vrow = smem + kOffV + st * 2 * kKVHalf + r * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            *reinterpret_cast<uint4*>(vrow + c * 16) = z;
            *reinterpret_cast<uint4*>(vrow + kKVHalf + c * 16) = z;
          }
          fence_proxy_async_smem();
        }
      }
      // P = exp2(scale*s - m_ref) as bf16 pairs, written over this S buffer
      // 32 keys at a time (packed column 16h + c holds keys 32h + 2c,
      // 32h + 2c + 1).  The row sum adds the fp32 exponentials; P carries
      // their bf16 rounding (a relative 2^-9 per term, unbiased).
      const float negm = m_ref == -INFINITY ? 0.f : -m_ref;   // all-masked rows: every s is -inf
      const uint64_t qs2 = f2pack(p.qscale, p.qscale), nm2 = f2pack(negm, negm);
      uint64_t ls2[4];                               // eight partial row sums, as four pairs
#pragma unroll
      for (int i = 0; i < 4; ++i) ls2[i] = f2pack(0.f, 0.f);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t pw[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          // exponents as one packed fp32 fma per pair, 2^x in fp32, one bf16
          // pair for the product, one packed add into the sums
          float x0, x1;
          f2unpack(ffma2(f2pack(__uint_as_float(v[hf][2 * c]), __uint_as_float(v[hf][2 * c + 1])), qs2, nm2), x0,
                   x1);
          const float p0 = ex2_f32(x0), p1 = ex2_f32(x1);
          const __nv_bfloat162 pk = __floats2bfloat162_rn(p0, p1);
          ls2[c & 3] = fadd2(ls2[c & 3], f2pack(p0, p1));
          pw[c] = *reinterpret_cast<const uint32_t*>(&pk);
        }
        tmem_st16(tmem + st * kKT + hf * 16 + lane_off, pw);
      }
      float ls8[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) f2unpack(ls2[i], ls8[2 * i], ls8[2 * i + 1]);
      lsum += ((ls8[0] + ls8[1]) + (ls8[2] + ls8[3])) + ((ls8[4] + ls8[5]) + (ls8[6] + ls8[7]));
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&bars->p[st]);
    }

    // epilogue: O / l -> bf16 rows
    bool have = nt > 0 && live;
    if (have) {
      const bool ok = wait_or_abort(&bars->pv[(nt - 1) & 1], (uint32_t)((nt - 1) >> 1) & 1u, abort_flag);
      have = __all_sync(0xffffffffu, ok);
      tc_fence_after();
    }
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    if (nt > 0 && q0 + p.QP <= nq) {
      // A full tile: O / l as bf16 rows staged in the Q buffer (its last
      // reader, S_{nt-1}, completed before P_{nt-1} V_{nt-1}) in the
      // 128-byte-swizzled layout of the tile's TMA box, then two TMA stores.
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        if (have) {
          tmem_ld32(tO + lane_off + c * 32, v);
          tmem_ld_wait();
        }
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float a0 = have ? __uint_as_float(v[g * 8 + 2 * e]) * inv : 0.f;
            const float a1 = have ? __uint_as_float(v[g * 8 + 2 * e + 1]) * inv : 0.f;
            const __nv_bfloat162 pk = __floats2bfloat162_rn(a0, a1);
            w[e] = *reinterpret_cast<const uint32_t*>(&pk);
          }
          const int ch = c * 4 + g;                 // 16-byte chunk of the row, 0..15
          *reinterpret_cast<uint4*>(smem + kOffQ + (ch >> 3) * kQHalf + r * 128 + (((ch & 7) ^ (r & 7)) << 4)) =
              make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
      fence_proxy_async_smem();
      named_sync(1, 128);
      if (warp == 2 && lane == 0) {
        tma_store_4d(&mapO, smem + kOffQ, 0, kvh * p.G, qrow0 + q0, 0);
        tma_store_4d(&mapO, smem + kOffQ + kQHalf, 64, kvh * p.G, qrow0 + q0, 0);
        bulk_commit();
        bulk_wait_all();
      }
    } else {
      unsigned char* orow = static_cast<unsigned char*>(p.out) +
                            (((size_t)qrow0 + q0 + qi) * p.Hq + (size_t)kvh * p.G + hh) * (kD * 2);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t v[32];
        if (have) {
          tmem_ld32(tO + lane_off + c * 32, v);
          tmem_ld_wait();
        }
        if (row_out) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float a0 = have ? __uint_as_float(v[g * 8 + 2 * e]) * inv : 0.f;
              const float a1 = have ? __uint_as_float(v[g * 8 + 2 * e + 1]) * inv : 0.f;
              const __nv_bfloat162 pk = __floats2bfloat162_rn(a0, a1);
              w[e] = *reinterpret_cast<const uint32_t*>(&pk);
            }
            st_v4(orow + (c * 32 + g * 8) * 2, make_uint4(w[0], w[1], w[2], w[3]));
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

unsigned fetch_status_prefill() {
  unsigned v = 0, zero = 0;
  if (cudaMemcpyFromSymbol(&v, g_status_prefill, sizeof(v)) != cudaSuccess) return 0xffffffffu;
  if (v && cudaMemcpyToSymbol(g_status_prefill, &zero, sizeof(zero)) != cudaSuccess) return 0xffffffffu;
  return v;
}

}  // namespace pa

using namespace pa;

// Shared by pa_prefill_paged (query_start null: num_queries per sequence)
// and pa_prefill_varlen (query_start [B+1]; rows = total query rows).
static int prefill_impl(void* out, const void* query, const int32_t* query_start, int num_queries, int rows,
                        const void* k_cache, const void* v_cache, const int32_t* block_tables,
                        int max_blocks_per_seq, const int32_t* context_lens, int num_seqs, int num_heads,
                        int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
                        pa_dtype dtype, void* stream) {
  if (dtype != PA_F32 && dtype != PA_BF16) return PA_ERR_DTYPE;
  if (dtype != PA_BF16 || head_dim != 128) return PA_ERR_SHAPE;
  if (num_seqs < 0 || num_queries < 0 || rows < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
      num_heads % num_kv_heads || num_blocks <= 0 || max_blocks_per_seq <= 0 ||
      !(block_size == 8 || block_size == 16 || block_size == 32))
    return PA_ERR_SHAPE;
  if (query_start && num_seqs > kVarlenMaxSeqs) return PA_ERR_SHAPE;
  const int G = num_heads / num_kv_heads;
  if (G > 16 || (128 % G) != 0 || !(scale > 0.f)) return PA_ERR_SHAPE;
  if (num_seqs == 0 || rows == 0) return PA_OK;
  if (!out || !query || !k_cache || !v_cache || !block_tables || !context_lens) return PA_ERR_NULL;
  if (!aligned16(out) || !aligned16(query) || !aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_ALIGN;

  const int QP = 128 / G;
  CUtensorMap mapQ, mapK, mapV, mapO;
  {
    // queries as [rows, Hq, D] (one more unit dimension for the 4-D copy)
    const uint64_t dims[4] = {128, (uint64_t)num_heads, (uint64_t)rows, 1};
    const uint64_t str[3] = {256, (uint64_t)num_heads * 256, (uint64_t)rows * num_heads * 256};
    const uint32_t box[4] = {64, (uint32_t)G, (uint32_t)QP, 1};
    if (!encode_map(&mapQ, query, PA_BF16, 4, dims, str, box, true)) {
      note_host_error("cuTensorMapEncodeTiled failed for the query tile");
      return PA_ERR_CUDA;
    }
    // the output as the same [rows, Hq, D] view, written one full tile per store
    if (!encode_map(&mapO, out, PA_BF16, 4, dims, str, box, true)) {
      note_host_error("cuTensorMapEncodeTiled failed for the output tile");
      return PA_ERR_CUDA;
    }
  }
  {
    const uint64_t dims[4] = {128, (uint64_t)num_kv_heads, (uint64_t)block_size, (uint64_t)num_blocks};
    const uint64_t str[3] = {256, (uint64_t)num_kv_heads * 256, (uint64_t)block_size * num_kv_heads * 256};
    const uint32_t box[4] = {64, 1, (uint32_t)block_size, 1};
    if (!encode_map(&mapK, k_cache, PA_BF16, 4, dims, str, box, true) ||
        !encode_map(&mapV, v_cache, PA_BF16, 4, dims, str, box, true)) {
      note_host_error("cuTensorMapEncodeTiled failed for the K/V pool");
      return PA_ERR_CUDA;
    }
  }
  int dev = 0;
  if (!ck(cudaGetDevice(&dev), "cudaGetDevice")) return PA_ERR_CUDA;
  if (!raise_smem_limit(reinterpret_cast<const void*>(&prefill_kernel), dev)) return PA_ERR_CUDA;

  PrefillParams prm;
  prm.out = out;
  prm.block_tables = block_tables;
  prm.context_lens = context_lens;
  prm.query_start = query_start;
  prm.B = num_seqs;
  prm.Tq = num_queries;
  prm.Hq = num_heads;
  prm.Hkv = num_kv_heads;
  prm.G = G;
  prm.QP = QP;
  prm.n_qt = (num_queries + QP - 1) / QP;
  prm.rows = rows;
  prm.max_blocks = max_blocks_per_seq;
  prm.bs = block_size;
  prm.num_blocks = num_blocks;
  prm.qscale = scale * kLog2e;
  // ragged: at most ceil(rows/QP) + B query tiles in all
  const long long tiles = query_start ? (long long)(rows + QP - 1) / QP + num_seqs
                                      : (long long)prm.n_qt * num_seqs;
  const long long grid = tiles * num_kv_heads;
  const size_t smem = kSmemBytes + (query_start ? 4 * ((size_t)num_seqs + 1 + 8) : 0);
  void* args[] = {&mapQ, &mapK, &mapV, &mapO, &prm};
  if (!ck(cudaLaunchKernel(reinterpret_cast<const void*>(&prefill_kernel), dim3((unsigned)grid), dim3(kThreads),
                           args, smem, (cudaStream_t)stream),
          "cudaLaunchKernel(prefill_kernel)"))
    return PA_ERR_CUDA;
  return PA_OK;
}

extern "C" int pa_prefill_paged(void* out, const void* query, int num_queries, const void* k_cache,
                                const void* v_cache, const int32_t* block_tables, int max_blocks_per_seq,
                                const int32_t* context_lens, int num_seqs, int num_heads, int num_kv_heads,
                                int head_dim, int block_size, int num_blocks, float scale, pa_dtype dtype,
                                void* stream) {
  if (num_seqs < 0 || num_queries < 0 || (long long)num_seqs * num_queries > 0x7fffffffll) return PA_ERR_SHAPE;
  return prefill_impl(out, query, nullptr, num_queries, num_seqs * num_queries, k_cache, v_cache, block_tables,
                      max_blocks_per_seq, context_lens, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                      num_blocks, scale, dtype, stream);
}

extern "C" int pa_prefill_varlen(void* out, const void* query, const int32_t* query_start, int total_queries,
                                 const void* k_cache, const void* v_cache, const int32_t* block_tables,
                                 int max_blocks_per_seq, const int32_t* context_lens, int num_seqs, int num_heads,
                                 int num_kv_heads, int head_dim, int block_size, int num_blocks, float scale,
                                 pa_dtype dtype, void* stream) {
  if (num_seqs > 0 && total_queries > 0 && !query_start) return PA_ERR_NULL;
  return prefill_impl(out, query, query_start, 0, total_queries, k_cache, v_cache, block_tables,
                      max_blocks_per_seq, context_lens, num_seqs, num_heads, num_kv_heads, head_dim, block_size,
                      num_blocks, scale, dtype, stream);
}
