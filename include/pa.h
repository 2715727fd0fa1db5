/*
 * pa.h — C ABI of libpa: paged KV-cache attention kernels for GB300 (sm_103a).
 *
 * The operations are the ones the paged-attention pages describe:
 *
 *   [KVS] "19.2 KV Cache 系统化管理" (paper.xwysyy.cn, llm-fullstack-book):
 *         §19.2.2 block pool / block table, Fig 19-5 block-wise attention,
 *         Fig 19-8 copy-on-write; §19.2.3 the simplified implementation
 *         (pool layout, slot writes, block-table append, paged attention with
 *         an online softmax checked against dense softmax attention);
 *         §19.2.4 KV quantisation (FP8); §19.2.6 swapping blocks to CPU
 *         memory on preemption.
 *   [OS]  "LLM 推理引擎的内存管理与调度：PagedAttention、Prefix Cache 与
 *         Continuous Batching" (zhouzhq2021.github.io): §三 the kernel looks a
 *         logical block up in the block table and forms the physical address
 *         and in-block offset; §四 shared blocks and copy-on-write; §8.1
 *         chunked prefill.
 *
 * Conventions shared by every call
 * --------------------------------
 *  - Pool layout (from [KVS] §19.2.3): k_cache and v_cache are each
 *    [num_blocks, block_size, num_kv_heads, head_dim], row-major, contiguous,
 *    one layer.  Call once per layer for a multi-layer cache.
 *  - Element type: PA_F32 or PA_BF16; K, V, Q and the output share it,
 *    except for the e4m3 pool calls (pa_reshape_and_cache_fp8,
 *    pa_decode_fp8), whose pools hold PA_FP8_E4M3 codes with fp32 scales.
 *    Accumulation is fp32 whatever the storage type (the tensor-core forms
 *    round their product operands as each call's description states); bf16
 *    results are rounded to nearest even.
 *  - Supported sizes: head_dim in {32, 64, 128}; block_size in {4, 8, 16,
 *    32}; num_heads a multiple of num_kv_heads.  Query head h reads KV head
 *    h / (num_heads / num_kv_heads) (grouped-query attention).
 *  - Every pointer argument is a DEVICE pointer unless stated otherwise; the
 *    caller owns all memory and the library allocates nothing per call.
 *    K/V pools, queries and outputs must be 16-byte aligned.
 *  - `stream` is a cudaStream_t (NULL: the legacy default stream).  Every
 *    call only enqueues work on it and returns without synchronising.
 *  - CUDA graphs: every argument the kernels read is a device pointer or a
 *    size, so a captured call replays with whatever the pointed-to buffers
 *    hold at replay time.  The first call with a new combination of sizes
 *    and pool (kernel variant, tensor map) does host-side set-up (function
 *    attributes, occupancy query, tensor-map encoding, cached afterwards):
 *    make one call outside the capture first.
 *  - Return value: 0 on success, or a negative PA_ERR_* code when the host
 *    side rejects the arguments — in that case nothing was launched.
 *  - Conditions only the device can see (a block id outside the pool, a slot
 *    outside the pool, a context longer than its block-table row, a
 *    pipeline wait that ran out) never trap: the affected item is skipped or
 *    zero-filled and a bit is OR-ed into a sticky device word that
 *    pa_last_error() returns and clears.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* PA_FP8_E4M3 is a storage type for K/V pools only: 8-bit e4m3 codes (4
 * exponent bits with bias 7, 3 mantissa bits, largest finite value 448)
 * with one fp32 scale per token for its K vector and one for its V vector.
 * See pa_reshape_and_cache_fp8 and pa_decode_fp8. */
typedef enum { PA_F32 = 0, PA_BF16 = 1, PA_FP8_E4M3 = 2 } pa_dtype;

/* host-detected errors (negative return values) */
#define PA_OK             0
#define PA_ERR_NULL      (-1) /* a required pointer is NULL */
#define PA_ERR_SHAPE     (-2) /* unsupported or inconsistent sizes */
#define PA_ERR_DTYPE     (-3) /* unknown pa_dtype */
#define PA_ERR_ALIGN     (-4) /* a K/V/Q/out pointer is not 16-byte aligned */
#define PA_ERR_WORKSPACE (-5) /* workspace missing or smaller than needed */
#define PA_ERR_CUDA      (-6) /* a CUDA runtime call failed (launch, attributes) */

/* device-detected conditions (bits of pa_last_error()'s positive result) */
#define PA_DEV_BAD_BLOCK  1u  /* block-table entry or pair id outside [0, num_blocks) */
#define PA_DEV_BAD_SLOT   2u  /* slot_mapping entry >= num_blocks * block_size */
#define PA_DEV_BAD_LEN    4u  /* context length < 0 or > max_blocks_per_seq * block_size */
#define PA_DEV_TIMEOUT    8u  /* a shared-memory pipeline wait exceeded its time limit */
#define PA_DEV_BAD_GROUP 16u  /* pa_decode_shared: a group descriptor that does not cover the batch,
                                or a member whose row does not hold its group's shared blocks */

/*
 * KV append ("reshape_and_cache").  [KVS] §19.2.3: a new token's key and
 * value are written into a slot of a physical block; the slot comes from the
 * block table (logical block = tokens so far / block_size, offset = tokens so
 * far % block_size).  Fig 19-6: decode appends into the partly filled block.
 *
 *   key, value     [num_tokens, num_kv_heads, head_dim]   (read)
 *   slot_mapping   [num_tokens] int64: physical_block * block_size + offset.
 *                  A negative slot is padding and is skipped.  Slots must be
 *                  distinct within one call (duplicates: unspecified winner).
 *   k_cache, v_cache  pool (written only at the addressed slots)
 *
 * Exact byte copy.  A slot >= num_blocks * block_size is skipped and sets
 * PA_DEV_BAD_SLOT.  num_tokens == 0 launches nothing.
 */
int pa_reshape_and_cache(const void* key, const void* value,
                         const int64_t* slot_mapping, int num_tokens,
                         void* k_cache, void* v_cache,
                         int num_blocks, int block_size, int num_kv_heads, int head_dim,
                         pa_dtype dtype, void* stream);

/*
 * Paged decode attention.  [KVS] §19.2.3 / Fig 19-5 and [OS] §三: for each
 * sequence b and query head h (KV head g = h / (num_heads/num_kv_heads)),
 *
 *   out[b,h,:] = sum_{t < L_b} softmax_t(scale * <q[b,h,:], K_b[t,g,:]>) V_b[t,g,:]
 *
 * where token t of sequence b sits in physical block
 * block_tables[b*max_blocks_per_seq + t/block_size] at slot t % block_size,
 * and L_b = context_lens[b] counts the newest token (append it first).
 * Only the valid slots of the last block are read; L_b == 0 gives zeros.
 *
 *   out            [num_seqs, num_heads, head_dim]        (written)
 *   query          [num_seqs, num_heads, head_dim]
 *   block_tables   [num_seqs, max_blocks_per_seq] int32
 *   context_lens   [num_seqs] int32
 *   scale          the pages use 1/sqrt(head_dim)
 *   partition_size split-K partition in tokens: 0 = automatic (256 tokens
 *                  when num_heads == num_kv_heads; 2048 for grouped-query
 *                  attention, unless num_seqs * ceil(num_kv_heads / 4) <
 *                  912, the unsplit work items being fewer than three per
 *                  CTA of the grid: then the largest power of two from
 *                  256 to 2048 not above max_blocks_per_seq * block_size *
 *                  num_seqs * ceil(num_kv_heads / 4) / 2432, or 256), < 0 = never
 *                  split, > 0 = a multiple of block_size.  A sequence longer
 *                  than one partition is processed as independent partitions
 *                  whose (max, sum, unnormalised output) states are merged by
 *                  log-sum-exp in a second kernel (outside stream capture it
 *                  is launched as a programmatic dependent of the first and
 *                  waits for it on the device; inside a capture, a plain
 *                  launch).
 *   workspace      device scratch of at least pa_decode_workspace_bytes()
 *                  with the same sizes (may be NULL when that is 0).  Its
 *                  contents on entry do not matter; calls that share one
 *                  workspace must be ordered (same stream).  Its last 256
 *                  bytes hold a work-item counter: a one-thread kernel clears
 *                  it, then the decode kernel's CTAs take their work items
 *                  from it as they free up (on eager calls the decode kernel
 *                  is that kernel's programmatic dependent and waits for it
 *                  on the device).  Without a workspace (no split needed) the
 *                  items are divided among the CTAs in advance.
 *
 * Output is fp32-accumulated; bf16 output is rounded to nearest even.  With
 * bf16, head_dim 64 or 128, block_size >= 8 and a power-of-two group G >= 2,
 * the G query heads of a KV head are computed together on tensor cores
 * (m16n8k16 bf16 products, fp32 accumulation; P is rounded to bf16 for the
 * P*V product): for G <= 8 the block's tokens are the M rows and the heads
 * the N columns; for G >= 16, subgroups of 16 heads are the M rows.
 * Everything else runs on CUDA cores in fp32.
 */
int pa_decode(void* out, const void* query,
              const void* k_cache, const void* v_cache,
              const int32_t* block_tables, int max_blocks_per_seq,
              const int32_t* context_lens, int num_seqs,
              int num_heads, int num_kv_heads, int head_dim,
              int block_size, int num_blocks, float scale, int partition_size,
              void* workspace, size_t workspace_bytes,
              pa_dtype dtype, void* stream);

/*
 * Paged decode attention for sequences that share prompt blocks.  [KVS]
 * §19.2.2 (Fig 19-8) and §19.2.5, [OS] §四: samples drawn from one prompt
 * (parallel sampling, beam search, a common system prompt) point their
 * block tables at the same physical blocks for the prompt, shared by
 * reference count.  The result is that of pa_decode on the same arguments;
 * the shared blocks' keys and values are read from memory once per group
 * for all of its members' query heads (one dense tensor-core product per
 * (shared block, KV head)) instead of once per member.
 *
 *   group_start    [num_groups + 1] int32, device: group g is sequences
 *                  group_start[g] .. group_start[g+1]-1 (non-decreasing,
 *                  from 0 to num_seqs; a sequence alone is a group of one)
 *   shared_blocks  [num_groups] int32, device: the number of leading
 *                  block-table entries every member of group g holds in
 *                  common.  The shared part used is
 *                    S_g = min(shared_blocks[g], floor(L_b / block_size)
 *                              over the group's members b)
 *                  whole blocks, read through the FIRST member's table row;
 *                  each member's tokens from S_g * block_size on are read
 *                  through its own row.  The two attention states are
 *                  merged by log-sum-exp (exact up to rounding: the online
 *                  softmax is associative).
 *   partition_size 0: automatic: partitions of the shared blocks of 1024,
 *                  512, 256 or 128 tokens, the largest that gives at least
 *                  152 shared items if every group shared its whole longest
 *                  context (host arithmetic on num_seqs, num_groups,
 *                  num_kv_heads and max_blocks_per_seq); the private tails
 *                  as pa_decode's automatic choice;
 *                  > 0: a multiple of block_size used for both; < 0: no
 *                  split of either.
 *   workspace      at least pa_decode_shared_workspace_bytes() with the same
 *                  sizes, 16-byte aligned (PA_ERR_ALIGN otherwise); contents
 *                  on entry do not matter
 *   other arguments as for pa_decode
 *
 * Device-detected conditions (PA_DEV_BAD_GROUP): a descriptor that is not
 * non-decreasing from 0 to num_seqs is ignored (the call computes plain
 * decode); a member whose row differs from the first member's within the
 * shared blocks is flagged and its shared part follows the first member's
 * row.  PA_BF16 with head_dim 64 or 128, block_size >= 8, G =
 * num_heads / num_kv_heads <= 8, num_seqs <= 1024 and 1 <= num_groups <=
 * 1024 run the shared path (tensor cores, m16n8k16 bf16 products with fp32
 * accumulation, P rounded to bf16); other arguments run pa_decode unchanged
 * (same result, no sharing exploited).  On the stream: a one-thread kernel
 * that clears the work-item counter the call keeps in the workspace, the
 * decode kernel (its CTAs take work items from that counter as they free
 * up, larger ones first; private tails largest first) and a merge kernel;
 * on eager calls the last two are launched as programmatic dependents of
 * the kernel before them and wait for it on the device.
 */
int pa_decode_shared(void* out, const void* query,
                     const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, int max_blocks_per_seq,
                     const int32_t* context_lens, int num_seqs,
                     const int32_t* group_start, const int32_t* shared_blocks, int num_groups,
                     int num_heads, int num_kv_heads, int head_dim,
                     int block_size, int num_blocks, float scale, int partition_size,
                     void* workspace, size_t workspace_bytes,
                     pa_dtype dtype, void* stream);

/* Bytes of workspace pa_decode_shared needs for these sizes (never less than
 * pa_decode_workspace_bytes()).  Pure host arithmetic; no CUDA call. */
size_t pa_decode_shared_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                        int max_blocks_per_seq, int block_size, int partition_size,
                                        int num_groups);

/*
 * KV append into an e4m3 pool.  The write of pa_reshape_and_cache, with each
 * token's K vector and V vector ([num_kv_heads, head_dim], every head)
 * quantised on its own ([KVS] §19.2.4: per-token scaled quantisation, FP8
 * at one byte per element).  The formula is not in the extracted page; the
 * reading implemented is absmax scaling onto the e4m3 range:
 *
 *   amax  = max |x| over the token's vector
 *   scale = amax / 448                 (fp32, correctly rounded)
 *   code  = e4m3(x * (448 / amax))     (fp32 product, nearest-even rounding,
 *                                       saturating at +-448)
 *
 * and amax == 0 gives scale 0 and all-zero codes.  A dequantised element is
 * e4m3_value(code) * scale.  Non-finite inputs give unspecified codes.
 *
 *   key, value        [num_tokens, num_kv_heads, head_dim], src_dtype
 *                     PA_BF16 or PA_F32
 *   slot_mapping      as for pa_reshape_and_cache
 *   k_cache, v_cache  e4m3 pools [num_blocks, block_size, num_kv_heads,
 *                     head_dim], one byte per element
 *   k_scale, v_scale  [num_blocks, block_size] fp32 (16-byte aligned): the
 *                     scale of the token in each slot
 */
int pa_reshape_and_cache_fp8(const void* key, const void* value,
                             const int64_t* slot_mapping, int num_tokens,
                             void* k_cache, void* v_cache, float* k_scale, float* v_scale,
                             int num_blocks, int block_size, int num_kv_heads, int head_dim,
                             pa_dtype src_dtype, void* stream);

/*
 * Paged decode attention over an e4m3 pool: the result of pa_decode over
 * the dequantised pool (K = e4m3_value(code) * k_scale[slot], likewise V).
 * The per-token scales are applied exactly in fp32: the K scale multiplies
 * the token's score, the V scale its softmax weight in the P*V sum (the
 * softmax normaliser uses the unscaled weights).  Halves the bytes read per
 * token against bf16 ([KVS] §19.2.4).
 *
 *   query, out        dtype must be PA_BF16
 *   k_cache, v_cache  e4m3 pools; k_scale, v_scale as written by
 *                     pa_reshape_and_cache_fp8 (16-byte aligned)
 *   partition_size    as for pa_decode, but the automatic choice is 512
 *                     tokens when num_heads == num_kv_heads (grouped-query
 *                     attention as for pa_decode); pa_decode_fp8_partition_size
 *                     returns the size used
 *   workspace         pa_decode_workspace_bytes() with the same sizes is
 *                     enough (the automatic partition here is never shorter
 *                     than pa_decode's, so no more partials are written)
 *   other arguments   as for pa_decode
 *
 * Power-of-two query groups (G >= 2; subgroups of 16 above 16) with
 * head_dim 128 and block_size >= 8 run on tensor cores: f16 m16n8k16 products of the exactly converted codes with
 * fp32 accumulation, Q scaled per work item by a power of two into f16
 * range, P carrying the V scale relative to a power-of-two reference (f16,
 * in [0, 1]).  Everything else runs on CUDA cores in fp32.
 */
int pa_decode_fp8(void* out, const void* query,
                  const void* k_cache, const void* v_cache,
                  const float* k_scale, const float* v_scale,
                  const int32_t* block_tables, int max_blocks_per_seq,
                  const int32_t* context_lens, int num_seqs,
                  int num_heads, int num_kv_heads, int head_dim,
                  int block_size, int num_blocks, float scale, int partition_size,
                  void* workspace, size_t workspace_bytes,
                  pa_dtype dtype, void* stream);

/*
 * Swap blocks between two pools (preemption by swapping).  [KVS] §19.2.6:
 * a preempted request's KV cache can be moved out to CPU memory and moved
 * back when GPU memory frees up; [OS] §九 names the same swap-out.  For each
 * pair i, block pairs[2i+1] of the destination pool (dst_k, dst_v) becomes a
 * byte-exact copy of block pairs[2i] of the source pool (src_k, src_v), all
 * slots and heads.  Both pools have the [num_blocks, block_size,
 * num_kv_heads, head_dim] layout; their block counts may differ.
 *
 *   dst_*, src_*  device-accessible addresses: device memory, or page-locked
 *                 host memory the device can address (on GB300 such host
 *                 memory is reached over NVLink-C2C by the copy kernel itself,
 *                 so no staging buffer is needed)
 *   pairs         [num_pairs, 2] int64 (src block, dst block), device memory;
 *                 destination blocks distinct, pools not overlapping
 *
 * A pair naming a block outside its pool is skipped and sets
 * PA_DEV_BAD_BLOCK.  num_pairs == 0 launches nothing.  Shapes and dtypes as
 * for pa_copy_blocks (an e4m3 pool swaps its scale rows by a second call).
 */
int pa_swap_blocks(void* dst_k, void* dst_v, int dst_num_blocks,
                   const void* src_k, const void* src_v, int src_num_blocks,
                   const int64_t* pairs, int num_pairs,
                   int block_size, int num_kv_heads, int head_dim,
                   pa_dtype dtype, void* stream);

/*
 * Decode that allocates nothing and takes no workspace.  This entry point
 * has no counterpart on the paged-attention pages; it exists for callers
 * that cannot allocate device memory at the point of the call — for example
 * a plug-in whose host engine owns every device allocation through its own
 * pool, or a latency-critical path that cannot afford an allocation call
 * that may synchronise the device.
 *
 * Same arguments and result as pa_decode, without workspace: the split-K
 * scratch is a PA_NOALLOC_SCRATCH_BYTES array compiled into the library,
 * held by every device that loads the library until the process exits.
 *  - Sizes whose pa_decode_workspace_bytes() exceeds that limit are rejected
 *    with PA_ERR_WORKSPACE (nothing launched; pa_last_host_error() says how
 *    much was needed).
 *  - The first call on a device looks up the array's device address (with
 *    that device current) and caches it, and so does the first call after
 *    the device's context has changed (e.g. after cudaDeviceReset()); make
 *    such a call before any stream capture.
 *  - Every call on a device shares the one array and it keeps the previous
 *    call's contents: calls whose GPU work overlaps (e.g. on two streams)
 *    race on it and must be ordered by the caller.  Nothing in it needs to
 *    start at zero.
 *  - It calls no cudaMalloc, cudaFree or other allocating routine.
 */
#define PA_NOALLOC_SCRATCH_BYTES (32u * 1024u * 1024u)
int pa_decode_noalloc(void* out, const void* query,
                      const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, int max_blocks_per_seq,
                      const int32_t* context_lens, int num_seqs,
                      int num_heads, int num_kv_heads, int head_dim,
                      int block_size, int num_blocks, float scale, int partition_size,
                      pa_dtype dtype, void* stream);

/* Bytes of workspace pa_decode needs for these sizes (0 when no sequence can
 * span more than one partition).  Pure host arithmetic; no CUDA call. */
size_t pa_decode_workspace_bytes(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                 int max_blocks_per_seq, int block_size, int partition_size);

/* The partition size (tokens) pa_decode will use for these arguments. */
int pa_decode_partition_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                             int max_blocks_per_seq, int block_size, int partition_size);

/* The partition size (tokens) pa_decode_fp8 will use for these arguments. */
int pa_decode_fp8_partition_size(int num_seqs, int num_heads, int num_kv_heads, int head_dim,
                                 int max_blocks_per_seq, int block_size, int partition_size);

/*
 * Copy-on-write block copy.  [KVS] Fig 19-8 and [OS] §四: before a sequence
 * writes into a block that other sequences still share, a new block is
 * allocated and the old contents are copied into it.  For each pair i,
 * block pairs[2i+1] of both k_cache and v_cache becomes a byte-exact copy of
 * block pairs[2i] (all block_size slots, all heads).
 *
 *   pairs   [num_pairs, 2] int64 (src, dst), device memory.  dsts must be
 *           distinct and no dst may be the src of another pair; if they are
 *           not, the contents of the blocks involved are undefined (nothing
 *           is flagged).  A pair whose src equals its dst changes nothing.
 *
 * A pair with an id outside [0, num_blocks) is skipped and sets
 * PA_DEV_BAD_BLOCK.  num_pairs == 0 launches nothing.
 *
 * Pure byte movement, so any dtype (PA_FP8_E4M3 included) and any
 * num_kv_heads, head_dim >= 1 whose block (block_size * num_kv_heads *
 * head_dim * element bytes) is a multiple of 16 bytes.  For an e4m3 pool,
 * copy its scale rows with a second call with the same pairs on
 * (k_scale, v_scale) as an fp32 pool with num_kv_heads = head_dim = 1.
 */
int pa_copy_blocks(void* k_cache, void* v_cache, const int64_t* pairs, int num_pairs,
                   int num_blocks, int block_size, int num_kv_heads, int head_dim,
                   pa_dtype dtype, void* stream);

/*
 * Causal chunked-prefill query tile over the paged cache ([OS] §8.1: a long
 * prompt is processed in chunks, each continuing from the tokens already in
 * the cache).  The tile is the LAST num_queries tokens of each sequence's
 * context, their K/V already appended: query i of sequence b sits at
 * position p = context_lens[b] - num_queries + i and attends to positions
 * 0..p of its paged context (query head h reads KV head h / G).  Rows with
 * p < 0 are written as zeros.
 *
 *   out, query  [num_seqs, num_queries, num_heads, head_dim]
 *   other arguments as for pa_decode.
 *
 * Runs on the tcgen05 tensor cores: PA_BF16, head_dim 128, block_size in
 * {8, 16, 32}, G = num_heads / num_kv_heads in {1, 2, 4, 8, 16}; anything
 * else returns PA_ERR_SHAPE, as does scale <= 0.  P is rounded to bf16 before
 * the P*V product; accumulation is fp32.
 */
int pa_prefill_paged(void* out, const void* query, int num_queries,
                     const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, int max_blocks_per_seq,
                     const int32_t* context_lens, int num_seqs,
                     int num_heads, int num_kv_heads, int head_dim,
                     int block_size, int num_blocks, float scale,
                     pa_dtype dtype, void* stream);

/*
 * Mixed round in one launch: decode requests and prefill chunks together
 * ([OS] §8.1 chunked prefill; §8.2: one round's token budget covers decode
 * tokens, new prefill tokens and chunked-prefill tokens).  Sequence b
 * contributes n_b = query_start[b+1] - query_start[b] query rows, its last
 * n_b tokens (K/V already appended): n_b = 1 for a decode request, the chunk
 * length for a prefill chunk, 0 for a sequence with no work this round.
 * Row i of sequence b sits at position p = context_lens[b] - n_b + i and
 * attends causally to positions 0..p (rows with p < 0 are zeros).
 *
 *   out, query     [total_queries, num_heads, head_dim], rows in sequence
 *                  order: sequence b's rows start at query_start[b]
 *   query_start    [num_seqs + 1] int32, device, non-decreasing, starting
 *                  at 0 and ending at total_queries (a decreasing pair, or
 *                  a start outside 0..total_queries, sets PA_DEV_BAD_LEN
 *                  and that sequence writes nothing)
 *   other arguments as for pa_prefill_paged; num_seqs <= 2048
 *
 * The same tcgen05 kernel as pa_prefill_paged: each (query tile, KV head)
 * is one CTA, tiles of 128 / G query positions; a decode request is a
 * tile with one position.
 */
int pa_prefill_varlen(void* out, const void* query, const int32_t* query_start, int total_queries,
                      const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, int max_blocks_per_seq,
                      const int32_t* context_lens, int num_seqs,
                      int num_heads, int num_kv_heads, int head_dim,
                      int block_size, int num_blocks, float scale,
                      pa_dtype dtype, void* stream);

/* Return the sticky device-detected condition bits (PA_DEV_*) and clear
 * them.  Synchronises the current device; 0 means nothing was detected.
 * Returns PA_ERR_CUDA if the device cannot be read. */
int pa_last_error(void);

/* Text of the last host-side failure on the calling thread (which CUDA call
 * failed and why) after a call returned PA_ERR_CUDA; "" if none yet.  The
 * string is owned by the library and overwritten by the next failure. */
const char* pa_last_host_error(void);

/* Human-readable text for a PA_ERR_* code or a PA_DEV_* bit. */
const char* pa_strerror(int code);

/*
 * Health check of the bounded pipeline waits (a library facility; the pages
 * have no counterpart).  Every mbarrier wait in the decode and prefill
 * kernels gives up after 2 s, sets PA_DEV_TIMEOUT and lets the kernel finish,
 * so a stalled pipeline leaves the CUDA context usable and shows up in
 * pa_last_error().  This call exercises that path on its own: it launches one
 * 32-thread CTA that waits on a shared-memory mbarrier nothing arrives at,
 * giving up after limit_ns nanoseconds (1 .. 2e9).  Once the launch has run,
 * pa_last_error() includes PA_DEV_TIMEOUT.  Asynchronous on `stream`; touches
 * no global memory other than the status bit.  A limit outside the range
 * returns PA_ERR_SHAPE and launches nothing.
 */
int pa_selftest_bounded_wait(unsigned long long limit_ns, void* stream);

/* Library ABI version (major*100 + minor). */
int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
