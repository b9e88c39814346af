/*
 * pa.h — C ABI of the paged KV-cache decode library (libpagedattn.so).
 *
 * What the calls compute comes from two web pages on PagedAttention:
 *   [Z]  zenaique, "How does PagedAttention enable prefix sharing across
 *        requests and what data structure makes it cheap?" (answer text;
 *        "Most common mistake"; interviewer follow-ups)
 *   [K]  kgptalkie, "Day 28: PagedAttention / vLLM" (sections named below)
 *
 * Conventions for every call
 *   - Return value: PA_OK (0) on success, a negative PA_ERR_* code otherwise.
 *     Errors a host check can see are returned at once and nothing is
 *     launched.  Errors only the GPU can see (a block id or slot outside the
 *     pool) make the kernel skip the offending access and record the first
 *     such code in the pool's device error word; pa_get_error reports it.
 *     No call traps or aborts.
 *   - Device pointers: every tensor argument marked "device" is GPU memory
 *     owned by the caller, on the device the pool was created on.  The
 *     library never frees caller memory.
 *   - Streams: `stream` is a cudaStream_t passed as void*.  NULL means the
 *     legacy default stream.  Every GPU call is asynchronous on it.
 *   - CUDA graphs: once the pool's workspace holds the batch (a first call of
 *     the same shape, or pa_decode_reserve), pa_append_kv, pa_copy_blocks,
 *     pa_decode, pa_append_decode, pa_decode_noalloc and pa_prefill only
 *     launch kernels on `stream`, so they may be captured into a graph and
 *     replayed.  pa_decode_shared uploads its group description with a
 *     pageable copy when the description changes, pa_get_error synchronises:
 *     keep those two out of a capture.
 *
 * Pool layout (owned by the pool, created zeroed):
 *   K: [num_blocks][kv_heads][block_size][head_dim]   keys, one row per token
 *   V: [num_blocks][kv_heads][head_dim][block_size]   values, transposed inside
 *                                                      each (block, head) tile
 *   Each (block, head) tile of K and of V is block_size * head_dim elements,
 *   contiguous (4 KiB at block_size 16, head_dim 128, bf16).  Values are
 *   stored transposed so the decode kernel loads them directly as
 *   tensor-core operand fragments.  A slot is physical_block * block_size +
 *   offset ([K] "Follow One Token Address"); a negative slot means "skip".
 */
#ifndef PAGED_KV_CACHE_PA_H
#define PAGED_KV_CACHE_PA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct pa_pool pa_pool;
typedef struct pa_bm pa_bm;

/* Element type of the pool, of q/k/v inputs and (for out) of the output.
 * PA_FP8E4M3 is a pool type only ([K] "Split the Cache Into Fixed Blocks": a
 * block's bytes depend on the dtype): each key and value element is one e4m3
 * byte (sign, 4 exponent bits with bias 7, 3 mantissa bits, no infinity,
 * largest magnitude 448) standing for code * the pool's K or V scale.  Such a
 * pool takes bf16 k/v to append and bf16 queries, quantizing on the GPU:
 * code = e4m3(fl32(x / scale)), to nearest, ties to even, beyond 448
 * saturating to 448. */
typedef enum { PA_F32 = 0, PA_BF16 = 1, PA_FP8E4M3 = 2 } pa_dtype;

enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = -1,     /* a size, pointer or enum out of range */
    PA_ERR_DTYPE = -2,           /* unsupported dtype combination */
    PA_ERR_CUDA = -3,            /* a CUDA runtime call failed */
    PA_ERR_NO_FREE_BLOCK = -4,   /* the free pool is empty */
    PA_ERR_BAD_BLOCK_ID = -5,    /* (device) block id outside [0, num_blocks) */
    PA_ERR_BAD_SLOT = -6,        /* (device) slot outside the pool */
    PA_ERR_REFCOUNT = -7,        /* reference count would go below zero */
    PA_ERR_UNKNOWN_REQUEST = -8, /* request id not live in the block manager */
    PA_ERR_OUT_OF_MEMORY = -9,   /* host or device allocation failed */
    PA_ERR_UNSUPPORTED = -10,    /* shape outside what the kernels handle */
    PA_ERR_OVERLAP = -11,        /* (device) a copy pair's block is also used by
                                    another pair of the same call */
    PA_ERR_BAD_LENGTH = -12      /* (device) context length beyond the table */
};

/* ---------------------------------------------------------------- pool --- */

/* Create a KV pool of `num_blocks` physical blocks of `block_size` token
 * positions each, for `kv_heads` heads of width `head_dim` ([K] "Split the
 * Cache Into Fixed Blocks": every block has room for the same number of token
 * positions, and its size in bytes follows from the heads, the head width and
 * the element type).  One pool holds one layer.
 * Allocates and zeroes K and V on the current CUDA device (synchronously).
 * Limits: block_size in [1, 1024]; head_dim in [4, 256], a multiple of 4;
 * kv_heads >= 1.
 * On success *out owns the pool; release it with pa_pool_destroy. */
int pa_pool_create(int num_blocks, int block_size, int kv_heads, int head_dim,
                   pa_dtype dtype, pa_pool **out);

/* Free the pool, its device arrays and its decode workspace.  NULL is a no-op. */
int pa_pool_destroy(pa_pool *pool);

/* Device addresses of the pool's K and V arrays (layout above), for tests
 * and for callers that fill the cache themselves.  Either may be NULL. */
int pa_pool_kv_ptrs(pa_pool *pool, void **k, void **v);

/* Copy the whole pool out to (export) or in from (import) caller buffers of
 * the pool's layout and size (num_blocks * kv_heads * block_size * head_dim
 * elements each), device or host memory, asynchronously on `stream`.  For
 * snapshots and tests; not on the decode path. */
int pa_pool_export(pa_pool *pool, void *k_dst, void *v_dst, void *stream);
int pa_pool_import(pa_pool *pool, const void *k_src, const void *v_src, void *stream);

/* Geometry of the pool: any output pointer may be NULL. */
int pa_pool_info(const pa_pool *pool, int *num_blocks, int *block_size, int *kv_heads,
                 int *head_dim, int *dtype);

/* Scales of a PA_FP8E4M3 pool: a K code c stands for e4m3(c) * k_scale, a V
 * code for e4m3(c) * v_scale (both 1.0 at creation).  Appends quantize with the
 * scales current at the call and decodes dequantize with those current at
 * theirs, so set them before the first append.  Both must be finite and > 0
 * (else PA_ERR_INVALID_ARG); another pool type gives PA_ERR_DTYPE.  Host only. */
int pa_pool_set_kv_scales(pa_pool *pool, float k_scale, float v_scale);
int pa_pool_kv_scales(const pa_pool *pool, float *k_scale, float *v_scale);

/* Kernel-choice options of a pool.  The library reads no environment
 * variables: every choice that is not automatic is set here, explicitly, by
 * the caller (host only; it applies from the next call on this pool).  All
 * options select among kernels that compute the same result within the
 * stated tolerances; none changes what is computed.
 *   PA_OPT_PARTITION_CAP   decode partitions of at most `value` tokens
 *                          (rounded down to a multiple of block_size, never
 *                          below the smallest partition); 0 = no cap;
 *                          -1 (default) = automatic: 2048 tokens when the
 *                          batch has more sequences than the GPU has SMs,
 *                          else no cap.
 *   PA_OPT_SHARED_KERNEL   shared-prefix items of pa_decode_shared: 0
 *                          (default) = the tcgen05 kernel where the shape
 *                          allows it, 1 = the mma.sync form.
 *   PA_OPT_PREFILL_KERNEL  pa_prefill: 0 (default) = the tcgen05 kernel where
 *                          the shape allows it, 1 = the mma.sync form.
 * An unknown option or a value out of range returns PA_ERR_INVALID_ARG and
 * changes nothing. */
typedef enum {
    PA_OPT_PARTITION_CAP = 0,
    PA_OPT_SHARED_KERNEL = 1,
    PA_OPT_PREFILL_KERNEL = 2
} pa_option;
int pa_pool_set_option(pa_pool *pool, pa_option option, int value);
int pa_pool_get_option(const pa_pool *pool, pa_option option, int *value);

/* Write each new token's keys and values into its slot ([Z] answer: the new
 * token's data goes into the slot its request was given; [K] "Growth Needs
 * Only Another Free Block").
 *   k, v          device [T][kv_heads][head_dim], pool dtype (bf16 for an fp8 pool),
 *                 row-major
 *   slot_mapping  device int64 [T]; slot = block * block_size + offset;
 *                 negative = skip; >= num_blocks * block_size records
 *                 PA_ERR_BAD_SLOT and is skipped
 * Slots of one call must be distinct (the host block manager guarantees it);
 * two tokens aimed at one slot leave either one's data.  T == 0 is a no-op. */
int pa_append_kv(pa_pool *pool, const void *k, const void *v, const int64_t *slot_mapping,
                 int num_tokens, void *stream);

/* Copy-on-write block copies ([K] "Shared Blocks Must Not Be Changed in
 * Place": a private copy of the shared block is made before the diverging
 * write; [Z] "Most common mistake": the copy is limited to the one block
 * where the requests diverge).
 *   pairs  device int64 [P][2] = (src, dst); each copies all kv_heads x
 *          block_size x head_dim elements of K and of V, bit for bit.
 * A pair whose block id is outside the pool records PA_ERR_BAD_BLOCK_ID; a
 * pair whose dst equals its own src, or whose src or dst is another pair's
 * dst (or whose dst is another pair's src), records PA_ERR_OVERLAP; such
 * pairs copy nothing, the others proceed.  Issue it before the appends into
 * the copied blocks on the same stream.  P == 0 is a no-op. */
int pa_copy_blocks(pa_pool *pool, const int64_t *pairs, int num_pairs, void *stream);

/* Decode attention through block tables ([K] "The Block Table Is the Map",
 * "Follow One Token Address", "Batching Becomes More Flexible"; verification
 * recipe under "A Tiny Block-Table Example").  For every sequence s and query
 * head h, with G = num_q_heads / kv_heads and kv = h / G:
 *   x_j = scale * <q[s][h], K_s[j][kv]>   for every cached position
 *                                         j = 0 .. context_lens[s]-1, where
 *   K_s[j] is the key in block block_tables[s][j / block_size] at offset
 *   j % block_size;   out[s][h] = sum_j softmax(x)_j * V_s[j][kv].
 *   q             device [S][num_q_heads][head_dim], pool dtype (bf16 for an
 *                 fp8 pool)
 *   block_tables  device int32 [S][max_blocks_per_seq]; entries past a
 *                 sequence's last block are never read
 *   context_lens  device int32 [S]; 0 gives an all-zero output row; larger
 *                 than max_blocks_per_seq * block_size records
 *                 PA_ERR_BAD_LENGTH and is clamped
 *   out           device [S][num_q_heads][head_dim] of out_dtype
 * Keys/values are read once per (sequence, KV head) for all G query heads;
 * long contexts are split over block ranges and merged by log-sum-exp in a
 * second kernel (two launches per call).  The partition length is chosen on
 * the device from the batch's total length, so that the work items fill
 * whole waves of one item per resident CTA (one wave for a small batch, a
 * few for a large one; on fp8 pools partitions of at least 256 tokens while
 * two items per SM remain); the output does not depend on that choice beyond
 * rounding.  Batches with more sequences than
 * the GPU has SMs use partitions of at most 2048 tokens (the pool's
 * PA_OPT_PARTITION_CAP option overrides); the split never produces more
 * partials than the workspace holds.
 * Arithmetic: bf16 pools use bf16 tensor-core products with fp32
 * accumulation and fp32 softmax (the probabilities enter the value product
 * as a bf16 high part plus a bf16 low part); f32 pools use fp32 CUDA cores.
 * Supported: num_q_heads a multiple of kv_heads with G <= 16; bf16 pools
 * with head_dim in {64, 128, 256}, block_size a multiple of 16 and G <= 8
 * take the tensor-core path, every other shape the fp32 CUDA-core path;
 * S <= 16384.
 * Workspace: the pool keeps a device workspace for the split partials; a
 * call that needs more than it holds grows it (cudaMalloc, synchronous).
 * pa_decode_reserve sizes it ahead of time.
 * fp8 pool: K and V above are the dequantized values (code * k_scale,
 * code * v_scale).  On the tensor-core shapes (block_size % 16 == 0, head_dim
 * 64/128/256, G <= 8) the codes are widened exactly to f16 and each query to
 * f16 (exact for bf16 values of magnitude 2^-17 .. 65504), products are summed
 * in fp32, k_scale is applied to the scores and v_scale to the sums; other
 * shapes run the fp32 CUDA-core kernel on the dequantized values. */
int pa_decode(pa_pool *pool, const void *q, int num_seqs, int num_q_heads,
              const int32_t *block_tables, int max_blocks_per_seq,
              const int32_t *context_lens, float scale, void *out, pa_dtype out_dtype,
              void *stream);

/* Append then decode in one call: for each sequence s, its new token's keys
 * and values k[s], v[s] ([S][kv_heads][head_dim], pool dtype (bf16 for an
 * fp8 pool), device) are
 * written to slot_mapping[s] (device int64 [S]; negative = no token), exactly
 * as pa_append_kv with T = S would, and then decode attention runs exactly as
 * pa_decode.  Each slot must be the slot of position context_lens[s] - 1 of
 * sequence s (the token the decode of s reads last); otherwise nothing is
 * written for it and PA_ERR_INVALID_ARG is recorded on the device.  On the
 * tensor-core path (bf16 pools, and fp8 pools whose codes the kernel widens)
 * the write is done inside the decode kernel by the warp that reads that block
 * (one launch fewer per step; an fp8 pool's codes are quantized there exactly
 * as pa_append_kv quantizes them); other shapes run pa_append_kv and pa_decode
 * back to back.  Copy-on-write copies, if any, must be issued before
 * (pa_copy_blocks). */
int pa_append_decode(pa_pool *pool, const void *k, const void *v, const int64_t *slot_mapping,
                     const void *q, int num_seqs, int num_q_heads, const int32_t *block_tables,
                     int max_blocks_per_seq, const int32_t *context_lens, float scale,
                     void *out, pa_dtype out_dtype, void *stream);

/* Size the pool's decode workspace for batches up to these bounds. */
int pa_decode_reserve(pa_pool *pool, int max_seqs, int max_q_heads);

/* Decode attention for batches whose requests share leading blocks, reading
 * each shared block once for all the queries that point at it ([Z] answer:
 * requests with one prefix point at one copy; [K] "Prefix Sharing Is a
 * Natural Extension").  Same arguments and result as pa_decode, plus a host
 * description of the sharing (pa_bm_prefix_groups produces it):
 *   group_seq_offsets   host int32 [num_groups + 1], offsets[0] == 0: group g
 *                       owns batch entries group_seqs[offsets[g] .. offsets[g+1])
 *   group_seqs          host int32: batch indices; each in at most one group
 *   group_shared_blocks host int32 [num_groups]: number of leading table
 *                       entries that name one physical block in every
 *                       member's table and lie wholly inside every member's context
 * For each group and KV head, tiles of up to 128 query rows (members x their
 * G heads) attend to 1024-token chunks of the shared span together on the
 * 5th-generation tensor cores (tcgen05: operands staged in shared memory,
 * accumulators in tensor memory; head_dim 128, block_size 16, G <= 8, bf16
 * pools or fp8 pools, whose codes are widened to f16 in shared memory and
 * whose queries are re-rounded to f16; other tensor-core shapes use 64-row
 * tiles on mma.sync, which the pool's PA_OPT_SHARED_KERNEL option also
 * selects); each member's private suffix goes through the ordinary split
 * path, and the partials are merged by log-sum-exp.  Groups with fewer than two members
 * or no shared block are ignored; shapes outside the bf16 tensor-core path
 * (see pa_decode) fall back to pa_decode.  The device checks that members'
 * leading entries agree and that their contexts cover the shared span, and
 * records PA_ERR_INVALID_ARG otherwise (the result is then undefined).
 * The description is uploaded to the device when it differs from the
 * previous call's (a synchronous copy); repeated steps with the same sharing
 * reuse it.  Calls on one pool must not overlap on the GPU. */
int pa_decode_shared(pa_pool *pool, const void *q, int num_seqs, int num_q_heads,
                     const int32_t *block_tables, int max_blocks_per_seq,
                     const int32_t *context_lens, float scale, void *out,
                     pa_dtype out_dtype, const int32_t *group_seq_offsets,
                     const int32_t *group_seqs, const int32_t *group_shared_blocks,
                     int num_groups, void *stream);

/* Decode without allocating: the same computation, arguments and result as
 * pa_decode, for callers that cannot let the library call cudaMalloc — a
 * process whose device memory is owned by another allocator (a framework's
 * caching allocator that has reserved the GPU, or a fixed memory budget set
 * by the application), or a serving loop that cannot pay for cudaMalloc's
 * implicit device-wide synchronisation.  The pages have no counterpart: this
 * is an interface choice of this library, not part of the method.
 * The split partials and arrival counters live in a fixed 32 MiB array inside
 * the library image that every GPU loading the library holds until the
 * process exits; nothing is allocated or freed by the call (it clears the
 * counters with cudaMemsetAsync on `stream`).  A batch whose partials do not
 * fit returns PA_ERR_UNSUPPORTED before launching anything (roughly:
 * sequences x KV heads up to about 14,000 at head_dim 128, G 4, on a 152-SM
 * GB300; when the array has less room than the partition cap would use, the
 * kernel takes longer partitions instead).
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current) and caches it.  Under lazy
 * module loading (CUDA's default) that lookup is what loads the library's
 * device code, so the 32 MiB are reserved during that first call: make it
 * before the process's own allocator reserves the GPU's memory, and before
 * any stream capture begins.  If the device has no room for it, the call
 * returns PA_ERR_OUT_OF_MEMORY.  The cached address does not survive a
 * cudaDeviceReset of that device: do not call this entry point on a device
 * after resetting it.  All calls on a device share the one array, which keeps the last
 * call's contents: calls that overlap on the GPU (other streams, other pools,
 * other threads) race and give wrong results; serialise them. */
int pa_decode_noalloc(pa_pool *pool, const void *q, int num_seqs, int num_q_heads,
                      const int32_t *block_tables, int max_blocks_per_seq,
                      const int32_t *context_lens, float scale, void *out,
                      pa_dtype out_dtype, void *stream);

/* Paged prefill attention of one chunk of new tokens per sequence.  The pages
 * name the prefill step only through what a prefix-cache hit saves ([Z]
 * answer and [K] "Prefix Sharing Is a Natural Extension": a hit means that
 * span needs no prefill); this library's reading: a chunk's keys and values are
 * appended first (pa_append_kv, the slots of positions L-n .. L-1), then chunk
 * token i of sequence s, at position L-n+i with L = context_lens[s] and
 * n = cu_seqlens_q[s+1] - cu_seqlens_q[s], attends to every cached key of s at
 * positions 0 .. L-n+i (the whole cached prefix, and the chunk causally):
 *   out[t][h] = sum_j softmax_j(scale * <q[t][h], K_s[j][h/G]>) * V_s[j][h/G]
 * over j <= its position, K_s / V_s found through block_tables[s] as in
 * pa_decode.
 *   q             device bf16 [T][num_q_heads][head_dim], the chunks packed
 *                 sequence after sequence (T = num_tokens)
 *   cu_seqlens_q  device int32 [S+1]: sequence s owns query rows
 *                 cu_seqlens_q[s] .. cu_seqlens_q[s+1]-1; cu_seqlens_q[0] = 0
 *   max_q_len     host int: no chunk is longer (sizes the launch)
 *   block_tables  device int32 [S][max_blocks_per_seq]
 *   context_lens  device int32 [S]: L after the chunk's append, L >= n
 *   out           device [T][num_q_heads][head_dim] of out_dtype (8-byte aligned)
 * Requires a bf16 or fp8 pool (else PA_ERR_DTYPE), block_size % 16 == 0
 * and head_dim 64/128/256 (else PA_ERR_UNSUPPORTED).  An fp8 pool's codes are
 * widened exactly to f16 and the bf16 queries re-rounded to f16 (exact for
 * magnitudes 2^-17 .. 65504); products are summed in fp32, k_scale is applied
 * to the scores and v_scale to the outputs (both kernels).  One kernel launch:
 * one CTA per (query rows, KV head, sequence) streams the keys up to its last
 * row's position through shared memory once for all its rows: 128 rows on the
 * tcgen05 tensor cores (keys/values staged by TMA for bf16 pools, an fp8
 * pool's codes by bulk copy and widened in shared memory; TMEM accumulators)
 * for 16-token blocks, head_dim 128 and a 16-byte-aligned out; 64 rows on
 * mma.sync otherwise (or when the pool's PA_OPT_PREFILL_KERNEL option selects
 * it).  Whatever
 * bits a block holds at positions at or past the sequence's length (a block
 * recycled from a finished request may hold anything, Inf and NaN included)
 * never reach the output.  A non-finite key or value inside the chunk itself
 * (a caller input) does reach the chunk's earlier rows, which weigh it by
 * zero (0 * Inf is NaN), as it reaches every later row.
 * On the device: a malformed cu_seqlens_q (decreasing, beyond T, a
 * chunk longer than its context or than max_q_len) records PA_ERR_INVALID_ARG,
 * a context beyond the table PA_ERR_BAD_LENGTH, a block id outside the pool
 * PA_ERR_BAD_BLOCK_ID; those sequences' rows are left unwritten. */
int pa_prefill(pa_pool *pool, const void *q, int num_tokens, int num_q_heads,
               const int32_t *cu_seqlens_q, int num_seqs, int max_q_len,
               const int32_t *block_tables, int max_blocks_per_seq,
               const int32_t *context_lens, float scale, void *out, pa_dtype out_dtype,
               void *stream);

/* Synchronize `stream`, then return and clear the first error the pool's
 * kernels recorded since the last call (PA_OK if none). */
int pa_get_error(pa_pool *pool, void *stream);

/* Static text for an error code. */
const char *pa_error_string(int code);

/* Number of kernels the library launched since it was loaded (all pools). */
uint64_t pa_launch_count(void);

/* ------------------------------------------------- host block manager --- */
/* Plain host bookkeeping, not on the GPU ([K] "Growth Needs Only Another
 * Free Block", "Shared Blocks Must Not Be Changed in Place"; [Z] answer and
 * follow-ups on the parent-chained hash and the cache key):
 *   - free pool: FIFO, initial order given; freed blocks join the tail in
 *     table order;
 *   - a request grows by one free block when its next token starts a block;
 *   - reference count per block = number of live requests pointing at it;
 *     a block returns to the free pool when its count reaches zero;
 *   - copy-on-write: the next token of a request whose last block another
 *     request also points at goes to a fresh block; the pair (old, fresh) is
 *     returned for pa_copy_blocks and only this request's entry is repointed;
 *   - prefix cache: each full block is hashed as FNV-1a-64 over (parent
 *     block's hash, 8 bytes LE; salt, 8 bytes LE; its token ids, 4 bytes LE
 *     each), the first block's parent hash being 0; a table maps hash to
 *     physical block; admission reuses leading cached blocks while the
 *     chain hits (token ids and parent block compared too) and stops at the
 *     first miss.  A block leaves the hash table when freed (unless
 *     retention is on: pa_bm_set_retention).
 * Not thread-safe: one manager per thread. */

/* free_order: host int32 [num_blocks], a permutation of 0..num_blocks-1 giving
 * the free pool's initial order; NULL means 0, 1, 2, ... */
int pa_bm_create(int num_blocks, int block_size, const int32_t *free_order, pa_bm **out);
int pa_bm_destroy(pa_bm *bm);

/* Admit a request with prompt token ids tokens[0..n); reuses cached full
 * blocks of the prompt's prefix.  *req = new request id, *cached_tokens =
 * number of leading prompt tokens already in the cache.  The caller appends
 * the remaining prompt tokens with pa_bm_append_slot(s). */
int pa_bm_add_request(pa_bm *bm, const int32_t *tokens, int n, uint64_t salt, int *req,
                      int *cached_tokens);

/* A new request sharing every block of `parent` (parallel sampling). */
int pa_bm_fork(pa_bm *bm, int parent, int *child);

/* Reserve the slot of request `req`'s next token (token id `token`).
 * *slot = block * block_size + offset.  *cow_src / *cow_dst = the copy pair
 * when copy-on-write happened, else -1 / -1.  On error nothing changes. */
int pa_bm_append_slot(pa_bm *bm, int req, int32_t token, int64_t *slot, int64_t *cow_src,
                      int64_t *cow_dst);

/* Batched form: for i in 0..n, append tokens[i] to reqs[i] in order.
 * slots[i] receives each slot; copy pairs are written to cow_pairs
 * ([*num_pairs][2], room for n pairs) in the order they arise.  Stops at the
 * first error; *num_done = entries applied before it. */
int pa_bm_append_slots(pa_bm *bm, int n, const int32_t *reqs, const int32_t *tokens,
                       int64_t *slots, int64_t *cow_pairs, int *num_pairs, int *num_done);

/* Release a finished request's blocks. */
int pa_bm_free_request(pa_bm *bm, int req);

/* Copy the request's block table into out[0..cap); *n = its length. */
int pa_bm_block_table(pa_bm *bm, int req, int32_t *out, int cap, int *n);

/* Fill tables [n][width] (host, int32) with the block tables of reqs[0..n),
 * padding with -1, and lens[n] with their token counts. */
int pa_bm_batch_tables(pa_bm *bm, int n, const int32_t *reqs, int width, int32_t *tables,
                       int32_t *lens);

/* *width = the longest block table among reqs[0..n) (0 for n = 0): the width
 * pa_bm_batch_tables needs for that batch.  PA_ERR_UNKNOWN_REQUEST if a
 * request is unknown (then *width is unchanged). */
int pa_bm_batch_width(pa_bm *bm, int n, const int32_t *reqs, int *width);

/* Number of tokens of a request; -1 if unknown. */
int pa_bm_seq_len(pa_bm *bm, int req);

/* Reference count of a block (0 = free); -1 if out of range. */
int pa_bm_refcount(pa_bm *bm, int block);

/* Number of free blocks. */
int pa_bm_num_free(pa_bm *bm);

/* Copy the free pool in FIFO order into out[0..cap); *n = its length. */
int pa_bm_free_list(pa_bm *bm, int32_t *out, int cap, int *n);

/* Sharing description of a decode batch for pa_decode_shared: batch entries
 * i (requests reqs[i]) whose tables start with the same physical block form
 * a group (in order of first appearance; singletons dropped); its shared
 * span is the longest run of leading entries that are the same physical
 * block for all members and full in every member.  Outputs (host, room for
 * n + 1 / n / n entries): group_offsets, group_seqs (batch indices),
 * group_shared_blocks; *num_groups = number of groups. */
int pa_bm_prefix_groups(pa_bm *bm, int n, const int32_t *reqs, int32_t *group_offsets,
                        int32_t *group_seqs, int32_t *group_shared_blocks, int *num_groups);

/* 1 if the block is registered in the prefix hash table, 0 if not, -1 if out
 * of range. */
int pa_bm_is_cached(pa_bm *bm, int block);

/* Retention of cached blocks after their last user leaves ([Z] follow-up on
 * how eviction interacts with the reference count, left unanswered there;
 * [K] "Prefix Reuse Also Needs Compatible Computation": what a system keeps
 * for later reuse is its own policy, over full blocks only).  Off by default (a freed block leaves
 * the hash table at once).  With on != 0:
 *   - a block still registered in the hash table whose count reaches zero
 *     stays registered and becomes evictable instead of joining the free
 *     pool; evictable blocks are kept in the order they were released;
 *   - pa_bm_free_request releases a request's blocks deepest first, so a
 *     chain's later blocks are evicted before its first ones;
 *   - a new block (growth or copy-on-write) comes from the free pool while it
 *     has one, else the least recently released evictable block is evicted:
 *     it leaves the hash table and is reused;
 *   - an admission hit on an evictable block takes it back (count 0 -> 1).
 * on == 0 returns every evictable block to the free pool's tail (in release
 * order), dropping its hash entry. */
int pa_bm_set_retention(pa_bm *bm, int on);

/* Number of evictable blocks (0 while retention is off); -1 for NULL. */
int pa_bm_num_evictable(pa_bm *bm);

/* Copy the evictable blocks, least recently released first, into
 * out[0..cap); *n = their number. */
int pa_bm_evictable_list(pa_bm *bm, int32_t *out, int cap, int *n);

/* FNV-1a-64 of a byte string (exposed so the hash can be checked). */
uint64_t pa_bm_fnv1a64(const uint8_t *data, size_t n);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_KV_CACHE_PA_H */
