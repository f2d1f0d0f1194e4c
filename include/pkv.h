/*
 * pkv.h -- C ABI of libpkv: paged KV-cache decode attention for GB300 (sm_103a).
 *
 * What the library computes (sources cited by page title and section):
 *
 *  - A flat pool of fixed-size physical KV blocks (16 tokens by default) and
 *    a per-sequence block table mapping logical block i (tokens 16i..16i+15)
 *    to a physical block ("The 8GB VRAM Breakthrough", §3 "How
 *    Logical-to-Physical Block Tables Work").  The pool is a stack of free
 *    block ids plus one reference count per block ("A Ideia de 60 Anos Que
 *    Domou a Memória da GPU", section "o código: a diferença entre reservar e
 *    mapear"); blocks are taken on demand when the current one is full (same
 *    page, section "a ideia roubada").
 *  - Prefix sharing by reference counts and copy-on-write of a *partially
 *    filled* shared block on the first divergent write ("The 8GB VRAM
 *    Breakthrough", §3 "Copy-on-Write (CoW) Prefix Sharing").
 *  - The KV-append write of each new token ("The 8GB VRAM Breakthrough", §1:
 *    every generated token writes one new KV vector back).
 *  - Single-query grouped-query attention through the block tables ("The 8GB
 *    VRAM Breakthrough", §3: the kernel gathers the scattered physical blocks
 *    for QK^T and the softmax-weighted sum of V).  Paging does not change the
 *    result ("PagedAttention aplica memória virtual ao cache KV de LLMs",
 *    section "Compartilhamento e compromissos"): the output is plain
 *    softmax(scale * q K^T) V over the sequence's tokens in logical order.
 *  - An INT4-asymmetric / FP8-E4M3 cache with the first n_sink tokens kept in
 *    16-bit, dequantised in registers inside the attention kernel ("The 8GB
 *    VRAM Breakthrough", §4 "The Hybrid Solution: Sink-FP16 + Group-Wise
 *    Asymmetric INT4 / FP8" and §5 "On-the-Fly Register Dequantization").
 *
 * Conventions (all entry points):
 *  - Every function returns an int status: PKV_OK (0) or a negative PKV_ERR_*.
 *    No exception or C++ object crosses the ABI; results go to out-params.
 *  - Host handles (pkv_pool*) are created and owned by the library; release
 *    them with pkv_pool_destroy.  Host calls on one pool are not thread-safe.
 *  - ALL device memory is owned by the caller (pools, tables, workspaces,
 *    outputs).  The library never allocates or frees device memory.
 *  - Device entry points are asynchronous on the caller's cudaStream_t,
 *    passed as void* (NULL = legacy default stream).  A failed launch returns
 *    PKV_ERR_CUDA.  Arguments are validated on the host before any launch
 *    (PKV_ERR_INVALID_ARG / PKV_ERR_UNSUPPORTED / PKV_ERR_MISALIGNED /
 *    PKV_ERR_WORKSPACE); data-dependent indices (table entries, slots, context
 *    lengths) are checked on the device: an out-of-range index is skipped (it
 *    is never dereferenced) and a bit is set in a per-device status word that
 *    pkv_device_status reads back.
 *  - Device pointers must be 16-byte aligned.  16-bit data is IEEE fp16
 *    (PKV_DTYPE_F16) or bfloat16 (PKV_DTYPE_BF16).
 *  - Layouts are row-major (last index fastest):
 *      q, out           [batch, num_q_heads, head_dim]          16-bit
 *      k, v (new rows)  [num_tokens, num_kv_heads, head_dim]    16-bit
 *      k_pool, v_pool   [num_blocks, num_kv_heads, block_size, head_dim]
 *      block_tables     [batch, max_blocks] int32, entries past the context
 *                       are not read (the host manager pads them with -1)
 *      context_lens     [batch] int32, tokens per sequence INCLUDING the
 *                       token appended in this decode step
 *      slot_mapping     [num_tokens] int64, slot = block * block_size + offset;
 *                       a negative slot skips that token
 *  - Query head h reads KV head h / (num_q_heads / num_kv_heads).
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- status */
enum {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = -1,   /* null pointer, bad size or shape            */
    PKV_ERR_OUT_OF_BLOCKS = -2, /* pool cannot supply the blocks; no change   */
    PKV_ERR_BAD_HANDLE = -3,    /* null pool handle                           */
    PKV_ERR_BAD_SEQ = -4,       /* unknown sequence id                        */
    PKV_ERR_DOUBLE_FREE = -5,   /* refcount of a free block would go below 0  */
    PKV_ERR_CUDA = -6,          /* a CUDA runtime call or launch failed       */
    PKV_ERR_DEVICE_BOUNDS = -7, /* device status word had an index error      */
    PKV_ERR_UNSUPPORTED = -8,   /* valid but not implemented shape / mode     */
    PKV_ERR_WORKSPACE = -9,     /* workspace missing or too small             */
    PKV_ERR_MISALIGNED = -10    /* a device pointer is not 16-byte aligned    */
};

enum { PKV_DTYPE_F16 = 0, PKV_DTYPE_BF16 = 1 };
enum { PKV_QMODE_INT4_ASYM = 1, PKV_QMODE_FP8_E4M3 = 2 };

/* Device status bits (see pkv_device_status). */
enum {
    PKV_STATUS_BAD_BLOCK = 1,   /* block-table entry outside [0, num_blocks)     */
    PKV_STATUS_BAD_SLOT = 2,    /* slot outside [0, num_blocks * block_size)     */
    PKV_STATUS_BAD_CONTEXT = 4, /* context_len < 0 or > max_blocks * block_size  */
    PKV_STATUS_BAD_PAIR = 8,    /* copy pair outside [0, num_blocks)             */
    PKV_STATUS_BAD_SINK = 16,   /* sink row / position outside its buffer        */
    PKV_STATUS_COPY_TIMEOUT = 32 /* a bounded wait for an asynchronous copy or a
                                  * tensor-core operation ran out; that call's
                                  * outputs are undefined                      */
};

/* Human-readable name of a status code (static string, never NULL). */
const char* pkv_status_string(int status);

/* Library ABI version (monotonic integer). */
int pkv_version(void);

/* ====================================================== host block manager
 * Physical block pool with a LIFO free stack and one reference count per
 * block, plus sequences with block tables ("A Ideia de 60 Anos...", section
 * "o código"; "The 8GB VRAM Breakthrough", §3).
 */
typedef struct pkv_pool pkv_pool;

/* Create a pool of num_blocks blocks of block_size tokens.  free_order
 * (host, nullable, num_blocks entries, a permutation of 0..num_blocks-1)
 * fixes the allocation order: successive allocations from a fresh pool
 * return free_order[0], free_order[1], ...; NULL means 0, 1, 2, ....
 * Errors: INVALID_ARG (sizes <= 0, not a permutation). */
int pkv_pool_create(int32_t num_blocks, int32_t block_size, const int32_t* free_order,
                    pkv_pool** out);
int pkv_pool_destroy(pkv_pool* pool);
int pkv_pool_num_free(const pkv_pool* pool, int32_t* out);
int pkv_pool_num_blocks(const pkv_pool* pool, int32_t* out);
int pkv_pool_block_size(const pkv_pool* pool, int32_t* out);

/* Pop a free block and set its count to 1.  OUT_OF_BLOCKS if none. */
int pkv_block_alloc(pkv_pool* pool, int32_t* block);
/* Add an owner to an allocated block.  DOUBLE_FREE if the block is free. */
int pkv_block_incref(pkv_pool* pool, int32_t block);
/* Drop an owner; at zero the block is pushed back on the free stack.
 * DOUBLE_FREE if the count is already zero. */
int pkv_block_decref(pkv_pool* pool, int32_t block);
int pkv_block_refcount(const pkv_pool* pool, int32_t block, int32_t* out);

/* New empty sequence.  Ids are 0, 1, 2, ... in creation order (forks too). */
int pkv_seq_create(pkv_pool* pool, int64_t* seq);
/* Give back every block of the sequence in logical order.  BAD_SEQ. */
int pkv_seq_free(pkv_pool* pool, int64_t seq);
/* Child sharing all of the parent's blocks (each count + 1), same length. */
int pkv_seq_fork(pkv_pool* pool, int64_t parent, int64_t* child);

/* Reserve slots for n_tokens new tokens of seq (the copy-on-write append).
 * If the tail block is partially filled and shared (count > 1) it is first
 * replaced by a fresh block and one (src, dst) copy is reported; then a new
 * block is taken each time the tail fills.
 *   slots_out       host int64[n_tokens]: slot of each new token
 *   copy_pairs_out  host int32[2] (nullable if the caller guarantees no CoW):
 *                   {src, dst} of the block the caller must copy (K, V and any
 *                   quantisation metadata) before writing the new tokens
 *   n_copies        host int32: 0 or 1
 * All-or-nothing: OUT_OF_BLOCKS leaves the pool and the sequence unchanged. */
int pkv_seq_append(pkv_pool* pool, int64_t seq, int32_t n_tokens, int64_t* slots_out,
                   int32_t* copy_pairs_out, int32_t* n_copies);

/* One decode step for n sequences: appends n_tokens_each tokens to each of
 * seqs[0..n-1] in order.  slots_out int64[n * n_tokens_each];
 * copy_pairs_out int32[2 * n] (pairs in sequence order); n_copies total.
 * All-or-nothing across the whole batch. */
int pkv_seq_append_batch(pkv_pool* pool, const int64_t* seqs, int32_t n, int32_t n_tokens_each,
                         int64_t* slots_out, int32_t* copy_pairs_out, int32_t* n_copies);

int pkv_seq_len(const pkv_pool* pool, int64_t seq, int64_t* out);
int pkv_seq_num_blocks(const pkv_pool* pool, int64_t seq, int32_t* out);
/* Copy the sequence's table into out[0..capacity); INVALID_ARG if it does
 * not fit. */
int pkv_seq_block_table(const pkv_pool* pool, int64_t seq, int32_t* out, int32_t capacity);

/* Build the decode inputs for seqs[0..n-1]: tables (host int32 [n, max_blocks],
 * unused entries -1) and context_lens (host int32 [n]).  INVALID_ARG if a
 * sequence has more than max_blocks blocks. */
int pkv_build_block_tables(const pkv_pool* pool, const int64_t* seqs, int32_t n, int32_t* tables,
                           int32_t max_blocks, int32_t* context_lens);

/* Fault injection: after n more successful block allocations, every further
 * allocation fails with OUT_OF_BLOCKS (appends stay all-or-nothing).
 * n < 0 disables. */
int pkv_debug_fail_after(pkv_pool* pool, int64_t n_allocs);

/* Test hook for the bounded waits of the tensor-core prefill kernel (the
 * multi-query path for long query spans): while tile >= 0, no CTA issues
 * the K copy of key tile `tile`, so the wait for it runs out after its time
 * limit (~0.3 s); the kernel then sets PKV_STATUS_COPY_TIMEOUT, lets its
 * copies and MMAs in flight finish (each wait again bounded) and stops,
 * leaving the context usable.  Outputs of such a call are undefined.
 * -1 (the default) turns it off; below -1 is INVALID_ARG.  Device-wide
 * (the current device), for tests only. */
int pkv_debug_prefill_drop_copy(int32_t tile);

/* ========================================================= prefix cache */

/* Prefix cache ("Capítulo 8 — Gerenciamento de KV Cache de Próxima Geração",
 * §8.3): prompts are cut into block_size-token chunks; a chunk already
 * computed under the same preceding chunks maps the cached physical block
 * into a new request's table, so its prefill is skipped.  An entry is one
 * full block keyed by (previous entry, its block_size token ids), compared
 * exactly (a 64-bit hash only buckets candidates).  The cache holds one
 * reference on every entry's block.  Token ids are opaque int32 values. */

/* Registers the full blocks of seq holding tokens[0 .. n_tokens) (the first
 * floor(n_tokens / block_size) blocks of its table; n_tokens <= its length).
 * Chunks already cached are skipped (the chain continues through them).
 * n_new (nullable): entries added. */
int pkv_prefix_register(pkv_pool* pool, int64_t seq, const int32_t* tokens, int32_t n_tokens,
                        int32_t* n_new);

/* Creates a sequence whose table is the longest chain of cached full blocks
 * matching tokens (each block's refcount + 1) and whose length is
 * matched_tokens (a multiple of block_size, <= n_tokens, 0 on a miss).  The
 * caller prefills tokens[matched_tokens ..] with pkv_seq_append. */
int pkv_prefix_match(pkv_pool* pool, const int32_t* tokens, int32_t n_tokens, int64_t* seq_out,
                     int32_t* matched_tokens);

/* Drops up to n_blocks entries, least recently matched or registered first,
 * among leaves (no cached chunk extends them) whose block no sequence holds;
 * their blocks return to the free stack.  n_freed (nullable): entries
 * dropped. */
int pkv_prefix_evict(pkv_pool* pool, int32_t n_blocks, int32_t* n_freed);

/* Drops every entry, releasing the cache's references in registration
 * order. */
int pkv_prefix_clear(pkv_pool* pool);

/* Entries held, pkv_prefix_match calls, and blocks those calls matched. */
int pkv_prefix_stats(const pkv_pool* pool, int64_t* entries, int64_t* lookups, int64_t* hit_blocks);

/* ================================================================ sizes */

/* Bytes of the split-K workspace pkv_paged_attention_decode* needs for this
 * shape.  Zero when a single partition covers max_blocks * block_size
 * (single-pass decode).  U = ceil(max_blocks * block_size / 16), the
 * tables' capacity in 16-token units (the kernels' token tile).
 *   - partition_size > 0 (a positive multiple of 16 and of block_size):
 *     fixed partitions, fp32 partial outputs [batch, num_q_heads, P,
 *     head_dim] and fp32 (max, sum) pairs [batch, num_q_heads, P, 2],
 *     P = ceil(max_blocks * block_size / partition_size).
 *   - partition_size 0 (automatic): the same for the automatic partition
 *     size (pkv_decode_auto_partition_size), or, when the automatic split
 *     may be balanced (batch <= 1024 and batch * num_q_heads * U >=
 *     32 * 16 * SMs), the larger of that and the balanced split's need:
 *     (nwt * 8 + batch * num_q_heads) * (head_dim + 2) * 4 bytes,
 *     nwt = min(20 * SMs, batch * num_q_heads * U / 2), the most warps a
 *     balanced kernel launches (SMs of the current device, 152 if none).
 * max_blocks * block_size above 2^30 is UNSUPPORTED. */
int pkv_decode_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t head_dim,
                               int32_t max_blocks, int32_t block_size, int32_t partition_size,
                               size_t* out);

/* The partition size of an automatic split that is not balanced (see
 * pkv_paged_attention_decode; the quantised decode follows the same rule),
 * and of _partials / _merge with partition_size 0: the largest of 512,
 * 256, 128, 64 tokens for which batch * num_q_heads * ceil(max_blocks *
 * block_size / size) >= 12 * (SM count of the current device, 152 if none),
 * else 64.  Small batches get finer splits so the GPU has enough partition
 * CTAs.  block_size 8, 16 or 32 (else UNSUPPORTED). */
int pkv_decode_auto_partition_size(int32_t batch, int32_t num_q_heads, int32_t max_blocks,
                                   int32_t block_size, int32_t* out);

/* =============================================================== device */

/* KV-append scatter: for every token t with slot_mapping[t] >= 0,
 * k_pool[slot / block_size, h, slot % block_size, :] = k[t, h, :] (and the
 * same for v), bit-exact.  head_dim % 8 == 0.  Slots beyond the pool set
 * PKV_STATUS_BAD_SLOT and are skipped. */
int pkv_kv_append(const void* k, const void* v, const int64_t* slot_mapping, int32_t num_tokens,
                  void* k_pool, void* v_pool, int32_t num_blocks, int32_t num_kv_heads,
                  int32_t head_dim, int32_t block_size, int dtype, void* stream);

/* Paged decode attention: out[b, h, :] = sum_t softmax_t(scale *
 * <q[b, h], K_t>) V_t over the tokens t < context_lens[b] of sequence b,
 * where K_t / V_t are read from k_pool / v_pool at block
 * block_tables[b, t / block_size], offset t % block_size, KV head
 * h / (num_q_heads / num_kv_heads).  fp32 accumulation; out has q's dtype;
 * a sequence with context 0 gets zeros.
 * Split-K: when more than one partition can occur (max_blocks * block_size
 * > the partition size) partial (max, sum, output) triples go to
 * `workspace` (device, >= pkv_decode_workspace_bytes) and a second kernel,
 * launched behind the first with programmatic dependent launch, merges them
 * with a log-sum-exp rescale (flash-decoding split-K); otherwise one pass
 * writes out directly.
 *   - partition_size > 0 (a multiple of 16 and of block_size, else
 *     INVALID_ARG): the context is cut into partitions of that many
 *     tokens, one CTA each.
 *   - partition_size 0 (automatic): if batch <= 1024 and batch *
 *     num_kv_heads * U (U = ceil(max_blocks * block_size / 16)) is at least
 *     32 items per launched warp (16 warps per SM) and below 2^30, a
 *     balanced split: the (sequence, KV head, 16-token unit) items of the
 *     call, in that order, are cut into one contiguous, equal share per
 *     warp, whatever the mix of context lengths; else partitions of
 *     pkv_decode_auto_partition_size tokens.
 * The kernels' token tile is 16 tokens: one block at block_size 16, half a
 * block at 32, two blocks at 8 (both table entries of a tile are checked;
 * a bad one skips the whole 16-token tile and sets PKV_STATUS_BAD_BLOCK).
 * Calls that share a workspace must not overlap on the GPU.
 * Supported: block_size 8, 16 or 32, head_dim 64 or 128, 1 <= num_q_heads /
 * num_kv_heads <= 8 (else UNSUPPORTED). */
int pkv_paged_attention_decode(const void* q, const void* k_pool, const void* v_pool,
                               const int32_t* block_tables, const int32_t* context_lens,
                               int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                               int32_t head_dim, int32_t num_blocks, int32_t block_size,
                               int32_t max_blocks, float scale, void* out, void* workspace,
                               size_t workspace_bytes, int32_t partition_size, int dtype,
                               void* stream);

/* One decode step in one kernel: for every sequence b with
 * slot_mapping[b] >= 0, writes k_new[b] / v_new[b] ([batch, num_kv_heads,
 * head_dim], 16-bit) into the pools at slot_mapping[b] and attends exactly
 * as pkv_paged_attention_decode, the new row being the last token
 * (position context_lens[b] - 1).  The slot must be that position's slot,
 * block_tables[b][(ctx-1)/block_size] * block_size + (ctx-1) % block_size
 * (what pkv_seq_append returned for the decode step); otherwise
 * PKV_STATUS_BAD_SLOT is set and the row is neither written nor used.
 * The new row is taken from k_new / v_new, never read back from the pool, so
 * no ordering against a separate append kernel is needed.  The pools are
 * written (not const).  Same workspace, shapes and errors as
 * pkv_paged_attention_decode. */
int pkv_paged_attention_decode_append(const void* q, const void* k_new, const void* v_new,
                                      const int64_t* slot_mapping, void* k_pool, void* v_pool,
                                      const int32_t* block_tables, const int32_t* context_lens,
                                      int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                      int32_t head_dim, int32_t num_blocks, int32_t block_size,
                                      int32_t max_blocks, float scale, void* out, void* workspace,
                                      size_t workspace_bytes, int32_t partition_size, int dtype,
                                      void* stream);

/* The two phases of a partitioned pkv_paged_attention_decode, for callers
 * that time or overlap them.  _partials always writes the workspace (never
 * out); _merge reads it and writes out.  Same arguments and requirements,
 * except that partition_size 0 means the automatic partition size
 * (pkv_decode_auto_partition_size), never the balanced split; size the
 * workspace with that partition size. */
int pkv_paged_attention_decode_partials(const void* q, const void* k_pool, const void* v_pool,
                                        const int32_t* block_tables, const int32_t* context_lens,
                                        int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                        int32_t head_dim, int32_t num_blocks, int32_t block_size,
                                        int32_t max_blocks, float scale, void* workspace,
                                        size_t workspace_bytes, int32_t partition_size, int dtype,
                                        void* stream);
int pkv_paged_attention_decode_merge(const int32_t* context_lens, int32_t batch,
                                     int32_t num_q_heads, int32_t head_dim, int32_t max_blocks,
                                     int32_t block_size, int32_t partition_size,
                                     const void* workspace, size_t workspace_bytes, void* out,
                                     int dtype, void* stream);

/* Multi-query paged attention: several new query tokens per sequence, each
 * attending causally to the cache up to its own position -- the target
 * model's one parallel pass over the gamma + 1 draft tokens of speculative
 * decoding ("The 8GB VRAM Breakthrough", §6), or one slice of a chunked
 * prefill (§5, "Chunked Prefill").
 *   q: [T, num_q_heads, head_dim] (dtype), T = q_start[batch]; the queries
 *     of sequence b are rows q_start[b] .. q_start[b+1] - 1 (device int32
 *     [batch + 1], non-decreasing; L_b = q_start[b+1] - q_start[b] <=
 *     max_q_len, which sizes the grid).
 *   The L_b new tokens are the last L_b of the context_lens[b] tokens in the
 *   pool (written before the call, e.g. by pkv_kv_append), so query i of
 *   sequence b sits at position p = context_lens[b] - L_b + i and
 *   out[q_start[b] + i, h] = sum_{t <= p} softmax_t(scale <q, K_t>) V_t
 *   over KV head h / (num_q_heads / num_kv_heads).  out: [T, num_q_heads,
 *   head_dim] (dtype).  L_b = 1 is pkv_paged_attention_decode.
 *   context_lens[b] < L_b sets PKV_STATUS_BAD_CONTEXT; rows at negative
 *   positions get zeros.  scale may have any sign (zero gives the mean of V
 *   up to each position).
 * Three kernels:
 *   - workspace (device, nullable) of at least
 *     pkv_multi_query_workspace_bytes bytes, and that size is non-zero
 *     (max_q_len * G <= 24, batch <= 1024, enough (sequence, KV head,
 *     block) items to fill the GPU): a balanced split.  Every warp streams
 *     an equal share of the call's (sequence, KV head, block) items, holding
 *     all L_b * G rows of its runs, so each K/V byte is read once.  A merge
 *     kernel follows behind it with programmatic dependent launch; the split
 *     kernel is itself launched that way and reads nothing before the
 *     stream's previous grid has completed (behind pkv_kv_append, its CTAs
 *     are made resident while the append runs).  L_b >
 *     max_q_len there sets PKV_STATUS_BAD_CONTEXT and only the first
 *     max_q_len * G rows are computed.  A workspace that is too small
 *     returns PKV_ERR_WORKSPACE.
 *   - otherwise, with head_dim 128, G in {1, 2, 4, 8} and max_q_len * G >
 *     64 (chunked-prefill slices): the 5th-generation tensor cores, one CTA
 *     per 128 (query token, query head) rows, tcgen05.mma with the
 *     accumulators in tensor memory and K/V tiles of 128 keys gathered from
 *     the blocks by TMA; a wait on those copies or MMAs that runs out sets
 *     PKV_STATUS_COPY_TIMEOUT.
 *   - otherwise one pass per (8 or 16 query rows, KV head, sequence).
 *   Only the balanced split touches the workspace.
 * Calls that share a workspace must not overlap on the GPU.
 * Supported: block_size 16, head_dim 64 or 128, 1 <= G <= 8. */
int pkv_paged_attention_multi_query(const void* q, const int32_t* q_start, const void* k_pool,
                                    const void* v_pool, const int32_t* block_tables,
                                    const int32_t* context_lens, int32_t batch, int32_t num_q_heads,
                                    int32_t num_kv_heads, int32_t head_dim, int32_t num_blocks,
                                    int32_t block_size, int32_t max_blocks, int32_t max_q_len,
                                    float scale, void* out, void* workspace, size_t workspace_bytes,
                                    int dtype, void* stream);

/* Workspace bytes for pkv_paged_attention_multi_query's balanced split:
 * (nwt + batch * num_kv_heads) * R * (head_dim + 2) * 4 with R =
 * 8 * ceil(max_q_len * G / 8) partial rows per slot and nwt the warps it
 * launches (at most 8 or 12 per SM).  0 when the split does not apply. */
int pkv_multi_query_workspace_bytes(int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                    int32_t head_dim, int32_t max_blocks, int32_t block_size,
                                    int32_t max_q_len, size_t* out);

/* Allocation-free decode.  The source pages have no counterpart for this
 * entry point: it exists for callers that cannot provide a device workspace
 * -- code running while a stream is captured into a CUDA graph (allocation
 * is not a capturable operation), plugins inside a host runtime that owns all
 * device memory and offers no allocator, and serving loops with a fixed,
 * pre-planned memory budget that must not call cudaMalloc / cudaFree (which
 * may synchronise the device) on the decode path.
 * Same arguments and result as pkv_paged_attention_decode, minus the
 * workspace: the split-K partials live in a fixed array inside the library
 * (PKV_STATIC_WORKSPACE_BYTES per GPU, held by every GPU that loads the
 * library until the process exits).  The call allocates nothing.
 *   - A shape whose pkv_decode_workspace_bytes exceeds
 *     PKV_STATIC_WORKSPACE_BYTES is rejected with PKV_ERR_WORKSPACE before
 *     any device work.
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current); make that first call before any
 *     stream capture.
 *   - All calls on a device share the one array and it keeps whatever the
 *     last call left in it; nothing in it needs to start at zero.  Calls whose
 *     kernels overlap on the GPU (different streams, no ordering) race on the
 *     array and give undefined results: order them on one stream or with
 *     events. */
#define PKV_STATIC_WORKSPACE_BYTES (16u << 20)
int pkv_paged_attention_decode_static_ws(const void* q, const void* k_pool, const void* v_pool,
                                         const int32_t* block_tables, const int32_t* context_lens,
                                         int32_t batch, int32_t num_q_heads, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t num_blocks, int32_t block_size,
                                         int32_t max_blocks, float scale, void* out,
                                         int32_t partition_size, int dtype, void* stream);

/* Quantised KV-append ("The 8GB VRAM Breakthrough", §4; §5 flowchart: fused
 * quantiser on the write path).  For every token t with slot >= 0 and every
 * KV head, K and V rows are quantised and written at the slot:
 *   INT4_ASYM: per group of group_size elements (group_size divides head_dim;
 *     supported: head_dim, 64, 32), binary32 steps in this order
 *     s = fp16(binary32(max - min) / 15), s = 1 if max == min or s == 0;
 *     z = fp16(binary32(-min) / s), -0 stored as +0;
 *     q = clamp(rint(binary32(x / s) + z), 0, 15)
 *     (fp16() rounds to nearest even, saturating at 65504); codes packed two
 *     per byte, element 2i in the low nibble.
 *     k_codes/v_codes u8 [num_blocks, Hkv, block_size, head_dim/2];
 *     k_scale/k_zero/v_scale/v_zero fp16 [num_blocks, Hkv, block_size,
 *     head_dim/group_size].  Dequantised value: (q - z) * s.
 *   FP8_E4M3: one scale per (token, head): s = fp16(max|x| / 448), 1 if 0;
 *     code = E4M3 (OCP e4m3fn) of binary32(x / s), nearest even, saturating
 *     at +-448.  k_codes/v_codes u8 [num_blocks, Hkv, block_size, head_dim];
 *     k_scale/v_scale fp16 [num_blocks, Hkv, block_size, 1]; zeros unused
 *     (may be NULL).  group_size is ignored.
 * Sinks: if positions[t] < n_sink, the 16-bit row is also copied to
 * sink_k/sink_v[seq_idx[t], positions[t], h, :]; sink buffers are
 * [sink_rows, n_sink, Hkv, head_dim] in dtype (nullable when n_sink == 0).
 * Local window ("The 8GB VRAM Breakthrough", §5 flowchart: the most recent
 * tokens go to the high-precision pool): with window > 0 (a multiple of
 * block_size) every row is also copied to the 16-bit ring win_k/win_v
 * [sink_rows, window / block_size + 1, Hkv, block_size, head_dim] (dtype)
 * at ring block (p / block_size) % (window / block_size + 1), offset
 * p % block_size, p = positions[t]; nullable when window == 0.  Within one
 * call, a row whose slot the entry one ring span (window + block_size)
 * further on takes again (same seq_idx, position p + span) is not written;
 * other layouts in which two rows of one call share a slot leave that slot
 * undefined, so pass a sequence's tokens as consecutive entries.
 * positions / seq_idx: device int32 [num_tokens]. */
int pkv_kv_append_quant(const void* k, const void* v, const int64_t* slot_mapping,
                        const int32_t* positions, const int32_t* seq_idx, int32_t num_tokens,
                        void* k_codes, void* k_scale, void* k_zero, void* v_codes,
                        void* v_scale, void* v_zero, void* sink_k, void* sink_v, int32_t n_sink,
                        int32_t sink_rows, void* win_k, void* win_v, int32_t window,
                        int32_t num_blocks, int32_t num_kv_heads,
                        int32_t head_dim, int32_t block_size, int32_t group_size, int qmode,
                        int dtype, void* stream);

/* Decode attention over a quantised cache: as pkv_paged_attention_decode
 * with K_t, V_t the dequantised values ((q - z) * s for INT4, e4m3 * s for
 * FP8), except that positions t < n_sink read sink_k/sink_v[b, t, kv_head]
 * (16-bit, row b of the sink buffers belongs to batch entry b), and, with
 * window > 0, the whole blocks from w0 = block_size * floor(max(ctx -
 * window, 0) / block_size) on read the 16-bit window ring win_k/win_v[b]
 * (see pkv_kv_append_quant; between window and window + block_size - 1
 * tokens).  q and out are 16-bit (dtype).  Supported: block_size 16, head_dim 128 or 64;
 * INT4 group_size == head_dim, or 64 at head_dim 128 (the pages' layout:
 * two (scale, zero) pairs per token and head); n_sink <= block_size (the
 * pages keep 8); 1 <= G <= 8. */
int pkv_paged_attention_decode_quant(const void* q, const void* k_codes, const void* k_scale,
                                     const void* k_zero, const void* v_codes, const void* v_scale,
                                     const void* v_zero, const void* sink_k, const void* sink_v,
                                     int32_t n_sink, const void* win_k, const void* win_v,
                                     int32_t window, const int32_t* block_tables,
                                     const int32_t* context_lens, int32_t batch,
                                     int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                     int32_t num_blocks, int32_t block_size, int32_t max_blocks,
                                     int32_t group_size, float scale, void* out, void* workspace,
                                     size_t workspace_bytes, int32_t partition_size, int qmode,
                                     int dtype, void* stream);

/* Copy-on-write block copy ("The 8GB VRAM Breakthrough", §3; "A Ideia de 60
 * Anos...", section "o bônus que paga o ingresso"): for each pair i,
 * block pairs[2i+1] of every pool becomes a byte copy of block pairs[2i].
 *   pools            host array of n_pools device pointers (1..8)
 *   bytes_per_block  host int64[n_pools], each a multiple of 16
 *   pairs            device int32 [n_pairs, 2] (src, dst)
 * Pairs outside [0, num_blocks) set PKV_STATUS_BAD_PAIR and are skipped.
 * Pairs must not chain (no dst used as another pair's src). */
int pkv_copy_blocks(void* const* pools, const int64_t* bytes_per_block, int32_t n_pools,
                    const int32_t* pairs, int32_t n_pairs, int32_t num_blocks, void* stream);

/* Read and clear the current device's status word (synchronises `stream`).
 * *status receives the PKV_STATUS_* bits seen since the last call; returns
 * PKV_ERR_DEVICE_BOUNDS if any bit was set, PKV_OK otherwise. */
int pkv_device_status(int32_t* status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
