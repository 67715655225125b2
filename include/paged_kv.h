/*
 * paged_kv.h -- C ABI of the GB300 (sm_103a) paged KV-cache library.
 *
 * The cache holds the keys and values of past tokens; each new token's
 * attention reads them again ("PagedAttention Nedir?", section "Once KV
 * Cache'i Anlamak Gerekir").  It is cut into fixed-size blocks of
 * block_size (= 16) tokens that may sit anywhere in a physical pool; a
 * per-sequence block table maps logical block i to a physical block id
 * ("Makale Bulteni -- PagedAttention ve vLLM", section "Iddia ve Gerceklik";
 * "PagedAttention Nedir?", section "PagedAttention Nasil Calisir?").  The
 * vAttention variant keeps each request's KV contiguous in virtual memory and
 * backs it with physical pages on demand ("Makale Bulteni -- vAttention",
 * section "Iddia ve Gerceklik: vAttention").
 *
 * Conventions for every call:
 *   - Returns a kv_status; never throws, never aborts the process.
 *   - Pointers documented "device" are CUDA device pointers (or managed /
 *     mapped memory) that stay valid until the work on `stream` completes;
 *     "host" pointers are read or written before the call returns.
 *   - Kernels run asynchronously on `stream` (a cudaStream_t passed as void*;
 *     NULL = the legacy default stream).
 *   - Argument errors detected on the host return KV_ERR_ARG or
 *     KV_ERR_UNSUPPORTED and launch nothing.  Errors the GPU detects
 *     (a block id or slot outside the pool, a position outside the mapped
 *     range, a pipeline wait that timed out) skip the offending element, let
 *     the kernel finish, and set bits in a device error word that
 *     kv_get_device_error / kv_contig_get_device_error read and clear.
 *   - A pool or contiguous context lives on the device that was current
 *     when it was created.  Every call that launches work or copies memory
 *     for it checks that this device is current; a call made while another
 *     device is current returns KV_ERR_ARG and launches nothing.  The
 *     destroy calls switch to the object's device to free it and switch back.
 *   - Host buffers.  The per-step arguments of paged_append_and_decode,
 *     paged_decode_attention_scheduled, kv_contig_append,
 *     contig_decode_attention and contig_append_and_decode (q, k_new, v_new,
 *     slot_mapping, positions, seq_lens, seq_order, schedule, out, lse_out)
 *     may be pinned host memory (cudaHostAlloc, cudaHostRegister) instead of
 *     device memory: the GPU reads and writes it directly over the host link
 *     (NVLink-C2C on GB300), with the same results as device buffers.  The host must not change
 *     such a buffer until the call has completed.  Block tables, request ids,
 *     the pool, the contexts' memory and workspaces are device memory.
 *   - Element types: KV_F32 (IEEE fp32), KV_BF16 (bfloat16) or KV_F16 (IEEE
 *     half precision).  q, k_new and v_new use the pool's type; out may be
 *     KV_F32 or the pool's type.  The cascade decode takes bf16 or fp16 pools.
 *   - head_dim must be 64 or 128, block_size must be 16, num_q_heads must be
 *     a multiple of num_kv_heads with num_q_heads / num_kv_heads <= 8.
 *
 * Pool layout (paged path): separate K and V arrays, each
 *     [num_blocks][num_kv_heads][block_size][head_dim]
 * so one (block, kv head) tile of 16 tokens is contiguous (4 KiB for bf16,
 * head_dim 128).  Slot s of the pool is block s / 16, offset s % 16.
 * Grouped-query attention: query head hq reads kv head hq / (Hq / Hkv).
 */
#ifndef PAGED_KV_H
#define PAGED_KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KV_OK = 0,
    KV_ERR_ARG = -1,            /* invalid argument (null pointer, bad size, bad id) */
    KV_ERR_OOM = -2,            /* no free block / device or physical memory exhausted */
    KV_ERR_UNSUPPORTED = -3,    /* shape or type outside what the kernels implement */
    KV_ERR_CUDA = -4,           /* a CUDA runtime or driver call failed */
    KV_ERR_DEVICE_BOUNDS = -5,  /* the GPU met an out-of-range block id, slot or position */
    KV_ERR_TIMEOUT = -6,        /* a bounded pipeline wait inside a kernel ran out */
    KV_ERR_STATE = -7           /* call not valid in the object's current state */
} kv_status;

/* Element types: IEEE fp32, bfloat16, IEEE half precision (binary16). */
typedef enum { KV_F32 = 0, KV_BF16 = 1, KV_F16 = 2 } kv_dtype;

/* Bits of the device error word. */
#define KV_DEVERR_BLOCK_RANGE 0x1   /* block-table entry outside [0, num_blocks) */
#define KV_DEVERR_SLOT_RANGE 0x2    /* slot_mapping entry >= num_blocks * block_size */
#define KV_DEVERR_TIMEOUT 0x4       /* an mbarrier wait exceeded its time limit */
#define KV_DEVERR_UNMAPPED 0x8      /* contiguous path: position beyond the mapped range */
#define KV_DEVERR_VALUE_RANGE 0x10  /* prefill: a V value of a key below the sequence length
                                       with |v| >= 65536 or infinite; the PV product, run on
                                       fp16 operands, used +-65504 in its place */

/* Default time limit of a pipeline wait inside a kernel (nanoseconds). */
#define KV_WAIT_LIMIT_DEFAULT_NS 2000000000ull

const char *kv_status_string(kv_status s);

/* Text of the last CUDA runtime error a call of this library met on the
 * calling thread (after a KV_ERR_CUDA or KV_ERR_OOM).  Owned by the library. */
const char *kv_last_cuda_error(void);

/* Number of blocks a sequence of n_tokens needs and the slots left unused in
 * its last block ("PagedAttention Nedir?", "Nasil Calisir?": 35 tokens at 16
 * per block need 3 blocks and leave 13 slots unused).  Host only. */
kv_status kv_blocks_for_tokens(int64_t n_tokens, int block_size, int64_t *blocks,
                               int64_t *unused_slots);

/* ======================================================================
 * Host block allocator: free list + reference counts.
 * "Makale Bulteni -- PagedAttention ve vLLM", "Iddia ve Gerceklik": when a
 * sequence's current block is full a free block is taken from the pool;
 * forked / branched sequences share blocks by pointer, copy-on-write.
 * "PagedAttention Nedir?", step 5: blocks no longer needed are reused.
 * Pure host code: usable without a GPU.  Not thread-safe.
 * ==================================================================== */
typedef struct kv_allocator *kv_allocator_t;

/* Creates an allocator over block ids 0..num_blocks-1, all free, handed out
 * in increasing id order.  *out owns host memory; free with
 * kv_allocator_destroy. */
kv_status kv_allocator_create(int num_blocks, kv_allocator_t *out);
kv_status kv_allocator_destroy(kv_allocator_t a);

/* Sets the order in which free blocks are handed out (a permutation of
 * 0..num_blocks-1, host array of n = num_blocks ids).  Only valid while every
 * block is free (KV_ERR_STATE otherwise). */
kv_status kv_allocator_set_order(kv_allocator_t a, const int32_t *order, int n);

/* Takes n free blocks (refcount becomes 1) into ids_out (host, n entries).
 * KV_ERR_OOM and no change if fewer than n are free. */
kv_status kv_allocator_alloc(kv_allocator_t a, int n, int32_t *ids_out);

/* refcount += 1 for each listed block (sharing a prefix, forking a
 * sequence).  Each id must be allocated (KV_ERR_ARG otherwise, no change). */
kv_status kv_allocator_share(kv_allocator_t a, int n, const int32_t *ids);

/* refcount -= 1 for each listed block; a block whose count reaches zero goes
 * back to the free list.  Freeing a free block is KV_ERR_ARG (no change). */
kv_status kv_allocator_free(kv_allocator_t a, int n, const int32_t *ids);

kv_status kv_allocator_refcount(kv_allocator_t a, int32_t id, int *refcount);
kv_status kv_allocator_num_free(kv_allocator_t a, int *num_free);

/* Host step of appending n_new tokens to one sequence (the block manager's
 * part of a decode or prefill step).
 *   table_row    host int32[max_blocks]: the sequence's block table row, updated
 *                in place;
 *   *num_blocks  blocks currently in the row (in/out);
 *   cur_len      tokens currently stored (positions 0..cur_len-1);
 *   slots_out    host int64[n_new]: pool slot of positions cur_len..cur_len+n_new-1;
 *   cow_src/cow_dst host int32[*n_cow] capacity; on return *n_cow pairs.
 * A new block is taken whenever a position opens one.  If a position falls in
 * an existing block whose refcount is > 1, that block is copied on write:
 * a fresh block is taken, the pair (old, new) is reported in cow_src/cow_dst,
 * the old block's refcount drops by one and the row points at the new block.
 * The caller must run kv_copy_blocks on the reported pairs before writing
 * the new tokens.  On KV_ERR_OOM (not enough free blocks) or KV_ERR_ARG
 * (row or cow capacity too small) nothing is changed. */
kv_status kv_prepare_append(kv_allocator_t a, int block_size, int32_t *table_row,
                            int max_blocks, int *num_blocks, int64_t cur_len, int n_new,
                            int64_t *slots_out, int32_t *cow_src, int32_t *cow_dst,
                            int *n_cow);

/* The host step of a whole batch in one call: kv_prepare_append for every
 * sequence b in order, with
 *   tables      host int32[batch][max_blocks] (rows updated in place);
 *   num_blocks  host int32[batch] (in/out);
 *   cur_lens    host int64[batch]; n_new host int32[batch];
 *   slots_out   host int64[sum n_new], sequence b's slots after those of b-1;
 *   cow_src/cow_dst host int32[*n_cow] capacity, *n_cow pairs on return.
 * The whole batch is planned before anything changes: on KV_ERR_OOM or
 * KV_ERR_ARG no table, count or refcount is modified.  A block shared by
 * several sequences of the batch is copied for every writer but the last. */
kv_status kv_prepare_append_batch(kv_allocator_t a, int block_size, int batch, int32_t *tables,
                                  int max_blocks, int32_t *num_blocks, const int64_t *cur_lens,
                                  const int32_t *n_new, int64_t *slots_out, int32_t *cow_src,
                                  int32_t *cow_dst, int *n_cow);

/* ======================================================================
 * Prefix cache ("PagedAttention Nedir?", "Prefix Sharing Nasil Calisir?":
 * the KV of a common prompt prefix is reused when the tokens and the context
 * before them match exactly; blocks are keyed by their contents plus the
 * preceding context).  Host only.
 *
 * Full blocks only.  Block i's key mixes block i-1's key with block i's token
 * ids; each entry also keeps its tokens and parent key and a lookup compares
 * them, so hash collisions cannot cause a false match.  The cache holds one
 * allocator reference on every block it lists; a match takes one more for
 * the caller (who frees it with kv_allocator_free like any block of its
 * table).  Not thread-safe.
 * ==================================================================== */
typedef struct kv_prefix_cache *kv_prefix_cache_t;

/* A cache listing at most capacity_blocks blocks of allocator a. */
kv_status kv_prefix_cache_create(kv_allocator_t a, int block_size, int capacity_blocks,
                                 kv_prefix_cache_t *out);
/* Drops the cache's references and frees the cache. */
kv_status kv_prefix_cache_destroy(kv_prefix_cache_t c);

/* Longest run of leading full blocks of tokens (host int32[n_tokens]) that
 * is cached: their ids go to blocks_out (host, up to max_blocks), each with
 * one more reference for the caller; *n_matched blocks. */
kv_status kv_prefix_cache_match(kv_prefix_cache_t c, const int32_t *tokens, int64_t n_tokens,
                                int32_t *blocks_out, int max_blocks, int *n_matched);

/* Lists the full blocks of a sequence (tokens host int32[n_tokens], blocks =
 * its table row, host int32[n_blocks]) for later matches, taking one
 * reference on each newly listed block.  Blocks already listed for the same
 * key keep the older copy.  At capacity, least recently used blocks that only
 * the cache holds are evicted first; if none can be, insertion stops.
 * *n_inserted (may be NULL) counts the new entries. */
kv_status kv_prefix_cache_insert(kv_prefix_cache_t c, const int32_t *tokens, int64_t n_tokens,
                                 const int32_t *blocks, int n_blocks, int *n_inserted);

/* Frees up to n_blocks listed blocks that nobody but the cache holds,
 * least recently used first. */
kv_status kv_prefix_cache_evict(kv_prefix_cache_t c, int n_blocks, int *n_freed);

kv_status kv_prefix_cache_stats(kv_prefix_cache_t c, int *cached_blocks, int64_t *lookups,
                                int64_t *hits);

/* ======================================================================
 * Device pool.
 * ==================================================================== */
typedef struct kv_pool *kv_pool_t;

/* Allocates the K and V pools (num_blocks * num_kv_heads * block_size *
 * head_dim elements each) on the current device, a device error word, and a
 * host allocator over the blocks.  Pool memory is uninitialised. */
kv_status kv_pool_create(int num_blocks, int block_size, int num_kv_heads, int head_dim,
                         kv_dtype dtype, kv_pool_t *out);
kv_status kv_pool_destroy(kv_pool_t p);

/* Device addresses of the K and V pools (owned by the pool). */
kv_status kv_pool_ptrs(kv_pool_t p, void **k_pool, void **v_pool);

/* The pool's allocator (borrowed; destroyed with the pool). */
kv_status kv_pool_allocator(kv_pool_t p, kv_allocator_t *out);

/* enable = 1: the tensor-core decode launches on this pool (paged decode,
 * the fused decode step, the scheduled decode) may begin while the previous
 * kernel in their stream is still running (a programmatic dependent launch).
 * The grid-indexed paged decode first reads its inputs that a decode step
 * never writes -- the block tables, seq_lens, seq_order and q -- and then
 * waits for that kernel to complete before it touches the pool, the
 * workspace, the outputs or the new rows; the scheduled decode waits before
 * it reads anything.  So the kernel launched right before such a decode must
 * not write those four inputs (a decode step does not; a copy in the stream
 * between the two launches ends the overlap anyway).  Results are unchanged
 * and the launch latency between back-to-back steps is hidden.  enable = 0
 * (the default): ordinary launches.  Host only; takes effect from the next
 * call. */
kv_status kv_pool_set_launch_overlap(kv_pool_t p, int enable);

/* Block manager calls on the pool's own allocator ("Makale Bulteni --
 * PagedAttention ve vLLM", "Iddia ve Gerceklik": blocks come from a free
 * pool on demand, are shared between sequences by reference and are copied
 * on write).  Host only, like the kv_allocator_* calls they wrap:
 *   kv_alloc_blocks   n free blocks (refcount 1) into ids_out; KV_ERR_OOM
 *                     (nothing taken) if fewer are free;
 *   kv_share_blocks   one more reference on each listed block;
 *   kv_free_blocks    one reference fewer; a block reaching 0 is free again. */
kv_status kv_alloc_blocks(kv_pool_t p, int n, int32_t *ids_out);
kv_status kv_share_blocks(kv_pool_t p, int n, const int32_t *ids);
kv_status kv_free_blocks(kv_pool_t p, int n, const int32_t *ids);

/* Copy-on-write of one block before a write into it: if *block_id_inout is
 * held by more than one reference, a free block is taken, the whole block
 * (all heads and slots of K and V) is copied into it on `stream`, the old
 * block loses this caller's reference, *block_id_inout becomes the new id
 * and *copied = 1.  A block held once is left as is (*copied = 0).
 * KV_ERR_ARG for a free or out-of-range id; KV_ERR_OOM (nothing changed)
 * when no block is free.  Batches: kv_prepare_append_batch + kv_copy_blocks. */
kv_status kv_cow_if_shared(kv_pool_t p, int32_t *block_id_inout, int *copied, void *stream);

/* KV append: writes the new tokens' keys and values into their pool slots
 * ("Makale Bulteni -- PagedAttention ve vLLM", "Iddia ve Gerceklik";
 * "PagedAttention Nedir?", "Nasil Calisir?" steps 1-3).
 *   k_new, v_new   device [num_tokens][num_kv_heads][head_dim], pool dtype;
 *   slot_mapping   device int64[num_tokens]; a negative slot is skipped; a
 *                  slot >= num_blocks*block_size is skipped and sets
 *                  KV_DEVERR_SLOT_RANGE.
 * Exact byte copy.  Two tokens naming the same slot: unspecified winner. */
kv_status kv_append(kv_pool_t p, const void *k_new, const void *v_new,
                    const int64_t *slot_mapping, int num_tokens, void *stream);

/* Copy-on-write block copies: for i < n, every head and slot of K and V of
 * block src[i] is copied to block dst[i] (device int32 arrays).  Pairs must
 * not overlap (no dst is another pair's src).  Out-of-range ids are skipped
 * and set KV_DEVERR_BLOCK_RANGE. */
kv_status kv_copy_blocks(kv_pool_t p, const int32_t *src, const int32_t *dst, int n,
                         void *stream);

/* Swap / preemption ("Makale Bulteni -- PagedAttention ve vLLM", "Iddia ve
 * Gerceklik": when GPU memory is full, blocks are moved to CPU memory).
 * kv_swap_out copies every head and slot of K and V of the listed blocks
 * (device int32[n]) into host_buf, laid out [n][K then V][num_kv_heads][16]
 * [head_dim]; kv_swap_in copies them back into the listed blocks (which may
 * differ from the ones swapped out).  host_buf must be addressable by the GPU
 * (pinned host memory: cudaHostAlloc / cudaHostRegister, or a torch pinned
 * tensor), 16-byte aligned, kv_swap_bytes(n) long; a kernel reads / writes it
 * directly, so on this machine the bytes cross NVLink-C2C.  Out-of-range ids
 * are skipped and set KV_DEVERR_BLOCK_RANGE.  The refcounts are the caller's
 * business: swap out, kv_allocator_free; later alloc + swap in. */
kv_status kv_swap_out(kv_pool_t p, const int32_t *block_ids, int n, void *host_buf, void *stream);
kv_status kv_swap_in(kv_pool_t p, const int32_t *block_ids, int n, const void *host_buf,
                     void *stream);
kv_status kv_swap_bytes(kv_pool_t p, int n, size_t *bytes);

/* Scratch memory the decode call needs for a split plan: partial outputs
 * fp32 [batch][num_q_heads][splits][head_dim] and their log-sum-exp
 * [batch][num_q_heads][splits].  num_splits as in paged_decode_attention
 * (0 = automatic).  Host only. */
kv_status kv_decode_workspace_size(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                   int max_blocks, int num_splits, size_t *bytes);

/* The split plan paged_decode_attention / contig_decode_attention will use:
 * each sequence's tokens are cut into partitions of *part_blocks blocks
 * (16 tokens each), at most *max_splits per sequence.  Host only. */
kv_status kv_decode_split_plan(int batch, int num_kv_heads, int max_blocks, int num_splits,
                               int *part_blocks, int *max_splits);

/* Chooses num_splits for paged_decode_attention / contig_decode_attention
 * from the sequence lengths as the host knows them (a serving host keeps its
 * own block tables, so it has them).  host_seq_lens: host int32[batch].
 * The bf16 / head_dim 128 decode runs partitions of 256 blocks or more with a
 * deep copy ring at three CTAs per SM, shorter ones at five CTAs per SM.  The
 * plan prefers one wave: the smallest long partitions whose CTAs fit in at
 * most 2.4 per SM (measured to stream fastest), else the smallest short
 * partitions that fit in five per SM; when no split fits, the largest
 * partitions that still give several full waves.  The result depends only on
 * the lengths, the batch shape and the SM count.  Host only; *num_splits >= 1. */
kv_status kv_decode_plan(const int32_t *host_seq_lens, int batch, int num_kv_heads,
                         int max_blocks, int *num_splits);

/* The batch's sequences ordered by length, longest first (ties in batch
 * order), for the seq_order argument of paged_append_and_decode.  Host only:
 * host_seq_lens and order_out are host int32[batch]. */
kv_status kv_decode_order(const int32_t *host_seq_lens, int batch, int32_t *order_out);

/* Paged decode attention: one query token per sequence attends all
 * seq_lens[b] tokens of its cache, reading K/V blocks through the block
 * table ("PagedAttention Nedir?", "Nasil Calisir?" step 4), with
 *     o = softmax(scale * q K^T) V,   lse = log sum_j exp(scale * q.k_j).
 *   q             device [batch][num_q_heads][head_dim], pool dtype;
 *   block_tables  device int32[batch][max_blocks]; entries at index >=
 *                 ceil(seq_lens[b]/16) are never read;
 *   seq_lens      device int32[batch], 0 <= seq_lens[b] <= max_blocks*16;
 *   out           device [batch][num_q_heads][head_dim] of out_dtype;
 *   lse_out       device fp32[batch][num_q_heads] or NULL;
 *   num_splits    0 = automatic; else the number of partitions the longest
 *                 possible sequence (max_blocks blocks) is cut into;
 *   workspace     device scratch of at least kv_decode_workspace_size bytes
 *                 (may be NULL when that size is 0).
 * An empty sequence gives out = 0 and lse = -inf.  The result does not depend
 * on where the blocks sit in the pool (bit-identical for any placement).
 * Decode calls on one pool must not run concurrently on the GPU (the fused
 * split merge uses the pool's arrival counters): order them on one stream. */
kv_status paged_decode_attention(kv_pool_t p, const void *q, const int32_t *block_tables,
                                 int max_blocks, const int32_t *seq_lens, int batch,
                                 int num_q_heads, float scale, void *out, kv_dtype out_dtype,
                                 float *lse_out, int num_splits, void *workspace,
                                 size_t workspace_bytes, void *stream);

/* One decode step: kv_append of one new token per sequence followed by
 * paged_decode_attention ("PagedAttention Nedir?", "Nasil Calisir?": the
 * new token's KV is written into its block, then the step attends all
 * tokens).  Same results as those two calls (the pool receives the same
 * bytes, the output is bit-identical).
 *   k_new, v_new   device [batch][num_kv_heads][head_dim], pool dtype, 16-byte
 *                  aligned: the token appended to each sequence;
 *   slot_mapping   device int64[batch]: its slot; negative = none.  The slot
 *                  must be position seq_lens[b] - 1 of sequence b (seq_lens
 *                  count the new token) in a block only sequence b holds
 *                  (copy shared blocks first: kv_cow_if_shared / kv_copy_blocks).
 *   seq_order      device int32[batch] or NULL: a permutation of the batch,
 *                  the order in which the kernel's grid takes the sequences
 *                  (kv_decode_order: longest first, so one wave of CTAs loads
 *                  the SMs evenly).  It changes no result.
 * Other arguments as paged_decode_attention.  For bf16 pools with head_dim
 * 128 and >= 3 query heads per kv head the append is fused into the decode
 * kernel (one launch); other shapes run the two calls. */
kv_status paged_append_and_decode(kv_pool_t p, const void *q, const void *k_new,
                                  const void *v_new, const int64_t *slot_mapping,
                                  const int32_t *block_tables, int max_blocks,
                                  const int32_t *seq_lens, const int32_t *seq_order, int batch,
                                  int num_q_heads, float scale,
                                  void *out, kv_dtype out_dtype, float *lse_out, int num_splits,
                                  void *workspace, size_t workspace_bytes, void *stream);

/* Balanced work schedule for paged_decode_attention_scheduled (the pages fix
 * no schedule: this is how this library spreads a decode step over the GPU).
 * The grid-indexed plan gives every (sequence, kv head, split) its own CTA,
 * so CTAs differ in length as the sequences do and a single wave ends with
 * the longest.  Here the blocks of all (sequence, kv head) pairs are laid end
 * to end and cut into C runs of equal length, one per CTA of a single wave
 * (five CTAs per SM, or 2.4 per SM with the deep ring when every run has at
 * least 256 blocks); a run that crosses pairs is several pieces, which the CTA
 * streams one after the other.  A pair's pieces are its split-KV partitions
 * (at most 32, merged inside the kernel).
 *   host_seq_lens  host int32[batch]: the lengths the decode will see on the
 *                  device (a decode step: after its append);
 *   num_sms        SMs to plan for, 0 = the current device's;
 *   num_ctas       0 = the rule above; else this many CTAs (at most one wave:
 *                  5 per SM with 4 ring stages, 3 per SM with 8);
 *   ring_stages    0 = the rule above; else 4 (the wide kernel) or 8 (the
 *                  deep ring);
 *   flags          0, or KV_SCHED_WHOLE_PIECES: instead of equal runs, each
 *                  (sequence, kv head) is cut into ceil(n / W) pieces of
 *                  near-equal length, one CTA per piece, the CTAs ordered
 *                  longest piece first (no CTA streams two pieces; the grid
 *                  is then a little more than one wave);
 *   schedule_out   host int32[capacity_ints]; *used_ints receives the words
 *                  written (the caller copies that many to the device).
 * Capacity: kv_decode_schedule_capacity's bound for this batch shape.  Host
 * only.  KV_ERR_UNSUPPORTED when a sequence would need more than 32 pieces
 * (more than 31 x 1024 blocks). */
kv_status kv_decode_schedule_capacity(int batch, int num_kv_heads, int max_blocks, int num_sms,
                                      size_t *ints);
#define KV_SCHED_WHOLE_PIECES 1
kv_status kv_decode_schedule(const int32_t *host_seq_lens, int batch, int num_kv_heads,
                             int max_blocks, int num_sms, int num_ctas, int ring_stages, int flags,
                             int32_t *schedule_out, size_t capacity_ints, size_t *used_ints);
/* Workspace bytes paged_decode_attention_scheduled needs with this schedule
 * (its host copy). */
kv_status kv_decode_schedule_workspace_size(const int32_t *host_schedule, int num_q_heads,
                                            int head_dim, size_t *bytes);

/* Paged decode attention (and, with k_new non-NULL, the decode step's append
 * of one token per sequence, as paged_append_and_decode) run on a balanced
 * schedule from kv_decode_schedule.  Same maths as paged_decode_attention;
 * the split points differ from the grid-indexed plan's, so results agree
 * within rounding, not bit for bit (they are bit-identical from one call to
 * the next with the same schedule).
 *   host_schedule  the host array kv_decode_schedule filled (its header is
 *                  read here);
 *   schedule       its device copy, 16-byte aligned, all used words;
 *   k_new, v_new, slot_mapping  as paged_append_and_decode, or k_new = NULL
 *                  for no append.
 * Other arguments as paged_decode_attention.  Requires pool dtype KV_BF16 or
 * KV_F16, head_dim 128, 3..8 query heads per kv head and batch *
 * num_kv_heads <= 65536, else KV_ERR_UNSUPPORTED.  Device lengths that do not match the
 * schedule's (a piece past a sequence's end, or a sequence's last piece
 * stopping short of it) are recorded as KV_ERR_DEVICE_BOUNDS; nothing outside
 * the sequence's table row and the pool is read. */
kv_status paged_decode_attention_scheduled(kv_pool_t p, const void *q, const void *k_new,
                                           const void *v_new, const int64_t *slot_mapping,
                                           const int32_t *block_tables, int max_blocks,
                                           const int32_t *seq_lens, int batch, int num_q_heads,
                                           float scale, const int32_t *host_schedule,
                                           const int32_t *schedule, void *out, kv_dtype out_dtype,
                                           float *lse_out, void *workspace,
                                           size_t workspace_bytes, void *stream);

/* paged_decode_attention without a workspace argument, for callers that
 * cannot allocate device memory where they run decode (a plugin whose host
 * framework owns all device memory; a serving loop that must not call
 * cudaMalloc after start-up).  The pages have no counterpart: this is a
 * packaging choice of this library.
 *
 * Same arguments, maths and results as paged_decode_attention with the same
 * num_splits.  The split-KV partial results live in one fixed 8 MiB array in
 * the library's device image (held on every GPU that loads the library until
 * the process exits).  A split plan needing more scratch than that
 * (kv_decode_workspace_size > 8 MiB) returns KV_ERR_UNSUPPORTED and launches
 * nothing.  The call itself allocates nothing.  The first call on each device
 * looks up the array's device address (cudaGetSymbolAddress, with that device
 * current); make that first call before any stream capture.  All calls share
 * the array: calls whose kernels overlap on the GPU (unordered streams) race
 * and give undefined results.  Nothing in the array has to start at zero. */
kv_status paged_decode_attention_noalloc(kv_pool_t p, const void *q, const int32_t *block_tables,
                                         int max_blocks, const int32_t *seq_lens, int batch,
                                         int num_q_heads, float scale, void *out,
                                         kv_dtype out_dtype, float *lse_out, int num_splits,
                                         void *stream);

/* Cascade decode over shared prefixes ("PagedAttention Nedir?", "Prefix
 * Sharing Nasil Calisir?"; "Makale Bulteni -- PagedAttention ve vLLM",
 * "Ticari Etki": sequences that start alike hold that part of the cache once,
 * as the same physical blocks).  Same result as paged_decode_attention (exact
 * maths; rounding differs), but each group's shared blocks are read once for
 * all its sequences instead of once per sequence.
 *
 *   group_seqs     device int32[num_groups][group_size]: the sequences of
 *                  each group (batch indices), -1 for an empty slot; a
 *                  sequence belongs to at most one group;
 *   shared_tokens  device int32[batch]: tokens at the start of sequence b that
 *                  it reads through its group's shared blocks, rounded down to
 *                  whole blocks and clamped to seq_lens[b]; 0 for a sequence
 *                  in no group.  The blocks are read from the table row of the
 *                  member with the most shared tokens; every member's row must
 *                  hold the same block ids for its own shared blocks;
 *   max_prefix_blocks  upper bound of any group's shared blocks (host-known;
 *                  <= max_blocks).  A group with more sets
 *                  KV_DEVERR_BLOCK_RANGE and its excess is not attended;
 *   prefix_splits  0 = automatic (kv_cascade_plan), else the number of
 *                  key-range partitions of each group's prefix;
 *   num_splits, workspace: as paged_decode_attention, for the suffix (the
 *                  blocks after each sequence's shared part); the workspace
 *                  must hold kv_cascade_workspace_size bytes;
 *   seq_order      device int32[batch] or NULL: the order in which the suffix
 *                  grid takes the sequences (as paged_append_and_decode; e.g.
 *                  kv_cascade_order of the suffix lengths).
 * Other arguments as paged_decode_attention.  Requires pool dtype KV_BF16 or
 * KV_F16, head_dim 128, out_dtype KV_F32 or the pool's type and
 * group_size * (num_q_heads / num_kv_heads) <= 128, else KV_ERR_UNSUPPORTED.
 * The prefix kernel multiplies its softmax weights, split into two parts of
 * the pool's type (about 16 significant bits with bf16, 22 with fp16), by V in
 * that type.  Two kernels run in stream order: the prefix kernel
 * (tcgen05; rows = a group's sequences x the query heads of one kv head) and
 * the decode kernel over the suffixes, whose split-KV merge also takes the
 * prefix's partial results. */
kv_status kv_cascade_plan(int num_groups, int num_kv_heads, int max_prefix_blocks, int requested,
                          int *prefix_splits);
/* A seq_order for paged_decode_attention_cascade's suffix grid, from the
 * number of tokens each sequence attends after its shared part (host int32
 * host_suffix_lens[batch]; order_out: host int32[batch]).  Sequences with more
 * than one block (16 tokens) of their own come longest first (ties in batch
 * order); those with at most one block, whose CTAs are mostly start-up and
 * merge latency, come as one run (longest first) after the first 40%
 * (rounded) of the others, so that they overlap the long ones' streaming
 * instead of forming the grid's tail.  The pages fix no order; the rule is
 * this library's, measured on GB300 (the shared-prefix step's decode 0.077 ms
 * against 0.085 ms longest first).  Host only. */
kv_status kv_cascade_order(const int32_t *host_suffix_lens, int batch, int32_t *order_out);
kv_status kv_cascade_workspace_size(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                    int max_blocks, int num_splits, int prefix_splits,
                                    size_t *bytes);
kv_status paged_decode_attention_cascade(
    kv_pool_t p, const void *q, const int32_t *block_tables, int max_blocks, const int32_t *seq_lens,
    int batch, int num_q_heads, float scale, const int32_t *group_seqs, int num_groups,
    int group_size, const int32_t *shared_tokens, int max_prefix_blocks, int prefix_splits,
    void *out, kv_dtype out_dtype, float *lse_out, int num_splits, const int32_t *seq_order,
    void *workspace, size_t workspace_bytes, void *stream);

/* Chunked causal paged prefill ("Makale Bulteni -- vAttention", "Iddia ve
 * Gerceklik": the prefill kernels are where paging costs most).  Sequence b
 * holds seq_lens[b] tokens in the cache, the last T_b = cu_q[b+1] - cu_q[b]
 * of which are the new chunk (already appended with kv_append).  Query row
 * r = cu_q[b] + i sits at position (seq_lens[b] - T_b) + i and attends keys
 * 0..(seq_lens[b] - T_b) + i.  QK^T and PV run on the tcgen05 tensor cores
 * with fp32 accumulation in tensor memory.  QK^T multiplies q by K in the
 * pool's type.  PV multiplies the softmax weights, rounded to fp16, by V in
 * fp16; a bf16 pool's V is converted in shared memory, exactly for
 * magnitudes up to 65280, and larger attended values are handled as
 * KV_DEVERR_VALUE_RANGE describes.  Requires pool dtype KV_BF16 or KV_F16
 * and head_dim 128.  The query tiles of a chunk are launched last (heaviest)
 * first.
 *   q         device [total_q][num_q_heads][head_dim], the pool's type;
 *   cu_q      device int32[batch + 1], cu_q[0] = 0, non-decreasing, cu_q[batch]
 *             <= total_q;
 *   total_q   host: rows of q and out;
 *   max_q_len host: max_b T_b (sizes the grid);
 *   out       device [total_q][num_q_heads][head_dim] of out_dtype; rows not
 *             covered by any chunk are left untouched;
 *   lse_out   device fp32[total_q][num_q_heads] or NULL.
 * A sequence with seq_lens[b] < T_b, seq_lens[b] > max_blocks*16 or a chunk
 * past total_q is skipped and sets KV_DEVERR_BLOCK_RANGE; so does an
 * out-of-range block id (its keys read as zeros).  Returns KV_ERR_ARG for a
 * NULL pointer, a negative size, num_q_heads not a multiple of the pool's kv
 * heads or q not 16-byte aligned, and KV_ERR_UNSUPPORTED for another pool
 * type or head_dim, an out_dtype other than KV_F32 or the pool's type,
 * batch > 65535, max_q_len > 65535 * 256, or a pool of more than 2^31 - 1
 * (block, kv head, token) rows. */
kv_status paged_prefill_attention(kv_pool_t p, const void *q, const int32_t *cu_q, int total_q,
                                  int max_q_len, const int32_t *block_tables, int max_blocks,
                                  const int32_t *seq_lens, int batch, int num_q_heads,
                                  float scale, void *out, kv_dtype out_dtype, float *lse_out,
                                  void *stream);

/* Synchronises `stream`, returns the device error word in *code (0 = none)
 * and clears it.  Returns KV_ERR_TIMEOUT if the timeout bit is set, else
 * KV_ERR_UNSUPPORTED if only KV_DEVERR_VALUE_RANGE is set, else
 * KV_ERR_DEVICE_BOUNDS if any bit is set, KV_OK otherwise. */
kv_status kv_get_device_error(kv_pool_t p, int *code, void *stream);

/* ======================================================================
 * Contiguous (vAttention-style) KV path.  "Makale Bulteni -- vAttention",
 * "Iddia ve Gerceklik: vAttention": for each request a contiguous virtual
 * range large enough for the maximum context is reserved
 * (cuMemAddressRangeReserve) without using physical memory; physical pages
 * are created and mapped (cuMemCreate, cuMemMap) only as the request grows,
 * so the attention kernel sees one contiguous tensor per request.
 *
 * Per-request layout: K region [num_kv_heads][head_stride][head_dim] followed
 * by the V region of the same shape, where head_stride >= max_tokens is
 * max_tokens rounded up to whole physical pages (kv_contig_layout).
 * Physical pages are the driver's minimum granularity (2 MiB on current
 * GPUs); each mapped page of every head's K and V region is its own physical
 * allocation.
 * ==================================================================== */
typedef struct kv_contig *kv_contig_t;

/* Creates a context for up to max_requests requests of up to max_tokens
 * tokens on the current device.  Reserves nothing yet. */
kv_status kv_contig_create(int max_requests, int max_tokens, int num_kv_heads, int head_dim,
                           kv_dtype dtype, kv_contig_t *out);
/* Unmaps, releases and frees everything the context holds. */
kv_status kv_contig_destroy(kv_contig_t c);

/* Layout facts: tokens per head region (head_stride), bytes of one physical
 * page, bytes of virtual range reserved per request. */
kv_status kv_contig_layout(kv_contig_t c, int64_t *head_stride, int64_t *page_bytes,
                           int64_t *reserved_bytes_per_request);

/* Reserves request req's virtual range (cuMemAddressRangeReserve).  No
 * physical memory is used.  KV_ERR_STATE if already reserved. */
kv_status kv_contig_reserve(kv_contig_t c, int req);

/* Makes positions 0..n_tokens-1 of every head of request req backed by
 * physical pages (cuMemCreate + cuMemMap + cuMemSetAccess for pages not yet
 * mapped).  Synchronous host call.  KV_ERR_OOM if physical memory runs out
 * (pages mapped by this call are undone). */
kv_status kv_contig_ensure(kv_contig_t c, int req, int64_t n_tokens);

/* Unmaps and releases all physical pages of request req and frees its
 * virtual range.  The caller must have finished all work that uses it. */
kv_status kv_contig_release(kv_contig_t c, int req);

/* Keeps physical pages ready off the request path ("Makale Bulteni --
 * vAttention", "Iddia ve Gerceklik": background pre-allocation and deferred
 * reclamation hide the VMM-call latency).  With low > 0 a background thread
 * creates pages (cuMemCreate) whenever fewer than `low` are spare, up to
 * `high`; kv_contig_ensure then only maps.  kv_contig_release hands its
 * pages back to the spare set (up to `high`) instead of releasing them.
 * (0, 0) stops the thread and releases every spare page.  Spare pages count
 * as used device memory. */
kv_status kv_contig_page_pool(kv_contig_t c, int low, int high);

/* Spare pages now, pages created and spare pages reused so far, and the mean
 * host time per page of mapping (kv_contig_ensure) and unmapping
 * (kv_contig_release). */
kv_status kv_contig_page_stats(kv_contig_t c, int *spare_pages, int64_t *created, int64_t *reused,
                               double *map_us_per_page, double *unmap_us_per_page);

/* Device base addresses of request req's K and V regions. */
kv_status kv_contig_ptrs(kv_contig_t c, int req, void **k_base, void **v_base);

/* Mapped tokens of request req and physical bytes mapped over all requests. */
kv_status kv_contig_stats(kv_contig_t c, int req, int64_t *mapped_tokens,
                          int64_t *mapped_bytes_total);

/* Append on the contiguous path: token t's K/V go to position positions[t]
 * of request req_ids[t] (device int32 arrays).  A position at or beyond the
 * request's mapped range, or an unreserved request, is skipped and sets
 * KV_DEVERR_UNMAPPED. */
kv_status kv_contig_append(kv_contig_t c, const void *k_new, const void *v_new,
                           const int32_t *req_ids, const int32_t *positions, int num_tokens,
                           void *stream);

/* Decode attention over the contiguous layout: sequence b is request
 * req_ids[b] (device int32[batch]) with seq_lens[b] tokens.  Same maths and
 * arguments as paged_decode_attention; max_tokens plays the role of
 * max_blocks*16 in the split plan, so with the same num_splits and a table
 * width of ceil(max_tokens/16) both paths cut the keys identically and give
 * bit-identical results.  seq_lens[b] beyond the mapped range sets
 * KV_DEVERR_UNMAPPED and is clamped. */
kv_status contig_decode_attention(kv_contig_t c, const void *q, const int32_t *req_ids,
                                  const int32_t *seq_lens, int batch, int num_q_heads,
                                  float scale, void *out, kv_dtype out_dtype, float *lse_out,
                                  int num_splits, void *workspace, size_t workspace_bytes,
                                  void *stream);

/* One decode step on the contiguous path: each sequence's new token (device
 * k_new / v_new [batch][num_kv_heads][head_dim], the context's type) goes to
 * position seq_lens[b] - 1 of request req_ids[b] (mapped beforehand with
 * kv_contig_ensure), then contig_decode_attention attends all seq_lens[b]
 * tokens ("Makale Bulteni -- vAttention", "Iddia ve Gerceklik: vAttention":
 * the request's KV grows in place at the end of its contiguous range).  Same
 * results as kv_contig_append at those positions followed by
 * contig_decode_attention.  One launch where the tensor-core decode applies
 * (16-bit storage, head_dim 128, 3..8 query heads per kv head): the last
 * partition of each (sequence, kv head) writes the row and patches it into
 * its own copy of the last block; otherwise the two calls.  A sequence with
 * seq_lens[b] = 0 has no new token; one beyond the mapped range sets
 * KV_DEVERR_UNMAPPED and appends nothing. */
kv_status contig_append_and_decode(kv_contig_t c, const void *q, const void *k_new,
                                   const void *v_new, const int32_t *req_ids,
                                   const int32_t *seq_lens, int batch, int num_q_heads,
                                   float scale, void *out, kv_dtype out_dtype, float *lse_out,
                                   int num_splits, void *workspace, size_t workspace_bytes,
                                   void *stream);

kv_status kv_contig_get_device_error(kv_contig_t c, int *code, void *stream);

/* As kv_pool_set_launch_overlap for a contiguous context: kv_contig_append and
 * the tensor-core contig_decode_attention / contig_append_and_decode may begin
 * while the previous kernel in their stream still runs, and wait for it before
 * touching memory.  Off by default.  Host only. */
kv_status kv_contig_set_launch_overlap(kv_contig_t c, int enable);

/* ======================================================================
 * Test hooks: failure paths made reachable without faulting a GPU.  Not for
 * production use.
 * ==================================================================== */

/* Every pipeline wait inside the kernels (for data a producer has to
 * deliver, or a stage a consumer has to release) gives up after
 * KV_WAIT_LIMIT_DEFAULT_NS, records KV_DEVERR_TIMEOUT and lets its kernel run
 * to the end.  This sets that limit for kernels launched afterwards on the
 * current device: 0 makes every wait that is not satisfied at its first poll
 * give up; KV_WAIT_LIMIT_DEFAULT_NS restores the default.  A warp's wait for
 * its own copies or tensor-core operations before its CTA ends keeps the
 * default in all cases, so nothing is in flight when the memory they write is
 * released.  Results of a call that timed out are undefined; the next
 * kv_get_device_error returns KV_ERR_TIMEOUT and clears the state a merge may
 * have left. */
kv_status kv_debug_set_wait_limit_ns(uint64_t ns);

/* Contiguous path: of the physical page creations kv_contig_ensure makes from
 * now on (pages taken from the background pool do not count), the one after
 * `after` more successful ones fails as if the device had no memory left, once.
 * kv_contig_ensure then unmaps what that call had mapped and returns
 * KV_ERR_OOM.  A negative `after` cancels a pending failure. */
kv_status kv_debug_fail_page_create(int after);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_KV_H */
