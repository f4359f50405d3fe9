/*
 * pagedkv.h -- C ABI of libpagedkv.so: the decode-phase hot path of paged KV
 * caching (PagedAttention), for NVIDIA GB300 (sm_103a).
 *
 * The operations, and where they are defined:
 *   - pkv_paged_attention_decode: exact single-query attention of every
 *     sequence over its K/V, which sit in fixed-size blocks scattered through
 *     a preallocated pool and are reached through a per-sequence block table.
 *     "Efficient Memory Management for Large Language Model Serving with
 *     PagedAttention" (wywy.jp notes), glossary entries "PagedAttention" and
 *     "Block table"; zhaifeiyue.github.io detail page, the block-indexed
 *     attention formula (paper section 4.1) and its equivalence to standard
 *     attention; ricepunchb garden "KV Cache Optimization", section 3.3 (each
 *     block's scores at kernel level, a final reduction completes the softmax).
 *   - pkv_reshape_and_cache: the write of each new token's K and V into the
 *     slot the block manager assigned (wywy.jp notes, autoregressive
 *     generation phase: only the new token's K/V is produced per iteration;
 *     garden section 3.2: slot = table[pos / B] * B + pos mod B).
 *   - pkv_copy_blocks: the block engine's block-granular copy used by
 *     copy-on-write (wywy.jp notes, parallel sampling walkthrough; detail
 *     page, Memory Management table, "Copy-on-Write: one block").
 *   - pkv_bm_*: the host KV block manager -- free list, reference counts,
 *     on-demand allocation, fork and copy-on-write of the last shared block
 *     (wywy.jp notes, "KV cache manager", "Reference count", "Copy-on-write";
 *     detail page, Memory Management table: Allocate / Free / Copy-on-Write).
 *
 * Memory layout (all 16-bit element types; the pages leave layout open):
 *   k_cache, v_cache  [num_blocks][num_heads][block_size][head_dim]   one pool each;
 *                     one physical block id addresses both pools (the paper
 *                     keeps K and V in separate blocks with their own tables;
 *                     two identical tables are read as one).
 *   q, out            [num_seqs][num_heads][head_dim]
 *   k, v (new tokens) [num_tokens][num_heads][head_dim]
 *   block_tables      int32 [num_seqs][max_blocks_per_seq]; row s lists the
 *                     physical blocks of sequence s in logical order; entries
 *                     past ceil(context_lens[s] / block_size) are never read.
 *   context_lens      int32 [num_seqs]: tokens sequence s attends (its newest
 *                     token, the query's own, included).
 *   slot_mapping      int64 [num_tokens]: physical block * block_size + offset,
 *                     or a negative value for "do not write".
 *   pairs             int32 [num_pairs][2] = (src, dst) physical block ids.
 *
 * Supported shapes: head_dim 64 or 128; block_size 8, 16, 32 or 64; fp16 or
 * bf16 storage; fp32 arithmetic; K/V heads == query heads.
 *
 * Ownership and execution: every pointer passed to a kernel entry point is a
 * device pointer owned by the caller and must stay valid until the work on
 * `stream` completes; calls are asynchronous on `stream`.  The library never
 * allocates device memory: the decode entry point takes a caller-provided
 * workspace (size from pkv_decode_workspace_size).  q/out/k/v/caches must be
 * 16-byte aligned, the workspace 256-byte aligned.
 *
 * Errors: argument problems found on the host return PKV_ERR_INVALID and
 * launch nothing; a failed launch returns PKV_ERR_CUDA; in both cases
 * pkv_last_error() (thread-local) describes it.  Kernels validate every block
 * id, slot and context length they use: a bad value is skipped or clamped
 * (never dereferenced) and sets a bit in the library's device error word,
 * which pkv_get_device_error reads.  Kernels never wait without a bound: a
 * wait that runs out sets PKV_DEVERR_TIMEOUT and the kernel returns.
 */
#ifndef PAGEDKV_H
#define PAGEDKV_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PKV_OK = 0,
    PKV_ERR_INVALID = 1,   /* bad argument, nothing launched / state unchanged */
    PKV_ERR_CUDA = 2,      /* a CUDA runtime call or launch failed */
    PKV_ERR_OOM = 3,       /* block manager: not enough free physical blocks */
    PKV_ERR_DEVICE = 4     /* pkv_get_device_error found device-side error bits */
} pkv_status;

typedef enum { PKV_F16 = 0, PKV_BF16 = 1 } pkv_dtype;

/* bits of the device error word */
#define PKV_DEVERR_BAD_BLOCK   1  /* a block id outside [0, num_blocks) was read */
#define PKV_DEVERR_BAD_SLOT    2  /* a slot >= num_blocks * block_size was given */
#define PKV_DEVERR_BAD_CONTEXT 4  /* context_lens[s] < 0 or > max_blocks_per_seq * block_size */
#define PKV_DEVERR_TIMEOUT     8  /* a bounded wait inside a kernel ran out */
#define PKV_DEVERR_WORKSPACE  16  /* the workspace was too small for the launch */

/* Largest grid the decode kernel uses (CTAs); bounds the workspace. */
#define PKV_MAX_GRID 4096
/* Largest batch of sequences per decode call. */
#define PKV_MAX_SEQS 16384

/* ------------------------------------------------------------------------ */
/* Decode attention                                                          */
/* ------------------------------------------------------------------------ */

/*
 * Bytes of workspace pkv_paged_attention_decode needs for these sizes.
 * partition_size: split length in tokens of the split-K pass, or 0 for the
 * balanced split (each CTA of a persistent grid takes an equal share of the
 * batch's K/V).  A nonzero value must be a positive multiple of the kernel's
 * step: 16 tokens for head_dim 128, 32 for head_dim 64 (4 KiB of K per step,
 * gathered from several blocks when block_size is smaller).  Host only; never
 * touches the GPU.
 */
pkv_status pkv_decode_workspace_size(int num_seqs, int num_heads, int head_dim,
                                     int block_size, int max_blocks_per_seq,
                                     int partition_size, size_t* bytes);

/*
 * out[s][h][:] = sum_t softmax_t(scale * q[s][h] . K_s[t][h]) V_s[t][h] over
 * t < context_lens[s], where K_s[t] = k_cache[block_tables[s][t / B]][h][t % B].
 * Exact attention (not an approximation); fp32 accumulation, output rounded
 * to nearest in the storage dtype.  context_lens[s] == 0 gives a zero row.
 *
 * Work split: a persistent grid; each CTA streams a contiguous share of the
 * batch's (sequence, head, K/V step) space, keeps an online-softmax state per
 * warp, and writes either the final row (when it saw the whole sequence/head)
 * or a partial (max, sum, unnormalised output) that a second kernel merges
 * with the log-sum-exp rule.  Two launches on `stream`.
 *
 * Reproducibility: with the balanced split (partition_size 0) the last
 * quarter of the work is claimed by CTAs at run time, which decides the order
 * in which a row's terms are summed, so two calls may differ in the last bits
 * (each within rounding of the exact result); a nonzero partition_size gives
 * every CTA the same work on every call and bit-identical results.
 *
 * workspace: device, >= pkv_decode_workspace_size(...) bytes, 256-B aligned;
 * its contents need no initialisation and are scratch between calls; two
 * calls in flight at once must not share it.
 */
pkv_status pkv_paged_attention_decode(void* out, const void* q, const void* k_cache,
                                      const void* v_cache, const int32_t* block_tables,
                                      const int32_t* context_lens, float scale,
                                      int num_seqs, int num_heads, int head_dim,
                                      int block_size, int max_blocks_per_seq,
                                      int64_t num_blocks, pkv_dtype dtype,
                                      int partition_size, void* workspace,
                                      size_t workspace_bytes, cudaStream_t stream);

/*
 * One decode step in one call: each sequence's newest token (the one at
 * position context_lens[s] - 1) is written into its cache slot and attended,
 * as pkv_reshape_and_cache with slot table[s][(ctx - 1) / B] * B + (ctx - 1) % B
 * followed by pkv_paged_attention_decode would (wywy.jp notes, "generation
 * phase": each iteration produces only the new token's K/V; the
 * zhaifeiyue.github.io detail page's block-indexed formula, the query
 * attending its own position).  The attention takes that token's K and V
 * from k_new / v_new rather than reading them back from the cache, so the
 * write and the attention need no ordering between them.
 *   k_new, v_new  [num_seqs][num_heads][head_dim], device, 16-byte aligned.
 *   k_cache, v_cache  written at the newest token's slot of every sequence
 *                 with context_lens[s] >= 1 (nothing else is written).
 * Cache contents are bit-identical to the two-call path, and so are outputs
 * with a fixed split (partition_size > 0; with the balanced split they agree
 * within rounding, as two calls of pkv_paged_attention_decode do).  A slot
 * whose table entry is out of [0, num_blocks) is not written
 * (PKV_DEVERR_BAD_BLOCK).  Every other argument and rule is that of
 * pkv_paged_attention_decode (same workspace size); two launches on `stream`.
 */
pkv_status pkv_paged_attention_decode_append(void* out, const void* q, const void* k_new,
                                             const void* v_new, void* k_cache, void* v_cache,
                                             const int32_t* block_tables,
                                             const int32_t* context_lens, float scale,
                                             int num_seqs, int num_heads, int head_dim,
                                             int block_size, int max_blocks_per_seq,
                                             int64_t num_blocks, pkv_dtype dtype,
                                             int partition_size, void* workspace,
                                             size_t workspace_bytes, cudaStream_t stream);

/*
 * The same decode attention for batches whose sequences share prefix blocks
 * (parallel sampling, beam search: sequences forked from one prompt hold the
 * prompt's blocks by reference; wywy.jp notes, "Copy-on-write" and the
 * parallel-sampling walkthrough; ricepunchb garden section 5.1, the shared
 * physical blocks of the sharing diagram).  The sharing structure is read from
 * the block tables themselves: sequences ADJACENT in the batch whose tables
 * begin with the same full blocks (at least 4 steps' worth: 64 tokens at
 * head_dim 128) form a group of at most 8; the group's common prefix is read
 * from HBM once and attended by every member together (tensor-core products of
 * the prefix's keys with the members' queries), and each member's own blocks
 * are read as usual; a merge pass combines both with the log-sum-exp rule.
 * Results are those of pkv_paged_attention_decode (same definition, within the
 * same tolerance; not bit-identical, the summation order differs).  Sharers
 * that are not adjacent are computed correctly, each reading its blocks.
 * Three launches on `stream` (a small group pass, the main pass, the merge).
 * Arguments as for pkv_paged_attention_decode; the workspace is sized by
 * pkv_decode_shared_workspace_size.  Batches above 4096 sequences run the
 * plain kernels (no grouping).
 */
pkv_status pkv_decode_shared_workspace_size(int num_seqs, int num_heads, int head_dim,
                                            int block_size, int max_blocks_per_seq,
                                            int partition_size, size_t* bytes);
pkv_status pkv_paged_attention_decode_shared(void* out, const void* q, const void* k_cache,
                                             const void* v_cache, const int32_t* block_tables,
                                             const int32_t* context_lens, float scale,
                                             int num_seqs, int num_heads, int head_dim,
                                             int block_size, int max_blocks_per_seq,
                                             int64_t num_blocks, pkv_dtype dtype,
                                             int partition_size, void* workspace,
                                             size_t workspace_bytes, cudaStream_t stream);

/*
 * The same decode attention over a CONTIGUOUS K/V layout, for measuring what
 * paging costs: the baseline the pages compare PagedAttention with keeps each
 * sequence's KV cache in one contiguous region reserved for its maximum
 * length (wywy.jp notes, "existing systems" in the WHAT section; the
 * zhaifeiyue.github.io detail page, "Kernel 开销 (§7.1)": the paged kernel is
 * 20-26% slower than FasterTransformer's contiguous attention kernel, Fig. 18a).
 *   k, v  [num_seqs][num_heads][max_context_len][head_dim], device; token t of
 *         sequence s, head h at ((s * num_heads + h) * max_context_len + t) * head_dim.
 *   out[s][h] = sum_{t < context_lens[s]} softmax_t(scale q[s][h] . k[s][h][t]) v[s][h][t]
 * No block table.  The kernel is the paged one with the table lookup replaced
 * by that address (same persistent split, copy ring, online softmax and merge),
 * so the two differ only in the indirection.  context_lens[s] above
 * max_context_len is clamped and sets PKV_DEVERR_BAD_CONTEXT.  The workspace
 * (pkv_contiguous_workspace_size) and every other rule are those of
 * pkv_paged_attention_decode.
 */
pkv_status pkv_contiguous_workspace_size(int num_seqs, int num_heads, int head_dim,
                                         int max_context_len, int partition_size,
                                         size_t* bytes);
pkv_status pkv_contiguous_attention_decode(void* out, const void* q, const void* k,
                                           const void* v, const int32_t* context_lens,
                                           float scale, int num_seqs, int num_heads,
                                           int head_dim, int max_context_len, pkv_dtype dtype,
                                           int partition_size, void* workspace,
                                           size_t workspace_bytes, cudaStream_t stream);

/*
 * Bound, in nanoseconds, of the decode kernels' pipeline waits (a consumer
 * warp waiting for a ring stage's copy, the producer waiting for a free stage
 * or for a claimed chunk's query slice, the consumer warps meeting at the end
 * of a piece), for every later launch of pkv_paged_attention_decode and
 * pkv_paged_attention_decode_noalloc from any host thread.  Default 1 s; at
 * most 10 s (larger values: PKV_ERR_INVALID, nothing changed).  A wait that
 * runs out sets PKV_DEVERR_TIMEOUT; the CTA then stops issuing copies, its
 * other waits give up at once, its results for the call are not valid, and it
 * returns after every copy it issued has landed (those waits always keep the
 * 1 s bound, so no copy lands in a CTA that has ended).  The next call starts
 * afresh.  A short limit exists to exercise that path (tests); 0 gives up on
 * the first check that finds a phase incomplete.  *previous (may be NULL)
 * receives the limit it replaces.  Host only; touches no GPU.
 * (Failure handling of the kernels; the pages have no counterpart.)
 */
pkv_status pkv_set_decode_wait_limit(uint64_t ns, uint64_t* previous);

/*
 * The same decode attention for callers that cannot allocate device memory
 * (the paper has no counterpart; this is an interface convenience).  Some
 * callers can neither allocate nor be handed a workspace -- a serving loop
 * whose device memory is planned once at start-up, or a plugin whose enqueue
 * callback must not allocate -- so this entry point keeps its scratch in a
 * fixed array of the library's own static device memory,
 * PKV_NOALLOC_SCRATCH_BYTES per device, held by every GPU that loads the
 * library until the process exits.  It allocates nothing itself (no
 * cudaMalloc, cudaFree or allocating library routine).
 *
 * Arguments as for pkv_paged_attention_decode, without the workspace.  Sizes
 * whose workspace (pkv_decode_workspace_size) exceeds the array are rejected
 * with PKV_ERR_INVALID and nothing is launched.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current and keeps it for the life
 * of the process; make that first call before any stream capture.  The kept
 * address belongs to the device's primary context: do not use this entry
 * point after cudaDeviceReset on that device or from another context (the
 * library's device error word is kept the same way).  All calls on a device
 * share the array, which keeps the last call's contents (nothing in it needs
 * to start at zero): calls whose work overlaps on the GPU (other streams,
 * other host threads) race on it and must be serialised by the caller.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (16u << 20)

pkv_status pkv_paged_attention_decode_noalloc(void* out, const void* q, const void* k_cache,
                                              const void* v_cache, const int32_t* block_tables,
                                              const int32_t* context_lens, float scale,
                                              int num_seqs, int num_heads, int head_dim,
                                              int block_size, int max_blocks_per_seq,
                                              int64_t num_blocks, pkv_dtype dtype,
                                              int partition_size, cudaStream_t stream);

/*
 * Prompt phase (wywy.jp notes, "prompt phase": every prompt token is known,
 * their K/V are produced together and attention runs as matrix-matrix work).
 * Sequence s has qlen = query_start[s+1] - query_start[s] new tokens whose
 * K/V are already in the cache (pkv_reshape_and_cache) at positions
 * ctx - qlen .. ctx - 1, ctx = context_lens[s].  Query row query_start[s] + i
 * (position p = ctx - qlen + i) attends positions 0 .. p (causal):
 *   out[row][h] = sum_{t <= p} softmax_t(scale * q[row][h] . K_s[t][h]) V_s[t][h]
 * A whole prompt is qlen == ctx; a prompt continued after a cached prefix
 * (shared prefix, chunked prefill) is qlen < ctx; qlen == 1 is one decode row.
 * q, out: [num_query_tokens][num_heads][head_dim] (num_query_tokens = the
 * rows of q and out, host); query_start: int32 [num_seqs + 1], device, with
 * every sequence's rows inside [0, num_query_tokens) (else the sequence is
 * skipped and PKV_DEVERR_BAD_CONTEXT set).  max_query_len (host) bounds every
 * qlen; a larger one sets PKV_DEVERR_BAD_CONTEXT and its extra rows are not
 * written.  num_blocks * num_heads * block_size must stay below 2^31 (the
 * tiled copies address cache rows with 32-bit coordinates).  The work is dealt
 * to the CTAs by 64-bit sums of estimated item costs: sizes whose bound on
 * those sums (ceil(num_heads / 2) * num_seqs * ceil(max_query_len / 256)
 * items, each at most 20 * (max_blocks_per_seq * block_size / 128 + 1) + 24)
 * reaches 2^60 are refused with PKV_ERR_INVALID (far beyond any call whose
 * tensors fit in memory).
 * Fifth-generation tensor cores (tcgen05, accumulators in tensor memory, TMA
 * tiled copies through the block table), fp32 accumulation, one launch, no
 * workspace.
 */
pkv_status pkv_paged_attention_prefill(void* out, const void* q, const void* k_cache,
                                       const void* v_cache, const int32_t* block_tables,
                                       const int32_t* context_lens, const int32_t* query_start,
                                       float scale, int num_seqs, int num_heads, int head_dim,
                                       int block_size, int max_blocks_per_seq, int64_t num_blocks,
                                       int max_query_len, int num_query_tokens, pkv_dtype dtype,
                                       cudaStream_t stream);

/*
 * The prompt phase with the prompts' cache write done by the same kernel,
 * for whole prompts (every sequence's qlen == context_lens[s]; a sequence
 * that is not is skipped and sets PKV_DEVERR_BAD_CONTEXT).  k, v:
 * [num_query_tokens][num_heads][head_dim], device, the prompt tokens' K and V
 * in the rows of q.  Computes out as pkv_paged_attention_prefill does, reading
 * the keys and values from k and v rather than from the cache, and writes
 * every prompt token's K and V into the cache at its position (slot
 * block_tables[s][t / B] * B + t mod B for position t: what
 * pkv_reshape_and_cache would write; other slots are left untouched).  One
 * launch instead of the cache write followed by the attention: the stores
 * run beside the tensor-core work (the wywy.jp notes' prompt phase, the block
 * manager's slot rule of the ricepunchb garden, section 3.2).  Other arguments
 * and rules as pkv_paged_attention_prefill; q, k, v 16-byte aligned.
 */
pkv_status pkv_paged_attention_prefill_write(void* out, const void* q, const void* k,
                                             const void* v, void* k_cache, void* v_cache,
                                             const int32_t* block_tables,
                                             const int32_t* context_lens,
                                             const int32_t* query_start, float scale,
                                             int num_seqs, int num_heads, int head_dim,
                                             int block_size, int max_blocks_per_seq,
                                             int64_t num_blocks, int max_query_len,
                                             int num_query_tokens, pkv_dtype dtype,
                                             cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Cache maintenance                                                         */
/* ------------------------------------------------------------------------ */

/*
 * For each token t with slot_mapping[t] >= 0 and each head h:
 *   k_cache[slot / B][h][slot % B][:] = k[t][h][:]   (same for v)
 * A bit copy.  Slots within one call must be distinct (else the result for
 * the duplicated slot is one of the writers').  A slot beyond the pool is
 * skipped and sets PKV_DEVERR_BAD_SLOT.  num_tokens == 0 launches nothing.
 */
pkv_status pkv_reshape_and_cache(const void* k, const void* v, void* k_cache, void* v_cache,
                                 const int64_t* slot_mapping, int num_tokens, int num_heads,
                                 int head_dim, int block_size, int64_t num_blocks,
                                 pkv_dtype dtype, cudaStream_t stream);

/*
 * For each pair p: k_cache[dst] = k_cache[src] and v_cache[dst] = v_cache[src],
 * whole blocks (all heads).  Destinations must be distinct and must not be the
 * source of any pair in the same call (copy-on-write always copies into a
 * freshly allocated block, so this holds for pairs the block manager emits).
 * A bad id skips the pair and sets PKV_DEVERR_BAD_BLOCK.
 * num_pairs == 0 launches nothing.
 */
pkv_status pkv_copy_blocks(void* k_cache, void* v_cache, const int32_t* pairs, int num_pairs,
                           int num_heads, int head_dim, int block_size, int64_t num_blocks,
                           pkv_dtype dtype, cudaStream_t stream);

/*
 * Block swap between a GPU pool and a CPU pool (either direction): for each
 * pair, dst_k_cache[dst] = src_k_cache[src] and the same for V, whole blocks.
 * Swapping evicts a preempted sequence's blocks to CPU RAM and brings them
 * back (wywy.jp notes, "Swapping" and the preemption section: the block
 * engine keeps a CPU pool split into blocks like the GPU one; swap space is
 * bounded by the GPU KV pool; zhaifeiyue.github.io detail page, Scheduling
 * table).  One kernel moves every pair at once, its SMs reading and writing
 * the host pool over the CPU-GPU link, so small blocks do not turn into many
 * small transfers.  Pools and pairs may be device memory, pinned (registered)
 * host memory or managed memory (checked with cudaPointerGetAttributes;
 * pageable host memory is refused with PKV_ERR_INVALID).  Both pools share
 * the [blocks][H][B][D] layout; destinations must be distinct.  A bad id
 * skips its pair and sets PKV_DEVERR_BAD_BLOCK.
 */
pkv_status pkv_swap_blocks(void* dst_k_cache, void* dst_v_cache, const void* src_k_cache,
                           const void* src_v_cache, const int32_t* pairs, int num_pairs,
                           int num_heads, int head_dim, int block_size, int64_t src_num_blocks,
                           int64_t dst_num_blocks, pkv_dtype dtype, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Errors                                                                    */
/* ------------------------------------------------------------------------ */

/*
 * Synchronises `stream`, then reads the device error word of the current
 * device into *bits (PKV_DEVERR_* bits, 0 = none) and, if clear != 0, resets
 * it.  Returns PKV_ERR_DEVICE when bits != 0, PKV_OK otherwise.
 */
pkv_status pkv_get_device_error(int32_t* bits, int clear, cudaStream_t stream);

/* Thread-local description of the last non-OK status of this thread. */
const char* pkv_last_error(void);

/* Library version string. */
const char* pkv_version(void);

/* ------------------------------------------------------------------------ */
/* Host block manager (host memory only; not thread-safe per handle)          */
/* ------------------------------------------------------------------------ */

/*
 * Policy: the free list starts as a seeded permutation of [0, num_blocks)
 * (Fisher-Yates driven by SplitMix64(seed), j = next() mod (i + 1) for
 * i = n-1 .. 1); allocation pops its front; a block whose count drops to zero
 * is pushed to its back (in block-table order).  A new block is allocated
 * only when the sequence's last block is full; writing into a partially
 * filled last block whose reference count is above one allocates a new block,
 * emits the (old, new) copy pair and decrements the old block's count.
 * Every failing call leaves the manager unchanged.
 */
typedef struct pkv_bm pkv_bm;

pkv_status pkv_bm_create(int64_t num_blocks, int block_size, uint64_t seed, pkv_bm** out);
void pkv_bm_destroy(pkv_bm* bm);

/* New sequence holding prompt_len tokens: allocates ceil(prompt_len / B)
 * blocks; writes the prompt tokens' slots to slots_out[prompt_len] (may be
 * NULL).  PKV_ERR_INVALID if seq_id exists; PKV_ERR_OOM if blocks run out. */
pkv_status pkv_bm_add_sequence(pkv_bm* bm, int64_t seq_id, int32_t prompt_len,
                               int64_t* slots_out);

/* child shares every block of parent (each block's count + 1). */
pkv_status pkv_bm_fork(pkv_bm* bm, int64_t parent, int64_t child);

/* Reserve the slot of the sequence's next token.  *cow_src / *cow_dst are the
 * copy pair the caller must apply (pkv_copy_blocks) before writing, or -1. */
pkv_status pkv_bm_append_slot(pkv_bm* bm, int64_t seq_id, int64_t* slot, int32_t* cow_src,
                              int32_t* cow_dst);

/* One decode step for n sequences, in order: slots[n]; copy pairs into
 * pairs[n][2] (at most one per sequence), their number in *num_pairs.
 * All-or-nothing: on failure the manager is unchanged. */
pkv_status pkv_bm_append_slots(pkv_bm* bm, const int64_t* seq_ids, int n, int64_t* slots,
                               int32_t* pairs, int32_t* num_pairs);

/* Release every block of the sequence (count - 1; zero -> free list). */
pkv_status pkv_bm_free_sequence(pkv_bm* bm, int64_t seq_id);

/* Copy the sequence's block table into out[cap]; *n = its length.
 * PKV_ERR_INVALID if cap is too small (nothing written). */
pkv_status pkv_bm_block_table(const pkv_bm* bm, int64_t seq_id, int32_t* out, int32_t cap,
                              int32_t* n);

/* Tokens held by the sequence. */
pkv_status pkv_bm_context_len(const pkv_bm* bm, int64_t seq_id, int32_t* n);

/* Decode-call inputs for n sequences: tables[n][max_blocks] (unused entries
 * set to -1) and context_lens[n].  PKV_ERR_INVALID if a table is longer than
 * max_blocks or a sequence is unknown. */
pkv_status pkv_bm_export(const pkv_bm* bm, const int64_t* seq_ids, int n, int32_t* tables,
                         int32_t max_blocks, int32_t* context_lens);

/* Reference count of a block (-1 if out of range); number of free blocks. */
int32_t pkv_bm_refcount(const pkv_bm* bm, int32_t block);
int64_t pkv_bm_num_free(const pkv_bm* bm);

/*
 * Swapping (wywy.jp notes, "Swapping", "All-or-nothing eviction" and the
 * preemption section; zhaifeiyue.github.io detail page, Scheduling table).
 * pkv_bm_add_cpu_pool gives the manager a CPU pool of num_cpu_blocks blocks
 * (its own seeded free list, same policy).  pkv_bm_swap_out moves a group of
 * resident sequences to the CPU pool, pkv_bm_swap_in moves swapped-out ones
 * back: all of the group's blocks move together; a block shared with a
 * sequence outside the group is refused (PKV_ERR_INVALID); each distinct
 * block (first-seen order: group order, then table order) gets a fresh block
 * in the other pool with the same reference count, the pair (old, new) is
 * written to pairs[cap][2] for pkv_swap_blocks, and the old block is freed.
 * Swapped-out sequences cannot append, fork or be exported until swapped in;
 * freeing one releases its CPU blocks.  All-or-nothing: on failure (OOM when
 * the other pool lacks blocks) nothing changes.
 */
pkv_status pkv_bm_add_cpu_pool(pkv_bm* bm, int64_t num_cpu_blocks, uint64_t seed);
pkv_status pkv_bm_swap_out(pkv_bm* bm, const int64_t* seq_ids, int n, int32_t* pairs,
                           int32_t cap, int32_t* num_pairs);
pkv_status pkv_bm_swap_in(pkv_bm* bm, const int64_t* seq_ids, int n, int32_t* pairs, int32_t cap,
                          int32_t* num_pairs);
/* 1 if swapped out, 0 if resident, -1 if unknown. */
int32_t pkv_bm_is_swapped(const pkv_bm* bm, int64_t seq_id);
int32_t pkv_bm_cpu_refcount(const pkv_bm* bm, int32_t block);
int64_t pkv_bm_num_free_cpu(const pkv_bm* bm);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDKV_H */
