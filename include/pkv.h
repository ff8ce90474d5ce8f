/*
 * pkv.h -- C ABI of the GB300 (sm_103a) paged-KV attention library.
 *
 * One attention step of an in-flight-batching engine over a paged KV cache,
 * as the page "TensorRT-LLM框架解析与高性能推理优化实践" describes it:
 * K/V of every live sequence sit in fixed-size pages of one shared pool
 * (§4.2 "KV缓存管理细节"), a per-sequence block table maps logical pages to
 * physical ones (§6.2 "Paged Attention优化": block_tables
 * [num_seqs, max_blocks]), sequences may share prefix pages (§6.2, the
 * list of its optimisations), the KV cache may be stored quantised and is
 * dequantised inside the attention kernel (§7.2 "KV Cache量化"), and long
 * prompts are processed as chunks interleaved with decode requests (§5.3
 * "分块上下文处理").
 *
 * Conventions for every entry point
 *  - Pointers named as device data are device memory owned by the caller;
 *    descriptors (pkv_pool_desc) are host memory.  The library allocates no
 *    device memory at run time: scratch space (workspace) is sized by a query
 *    and passed in (pkv_paged_attention_noalloc instead uses a fixed array
 *    held from load time).  The host page manager (pkv_cache_*) keeps its
 *    own state in host memory.
 *  - All work is enqueued asynchronously on `stream` (a cudaStream_t; NULL
 *    is the legacy default stream), in stream order.  Nothing synchronises
 *    the host except pkv_get_device_error.  Kernels are launched with
 *    programmatic stream serialization so that consecutive kernels overlap
 *    their launch; each waits for the earlier kernels of the stream before
 *    touching memory they use, so the ordering is that of plain launches.
 *  - Arguments are validated on the host before anything is enqueued;
 *    an invalid call returns an error and enqueues nothing.
 *  - Device data (block-table entries, context lengths, slots) is not read by
 *    the host.  Kernels check it: an out-of-range page id or slot is skipped
 *    (never dereferenced) and recorded in a sticky per-device error word that
 *    pkv_get_device_error returns.  Kernels never trap and every wait in them
 *    is bounded; a wait that runs out is recorded the same way.
 *  - Host threads: the entry points may be called from several host threads
 *    at once (each on its own stream and buffers); the per-device set-up done
 *    on first use (SM count, kernel shared-memory attributes) is guarded.
 *    A pkv_cache_* handle is not synchronised: use each from one thread at a
 *    time.
 *
 * Data layout
 *  - KV pool: k_pool, v_pool = [num_blocks][num_kv_heads][block_size][head_dim],
 *    row-major, element type bf16 or FP8 E4M3 (OCP OFP8).  One (page, kv head)
 *    is a contiguous block_size*head_dim run.
 *  - Pool slot: slot = page * block_size + offset (offset < block_size).
 *  - GQA: q head a reads kv head a / (num_q_heads / num_kv_heads).
 *  - context_lens[s] counts every token of sequence s INCLUDING the ones
 *    appended in this step: append first (pkv_kv_append), then attend.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define PKV_API __attribute__((visibility("default")))
#else
#define PKV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_ERR_INVALID_ARG = 1,   /* null pointer, bad size, misalignment */
    PKV_ERR_UNSUPPORTED = 2,   /* valid but not built: head_dim, group size, ... */
    PKV_ERR_WORKSPACE = 3,     /* workspace too small or misaligned */
    PKV_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    PKV_ERR_DEVICE_BOUNDS = 5, /* a kernel met an out-of-range page id or slot */
    PKV_ERR_DEVICE_TIMEOUT = 6, /* a bounded wait inside a kernel ran out */
    PKV_ERR_OUT_OF_BLOCKS = 7   /* host page manager: the pool cannot supply the blocks */
} pkv_status;

typedef enum pkv_kv_dtype {
    PKV_KV_BF16 = 0,
    PKV_KV_FP8_E4M3 = 1        /* per-tensor scales: value = e4m3(code) * scale */
} pkv_kv_dtype;

/* Shape of the paged pool.  head_dim in {64, 128}; block_size in
 * {16, 32, 64, 128}.  FP8 only: one scale per tensor (k_scale / v_scale, > 0 and
 * finite), or one per kv head as the page's KV-cache quantisation section
 * describes (§7.2 "KV Cache量化", its first item): k_scales / v_scales,
 * optional device arrays of num_kv_heads positive finite floats (4-byte
 * aligned) that override the scalars when non-NULL.  Values in those arrays
 * are device data and are not checked. */
typedef struct pkv_pool_desc {
    int32_t num_blocks;
    int32_t num_kv_heads;
    int32_t block_size;
    int32_t head_dim;
    int32_t kv_dtype;          /* pkv_kv_dtype */
    float k_scale;
    float v_scale;
    const float *k_scales;     /* optional, device [num_kv_heads] */
    const float *v_scales;     /* optional, device [num_kv_heads] */
} pkv_pool_desc;

/*
 * pkv_kv_append -- write this step's new tokens into their pool slots.
 * (§4.2: pages allow non-contiguous storage of a growing sequence.)
 *
 *   k_new, v_new   device, bf16 [num_tokens][num_kv_heads][head_dim], 16-byte aligned
 *   slot_mapping   device, int64 [num_tokens]; token t goes to page
 *                  slot/block_size, offset slot%block_size.  slot < 0: skipped
 *                  (padding).  slot >= num_blocks*block_size: skipped and
 *                  recorded as PKV_ERR_DEVICE_BOUNDS.
 *   k_pool, v_pool device pools (see layout above), 16-byte aligned
 *   pool           host descriptor
 * bf16 pools store the bits unchanged.  FP8 pools store
 * e4m3_rn_satfinite(x / scale), the quotient taken in IEEE binary32, with
 * the token's kv head's scale when per-head scales are given.
 * num_tokens == 0 is a no-op.  Two tokens with the same slot race.
 */
PKV_API pkv_status pkv_kv_append(const void *k_new, const void *v_new,
                         const int64_t *slot_mapping, int32_t num_tokens,
                         void *k_pool, void *v_pool, const pkv_pool_desc *pool,
                         void *stream);

/*
 * Bytes of workspace pkv_paged_attention needs for these sizes (0 never
 * returned; at most a few hundred bytes per (sequence, q head, partition)).
 * partition_tokens as for pkv_paged_attention.  Returns 0 for invalid sizes.
 */
PKV_API size_t pkv_paged_attention_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                          int32_t max_context_len,
                                          int32_t partition_tokens,
                                          const pkv_pool_desc *pool);

/*
 * The split plan pkv_paged_attention uses for these sizes: *partition_out
 * receives the partition length in tokens (partition_tokens if > 0, else the
 * automatic choice) and *max_splits_out the largest number of partitions of
 * one sequence (1 = no split, the merge kernel is not launched).  Host-only.
 */
PKV_API pkv_status pkv_paged_attention_plan(int32_t num_seqs, int32_t num_q_heads,
                                            int32_t max_context_len, int32_t partition_tokens,
                                            const pkv_pool_desc *pool, int32_t *partition_out,
                                            int32_t *max_splits_out);

/*
 * pkv_paged_attention -- decode attention for a batch of sequences, one
 * query token each (§6.2 "Paged Attention优化"; running max/sum of §6.1).
 *
 *   out[s][a][:] = sum_i softmax_i(scale * <q[s][a], K_s[i]>) * V_s[i]
 *   over i < context_lens[s], K_s[i] = k_pool[block_tables[s][i/P]][a/G][i%P].
 *
 *   q               device, bf16 [num_seqs][num_q_heads][head_dim], 16-byte aligned
 *   k_pool, v_pool  device pools, 16-byte aligned
 *   block_tables    device, int32 [num_seqs][max_blocks_per_seq]
 *   context_lens    device, int32 [num_seqs]; each in [0, max_context_len]
 *                   (length 0 gives a zero output row)
 *   max_context_len host upper bound of context_lens (sizes the split plan)
 *   scale           softmax scale (e.g. 1/sqrt(head_dim)); FP8 scores are
 *                   additionally multiplied by k_scale and outputs by v_scale
 *                   (those of the kv head, with per-head scales)
 *   partition_tokens split-K partition length in tokens: a sequence longer
 *                   than it is processed as ceil(L/partition) independent
 *                   partitions merged by a second kernel.  0 = automatic.
 *                   Must be a multiple of block_size otherwise.
 *   workspace       device scratch of >= pkv_paged_attention_workspace_size
 *                   bytes, 256-byte aligned; contents need not be initialised
 *                   and are clobbered.  Calls sharing a workspace must be
 *                   stream-ordered.
 *   out             device, bf16 [num_seqs][num_q_heads][head_dim]
 * num_q_heads must be a multiple of num_kv_heads with a group size of
 * 1, 2, 4 or 8.  num_seqs == 0 is a no-op.
 */
PKV_API pkv_status pkv_paged_attention(const void *q, const void *k_pool, const void *v_pool,
                               const pkv_pool_desc *pool, const int32_t *block_tables,
                               int32_t max_blocks_per_seq, const int32_t *context_lens,
                               int32_t num_seqs, int32_t num_q_heads,
                               int32_t max_context_len, float scale,
                               int32_t partition_tokens, void *workspace,
                               size_t workspace_bytes, void *out, void *stream);

/*
 * pkv_paged_attention_noalloc -- the same decode attention as
 * pkv_paged_attention, for callers that cannot allocate device memory (the
 * pages describe no counterpart; this is a library convenience).  Some
 * callers receive only their input and output buffers -- a plugin run by a
 * host engine that owns all device allocations and exposes no workspace, or
 * a latency-critical step that must not call cudaMalloc -- so this entry
 * point takes no workspace and allocates nothing.  Its scratch is a fixed
 * device array inside the library of pkv_paged_attention_noalloc_max_scratch()
 * bytes (64 MiB), held on every GPU that loads the library until the process
 * exits.
 *   Arguments as for pkv_paged_attention, minus workspace / workspace_bytes.
 *   Returns PKV_ERR_WORKSPACE when these sizes need more scratch than the
 *   fixed maximum (see pkv_paged_attention_workspace_size); nothing is
 *   enqueued then.
 *   The first call on a device resolves the array's device address (a host
 *   call, once per device); make that first call before any stream capture.
 *   Every call shares the one array and the scratch needs no initial
 *   contents.  Calls whose work overlaps on the GPU (different streams
 *   without ordering between them) race on the array and give wrong results.
 */
PKV_API pkv_status pkv_paged_attention_noalloc(const void *q, const void *k_pool,
                                               const void *v_pool, const pkv_pool_desc *pool,
                                               const int32_t *block_tables,
                                               int32_t max_blocks_per_seq,
                                               const int32_t *context_lens, int32_t num_seqs,
                                               int32_t num_q_heads, int32_t max_context_len,
                                               float scale, int32_t partition_tokens, void *out,
                                               void *stream);

/* Size in bytes of the fixed scratch array pkv_paged_attention_noalloc uses. */
PKV_API size_t pkv_paged_attention_noalloc_max_scratch(void);

/*
 * pkv_paged_prefill -- causal attention of prefill-chunk tokens over their
 * sequences' pages (§5.3 "分块上下文处理": chunked context).
 *
 *   Sequence s owns packed query rows cu_seqlens_q[s] .. cu_seqlens_q[s+1]-1
 *   (C_s rows).  context_lens[s] = L_s counts the chunk, whose K/V must have
 *   been appended already.  Row i of sequence s (position L_s - C_s + i)
 *   attends to keys 0 .. L_s - C_s + i.
 *
 *   q               device, bf16 [num_q_tokens][num_q_heads][head_dim], 16-byte aligned
 *   cu_seqlens_q    device, int32 [num_seqs + 1], non-decreasing, [0] = 0,
 *                   [num_seqs] = num_q_tokens, each C_s <= min(max_q_len, L_s)
 *   k_pool, v_pool  device pools, bf16 or FP8 E4M3 (scales as in the pool
 *                   descriptor: k_scale multiplies the scores, v_scale the
 *                   output), 16-byte aligned
 *   block_tables    device, int32 [num_seqs][max_blocks_per_seq]
 *   context_lens    device, int32 [num_seqs]
 *   max_q_len       host upper bound of C_s
 *   scale           softmax scale, finite and > 0
 *   out             device, bf16 [num_q_tokens][num_q_heads][head_dim]
 * head_dim 64 or 128; the group size num_q_heads/num_kv_heads must divide
 * 128.  Uses tcgen05 tensor cores and TMA; needs no workspace.  An FP8 pool
 * is dequantised inside the kernel (§7.2, its third item): the codes are
 * converted exactly to f16 in shared memory, q is converted to f16 after an
 * exact power-of-two scaling per query row (undone on the scores), and both
 * products run on f16 operands with fp32 accumulation.
 * Device data: a sequence whose rows fall outside 0 .. num_q_tokens-1, whose
 * chunk is longer than max_q_len or than L_s, or whose L_s exceeds
 * max_blocks_per_seq pages is skipped (its rows are not written) and
 * recorded for pkv_get_device_error (PKV_ERR_DEVICE_BOUNDS); a page id out of
 * range is recorded and read as zeros.
 */
PKV_API pkv_status pkv_paged_prefill(const void *q, const int32_t *cu_seqlens_q,
                             const void *k_pool, const void *v_pool,
                             const pkv_pool_desc *pool, const int32_t *block_tables,
                             int32_t max_blocks_per_seq, const int32_t *context_lens,
                             int32_t num_seqs, int32_t num_q_heads, int32_t max_q_len,
                             int32_t num_q_tokens, float scale, void *out,
                             void *stream);

/*
 * pkv_get_device_error -- read and clear the current device's sticky error
 * word after the work already enqueued on `stream`: one small kernel on
 * `stream` swaps the word for zero atomically, the value is copied back on
 * the same stream and the stream is synchronised.  *code receives PKV_OK,
 * PKV_ERR_DEVICE_BOUNDS or PKV_ERR_DEVICE_TIMEOUT (the first error recorded
 * since the last read).  An error that a kernel on another stream records
 * meanwhile is returned by this read or kept for the next one, never lost.
 * Returns PKV_ERR_CUDA if the launch, the copy or the synchronisation fails.
 */
PKV_API pkv_status pkv_get_device_error(int32_t *code, void *stream);

/*
 * pkv_self_test_bounded_wait -- a check of the kernels' failure path on the
 * current device: one small kernel waits, with a limit of limit_cycles SM
 * clock cycles (0 < limit_cycles <= 2e9), on a barrier that nothing arrives
 * at.  The wait must give up, record PKV_ERR_DEVICE_TIMEOUT in the sticky
 * error word (read it with pkv_get_device_error) and raise the kernel's
 * abort flag, after which a second wait returns at once; the kernel then
 * ends normally and the context stays usable.
 *   out   device, int32 [5], 4-byte aligned: first wait's result (expect 0),
 *         second wait's result (0), abort flag (1), first wait lasted at
 *         least limit_cycles (1), second lasted less than limit_cycles / 4 (1).
 * Enqueued on `stream`; PKV_ERR_INVALID_ARG for a bad pointer or limit.
 */
PKV_API pkv_status pkv_self_test_bounded_wait(int64_t limit_cycles, int32_t *out, void *stream);

/* Text of the last CUDA error a call of this library met on the calling
 * thread (explains PKV_ERR_CUDA; "no error" if none).  Never NULL. */
PKV_API const char *pkv_last_cuda_error(void);

/* One decode step in one call: the same result as pkv_kv_append(k_new, v_new,
 * slot_mapping, num_new_tokens, ...) followed by pkv_paged_attention(...) on
 * the same stream, with the append fused into the attention's planning
 * launch (one kernel launch fewer per step).  Arguments as in those two
 * calls (k_new / v_new: device bf16 [num_new_tokens][Hkv][D]; slot_mapping:
 * device int64 [num_new_tokens], slot < 0 = padding); the appended tokens are
 * visible to the attention (context_lens count them).  The workspace is the
 * same as pkv_paged_attention's.  num_new_tokens = 0 is a plain
 * pkv_paged_attention; num_seqs = 0 a plain pkv_kv_append.  Errors: any status
 * of either call, returned before anything is enqueued when it comes from
 * host validation. */
PKV_API pkv_status pkv_paged_attention_append(
    const void *q, const void *k_new, const void *v_new, const int64_t *slot_mapping,
    int32_t num_new_tokens, void *k_pool, void *v_pool, const pkv_pool_desc *pool,
    const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *context_lens,
    int32_t num_seqs, int32_t num_q_heads, int32_t max_context_len, float scale,
    int32_t partition_tokens, void *workspace, size_t workspace_bytes, void *out, void *stream);

/* Copy whole blocks for copy-on-write of shared prefix pages (the page's
 * §4.1 / §4.2: blocks are reused and shared between sequences; a shared
 * block must be duplicated before one of its owners writes into it).
 *   pairs        device, int32 [num_pairs][2]: (source block, destination
 *                block), 4-byte aligned, as pkv_cache_append reports them.
 *                Every destination must be distinct and must not be the
 *                source of any pair in the same call (the manager's
 *                destinations are freshly popped blocks, so this holds).
 *   k_pool/v_pool as in pkv_kv_append; the whole block (all kv heads) of
 *                both pools is copied.
 * Asynchronous on `stream`; order it before the pkv_kv_append that writes
 * into the destinations.  An out-of-range block id is skipped and recorded
 * for pkv_get_device_error (PKV_ERR_DEVICE_BOUNDS). */
PKV_API pkv_status pkv_copy_blocks(void *k_pool, void *v_pool, const pkv_pool_desc *pool,
                                   const int32_t *pairs, int32_t num_pairs, void *stream);

/* ---- Host KV-cache page manager ------------------------------------------
 * The page "TensorRT-LLM框架解析与高性能推理优化实践", §4.1 (a KV-cache
 * manager: paged cache, block reuse and prefix sharing, memory reclaim),
 * §4.2 (KV缓存管理细节: blocks of one pool handed out and taken back, a block
 * list per sequence that is its block table) and §5.2 (抢占策略实现:
 * last-in-first-out preemption of running requests when the pool is short).
 *
 * Host memory only; no CUDA call.  A manager is not thread-safe: one caller
 * at a time.  Its outputs are the device calls' inputs: slot mappings for
 * pkv_kv_append, block pairs for pkv_copy_blocks, block tables and lengths
 * for pkv_paged_attention / pkv_paged_prefill (copied to the device by the
 * caller).  Sequence ids are caller-chosen non-negative int64 values.
 *
 * Policy, fixed so that results are reproducible:
 *   - free blocks form a stack with block 0 on top at creation; allocation
 *     pops the top, release pushes;
 *   - a sequence forked from another shares the parent's first
 *     ceil(num_tokens / block_size) blocks;
 *   - a block with more than one owner is copied before a sequence writes
 *     into it: a fresh block is popped and (old, new) reported;
 *   - an append over several sequences is all-or-nothing;
 *   - release pushes a sequence's blocks last page first; a block returns to
 *     the free stack when its owner count reaches zero;
 *   - preemption frees whole sequences, most recently admitted (added or
 *     forked) first, skipping protected ones; nothing changes if that cannot
 *     free enough.
 * Errors: PKV_ERR_INVALID_ARG (null pointer, unknown or duplicate id, a
 * count that would exceed max_blocks_per_seq, too small an output buffer)
 * and PKV_ERR_OUT_OF_BLOCKS leave the manager unchanged. */
typedef struct pkv_cache pkv_cache;

/* Create a manager for a pool of num_blocks blocks of block_size tokens;
 * tables have max_blocks_per_seq entries.  *out is owned by the caller and
 * freed by pkv_cache_destroy. */
PKV_API pkv_status pkv_cache_create(int32_t num_blocks, int32_t block_size,
                                    int32_t max_blocks_per_seq, pkv_cache **out);
PKV_API void pkv_cache_destroy(pkv_cache *cache);

/* Free blocks / live sequences (-1 for a NULL manager). */
PKV_API int32_t pkv_cache_num_free(const pkv_cache *cache);
PKV_API int32_t pkv_cache_num_seqs(const pkv_cache *cache);
/* Tokens held by a sequence, -1 if unknown. */
PKV_API int32_t pkv_cache_length(const pkv_cache *cache, int64_t seq_id);

/* Admit an empty sequence. */
PKV_API pkv_status pkv_cache_add(pkv_cache *cache, int64_t seq_id);
/* Admit `child` as the first num_tokens tokens of `parent` (0 <= num_tokens
 * <= parent's length), sharing the blocks that hold them. */
PKV_API pkv_status pkv_cache_fork(pkv_cache *cache, int64_t parent, int64_t child,
                                  int32_t num_tokens);
/* Give back a sequence's blocks and forget it. */
PKV_API pkv_status pkv_cache_release(pkv_cache *cache, int64_t seq_id);

/* Blocks (new pages plus copies) that pkv_cache_append of the same arguments
 * would take; -1 if the request is invalid. */
PKV_API int64_t pkv_cache_blocks_needed(pkv_cache *cache, const int64_t *seq_ids,
                                        const int32_t *counts, int32_t n);

/* Reserve slots for counts[i] new tokens of seq_ids[i] (distinct ids), in
 * that order.  Writes the slots (block * block_size + offset) of the
 * sum(counts) tokens, sequence after sequence, into slot_mapping
 * (slot_capacity entries), and the copy-on-write pairs into copies
 * (copy_capacity >= n pairs of int32: each sequence copies at most one
 * block per call).  *num_slots and *num_copies receive the counts. */
PKV_API pkv_status pkv_cache_append(pkv_cache *cache, const int64_t *seq_ids,
                                    const int32_t *counts, int32_t n, int64_t *slot_mapping,
                                    int64_t slot_capacity, int32_t *copies,
                                    int32_t copy_capacity, int64_t *num_slots,
                                    int32_t *num_copies);

/* Release whole sequences, most recently admitted first and skipping the
 * num_protected ids in protected_ids, until at least `needed` blocks are
 * free.  The released ids go to victims (victim_capacity entries), in
 * release order; *num_victims receives their count (0 if enough blocks were
 * already free).  PKV_ERR_OUT_OF_BLOCKS if even releasing every unprotected
 * sequence would not be enough. */
PKV_API pkv_status pkv_cache_preempt_for(pkv_cache *cache, int32_t needed,
                                         const int64_t *protected_ids, int32_t num_protected,
                                         int64_t *victims, int32_t victim_capacity,
                                         int32_t *num_victims);

/* Block tables (int32 [n][max_blocks_per_seq], -1 past each sequence's last
 * block) and context lengths (int32 [n]) of the listed sequences, in host
 * memory, ready for one host-to-device copy. */
PKV_API pkv_status pkv_cache_block_tables(const pkv_cache *cache, const int64_t *seq_ids,
                                          int32_t n, int32_t *block_tables,
                                          int32_t *context_lens);

/* Static string for a status code (never NULL). */
PKV_API const char *pkv_status_string(int32_t status);

/* Library ABI version (major * 100 + minor).  101: pkv_paged_prefill accepts
 * FP8 E4M3 pools. */
PKV_API int32_t pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
