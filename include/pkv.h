/*
 * pkv.h -- C ABI of libpkv: the decode hot path of PagedAttention on GB300.
 *
 * The operations follow the statement of the problem in "vLLM &
 * PagedAttention: Efficient Memory Management for LLM Serving" (§III
 * blockwise attention, §V request flow, §VII sharing and copy-on-write, §X
 * the three fused kernels and the fork/append/free primitives) and
 * "PagedAttention and vLLM, annotated" (§4.1 blockwise attention, §4.2 block
 * tables, §4.4 copy-on-write).
 *
 * Conventions for every call:
 *   - Returns pkv_status; PKV_OK is 0.  On failure pkv_last_error_string()
 *     describes the last error of the calling thread.
 *   - Pointers named *_dev are device pointers; the caller owns all device
 *     memory (the library allocates none for these calls) and must keep it
 *     alive until the work on `stream` has finished.  Device pointers must be
 *     16-byte aligned.
 *   - Device work is asynchronous on `stream` (a cudaStream_t; NULL is the
 *     legacy default stream).  Arguments are checked on the host before any
 *     launch; a bad argument returns PKV_EINVAL and launches nothing.
 *   - Index errors that only the device can see (a slot or block id outside
 *     the pool, a context longer than its table) are latched in a per-device
 *     status word; the offending access is skipped and the affected outputs
 *     are unspecified.  pkv_check() synchronises `stream`, reports the
 *     latched error (PKV_EINDEX, or PKV_ETIMEOUT when a bounded device-side
 *     wait gave up) and clears it.  Device errors are never raised with
 *     traps or asserts: the CUDA context stays usable.
 *   - 16-bit data are fp16 or bf16 (pkv_dtype); the library copies their bit
 *     patterns and computes in fp32.
 *
 * Layouts (row-major, innermost last):
 *   key_cache, value_cache   [num_blocks][num_kv_heads][block_size][head_dim]
 *   key, value (new tokens)  [num_tokens][num_kv_heads][head_dim]
 *   query, out               [num_seqs][num_heads][head_dim]
 *   block_tables             [num_seqs][max_blocks_per_seq] int32
 *   context_lens             [num_seqs] int32 (includes the decode token)
 * Query head h reads kv head h / (num_heads / num_kv_heads).
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;                       /* cudaStream_t is struct CUstream_st* */

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_EINVAL = 1,    /* bad argument; nothing was launched */
    PKV_ENOMEM = 2,    /* allocator: too few free blocks; state unchanged */
    PKV_EINDEX = 3,    /* device saw an index outside the pool or table */
    PKV_ECUDA = 4,     /* a CUDA runtime call failed */
    PKV_ETIMEOUT = 5   /* a bounded device-side wait gave up */
} pkv_status;

typedef enum pkv_dtype { PKV_F16 = 0, PKV_BF16 = 1 } pkv_dtype;

/* ---------------------------------------------------------------------------
 * kv_reshape_and_cache -- the fused reshape + block write ("vLLM &
 * PagedAttention" §X, first kernel; §V steps 2-3).
 *
 * For each token t with s = slot_mapping[t] >= 0: block b = s / block_size,
 * offset o = s % block_size, and for every kv head h
 *   key_cache[b][h][o][:] = key[t][h][:],  value_cache[b][h][o][:] = value[t][h][:]
 * copied bit for bit.  A negative slot marks a padding token and is skipped.
 * A slot >= num_blocks * block_size latches PKV_EINDEX and is skipped.
 * Slots must be distinct (two tokens with one slot race).
 *   key_dev, value_dev           [num_tokens][num_kv_heads][head_dim] 16-bit
 *   key_cache_dev, value_cache_dev  the pool, see Layouts
 *   slot_mapping_dev             [num_tokens] int64
 * head_dim must be a multiple of 8; block_size a power of two; num_tokens
 * may be 0 (nothing launched).
 * ------------------------------------------------------------------------- */
pkv_status kv_reshape_and_cache(const void *key_dev, const void *value_dev,
                                void *key_cache_dev, void *value_cache_dev,
                                const int64_t *slot_mapping_dev, int num_tokens,
                                int num_kv_heads, int head_dim, int block_size,
                                int num_blocks, pkv_dtype dtype, struct CUstream_st *stream);

/* ---------------------------------------------------------------------------
 * paged_attention_decode -- block-table gather + decode attention ("vLLM &
 * PagedAttention" §I attention equation, §III blockwise equation, §X second
 * kernel; "PagedAttention and vLLM, annotated" §4.1).
 *
 * For every sequence s and query head h, with g = h / (num_heads/num_kv_heads)
 * and n = context_lens[s]:
 *   x_t = scale * query[s][h] . K_t,   K_t = key_cache[block_tables[s][t / B]][g][t % B]
 *   out[s][h] = sum_{t<n} softmax(x)_t * V_t          (V_t likewise)
 * rounded to `dtype`.  n = 0 gives zeros.  scale is usually 1/sqrt(head_dim).
 *
 * Long contexts are split into partitions of partition_size tokens; each is
 * reduced to (max, sum of exponentials, un-normalised value sum) and the
 * partitions are merged by log-sum-exp: inside the attention kernel for
 * splits of up to 16 partitions, by a second kernel for longer ones.
 * partition_size = 0 lets the library
 * choose; otherwise it must be a positive multiple of 32.
 *   max_context_len   host-side upper bound on every context_lens[s]
 *                     (0 = max_blocks_per_seq * block_size); a larger
 *                     context latches PKV_EINDEX.
 *   num_blocks        pool size; a table entry outside [0, num_blocks)
 *                     within a context latches PKV_EINDEX.  Entries past
 *                     ceil(n / B) are never read.
 *   workspace_dev     at least paged_attention_workspace_size(...) bytes of
 *                     device scratch owned by the caller, initialised once
 *                     with paged_attention_workspace_init before its first
 *                     use.  It holds the work-ticket and merge counters,
 *                     which every completed call leaves ready for the next,
 *                     and the partition partials, which are clobbered.  The
 *                     merge counters move with the call's sizes: a call whose
 *                     sizes differ from the previous call's on the same
 *                     workspace first zeroes them (one more small launch).
 *                     Calls that may overlap on the GPU
 *                     need separate workspaces.  After a call that reported
 *                     PKV_ETIMEOUT, initialise it again.  An uninitialised
 *                     workspace makes the call do nothing and pkv_check
 *                     report PKV_EINVAL.
 * head_dim in {64, 128}; block_size a power of two in [4, 128];
 * num_heads % num_kv_heads == 0.
 * ------------------------------------------------------------------------- */
pkv_status paged_attention_decode(void *out_dev, const void *query_dev,
                                  const void *key_cache_dev, const void *value_cache_dev,
                                  const int32_t *block_tables_dev,
                                  const int32_t *context_lens_dev, int num_seqs,
                                  int max_blocks_per_seq, int max_context_len,
                                  int block_size, int num_blocks, int num_heads,
                                  int num_kv_heads, int head_dim, float scale,
                                  int partition_size, void *workspace_dev,
                                  size_t workspace_bytes, pkv_dtype dtype,
                                  struct CUstream_st *stream);

/* ---------------------------------------------------------------------------
 * paged_attention_decode_write -- kv_reshape_and_cache and
 * paged_attention_decode of one decode step in one launch ("vLLM &
 * PagedAttention" §X: the fused reshape-and-block-write beside the
 * attention).  The pages have no single call for the pair; it saves the
 * write's launch.
 *
 * key_dev, value_dev [num_seqs][num_kv_heads][head_dim] hold each sequence's
 * new token, slot_mapping_dev[num_seqs] (int64) its slot, which must be the
 * slot of position context_lens[s] - 1 of sequence s's table (as the
 * allocator returns it); a negative slot writes nothing; a slot beyond the
 * pool, or any other slot than that position's (a slot the launch's other
 * work items may be reading), latches PKV_EINDEX and is not written.  The
 * result is that of kv_reshape_and_cache on
 * the same arguments followed by paged_attention_decode: the caches hold the
 * new tokens bit for bit and out is the attention over contexts that include
 * them.  When the batch takes the grid kernel (more than 4096 sequences) the
 * call launches the write first.  Other arguments as for
 * paged_attention_decode.
 * ------------------------------------------------------------------------- */
pkv_status paged_attention_decode_write(void *out_dev, const void *query_dev, const void *key_dev,
                                        const void *value_dev, void *key_cache_dev,
                                        void *value_cache_dev, const int64_t *slot_mapping_dev,
                                        const int32_t *block_tables_dev,
                                        const int32_t *context_lens_dev, int num_seqs,
                                        int max_blocks_per_seq, int max_context_len,
                                        int block_size, int num_blocks, int num_heads,
                                        int num_kv_heads, int head_dim, float scale,
                                        int partition_size, void *workspace_dev,
                                        size_t workspace_bytes, pkv_dtype dtype,
                                        struct CUstream_st *stream);

/* ---------------------------------------------------------------------------
 * paged_attention_decode_noalloc -- paged_attention_decode for callers that
 * cannot allocate device memory.  The pages have no counterpart: this is an
 * interface convenience of this library.
 *
 * Some callers may not call cudaMalloc where they run attention: a plugin
 * that a host framework invokes while it captures a CUDA graph or from a
 * latency-critical execution callback (allocating there synchronises the
 * device or is refused), or a service that fixes its device-memory budget at
 * start-up.  This call takes no workspace: the partition partials live in a
 * fixed 16 MiB array in the library's own device memory, which every GPU that
 * loads the library holds until the process exits.  The caller still owns
 * and passes every input and output; the arguments and results are those of
 * paged_attention_decode.
 *   - Sizes whose partials would exceed 16 MiB (see
 *     paged_attention_workspace_size) return PKV_EINVAL, launching nothing.
 *   - The first call on each device looks up the array's device address and
 *     prepares its counters (no allocation; one small kernel on `stream`,
 *     which the call waits for).  pkv_check reporting PKV_ETIMEOUT marks the
 *     array for preparation again, done the same way by the next call.  A
 *     call that has to prepare the array while `stream` is capturing a CUDA
 *     graph returns PKV_EINVAL and launches nothing: make the first call on
 *     a device, and the first after a reported timeout, outside capture.
 *   - All calls on a device share the one array: calls that may overlap on
 *     the GPU (other streams, other threads) race and give wrong results; one
 *     call at a time per device.  Each completed call leaves the array ready
 *     for the next.
 * ------------------------------------------------------------------------- */
pkv_status paged_attention_decode_noalloc(void *out_dev, const void *query_dev,
                                          const void *key_cache_dev, const void *value_cache_dev,
                                          const int32_t *block_tables_dev,
                                          const int32_t *context_lens_dev, int num_seqs,
                                          int max_blocks_per_seq, int max_context_len,
                                          int block_size, int num_blocks, int num_heads,
                                          int num_kv_heads, int head_dim, float scale,
                                          int partition_size, pkv_dtype dtype,
                                          struct CUstream_st *stream);

/* ---------------------------------------------------------------------------
 * paged_attention_prefill -- attention of the prompt phase over the paged
 * cache: many new tokens per sequence, causal, after an optional cached
 * prefix ("vLLM & PagedAttention", §I attention equation with its sum over
 * t <= i; §II and §V, the prompt phase; §VII, a shared prefix whose blocks
 * are already cached, so that only the request's own input is computed).
 *
 * Sequence s has n_s = query_start[s+1] - query_start[s] new tokens, the
 * last n_s of its context_lens[s] tokens; their keys and values must already
 * be in the cache (kv_reshape_and_cache first).  New token j of sequence s,
 * row i = query_start[s] + j of query and out, sits at position
 * p = context_lens[s] - n_s + j and gives, for every query head h
 * (kv head g = h / (num_heads / num_kv_heads)):
 *   x_t = scale * query[i][h] . K_t  for t = 0..p   (K_t, V_t as above)
 *   out[i][h] = sum_{t<=p} softmax(x)_t * V_t, rounded to `dtype`.
 * n_s = context_lens[s] is a plain prompt; n_s = 1 is one decode step.
 *
 *   out_dev, query_dev  [num_tokens][num_heads][head_dim], 16-byte aligned;
 *                       num_tokens = query_start[num_seqs].
 *   query_start_dev     int32 [num_seqs + 1], query_start[0] = 0,
 *                       non-decreasing.  A sequence with n_s < 0,
 *                       n_s > context_lens[s], a context beyond its table
 *                       row or query_start[s+1] > num_tokens latches
 *                       PKV_EINDEX and writes none of its rows.
 *   max_query_len       host-side bound on every n_s (0 = num_tokens); it
 *                       sizes the grid, so a larger n_s leaves rows unwritten.
 *   num_blocks          table entries outside [0, num_blocks) latch
 *                       PKV_EINDEX (the call reads block 0 instead).
 *   workspace_dev       NULL, or at least 256 bytes prepared once by
 *                       paged_attention_workspace_init (a decode workspace
 *                       serves as well).  The work -- pairs of 128-row query
 *                       tiles of one (sequence, head), or with an even number
 *                       of query heads per kv head the same 128 rows of two
 *                       query heads that share a kv head -- is spread over one
 *                       CTA per SM; with a workspace the CTAs take items from
 *                       a counter in it (balanced), without one each takes a
 *                       fixed share (round robin).  The call leaves the
 *                       counter ready for the next; calls sharing a workspace
 *                       must not overlap on the GPU.  A workspace that was
 *                       never prepared latches PKV_EINVAL on the device
 *                       (pkv_check) and computes nothing.
 * The call allocates nothing.  num_seqs <= 65535; head_dim in {64, 128};
 * block_size a power of two in [4, 128]; num_heads % num_kv_heads == 0;
 * scale > 0 (usually 1/sqrt(head_dim)); the work items (ceil(max_query_len /
 * 256) x num_heads x num_seqs, or ceil(max_query_len / 128) x num_heads / 2 x
 * num_seqs for paired heads) <= 2^30.  Asynchronous on `stream`; PKV_EINVAL for
 * bad arguments, launching nothing.
 * ------------------------------------------------------------------------- */
pkv_status paged_attention_prefill(void *out_dev, const void *query_dev,
                                   const void *key_cache_dev, const void *value_cache_dev,
                                   const int32_t *block_tables_dev,
                                   const int32_t *context_lens_dev,
                                   const int32_t *query_start_dev, int num_seqs, int num_tokens,
                                   int max_query_len, int max_blocks_per_seq, int block_size,
                                   int num_blocks, int num_heads, int num_kv_heads, int head_dim,
                                   float scale, void *workspace_dev, size_t workspace_bytes,
                                   pkv_dtype dtype, struct CUstream_st *stream);

/* Bytes of workspace paged_attention_decode needs for these sizes: 256 for
 * the counters, plus the partition partials when a context can span more
 * than one partition.  partition_size as above. */
size_t paged_attention_workspace_size(int num_seqs, int num_heads, int num_kv_heads,
                                      int head_dim, int max_context_len,
                                      int partition_size);

/* Prepare a workspace for paged_attention_decode (asynchronous on `stream`;
 * one small kernel).  workspace_bytes >= 256. */
pkv_status paged_attention_workspace_init(void *workspace_dev, size_t workspace_bytes,
                                          struct CUstream_st *stream);

/* The partition size paged_attention_decode uses for these arguments:
 * partition_size when positive, else 512 tokens at head_dim 128 and 2048 at
 * head_dim 64 (the same bytes per work item), halved down to 512 while
 * num_seqs x num_kv_heads x ceil(max_context_len / P) stays below 2048. */
int paged_attention_partition_size(int num_seqs, int num_heads, int num_kv_heads,
                                   int head_dim, int max_context_len, int partition_size);

/* ---------------------------------------------------------------------------
 * copy_blocks -- the fused block copy for copy-on-write ("vLLM &
 * PagedAttention" §X, third kernel; §VII Figure 8).
 *
 * For each pair p: block dst = src_dst_pairs[2p+1] of `cache` becomes a copy
 * of block src = src_dst_pairs[2p], block_bytes bytes each (for the layout
 * above, block_bytes = num_kv_heads * block_size * head_dim * 2).  Call once
 * for the key cache and once for the value cache.
 *   cache_dev          [num_blocks] blocks of block_bytes bytes
 *   src_dst_pairs_dev  [num_pairs][2] int32, device memory
 * block_bytes must be a positive multiple of 16.  A block id outside
 * [0, num_blocks) latches PKV_EINDEX and that pair is skipped.  Destinations
 * must be distinct and no destination may also be a source (the pairs an
 * allocator's copy-on-write produces always are); pkv_validate_copy_pairs
 * checks this on a host copy.  num_pairs may be 0 (nothing launched).
 * ------------------------------------------------------------------------- */
pkv_status copy_blocks(void *cache_dev, const int32_t *src_dst_pairs_dev, int num_pairs,
                       int64_t block_bytes, int num_blocks, struct CUstream_st *stream);

/* ---------------------------------------------------------------------------
 * swap_blocks -- block copies between two pools, for swapping an evicted
 * group's blocks to the CPU and back ("vLLM & PagedAttention" §VIII and
 * Figure 4: a GPU block allocator for the live cache, a CPU block allocator
 * for swapped-out blocks).
 *
 * For each pair p: block pairs[2p+1] of dst_pool becomes a copy of block
 * pairs[2p] of src_pool, block_bytes bytes each (the pools share the layout
 * above).  One launch copies every pair, so small blocks cost no more
 * transfers than large ones.  Call once for keys and once for values.
 *   dst_pool, src_pool  [dst_blocks] / [src_blocks] blocks: device memory, or
 *                       host memory the GPU can address (pinned, e.g.
 *                       cudaHostAlloc), 16-byte aligned, distinct.
 *   pairs               [num_pairs][2] int32 in device or pinned host memory;
 *                       destinations distinct (pkv_move_group's pairs are).
 * A block id out of range latches PKV_EINDEX and that pair is skipped.
 * num_pairs may be 0 (nothing launched).  Asynchronous on `stream`: host
 * buffers must stay alive until it completes.
 * ------------------------------------------------------------------------- */
pkv_status swap_blocks(void *dst_pool, const void *src_pool, const int32_t *pairs, int num_pairs,
                       int64_t block_bytes, int src_blocks, int dst_blocks, struct CUstream_st *stream);

/* Host-side check of a pair list: ids in range, distinct destinations, no
 * destination that is also a source.  PKV_EINVAL if any fails. */
pkv_status pkv_validate_copy_pairs(const int32_t *src_dst_pairs_host, int num_pairs,
                                   int num_blocks);

/* ---------------------------------------------------------------------------
 * Status and introspection
 * ------------------------------------------------------------------------- */

/* Synchronise `stream`, then report and clear the error latched on the
 * current device (PKV_OK, PKV_EINDEX, PKV_ETIMEOUT, or PKV_EINVAL for an
 * attention workspace that was not initialised; PKV_ECUDA when the stream
 * itself failed). */
pkv_status pkv_check(struct CUstream_st *stream);

/* Message for the last failing call of this thread (never NULL). */
const char *pkv_last_error_string(void);

/* Number of kernels this library has launched in this process. */
uint64_t pkv_launch_count(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int pkv_version(void);

/* Self-test of the bounded device-side wait: launches one CTA that waits on
 * an mbarrier nothing ever arrives on, for at most limit_cycles clock
 * cycles (0 < limit_cycles <= 2^32).  The wait gives up, latches the timeout
 * and the kernel returns, so that a later pkv_check reports PKV_ETIMEOUT and
 * the context stays usable.  No counterpart on the pages: it exercises the
 * library's failure path without faulting or hanging the GPU. */
pkv_status pkv_selftest_wait_timeout(long long limit_cycles, struct CUstream_st *stream);

/* ---------------------------------------------------------------------------
 * Host block allocator ("vLLM & PagedAttention" §V, §VII, §X; "How
 * PagedAttention changed LLM serving throughput": a sequence uses exactly
 * ceil(len / block_size) blocks).
 *
 * A pool of num_blocks physical blocks with a reference count each.  Blocks
 * are handed out in the order `free_order` lists (a permutation of
 * 0..num_blocks-1; NULL = ascending); freed blocks are pushed back in the
 * freed sequence's logical order and handed out again last-in, first-out.
 * Sequence ids are assigned 0, 1, 2, ... in creation order and never reused.
 * A call that returns PKV_ENOMEM leaves the allocator unchanged.  The
 * allocator is not thread-safe; it makes no CUDA calls.
 * ------------------------------------------------------------------------- */
typedef struct pkv_allocator pkv_allocator;

pkv_status pkv_alloc_create(int num_blocks, int block_size, const int32_t *free_order,
                            pkv_allocator **out);
void pkv_alloc_destroy(pkv_allocator *a);

/* A new sequence of len tokens holding ceil(len / block_size) fresh blocks. */
pkv_status pkv_seq_new(pkv_allocator *a, int64_t len, int32_t *seq);
/* A new sequence sharing every block of `seq` (each count + 1). */
pkv_status pkv_seq_fork(pkv_allocator *a, int32_t seq, int32_t *child);
/* Add one token.  A full (or absent) last block gets a fresh block appended;
 * a shared (count > 1) partly filled last block is replaced by a fresh block
 * and (cow_src, cow_dst) = (old, new) is returned for copy_blocks, else both
 * are -1.  *slot = table[len / B] * B + len % B for the token's position. */
pkv_status pkv_seq_append(pkv_allocator *a, int32_t seq, int64_t *slot, int32_t *cow_src,
                          int32_t *cow_dst);
/* One token for each of seqs[0..n-1] in order (all or nothing).  slots[n];
 * cow_pairs has room for n pairs; *num_pairs receives the count. */
pkv_status pkv_seq_append_batch(pkv_allocator *a, const int32_t *seqs, int n, int64_t *slots,
                                int32_t *cow_pairs, int *num_pairs);
/* Drop the sequence; blocks whose count reaches 0 return to the pool. */
pkv_status pkv_seq_free(pkv_allocator *a, int32_t seq);
pkv_status pkv_seq_len(const pkv_allocator *a, int32_t seq, int64_t *len);
/* Copy the block table (at most cap entries) and its length. */
pkv_status pkv_seq_block_table(const pkv_allocator *a, int32_t seq, int32_t *out, int cap,
                               int *n);
/* Fill tables[n][max_blocks] (unused entries -1) and context_lens[n] for a
 * batch of sequences, ready to upload for paged_attention_decode. */
pkv_status pkv_build_block_tables(const pkv_allocator *a, const int32_t *seqs, int n,
                                  int32_t *tables, int max_blocks, int32_t *context_lens);
/* Reference count of a block (-1 if out of range). */
int pkv_block_ref(const pkv_allocator *a, int32_t block);
int pkv_num_free(const pkv_allocator *a);
/* Free blocks in the order they would be handed out (at most cap). */
pkv_status pkv_free_list(const pkv_allocator *a, int32_t *out, int cap, int *n);

/* One beam-search step ("vLLM & PagedAttention" §VII, Figure 9): the kn new
 * candidates continue beams[parents[i]] (0 <= parents[i] < k).
 *   - The first candidate naming a parent continues the parent's sequence
 *     (new_beams[i] = that id); each further one forks it (a new id).
 *   - Every candidate then appends one token, in order: slots[i] receives its
 *     slot; a write into a shared, partly filled last block copies that block
 *     first (cow_pairs gets (src, dst); room for kn pairs, *num_pairs of
 *     them).
 *   - Beams no candidate names are freed last.
 * All or nothing: PKV_ENOMEM (too few free blocks) or PKV_EINVAL (unknown
 * or repeated beam, bad parent index) change nothing. */
pkv_status pkv_beam_step(pkv_allocator *a, const int32_t *beams, int k, const int32_t *parents, int kn,
                         int32_t *new_beams, int64_t *slots, int32_t *cow_pairs, int *num_pairs);
/* Blocks currently held by some sequence (num_blocks - free). */
int pkv_blocks_in_use(const pkv_allocator *a);

/* Swapping ("vLLM & PagedAttention" §VIII): move the sequence group
 * seqs[0..n-1] from allocator `src` to allocator `dst` (a GPU and a CPU pool
 * of the same block size), all or nothing.
 *   - The group must hold every reference to its blocks (sequences that
 *     share blocks are evicted together); otherwise PKV_EINVAL.
 *   - Each distinct block, in first-seen order (the sequences in the given
 *     order, each in logical order), takes a block of `dst` with the same
 *     reference count; pairs[2k], pairs[2k+1] = (block in src, block in
 *     dst); *num_pairs of them (room for pairs_cap).  new_ids[i] is
 *     seqs[i]'s id in `dst`, with the same length and a table over the new
 *     blocks.
 *   - Then the group is freed in `src` (sequence by sequence, as
 *     pkv_seq_free).  The caller copies the pairs' blocks with swap_blocks
 *     (keys and values) before any of the freed blocks is written again.
 * Too few free blocks in `dst`: PKV_ENOMEM; on every error nothing changes. */
pkv_status pkv_move_group(pkv_allocator *src, pkv_allocator *dst, const int32_t *seqs, int n,
                          int32_t *new_ids, int32_t *pairs, int pairs_cap, int *num_pairs);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
