/*
 * libpagedattn — PagedAttention decode on GB300 (sm_103a), C ABI.
 *
 * The KV cache of every sequence lives in fixed-size physical blocks of one
 * preallocated pool; a per-sequence block table maps logical block i to a
 * physical block id ("PagedAttention" glossary entry, block tables; "10 — Paged
 * Attention" tutorial, §1 "What is it?").  This library provides the three
 * device operations of a decode step over such a pool:
 *
 *   pa_decode             attention of one query token per sequence over its
 *                         paged keys/values, the gather fused into the math
 *                         (tutorial §5 "The kernel side"; glossary entry, the
 *                         kernel duties: read the table, gather, handle a
 *                         partly filled last block);
 *   pa_reshape_and_cache  store new tokens' keys/values in pool slots;
 *   pa_copy_blocks        whole-block copies for copy-on-write (tutorial §5
 *                         "Copy-on-write sharing"; subroutine-cs article §3);
 *
 * plus pa_decode_slots (the slot of each sequence's newest token, the
 * tutorial's PhysicalIndex, §4) and a host-side block manager (pa_bm_*,
 * tutorial §4 "Tiny example": allocate / free / fork / append).
 *
 * Conventions for every device call
 *   - All tensors are dense, row-major, in device memory owned by the caller.
 *     The library allocates no device memory and keeps no global device state;
 *     pa_decode's scratch space is a caller-provided workspace.
 *   - K and V pools share one layout: [num_blocks, block_size, num_kv_heads,
 *     head_dim], so slot s (= block * block_size + row) of the pool is one
 *     contiguous row of num_kv_heads * head_dim elements.
 *   - Element type is fp16 or bf16 (pa_dtype); q, out, key, value and the
 *     pools of one call share it.  Index arrays are int32.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream).  Host-side
 *     argument checks run before any launch and return an error code without
 *     launching; a launch failure returns PA_ERR_CUDA.  No call aborts.
 *   - status_dev (nullable): an int32 in device memory.  When non-NULL the call
 *     runs in checked mode: invalid device-side data (a block id outside
 *     [0, num_blocks), a slot outside the pool, a sequence longer than its
 *     table) is reported by storing the error code there, and the offending
 *     access is skipped.  The caller zeroes it beforehand.  With NULL such data
 *     is a caller error (reads through the tensor-map path stay inside the
 *     pool; other accesses are unchecked).
 */
#ifndef PAGEDATTN_H
#define PAGEDATTN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1,   /* null pointer, bad shape or size            */
  PA_ERR_UNSUPPORTED = 2,   /* dtype / head_dim / block_size not built     */
  PA_ERR_WORKSPACE = 3,     /* workspace missing or too small              */
  PA_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed        */
  PA_ERR_BAD_BLOCK_ID = 5,  /* checked mode: bad block id / slot / length  */
  PA_ERR_OUT_OF_BLOCKS = 6, /* block manager: free pool too small          */
  PA_ERR_BLOCK_STATE = 7,   /* block manager: unreferenced block freed or
                               forked, unknown sequence                    */
  PA_ERR_TIMEOUT = 8        /* a kernel's bounded internal wait expired and
                               it stopped early (reported via status_dev)  */
} pa_status;

typedef enum pa_dtype { PA_FLOAT16 = 0, PA_BFLOAT16 = 1 } pa_dtype;

/* Human-readable name of a status code (static string). */
const char* pa_status_string(int status);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int pa_version(void);

/* ------------------------------------------------------------------------ */
/* Decode attention                                                          */
/* ------------------------------------------------------------------------ */

/*
 * Workspace bytes pa_decode needs for a batch of num_seqs sequences no longer
 * than max_seq_len tokens, whichever decode kernel serves the call (an upper
 * bound over the kernels).  partition_tokens: 0 selects the default (512).
 * Returns 0 for invalid arguments.
 */
size_t pa_decode_workspace_bytes(int num_seqs, int num_q_heads, int head_dim,
                                 int max_seq_len, int partition_tokens);

/*
 * Workspace bytes of the decode kernel that a pa_decode call with these
 * arguments runs under the current kernel selection (pa_set_decode_path): the
 * grouped tensor-core kernel needs only its stream-K area (per-CTA partials,
 * independent of the sequence lengths), the others the [num_seqs, num_q_heads,
 * partitions] partials.  At most pa_decode_workspace_bytes(...).  Returns 0 for
 * arguments pa_decode would reject.  Host only; reads no device memory.
 */
size_t pa_decode_workspace_bytes_for(int num_seqs, int num_q_heads, int num_kv_heads,
                                     int head_dim, int block_size, int max_blocks,
                                     int num_blocks, int max_seq_len, int dtype,
                                     int partition_tokens);

/*
 * out[b, hq, :] = sum_t softmax_t(scale * q[b, hq, :] . K[slot_t, hq / G, :])
 *                       * V[slot_t, hq / G, :]
 * over t < seq_lens[b], slot_t = block_tables[b][t / block_size] * block_size
 * + t % block_size, G = num_q_heads / num_kv_heads (query head hq reads KV
 * head hq / G).  This is exact softmax attention; the pool indirection only
 * decides where rows are read from (glossary entry, the kernel duties; tutorial
 * §4 PhysicalIndex and §5 "The kernel side").
 *
 * out, q        [num_seqs, num_q_heads, head_dim]          dtype
 * k_pool/v_pool [num_blocks, block_size, num_kv_heads, head_dim]   dtype
 * block_tables  [num_seqs, max_blocks] int32; entries past
 *               ceil(seq_len / block_size) are never read
 * seq_lens      [num_seqs] int32, 0 <= seq_len <= max_seq_len; a sequence of
 *               length 0 gets a zero output row
 * max_seq_len   host-side upper bound on seq_lens (sizes the launch without a
 *               device-to-host read); a longer or negative seq_len is clamped
 *               to [0, max_seq_len] (and reported in checked mode)
 * scale         softmax scale applied to q.k (fp32)
 * partition_tokens  tokens per split-K partition (multiple of 128 and of
 *               block_size); 0 = default 512.  Sequences longer than one
 *               partition are processed as independent partitions whose
 *               partial (max, sum, accumulator) are merged by a second pass.
 * workspace     device scratch of at least pa_decode_workspace_bytes_for(...)
 *               (pa_decode_workspace_bytes(...) always suffices), 256-byte
 *               aligned; contents need not be initialised; it may not be
 *               shared by calls that overlap on the GPU.
 * Supported: dtype fp16/bf16, head_dim 64 or 128, block_size 8/16/32/64,
 * num_q_heads a multiple of num_kv_heads.
 */
pa_status pa_decode(void* out, const void* q, const void* k_pool, const void* v_pool,
                    const int32_t* block_tables, const int32_t* seq_lens,
                    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                    int block_size, int max_blocks, int num_blocks, int max_seq_len,
                    float scale, int dtype, int partition_tokens,
                    void* workspace, size_t workspace_bytes,
                    int32_t* status_dev, cudaStream_t stream);

/*
 * Kernel selection for pa_decode / pa_decode_noalloc (process-wide setting).
 * Three decode kernels exist:
 *   grouped tensor-core kernel (tcgen05 + TMA): each CTA reads whole blocks,
 *     all KV heads at once, over an equal share of the batch's tokens;
 *     head_dim 128, num_q_heads / num_kv_heads in {1,2,4,8,16} (or 3, 5, 6, 7
 *     when num_kv_heads is a multiple of 4: passes of 4 or 8 KV heads),
 *     num_seqs <= 32768; more than 64 query heads run as passes over groups of
 *     1-32 KV heads (a group must divide num_kv_heads);
 *   per-head tensor-core kernel (tcgen05 + TMA): one KV head per work item;
 *     head_dim 128, any grouping;
 *   CUDA-core kernel: every supported shape.
 *   PA_DECODE_AUTO     the first of the three that serves the call (default);
 *   PA_DECODE_SIMT     always the CUDA-core kernel;
 *   PA_DECODE_TC       a tensor-core kernel (grouped when it serves the call);
 *   PA_DECODE_TC_HEAD  the per-head tensor-core kernel;
 * a tensor-core setting returns PA_ERR_UNSUPPORTED for calls no tensor-core
 * kernel serves.  Returns PA_ERR_INVALID_ARG for an unknown value.  Not
 * synchronised with calls in flight on other host threads.
 */
typedef enum pa_decode_path {
  PA_DECODE_AUTO = 0, PA_DECODE_SIMT = 1, PA_DECODE_TC = 2, PA_DECODE_TC_HEAD = 3
} pa_decode_path;
pa_status pa_set_decode_path(int path);

/*
 * Which decode kernel a pa_decode call with these arguments runs under the
 * current selection: PA_KERNEL_GROUPED, PA_KERNEL_PER_HEAD or PA_KERNEL_SIMT;
 * -1 for arguments pa_decode rejects (or a tensor-core selection that no
 * tensor-core kernel serves).  Host only; reads no device memory.
 */
typedef enum pa_decode_kernel {
  PA_KERNEL_GROUPED = 0, PA_KERNEL_PER_HEAD = 1, PA_KERNEL_SIMT = 2
} pa_decode_kernel;
int pa_decode_kernel_for(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                         int block_size, int max_blocks, int num_blocks, int max_seq_len,
                         int dtype, int partition_tokens);

/*
 * pa_decode for callers that cannot allocate device memory.  The pages have no
 * counterpart: this is a deployment convenience of this library.
 *
 * pa_decode needs a scratch workspace for its split-K partials, normally
 * allocated by the caller.  Some callers cannot allocate when they call: code
 * recorded into a CUDA graph where allocation is not permitted, plug-ins that
 * only receive device pointers from a host application that owns every
 * allocation, or latency-critical loops that must stay off the allocator.
 * This entry point has the arguments of pa_decode minus the workspace and
 * takes its scratch from a fixed array of PA_DECODE_NOALLOC_SCRATCH_BYTES
 * (32 MiB) that is part of the library's device image: every device that
 * loads the library holds it until the process exits.  It calls no
 * allocating routine.
 *
 *  - Limit: a batch whose pa_decode_workspace_bytes_for(...) exceeds
 *    PA_DECODE_NOALLOC_SCRATCH_BYTES is rejected with PA_ERR_WORKSPACE before
 *    any device work.  The grouped tensor-core kernel (the default where it
 *    serves the shape) needs about 5.1 MiB per 32 query heads whatever the
 *    lengths (batches of up to 192 query heads fit); the
 *    other kernels need [num_seqs, num_q_heads, partitions] partials, e.g.
 *    8 sequences x 64 query heads up to 128K tokens about 65 MiB, which is
 *    rejected.  Other errors are those of pa_decode.
 *  - Set-up: the first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current; this may load the module).
 *    Make that first call before any stream capture.  The current device must
 *    be the device of the buffers and of `stream`.  The address is kept per
 *    device context: after cudaDeviceReset the next call looks it up again
 *    (so, again, before any capture).
 *  - Sharing: all calls share the one array, which keeps the last call's
 *    contents; nothing in it needs to start at zero.  Calls that overlap on the
 *    GPU (different streams, or different host threads without ordering) race
 *    on it and give wrong results: serialise them.
 */
#define PA_DECODE_NOALLOC_SCRATCH_BYTES (32u << 20)

pa_status pa_decode_noalloc(void* out, const void* q, const void* k_pool, const void* v_pool,
                            const int32_t* block_tables, const int32_t* seq_lens,
                            int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                            int block_size, int max_blocks, int num_blocks, int max_seq_len,
                            float scale, int dtype, int partition_tokens,
                            int32_t* status_dev, cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Cache writes                                                              */
/* ------------------------------------------------------------------------ */

/*
 * For i < num_tokens with slot = slot_mapping[i] >= 0:
 *   k_pool[slot / block_size][slot % block_size][:, :] = key[i][:, :]
 *   v_pool[...same...]                                   = value[i][:, :]
 * i.e. token i's [num_kv_heads, head_dim] rows land in pool slot `slot`, the
 * tutorial's PhysicalIndex of the token's position (§4).  Negative slots mark
 * padding and are skipped.  Exact bit copies.
 *
 * key/value     [num_tokens, num_kv_heads, head_dim] with token stride
 *               kv_token_stride elements (0 = num_kv_heads * head_dim); rows
 *               must be 16-byte aligned.
 * Two tokens mapped to the same slot in one call is a caller error.
 */
pa_status pa_reshape_and_cache(void* k_pool, void* v_pool, const void* key, const void* value,
                               const int32_t* slot_mapping, int num_tokens,
                               int64_t kv_token_stride, int num_kv_heads, int head_dim,
                               int block_size, int num_blocks, int dtype,
                               int32_t* status_dev, cudaStream_t stream);

/*
 * Copy-on-write clone: for each pair (src, dst) = (block_pairs[2i],
 * block_pairs[2i+1]), i < num_pairs, copy every slot of block src to block dst,
 * in both pools (tutorial §5 "Copy-on-write sharing": copy first, then write).
 * Pairs are copied concurrently: a dst that is also a src, or a dst that
 * appears twice, in one call is a caller error.  Exact bit copies.
 */
pa_status pa_copy_blocks(void* k_pool, void* v_pool, const int32_t* block_pairs, int num_pairs,
                         int num_kv_heads, int head_dim, int block_size, int num_blocks,
                         int dtype, int32_t* status_dev, cudaStream_t stream);

/*
 * slot_mapping[b] = slot of token seq_lens[b] - 1 of sequence b (its newest
 * token), block_tables[b][(L-1) / block_size] * block_size + (L-1) % block_size,
 * or -1 when seq_lens[b] == 0 (tutorial §4 PhysicalIndex).  Feeds
 * pa_reshape_and_cache in a decode step.  A negative length, a length past
 * max_blocks * block_size, or a block id outside [0, num_blocks) also gives -1
 * and is reported through status_dev (checked mode), so the token is never
 * written anywhere.  num_blocks * block_size must fit an int32.
 */
pa_status pa_decode_slots(int32_t* slot_mapping, const int32_t* block_tables,
                          const int32_t* seq_lens, int num_seqs, int max_blocks,
                          int block_size, int num_blocks, int32_t* status_dev,
                          cudaStream_t stream);

/*
 * Decode-step cache write in one launch: pa_decode_slots followed by
 * pa_reshape_and_cache.  For every sequence b with L = seq_lens[b] > 0, token
 * L - 1 (the newest, already counted in L) is stored at its pool slot
 *   slot = block_tables[b][(L-1) / block_size] * block_size + (L-1) % block_size
 * (tutorial §4 PhysicalIndex): k_pool/v_pool rows of that slot = key[b] / value[b]
 * ([num_kv_heads, head_dim], token stride kv_token_stride elements, 0 = packed).
 * slot_mapping (nullable, [num_seqs] int32) receives the slots, -1 for empty
 * sequences.  A length beyond max_blocks * block_size or a slot outside the pool
 * is skipped (and reported in checked mode).  Exact bit copies.
 */
pa_status pa_append_tokens(void* k_pool, void* v_pool, const void* key, const void* value,
                           const int32_t* block_tables, const int32_t* seq_lens,
                           int32_t* slot_mapping, int num_seqs, int64_t kv_token_stride,
                           int num_kv_heads, int head_dim, int block_size, int max_blocks,
                           int num_blocks, int dtype, int32_t* status_dev, cudaStream_t stream);

/*
 * One whole decode step: the cache write of pa_append_tokens (key / value
 * packed [num_seqs, num_kv_heads, head_dim], no slot_mapping output), then
 * pa_decode over the grown sequences ("10 — Paged Attention" tutorial, §4: the
 * newest token gets its slot, then §5 "The kernel side": attention through the
 * table).  Results and pools are bit-identical to those two calls in that
 * order; the other arguments, the workspace and the error behaviour are those
 * of pa_decode (key and value 16-byte aligned).  Where pa_decode runs its
 * grouped tensor-core kernel, the write happens inside it: the CTA that reads a
 * sequence's last tile stores the newest token before loading that tile, which
 * saves one launch per step.  The CUDA-core kernel writes it inside too (one
 * CTA per sequence and KV head stores the row; every CTA reads that token from
 * key / value); with the per-head tensor-core kernel it is a launch before it.  The block receiving a sequence's newest token must
 * not be in another sequence's table (copy-on-write it first, as for any write).
 */
pa_status pa_decode_append(void* out, const void* q, void* k_pool, void* v_pool,
                           const void* key, const void* value, const int32_t* block_tables,
                           const int32_t* seq_lens, int num_seqs, int num_q_heads,
                           int num_kv_heads, int head_dim, int block_size, int max_blocks,
                           int num_blocks, int max_seq_len, float scale, int dtype,
                           int partition_tokens, void* workspace, size_t workspace_bytes,
                           int32_t* status_dev, cudaStream_t stream);

/*
 * Paged multi-query attention with a causal mask: prefill, chunked prefill and
 * verification of several drafted tokens (subroutine-cs article, introduction:
 * the prefill phase computes all prompt tokens at once; "10 — Paged Attention"
 * §5 "The kernel side" for the gather through the block table).
 *   q, out      [total_q, num_q_heads, head_dim]; rows q_start[b] .. q_start[b+1]-1
 *               are sequence b's n_b = q_start[b+1] - q_start[b] query tokens,
 *               which are its LAST n_b tokens: row q_start[b] + i is position
 *               seq_lens[b] - n_b + i.  Their K/V must already be in the pool
 *               (pa_reshape_and_cache).
 *   q_start     [num_seqs + 1] int32, non-decreasing, q_start[0] = 0,
 *               q_start[num_seqs] = total_q (device memory).
 *   max_q_len   host upper bound of every n_b (sizes the grid, no device sync).
 * For query head hq of that row, with KV head h = hq / (num_q_heads /
 * num_kv_heads):  out = softmax_t(scale * q . K[slot_t, h]) . V[slot_t, h] over
 * t = 0 .. position, slot_t as in pa_decode.  fp32 accumulation, output rounded
 * to the storage type.  Supported: head_dim 64 or 128, any num_q_heads /
 * num_kv_heads, block_size in {8, 16, 32, 64}, fp16 / bf16.  head_dim 128 with
 * query groups of 1 to 8 or 16 runs on the tensor cores (tcgen05, TMA); every
 * other shape on a CUDA-core kernel.  A sequence with n_b > seq_lens[b], n_b > max_q_len,
 * seq_lens[b] > max_blocks * block_size, or rows outside [0, total_q) is skipped
 * (rows untouched; reported in checked mode); out-of-range block ids read zeros
 * (reported in checked mode).
 * No workspace.
 */
pa_status pa_prefill(void* out, const void* q, const void* k_pool, const void* v_pool,
                     const int32_t* block_tables, const int32_t* seq_lens,
                     const int32_t* q_start, int num_seqs, int total_q, int num_q_heads,
                     int num_kv_heads, int head_dim, int block_size, int max_blocks,
                     int num_blocks, int max_q_len, float scale, int dtype,
                     int32_t* status_dev, cudaStream_t stream);

/* Kernel choice for pa_prefill (process-wide; for tests and measurements):
 * AUTO picks the tensor-core kernel where it serves the shape. */
typedef enum pa_prefill_path {
  PA_PREFILL_AUTO = 0, PA_PREFILL_SIMT = 1, PA_PREFILL_TC = 2
} pa_prefill_path;
pa_status pa_set_prefill_path(int path);

/*
 * Copy-on-write across a whole model in one launch ("10 — Paged Attention"
 * tutorial §5 "Copy-on-write sharing"; a model keeps one K and one V pool per
 * layer, subroutine-cs article §1 bytes-per-token formula).  For every pair
 * (src, dst) of block_pairs ([num_pairs, 2] int32, device memory) and every
 * pool i < num_pools: block dst of pools[i] = block src of pools[i].
 *   pools        host array of num_pools device pointers (the K and V pools of
 *                every layer, any order), each num_blocks blocks of block_bytes
 *                bytes (block_size * num_kv_heads * head_dim * element size for
 *                the [num_blocks, block_size, num_kv_heads, head_dim] layout);
 *                16-byte aligned; read during the call only.
 *   block_bytes  a multiple of 16.  num_pools <= 512.
 * A block id outside [0, num_blocks) skips its pair (reported in checked mode).
 * A dst that is also a src, or appears twice, is a caller error.  Exact bit
 * copies.
 */
pa_status pa_copy_blocks_multi(void* const* pools, int num_pools, const int32_t* block_pairs,
                               int num_pairs, int64_t block_bytes, int num_blocks,
                               int32_t* status_dev, cudaStream_t stream);

/*
 * Block swap between GPU pools and pools in CPU RAM (the PagedAttention glossary
 * page, allocation and eviction: evicted blocks moved to host memory).
 * For every pair (src, dst) of block_pairs and every pool i < num_pools: block
 * dst of dst_pools[i] = block src of src_pools[i].  Swap-out passes GPU pools as
 * src and host pools as dst; swap-in the reverse; GPU-to-GPU also works.
 *   dst_pools, src_pools  host arrays of num_pools pointers, each to device
 *                memory or to page-locked host memory (cudaHostAlloc, or
 *                cudaHostRegister'ed) that the GPU can address; pageable host
 *                memory is rejected with PA_ERR_INVALID_ARG.  16-byte aligned.
 *   block_pairs  [num_pairs, 2] int32 (src id, dst id) in device or page-locked
 *                host memory; src ids index [0, src_num_blocks), dst ids
 *                [0, dst_num_blocks).
 *   block_bytes  bytes of one block of one pool, a multiple of 16.
 * One kernel moves every block of every pool over NVLink-C2C with plain loads and
 * stores.  Out-of-range ids skip the pair (reported in checked mode).  The host
 * memory must stay untouched by the CPU until the stream has passed the call.
 */
pa_status pa_swap_blocks(void* const* dst_pools, const void* const* src_pools, int num_pools,
                         const int32_t* block_pairs, int num_pairs, int64_t block_bytes,
                         int src_num_blocks, int dst_num_blocks, int32_t* status_dev,
                         cudaStream_t stream);

/* ------------------------------------------------------------------------ */
/* Host block manager                                                        */
/* ------------------------------------------------------------------------ */
/*
 * Refcounted allocator of physical block ids (tutorial §4 "Tiny example"):
 * a LIFO free stack; allocating n blocks hands out the top n entries in stack
 * order with refcount 1, or fails leaving the state unchanged; freeing drops
 * a refcount and returns the block to the stack at zero; forking raises the
 * refcount of every block of a table.  Sequences (block table + length) grow
 * one token at a time; a token that lands in a shared block triggers
 * copy-on-write (new block, (old, new) pair reported for pa_copy_blocks,
 * old refcount - 1).  Host memory only; not thread-safe per handle.
 */
typedef struct pa_block_manager pa_block_manager;

/* initial_free_stack: NULL = ids num_blocks-1 .. 0 pushed in that order (id 0 on
 * top); else a permutation of [0, num_blocks) listed bottom to top. */
pa_status pa_bm_create(int num_blocks, int block_size, const int32_t* initial_free_stack,
                       pa_block_manager** out);
void pa_bm_destroy(pa_block_manager* bm);
int pa_bm_num_free(const pa_block_manager* bm);
/* Cached blocks with refcount 0 waiting for eviction (not on the free stack). */
int pa_bm_num_evictable(const pa_block_manager* bm);
/* Refcount of a block id (0 when free, -1 when out of range). */
int pa_bm_refcount(const pa_block_manager* bm, int block_id);
pa_status pa_bm_allocate(pa_block_manager* bm, int n, int32_t* out_ids);
pa_status pa_bm_free(pa_block_manager* bm, const int32_t* ids, int n);
pa_status pa_bm_fork(pa_block_manager* bm, const int32_t* ids, int n);

/* Sequences are numbered by the manager; ids are never reused. */
pa_status pa_bm_seq_create(pa_block_manager* bm, int prompt_len, int* seq_id);
pa_status pa_bm_seq_fork(pa_block_manager* bm, int parent, int* child);
pa_status pa_bm_seq_release(pa_block_manager* bm, int seq_id);
/* Append one token.  *slot = its pool slot; (*cow_src, *cow_dst) = the block
 * copy the caller must run before writing the token, or (-1, -1). */
pa_status pa_bm_seq_append(pa_block_manager* bm, int seq_id, int32_t* slot,
                           int32_t* cow_src, int32_t* cow_dst);
int pa_bm_seq_len(const pa_block_manager* bm, int seq_id);
/*
 * Prefix cache ("10 — Paged Attention" tutorial §5, the relationship to prefix
 * caching): create a sequence holding token_ids[0 .. num_tokens).  Full block i
 * is keyed by key_i = FNV-1a-64(key_{i-1} as 8 little-endian bytes, then the
 * block's token ids as 4 little-endian bytes each), key_{-1} = 0, so a key
 * names the whole prefix.  The leading blocks whose keys (and stored parent key
 * and token ids) are cached are shared (refcount + 1, or taken off the
 * eviction queue with refcount 1), up to the first miss; the rest are allocated
 * and their full blocks registered.  *cached_tokens = tokens whose KV is
 * already in the pool (a multiple of block_size); the caller computes the KV of
 * the others before anything reads them.  A cached block whose refcount drops to
 * zero waits on an eviction queue (blocks of one release last block first) and
 * is evicted, front first, only when an allocation finds the free stack short.
 * PA_ERR_OUT_OF_BLOCKS (state unchanged) when free + evictable blocks, minus
 * the queued blocks this call revives, cannot cover the new blocks.
 */
pa_status pa_bm_seq_create_cached(pa_block_manager* bm, const int32_t* token_ids,
                                  int num_tokens, int* seq_id, int* cached_tokens);
int pa_bm_seq_num_blocks(const pa_block_manager* bm, int seq_id);
/* Copy sequence tables into a [n, max_blocks] int32 array (padding with pad_id)
 * and their lengths into seq_lens[n]; fails if a table is longer than max_blocks. */
pa_status pa_bm_export(const pa_block_manager* bm, const int* seq_ids, int n, int max_blocks,
                       int32_t pad_id, int32_t* block_tables, int32_t* seq_lens);

/* ------------------------------------------------------------------------ */
/* Allocator simulator                                                       */
/* ------------------------------------------------------------------------ */
/*
 * A contiguous and a paged KV allocator serving one request stream
 * ("10 — Paged Attention" tutorial, §10 exercises B and C; the 20-38% vs 96%+
 * memory-utilisation comparison of §7).  Host code.  Time advances in decode
 * steps t = 0, 1, ...; each step:
 *   1. requests with arrival_step <= t join the back of the waiting queue;
 *   2. admission: the queue head is admitted while its allocation succeeds; the
 *      first failure ends admission for the step (one failed allocation);
 *      an admitted request holds len tokens (its prompt, or after a preemption
 *      all it had: the KV is recomputed);
 *   3. growth: each request admitted in an earlier step, in admission order,
 *      appends one token; paged: with its blocks full it takes one more block,
 *      or, with none free, is preempted (one failed allocation, one preemption):
 *      its blocks are freed and it goes back to the front of the queue (those
 *      preempted in one step in admission order);
 *   4. measurement (when any request runs): tokens stored = sum of len, memory
 *      held (contiguous: sum of reservations; paged: blocks x block_size),
 *      running requests, blocks per request (paged);
 *   5. requests with len == prompt + output finish and release their memory.
 * Contiguous: one extent of `reserve` slots of a linear space of
 * capacity_tokens, first fit at the lowest address, freed extents merged;
 * reserve = max_seq_len (MAX), next power of two of prompt + output (POW2) or
 * prompt + output (EXACT).  A failed admission while the free total covers the
 * request is also a fragmentation failure.  Paged: capacity_tokens / block_size
 * blocks, admission needs ceil(len / block_size) free blocks.
 * Requests: arrival_step non-decreasing; 1 <= prompt, 1 <= output,
 * prompt + output <= max_seq_len; each must fit an empty pool.  Stops after
 * max_steps steps (result.completed < num_requests then).
 */
enum { PA_SIM_CONTIGUOUS = 0, PA_SIM_PAGED = 1 };
enum { PA_SIM_RESERVE_MAX = 0, PA_SIM_RESERVE_POW2 = 1, PA_SIM_RESERVE_EXACT = 2 };

typedef struct {
  int allocator;              /* PA_SIM_CONTIGUOUS or PA_SIM_PAGED */
  int reserve;                /* contiguous reservation rule, PA_SIM_RESERVE_* */
  int block_size;             /* paged */
  int max_seq_len;            /* longest request; the MAX reservation */
  int64_t capacity_tokens;    /* KV slots of the pool */
  int64_t max_steps;
} pa_sim_config;

typedef struct {
  int64_t steps;                    /* steps simulated */
  int64_t completed;                /* requests finished */
  int64_t failed_allocations;       /* failed admissions + failed growths */
  int64_t fragmentation_failures;   /* contiguous: failed although enough was free */
  int64_t preemptions;              /* paged: growths that found no free block */
  int64_t max_concurrency;          /* most requests running in one step */
  int64_t sum_concurrency;          /* sums over the steps with a running request: */
  int64_t busy_steps;               /*   that many steps */
  int64_t sum_stored;               /*   tokens stored */
  int64_t sum_held;                 /*   slots held by the allocator */
  int64_t peak_stored, peak_held;
  int64_t sum_table_len;            /* paged: blocks held, summed over requests and steps */
  int64_t max_table_len;            /* paged: longest block table */
} pa_sim_result;

/* Arrays of num_requests int32 in host memory.  PA_ERR_INVALID_ARG on a bad
 * configuration or request (nothing simulated). */
pa_status pa_sim_run(const pa_sim_config* cfg, const int32_t* arrival_step,
                     const int32_t* prompt_len, const int32_t* output_len, int num_requests,
                     pa_sim_result* out);

/* ------------------------------------------------------------------------ */
/* Measurement aid                                                           */
/* ------------------------------------------------------------------------ */
/*
 * A plain read stream over `bytes` bytes of device memory at `src` (16-byte
 * aligned, bytes a multiple of 16): every byte read once, contiguously, with
 * no gather and no compute.  Not part of the decode path: timing it in the same
 * run as pa_decode gives the read bandwidth a kernel reaches on this GPU, next
 * to which the decode kernels' bandwidth is read.  `sink` (nullable, device) is
 * incremented only when the XOR of all words read equals 0x9E3779B9, so the
 * loads cannot be dropped.  Asynchronous on `stream`.
 */
pa_status pa_stream_read(const void* src, size_t bytes, unsigned long long* sink,
                         cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_H */
