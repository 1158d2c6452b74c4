// Cache writes of a decode step: reshape_and_cache (new tokens into pool
// slots), copy_blocks (copy-on-write clones) and decode_slots (the slot of each
// sequence's newest token).
//
// All three are bandwidth-trivial bit copies; they move 16-byte vectors so a
// warp touches whole 512-byte spans.  Pool slot s is the contiguous row of
// Hkv * D elements at s * Hkv * D ("10 — Paged Attention" tutorial, §4
// PhysicalIndex: slot = block * block_size + row).
#include "pa_common.cuh"

namespace pa {

// One thread per 16-byte vector of one token's K (and V) row.
__global__ void __launch_bounds__(256)
reshape_and_cache_kernel(uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                         const uint4* __restrict__ key, const uint4* __restrict__ value,
                         const int32_t* __restrict__ slot_mapping, int num_tokens,
                         int64_t src_token_vecs, int row_vecs, int64_t num_slots,
                         int32_t* status_dev) {
  allow_next_grid();
  wait_prior_grid();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t total = (int64_t)num_tokens * row_vecs;
  if (i >= total) return;
  const int token = (int)(i / row_vecs);
  const int v = (int)(i - (int64_t)token * row_vecs);
  const int32_t slot = slot_mapping[token];
  if (slot < 0) return;                       // padding token
  if ((int64_t)slot >= num_slots) {           // never write outside the pool
    report(status_dev, PA_ERR_BAD_BLOCK_ID);
    return;
  }
  const int64_t src = (int64_t)token * src_token_vecs + v;
  const int64_t dst = (int64_t)slot * row_vecs + v;
  k_pool[dst] = key[src];
  v_pool[dst] = value[src];
}

// One CTA per (pair, pool); its threads stride over the block's vectors.
__global__ void __launch_bounds__(256)
copy_blocks_kernel(uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                   const int32_t* __restrict__ pairs, int block_vecs, int num_blocks,
                   int32_t* status_dev) {
  allow_next_grid();
  wait_prior_grid();
  const int pair = blockIdx.x;
  const int32_t src = pairs[2 * pair], dst = pairs[2 * pair + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (threadIdx.x == 0 && blockIdx.y == 0) report(status_dev, PA_ERR_BAD_BLOCK_ID);
    return;
  }
  uint4* pool = blockIdx.y == 0 ? k_pool : v_pool;
  const uint4* from = pool + (int64_t)src * block_vecs;
  uint4* to = pool + (int64_t)dst * block_vecs;
  // four independent 16-byte loads in flight per thread
  int v = threadIdx.x;
  for (; v + 3 * 256 < block_vecs; v += 4 * 256) {
    uint4 a = from[v], b = from[v + 256], c = from[v + 512], d = from[v + 768];
    to[v] = a;
    to[v + 256] = b;
    to[v + 512] = c;
    to[v + 768] = d;
  }
  for (; v < block_vecs; v += 256) to[v] = from[v];
}

// Slot of each sequence's newest token, or -1.  A length past the table or a
// block id outside [0, num_blocks) gives -1 and is reported (checked mode), as
// in append_tokens_kernel, so that a bad table entry never turns into a slot
// that a later cache write would silently treat as padding or write through.
__global__ void decode_slots_kernel(int32_t* __restrict__ slot_mapping,
                                    const int32_t* __restrict__ block_tables,
                                    const int32_t* __restrict__ seq_lens, int num_seqs,
                                    int max_blocks, int block_size, int num_blocks,
                                    int32_t* status_dev) {
  allow_next_grid();
  wait_prior_grid();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= num_seqs) return;
  const int len = seq_lens[b];
  if (len <= 0 || len > max_blocks * block_size) {
    if (len != 0) report(status_dev, PA_ERR_BAD_BLOCK_ID);
    slot_mapping[b] = -1;
    return;
  }
  const int pos = len - 1;
  const int32_t blk = block_tables[(int64_t)b * max_blocks + pos / block_size];
  if (blk < 0 || blk >= num_blocks) {
    report(status_dev, PA_ERR_BAD_BLOCK_ID);
    slot_mapping[b] = -1;
    return;
  }
  slot_mapping[b] = blk * block_size + pos % block_size;
}

// Newest token of each sequence: slot from the block table, then the copy.
// One thread per 16-byte vector of one sequence's K (and V) row.
__global__ void __launch_bounds__(256)
append_tokens_kernel(uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                     const uint4* __restrict__ key, const uint4* __restrict__ value,
                     const int32_t* __restrict__ block_tables,
                     const int32_t* __restrict__ seq_lens, int32_t* __restrict__ slot_mapping,
                     int num_seqs, int64_t src_token_vecs, int row_vecs, int block_size,
                     int max_blocks, int64_t num_slots, int32_t* status_dev) {
  allow_next_grid();
  wait_prior_grid();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)num_seqs * row_vecs) return;
  const int b = (int)(i / row_vecs);
  const int v = (int)(i - (int64_t)b * row_vecs);
  const int L = seq_lens[b];
  int64_t slot = -1;
  if (L > 0 && L <= max_blocks * block_size) {
    const int pos = L - 1;
    slot = (int64_t)block_tables[(int64_t)b * max_blocks + pos / block_size] * block_size +
           pos % block_size;
    if (slot < 0 || slot >= num_slots) {
      if (v == 0) report(status_dev, PA_ERR_BAD_BLOCK_ID);
      slot = -1;
    }
  } else if (L != 0 && v == 0) {
    report(status_dev, PA_ERR_BAD_BLOCK_ID);
  }
  if (slot_mapping && v == 0) slot_mapping[b] = (int32_t)slot;
  if (slot < 0) return;
  const int64_t src = (int64_t)b * src_token_vecs + v;
  const int64_t dst = slot * row_vecs + v;
  k_pool[dst] = key[src];
  v_pool[dst] = value[src];
}

}  // namespace pa

using namespace pa;

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

static bool supported_shape(int head_dim, int block_size, int dtype) {
  return (head_dim == 64 || head_dim == 128) &&
         (block_size == 8 || block_size == 16 || block_size == 32 || block_size == 64) &&
         (dtype == PA_FLOAT16 || dtype == PA_BFLOAT16);
}

extern "C" pa_status pa_reshape_and_cache(void* k_pool, void* v_pool, const void* key,
                                          const void* value, const int32_t* slot_mapping,
                                          int num_tokens, int64_t kv_token_stride,
                                          int num_kv_heads, int head_dim, int block_size,
                                          int num_blocks, int dtype, int32_t* status_dev,
                                          cudaStream_t stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || num_blocks <= 0) return PA_ERR_INVALID_ARG;
  if (!supported_shape(head_dim, block_size, dtype)) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!k_pool || !v_pool || !key || !value || !slot_mapping) return PA_ERR_INVALID_ARG;
  const int64_t row_elems = (int64_t)num_kv_heads * head_dim;
  const int64_t stride = kv_token_stride == 0 ? row_elems : kv_token_stride;
  if (stride < row_elems || (stride % 8) != 0) return PA_ERR_INVALID_ARG;
  if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(key) || !aligned16(value))
    return PA_ERR_INVALID_ARG;
  const int row_vecs = (int)(row_elems / 8);
  const int64_t total = (int64_t)num_tokens * row_vecs;
  const int64_t grid = (total + 255) / 256;
  if (grid > 0x7FFFFFFF) return PA_ERR_INVALID_ARG;
  if (launch_pdl(reshape_and_cache_kernel, dim3((unsigned)grid), 256, 0, stream, (uint4*)k_pool,
                 (uint4*)v_pool, (const uint4*)key, (const uint4*)value, slot_mapping, num_tokens,
                 (int64_t)(stride / 8), row_vecs, (int64_t)num_blocks * block_size,
                 status_dev) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

extern "C" pa_status pa_copy_blocks(void* k_pool, void* v_pool, const int32_t* block_pairs,
                                    int num_pairs, int num_kv_heads, int head_dim,
                                    int block_size, int num_blocks, int dtype,
                                    int32_t* status_dev, cudaStream_t stream) {
  if (num_pairs < 0 || num_kv_heads <= 0 || num_blocks <= 0) return PA_ERR_INVALID_ARG;
  if (!supported_shape(head_dim, block_size, dtype)) return PA_ERR_UNSUPPORTED;
  if (num_pairs == 0) return PA_OK;
  if (!k_pool || !v_pool || !block_pairs) return PA_ERR_INVALID_ARG;
  if (!aligned16(k_pool) || !aligned16(v_pool)) return PA_ERR_INVALID_ARG;
  const int64_t block_elems = (int64_t)block_size * num_kv_heads * head_dim;
  if (block_elems / 8 > 0x7FFFFFFF) return PA_ERR_INVALID_ARG;
  if (launch_pdl(copy_blocks_kernel, dim3((unsigned)num_pairs, 2), 256, 0, stream, (uint4*)k_pool,
                 (uint4*)v_pool, block_pairs, (int)(block_elems / 8), num_blocks,
                 status_dev) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

extern "C" pa_status pa_decode_slots(int32_t* slot_mapping, const int32_t* block_tables,
                                     const int32_t* seq_lens, int num_seqs, int max_blocks,
                                     int block_size, int num_blocks, int32_t* status_dev,
                                     cudaStream_t stream) {
  if (num_seqs < 0 || max_blocks <= 0 || block_size <= 0 || num_blocks <= 0)
    return PA_ERR_INVALID_ARG;
  // every slot of the pool is an int32
  if ((long long)num_blocks * block_size > 0x7FFFFFFFll) return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) return PA_OK;
  if (!slot_mapping || !block_tables || !seq_lens) return PA_ERR_INVALID_ARG;
  if (launch_pdl(decode_slots_kernel, dim3((unsigned)((num_seqs + 127) / 128)), 128, 0, stream,
                 slot_mapping, block_tables, seq_lens, num_seqs, max_blocks, block_size,
                 num_blocks, status_dev) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

extern "C" pa_status pa_append_tokens(void* k_pool, void* v_pool, const void* key,
                                      const void* value, const int32_t* block_tables,
                                      const int32_t* seq_lens, int32_t* slot_mapping,
                                      int num_seqs, int64_t kv_token_stride, int num_kv_heads,
                                      int head_dim, int block_size, int max_blocks,
                                      int num_blocks, int dtype, int32_t* status_dev,
                                      cudaStream_t stream) {
  if (num_seqs < 0 || num_kv_heads <= 0 || num_blocks <= 0 || max_blocks <= 0)
    return PA_ERR_INVALID_ARG;
  if (!supported_shape(head_dim, block_size, dtype)) return PA_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PA_OK;
  if (!k_pool || !v_pool || !key || !value || !block_tables || !seq_lens)
    return PA_ERR_INVALID_ARG;
  const int64_t row_elems = (int64_t)num_kv_heads * head_dim;
  const int64_t stride = kv_token_stride == 0 ? row_elems : kv_token_stride;
  if (stride < row_elems || (stride % 8) != 0) return PA_ERR_INVALID_ARG;
  if (!aligned16(k_pool) || !aligned16(v_pool) || !aligned16(key) || !aligned16(value))
    return PA_ERR_INVALID_ARG;
  const int row_vecs = (int)(row_elems / 8);
  const int64_t grid = ((int64_t)num_seqs * row_vecs + 255) / 256;
  if (grid > 0x7FFFFFFF) return PA_ERR_INVALID_ARG;
  if (launch_pdl(append_tokens_kernel, dim3((unsigned)grid), 256, 0, stream, (uint4*)k_pool,
                 (uint4*)v_pool, (const uint4*)key, (const uint4*)value, block_tables, seq_lens,
                 slot_mapping, num_seqs, (int64_t)(stride / 8), row_vecs, block_size, max_blocks,
                 (int64_t)num_blocks * block_size, status_dev) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}
