// C ABI of pa_decode: argument checks, workspace carve-up, kernel choice.
#include <math.h>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Each kernel lays out only what it uses, from offset 0: the grouped kernel its
// stream-K area; the per-head kernel the work queue, the (sequence, partition)
// items and the [B, Hq, P] partials; the CUDA-core kernel the partials.
WorkspaceLayout workspace_layout(DecodeKernel k, int B, int Hq, int D, int P) {
  const size_t rows = (size_t)B * Hq * P;
  WorkspaceLayout w = {};
  if (k == DecodeKernel::kGrouped) {      // the partials of every query head
    w.sk_off = 0;
    w.total = sk_layout(B, Hq).total;
    return w;
  }
  size_t off = 0;
  if (k == DecodeKernel::kPerHead) {
    w.queue_off = 0;                                 // work-queue counters
    w.items_off = 256;                               // (sequence, partition) pairs
    off = w.items_off + align256((size_t)B * P * 2 * sizeof(int));
  }
  w.m_off = off;
  w.l_off = w.m_off + align256(rows * sizeof(float));
  w.acc_off = w.l_off + align256(rows * sizeof(float));
  w.total = w.acc_off + align256(rows * D * sizeof(float));
  return w;
}

// Process-wide kernel choice: a switch for tests and measurements (see
// pa_set_decode_path), read once per call.
static int g_decode_path = PA_DECODE_AUTO;

static bool valid_partition(int pt) { return pt >= 128 && pt <= 1024 && pt % 128 == 0; }

// The kernel a call runs: the grouped tensor-core kernel where it serves the
// shape, else the per-head tensor-core kernel (head_dim 128), else the CUDA-core
// kernel; kNone when the path setting asks for a tensor-core kernel that does
// not serve the call.
DecodeKernel choose_decode_kernel(const DecodeParams& p, int path) {
  if (path != PA_DECODE_SIMT && path != PA_DECODE_TC_HEAD && tcg_supported(p))
    return DecodeKernel::kGrouped;
  const bool per_head = path != PA_DECODE_SIMT && tc_supported(p);
  if ((path == PA_DECODE_TC || path == PA_DECODE_TC_HEAD) && !per_head)
    return DecodeKernel::kNone;
  return per_head ? DecodeKernel::kPerHead : DecodeKernel::kSimt;
}

}  // namespace pa

using namespace pa;

extern "C" const char* pa_status_string(int status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported dtype, head_dim or block_size";
    case PA_ERR_WORKSPACE: return "workspace missing or too small";
    case PA_ERR_CUDA: return "CUDA error";
    case PA_ERR_BAD_BLOCK_ID: return "invalid block id, slot or sequence length in device data";
    case PA_ERR_OUT_OF_BLOCKS: return "no free KV block left";
    case PA_ERR_BLOCK_STATE: return "block or sequence in the wrong state";
    case PA_ERR_TIMEOUT: return "a kernel's bounded wait expired; results are incomplete";
    default: return "unknown status";
  }
}

extern "C" int pa_version(void) { return 100; }

extern "C" size_t pa_decode_workspace_bytes(int num_seqs, int num_q_heads, int head_dim,
                                            int max_seq_len, int partition_tokens) {
  const int pt = partition_tokens == 0 ? kDefaultPartitionTokens : partition_tokens;
  if (num_seqs < 0 || num_q_heads <= 0 || head_dim <= 0 || max_seq_len < 0 ||
      !valid_partition(pt))
    return 0;
  const int P = max(1, num_partitions(max_seq_len, pt));
  // enough for whichever kernel runs
  const size_t a = workspace_layout(DecodeKernel::kGrouped, num_seqs, num_q_heads, head_dim, P).total;
  const size_t b = workspace_layout(DecodeKernel::kPerHead, num_seqs, num_q_heads, head_dim, P).total;
  return a > b ? a : b;
}

// Host-side checks shared by pa_decode and the workspace query: fills the
// shape fields of p; returns PA_OK or the status pa_decode would return.
static pa_status check_shape(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                             int block_size, int max_blocks, int num_blocks, int max_seq_len,
                             int dtype, int partition_tokens, DecodeParams* p) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_blocks <= 0 ||
      num_blocks <= 0 || max_seq_len < 0)
    return PA_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads) return PA_ERR_INVALID_ARG;
  if (!(head_dim == 64 || head_dim == 128)) return PA_ERR_UNSUPPORTED;
  if (!(block_size == 8 || block_size == 16 || block_size == 32 || block_size == 64))
    return PA_ERR_UNSUPPORTED;
  if (dtype != PA_FLOAT16 && dtype != PA_BFLOAT16) return PA_ERR_UNSUPPORTED;
  const int pt = partition_tokens == 0 ? kDefaultPartitionTokens : partition_tokens;
  if (!valid_partition(pt) || pt % block_size) return PA_ERR_INVALID_ARG;
  if ((long long)max_seq_len > (long long)max_blocks * block_size) return PA_ERR_INVALID_ARG;
  *p = DecodeParams{};
  p->B = num_seqs;
  p->Hq = num_q_heads;
  p->Hkv = num_kv_heads;
  p->D = head_dim;
  p->bs = block_size;
  p->max_blocks = max_blocks;
  p->num_blocks = num_blocks;
  p->max_seq_len = max_seq_len;
  p->dtype = dtype;
  p->PT = pt;
  p->P = max(1, num_partitions(max_seq_len, pt));
  p->Hkv_all = num_kv_heads;
  p->Hq_all = num_q_heads;
  p->head_off = 0;
  return PA_OK;
}

extern "C" size_t pa_decode_workspace_bytes_for(int num_seqs, int num_q_heads, int num_kv_heads,
                                                int head_dim, int block_size, int max_blocks,
                                                int num_blocks, int max_seq_len, int dtype,
                                                int partition_tokens) {
  DecodeParams p;
  if (check_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks,
                  num_blocks, max_seq_len, dtype, partition_tokens, &p) != PA_OK)
    return 0;
  const DecodeKernel k = choose_decode_kernel(p, g_decode_path);
  if (k == DecodeKernel::kNone) return 0;
  return workspace_layout(k, p.B, p.Hq, p.D, p.P).total;
}

extern "C" int pa_decode_kernel_for(int num_seqs, int num_q_heads, int num_kv_heads,
                                    int head_dim, int block_size, int max_blocks, int num_blocks,
                                    int max_seq_len, int dtype, int partition_tokens) {
  DecodeParams p;
  if (check_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, max_blocks,
                  num_blocks, max_seq_len, dtype, partition_tokens, &p) != PA_OK)
    return -1;
  switch (choose_decode_kernel(p, g_decode_path)) {
    case DecodeKernel::kGrouped: return PA_KERNEL_GROUPED;
    case DecodeKernel::kPerHead: return PA_KERNEL_PER_HEAD;
    case DecodeKernel::kSimt: return PA_KERNEL_SIMT;
    default: return -1;
  }
}

// pa_decode, optionally preceded by the decode-step cache write of
// pa_append_tokens (new_k / new_v non-null): fused into the grouped tensor-core
// kernel and into the CUDA-core kernel, two launches with the per-head kernel.  Every argument is
// checked before anything is launched.
static pa_status decode_impl(void* out, const void* q, const void* k_pool, const void* v_pool,
                             const void* new_k, const void* new_v,
                             const int32_t* block_tables, const int32_t* seq_lens,
                             int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                             int block_size, int max_blocks, int num_blocks, int max_seq_len,
                             float scale, int dtype, int partition_tokens, void* workspace,
                             size_t workspace_bytes, int32_t* status_dev, cudaStream_t stream) {
  DecodeParams p;
  pa_status st = check_shape(num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                             max_blocks, num_blocks, max_seq_len, dtype, partition_tokens, &p);
  if (st != PA_OK) return st;
  if (!isfinite(scale)) return PA_ERR_INVALID_ARG;
  if (num_seqs == 0) return PA_OK;
  if (!out || !q || !k_pool || !v_pool || !block_tables || !seq_lens) return PA_ERR_INVALID_ARG;
  if ((((uintptr_t)out | (uintptr_t)q | (uintptr_t)k_pool | (uintptr_t)v_pool) & 15u) != 0)
    return PA_ERR_INVALID_ARG;
  const bool append = new_k != nullptr || new_v != nullptr;
  if (append && (!new_k || !new_v || (((uintptr_t)new_k | (uintptr_t)new_v) & 15u) != 0))
    return PA_ERR_INVALID_ARG;
  const DecodeKernel kernel = choose_decode_kernel(p, g_decode_path);
  if (kernel == DecodeKernel::kNone) return PA_ERR_UNSUPPORTED;
  const WorkspaceLayout wl = workspace_layout(kernel, num_seqs, num_q_heads, head_dim, p.P);
  if (!workspace || workspace_bytes < wl.total || ((uintptr_t)workspace & 255u) != 0)
    return PA_ERR_WORKSPACE;

  p.out = out;
  p.q = q;
  p.k_pool = k_pool;
  p.v_pool = v_pool;
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.scale_log2 = (float)((double)scale * 1.4426950408889634);
  char* ws = static_cast<char*>(workspace);
  p.ws_m = reinterpret_cast<float*>(ws + wl.m_off);
  p.ws_l = reinterpret_cast<float*>(ws + wl.l_off);
  p.ws_acc = reinterpret_cast<float*>(ws + wl.acc_off);
  p.status_dev = status_dev;
  p.new_k = nullptr;
  p.new_v = nullptr;

  if (kernel == DecodeKernel::kGrouped) {
    p.new_k = new_k;
    p.new_v = new_v;
    return launch_decode_tcg(p, ws + wl.sk_off, stream);
  }
  const bool per_head = kernel == DecodeKernel::kPerHead;
  const int P = p.P;
  if (append && per_head) {
    st = pa_append_tokens(const_cast<void*>(k_pool), const_cast<void*>(v_pool), new_k, new_v,
                          block_tables, seq_lens, nullptr, num_seqs, 0, num_kv_heads, head_dim,
                          block_size, max_blocks, num_blocks, dtype, status_dev, stream);
    if (st != PA_OK) return st;
  } else if (append) {          // the CUDA-core kernel writes the newest tokens itself
    p.new_k = new_k;
    p.new_v = new_v;
  }
  if (per_head) {
    st = launch_decode_tc(p, reinterpret_cast<int2*>(ws + wl.items_off),
                          reinterpret_cast<int*>(ws + wl.queue_off), stream);
  } else {
    st = launch_decode_simt(p, stream);
  }
  if (st != PA_OK || P == 1) return st;
  return launch_combine(p, stream);
}

extern "C" pa_status pa_decode(void* out, const void* q, const void* k_pool, const void* v_pool,
                               const int32_t* block_tables, const int32_t* seq_lens,
                               int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                               int block_size, int max_blocks, int num_blocks, int max_seq_len,
                               float scale, int dtype, int partition_tokens, void* workspace,
                               size_t workspace_bytes, int32_t* status_dev,
                               cudaStream_t stream) {
  return decode_impl(out, q, k_pool, v_pool, nullptr, nullptr, block_tables, seq_lens, num_seqs,
                     num_q_heads, num_kv_heads, head_dim, block_size, max_blocks, num_blocks,
                     max_seq_len, scale, dtype, partition_tokens, workspace, workspace_bytes,
                     status_dev, stream);
}

extern "C" pa_status pa_decode_append(void* out, const void* q, void* k_pool, void* v_pool,
                                      const void* key, const void* value,
                                      const int32_t* block_tables, const int32_t* seq_lens,
                                      int num_seqs, int num_q_heads, int num_kv_heads,
                                      int head_dim, int block_size, int max_blocks,
                                      int num_blocks, int max_seq_len, float scale, int dtype,
                                      int partition_tokens, void* workspace,
                                      size_t workspace_bytes, int32_t* status_dev,
                                      cudaStream_t stream) {
  if (num_seqs > 0 && (!key || !value)) return PA_ERR_INVALID_ARG;
  return decode_impl(out, q, k_pool, v_pool, key, value, block_tables, seq_lens, num_seqs,
                     num_q_heads, num_kv_heads, head_dim, block_size, max_blocks, num_blocks,
                     max_seq_len, scale, dtype, partition_tokens, workspace, workspace_bytes,
                     status_dev, stream);
}

extern "C" pa_status pa_set_decode_path(int path) {
  if (path != PA_DECODE_AUTO && path != PA_DECODE_SIMT && path != PA_DECODE_TC &&
      path != PA_DECODE_TC_HEAD)
    return PA_ERR_INVALID_ARG;
  g_decode_path = path;
  return PA_OK;
}
