// pa_decode_noalloc: decode attention for callers that cannot allocate device
// memory.
//
// pa_decode needs a scratch workspace for its split-K partials, which the
// caller normally allocates (cudaMalloc or a framework allocator).  Some
// callers cannot do that at call time: code running inside a CUDA graph
// capture where allocation is not allowed, plug-ins that are handed device
// pointers by a host application that owns all allocations, or real-time
// loops that must not touch the allocator.  This entry point takes its scratch
// from a fixed array that is part of the library's device image instead.
//
// The array is a file-scope __device__ object: it is created when the module
// is loaded on a device and every device that loads the library keeps it
// until the process exits.  In host code the array's name only stands for the
// symbol; its device address is looked up once per device with
// cudaGetSymbolAddress while that device is current, and the pointer is passed
// to the kernels.
#include <mutex>

#include "pa_common.cuh"

static __device__ __align__(256) unsigned char g_decode_scratch[PA_DECODE_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_address[kMaxDevices];   // per device; null until looked up

// Device address of the scratch array on the current device.
pa_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (!g_scratch_address[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return PA_ERR_CUDA;
    g_scratch_address[dev] = p;
  }
  *out = g_scratch_address[dev];
  return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_noalloc(void* out, const void* q, const void* k_pool,
                                       const void* v_pool, const int32_t* block_tables,
                                       const int32_t* seq_lens, int num_seqs, int num_q_heads,
                                       int num_kv_heads, int head_dim, int block_size,
                                       int max_blocks, int num_blocks, int max_seq_len,
                                       float scale, int dtype, int partition_tokens,
                                       int32_t* status_dev, cudaStream_t stream) {
  // Reject before any device work when the batch needs more scratch than the
  // array holds.  (Invalid shapes give 0 here and are reported by pa_decode.)
  const size_t need = pa_decode_workspace_bytes(num_seqs, num_q_heads, head_dim, max_seq_len,
                                                partition_tokens);
  if (need > (size_t)PA_DECODE_NOALLOC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const pa_status st = scratch_address(&scratch);
  if (st != PA_OK) return st;
  // Nothing in the scratch has to start at zero: every partial the combine
  // pass reads is written earlier in the same call.
  return pa_decode(out, q, k_pool, v_pool, block_tables, seq_lens, num_seqs, num_q_heads,
                   num_kv_heads, head_dim, block_size, max_blocks, num_blocks, max_seq_len,
                   scale, dtype, partition_tokens, scratch,
                   (size_t)PA_DECODE_NOALLOC_SCRATCH_BYTES, status_dev, stream);
}
