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
// to the kernels.  The address belongs to the device's current context: when
// that context is destroyed and a new one made (cudaDeviceReset), the module is
// loaded again and the array may move, so the cached address is keyed on the
// context's unique id and looked up again when the id changes.
#include <cuda.h>

#include <mutex>

#include "pa_common.cuh"
#include "pa_internal.h"

static __device__ __align__(256) unsigned char g_decode_scratch[PA_DECODE_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
struct ScratchEntry {
  unsigned long long ctx_id;     // context the address belongs to (0: none yet)
  void* address;
};
ScratchEntry g_scratch[kMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (driver entry points
// looked up once; CUDA 12.0 and later give every context a process-unique id).
pa_status current_context_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* a = nullptr;
    void* b = nullptr;
    cudaDriverEntryPointQueryResult qa, qb;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault,
                                         &qa) == cudaSuccess &&
        qa == cudaDriverEntryPointSuccess &&
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &qb) ==
            cudaSuccess &&
        qb == cudaDriverEntryPointSuccess) {
      get_current = reinterpret_cast<CtxGetCurrentFn>(a);
      get_id = reinterpret_cast<CtxGetIdFn>(b);
    }
  });
  if (!get_current || !get_id) return PA_ERR_CUDA;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return PA_ERR_CUDA;
  return get_id(ctx, id) == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

// Device address of the scratch array on the current device.
pa_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
  // make sure the device's primary context exists and is current (CUDA 12 and
  // later initialise it here; it allocates nothing)
  if (cudaSetDevice(dev) != cudaSuccess) return PA_ERR_CUDA;
  unsigned long long ctx_id = 0;
  const pa_status st = current_context_id(&ctx_id);
  if (st != PA_OK) return st;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  ScratchEntry& e = g_scratch[dev];
  if (e.address == nullptr || e.ctx_id != ctx_id) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return PA_ERR_CUDA;
    e.address = p;
    e.ctx_id = ctx_id;
  }
  *out = e.address;
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
  // Reject before any device work when the kernel that serves the batch needs
  // more scratch than the array holds.  (Invalid shapes give 0 here and are
  // reported by pa_decode.)
  const size_t need = pa_decode_workspace_bytes_for(num_seqs, num_q_heads, num_kv_heads,
                                                    head_dim, block_size, max_blocks, num_blocks,
                                                    max_seq_len, dtype, partition_tokens);
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
