// Whole-block moves between pools, many pools per launch:
//
//   pa_copy_blocks_multi  copy-on-write clones in the K and V pools of every
//                         layer at once (one launch instead of one per layer);
//   pa_swap_blocks        blocks between the GPU pools and pools in page-locked
//                         host memory (the PagedAttention glossary page names
//                         moving evicted blocks to host memory as an extension).
//
// Both are the same gather/scatter: for every (src, dst) pair and every pool i,
// block dst of dst_pools[i] receives the bytes of block src of src_pools[i].
// On GB300 the host pools sit behind NVLink-C2C, which the GPU reaches with
// ordinary loads and stores through the mapped address of page-locked memory, so
// a swap is one kernel over all blocks and layers rather than one copy-engine
// transfer per block and layer.  The kernel keeps many 16-byte accesses in
// flight per thread: the host link has microseconds of latency.
#include <mutex>

#include "pa_common.cuh"

namespace pa {
namespace {

constexpr int kMaxPools = 512;          // 2 pools (K, V) x 256 layers
constexpr int kSegThreads = 256;
constexpr int kSegUnroll = 8;           // 16-byte vectors per thread per segment
constexpr int kSegVecs = kSegThreads * kSegUnroll;   // 32 KiB per segment

struct PoolSet {
  uint4* dst[kMaxPools];
  const uint4* src[kMaxPools];
};

// Work item u = ((pair * num_pools) + pool) * segs + seg; a persistent grid
// strides over the items so consecutive CTAs copy neighbouring segments.
__global__ void __launch_bounds__(kSegThreads)
block_move_kernel(const __grid_constant__ PoolSet ps, const int32_t* __restrict__ pairs,
                  int num_pairs, int num_pools, int64_t block_vecs, int segs,
                  int src_num_blocks, int dst_num_blocks, int32_t* status_dev) {
  allow_next_grid();
  wait_prior_grid();
  const int64_t items = (int64_t)num_pairs * num_pools * segs;
  for (int64_t u = blockIdx.x; u < items; u += gridDim.x) {
    const int seg = (int)(u % segs);
    const int64_t pp = u / segs;
    const int pool = (int)(pp % num_pools);
    const int pair = (int)(pp / num_pools);
    const int32_t s = pairs[2 * pair], d = pairs[2 * pair + 1];
    if (s < 0 || s >= src_num_blocks || d < 0 || d >= dst_num_blocks) {
      if (threadIdx.x == 0 && pool == 0 && seg == 0) report(status_dev, PA_ERR_BAD_BLOCK_ID);
      continue;
    }
    const int64_t base = (int64_t)seg * kSegVecs;
    const uint4* from = ps.src[pool] + (int64_t)s * block_vecs + base;
    uint4* to = ps.dst[pool] + (int64_t)d * block_vecs + base;
    const int64_t n = block_vecs - base < kSegVecs ? block_vecs - base : kSegVecs;
    if (n == kSegVecs) {
      uint4 r[kSegUnroll];
#pragma unroll
      for (int k = 0; k < kSegUnroll; ++k) r[k] = from[threadIdx.x + k * kSegThreads];
#pragma unroll
      for (int k = 0; k < kSegUnroll; ++k) to[threadIdx.x + k * kSegThreads] = r[k];
    } else {
      for (int64_t v = threadIdx.x; v < n; v += kSegThreads) to[v] = from[v];
    }
  }
}

int num_sms() {
  static int n = 0;
  static std::once_flag once;
  std::call_once(once, [] {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      n = 0;
  });
  return n > 0 ? n : 1;
}

// Address the GPU uses for p: itself for device memory, the mapped alias for
// page-locked host memory, nullptr for memory the GPU cannot reach (pageable
// host memory, or a pointer the runtime does not know).
const void* device_alias(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();            // a failed query also sets the last-error slot
    return nullptr;
  }
  switch (a.type) {
    case cudaMemoryTypeDevice:
    case cudaMemoryTypeManaged:
      return p;
    case cudaMemoryTypeHost:
      if (!a.devicePointer) return nullptr;
      // the alias of p itself, not of the start of its allocation
      return static_cast<const char*>(a.devicePointer) +
             (static_cast<const char*>(p) - static_cast<const char*>(a.hostPointer));
    default:
      return nullptr;
  }
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

pa_status launch_block_move(PoolSet& ps, const int32_t* pairs, int num_pairs, int num_pools,
                            int64_t block_bytes, int src_num_blocks, int dst_num_blocks,
                            int32_t* status_dev, cudaStream_t stream) {
  const int64_t block_vecs = block_bytes / 16;
  const int64_t segs = (block_vecs + kSegVecs - 1) / kSegVecs;
  const int64_t items = (int64_t)num_pairs * num_pools * segs;
  if (segs > 0x7FFFFFFF || items / num_pools / segs != num_pairs) return PA_ERR_INVALID_ARG;
  // 4 resident CTAs of 256 threads per SM are enough bytes in flight for HBM
  // and for the host link; more CTAs only add scheduling work.
  const int64_t grid = items < (int64_t)num_sms() * 4 ? items : (int64_t)num_sms() * 4;
  if (launch_pdl(block_move_kernel, dim3((unsigned)grid), kSegThreads, 0, stream, ps, pairs,
                 num_pairs, num_pools, block_vecs, (int)segs, src_num_blocks, dst_num_blocks,
                 status_dev) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" pa_status pa_copy_blocks_multi(void* const* pools, int num_pools,
                                          const int32_t* block_pairs, int num_pairs,
                                          int64_t block_bytes, int num_blocks,
                                          int32_t* status_dev, cudaStream_t stream) {
  if (num_pairs < 0 || num_pools <= 0 || num_pools > kMaxPools || block_bytes <= 0 ||
      (block_bytes % 16) != 0 || num_blocks <= 0 || !pools)
    return PA_ERR_INVALID_ARG;
  if (num_pairs == 0) return PA_OK;
  if (!block_pairs) return PA_ERR_INVALID_ARG;
  const int32_t* pairs = static_cast<const int32_t*>(device_alias(block_pairs));
  if (!pairs) return PA_ERR_INVALID_ARG;
  PoolSet ps;
  for (int i = 0; i < num_pools; ++i) {
    if (!pools[i] || !aligned16(pools[i])) return PA_ERR_INVALID_ARG;
    ps.dst[i] = static_cast<uint4*>(pools[i]);
    ps.src[i] = static_cast<const uint4*>(pools[i]);
  }
  return launch_block_move(ps, pairs, num_pairs, num_pools, block_bytes, num_blocks, num_blocks,
                           status_dev, stream);
}

extern "C" pa_status pa_swap_blocks(void* const* dst_pools, const void* const* src_pools,
                                    int num_pools, const int32_t* block_pairs, int num_pairs,
                                    int64_t block_bytes, int src_num_blocks, int dst_num_blocks,
                                    int32_t* status_dev, cudaStream_t stream) {
  if (num_pairs < 0 || num_pools <= 0 || num_pools > kMaxPools || block_bytes <= 0 ||
      (block_bytes % 16) != 0 || src_num_blocks <= 0 || dst_num_blocks <= 0 || !dst_pools ||
      !src_pools)
    return PA_ERR_INVALID_ARG;
  if (num_pairs == 0) return PA_OK;
  if (!block_pairs) return PA_ERR_INVALID_ARG;
  const int32_t* pairs = static_cast<const int32_t*>(device_alias(block_pairs));
  if (!pairs) return PA_ERR_INVALID_ARG;
  PoolSet ps;
  for (int i = 0; i < num_pools; ++i) {
    if (!dst_pools[i] || !src_pools[i]) return PA_ERR_INVALID_ARG;
    void* d = const_cast<void*>(device_alias(dst_pools[i]));
    const void* s = device_alias(src_pools[i]);
    if (!d || !s || !aligned16(d) || !aligned16(s)) return PA_ERR_INVALID_ARG;
    ps.dst[i] = static_cast<uint4*>(d);
    ps.src[i] = static_cast<const uint4*>(s);
  }
  return launch_block_move(ps, pairs, num_pairs, num_pools, block_bytes, src_num_blocks,
                           dst_num_blocks, status_dev, stream);
}
