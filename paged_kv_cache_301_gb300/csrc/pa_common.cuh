// Shared device helpers of libpagedattn (storage conversions, launch checks).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pagedattn.h"

namespace pa {

constexpr int kDefaultPartitionTokens = 512;

// Number of split-K partitions a sequence of `len` tokens covers.
__host__ __device__ inline int num_partitions(int len, int partition_tokens) {
  return (len + partition_tokens - 1) / partition_tokens;
}

// Two storage elements (one 32-bit word) widened to fp32.
template <int DT>
__device__ __forceinline__ float2 widen2(uint32_t w);

template <>
__device__ __forceinline__ float2 widen2<PA_BFLOAT16>(uint32_t w) {
  // bf16 -> fp32 is the 16-bit pattern placed in the high half of the word
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

template <>
__device__ __forceinline__ float2 widen2<PA_FLOAT16>(uint32_t w) {
  __half2 h = *reinterpret_cast<__half2*>(&w);
  return __half22float2(h);
}

template <int DT>
__device__ __forceinline__ uint16_t narrow(float x);

template <>
__device__ __forceinline__ uint16_t narrow<PA_BFLOAT16>(float x) {
  return __bfloat16_as_ushort(__float2bfloat16_rn(x));
}

template <>
__device__ __forceinline__ uint16_t narrow<PA_FLOAT16>(float x) {
  return __half_as_ushort(__float2half_rn(x));
}

template <int DT>
__device__ __forceinline__ uint32_t narrow2(float a, float b) {
  return (uint32_t)narrow<DT>(a) | ((uint32_t)narrow<DT>(b) << 16);
}

__device__ __forceinline__ void report(int32_t* status_dev, int code) {
  if (status_dev) atomicCAS(status_dev, 0, code);
}

// Programmatic dependent launch.  A kernel launched with launch_pdl may be
// scheduled before the previous kernel in the stream has finished; it calls
// wait_prior_grid() before touching data that kernel produces (returns at once
// when there is no such dependency).  allow_next_grid() lets the next kernel be
// scheduled early; that kernel still waits for this grid to complete.
__device__ __forceinline__ void wait_prior_grid() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void allow_next_grid() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, int threads, int smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

}  // namespace pa

// Map the last launch error to a status code.
#define PA_CHECK_LAUNCH()                                  \
  do {                                                     \
    if (cudaGetLastError() != cudaSuccess) return PA_ERR_CUDA; \
  } while (0)
