// pa_prefill on the CUDA cores: the same causal multi-query attention over the
// paged pool as the tensor-core kernel (subroutine-cs article, introduction: the
// prefill phase; "10 — Paged Attention" §5 "The kernel side" for the gather), for
// the shapes that kernel does not serve (head_dim 64, query groups other than
// 1/2/4/8/16).
//
// One warp per (query row, query head).  Keys are visited in chunks of 32: each
// lane scores one key (its K row read whole, q from shared memory), the warp
// takes the chunk's max and sum (online softmax in base 2), then the lanes switch
// to columns and accumulate the chunk's V rows (coalesced, p passed by shuffle).
#include <math_constants.h>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr int kWarps = 8;

template <int DT, int D>
__global__ void __launch_bounds__(32 * kWarps)
prefill_simt_kernel(const PrefillArgs a) {
  constexpr int PER = D / 32;                    // output columns per lane
  __shared__ float qsh[kWarps][D];
  allow_next_grid();
  wait_prior_grid();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t wid = (int64_t)blockIdx.x * kWarps + warp;
  if (wid >= (int64_t)a.total_q * a.Hq) return;  // whole warps only
  const int row = (int)(wid / a.Hq), hq = (int)(wid - (int64_t)row * a.Hq);
  int lo = 0, hi = a.B - 1;                      // the sequence holding the row
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (a.q_start[mid] <= row) lo = mid;
    else hi = mid - 1;
  }
  const int b = lo, qs = a.q_start[b], n = a.q_start[b + 1] - qs, L = a.seq_lens[b];
  if (qs < 0 || row < qs || row >= qs + n || n > L || n > a.max_q_len ||
      L > a.max_blocks * a.bs || qs + n > a.total_q) {
    if (lane == 0) report(a.status_dev, PA_ERR_BAD_BLOCK_ID);
    return;
  }
  const int pos = L - n + (row - qs);            // keys 0 .. pos are visible
  const int h = hq / (a.Hq / a.Hkv);
  const uint16_t* qrow = static_cast<const uint16_t*>(a.q) + ((int64_t)row * a.Hq + hq) * D;
  for (int d = lane; d < D; d += 32) {
    uint32_t w = qrow[d];
    qsh[warp][d] = widen2<DT>(w).x * a.scale_log2;
  }
  __syncwarp();
  const int32_t* table = a.tables + (int64_t)b * a.max_blocks;
  const uint16_t* kp = static_cast<const uint16_t*>(a.k_pool);
  const uint16_t* vp = static_cast<const uint16_t*>(a.v_pool);
  const int64_t num_slots = (int64_t)a.num_blocks * a.bs;
  float m = -CUDART_INF_F, l = 0.f, acc[PER];
#pragma unroll
  for (int e = 0; e < PER; ++e) acc[e] = 0.f;
  for (int j0 = 0; j0 <= pos; j0 += 32) {
    const int j = j0 + lane;
    float s = -CUDART_INF_F;
    int64_t slot = -1;                           // -1: no row (zeros), past the row or bad id
    if (j <= pos) {
      const int32_t blk = table[j / a.bs];
      slot = (int64_t)blk * a.bs + j % a.bs;
      if (blk < 0 || slot >= num_slots) {        // outside the pool: a zero row
        if (a.status_dev) report(a.status_dev, PA_ERR_BAD_BLOCK_ID);
        slot = -1;
        s = 0.f;
      } else {
        const uint4* k4 = reinterpret_cast<const uint4*>(kp + (slot * a.Hkv + h) * D);
        float dot = 0.f;
#pragma unroll
        for (int c = 0; c < D / 8; ++c) {
          const uint4 v = k4[c];
          const float2 x0 = widen2<DT>(v.x), x1 = widen2<DT>(v.y);
          const float2 x2 = widen2<DT>(v.z), x3 = widen2<DT>(v.w);
          const float* qc = &qsh[warp][c * 8];
          dot = fmaf(qc[0], x0.x, dot);
          dot = fmaf(qc[1], x0.y, dot);
          dot = fmaf(qc[2], x1.x, dot);
          dot = fmaf(qc[3], x1.y, dot);
          dot = fmaf(qc[4], x2.x, dot);
          dot = fmaf(qc[5], x2.y, dot);
          dot = fmaf(qc[6], x3.x, dot);
          dot = fmaf(qc[7], x3.y, dot);
        }
        s = dot;
      }
    }
    float mc = s;
#pragma unroll
    for (int o = 16; o; o >>= 1) mc = fmaxf(mc, __shfl_xor_sync(0xFFFFFFFFu, mc, o));
    const float m_new = fmaxf(m, mc);            // finite: key j0 <= pos is visible
    const float alpha = exp2f(m - m_new);        // 0 on the first chunk
    const float pj = j <= pos ? exp2f(s - m_new) : 0.f;
    float ps = pj;
#pragma unroll
    for (int o = 16; o; o >>= 1) ps += __shfl_xor_sync(0xFFFFFFFFu, ps, o);
    l = fmaf(l, alpha, ps);
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] *= alpha;
    const int kmax = min(32, pos - j0 + 1);
    for (int k = 0; k < kmax; ++k) {
      const float pk = __shfl_sync(0xFFFFFFFFu, pj, k);
      const long long sk = __shfl_sync(0xFFFFFFFFu, (long long)slot, k);
      if (sk < 0) continue;                      // zero row
      const uint16_t* vrow = vp + (sk * a.Hkv + h) * D + lane * PER;
      if constexpr (PER == 4) {
        const uint2 v = *reinterpret_cast<const uint2*>(vrow);
        const float2 x0 = widen2<DT>(v.x), x1 = widen2<DT>(v.y);
        acc[0] = fmaf(pk, x0.x, acc[0]);
        acc[1] = fmaf(pk, x0.y, acc[1]);
        acc[2] = fmaf(pk, x1.x, acc[2]);
        acc[3] = fmaf(pk, x1.y, acc[3]);
      } else {
        const float2 x0 = widen2<DT>(*reinterpret_cast<const uint32_t*>(vrow));
        acc[0] = fmaf(pk, x0.x, acc[0]);
        acc[1] = fmaf(pk, x0.y, acc[1]);
      }
    }
    m = m_new;
  }
  const float inv = 1.f / l;
  uint16_t* orow = static_cast<uint16_t*>(a.out) + ((int64_t)row * a.Hq + hq) * D + lane * PER;
  if constexpr (PER == 4) {
    uint2 o;
    o.x = narrow2<DT>(acc[0] * inv, acc[1] * inv);
    o.y = narrow2<DT>(acc[2] * inv, acc[3] * inv);
    *reinterpret_cast<uint2*>(orow) = o;
  } else {
    *reinterpret_cast<uint32_t*>(orow) = narrow2<DT>(acc[0] * inv, acc[1] * inv);
  }
}

template <int DT, int D>
pa_status launch(const PrefillArgs& a, cudaStream_t stream) {
  const int64_t warps = (int64_t)a.total_q * a.Hq;
  const int64_t grid = (warps + kWarps - 1) / kWarps;
  if (grid > 0x7FFFFFFF) return PA_ERR_INVALID_ARG;
  if (launch_pdl(prefill_simt_kernel<DT, D>, dim3((unsigned)grid), 32 * kWarps, 0, stream, a) !=
      cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

}  // namespace

pa_status launch_prefill_simt(const PrefillArgs& a, cudaStream_t stream) {
  if (a.dtype == PA_BFLOAT16)
    return a.D == 128 ? launch<PA_BFLOAT16, 128>(a, stream) : launch<PA_BFLOAT16, 64>(a, stream);
  return a.D == 128 ? launch<PA_FLOAT16, 128>(a, stream) : launch<PA_FLOAT16, 64>(a, stream);
}

}  // namespace pa
