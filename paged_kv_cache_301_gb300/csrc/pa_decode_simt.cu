// pa_decode on CUDA cores, and the split-K combine pass.
//
// One CTA (4 warps) per (partition, KV head, query-head chunk, sequence).  The
// CTA walks the block table of its sequence over its partition's tokens
// ("10 — Paged Attention" tutorial, §5 "The kernel side": one table load per
// block, then the rows of that physical block), in three phases:
//   1. scores  s_t = log2(e) * scale * q . K[slot_t]: a token's row is split
//      over D/8 lanes that each load one 16-byte vector and reduce the partial
//      dot products with warp shuffles; several rows in flight per lane;
//   2. softmax over the partition (max, exp2, sum) per query head;
//   3. p . V: each lane owns one 16-byte slice of head_dim and accumulates
//      p_t * V[slot_t] over a subset of tokens; partial sums meet in shared
//      memory.
// The query heads of a KV head (G = Hq / Hkv) share every K/V row the CTA
// loads, so rows are read once per KV head, not once per query head.
// A sequence that fits one partition writes its output directly; otherwise the
// partition's (max, sum, accumulator) go to the workspace and the combine
// kernel merges them (exact: rescaling by exp2(m_p - M)).
#include <math_constants.h>

#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

constexpr unsigned kFull = 0xFFFFFFFFu;

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}

__device__ __forceinline__ uint4 load_nc(const void* p) {
  return __ldg(reinterpret_cast<const uint4*>(p));
}

template <int DT>
__device__ __forceinline__ void widen8(const uint4& w, float (&x)[8]) {
  float2 a = widen2<DT>(w.x), b = widen2<DT>(w.y), c = widen2<DT>(w.z), d = widen2<DT>(w.w);
  x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
  x[4] = c.x; x[5] = c.y; x[6] = d.x; x[7] = d.y;
}

// Clamp a sequence length to [0, max_seq_len] (the host checked max_seq_len
// against the table capacity), reporting an out-of-range length in checked mode.
__device__ __forceinline__ int clamp_len(const DecodeParams& p, int b, bool report_here) {
  int L = p.seq_lens[b];
  if (L < 0 || L > p.max_seq_len) {
    if (report_here) report(p.status_dev, PA_ERR_BAD_BLOCK_ID);
    L = L < 0 ? 0 : p.max_seq_len;
  }
  return L;
}

template <int DT, int D, int GP>
__global__ void __launch_bounds__(128)
decode_simt_kernel(const DecodeParams p) {
  constexpr int VEC = 8;           // elements per 16-byte vector
  constexpr int TG = D / VEC;      // lanes sharing one token row
  constexpr int TPW = 32 / TG;     // rows a warp covers per pass
  constexpr int NW = 4;            // warps per CTA
  constexpr int U = 4;             // rows in flight per lane
  constexpr int NGRP = 128 / TG;   // token groups in the p.V phase
  extern __shared__ float smem[];  // scores [GP][PT], then partial sums [NW][GP][D]
  __shared__ float s_m[GP], s_l[GP];

  const int part = blockIdx.x;
  const int G = p.Hq / p.Hkv;
  const int chunks = (G + GP - 1) / GP;
  const int h = blockIdx.y / chunks;
  const int g0 = (blockIdx.y - h * chunks) * GP;
  const int gn = min(GP, G - g0);
  const int b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int L = clamp_len(p, b, part == 0 && blockIdx.y == 0 && tid == 0);
  const int hq0 = h * G + g0;
  const int32_t* table = p.block_tables + (int64_t)b * p.max_blocks;
  // Decode-step cache write (pa_decode_append: new_k / new_v non-null): the CTA
  // of partition 0 and the first query-head chunk of each (sequence, KV head)
  // stores head h of the newest token, position seq_lens[b] - 1, in its slot
  // (nothing for a length of 0, or past the table; a bad block id is reported);
  // every CTA that reads that token takes it from new_k / new_v, so no CTA reads
  // a slot while it is written.
  int newest = -1;
  if (p.new_k != nullptr) {
    const int L_raw = p.seq_lens[b];
    if (L_raw == L) newest = L - 1;
    if (part == 0 && g0 == 0) {
      if (L_raw > 0 && L_raw <= p.max_blocks * p.bs) {
        const int pos = L_raw - 1;
        const int32_t blk = table[pos / p.bs];
        if (blk < 0 || blk >= p.num_blocks) {
          if (tid == 0) report(p.status_dev, PA_ERR_BAD_BLOCK_ID);
        } else {
          const int64_t dst = (((int64_t)blk * p.bs + pos % p.bs) * p.Hkv + h) * D;
          const int64_t src = ((int64_t)b * p.Hkv + h) * D;
          for (int v = tid; v < D / VEC; v += 128) {
            reinterpret_cast<uint4*>(const_cast<void*>(p.k_pool))[dst / VEC + v] =
                reinterpret_cast<const uint4*>(p.new_k)[src / VEC + v];
            reinterpret_cast<uint4*>(const_cast<void*>(p.v_pool))[dst / VEC + v] =
                reinterpret_cast<const uint4*>(p.new_v)[src / VEC + v];
          }
        }
      } else if (L_raw != 0 && tid == 0) {
        report(p.status_dev, PA_ERR_BAD_BLOCK_ID);
      }
    }
  }
  if (L == 0) {   // empty context: a zero output row (+0.0 in fp16 and bf16)
    if (part == 0)
      for (int o = tid; o < gn * D; o += 128)
        static_cast<uint16_t*>(p.out)[((int64_t)b * p.Hq + hq0) * D + o] = 0;
    return;
  }
  const int start = part * p.PT;
  if (start >= L) return;
  const int n = min(p.PT, L - start);
  const int nparts = num_partitions(L, p.PT);
  const int li = lane % TG, sub = lane / TG;
  const bool checked = p.status_dev != nullptr;
  const int bs_shift = __ffs(p.bs) - 1;   // block_size is a power of two
  const int bs_mask = p.bs - 1;

  // this lane's head_dim slice of each query head, scaled into base 2
  float qr[GP][VEC];
  {
    const uint16_t* qb = static_cast<const uint16_t*>(p.q) + ((int64_t)b * p.Hq + hq0) * D + li * VEC;
#pragma unroll
    for (int g = 0; g < GP; ++g) {
      if (g < gn) {
        float x[8];
        widen8<DT>(load_nc(qb + g * D), x);
#pragma unroll
        for (int j = 0; j < VEC; ++j) qr[g][j] = x[j] * p.scale_log2;
      } else {
#pragma unroll
        for (int j = 0; j < VEC; ++j) qr[g][j] = 0.f;
      }
    }
  }

  const int64_t slot_elems = (int64_t)p.Hkv * D;
  const int64_t new_row = ((int64_t)b * p.Hkv + h) * D + li * VEC;   // newest token, head h
  const uint16_t* kbase = static_cast<const uint16_t*>(p.k_pool) + (int64_t)h * D + li * VEC;
  const uint16_t* vbase = static_cast<const uint16_t*>(p.v_pool) + (int64_t)h * D + li * VEC;
  float* s_scores = smem;

  // Phase 1: scores.  The loop bound is uniform per warp (shuffles below).
  for (int wbase = warp * TPW; wbase < n; wbase += NW * TPW * U) {
    uint4 kv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int tl = wbase + sub + u * NW * TPW;
      kv[u] = make_uint4(0, 0, 0, 0);
      if (tl < n) {
        const int t = start + tl;
        const int32_t blk = table[t >> bs_shift];
        if (checked && (blk < 0 || blk >= p.num_blocks)) {
          report(p.status_dev, PA_ERR_BAD_BLOCK_ID);
        } else {
          kv[u] = t == newest ? load_nc(static_cast<const uint16_t*>(p.new_k) + new_row)
                              : load_nc(kbase + (((int64_t)blk << bs_shift) + (t & bs_mask)) * slot_elems);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int tl = wbase + sub + u * NW * TPW;
      float k[8];
      widen8<DT>(kv[u], k);
      float dot[GP];
#pragma unroll
      for (int g = 0; g < GP; ++g) {
        float a = 0.f;
#pragma unroll
        for (int j = 0; j < VEC; ++j) a = fmaf(qr[g][j], k[j], a);
        dot[g] = a;
      }
#pragma unroll
      for (int o = TG / 2; o; o >>= 1) {
#pragma unroll
        for (int g = 0; g < GP; ++g) dot[g] += __shfl_xor_sync(kFull, dot[g], o);
      }
      if (li == 0 && tl < n) {
#pragma unroll
        for (int g = 0; g < GP; ++g)
          if (g < gn) s_scores[g * p.PT + tl] = dot[g];
      }
    }
  }
  __syncthreads();

  // Phase 2: per-head max, exp2 and sum over the partition.
  for (int g = warp; g < gn; g += NW) {
    float* s = s_scores + g * p.PT;
    float m = -CUDART_INF_F;
    for (int i = lane; i < n; i += 32) m = fmaxf(m, s[i]);
    m = warp_max(m);
    float l = 0.f;
    for (int i = lane; i < n; i += 32) {
      const float e = exp2f(s[i] - m);
      s[i] = e;
      l += e;
    }
    l = warp_sum(l);
    if (lane == 0) {
      s_m[g] = m;
      s_l[g] = l;
    }
  }
  __syncthreads();

  // Phase 3: p . V over this thread's token group.
  const int grp = tid / TG;
  float acc[GP][VEC];
#pragma unroll
  for (int g = 0; g < GP; ++g)
#pragma unroll
    for (int j = 0; j < VEC; ++j) acc[g][j] = 0.f;
  for (int tb = grp; tb < n; tb += NGRP * U) {
    uint4 vv[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int tl = tb + u * NGRP;
      vv[u] = make_uint4(0, 0, 0, 0);
      if (tl < n) {
        const int t = start + tl;
        const int32_t blk = table[t >> bs_shift];
        if (!checked || (blk >= 0 && blk < p.num_blocks))
          vv[u] = t == newest ? load_nc(static_cast<const uint16_t*>(p.new_v) + new_row)
                              : load_nc(vbase + (((int64_t)blk << bs_shift) + (t & bs_mask)) * slot_elems);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int tl = tb + u * NGRP;
      if (tl < n) {
        float v[8];
        widen8<DT>(vv[u], v);
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          const float pg = g < gn ? s_scores[g * p.PT + tl] : 0.f;
#pragma unroll
          for (int j = 0; j < VEC; ++j) acc[g][j] = fmaf(pg, v[j], acc[g][j]);
        }
      }
    }
  }
  // token groups inside a warp hold the same head_dim slice: fold them
#pragma unroll
  for (int o = TG; o < 32; o <<= 1)
#pragma unroll
    for (int g = 0; g < GP; ++g)
#pragma unroll
      for (int j = 0; j < VEC; ++j) acc[g][j] += __shfl_xor_sync(kFull, acc[g][j], o);
  __syncthreads();   // scores are dead; reuse the buffer for per-warp sums
  float* red = smem;
  if (lane < TG) {
#pragma unroll
    for (int g = 0; g < GP; ++g)
#pragma unroll
      for (int j = 0; j < VEC; ++j) red[(warp * GP + g) * D + li * VEC + j] = acc[g][j];
  }
  __syncthreads();

  for (int o = tid; o < gn * D; o += 128) {
    const int g = o / D, d = o - g * D;
    float a = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) a += red[(w * GP + g) * D + d];
    const int64_t row = (int64_t)b * p.Hq + hq0 + g;
    if (nparts == 1) {
      static_cast<uint16_t*>(p.out)[row * D + d] = narrow<DT>(a / s_l[g]);
    } else {
      const int64_t idx = row * p.P + part;
      p.ws_acc[idx * D + d] = a;
      if (d == 0) {
        p.ws_m[idx] = s_m[g];
        p.ws_l[idx] = s_l[g];
      }
    }
  }
}

// Merge split-K partials: one warp per (sequence, query head).
//   M = max_p m_p,  out = sum_p acc_p 2^(m_p - M) / sum_p l_p 2^(m_p - M)
template <int DT, int D>
__global__ void __launch_bounds__(128)
combine_kernel(const DecodeParams p) {
  constexpr int PER = D / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 4 + warp;
  if (row >= (int64_t)p.B * p.Hq) return;
  const int b = (int)(row / p.Hq);
  const int L = clamp_len(p, b, false);
  uint16_t* out = static_cast<uint16_t*>(p.out) + row * D + lane * PER;
  const int nparts = num_partitions(L, p.PT);
  if (nparts <= 1) return;                       // written by the main kernel
  const float* m = p.ws_m + row * p.P;
  const float* l = p.ws_l + row * p.P;
  const float* acc = p.ws_acc + row * p.P * D + lane * PER;
  float M = -CUDART_INF_F;
  for (int i = lane; i < nparts; i += 32) M = fmaxf(M, m[i]);
  M = warp_max(M);
  float den = 0.f, o[PER];
#pragma unroll
  for (int j = 0; j < PER; ++j) o[j] = 0.f;
#pragma unroll 4
  for (int i = 0; i < nparts; ++i) {
    const float w = exp2f(m[i] - M);
    den = fmaf(w, l[i], den);
#pragma unroll
    for (int j = 0; j < PER; ++j) o[j] = fmaf(w, acc[(int64_t)i * D + j], o[j]);
  }
  const float inv = 1.f / den;
#pragma unroll
  for (int j = 0; j < PER; ++j) out[j] = narrow<DT>(o[j] * inv);
}

template <int DT, int D, int GP>
static pa_status launch_simt_t(const DecodeParams& p, cudaStream_t stream) {
  const int G = p.Hq / p.Hkv;
  const int chunks = (G + GP - 1) / GP;
  const size_t smem = sizeof(float) * (size_t)max(GP * p.PT, 4 * GP * D);
  if (smem > 48 * 1024) return PA_ERR_UNSUPPORTED;
  const long long gy = (long long)p.Hkv * chunks;
  if (gy > 65535 || p.B > 65535) return PA_ERR_INVALID_ARG;
  dim3 grid((unsigned)p.P, (unsigned)gy, (unsigned)p.B);
  decode_simt_kernel<DT, D, GP><<<grid, 128, smem, stream>>>(p);
  PA_CHECK_LAUNCH();
  return PA_OK;
}

template <int DT, int D>
static pa_status launch_simt_d(const DecodeParams& p, cudaStream_t stream) {
  const int G = p.Hq / p.Hkv;
  if (G <= 1) return launch_simt_t<DT, D, 1>(p, stream);
  if (G <= 2) return launch_simt_t<DT, D, 2>(p, stream);
  if (G <= 4) return launch_simt_t<DT, D, 4>(p, stream);
  return launch_simt_t<DT, D, 8>(p, stream);
}

pa_status launch_decode_simt(const DecodeParams& p, cudaStream_t stream) {
  if (p.dtype == PA_BFLOAT16)
    return p.D == 128 ? launch_simt_d<PA_BFLOAT16, 128>(p, stream)
                      : launch_simt_d<PA_BFLOAT16, 64>(p, stream);
  return p.D == 128 ? launch_simt_d<PA_FLOAT16, 128>(p, stream)
                    : launch_simt_d<PA_FLOAT16, 64>(p, stream);
}

pa_status launch_combine(const DecodeParams& p, cudaStream_t stream) {
  const long long rows = (long long)p.B * p.Hq;
  if (rows == 0) return PA_OK;
  const unsigned grid = (unsigned)((rows + 3) / 4);
  if (p.dtype == PA_BFLOAT16) {
    if (p.D == 128) combine_kernel<PA_BFLOAT16, 128><<<grid, 128, 0, stream>>>(p);
    else combine_kernel<PA_BFLOAT16, 64><<<grid, 128, 0, stream>>>(p);
  } else {
    if (p.D == 128) combine_kernel<PA_FLOAT16, 128><<<grid, 128, 0, stream>>>(p);
    else combine_kernel<PA_FLOAT16, 64><<<grid, 128, 0, stream>>>(p);
  }
  PA_CHECK_LAUNCH();
  return PA_OK;
}

}  // namespace pa
