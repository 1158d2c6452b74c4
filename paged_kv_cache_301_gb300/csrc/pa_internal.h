// Internal launch interface shared by libpagedattn's translation units.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/pagedattn.h"

namespace pa {

// Everything a decode launch needs, resolved on the host.
struct DecodeParams {
  void* out;
  const void* q;
  const void* k_pool;
  const void* v_pool;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  int B, Hq, Hkv, D, bs, max_blocks, num_blocks, max_seq_len;
  float scale_log2;      // softmax scale * log2(e): scores are kept in base 2
  int dtype;
  int PT;                // tokens per split-K partition
  int P;                 // partitions of the longest allowed sequence
  float* ws_m;           // [B, Hq, P] running max (base 2) per partition
  float* ws_l;           // [B, Hq, P] sum of exp2(s - m) per partition
  float* ws_acc;         // [B, Hq, P, D] unnormalised partial outputs
  int32_t* status_dev;   // nullable: checked mode
  // Decode-step cache write done inside the grouped kernel (both null: none).
  // new_k[b] / new_v[b] ([Hkv, D], packed) become the pool rows of token
  // seq_lens[b] - 1 before any load of that token's tile.
  const void* new_k;
  const void* new_v;
  // Head group served by this launch (the grouped tensor-core kernel splits
  // wide head counts into passes): KV heads head_off .. head_off + Hkv - 1 of
  // Hkv_all in every pool and new-token row, query heads head_off * G .. of
  // Hq_all in every q / out row.  Hkv_all = Hkv, Hq_all = Hq, head_off = 0 for
  // a launch over all heads.
  int Hkv_all, Hq_all, head_off;
};

// The decode kernels; which one serves a call depends on its shape and on the
// process-wide path setting (pa_set_decode_path).
enum class DecodeKernel { kGrouped, kPerHead, kSimt, kNone };
DecodeKernel choose_decode_kernel(const DecodeParams& p, int path);

// Workspace carve-up of one kernel (offsets of the parts it uses; total bytes).
struct WorkspaceLayout {
  size_t queue_off, items_off, m_off, l_off, acc_off, sk_off, total;
};
WorkspaceLayout workspace_layout(DecodeKernel k, int B, int Hq, int D, int P);

pa_status launch_decode_simt(const DecodeParams& p, cudaStream_t stream);
pa_status launch_combine(const DecodeParams& p, cudaStream_t stream);

// Tensor-core path, one KV head per work item (head_dim 128): plan kernel +
// persistent tcgen05 kernel; partials go to the [B, Hq, P] workspace arrays.
bool tc_supported(const DecodeParams& p);
pa_status launch_decode_tc(const DecodeParams& p, int2* items, int* queue, cudaStream_t stream);

// Tensor-core path, all KV heads of a block per CTA with a stream-K split
// (head_dim 128, G in {1,2,4,8,16}, or 3, 5, 6, 7 in passes of 4 or 8 KV
// heads; up to 32768 sequences): main + combine,
// once per group of KV heads with at most 64 query heads.
constexpr int kSkMaxGrid = 160;          // persistent CTAs at most (GB300: 152 SMs)
struct SkLayout {
  size_t prefix_off, wprefix_off, m_off, l_off, acc_off, total;
};
SkLayout sk_layout(int B, int Hq);
bool tcg_supported(const DecodeParams& p);
pa_status launch_decode_tcg(const DecodeParams& p, void* sk_ws, cudaStream_t stream);

// Prefill (causal multi-query attention over the pool), resolved on the host.
struct PrefillArgs {
  void* out;
  const void* q;
  const void* k_pool;
  const void* v_pool;
  const int32_t* tables;
  const int32_t* seq_lens;
  const int32_t* q_start;
  int B, total_q, Hq, Hkv, D, bs, max_blocks, num_blocks, max_q_len;
  float scale_log2;
  int dtype;
  int32_t* status_dev;
};
// CUDA-core kernel for every supported shape (head_dim 64 or 128, any group).
pa_status launch_prefill_simt(const PrefillArgs& a, cudaStream_t stream);

}  // namespace pa
