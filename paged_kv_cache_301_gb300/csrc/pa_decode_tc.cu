// pa_decode on the Blackwell tensor cores (tcgen05 + TMEM) with TMA staging.
//
// The gather of a sequence's K/V rows through its block table ("10 — Paged
// Attention" tutorial, §5 "The kernel side") is done by TMA: one 3-D tiled copy
// per (physical block, 64-element half of head_dim), box {64, 1, block_size}
// over the pool viewed as [NB*bs tokens][Hkv][D], into 128-byte-swizzled shared
// memory.  Tokens are processed in tiles of 128; a work item is one
// (sequence, KV head, query-head chunk, partition).
//
// Per tile, with the G <= 16 query heads of the KV head packed as the N=16
// dimension of the MMA:
//   S^T[128 tok x 16] = K_tile[128 x D] . Q^T[D x 16]        (tcgen05, TMEM)
//   softmax warps: scores -> running max (base 2) -> P = exp2(s - m), stored as
//     two storage-type terms P_hi + P_lo (about 16 significant bits: one bf16
//     term alone would perturb each weight by up to 2^-9)
//   O^T[D x 16] = V_tile^T . P_hi^T + V_tile^T . P_lo^T      (tcgen05, TMEM)
//   O accumulates in registers (thread d owns row d of O^T) with the
//   online-softmax rescale exp2(m_old - m_new).
//
// Roles (192 threads, one persistent CTA per SM):
//   warp 0      producer: fetches work items from a queue, loads block ids, issues TMA
//   warp 1      TMEM allocation and the single-thread MMA issue
//   warps 2-5   softmax / epilogue; warp w reads TMEM lanes 32*(w%4) .. +31
// Stages flow through a 6-deep ring of 32 KB shared-memory buffers (K and V
// tiles alternate), tracked by mbarriers.  Every wait is bounded: on timeout the
// CTA raises an abort flag, drains its in-flight copies and MMAs, frees TMEM and
// reports PA_ERR_TIMEOUT through status_dev.
//
// A plan kernel (one CTA) runs first: it lists the (sequence, partition) pairs
// to process, full partitions first and each sequence's partial last partition
// after them, writes zero rows for empty sequences, and resets the queue.
#include <math_constants.h>

#include <mutex>

#include "pa_common.cuh"
#include "pa_internal.h"
#include "pa_sm100.cuh"

namespace pa {
namespace {

using namespace sm100;

constexpr int kD = 128;               // head_dim handled by this kernel
constexpr int kTile = 128;            // tokens per MMA tile (M of the S MMA)
constexpr int kN = 16;                // query heads per MMA (N)
constexpr int kStages = 6;            // K/V ring depth
constexpr int kSlabBytes = kTile * 128;        // 128 rows x 128 B (64 elements)
constexpr int kStageBytes = 2 * kSlabBytes;    // one K or V tile, D = 128
constexpr int kQBytes = 2 * kN * 128;          // 16 rows x 256 B
constexpr int kPHalf = 2 * kN * 128;           // 16 heads x 128 tokens x 2 B
constexpr int kPBytes = 2 * kPHalf;            // P split into hi + lo storage values
constexpr int kMaxIds = 1024 / 8;     // block ids per item (partition <= 1024, bs >= 8)
constexpr int kThreads = 192;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s
constexpr uint32_t kTmemCols = 64;    // S: cols [0,32), O: cols [32,64)

struct ItemInfo {
  int b, h, g0, gn, part, start, n, single;   // single: the sequence has one partition
  int valid;                                   // 1 = work, 0 = end of queue
  int pad[3];
};

struct alignas(8) Barriers {
  uint64_t full[kStages], empty[kStages];
  uint64_t item_full[2], item_empty[2];
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full[2], s_empty[2];
  uint64_t p_full[2], p_empty[2];
  uint64_t o_full[2], o_empty[2];
  uint64_t red[2], lsum, drain;
};

struct SmemTail {
  Barriers bar;
  ItemInfo items[2];
  int ids[kMaxIds];
  float red[2][4][kN];
  float lred[4][kN];
  uint32_t tmem_base;
  int abort_flag;
};

constexpr int kRingOff = 0;
constexpr int kQOff = kRingOff + kStages * kStageBytes;
constexpr int kPOff = kQOff + 2 * kQBytes;
constexpr int kTailOff = kPOff + 2 * kPBytes;
constexpr int kSmemBytes = kTailOff + (int)sizeof(SmemTail) + 1024;   // + alignment slack
static_assert(kSmemBytes <= 232448, "shared memory over the per-block limit");

struct TcParams {
  DecodeParams p;
  int2* items;         // (b, partition) pairs, written by the plan kernel
  int* queue;          // [0]: next work item, [1]: number of pairs
  int hc;              // Hkv * query-head chunks
  int chunks;
};

__device__ __forceinline__ void set_abort(SmemTail* t, int32_t* status_dev) {
  t->abort_flag = 1;
  report(status_dev, PA_ERR_TIMEOUT);
}

__device__ __forceinline__ int clamp_seq_len(const DecodeParams& p, int b) {
  int L = p.seq_lens[b];
  return L < 0 ? 0 : (L > p.max_seq_len ? p.max_seq_len : L);
}

// Reduce N values (one per query head) over the 32 lanes of a warp.  Halving
// exchanges: after them lane l holds the reduction of head l >> (5 - log2 N).
template <int N, bool MAX>
__device__ __forceinline__ float warp_reduce_heads(const float (&v)[N], int lane) {
  float cur[N];
#pragma unroll
  for (int i = 0; i < N; ++i) cur[i] = v[i];
  int width = N;
  int bit = 16;
#pragma unroll
  for (int step = 0; step < 5; ++step) {
    if (width > 1) {
      const int half = width >> 1;
      const bool upper = (lane & bit) != 0;
#pragma unroll
      for (int i = 0; i < N / 2; ++i) {
        if (i < half) {
          const float send = upper ? cur[i] : cur[i + half];
          const float keep = upper ? cur[i + half] : cur[i];
          const float got = __shfl_xor_sync(0xFFFFFFFFu, send, bit);
          cur[i] = MAX ? fmaxf(keep, got) : keep + got;
        }
      }
      width = half;
    } else {
      const float got = __shfl_xor_sync(0xFFFFFFFFu, cur[0], bit);
      cur[0] = MAX ? fmaxf(cur[0], got) : cur[0] + got;
    }
    bit >>= 1;
  }
  return cur[0];
}

template <int N>
__device__ __forceinline__ constexpr int head_shift() {
  return N == 16 ? 1 : (N == 8 ? 2 : (N == 4 ? 3 : (N == 2 ? 4 : 5)));
}

template <int DT, int GP>
__global__ void __launch_bounds__(kThreads, 1)
decode_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v,
                 const __grid_constant__ CUtensorMap tm_q, const TcParams tp) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  SmemTail* tail = reinterpret_cast<SmemTail*>(smem + kTailOff);
  Barriers& bar = tail->bar;
  volatile int* abort_flag = &tail->abort_flag;
  const DecodeParams& p = tp.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.Hq / p.Hkv;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bar.full[s], 1);
      mbar_init(&bar.empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar.item_full[i], 1);
      mbar_init(&bar.item_empty[i], 5);     // MMA warp + 4 softmax warps
      mbar_init(&bar.q_full[i], 1);
      mbar_init(&bar.q_empty[i], 1);
      mbar_init(&bar.s_full[i], 1);
      mbar_init(&bar.s_empty[i], 4);
      mbar_init(&bar.p_full[i], 4);
      mbar_init(&bar.p_empty[i], 1);
      mbar_init(&bar.o_full[i], 1);
      mbar_init(&bar.o_empty[i], 4);
      mbar_init(&bar.red[i], 4);
    }
    mbar_init(&bar.lsum, 4);
    mbar_init(&bar.drain, 1);
    tail->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_q);
  }
  if (warp == 1) {
    tmem_alloc(&tail->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tail->tmem_base;

  const uint32_t ring_addr = smem_addr(smem + kRingOff);
  const uint32_t q_addr = smem_addr(smem + kQOff);
  const uint32_t p_addr = smem_addr(smem + kPOff);

  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    const uint64_t policy = policy_evict_first();
    const int total = tp.queue[1] * tp.hc;
    int stage = 0, stage_phase = 0;       // next ring slot to fill
    int issued[kStages];                  // last fill phase of each slot, -1 = never
#pragma unroll
    for (int s = 0; s < kStages; ++s) issued[s] = -1;
    int q_issued[2] = {-1, -1};
    int item_idx = 0;
    int next = 0;
    if (lane == 0) next = atomicAdd(&tp.queue[0], 1);
    next = __shfl_sync(0xFFFFFFFFu, next, 0);
    bool ok = true;
    for (;;) {
      const int k = next;
      const bool have = k < total;
      if (have) {
        if (lane == 0) next = atomicAdd(&tp.queue[0], 1);   // one item ahead
        next = __shfl_sync(0xFFFFFFFFu, next, 0);
      }
      const int islot = item_idx & 1;
      const int iphase = (item_idx >> 1) & 1;
      ItemInfo it;
      it.valid = 0;
      if (have) {
        const int2 pr = tp.items[k / tp.hc];
        const int hcv = k - (k / tp.hc) * tp.hc;
        it.b = pr.x;
        it.part = pr.y;
        it.h = hcv / tp.chunks;
        it.g0 = (hcv - it.h * tp.chunks) * kN;
        it.gn = min(kN, G - it.g0);
        const int L = clamp_seq_len(p, it.b);
        it.start = it.part * p.PT;
        it.n = min(p.PT, L - it.start);
        it.single = num_partitions(L, p.PT) == 1;
        it.valid = 1;
        // this item's block ids, one lane per block
        const int nblk = (it.n + p.bs - 1) / p.bs;
        const int32_t* table = p.block_tables + (int64_t)it.b * p.max_blocks + it.start / p.bs;
        for (int j = lane; j < nblk; j += 32) {
          const int32_t id = table[j];
          if (p.status_dev && (id < 0 || id >= p.num_blocks))
            report(p.status_dev, PA_ERR_BAD_BLOCK_ID);   // TMA reads zeros out of range
          tail->ids[j] = id;
        }
      }
      __syncwarp();
      // hand the item to the consumers
      if (lane == 0) {
        ok = mbar_wait(&bar.item_empty[islot], iphase ^ 1, abort_flag, kWaitLimitNs);
        if (ok) {
          tail->items[islot] = it;
          mbar_arrive(&bar.item_full[islot]);
        } else {
          set_abort(tail, p.status_dev);
        }
      }
      ok = __shfl_sync(0xFFFFFFFFu, (int)ok, 0) != 0;
      if (!ok || !have) break;
      // query rows of this item (16 rows; rows past the chunk are never used)
      const int qb = item_idx & 1;
      if (lane == 0) {
        ok = mbar_wait(&bar.q_empty[qb], ((item_idx >> 1) & 1) ^ 1, abort_flag, kWaitLimitNs);
        if (ok) {
          mbar_arrive_expect_tx(&bar.q_full[qb], kQBytes);
          const int row0 = it.b * p.Hq + it.h * G + it.g0;
          tma_load_2d(smem + kQOff + qb * kQBytes, &tm_q, &bar.q_full[qb], 0, row0);
          tma_load_2d(smem + kQOff + qb * kQBytes + kN * 128, &tm_q, &bar.q_full[qb], 64, row0);
          q_issued[qb] = (item_idx >> 1) & 1;
        } else {
          set_abort(tail, p.status_dev);
        }
      }
      ok = __shfl_sync(0xFFFFFFFFu, (int)ok, 0) != 0;
      if (!ok) break;
      const int ntiles = (it.n + kTile - 1) / kTile;
      const int blocks_per_tile = kTile / p.bs;
      for (int j = 0; j < ntiles && ok; ++j) {
        const int tile_tokens = min(kTile, it.n - j * kTile);
        const int nb = (tile_tokens + p.bs - 1) / p.bs;
        const uint32_t bytes = (uint32_t)nb * p.bs * 128u * 2u;
        for (int kv = 0; kv < 2 && ok; ++kv) {
          if (lane == 0) {
            ok = mbar_wait(&bar.empty[stage], stage_phase ^ 1, abort_flag, kWaitLimitNs);
            if (ok) mbar_arrive_expect_tx(&bar.full[stage], bytes);
            else set_abort(tail, p.status_dev);
          }
          ok = __shfl_sync(0xFFFFFFFFu, (int)ok, 0) != 0;
          if (!ok) break;
          const CUtensorMap* map = kv == 0 ? &tm_k : &tm_v;
          uint8_t* dst = smem + kRingOff + stage * kStageBytes;
          for (int i = lane; i < nb; i += 32) {
            const int32_t blk = tail->ids[j * blocks_per_tile + i];
            const int row = blk * p.bs;
            tma_load_3d_hint(dst + i * p.bs * 128, map, &bar.full[stage], 0, it.h, row, policy);
            tma_load_3d_hint(dst + kSlabBytes + i * p.bs * 128, map, &bar.full[stage], 64, it.h,
                             row, policy);
          }
          issued[stage] = stage_phase;
          if (++stage == kStages) {
            stage = 0;
            stage_phase ^= 1;
          }
        }
      }
      if (!ok) break;
      ++item_idx;
      __syncwarp();
    }
    if (*abort_flag && lane == 0) {
      // let every copy this warp started land before the CTA exits
      for (int s = 0; s < kStages; ++s)
        if (issued[s] >= 0) mbar_wait_drain(&bar.full[s], issued[s], kWaitLimitNs);
      for (int i = 0; i < 2; ++i)
        if (q_issued[i] >= 0) mbar_wait_drain(&bar.q_full[i], q_issued[i], kWaitLimitNs);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issue --
    constexpr uint32_t ab = DT == PA_BFLOAT16 ? 1u : 0u;
    constexpr uint32_t idesc_s = idesc_f16(ab, 0, 0, kTile, kN);   // K (K-major) x Q (K-major)
    constexpr uint32_t idesc_o = idesc_f16(ab, 1, 0, kD, kN);      // V (MN-major) x P (K-major)
    int stage = 0, stage_phase = 0;
    int tile_g = 0;
    int item_idx = 0;
    bool ok = true;
    bool committed_any = false;
    // p.V for global tile t whose V sits in ring slot vs (fill phase vph)
    auto issue_pv = [&](int t, int vs, int vph) -> bool {
      const int slot = t & 1, ph = (t >> 1) & 1;
      if (!mbar_wait(&bar.full[vs], vph, abort_flag, kWaitLimitNs)) return false;
      if (!mbar_wait(&bar.p_full[slot], ph, abort_flag, kWaitLimitNs)) return false;
      if (!mbar_wait(&bar.o_empty[slot], ph ^ 1, abort_flag, kWaitLimitNs)) return false;
      tc_fence_after();
      const uint32_t vaddr = ring_addr + vs * kStageBytes;
      const uint32_t paddr = p_addr + slot * kPBytes;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint64_t a = smem_desc_sw128(vaddr + kk * 16 * 128, kSlabBytes, 1024);
          const uint64_t b = smem_desc_sw128(
              paddr + half * kPHalf + (kk >> 2) * (kN * 128) + (kk & 3) * 32, 16, 1024);
          mma_f16(tmem + 32 + slot * kN, a, b, idesc_o, (half | kk) != 0);
        }
      }
      mma_commit(&bar.empty[vs]);
      mma_commit(&bar.o_full[slot]);
      mma_commit(&bar.p_empty[slot]);
      return true;
    };
    for (;;) {
      const int islot = item_idx & 1;
      int valid = 0, n = 0;
      if (lane == 0) {
        ok = mbar_wait(&bar.item_full[islot], (item_idx >> 1) & 1, abort_flag, kWaitLimitNs);
        if (ok) {
          valid = tail->items[islot].valid;
          n = tail->items[islot].n;
          mbar_arrive(&bar.item_empty[islot]);
        }
      }
      ok = __shfl_sync(0xFFFFFFFFu, (int)ok, 0) != 0;
      valid = __shfl_sync(0xFFFFFFFFu, valid, 0);
      n = __shfl_sync(0xFFFFFFFFu, n, 0);
      if (!ok) {
        if (lane == 0) set_abort(tail, p.status_dev);
        break;
      }
      if (!valid) break;
      const int qb = item_idx & 1;
      const int ntiles = (n + kTile - 1) / kTile;
      if (lane == 0) {
        ok = mbar_wait(&bar.q_full[qb], (item_idx >> 1) & 1, abort_flag, kWaitLimitNs);
        int prev_vs = -1, prev_vph = 0;
        for (int j = 0; j < ntiles && ok; ++j) {
          const int t = tile_g + j;
          const int slot = t & 1, ph = (t >> 1) & 1;
          const int ks = stage, kph = stage_phase;
          if (++stage == kStages) { stage = 0; stage_phase ^= 1; }
          const int vs = stage, vph = stage_phase;
          if (++stage == kStages) { stage = 0; stage_phase ^= 1; }
          ok = mbar_wait(&bar.full[ks], kph, abort_flag, kWaitLimitNs) &&
               mbar_wait(&bar.s_empty[slot], ph ^ 1, abort_flag, kWaitLimitNs);
          if (!ok) break;
          tc_fence_after();
          const uint32_t kaddr = ring_addr + ks * kStageBytes;
          const uint32_t qaddr = q_addr + qb * kQBytes;
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kSlabBytes + (kk & 3) * 32;
            const uint32_t qoff = (kk >> 2) * (kN * 128) + (kk & 3) * 32;
            mma_f16(tmem + slot * kN, smem_desc_sw128(kaddr + off, 16, 1024),
                    smem_desc_sw128(qaddr + qoff, 16, 1024), idesc_s, kk > 0);
          }
          mma_commit(&bar.empty[ks]);
          mma_commit(&bar.s_full[slot]);
          if (j == ntiles - 1) mma_commit(&bar.q_empty[qb]);
          committed_any = true;
          if (j > 0) ok = issue_pv(t - 1, prev_vs, prev_vph);
          prev_vs = vs;
          prev_vph = vph;
        }
        if (ok) ok = issue_pv(tile_g + ntiles - 1, prev_vs, prev_vph);
        if (!ok) set_abort(tail, p.status_dev);
      }
      ok = __shfl_sync(0xFFFFFFFFu, (int)ok, 0) != 0;
      if (!ok) break;
      tile_g += ntiles;
      ++item_idx;
    }
    if (*abort_flag && lane == 0 && committed_any) {
      // wait (bounded) for the MMAs already issued before TMEM is released
      mma_commit(&bar.drain);
      mbar_wait_drain(&bar.drain, 0, kWaitLimitNs);
    }
  } else {
    // ----------------------------------------------------- softmax / epilogue --
    const int wq = warp & 3;                 // TMEM lane quarter of this warp
    const int r = wq * 32 + lane;            // token row of S, d row of O
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    int tile_g = 0;
    int item_idx = 0;
    int red_round = 0;
    int lsum_round = 0;
    bool ok = true;
    auto wait_all = [&](uint64_t* b, int parity) -> bool {
      const bool w = mbar_wait(b, parity, abort_flag, kWaitLimitNs);
      return __all_sync(0xFFFFFFFFu, w);
    };
    for (;;) {
      const int islot = item_idx & 1;
      if (!wait_all(&bar.item_full[islot], (item_idx >> 1) & 1)) { ok = false; break; }
      const ItemInfo it = tail->items[islot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bar.item_empty[islot]);
      if (!it.valid) break;
      const int ntiles = (it.n + kTile - 1) / kTile;
      float m_run[GP], l_t[GP], acc[GP], alpha_prev[GP];
#pragma unroll
      for (int g = 0; g < GP; ++g) {
        m_run[g] = -CUDART_INF_F;
        l_t[g] = 0.f;
        acc[g] = 0.f;
        alpha_prev[g] = 0.f;
      }
      // acc <- acc * exp2(m_{t-1} - m_t) + O_t, the rescale saved from tile t's softmax
      auto accumulate = [&](int t) -> bool {
        const int slot = t & 1, ph = (t >> 1) & 1;
        if (!wait_all(&bar.o_full[slot], ph)) return false;
        tc_fence_after();
        float o[16];
        tmem_ld16(tmem + lane_base + 32 + slot * kN, o);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.o_empty[slot]);
#pragma unroll
        for (int g = 0; g < GP; ++g) acc[g] = fmaf(acc[g], alpha_prev[g], o[g]);
        return true;
      };
      for (int j = 0; j < ntiles && ok; ++j) {
        const int t = tile_g + j;
        const int slot = t & 1, ph = (t >> 1) & 1;
        // scores of this tile
        if (!wait_all(&bar.s_full[slot], ph)) { ok = false; break; }
        tc_fence_after();
        float s[16];
        tmem_ld16(tmem + lane_base + slot * kN, s);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.s_empty[slot]);
        const bool valid = j * kTile + r < it.n;
        float x[GP];
#pragma unroll
        for (int g = 0; g < GP; ++g) x[g] = valid ? s[g] * p.scale_log2 : -CUDART_INF_F;
        // tile maximum per head across the 128 rows
        const float wmax = warp_reduce_heads<GP, true>(x, lane);
        constexpr int hs = head_shift<GP>();
        const int rb = red_round & 1;
        if ((lane & ((1 << hs) - 1)) == 0) tail->red[rb][wq][lane >> hs] = wmax;
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.red[rb]);
        if (!wait_all(&bar.red[rb], (red_round >> 1) & 1)) { ok = false; break; }
        ++red_round;
        float alpha[GP], pr[GP];
#pragma unroll
        for (int g = 0; g < GP; ++g) {
          const float tm = fmaxf(fmaxf(tail->red[rb][0][g], tail->red[rb][1][g]),
                                 fmaxf(tail->red[rb][2][g], tail->red[rb][3][g]));
          const float m_new = fmaxf(m_run[g], tm);
          alpha[g] = exp2f(m_run[g] - m_new);
          pr[g] = valid ? exp2f(x[g] - m_new) : 0.f;
          l_t[g] = fmaf(l_t[g], alpha[g], pr[g]);
          m_run[g] = m_new;
        }
        // P^T operand: row = head, column = token, K-major, 128-byte swizzle
        if (!wait_all(&bar.p_empty[slot], ph ^ 1)) { ok = false; break; }
        uint8_t* pbuf = smem + kPOff + slot * kPBytes + (r >> 6) * (kN * 128);
        const int chunk = (r & 63) >> 3;
#pragma unroll
        for (int g = 0; g < kN; ++g) {
          const float v = (g < GP && g < it.gn) ? pr[g < GP ? g : 0] : 0.f;
          const uint16_t hi = narrow<DT>(v);
          const uint16_t lo = narrow<DT>(v - widen2<DT>(hi).x);
          const int off = g * 128 + ((chunk ^ (g & 7)) << 4) + (r & 7) * 2;
          *reinterpret_cast<uint16_t*>(pbuf + off) = hi;
          *reinterpret_cast<uint16_t*>(pbuf + kPHalf + off) = lo;
        }
        // rows past the end of the sequence: zero their V row so 0 * garbage
        // cannot reach the accumulator
        if ((j + 1) * kTile > it.n) {
          const int u = 2 * t + 1;                 // ring use index of this tile's V
          const int vs = u % kStages, vph = (u / kStages) & 1;
          if (!wait_all(&bar.full[vs], vph)) { ok = false; break; }
          if (!valid) {
            uint4* row0 = reinterpret_cast<uint4*>(smem + kRingOff + vs * kStageBytes + r * 128);
            uint4* row1 = reinterpret_cast<uint4*>(smem + kRingOff + vs * kStageBytes +
                                                   kSlabBytes + r * 128);
            const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
            for (int c = 0; c < 8; ++c) {
              row0[c] = z;
              row1[c] = z;
            }
          }
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.p_full[slot]);
        if (j > 0 && !accumulate(t - 1)) { ok = false; break; }
#pragma unroll
        for (int g = 0; g < GP; ++g) alpha_prev[g] = alpha[g];
      }
      if (!ok) break;
      if (!accumulate(tile_g + ntiles - 1)) { ok = false; break; }
      // softmax denominators: sum the per-row partial sums over the 128 rows
      {
        const float wsum = warp_reduce_heads<GP, false>(l_t, lane);
        constexpr int hs = head_shift<GP>();
        if ((lane & ((1 << hs) - 1)) == 0) tail->lred[wq][lane >> hs] = wsum;
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar.lsum);
        if (!wait_all(&bar.lsum, lsum_round & 1)) { ok = false; break; }
        ++lsum_round;
      }
      const int64_t row0 = (int64_t)it.b * p.Hq + it.h * G + it.g0;
#pragma unroll
      for (int g = 0; g < GP; ++g) {
        if (g < it.gn) {
          const float l = tail->lred[0][g] + tail->lred[1][g] + tail->lred[2][g] +
                          tail->lred[3][g];
          if (it.single) {
            static_cast<uint16_t*>(p.out)[(row0 + g) * kD + r] = narrow<DT>(acc[g] / l);
          } else {
            const int64_t idx = (row0 + g) * p.P + it.part;
            p.ws_acc[idx * kD + r] = acc[g];
            if (r == 0) {
              p.ws_m[idx] = m_run[g];
              p.ws_l[idx] = l;
            }
          }
        }
      }
      // lred is rewritten by the next item only after every warp has passed
      // the next item's first red barrier, which follows these reads
      tile_g += ntiles;
      ++item_idx;
    }
    if (!ok) set_abort(tail, p.status_dev);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// List the (sequence, partition) pairs: full partitions first, then the partial
// last partition of each sequence; zero the output rows of empty sequences;
// reset the work queue.  One CTA of 1024 threads.
__global__ void __launch_bounds__(1024) plan_kernel(const DecodeParams p, int2* items, int* queue) {
  __shared__ int warp_tot[2][32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (p.B + 1023) / 1024;
  const int b0 = min(p.B, tid * per), b1 = min(p.B, b0 + per);
  int full = 0, part = 0;
  for (int b = b0; b < b1; ++b) {
    const int raw = p.seq_lens[b];
    if (raw < 0 || raw > p.max_seq_len) report(p.status_dev, PA_ERR_BAD_BLOCK_ID);
    const int L = clamp_seq_len(p, b);
    const int np = num_partitions(L, p.PT);
    const int f = (L % p.PT == 0) ? np : np - 1;
    full += f;
    part += np - f;
  }
  // exclusive scans of (full, part) over the 1024 threads
  int fi = full, pi = part;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a = __shfl_up_sync(0xFFFFFFFFu, fi, o), c = __shfl_up_sync(0xFFFFFFFFu, pi, o);
    if (lane >= o) {
      fi += a;
      pi += c;
    }
  }
  if (lane == 31) {
    warp_tot[0][warp] = fi;
    warp_tot[1][warp] = pi;
  }
  __syncthreads();
  if (warp == 0) {
    int a = warp_tot[0][lane], c = warp_tot[1][lane];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int x = __shfl_up_sync(0xFFFFFFFFu, a, o), y = __shfl_up_sync(0xFFFFFFFFu, c, o);
      if (lane >= o) {
        a += x;
        c += y;
      }
    }
    warp_tot[0][lane] = a;     // inclusive over warps
    warp_tot[1][lane] = c;
  }
  __syncthreads();
  const int full_total = warp_tot[0][31];
  int foff = fi - full + (warp ? warp_tot[0][warp - 1] : 0);
  int poff = full_total + pi - part + (warp ? warp_tot[1][warp - 1] : 0);
  for (int b = b0; b < b1; ++b) {
    const int L = clamp_seq_len(p, b);
    const int np = num_partitions(L, p.PT);
    const int f = (L % p.PT == 0) ? np : np - 1;
    for (int q = 0; q < f; ++q) items[foff++] = make_int2(b, q);
    if (np > f) items[poff++] = make_int2(b, np - 1);
    if (L == 0) {
      uint16_t* o = static_cast<uint16_t*>(p.out) + (int64_t)b * p.Hq * p.D;
      for (int e = 0; e < p.Hq * p.D; ++e) o[e] = 0;
    }
  }
  if (tid == 0) {
    queue[0] = 0;
    queue[1] = full_total + warp_tot[1][31];
  }
}

// ------------------------------------------------------------ host side --

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

template <int DT, int GP>
pa_status launch_tc_t(const TcParams& tp, const CUtensorMap& k, const CUtensorMap& v,
                      const CUtensorMap& q, int grid, cudaStream_t stream) {
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [] {
    attr_err = cudaFuncSetAttribute(decode_tc_kernel<DT, GP>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  });
  if (attr_err != cudaSuccess) return PA_ERR_CUDA;
  decode_tc_kernel<DT, GP><<<grid, kThreads, kSmemBytes, stream>>>(k, v, q, tp);
  PA_CHECK_LAUNCH();
  return PA_OK;
}

}  // namespace

bool tc_supported(const DecodeParams& p) {
  if (p.D != kD) return false;
  if ((long long)p.num_blocks * p.bs >= (1ll << 31)) return false;
  if ((long long)p.B * p.Hq >= (1ll << 31)) return false;
  if (p.PT > 1024 || p.PT % kTile) return false;
  return encode_fn() != nullptr;
}

pa_status launch_decode_tc(const DecodeParams& p, int2* items, int* queue,
                           cudaStream_t stream) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return PA_ERR_UNSUPPORTED;
  const CUtensorMapDataType dt =
      p.dtype == PA_BFLOAT16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUtensorMap tk, tv, tq;
  const cuuint64_t kv_dims[3] = {(cuuint64_t)kD, (cuuint64_t)p.Hkv,
                                 (cuuint64_t)p.num_blocks * p.bs};
  const cuuint64_t kv_strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)p.Hkv * kD * 2};
  const cuuint32_t kv_box[3] = {64, 1, (cuuint32_t)p.bs};
  const cuuint32_t ones[3] = {1, 1, 1};
  if (enc(&tk, dt, 3, const_cast<void*>(p.k_pool), kv_dims, kv_strides, kv_box, ones,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return PA_ERR_INVALID_ARG;
  if (enc(&tv, dt, 3, const_cast<void*>(p.v_pool), kv_dims, kv_strides, kv_box, ones,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return PA_ERR_INVALID_ARG;
  const cuuint64_t q_dims[2] = {(cuuint64_t)kD, (cuuint64_t)p.B * p.Hq};
  const cuuint64_t q_strides[1] = {(cuuint64_t)kD * 2};
  const cuuint32_t q_box[2] = {64, (cuuint32_t)kN};
  if (enc(&tq, dt, 2, const_cast<void*>(p.q), q_dims, q_strides, q_box, ones,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return PA_ERR_INVALID_ARG;

  TcParams tp;
  tp.p = p;
  tp.items = items;
  tp.queue = queue;
  const int G = p.Hq / p.Hkv;
  tp.chunks = (G + kN - 1) / kN;
  tp.hc = p.Hkv * tp.chunks;

  plan_kernel<<<1, 1024, 0, stream>>>(p, items, queue);
  PA_CHECK_LAUNCH();
  const int grid = sm_count();
  if (grid <= 0) return PA_ERR_CUDA;
  const int gp = G > 8 ? 16 : (G > 4 ? 8 : 4);
  if (p.dtype == PA_BFLOAT16) {
    if (gp == 4) return launch_tc_t<PA_BFLOAT16, 4>(tp, tk, tv, tq, grid, stream);
    if (gp == 8) return launch_tc_t<PA_BFLOAT16, 8>(tp, tk, tv, tq, grid, stream);
    return launch_tc_t<PA_BFLOAT16, 16>(tp, tk, tv, tq, grid, stream);
  }
  if (gp == 4) return launch_tc_t<PA_FLOAT16, 4>(tp, tk, tv, tq, grid, stream);
  if (gp == 8) return launch_tc_t<PA_FLOAT16, 8>(tp, tk, tv, tq, grid, stream);
  return launch_tc_t<PA_FLOAT16, 16>(tp, tk, tv, tq, grid, stream);
}

}  // namespace pa
