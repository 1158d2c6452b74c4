// pa_decode on the tensor cores, all KV heads of a block per CTA (grouped).
//
// A K/V block of the pool stores, per token, the rows of all Hkv heads next to
// each other ([block_size][Hkv][D]), so one TMA copy with box
// {64, Hkv, tokens} fetches a contiguous stretch of the block for all heads.
// Per-head copies fetch 128-byte pieces 2 KB apart, which measured ~30% slower
// on GB300 than whole-block copies.  This kernel therefore gives each CTA all
// heads of a token range:
//
//   tile      = 128 rows = TT = 128 / Hkv tokens x Hkv heads, row = token * Hkv + head
//   S         = K_tile[128 x 128] . Q^T[128 x N]       N = Hq rounded up to 16
//   softmax   row (t, h) keeps the G columns of its own query heads h*G .. h*G+G-1
//   P'        [128 rows x N], block diagonal: P'[(t,h), hq] = p(t, hq) when hq / G == h
//   O^T       [128 x N] += V_tile^T . P'                (V read MN-major from the tile)
// so every query head meets only the rows of its own KV head ("10 — Paged
// Attention" tutorial, §5 "The kernel side": gather through the table; the head
// mapping hq -> hq / G is this library's reading of grouped-query attention).
// P' is stored as two storage-type terms (hi + lo, ~16 significant bits).
//
// Work split (stream-K): the batch is a sequence of token tiles, each sequence
// padded to whole tiles.  A sequence weighs a start weight sw + its tiles
// (starting a sequence costs a CTA its epilogue, the next Q and the refill of
// its pipeline: about one tile's time with two Q / P' buffers, three with one,
// so sw = 1 or 3), and CTA c of the persistent grid
// takes the tiles whose weighted positions fall in [c*W/grid, (c+1)*W/grid), W
// the batch's total weight.  Every CTA gets the same weight to within one,
// whatever the length mix.  A sequence that lies inside one CTA's range is
// written directly; a sequence cut by range boundaries leaves one partial
// (max, sum, accumulator) per CTA, merged by the combine kernel.  Each CTA
// keeps in shared memory only the window of sequences its range meets (at most
// kWin), so the batch size is not bounded by shared memory.  A range of R units
// meets at most R / (sw + 1) + 2 sequences; in a batch so long that R / 2 + 2
// could exceed kWin (more than ~190K tiles, i.e. > 6 GB of K/V, beside hundreds
// of short sequences), sw is raised until it cannot.
//
// Roles (192 threads, one CTA per SM): warp 0 issues TMA, warp 1 issues MMA,
// warps 2-5 run the softmax and the epilogue (and, in pa_decode_append, the
// newest tokens' cache write).  All waits are bounded.
#include <math_constants.h>

#include <mutex>
#include <utility>

#include "pa_common.cuh"
#include "pa_internal.h"
#include "pa_sm100.cuh"

namespace pa {
namespace {

using namespace sm100;

constexpr int kD = 128;
constexpr int kRows = 128;                   // rows per tile (M of the S MMA)
constexpr int kSlab = kRows * 128;           // 128 rows x 128 B
constexpr int kStage = 2 * kSlab;            // one K or V tile
constexpr int kThreads = 192;
constexpr uint64_t kWaitNs = 2000000000ull;

constexpr int kMaxStages = 6;
constexpr int kSmemBudget = 232448 - 1024;   // per-block limit minus alignment slack
constexpr float kRescaleLog2 = 8.f;          // raise a running max only past this (base 2)
constexpr int kWin = 640;                    // sequences of one CTA's range (shared memory)
constexpr int kMaxSeqs = 32768;              // batch size served (also B <= (kWin - 2) grid / 2)


struct SegInfo {
  int b, L, j0, j1;       // sequence, its length, tile range [j0, j1) within it
  int direct, slot;       // direct output, or partial slot 0/1 of this CTA
  int valid, last;        // last: the CTA's final segment
};

template <int N>
struct Tail {
  uint64_t full[kMaxStages], empty[kMaxStages];
  uint64_t seg_full[2], seg_empty[2];
  uint64_t q_full[2], q_empty[2];
  uint64_t s_full[2], s_empty[2];
  uint64_t p_full[2], p_empty[2];
  uint64_t o_full[2], o_empty[2];
  uint64_t red[2], lsum, drain;
  uint64_t red2[2];           // second exchange of a tile whose running maxima rise
  uint64_t app_done;          // newest tokens of this CTA's sequences are in the pool
  uint64_t staged;            // final outputs staged in the ring (one arrive per softmax warp)
  uint64_t p_staged[2];       // a segment's outputs staged in P' buffer i (one arrive per softmax warp)
  uint64_t p_released[2];     // the bulk copy has read P' buffer i
  SegInfo seg[2];
  float red_buf[2][4][N];
  alignas(16) int vote[2][4]; // per tile and softmax warp: a row exceeds its running max + 8
  float alpha[2][N];
  alignas(16) float lred[4][N];
  float m_fin[N];
  // The CTA's window: the non-empty sequences whose tiles meet its range, in
  // batch order.  Entry k is sequence win_b[k], whose tiles are the batch tiles
  // [win_tp[k], win_tp[k+1]).
  int win_b[kWin];
  int win_len[kWin];          // its length (clamped to [0, max_seq_len])
  int win_tp[kWin + 1];
  int nwin;
  int cut[2];                 // the CTA's tile range [cut[0], cut[1])
  int win_n[2];               // non-empty sequences before the window's first / after its last
  int scan[2][4];
  uint32_t tmem_base;
  int abort_flag;
};

template <int H, int G>
struct Geo {
  static constexpr int Hq = H * G;
  static constexpr int N = (Hq + 15) / 16 * 16;
  static constexpr int TT = kRows / H;                   // tokens per tile
  static constexpr int kQBytes = N * 256;
  // For N = 64, Q and P' are single-buffered and the room goes to a fifth ring
  // stage (measured on GB300: long-context decode 90% -> 95% of the HBM peak;
  // N = 48, 40 query heads: 0.90 -> 0.91).  For N = 32 the same trade (six
  // stages) measured slower (82% -> 79.5%): the softmax then waits for the
  // previous P'.V before writing P'.
  static constexpr int kQBufs = N >= 48 ? 1 : 2;
  static constexpr int kPBufs = N >= 48 ? 1 : 2;
  // Least start weight of a sequence, in tiles.  With one Q / P' buffer the
  // next sequence's Q and first scores wait for the previous one's last tile,
  // so nothing of a sequence start overlaps; on GB300 a weight of 3 measured
  // best there (Llama-3-405B-shaped, N = 64: 109.7 -> 104.8 us per step; 40
  // query heads, N = 48: 101.3 -> 97.7 us), and 1 with two buffers (N = 32:
  // 97.9 us at 1, 98.4 at 3).
  static constexpr int kStartWeight = kQBufs == 1 ? 3 : 1;
  static constexpr int kPHalf = N * 256;
  static constexpr int kPBytes = 2 * kPHalf;
  // as many 32 KB ring stages as the shared memory left over allows
  static constexpr int kFree =
      kSmemBudget - (int)sizeof(Tail<N>) - kQBufs * kQBytes - kPBufs * kPBytes;
  static constexpr int kStages = kFree / kStage > kMaxStages ? kMaxStages : kFree / kStage;
  // S and O^T, two slots each: 4N columns, allocated as a power of two
  static constexpr uint32_t kTmemCols = 4 * N <= 64 ? 64 : 4 * N <= 128 ? 128 : 4 * N <= 256 ? 256 : 512;
  static constexpr int kRingOff = 0;
  static constexpr int kQOff = kStages * kStage;
  static constexpr int kPOff = kQOff + kQBufs * kQBytes;
  static constexpr int kTailOff = kPOff + kPBufs * kPBytes;
};

template <int DT, int H, int G>
constexpr int smem_bytes() {
  return Geo<H, G>::kTailOff + (int)sizeof(Tail<Geo<H, G>::N>) + 1024;
}

// Head-group passes of one call (p.head_off > 0 or p.Hkv < p.Hkv_all) run as a
// chain: every pass but the last lets the next one launch once it has passed its
// own dependency wait (its CTAs take the SMs as this pass's CTAs leave), and
// every pass but the first reads only data that the first pass's wait already
// covers, so it defers its wait to its end, where it makes its own completion
// imply the previous pass's.
constexpr int kChainTrigger = 1;
constexpr int kChainLateWait = 2;

struct SkParams {
  DecodeParams p;
  int chain;                // kChainTrigger | kChainLateWait for head-group passes
  int* tile_prefix;         // [B + 1] tiles before sequence b (written by CTA 0 for the combine)
  int* weight_prefix;       // [B + 2] weight before sequence b, then the start weight (the same)
  float* part_m;            // [grid * 2][Hq_all]: each pass its own heads
  float* part_l;
  float* part_acc;          // [grid * 2][Hq_all][D]
};

__device__ __forceinline__ int clamp_len(const DecodeParams& p, int b) {
  const int L = p.seq_lens[b];
  return L < 0 ? 0 : (L > p.max_seq_len ? p.max_seq_len : L);
}

// Start of CTA c's share of W units over `grid` CTAs.
__device__ __forceinline__ int range_start(int c, int W, int grid) {
  return (int)((unsigned long long)c * (unsigned)W / (unsigned)grid);
}

// The CTA whose share [range_start(c), range_start(c + 1)) holds unit x.
__device__ __forceinline__ int range_owner(int x, int W, int grid) {
  return (int)(((unsigned long long)(x + 1) * (unsigned)grid - 1ull) / (unsigned)W);
}

// Decode-step cache write of sequence b, vectors first, first + stride, ...:
// the K/V rows of token L - 1 (all H heads, 16-byte vectors) go to its slot
// table[(L-1) / bs] * bs + (L-1) % bs ("10 — Paged Attention" tutorial, §4
// PhysicalIndex).  L <= 0 or past the table writes nothing (the length check
// reports it); a block id outside the pool is reported and skipped.
template <int H>
__device__ __forceinline__ void store_newest(const DecodeParams& p, int b, int first, int stride) {
  constexpr int kRowVecs = H * kD * 2 / 16;     // this launch's heads of a token
  const int64_t all_vecs = (int64_t)p.Hkv_all * kD * 2 / 16, off_vecs = (int64_t)p.head_off * kD * 2 / 16;
  const int L = p.seq_lens[b];
  if (L <= 0 || L > p.max_blocks * p.bs) return;
  const int pos = L - 1;
  const int32_t id = p.block_tables[(int64_t)b * p.max_blocks + pos / p.bs];
  if (id < 0 || id >= p.num_blocks) {
    if (first == 0) report(p.status_dev, PA_ERR_BAD_BLOCK_ID);
    return;
  }
  const int64_t dst = ((int64_t)id * p.bs + pos % p.bs) * all_vecs + off_vecs;
  const uint4* sk = static_cast<const uint4*>(p.new_k) + (int64_t)b * all_vecs + off_vecs;
  const uint4* sv = static_cast<const uint4*>(p.new_v) + (int64_t)b * all_vecs + off_vecs;
  uint4* dk = static_cast<uint4*>(const_cast<void*>(p.k_pool)) + dst;
  uint4* dv = static_cast<uint4*>(const_cast<void*>(p.v_pool)) + dst;
  for (int v = first; v < kRowVecs; v += stride) {
    dk[v] = sk[v];
    dv[v] = sv[v];
  }
}

template <int DT, int H, int G>
__global__ void __launch_bounds__(kThreads, 1)
decode_tcg_kernel(const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_q, const SkParams sp) {
  using Gm = Geo<H, G>;
  constexpr int N = Gm::N, TT = Gm::TT, S = Gm::kStages;
  static_assert(S >= 3, "ring too shallow");
  static_assert(Gm::kTailOff + (int)sizeof(Tail<N>) <= kSmemBudget, "shared memory layout");
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  Tail<N>* tl = reinterpret_cast<Tail<N>*>(smem + Gm::kTailOff);
  volatile int* abort_flag = &tl->abort_flag;
  const DecodeParams& p = sp.p;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x, grid = gridDim.x;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&tl->full[s], 1);
      mbar_init(&tl->empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tl->seg_full[i], 1);
      mbar_init(&tl->seg_empty[i], 5);
      mbar_init(&tl->q_full[i], 1);
      mbar_init(&tl->q_empty[i], 1);
      mbar_init(&tl->s_full[i], 1);
      mbar_init(&tl->s_empty[i], 4);
      mbar_init(&tl->p_full[i], 4);
      mbar_init(&tl->p_empty[i], 1);
      mbar_init(&tl->o_full[i], 1);
      mbar_init(&tl->o_empty[i], 4);
      mbar_init(&tl->red[i], 4);
      mbar_init(&tl->red2[i], 4);
    }
    mbar_init(&tl->lsum, 4);
    mbar_init(&tl->drain, 1);
    mbar_init(&tl->app_done, 128);
    mbar_init(&tl->staged, 4);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tl->p_staged[i], 4);
      mbar_init(&tl->p_released[i], 1);
    }
    tl->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_q);
  }
  if (warp == 1) {
    tmem_alloc(&tl->tmem_base, Gm::kTmemCols);
    tmem_relinquish();
  }
  if (warp >= 2) {
    // P' is block diagonal: entries outside a row's query group stay zero forever
    uint4* pz = reinterpret_cast<uint4*>(smem + Gm::kPOff);
    for (int i = threadIdx.x - 64; i < Gm::kPBufs * Gm::kPBytes / 16; i += 128) pz[i] = make_uint4(0, 0, 0, 0);
    fence_async_smem();
  }
  // No early launch of the dependent kernel (the combine): its CTAs, resident
  // and waiting while this grid streams, cost this grid 0.9 us on the
  // Llama-shaped batch and 2.8 us on the long-context one (GB300, back-to-back
  // steps); triggering when the producer has issued its last copy, or at the
  // CTA's last segment, measured in between.  The next pass of a head-group
  // chain is launched early: it cannot become resident before this pass's
  // CTAs leave (shared memory).
  if (!(sp.chain & kChainLateWait)) wait_prior_grid();   // inputs may come from the previous kernel
  if (sp.chain & kChainTrigger) allow_next_grid();
  if (warp >= 2) {
    // The split (every CTA computes it; CTA 0 also stores the prefixes for the
    // combine pass), zero rows of empty sequences, length checks.  Thread et
    // walks the sequences [b0, b1) three times: totals, then prefixes and the
    // CTA's cuts, then its window entries.
    const int et = threadIdx.x - 64, ew = et >> 5;
    const int per = (p.B + 127) / 128;
    const int b0 = min(p.B, et * per), b1 = min(p.B, b0 + per);
    int my_t = 0, my_n = 0;
    for (int b = b0; b < b1; ++b) {
      const int nt = (clamp_len(p, b) + TT - 1) / TT;
      my_t += nt;
      my_n += nt > 0;
    }
    int inc_t = my_t, inc_n = my_n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int vt = __shfl_up_sync(0xFFFFFFFFu, inc_t, o);
      const int vn = __shfl_up_sync(0xFFFFFFFFu, inc_n, o);
      if (lane >= o) {
        inc_t += vt;
        inc_n += vn;
      }
    }
    if (lane == 31) {
      tl->scan[0][ew] = inc_t;
      tl->scan[1][ew] = inc_n;
    }
    named_barrier(1, 128);
    int run_t = inc_t - my_t, run_n = inc_n - my_n, T = 0, NE = 0;
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      if (w < ew) {
        run_t += tl->scan[0][w];
        run_n += tl->scan[1][w];
      }
      T += tl->scan[0][w];
      NE += tl->scan[1][w];
    }
    // start weight: the least >= Gm::kStartWeight with (T + sw NE) / grid + 1 <=
    // (kWin - 2)(sw + 1), so that no range meets more than kWin sequences (the
    // host keeps NE <= (kWin - 2) grid / 2, so den > 0)
    int sw = Gm::kStartWeight;
    {
      const long long num = (long long)T + grid - (long long)(kWin - 2) * grid;
      const long long den = (long long)(kWin - 2) * grid - NE;
      if (num > 0) sw = max(sw, (int)((num + den - 1) / den));
    }
    const int W = T + sw * NE;
    const int x0 = range_start(c, W, grid), x1 = range_start(c + 1, W, grid);
    const int first_t = run_t, first_n = run_n;
    for (int b = b0; b < b1; ++b) {
      const int raw = p.seq_lens[b];
      const int L = clamp_len(p, b);
      const int nt = (L + TT - 1) / TT;
      const int run_w = run_t + sw * run_n;
      if (c == 0) {
        sp.tile_prefix[b] = run_t;
        sp.weight_prefix[b] = run_w;
        if (raw < 0 || raw > p.max_seq_len) report(p.status_dev, PA_ERR_BAD_BLOCK_ID);
      }
      if (L == 0 && b % grid == c) {
        uint16_t* o = static_cast<uint16_t*>(p.out) + ((int64_t)b * p.Hq_all + p.head_off * G) * kD;
        for (int e = 0; e < p.Hq * kD; ++e) o[e] = 0;
        if (p.new_k != nullptr) store_newest<H>(p, b, 0, 1);   // no tile reads it
      }
      if (nt > 0) {
        // weighted span [run_w, run_w + sw + nt): the start, then the
        // tiles; a cut in it falls before tile clamp(x - run_w - start, 0, nt)
        const int span_end = run_w + sw + nt;
        if (run_w <= x0 && x0 < span_end) {
          const int tb = run_t + min(max(x0 - run_w - sw, 0), nt);
          tl->cut[0] = tb;
          // the window starts at the sequence holding tile tb (tb < run_t + nt
          // here); its first block ids go to L2 now, so that the producer's
          // first load of them does not wait for DRAM
          tl->win_n[0] = run_n;
          const int kf = (tb - run_t) * TT / p.bs;
          const int32_t* ids = p.block_tables + (int64_t)b * p.max_blocks + kf;
          prefetch_l2(ids);
          if (kf + 32 < p.max_blocks) prefetch_l2(ids + 32);
        }
        if (run_w <= x1 && x1 < span_end) {
          const int te = run_t + min(max(x1 - run_w - sw, 0), nt);
          tl->cut[1] = te;
          tl->win_n[1] = te > run_t ? run_n + 1 : run_n;   // sequences before the end cut
        }
      }
      run_t += nt;
      run_n += nt > 0;
    }
    if (et == 127) {
      if (c == 0) {
        sp.tile_prefix[p.B] = run_t;
        sp.weight_prefix[p.B] = run_t + sw * run_n;
        sp.weight_prefix[p.B + 1] = sw;
      }
      if (x0 >= W) {              // cuts at the batch's end (or an empty batch)
        tl->cut[0] = T;
        tl->win_n[0] = NE;
      }
      if (x1 >= W) {
        tl->cut[1] = T;
        tl->win_n[1] = NE;
      }
    }
    named_barrier(1, 128);
    const int wn0 = tl->win_n[0], wn1 = tl->cut[0] < tl->cut[1] ? tl->win_n[1] : wn0;
    run_t = first_t;
    run_n = first_n;
    for (int b = b0; b < b1; ++b) {
      const int nt = (clamp_len(p, b) + TT - 1) / TT;
      if (nt > 0 && run_n >= wn0 && run_n < wn1) {
        const int k = run_n - wn0;          // < kWin: the host bounds B by kWin * grid
        if (k < kWin) {
          tl->win_b[k] = b;
          tl->win_len[k] = clamp_len(p, b);
          tl->win_tp[k] = run_t;
          if (run_n == wn1 - 1) tl->win_tp[k + 1] = run_t + nt;
        }
      }
      run_t += nt;
      run_n += nt > 0;
    }
    if (et == 0) tl->nwin = min(wn1 - wn0, kWin);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int t_begin = tl->cut[0], t_end = tl->nwin > 0 ? tl->cut[1] : tl->cut[0];
  const int nwin = tl->nwin;
  if (warp >= 2) {
    // Decode-step cache write: the newest token of a sequence lies in its last
    // tile, and tiles cover disjoint token ranges, so the CTA whose range holds
    // that tile stores the token.  The writes are fenced against the async
    // proxy; the producer waits for app_done before it loads such a tile.
    if (p.new_k != nullptr) {
      for (int k = 0; k < nwin && tl->win_tp[k + 1] <= t_end; ++k)
        store_newest<H>(p, tl->win_b[k], threadIdx.x - 64, 128);
    }
    fence_async_global();
    mbar_arrive(&tl->app_done);
  }
  // Ring order follows the MMA's consumption order: K(0), then for t >= 1 K(t)
  // before V(t-1), and V(last) at the end.  Positions in that sequence:
  const int t_last = t_end - t_begin - 1;
  auto pos_k = [](int t) { return t == 0 ? 0 : 2 * t - 1; };
  auto pos_v = [t_last](int t) { return t < t_last ? 2 * t + 2 : 2 * t + 1; };
  const uint32_t tmem = tl->tmem_base;
  const uint32_t ring_addr = smem_addr(smem + Gm::kRingOff);
  const uint32_t q_addr = smem_addr(smem + Gm::kQOff);
  const uint32_t p_addr = smem_addr(smem + Gm::kPOff);

  auto set_abort = [&]() {
    tl->abort_flag = 1;
    report(p.status_dev, PA_ERR_TIMEOUT);
  };

  if (warp == 0) {
    // -------------------------------------------------------------- producer --
    const uint64_t policy = policy_evict_first();
    int stage = 0, sphase = 0;
    int issued[kMaxStages] = {-1, -1, -1, -1, -1, -1};
    int q_issued[2] = {-1, -1};
    int seg_idx = 0;
    bool ok = true;
    bool appended = p.new_k == nullptr;   // newest tokens already in the pool
    int tile = t_begin;
    // V tile of the previous K tile, issued after the next K tile
    bool pend = false;
    int pend_nbox = 0, pend_box = 0, pend_tok = 0;
    int32_t pend_blk = 0;
    // One tile: lanes < nbox each copy one box of box_tokens tokens x H heads,
    // lane i at (token-in-block tok, block blk) of the [blocks][bs][H][D] pool;
    // the boxes fill the stage (nbox * box_tokens = TT tokens).
    auto issue = [&](const CUtensorMap* map, int nbox, int box_tokens, int tok,
                     int32_t blk) -> bool {
      const uint32_t bytes = (uint32_t)nbox * box_tokens * H * 128u * 2u;
      bool good = true;
      if (lane == 0) {
        good = mbar_wait(&tl->empty[stage], sphase ^ 1, abort_flag, kWaitNs);
        if (good) mbar_arrive_expect_tx(&tl->full[stage], bytes);
        else set_abort();
      }
      good = __shfl_sync(0xFFFFFFFFu, (int)good, 0) != 0;
      if (!good) return false;
      if (lane < nbox) {
        uint8_t* dst = smem + Gm::kRingOff + stage * kStage + lane * box_tokens * H * 128;
        tma_load_4d_hint(dst, map, &tl->full[stage], 0, 0, tok, blk, policy);
        tma_load_4d_hint(dst + kSlab, map, &tl->full[stage], 64, 0, tok, blk, policy);
      }
      issued[stage] = sphase;
      if (++stage == S) {
        stage = 0;
        sphase ^= 1;
      }
      return true;
    };
    // Block ids of a segment, 32 per chunk held one per lane (ids past the
    // sequence's blocks are loaded but never used).  A segment's length and first
    // two chunks are loaded while the previous segment streams: waiting for those
    // dependent loads at the segment start left the ring without new copies for
    // their latency (measured on GB300: ~4 us per segment boundary).
    auto raw_ids = [&](int bb, int base) -> int32_t {
      const int k = base + lane;
      return k < p.max_blocks ? p.block_tables[(int64_t)bb * p.max_blocks + k] : 0;
    };
    int pf_b = -1;
    int32_t pf_cur = 0, pf_nxt = 0;
    // With two Q buffers the next segment's Q is copied as soon as its buffer is
    // free (polled once per tile, never waited on), instead of at the segment's
    // start, one ring-depth before the MMA needs it: the copy's latency there
    // (~4 us under load on GB300) held up the first S of every segment.
    int next_b = -1;                   // sequence of the next segment, -1: none
    bool q_early = false;              // the next segment's Q is already on its way
    int wk = 0;                        // window entry of the next segment
    int tpb = 0, tpb1 = 0;             // batch tiles of the segment's sequence
    while (ok) {
      SegInfo sg;
      sg.valid = 0;
      if (tile < t_end) {
        tpb = tl->win_tp[wk];
        tpb1 = tl->win_tp[wk + 1];
        sg.b = tl->win_b[wk];
        if (pf_b != sg.b) {              // first segment: nothing prefetched
          pf_b = sg.b;
          const int kf = ((tile - tpb) * TT) / p.bs;
          pf_cur = raw_ids(sg.b, kf);
          pf_nxt = raw_ids(sg.b, kf + 32);
        }
        sg.L = tl->win_len[wk];
        sg.j0 = tile - tpb;
        sg.j1 = min(t_end, tpb1) - tpb;
        sg.direct = (sg.j0 == 0 && sg.j1 == tpb1 - tpb);
        sg.slot = seg_idx == 0 ? 0 : 1;
        sg.valid = 1;
        sg.last = tpb1 >= t_end;
      }
      if (!sg.valid && pend) {           // the last V tile of this CTA
        ok = issue(&tm_v, pend_nbox, pend_box, pend_tok, pend_blk);
        pend = false;
        if (!ok) break;
      }
      const int islot = seg_idx & 1;
      if (lane == 0) {
        ok = mbar_wait(&tl->seg_empty[islot], ((seg_idx >> 1) & 1) ^ 1, abort_flag, kWaitNs);
        if (ok) {
          tl->seg[islot] = sg;
          mbar_arrive(&tl->seg_full[islot]);
        } else {
          set_abort();
        }
      }
      ok = __shfl_sync(0xFFFFFFFFu, (int)ok, 0) != 0;
      if (!ok || !sg.valid) break;
      // all query heads of the sequence (N rows; rows past Hq are never used)
      const int qb = seg_idx % Gm::kQBufs, qph = (seg_idx / Gm::kQBufs) & 1;
      if (q_early) {
        q_early = false;
      } else if (lane == 0) {
        ok = mbar_wait(&tl->q_empty[qb], qph ^ 1, abort_flag, kWaitNs);
        if (ok) {
          mbar_arrive_expect_tx(&tl->q_full[qb], Gm::kQBytes);
          tma_load_2d(smem + Gm::kQOff + qb * Gm::kQBytes, &tm_q, &tl->q_full[qb], 0,
                      sg.b * p.Hq_all + p.head_off * G);
          tma_load_2d(smem + Gm::kQOff + qb * Gm::kQBytes + N * 128, &tm_q, &tl->q_full[qb], 64,
                      sg.b * p.Hq_all + p.head_off * G);
          q_issued[qb] = qph;
        } else {
          set_abort();
        }
      }
      ok = __shfl_sync(0xFFFFFFFFu, (int)ok, 0) != 0;
      if (!ok) break;
      const int nblk_seq = (sg.L + p.bs - 1) / p.bs;
      int kb = (sg.j0 * TT) / p.bs;
      int32_t cur = pf_cur, nxt = pf_nxt;
      const int seq_tiles = tpb1 - tpb;
      next_b = -1;
      if (tpb + sg.j1 < t_end) {       // the next segment: the next window entry
        const int nb = tl->win_b[wk + 1];
        next_b = nb;
        pf_b = nb;
        pf_cur = raw_ids(nb, 0);
        pf_nxt = raw_ids(nb, 32);
      }
      for (int j = sg.j0; j < sg.j1 && ok; ++j) {
        // boxes of the tile: TT / bs whole blocks, or one TT-token piece of a block
        const int tok0 = j * TT;
        const int box_tokens = TT >= p.bs ? p.bs : TT;
        const int nbox = TT / box_tokens;
        const int k0 = tok0 / p.bs;
        const int tok_off = TT >= p.bs ? 0 : tok0 % p.bs;
        // The box holding the sequence's last token is shifted back by sh rows so
        // that it ends at that token: its first sh rows read a negative in-block
        // coordinate (zeros) or the sequence's earlier tokens.  Boxes after it
        // read block -1 (zeros).  Every row is finite and the softmax masks the
        // rows that are not this tile's tokens, so no copy has to be waited for
        // to clean rows.
        const int n_valid = sg.L - tok0;
        const int il = n_valid >= TT ? nbox : (n_valid - 1) / box_tokens;
        const int sh = n_valid >= TT ? 0 : box_tokens - (n_valid - il * box_tokens);
        while (k0 - kb >= 32) {          // advance the id window
          kb += 32;
          cur = nxt;
          nxt = raw_ids(sg.b, kb + 32);
        }
        const int src = min(k0 + lane, nblk_seq - 1) - kb;     // < 64: nbox <= 16
        const int32_t a = __shfl_sync(0xFFFFFFFFu, cur, src & 31);
        const int32_t bb = __shfl_sync(0xFFFFFFFFu, nxt, src & 31);
        int32_t blk = src < 32 ? a : bb;
        int tok = tok_off;
        if (lane > il) {
          blk = -1;
        } else {
          if (lane == il) tok = tok_off - sh;
          if (blk < 0 || blk >= p.num_blocks) {   // outside the pool: the copy reads zeros
            if (lane < nbox) report(p.status_dev, PA_ERR_BAD_BLOCK_ID);
            blk = p.num_blocks;
          }
        }
        if (!appended && j == seq_tiles - 1) {   // holds the newest token: wait for its write
          bool good = mbar_wait(&tl->app_done, 0, abort_flag, kWaitNs);
          good = __all_sync(0xFFFFFFFFu, good);
          if (!good) {
            if (lane == 0) set_abort();
            ok = false;
            break;
          }
          appended = true;
        }
        ok = issue(&tm_k, nbox, box_tokens, tok, blk);
        if (ok && pend) ok = issue(&tm_v, pend_nbox, pend_box, pend_tok, pend_blk);
        if (Gm::kQBufs == 2 && next_b >= 0 && !q_early) {
          const int nqb = (seg_idx + 1) % Gm::kQBufs, nqph = ((seg_idx + 1) / Gm::kQBufs) & 1;
          int go = 0;
          if (lane == 0 && mbar_try_wait(&tl->q_empty[nqb], nqph ^ 1)) {
            mbar_arrive_expect_tx(&tl->q_full[nqb], Gm::kQBytes);
            tma_load_2d(smem + Gm::kQOff + nqb * Gm::kQBytes, &tm_q, &tl->q_full[nqb], 0,
                        next_b * p.Hq_all + p.head_off * G);
            tma_load_2d(smem + Gm::kQOff + nqb * Gm::kQBytes + N * 128, &tm_q, &tl->q_full[nqb],
                        64, next_b * p.Hq_all + p.head_off * G);
            q_issued[nqb] = nqph;
            go = 1;
          }
          q_early = __shfl_sync(0xFFFFFFFFu, go, 0) != 0;
        }
        pend = true;
        pend_nbox = nbox;
        pend_box = box_tokens;
        pend_tok = tok;
        pend_blk = blk;
      }
      if (!ok) break;
      tile = tpb + sg.j1;
      ++wk;
      ++seg_idx;
      __syncwarp();
    }
    if (*abort_flag && lane == 0) {
      for (int s = 0; s < S; ++s)
        if (issued[s] >= 0) mbar_wait_drain(&tl->full[s], issued[s], kWaitNs);
      for (int i = 0; i < 2; ++i)
        if (q_issued[i] >= 0) mbar_wait_drain(&tl->q_full[i], q_issued[i], kWaitNs);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue --
    constexpr uint32_t ab = DT == PA_BFLOAT16 ? 1u : 0u;
    constexpr uint32_t idesc_s = idesc_f16(ab, 0, 0, kRows, N);
    constexpr uint32_t idesc_o = idesc_f16(ab, 1, 0, kD, N);
    int tile_g = 0, seg_idx = 0;
    bool ok = true, committed = false;
    auto issue_pv = [&](int t, int vs, int vph) -> bool {
      const int slot = t & 1, ph = (t >> 1) & 1;
      if (!mbar_wait(&tl->full[vs], vph, abort_flag, kWaitNs)) return false;
      const int ps = t % Gm::kPBufs, pph = (t / Gm::kPBufs) & 1;
      if (!mbar_wait(&tl->p_full[ps], pph, abort_flag, kWaitNs)) return false;
      if (!mbar_wait(&tl->o_empty[slot], ph ^ 1, abort_flag, kWaitNs)) return false;
      tc_fence_after();
      // descriptors built once and stepped by compile-time offsets (address / 16):
      // one thread issues every MMA
      const uint64_t vdesc = smem_desc_sw128(ring_addr + vs * kStage, kSlab, 1024);
      const uint64_t pdesc = smem_desc_sw128(p_addr + ps * Gm::kPBytes, 16, 1024);
      const uint32_t d = tmem + 2 * N + slot * N;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
#pragma unroll
        for (int kk = 0; kk < kRows / 16; ++kk) {
          const uint64_t a = vdesc + (uint64_t)((kk * 16 * 128) >> 4);
          const uint64_t bd =
              pdesc + (uint64_t)((half * Gm::kPHalf + (kk >> 2) * (N * 128) + (kk & 3) * 32) >> 4);
          mma_f16(d, a, bd, idesc_o, (half | kk) != 0);
        }
      }
      mma_commit(&tl->empty[vs]);
      mma_commit(&tl->o_full[slot]);
      mma_commit(&tl->p_empty[ps]);
      return true;
    };
    for (;;) {
      const int islot = seg_idx & 1;
      int valid = 0, ntiles = 0;
      if (lane == 0) {
        ok = mbar_wait(&tl->seg_full[islot], (seg_idx >> 1) & 1, abort_flag, kWaitNs);
        if (ok) {
          valid = tl->seg[islot].valid;
          ntiles = tl->seg[islot].j1 - tl->seg[islot].j0;
          mbar_arrive(&tl->seg_empty[islot]);
        }
      }
      ok = __shfl_sync(0xFFFFFFFFu, (int)ok, 0) != 0;
      valid = __shfl_sync(0xFFFFFFFFu, valid, 0);
      ntiles = __shfl_sync(0xFFFFFFFFu, ntiles, 0);
      if (!ok) {
        if (lane == 0) set_abort();
        break;
      }
      if (!valid) break;
      const int qb = seg_idx % Gm::kQBufs;
      if (lane == 0) {
        ok = mbar_wait(&tl->q_full[qb], (seg_idx / Gm::kQBufs) & 1, abort_flag, kWaitNs);
        int pvs = 0, pvph = 0;
        for (int j = 0; j < ntiles && ok; ++j) {
          const int t = tile_g + j;
          const int slot = t & 1, ph = (t >> 1) & 1;
          const int ks = pos_k(t) % S, kph = (pos_k(t) / S) & 1;
          const int vs = pos_v(t) % S, vph = (pos_v(t) / S) & 1;
          ok = mbar_wait(&tl->full[ks], kph, abort_flag, kWaitNs) &&
               mbar_wait(&tl->s_empty[slot], ph ^ 1, abort_flag, kWaitNs);
          if (!ok) break;
          tc_fence_after();
          const uint64_t kdesc = smem_desc_sw128(ring_addr + ks * kStage, 16, 1024);
          const uint64_t qdesc = smem_desc_sw128(q_addr + qb * Gm::kQBytes, 16, 1024);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kSlab + (kk & 3) * 32;
            const uint32_t qoff = (kk >> 2) * (N * 128) + (kk & 3) * 32;
            mma_f16(tmem + slot * N, kdesc + (uint64_t)(off >> 4), qdesc + (uint64_t)(qoff >> 4),
                    idesc_s, kk > 0);
          }
          mma_commit(&tl->empty[ks]);
          mma_commit(&tl->s_full[slot]);
          if (j == ntiles - 1) mma_commit(&tl->q_empty[qb]);
          committed = true;
          if (j > 0) ok = issue_pv(t - 1, pvs, pvph);
          pvs = vs;
          pvph = vph;
        }
        if (ok) ok = issue_pv(tile_g + ntiles - 1, pvs, pvph);
        if (!ok) set_abort();
      }
      ok = __shfl_sync(0xFFFFFFFFu, (int)ok, 0) != 0;
      if (!ok) break;
      tile_g += ntiles;
      ++seg_idx;
    }
    if (*abort_flag && lane == 0 && committed) {
      mma_commit(&tl->drain);
      mbar_wait_drain(&tl->drain, 0, kWaitNs);
    }
  } else {
    // ------------------------------------------------- softmax / epilogue --
    const int wq = warp & 3;
    const int r = wq * 32 + lane;            // tile row (token r / H, head r % H); O row d
    const int tt = r / H, h = lane % H;      // H divides 32
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    int tile_g = 0, seg_idx = 0, round = 0, lround = 0, rround = 0;
    bool raised[2] = {true, true};         // per round parity: the tile moved its maxima
    bool ok = true;
    auto wait_all = [&](uint64_t* bar, int parity) -> bool {
      const bool w = mbar_wait(bar, parity, abort_flag, kWaitNs);
      return __all_sync(0xFFFFFFFFu, w);
    };
    // A segment's outputs leave through the TMA unit.  Global stores issued by
    // these warps while the TMA copies keep the memory system saturated stall
    // each warp ~190 cycles per store on GB300 (~3 us per segment, in a burst
    // or spread over the following tiles alike).  So the outputs are written to
    // shared memory and sent with one bulk copy: the CTA's final segment stages
    // them in the idle ring; another segment (N <= 32, two P' buffers) in the
    // P' buffer of its last tile, which its P'.V has finished reading and which
    // the next tile does not use.  Before that buffer takes a P' again, the bulk
    // copy must have read it and each thread re-zeroes its row (P' relies on
    // zeros off the block diagonal).  For N = 64 (one P' buffer; few segments
    // per CTA in its batches) other segments store directly.
    constexpr bool kStageP = Gm::kPBufs == 2;
    int stg_pend = 0;                  // bit i: P' buffer i holds staged outputs
    int stg_phase = 0;                 // bit i: parity of P' buffer i's next staging
    auto release_p = [&](int ps) -> bool {
      if (!(stg_pend >> ps & 1)) return true;
      if (threadIdx.x == 64) {
        asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
        mbar_arrive(&tl->p_released[ps]);
      }
      if (!wait_all(&tl->p_released[ps], stg_phase >> ps & 1)) return false;
      uint8_t* pb = smem + Gm::kPOff + ps * Gm::kPBytes + (r >> 6) * (N * 128);
      const int chunk = (r & 63) >> 3;
#pragma unroll
      for (int q = 0; q < N; ++q) {
        const int off = q * 128 + ((chunk ^ (q & 7)) << 4) + (r & 7) * 2;
        *reinterpret_cast<uint16_t*>(pb + off) = 0;
        *reinterpret_cast<uint16_t*>(pb + Gm::kPHalf + off) = 0;
      }
      stg_pend &= ~(1 << ps);
      stg_phase ^= 1 << ps;
      return true;
    };
    for (;;) {
      const int islot = seg_idx & 1;
      if (!wait_all(&tl->seg_full[islot], (seg_idx >> 1) & 1)) { ok = false; break; }
      const SegInfo sg = tl->seg[islot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&tl->seg_empty[islot]);
      if (!sg.valid) break;
      const int ntiles = sg.j1 - sg.j0;
      float m_run[G], l_t[G], acc[N];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        m_run[g] = -CUDART_INF_F;
        l_t[g] = 0.f;
      }
#pragma unroll
      for (int q = 0; q < N; ++q) acc[q] = 0.f;
      // acc <- acc * alpha(t) + O_t, alpha(t) from round `rnd` (all query heads)
      auto accumulate = [&](int t, int rnd) -> bool {
        const int slot = t & 1, ph = (t >> 1) & 1;
        if (!wait_all(&tl->o_full[slot], ph)) return false;
        tc_fence_after();
        if (raised[rnd & 1]) {
          const float* al = tl->alpha[rnd & 1];
#pragma unroll
          for (int c0 = 0; c0 < N; c0 += 16) {
            float o[16];
            tmem_ld16(tmem + lane_base + 2 * N + slot * N + c0, o);
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[c0 + i] = fmaf(acc[c0 + i], al[c0 + i], o[i]);
          }
        } else {                 // the round kept every running max: alpha = 1
#pragma unroll
          for (int c0 = 0; c0 < N; c0 += 16) {
            float o[16];
            tmem_ld16(tmem + lane_base + 2 * N + slot * N + c0, o);
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[c0 + i] += o[i];
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tl->o_empty[slot]);
        return true;
      };
      for (int j = 0; j < ntiles && ok; ++j) {
        const int t = tile_g + j;
        const int slot = t & 1, ph = (t >> 1) & 1;
        if (!wait_all(&tl->s_full[slot], ph)) { ok = false; break; }
        tc_fence_after();
        float x[G];
        {
          float s[N];
#pragma unroll
          for (int c0 = 0; c0 < N; c0 += 16) {
            float v[16];
            tmem_ld16(tmem + lane_base + slot * N + c0, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) s[c0 + i] = v[i];
          }
#pragma unroll
          for (int hh = 0; hh < H; ++hh)
            if (h == hh) {
#pragma unroll
              for (int g = 0; g < G; ++g) x[g] = s[hh * G + g];
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tl->s_empty[slot]);
        // rows of this tile's tokens: all rows of an interior tile; in a
        // sequence's last tile the boxes before the last one and the last box's
        // rows from its shift on (the producer's layout of that tile)
        bool valid = true;
        {
          const int n_valid = sg.L - (sg.j0 + j) * TT;
          if (n_valid < TT) {
            const int bx = TT >= p.bs ? p.bs : TT;
            const int il = (n_valid - 1) / bx;
            const int sh = bx - (n_valid - il * bx);
            const int ib = tt / bx;
            valid = ib < il || (ib == il && tt - ib * bx >= sh);
          }
        }
        bool exceed = false;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          x[g] = valid ? x[g] * p.scale_log2 : -CUDART_INF_F;
          exceed |= x[g] > m_run[g] + kRescaleLog2;
        }
        // Running maxima rise only where a score exceeds them by more than 2^8
        // (always on a segment's first tile, where they are -inf): the four
        // warps vote, and only then is the tile's max per query head reduced
        // and every running max moved to it.  Otherwise p = 2^(s - m) may
        // reach 2^8, which fp32 sums and the hi + lo terms of P' carry, and the
        // accumulators need no rescale; the final division by the sum removes
        // the choice of max.
        const int rb = round & 1;
        {
          const bool wv = __any_sync(0xFFFFFFFFu, exceed);
          if (lane == 0) {
            tl->vote[rb][wq] = wv ? 1 : 0;
            mbar_arrive(&tl->red[rb]);
          }
        }
        if (!wait_all(&tl->red[rb], (round >> 1) & 1)) { ok = false; break; }
        const int4 vt = *reinterpret_cast<const int4*>(tl->vote[rb]);
        const bool raise = (vt.x | vt.y | vt.z | vt.w) != 0;
        raised[rb] = raise;
        float pr[G];
        if (raise) {
          float wm[G];
#pragma unroll
          for (int g = 0; g < G; ++g) wm[g] = x[g];
          // rows of the same KV head in this warp: lanes h, h+H, ... (xor H .. 16)
#pragma unroll
          for (int off = H; off < 32; off <<= 1)
#pragma unroll
            for (int g = 0; g < G; ++g) wm[g] = fmaxf(wm[g], __shfl_xor_sync(0xFFFFFFFFu, wm[g], off));
          const int rr = rround & 1;
          if (lane < H)
#pragma unroll
            for (int g = 0; g < G; ++g) tl->red_buf[rr][wq][h * G + g] = wm[g];
          __syncwarp();
          if (lane == 0) mbar_arrive(&tl->red2[rr]);
          if (!wait_all(&tl->red2[rr], (rround >> 1) & 1)) { ok = false; break; }
          ++rround;
          float alpha[G];
#pragma unroll
          for (int g = 0; g < G; ++g) {
            const int q = h * G + g;
            const float tm = fmaxf(fmaxf(tl->red_buf[rr][0][q], tl->red_buf[rr][1][q]),
                                   fmaxf(tl->red_buf[rr][2][q], tl->red_buf[rr][3][q]));
            const float m_new = fmaxf(m_run[g], tm);
            alpha[g] = exp2f(m_run[g] - m_new);
            pr[g] = valid ? exp2f(x[g] - m_new) : 0.f;
            l_t[g] = fmaf(l_t[g], alpha[g], pr[g]);
            m_run[g] = m_new;
          }
          if (wq == 0 && lane < H) {
#pragma unroll
            for (int g = 0; g < G; ++g) tl->alpha[rb][h * G + g] = alpha[g];
          }
        } else {
#pragma unroll
          for (int g = 0; g < G; ++g) {
            pr[g] = valid ? exp2f(x[g] - m_run[g]) : 0.f;
            l_t[g] += pr[g];
          }
        }
        // P' entries of this row: (head h*G+g, column r)
        const int ps = t % Gm::kPBufs, pph = (t / Gm::kPBufs) & 1;
        if (!wait_all(&tl->p_empty[ps], pph ^ 1)) { ok = false; break; }
        if (kStageP && !release_p(ps)) { ok = false; break; }
        uint8_t* pbuf = smem + Gm::kPOff + ps * Gm::kPBytes + (r >> 6) * (N * 128);
        const int chunk = (r & 63) >> 3;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const int q = h * G + g;
          const uint16_t hi = narrow<DT>(pr[g]);
          const uint16_t lo = narrow<DT>(pr[g] - widen2<DT>(hi).x);
          const int off = q * 128 + ((chunk ^ (q & 7)) << 4) + (r & 7) * 2;
          *reinterpret_cast<uint16_t*>(pbuf + off) = hi;
          *reinterpret_cast<uint16_t*>(pbuf + Gm::kPHalf + off) = lo;
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tl->p_full[ps]);
        if (j > 0 && !accumulate(t - 1, round - 1)) { ok = false; break; }
        ++round;
      }
      if (!ok) break;
      // denominators (and final maxima) of the segment, per query head
      {
        float ls[G];
#pragma unroll
        for (int g = 0; g < G; ++g) ls[g] = l_t[g];
#pragma unroll
        for (int off = H; off < 32; off <<= 1)
#pragma unroll
          for (int g = 0; g < G; ++g) ls[g] += __shfl_xor_sync(0xFFFFFFFFu, ls[g], off);
        if (lane < H)
#pragma unroll
          for (int g = 0; g < G; ++g) tl->lred[wq][h * G + g] = ls[g];
        if (wq == 0 && lane < H)
#pragma unroll
          for (int g = 0; g < G; ++g) tl->m_fin[h * G + g] = m_run[g];
        __syncwarp();
        if (lane == 0) mbar_arrive(&tl->lsum);
        if (!wait_all(&tl->lsum, lround & 1)) { ok = false; break; }
        ++lround;
      }
      if (!accumulate(tile_g + ntiles - 1, round - 1)) { ok = false; break; }
      const int Hq = p.Hq;
      // direct: normalised output; partial: the unnormalised accumulator, with
      // its (max, sum) per query head stored by the lanes of one warp.  The
      // division is the fast one (at most 2 ulp in fp32 for l in [1, 2^31], far
      // below the output's storage rounding): the IEEE one, with its slow-path
      // branch per element, cost ~2.3 us per segment on GB300.
      // The sums are read as vectors with no per-head branch, so that the loads
      // overlap (heads >= Hq divide by unwritten sums and are never stored); for
      // N = 64 the registers are not there (and its batches' segments are nearly
      // all partial).
      if (N <= 32 && sg.direct) {
#pragma unroll
        for (int q = 0; q < N; q += 4) {
          const float4 a = *reinterpret_cast<const float4*>(&tl->lred[0][q]);
          const float4 b = *reinterpret_cast<const float4*>(&tl->lred[1][q]);
          const float4 e = *reinterpret_cast<const float4*>(&tl->lred[2][q]);
          const float4 f = *reinterpret_cast<const float4*>(&tl->lred[3][q]);
          acc[q] = __fdividef(acc[q], a.x + b.x + e.x + f.x);
          acc[q + 1] = __fdividef(acc[q + 1], a.y + b.y + e.y + f.y);
          acc[q + 2] = __fdividef(acc[q + 2], a.z + b.z + e.z + f.z);
          acc[q + 3] = __fdividef(acc[q + 3], a.w + b.w + e.w + f.w);
        }
      } else if (sg.direct) {
#pragma unroll
        for (int q = 0; q < N; ++q) {
          if (q < Hq) {
            const float l = tl->lred[0][q] + tl->lred[1][q] + tl->lred[2][q] + tl->lred[3][q];
            acc[q] = __fdividef(acc[q], l);
          }
        }
      }
      // partial index of this pass's head 0 (partials of all heads side by side)
      const int64_t part0 = ((int64_t)c * 2 + sg.slot) * p.Hq_all + (int64_t)p.head_off * G;
      if (!sg.direct && wq == 0) {
        for (int q = lane; q < Hq; q += 32) {
          sp.part_m[part0 + q] = tl->m_fin[q];
          sp.part_l[part0 + q] = tl->lred[0][q] + tl->lred[1][q] + tl->lred[2][q] + tl->lred[3][q];
        }
      }
      const int64_t out0 =
          sg.direct ? ((int64_t)sg.b * p.Hq_all + p.head_off * G) * kD : part0 * kD;
      const int last_ps = (tile_g + ntiles - 1) % Gm::kPBufs;
      if (sg.last || kStageP) {
        // final segment: every MMA has completed and every copy has landed, the
        // ring is idle; otherwise the P' buffer of the segment's last tile
        uint8_t* stg = sg.last ? smem + Gm::kRingOff : smem + Gm::kPOff + last_ps * Gm::kPBytes;
        uint64_t* bar = sg.last ? &tl->staged : &tl->p_staged[last_ps];
        const int par = sg.last ? 0 : (stg_phase >> last_ps & 1);
#pragma unroll
        for (int q = 0; q < N; ++q) {
          if (q < Hq) {
            if (sg.direct) reinterpret_cast<uint16_t*>(stg)[q * kD + r] = narrow<DT>(acc[q]);
            else reinterpret_cast<float*>(stg)[q * kD + r] = acc[q];
          }
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar);
        if (threadIdx.x == 64) {
          if (mbar_wait(bar, par, abort_flag, kWaitNs)) {
            void* dst = sg.direct ? static_cast<void*>(static_cast<uint16_t*>(p.out) + out0)
                                  : static_cast<void*>(sp.part_acc + out0);
            const uint32_t bytes = (uint32_t)Hq * kD * (sg.direct ? 2u : 4u);
            if (sg.last) {
              bulk_store_and_release(dst, stg, bytes);
            } else {
              asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst),
                           "r"(smem_addr(stg)), "r"(bytes)
                           : "memory");
              asm volatile("cp.async.bulk.commit_group;" ::: "memory");
            }
          } else {
            ok = false;
          }
        }
        if (!sg.last) stg_pend |= 1 << last_ps;
        ok = __all_sync(0xFFFFFFFFu, ok);    // one lane's failed wait ends the warp's loop
        if (!ok) break;
      } else {
#pragma unroll
        for (int q = 0; q < N; ++q) {
          if (q < Hq) {
            if (sg.direct) static_cast<uint16_t*>(p.out)[out0 + (int64_t)q * kD + r] = narrow<DT>(acc[q]);
            else sp.part_acc[out0 + (int64_t)q * kD + r] = acc[q];
          }
        }
      }
      tile_g += ntiles;
      ++seg_idx;
    }
    if (threadIdx.x == 64) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
    if (!ok) set_abort();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Gm::kTmemCols);
  }
  if (sp.chain & kChainLateWait) wait_prior_grid();   // complete only after the previous pass
}

// Merge the partials of sequences cut by CTA range boundaries.  One warp per
// (sequence, query head).  Two rounds of loads: the sequence's prefixes, then,
// all at once, every part's (max, sum) (lane i: part i) and the first eight
// parts' accumulators (each lane its four columns); parts past the eighth are
// read afterwards, eight in flight.
// No early launch of the next kernel: letting the next decode's CTAs become
// resident while this grid runs measured 3% slower on the long-context batch
// on GB300 (and no faster on the others).
template <int DT>
__global__ void __launch_bounds__(128)
combine_sk_kernel(const SkParams sp, int grid) {
  const DecodeParams& p = sp.p;
  constexpr int PER = kD / 32;
  constexpr int kEarly = 8;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  wait_prior_grid();           // partials and the prefixes come from the main kernel
  const int64_t row = (int64_t)blockIdx.x * 4 + warp;
  if (row >= (int64_t)p.B * p.Hq) return;
  const int b = (int)(row / p.Hq), q = (int)(row - (int64_t)b * p.Hq);
  const int W = sp.weight_prefix[p.B], sw = sp.weight_prefix[p.B + 1];
  const int tpb = sp.tile_prefix[b], tpb1 = sp.tile_prefix[b + 1];
  const int pwb = sp.weight_prefix[b];
  if (tpb1 <= tpb) return;                                  // empty: zeroed by the main kernel
  // weighted position of the sequence's tile j: pwb + sw + j
  const int cf = range_owner(pwb + sw, W, grid);
  const int cl = range_owner(pwb + sw + (tpb1 - tpb) - 1, W, grid);
  if (cf == cl) return;                                     // written directly
  const int nparts = cl - cf + 1;
  // part i: CTA cf + i, slot 0 when the sequence is that CTA's first segment
  // (every CTA after cf; cf when its range starts at or after the sequence's
  // start), else 1; -1 for a CTA with an empty range
  auto part_index = [&](int i) -> int64_t {
    const int cc = cf + i;
    const int st = range_start(cc, W, grid);
    if (st == range_start(cc + 1, W, grid)) return -1;
    const int slot = (cc > cf || st >= pwb) ? 0 : 1;
    return ((int64_t)cc * 2 + slot) * p.Hq + q;
  };
  const int64_t idx0 = lane < nparts ? part_index(lane) : -1;
  float m0 = -CUDART_INF_F, l0 = 0.f;
  if (idx0 >= 0) {
    m0 = sp.part_m[idx0];
    l0 = sp.part_l[idx0];
  }
  float4 early[kEarly];
#pragma unroll
  for (int k = 0; k < kEarly; ++k) {
    const long long ik = __shfl_sync(0xFFFFFFFFu, (long long)idx0, k);
    early[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (k < nparts && ik >= 0)
      early[k] = *reinterpret_cast<const float4*>(sp.part_acc + ik * kD + lane * PER);
  }
  // the first 32 parts' (max, sum) stay in registers; more parts are read again
  float M = m0;
  for (int i = lane + 32; i < nparts; i += 32) {
    const int64_t idx = part_index(i);
    if (idx >= 0) M = fmaxf(M, sp.part_m[idx]);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
  const float w0 = idx0 >= 0 ? exp2f(m0 - M) : 0.f;
  float den = w0 * l0, acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
#pragma unroll
  for (int k = 0; k < kEarly; ++k) {
    const float wk = __shfl_sync(0xFFFFFFFFu, w0, k);      // 0 for missing parts
    acc[0] = fmaf(wk, early[k].x, acc[0]);
    acc[1] = fmaf(wk, early[k].y, acc[1]);
    acc[2] = fmaf(wk, early[k].z, acc[2]);
    acc[3] = fmaf(wk, early[k].w, acc[3]);
  }
  for (int base = 0; base < nparts; base += 32) {
    const int i = base + lane;
    int64_t idx = -1;
    float w = 0.f;
    if (base == 0) {
      idx = idx0;
      w = w0;
    } else if (i < nparts) {
      idx = part_index(i);
      if (idx >= 0) {
        w = exp2f(sp.part_m[idx] - M);
        den = fmaf(w, sp.part_l[idx], den);
      }
    }
    const int cnt = min(32, nparts - base);
#pragma unroll 8
    for (int k = base == 0 ? kEarly : 0; k < cnt; ++k) {
      const float wk = __shfl_sync(0xFFFFFFFFu, w, k);
      const long long ik = __shfl_sync(0xFFFFFFFFu, (long long)idx, k);
      if (ik >= 0) {
        const float4 v = *reinterpret_cast<const float4*>(sp.part_acc + ik * kD + lane * PER);
        acc[0] = fmaf(wk, v.x, acc[0]);
        acc[1] = fmaf(wk, v.y, acc[1]);
        acc[2] = fmaf(wk, v.z, acc[2]);
        acc[3] = fmaf(wk, v.w, acc[3]);
      }
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) den += __shfl_xor_sync(0xFFFFFFFFu, den, o);
  const float inv = 1.f / den;
  const int64_t orow = (int64_t)b * p.Hq_all + (int64_t)p.head_off * (p.Hq / p.Hkv) + q;
  uint16_t* out = static_cast<uint16_t*>(p.out) + orow * kD + lane * PER;
  uint2 packed;
  packed.x = narrow2<DT>(acc[0] * inv, acc[1] * inv);
  packed.y = narrow2<DT>(acc[2] * inv, acc[3] * inv);
  *reinterpret_cast<uint2*>(out) = packed;
}

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

int device_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

template <int DT, int H, int G>
pa_status launch_t(const SkParams& sp, const CUtensorMap& k, const CUtensorMap& v,
                   const CUtensorMap& q, int grid, cudaStream_t stream) {
  constexpr int bytes = smem_bytes<DT, H, G>();
  static_assert(bytes <= 232448, "shared memory over the per-block limit");
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(decode_tcg_kernel<DT, H, G>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  });
  if (attr != cudaSuccess) return PA_ERR_CUDA;
  if (launch_pdl(decode_tcg_kernel<DT, H, G>, dim3((unsigned)grid), kThreads, bytes, stream, k,
                 v, q, sp) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

// Query heads of a sequence: at most kMaxHq (thread d of the softmax warps holds
// one accumulator per query head).
constexpr int kMaxHq = 64;

template <int DT, int H, int G>
pa_status launch_hg(const SkParams& sp, const CUtensorMap& k, const CUtensorMap& v,
                    const CUtensorMap& q, int grid, cudaStream_t stream) {
  if constexpr (H * G <= kMaxHq) return launch_t<DT, H, G>(sp, k, v, q, grid, stream);
  else return PA_ERR_UNSUPPORTED;
}

// Query heads per KV head other than a power of two (3, 5, 6, 7: e.g. 40 / 8 or
// 28 / 4 heads) are built for 4 and 8 KV heads per pass only.
template <int H>
constexpr bool odd_groups_built() { return H == 4 || H == 8; }

template <int DT, int H>
pa_status launch_h(int G, const SkParams& sp, const CUtensorMap& k, const CUtensorMap& v,
                   const CUtensorMap& q, int grid, cudaStream_t stream) {
  switch (G) {
    case 1: return launch_hg<DT, H, 1>(sp, k, v, q, grid, stream);
    case 2: return launch_hg<DT, H, 2>(sp, k, v, q, grid, stream);
    case 4: return launch_hg<DT, H, 4>(sp, k, v, q, grid, stream);
    case 8: return launch_hg<DT, H, 8>(sp, k, v, q, grid, stream);
    case 16: return launch_hg<DT, H, 16>(sp, k, v, q, grid, stream);
    default: break;
  }
  if constexpr (odd_groups_built<H>()) {
    switch (G) {
      case 3: return launch_hg<DT, H, 3>(sp, k, v, q, grid, stream);
      case 5: return launch_hg<DT, H, 5>(sp, k, v, q, grid, stream);
      case 6: return launch_hg<DT, H, 6>(sp, k, v, q, grid, stream);
      case 7: return launch_hg<DT, H, 7>(sp, k, v, q, grid, stream);
      default: break;
    }
  }
  return PA_ERR_UNSUPPORTED;
}

// KV heads per block: a tile is 128 rows = 128 / H tokens x H heads
template <int DT>
pa_status launch_dt(int H, int G, const SkParams& sp, const CUtensorMap& k, const CUtensorMap& v,
                    const CUtensorMap& q, int grid, cudaStream_t stream) {
  switch (H) {
    case 1: return launch_h<DT, 1>(G, sp, k, v, q, grid, stream);
    case 2: return launch_h<DT, 2>(G, sp, k, v, q, grid, stream);
    case 4: return launch_h<DT, 4>(G, sp, k, v, q, grid, stream);
    case 8: return launch_h<DT, 8>(G, sp, k, v, q, grid, stream);
    case 16: return launch_h<DT, 16>(G, sp, k, v, q, grid, stream);
    case 32: return launch_h<DT, 32>(G, sp, k, v, q, grid, stream);
    default: return PA_ERR_UNSUPPORTED;
  }
}

}  // namespace

static bool pow2_group(int G) { return G == 1 || G == 2 || G == 4 || G == 8 || G == 16; }

// KV heads per pass: all of them when their query heads fit one pass (thread d
// of the softmax warps keeps one accumulator per query head, at most kMaxHq),
// else the largest group of 1, 2, 4, 8, 16 or 32 heads that divides Hkv and
// whose query heads fit (for G of 3, 5, 6 or 7: a group of 8 or 4 heads, the
// ones built); 0 when none does.
int heads_per_pass(int Hkv, int G) {
  const bool odd = !pow2_group(G);
  if (odd && G != 3 && G != 5 && G != 6 && G != 7) return 0;
  for (int hg = 32; hg >= 1; hg >>= 1)
    if (hg <= Hkv && Hkv % hg == 0 && hg * G <= kMaxHq && (!odd || hg == 4 || hg == 8))
      return hg;
  return 0;
}

bool tcg_supported(const DecodeParams& p) {
  const int G = p.Hq / p.Hkv;
  if (p.D != kD) return false;
  const int hg = heads_per_pass(p.Hkv, G);
  if (hg == 0) return false;
  if (p.B > kMaxSeqs) return false;
  // a bad block id is redirected to row num_blocks * bs (+ offset < 64): stays an int
  if ((long long)p.num_blocks * p.bs + 64 >= (1ll << 31)) return false;
  if ((long long)p.B * p.Hq >= (1ll << 31)) return false;
  // The start weight keeps every range within its window when B <= (kWin - 2)
  // grid / 2; it is then at most max(3, T / den + 1) with den >= B, so the
  // batch's weight T + sw B <= max(T + 3 B, 2 T + B) stays an int.
  const int grid = device_sms() < kSkMaxGrid ? device_sms() : kSkMaxGrid;
  if (grid <= 0 || 2ll * p.B > (long long)(kWin - 2) * grid) return false;
  const long long TT = kRows / hg;
  if (2ll * p.B * ((p.max_seq_len + TT - 1) / TT + 1) >= (1ll << 31)) return false;
  return encode_fn() != nullptr;
}

SkLayout sk_layout(int B, int Hq) {
  auto a = [](size_t x) { return (x + 255) & ~(size_t)255; };
  SkLayout l;
  l.prefix_off = 0;
  l.wprefix_off = l.prefix_off + a((size_t)(B + 1) * sizeof(int));
  l.m_off = l.wprefix_off + a((size_t)(B + 2) * sizeof(int));
  const size_t parts = (size_t)kSkMaxGrid * 2 * Hq;
  l.l_off = l.m_off + a(parts * sizeof(float));
  l.acc_off = l.l_off + a(parts * sizeof(float));
  l.total = l.acc_off + a(parts * kD * sizeof(float));
  return l;
}

// The stream-K area's pointers for a call over p.Hq_all query heads.
static SkParams sk_params(const DecodeParams& p, void* sk_ws, int chain) {
  const SkLayout l = sk_layout(p.B, p.Hq_all);
  char* ws = static_cast<char*>(sk_ws);
  SkParams sp;
  sp.p = p;
  sp.chain = chain;
  sp.tile_prefix = reinterpret_cast<int*>(ws + l.prefix_off);
  sp.weight_prefix = reinterpret_cast<int*>(ws + l.wprefix_off);
  sp.part_m = reinterpret_cast<float*>(ws + l.m_off);
  sp.part_l = reinterpret_cast<float*>(ws + l.l_off);
  sp.part_acc = reinterpret_cast<float*>(ws + l.acc_off);
  return sp;
}

static int launch_grid() {
  const int grid = device_sms();
  return grid > kSkMaxGrid ? kSkMaxGrid : grid;
}

// One pass's main kernel: the KV heads p.head_off .. p.head_off + p.Hkv - 1 (of
// p.Hkv_all).
static pa_status launch_pass(const DecodeParams& p, void* sk_ws, int chain, cudaStream_t stream) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return PA_ERR_UNSUPPORTED;
  const int H = p.Hkv, G = p.Hq / p.Hkv;
  const int TT = kRows / H;
  const int N = (p.Hq + 15) / 16 * 16;
  const CUtensorMapDataType dt =
      p.dtype == PA_BFLOAT16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const int box_tokens = p.bs < TT ? p.bs : TT;
  CUtensorMap tk, tv, tq;
  // [blocks][bs][Hkv_all][D] as a 4-D tensor over this pass's H heads: a box
  // whose in-block coordinate is negative reads zeros there instead of the
  // previous block's tokens
  const cuuint64_t kv_dims[4] = {(cuuint64_t)kD, (cuuint64_t)H, (cuuint64_t)p.bs,
                                 (cuuint64_t)p.num_blocks};
  const cuuint64_t kv_strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)p.Hkv_all * kD * 2,
                                    (cuuint64_t)p.bs * p.Hkv_all * kD * 2};
  const cuuint32_t kv_box[4] = {64, (cuuint32_t)H, (cuuint32_t)box_tokens, 1};
  const cuuint32_t ones[4] = {1, 1, 1, 1};
  const size_t head_bytes = (size_t)p.head_off * kD * 2;
  void* kbase = static_cast<char*>(const_cast<void*>(p.k_pool)) + head_bytes;
  void* vbase = static_cast<char*>(const_cast<void*>(p.v_pool)) + head_bytes;
  if (enc(&tk, dt, 4, kbase, kv_dims, kv_strides, kv_box, ones,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return PA_ERR_INVALID_ARG;
  if (enc(&tv, dt, 4, vbase, kv_dims, kv_strides, kv_box, ones,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return PA_ERR_INVALID_ARG;
  const cuuint64_t q_dims[2] = {(cuuint64_t)kD, (cuuint64_t)p.B * p.Hq_all};
  const cuuint64_t q_strides[1] = {(cuuint64_t)kD * 2};
  const cuuint32_t q_box[2] = {64, (cuuint32_t)N};
  if (enc(&tq, dt, 2, const_cast<void*>(p.q), q_dims, q_strides, q_box, ones,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return PA_ERR_INVALID_ARG;

  const int grid = launch_grid();
  if (grid <= 0) return PA_ERR_CUDA;
  const SkParams sp = sk_params(p, sk_ws, chain);
  return p.dtype == PA_BFLOAT16 ? launch_dt<PA_BFLOAT16>(H, G, sp, tk, tv, tq, grid, stream)
                                : launch_dt<PA_FLOAT16>(H, G, sp, tk, tv, tq, grid, stream);
}

// The combine over every query head of the call (p: all heads, head_off 0).
static pa_status launch_combine_sk(const DecodeParams& p, void* sk_ws, cudaStream_t stream) {
  const int grid = launch_grid();
  if (grid <= 0) return PA_ERR_CUDA;
  const SkParams sp = sk_params(p, sk_ws, 0);
  const long long rows = (long long)p.B * p.Hq;
  if (rows == 0) return PA_OK;
  const int cgrid = (int)((rows + 3) / 4);
  // The combine keeps the main kernel's shared-memory carve-out, so an SM does
  // not switch L1 / shared-memory configuration between the two kernels.
  static std::once_flag carve_once;
  std::call_once(carve_once, [] {
    cudaFuncSetAttribute(combine_sk_kernel<PA_BFLOAT16>,
                         cudaFuncAttributePreferredSharedMemoryCarveout,
                         (int)cudaSharedmemCarveoutMaxShared);
    cudaFuncSetAttribute(combine_sk_kernel<PA_FLOAT16>,
                         cudaFuncAttributePreferredSharedMemoryCarveout,
                         (int)cudaSharedmemCarveoutMaxShared);
  });
  const cudaError_t e =
      p.dtype == PA_BFLOAT16
          ? launch_pdl(combine_sk_kernel<PA_BFLOAT16>, dim3((unsigned)cgrid), 128, 0, stream, sp, grid)
          : launch_pdl(combine_sk_kernel<PA_FLOAT16>, dim3((unsigned)cgrid), 128, 0, stream, sp, grid);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// Query heads beyond kMaxHq (G = 16, or wide multi-head attention) run as
// passes over groups of KV heads; the passes read disjoint heads of every pool
// row, so the bytes read are the same as one pass over all heads.  The passes
// form a chain (kChainTrigger, kChainLateWait): each writes its own heads'
// partials into the shared stream-K area (partials of all heads side by side;
// the tile and weight prefixes are the same for every pass), so one pass can
// start while the previous one ends, and one combine merges every head.
pa_status launch_decode_tcg(const DecodeParams& p, void* sk_ws, cudaStream_t stream) {
  const int G = p.Hq / p.Hkv;
  const int hg = heads_per_pass(p.Hkv, G);
  if (hg == 0) return PA_ERR_UNSUPPORTED;
  for (int off = 0; off < p.Hkv; off += hg) {
    DecodeParams pp = p;
    pp.Hkv = hg;
    pp.Hq = hg * G;
    pp.head_off = p.head_off + off;
    const int chain = (off + hg < p.Hkv ? kChainTrigger : 0) | (off > 0 ? kChainLateWait : 0);
    const pa_status st = launch_pass(pp, sk_ws, chain, stream);
    if (st != PA_OK) return st;
  }
  return launch_combine_sk(p, sk_ws, stream);
}

}  // namespace pa
