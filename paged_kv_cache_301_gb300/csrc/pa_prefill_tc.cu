// pa_prefill on the tensor cores: causal multi-query attention over the paged
// KV pool (prefill, chunked prefill, verification of drafted tokens).
//
// The subroutine-cs article's introduction splits serving into a prefill phase
// (all prompt tokens at once) and a decode phase (one token, attending to all
// earlier ones).  Once the new tokens' K/V sit in their blocks (written by
// pa_reshape_and_cache), prefill attention is the decode gather of "10 — Paged
// Attention" §5 "The kernel side" for many queries, each limited to the
// positions up to its own.
//
// Work item (one CTA): sequence b, KV head h and two adjacent query tiles A, B
// of 128 rows each = TQ = 128 / G query tokens x the G query heads of h
// (row = token * G + g; for G = 3, 5, 6, 7, 128 / G rounded down, and the last
// 2 or 3 rows unused).  Every K/V tile loaded serves both, 256 query rows, so
// the per-head gather (128-byte rows 2 KB apart, ~35 GB/s per SM through TMA on
// GB300) feeds twice the tensor work of a single tile.  For KV tiles of 128 keys
// and each query tile k:
//
//   S_k  = Q_k[128 x D] . K_tile^T           (TMEM, 128 fp32 columns)
//   row r: mask keys past its position, running max m, p = 2^(s - m)
//   P_k  [128 x 128 keys] as two storage-type terms hi + lo, written to tensor
//        memory over the S columns it replaces
//   O_k += P_k . V_tile   [128 x D]          (P from TMEM, V from shared memory,
//                                             O accumulated in TMEM)
//
// The tensor core alternates between the tiles (P_A.V, S_A next, P_B.V, S_B
// next) while the softmax warps of the other tile work.  The running max is
// raised only when a tile's max exceeds it by more than 8 (a factor 2^8): O and
// the row sum are then rescaled by 2^(m_old - m_new) before the tile's product;
// otherwise p may reach 2^8, which fp32 sums and the hi + lo terms carry as
// well.  The final division by the row sum removes the choice of max.
//
// Roles (320 threads): warp 0 issues TMA (both Q tiles, then K(t), V(t) into a
// ring of 32 KB stages), warp 1 issues tcgen05.mma, warps 2-5 run tile A's
// softmax and warps 6-9 tile B's, one thread per row (all 128 keys of a tile,
// all 128 output columns: no exchange between warps).  Every wait is bounded.
#include <math_constants.h>

#include <mutex>

#include "pa_common.cuh"
#include "pa_internal.h"
#include "pa_sm100.cuh"

namespace pa {
namespace {

using namespace sm100;

constexpr int kD = 128;
constexpr int kRows = 128;                  // query rows per tile (M)
constexpr int kKeys = 128;                  // keys per KV tile (N of S, K of P.V)
constexpr int kSlab = 128 * 128;            // 128 rows x 128 bytes
constexpr int kTile = 2 * kSlab;            // 128 rows x 256 bytes (D = 128, 16-bit)
constexpr int kQOff = 0;                    // Q_A, then Q_B
constexpr int kRingOff = kQOff + 2 * kTile;
constexpr int kSoftWarps = 8;               // four per query tile, one thread per row
constexpr int kThreads = 64 + 32 * kSoftWarps;
constexpr float kRescaleLog2 = 8.f;         // raise the running max only past this
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kSmemBudget = 232448 - 1024;  // per-block limit minus alignment slack
constexpr int kTailBytes = 8192;
constexpr int kStages = (kSmemBudget - kRingOff - kTailBytes) / kTile > 6
                            ? 6 : (kSmemBudget - kRingOff - kTailBytes) / kTile;
// TMEM: S/P_A at column 0, S/P_B at 128 (P overwrites the S it was computed
// from), O_A at 256, O_B at 384
constexpr uint32_t kTmemCols = 512;

struct Tail {
  uint64_t full[kStages], empty[kStages];
  uint64_t q_full;
  uint64_t s_full[2], p_full[2], pv_done[2];   // per query tile
  uint64_t drain;
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(Tail) <= kTailBytes, "barrier block");
constexpr int kTailOff = kRingOff + kStages * kTile;
constexpr int kSmemBytes = kTailOff + kTailBytes + 1024;
static_assert(kStages >= 3, "ring too shallow");
static_assert(kSmemBytes <= 232448, "shared memory over the per-block limit");

struct PrefillParams {
  void* out;                    // [total_q, Hq, D]
  const int32_t* tables;        // [B, max_blocks]
  const int32_t* seq_lens;      // [B]
  const int32_t* q_start;       // [B + 1]
  int B, total_q, Hq, Hkv, bs, max_blocks, num_blocks, max_q_len, n_qpairs;
  float scale_log2;
  int32_t* status_dev;
};

template <int DT, int G>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_q, const PrefillParams p) {
  constexpr int TQ = kRows / G;                 // query tokens per tile
  constexpr int kUsedRows = TQ * G;             // 128, or 125 / 126 when G does not divide it
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  Tail* tl = reinterpret_cast<Tail*>(smem + kTailOff);
  volatile int* abort_flag = &tl->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  allow_next_grid();
  wait_prior_grid();               // q, the pools and the tables may come from the previous kernel
  // blockIdx.x walks the (sequence, KV head) pairs and blockIdx.y the query-tile
  // pairs, longest causal work first: CTAs resident together read different
  // K/V, and each (sequence, KV head)'s K/V stays in L2 for its later query tiles
  const int b = blockIdx.x / p.Hkv, h = blockIdx.x - b * p.Hkv;
  const int qp = p.n_qpairs - 1 - (int)blockIdx.y;
  const int qs = p.q_start[b];
  const int n = p.q_start[b + 1] - qs;
  const int L = p.seq_lens[b];
  if (n < 0 || n > L || n > p.max_q_len || L > p.max_blocks * p.bs || qs < 0 ||
      qs + n > p.total_q) {
    if (threadIdx.x == 0 && h == 0 && qp == 0) report(p.status_dev, PA_ERR_BAD_BLOCK_ID);
    return;
  }
  // query tile k = 0 (A), 1 (B): first query token, and the KV tiles 0 .. last_k
  // its causal rows reach (-1: no rows)
  const int q0a = 2 * qp * TQ, q0b = q0a + TQ;
  if (q0a >= n) return;                         // uniform: no rows in this pair
  const int last_a = (L - n + min(q0a + TQ, n) - 1) / kKeys;
  const int last_b = q0b < n ? (L - n + min(q0b + TQ, n) - 1) / kKeys : -1;
  const int last_all = last_b >= 0 ? last_b : last_a;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&tl->full[s], 1);
      mbar_init(&tl->empty[s], 1);
    }
    mbar_init(&tl->q_full, 1);
    for (int k = 0; k < 2; ++k) {
      mbar_init(&tl->s_full[k], 1);
      mbar_init(&tl->p_full[k], kSoftWarps / 2);
      mbar_init(&tl->pv_done[k], 1);
    }
    mbar_init(&tl->drain, 1);
    tl->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_q);
  }
  if (warp == 1) {
    tmem_alloc(&tl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tl->tmem_base;
  auto set_abort = [&]() {
    tl->abort_flag = 1;
    report(p.status_dev, PA_ERR_TIMEOUT);
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- producer --
    const uint64_t q_policy = policy_evict_first();     // read by this CTA only
    const uint64_t kv_policy = policy_evict_last();     // re-read by the sequence's other tiles
    const int32_t* table = p.tables + (int64_t)b * p.max_blocks;
    const int blocks_per_tile = kKeys / p.bs;          // bs divides 128
    const int nblk_seq = (L + p.bs - 1) / p.bs;
    int stage = 0, sphase = 0;
    int issued[kStages];
#pragma unroll
    for (int s = 0; s < kStages; ++s) issued[s] = -1;
    bool ok = true, q_issued = false;
    if (lane == 0) {            // both query tiles (rows past the batch read as zeros)
      mbar_arrive_expect_tx(&tl->q_full, 2u * 2u * kUsedRows * 128u);
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        uint8_t* dst = smem + kQOff + k * kTile;
        const int z = qs + (k ? q0b : q0a);
        tma_load_3d_hint(dst, &tm_q, &tl->q_full, 0, h * G, z, q_policy);
        tma_load_3d_hint(dst + kSlab, &tm_q, &tl->q_full, 64, h * G, z, q_policy);
      }
      q_issued = true;
    }
    // one K or V tile: lanes < nops each copy one block (both 64-column slabs)
    auto issue = [&](const CUtensorMap* map, int t) -> bool {
      const int kb = t * blocks_per_tile;
      const int nops = min(blocks_per_tile, nblk_seq - kb);
      bool good = true;
      if (lane == 0) {
        good = mbar_wait(&tl->empty[stage], sphase ^ 1, abort_flag, kWaitNs);
        if (good) mbar_arrive_expect_tx(&tl->full[stage], (uint32_t)nops * p.bs * 256u);
        else set_abort();
      }
      good = __shfl_sync(0xFFFFFFFFu, (int)good, 0) != 0;
      if (!good) return false;
      if (lane < nops) {
        const int32_t blk = table[kb + lane];
        if (p.status_dev && (blk < 0 || blk >= p.num_blocks))
          report(p.status_dev, PA_ERR_BAD_BLOCK_ID);      // TMA reads outside the pool as zeros
        uint8_t* dst = smem + kRingOff + stage * kTile + lane * p.bs * 128;
        tma_load_3d_hint(dst, map, &tl->full[stage], 0, h, blk * p.bs, kv_policy);
        tma_load_3d_hint(dst + kSlab, map, &tl->full[stage], 64, h, blk * p.bs, kv_policy);
      }
      __syncwarp();
      issued[stage] = sphase;
      if (++stage == kStages) {
        stage = 0;
        sphase ^= 1;
      }
      return true;
    };
    for (int t = 0; t <= last_all && ok; ++t) {      // ring order: K(0), V(0), K(1), V(1), ...
      ok = issue(&tm_k, t);
      if (ok) ok = issue(&tm_v, t);
    }
    if (*abort_flag && lane == 0) {            // let copies in flight land before exit
      for (int s = 0; s < kStages; ++s)
        if (issued[s] >= 0) mbar_wait_drain(&tl->full[s], issued[s], kWaitNs);
      if (q_issued) mbar_wait_drain(&tl->q_full, 0, kWaitNs);
    }
  } else if (warp == 1) {
    // -------------------------------------------------------------- MMA issue --
    constexpr uint32_t ab = DT == PA_BFLOAT16 ? 1u : 0u;
    constexpr uint32_t idesc_s = idesc_f16(ab, 0, 0, kRows, kKeys);   // Q, K both K-major
    constexpr uint32_t idesc_o = idesc_f16(ab, 0, 1, kRows, kD);      // P (TMEM), V MN-major
    const uint32_t ring = smem_addr(smem + kRingOff);
    const uint32_t qaddr = smem_addr(smem + kQOff);
    bool ok = true, committed = false;
    // One thread issues every MMA, one per 64 tensor cycles at full rate, so the
    // shared-memory descriptors are built once per operand and stepped by
    // compile-time offsets (the start-address field holds address / 16).
    const uint64_t qdesc_a = smem_desc_sw128(qaddr, 16, 1024);
    const uint64_t qdesc_b = smem_desc_sw128(qaddr + kTile, 16, 1024);
    // S_k = Q_k . K(t)^T into S/P buffer k
    auto issue_s = [&](int k, int t) {
      const uint64_t kdesc = smem_desc_sw128(ring + ((2 * t) % kStages) * kTile, 16, 1024);
      const uint64_t q0d = k ? qdesc_b : qdesc_a;
      const uint32_t d = tmem + k * kKeys;
#pragma unroll
      for (int kk = 0; kk < kD / 16; ++kk) {
        const uint64_t off = (uint64_t)(((kk >> 2) * kSlab + (kk & 3) * 32) >> 4);
        mma_f16(d, q0d + off, kdesc + off, idesc_s, kk > 0);
      }
      mma_commit(&tl->s_full[k]);
    };
    // O_k += (P_hi + P_lo) . V(t).  P sits in S/P buffer k: 16-key group g occupies
    // columns 16g .. 16g+7 (hi) and 16g+8 .. 16g+15 (lo).
    auto issue_pv = [&](int k, int t) {
      const uint64_t vdesc = smem_desc_sw128(ring + ((2 * t + 1) % kStages) * kTile, kSlab, 1024);
      const uint32_t d = tmem + 256 + k * kD, pcol = tmem + k * kKeys;
#pragma unroll
      for (int kk = 0; kk < kKeys / 16; ++kk) {
        const uint64_t bd = vdesc + (uint64_t)((kk * 16 * 128) >> 4);
#pragma unroll
        for (int term = 0; term < 2; ++term)
          mma_f16_ts(d, pcol + kk * 16 + term * 8, bd, idesc_o, (t | kk | term) != 0);
      }
      mma_commit(&tl->pv_done[k]);
    };
    auto stage_wait = [&](int pos) -> bool {
      return mbar_wait(&tl->full[pos % kStages], (pos / kStages) & 1, abort_flag, kWaitNs);
    };
    if (lane == 0) {
      ok = mbar_wait(&tl->q_full, 0, abort_flag, kWaitNs) && stage_wait(0);
      if (ok) {
        tc_fence_after();
        issue_s(0, 0);
        if (last_b >= 0) issue_s(1, 0);
        mma_commit(&tl->empty[0]);
        committed = true;
      }
      for (int t = 0; t <= last_all && ok; ++t) {
        ok = stage_wait(2 * t + 1);                      // V(t)
        bool next_k = false;                             // K(t+1) landed
        for (int k = 0; k < 2 && ok; ++k) {
          const int last_k = k ? last_b : last_a;
          if (t > last_k) continue;
          ok = mbar_wait(&tl->p_full[k], t & 1, abort_flag, kWaitNs);
          if (!ok) break;
          tc_fence_after();
          issue_pv(k, t);
          if (t + 1 <= last_k) {
            // S_k(t+1) overwrites P_k(t): after P_k(t).V(t) has read it
            ok = (next_k || stage_wait(2 * t + 2)) &&
                 mbar_wait(&tl->pv_done[k], t & 1, abort_flag, kWaitNs);
            if (!ok) break;
            next_k = true;
            tc_fence_after();
            issue_s(k, t + 1);
          }
        }
        if (!ok) break;
        mma_commit(&tl->empty[(2 * t + 1) % kStages]);   // V(t) read by every product
        if (t + 1 <= last_all) mma_commit(&tl->empty[(2 * t + 2) % kStages]);   // K(t+1)
      }
      if (!ok) set_abort();
      if (*abort_flag && committed) {          // let issued MMAs finish before TMEM is freed
        mma_commit(&tl->drain);
        mbar_wait_drain(&tl->drain, 0, kWaitNs);
      }
    }
    __syncwarp();
  }
  else {
    // ------------------------------------------------ softmax and output rows --
    // Tile k = 0 (A, warps 2-5) or 1 (B, warps 6-9); warp w reads the TMEM lane
    // quarter w % 4, so thread r = 32 (w % 4) + lane owns tile row r: all 128 keys
    // of every S tile (no exchange with another warp) and all 128 output columns.
    const int k = (warp - 2) >> 2;
    const int wq = warp & 3;                     // TMEM lane quarter of this warp
    const int r = wq * 32 + lane;                // tile row = query token r / G, head r % G
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const int i = (k ? q0b : q0a) + r / G;       // query token within the sequence's queries
    // rows past TQ * G (G not a power of two) hold no query: their Q rows in
    // shared memory are never written, and every key is masked for them
    const bool row_valid = r < kUsedRows && i < n;
    const int pos = row_valid ? L - n + i : -1;  // keys 0 .. pos are visible
    const uint32_t scol = tmem + lane_base + k * kKeys;
    const uint32_t ocol = tmem + lane_base + 256 + k * kD;
    const float sl2 = p.scale_log2;
    float m_run = -CUDART_INF_F, l_run = 0.f;
    bool ok = true;
    auto wait_all = [&](uint64_t* bar, int parity) -> bool {
      const bool w = mbar_wait(bar, parity, abort_flag, kWaitNs);
      return __all_sync(0xFFFFFFFFu, w);
    };
    const int my_last = k ? last_b : last_a;
    for (int t = 0; t <= my_last && ok; ++t) {
      if (!wait_all(&tl->s_full[k], t & 1)) { ok = false; break; }
      tc_fence_after();
      const int kc = t * kKeys;                  // key of column 0
      const bool partial = kc + kKeys - 1 > pos; // some keys lie past the row
      // S is read from tensor memory once and kept in registers (fewer TMEM
      // reads competing with the tensor core's); masked keys become -inf
      float sv[kKeys];
      {
        float h0[64], h1[64];
        tmem_ld64(scol, h0);
        tmem_ld64(scol + 64, h1);
#pragma unroll
        for (int e = 0; e < 64; ++e) {
          sv[e] = h0[e];
          sv[64 + e] = h1[e];
        }
      }
      if (partial) {
#pragma unroll
        for (int e = 0; e < kKeys; ++e) sv[e] = kc + e <= pos ? sv[e] : -CUDART_INF_F;
      }
      // the softmax is bound by instruction issue: three-input max, and packed
      // two-wide fp32 arithmetic below
      float mx4[4] = {-CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
      for (int e = 0; e < kKeys; e += 8) {
#pragma unroll
        for (int c = 0; c < 4; ++c) mx4[c] = fmax3(mx4[c], sv[e + 2 * c], sv[e + 2 * c + 1]);
      }
      const float mt = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
      const float m_tile = mt * sl2;
      // Rows whose max grows by more than 2^8 raise it; O (complete up to tile
      // t-1) and l scale by 2^(m_old - m_new).  TMEM access is warp-wide, so the
      // warp rescales when any of its rows needs it (the others by 1).
      const bool raise = m_run != -CUDART_INF_F && m_tile > m_run + kRescaleLog2;
      const float alpha = raise ? ex2_approx(m_run - m_tile) : 1.f;
      if (m_run == -CUDART_INF_F || raise) m_run = m_tile;   // first visible tile, or raised
      const float neg_m = m_run == -CUDART_INF_F ? 0.f : -m_run;
      // p = 2^(s * scale * log2 e - m), written back over the S columns as
      // hi / lo storage-type pairs (16-key group: 8 hi words, then 8 lo words);
      // masked keys hold -inf and give p = 0
      const uint64_t sl2x2 = f2_pack(sl2, sl2), negm2 = f2_pack(neg_m, neg_m);
      uint64_t ls2[2] = {f2_pack(0.f, 0.f), f2_pack(0.f, 0.f)};
#pragma unroll
      for (int g = 0; g < kKeys; g += 16) {
        uint32_t pw[16];
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          float ta, tb;
          f2_unpack(f2_fma(f2_pack(sv[g + e], sv[g + e + 1]), sl2x2, negm2), ta, tb);
          const float pa_ = ex2_approx(ta);
          const float pb_ = ex2_approx(tb);
          const uint64_t p2 = f2_pack(pa_, pb_);
          ls2[(e >> 1) & 1] = f2_add(ls2[(e >> 1) & 1], p2);
          if (DT == PA_BFLOAT16) {
            // hi = the top 16 bits (truncation), lo = the remainder, truncated
            // too: hi + lo carries ~15 significant bits with byte permutes only
            // (no conversion instruction)
            const uint32_t ua = __float_as_uint(pa_), ub = __float_as_uint(pb_);
            pw[e >> 1] = __byte_perm(ua, ub, 0x7632);
            float ra, rb;
            f2_unpack(f2_sub(p2, f2_pack(__uint_as_float(ua & 0xFFFF0000u),
                                         __uint_as_float(ub & 0xFFFF0000u))), ra, rb);
            pw[8 + (e >> 1)] = __byte_perm(__float_as_uint(ra), __float_as_uint(rb), 0x7632);
          } else {
            const uint32_t h2 = narrow2<DT>(pa_, pb_);
            const float2 hf = widen2<DT>(h2);
            pw[e >> 1] = h2;
            pw[8 + (e >> 1)] = narrow2<DT>(pa_ - hf.x, pb_ - hf.y);
          }
        }
        tmem_st16_nowait(scol + g, pw);          // over S columns already read
      }
      float ls4[4];
      f2_unpack(ls2[0], ls4[0], ls4[1]);
      f2_unpack(ls2[1], ls4[2], ls4[3]);
      const float ls = (ls4[0] + ls4[1]) + (ls4[2] + ls4[3]);
      // Rows that raised their max rescale O (complete up to tile t-1, P.V(t) not
      // yet issued) and l.
      if (__any_sync(0xFFFFFFFFu, raise)) {
        if (!wait_all(&tl->pv_done[k], (t - 1) & 1)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int c0 = 0; c0 < kD; c0 += 32) {
          float o[32];
          tmem_ld32(ocol + c0, o);
          uint32_t ow[32];
#pragma unroll
          for (int e = 0; e < 32; ++e) ow[e] = __float_as_uint(o[e] * alpha);
          tmem_st32(ocol + c0, ow);
        }
      }
      l_run = fmaf(l_run, alpha, ls);
      // keys at or past L: their V rows hold whatever the slot or an earlier tile
      // left (0 * NaN must not reach O).  The first tile whose product reads V(t)
      // zeroes them before releasing its P.
      if (kc + kKeys > L && (k == 0 || t > last_a)) {
        const int u = 2 * t + 1;
        if (!wait_all(&tl->full[u % kStages], (u / kStages) & 1)) { ok = false; break; }
        if (kc + r >= L) {                       // V row r, both 64-column slabs
          uint4* v0 = reinterpret_cast<uint4*>(smem + kRingOff + (u % kStages) * kTile + r * 128);
          uint4* v1 = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(v0) + kSlab);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            v0[e] = make_uint4(0, 0, 0, 0);
            v1[e] = make_uint4(0, 0, 0, 0);
          }
        }
      }
      // consume P.V(t-1)'s completion before P(t) is released, so the barrier
      // cannot run two phases ahead of any waiting warp
      if (t > 0 && !wait_all(&tl->pv_done[k], (t - 1) & 1)) { ok = false; break; }
      tmem_wait_st();                            // every P word is in tensor memory
      tc_fence_before();
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tl->p_full[k]);
    }
    if (my_last >= 0) {
      if (ok) ok = wait_all(&tl->pv_done[k], my_last & 1);
      if (!ok) {
        if (lane == 0) set_abort();
      } else {
        tc_fence_after();
        const float inv = 1.f / l_run;
        uint4* dst = reinterpret_cast<uint4*>(
            static_cast<uint16_t*>(p.out) + ((int64_t)(qs + (row_valid ? i : 0)) * p.Hq + h * G +
                                             r % G) * kD);
#pragma unroll
        for (int c0 = 0; c0 < kD; c0 += 32) {
          float o[32];
          tmem_ld32(ocol + c0, o);
          if (row_valid) {
#pragma unroll
            for (int c = 0; c < 4; ++c)
              dst[c0 / 8 + c] = make_uint4(narrow2<DT>(o[8 * c] * inv, o[8 * c + 1] * inv),
                                           narrow2<DT>(o[8 * c + 2] * inv, o[8 * c + 3] * inv),
                                           narrow2<DT>(o[8 * c + 4] * inv, o[8 * c + 5] * inv),
                                           narrow2<DT>(o[8 * c + 6] * inv, o[8 * c + 7] * inv));
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
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

template <int DT, int G>
pa_status launch_g(const PrefillParams& p, const CUtensorMap& k, const CUtensorMap& v,
                   const CUtensorMap& q, cudaStream_t stream) {
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(prefill_tc_kernel<DT, G>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  });
  if (attr != cudaSuccess) return PA_ERR_CUDA;
  const dim3 grid((unsigned)(p.Hkv * p.B), (unsigned)p.n_qpairs);
  if (launch_pdl(prefill_tc_kernel<DT, G>, grid, kThreads, kSmemBytes, stream, k, v, q, p) !=
      cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

template <int DT>
pa_status launch_dt(int G, const PrefillParams& p, const CUtensorMap& k, const CUtensorMap& v,
                    const CUtensorMap& q, cudaStream_t stream) {
  switch (G) {
    case 1: return launch_g<DT, 1>(p, k, v, q, stream);
    case 2: return launch_g<DT, 2>(p, k, v, q, stream);
    case 3: return launch_g<DT, 3>(p, k, v, q, stream);
    case 4: return launch_g<DT, 4>(p, k, v, q, stream);
    case 5: return launch_g<DT, 5>(p, k, v, q, stream);
    case 6: return launch_g<DT, 6>(p, k, v, q, stream);
    case 7: return launch_g<DT, 7>(p, k, v, q, stream);
    case 8: return launch_g<DT, 8>(p, k, v, q, stream);
    case 16: return launch_g<DT, 16>(p, k, v, q, stream);
    default: return PA_ERR_UNSUPPORTED;
  }
}

bool aligned16(const void* ptr) { return ((uintptr_t)ptr & 15u) == 0; }

}  // namespace
}  // namespace pa

using namespace pa;

static int g_prefill_path = PA_PREFILL_AUTO;

extern "C" pa_status pa_set_prefill_path(int path) {
  if (path < PA_PREFILL_AUTO || path > PA_PREFILL_TC) return PA_ERR_INVALID_ARG;
  g_prefill_path = path;
  return PA_OK;
}

extern "C" pa_status pa_prefill(void* out, const void* q, const void* k_pool, const void* v_pool,
                                const int32_t* block_tables, const int32_t* seq_lens,
                                const int32_t* q_start, int num_seqs, int total_q,
                                int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                int max_blocks, int num_blocks, int max_q_len, float scale,
                                int dtype, int32_t* status_dev, cudaStream_t stream) {
  if (num_seqs < 0 || total_q < 0 || max_q_len < 0 || num_kv_heads <= 0 || num_q_heads <= 0 ||
      num_q_heads % num_kv_heads != 0 || max_blocks <= 0 || num_blocks <= 0 ||
      !(scale > 0.f) || !(scale < 3.0e38f))
    return PA_ERR_INVALID_ARG;
  const int G = num_q_heads / num_kv_heads;
  if ((head_dim != 64 && head_dim != 128) ||
      (block_size != 8 && block_size != 16 && block_size != 32 && block_size != 64) ||
      (dtype != PA_FLOAT16 && dtype != PA_BFLOAT16))
    return PA_ERR_UNSUPPORTED;
  const int path = g_prefill_path;
  // a query tile holds 128 / G query tokens (G = 3, 5, 6, 7: 125 or 126 of its
  // 128 rows used)
  const bool tc_shape = head_dim == kD && ((G >= 1 && G <= 8) || G == 16);
  if (path == PA_PREFILL_TC && !tc_shape) return PA_ERR_UNSUPPORTED;
  if (num_seqs == 0 || total_q == 0 || max_q_len == 0) return PA_OK;
  if (!out || !q || !k_pool || !v_pool || !block_tables || !seq_lens || !q_start)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool))
    return PA_ERR_INVALID_ARG;
  if ((int64_t)num_blocks * block_size >= (1ll << 31) ||
      (int64_t)total_q * num_q_heads >= (1ll << 31))
    return PA_ERR_INVALID_ARG;
  EncodeTiledFn enc = encode_fn();
  if (!tc_shape || path == PA_PREFILL_SIMT || !enc) {
    PrefillArgs a;
    a.out = out;
    a.q = q;
    a.k_pool = k_pool;
    a.v_pool = v_pool;
    a.tables = block_tables;
    a.seq_lens = seq_lens;
    a.q_start = q_start;
    a.B = num_seqs;
    a.total_q = total_q;
    a.Hq = num_q_heads;
    a.Hkv = num_kv_heads;
    a.D = head_dim;
    a.bs = block_size;
    a.max_blocks = max_blocks;
    a.num_blocks = num_blocks;
    a.max_q_len = max_q_len;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.dtype = dtype;
    a.status_dev = status_dev;
    return launch_prefill_simt(a, stream);
  }
  const int TQ = kRows / G;
  const int64_t n_qtiles = ((int64_t)max_q_len + TQ - 1) / TQ;
  if ((n_qtiles + 1) / 2 > 65535 || (int64_t)num_seqs * num_kv_heads > 0x7FFFFFFF)
    return PA_ERR_INVALID_ARG;                                              // grid y, x

  const CUtensorMapDataType dt =
      dtype == PA_BFLOAT16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const cuuint32_t ones[3] = {1, 1, 1};
  CUtensorMap tk, tv, tq;
  const cuuint64_t kv_dims[3] = {(cuuint64_t)kD, (cuuint64_t)num_kv_heads,
                                 (cuuint64_t)num_blocks * block_size};
  const cuuint64_t kv_strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)num_kv_heads * kD * 2};
  const cuuint32_t kv_box[3] = {64, 1, (cuuint32_t)block_size};
  if (enc(&tk, dt, 3, const_cast<void*>(k_pool), kv_dims, kv_strides, kv_box, ones,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
      enc(&tv, dt, 3, const_cast<void*>(v_pool), kv_dims, kv_strides, kv_box, ones,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return PA_ERR_INVALID_ARG;
  const cuuint64_t q_dims[3] = {(cuuint64_t)kD, (cuuint64_t)num_q_heads, (cuuint64_t)total_q};
  const cuuint64_t q_strides[2] = {(cuuint64_t)kD * 2, (cuuint64_t)num_q_heads * kD * 2};
  const cuuint32_t q_box[3] = {64, (cuuint32_t)G, (cuuint32_t)TQ};
  if (enc(&tq, dt, 3, const_cast<void*>(q), q_dims, q_strides, q_box, ones,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return PA_ERR_INVALID_ARG;

  PrefillParams p;
  p.out = out;
  p.tables = block_tables;
  p.seq_lens = seq_lens;
  p.q_start = q_start;
  p.B = num_seqs;
  p.total_q = total_q;
  p.Hq = num_q_heads;
  p.Hkv = num_kv_heads;
  p.bs = block_size;
  p.max_blocks = max_blocks;
  p.num_blocks = num_blocks;
  p.max_q_len = max_q_len;
  p.n_qpairs = (int)((n_qtiles + 1) / 2);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status_dev = status_dev;
  return dtype == PA_BFLOAT16 ? launch_dt<PA_BFLOAT16>(G, p, tk, tv, tq, stream)
                              : launch_dt<PA_FLOAT16>(G, p, tk, tv, tq, stream);
}
