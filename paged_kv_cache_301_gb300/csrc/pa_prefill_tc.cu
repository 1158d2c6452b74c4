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
// Work item (one CTA): sequence b, KV head h, query tile of 128 rows =
// TQ = 128 / G query tokens x the G query heads of h (row = token * G + g), so a
// loaded K/V tile serves all heads of its group.  For KV tiles of 128 keys:
//
//   S   = Q_tile[128 x D] . K_tile^T           (TMEM, 128 fp32 columns, 2 buffers)
//   row r: mask keys past its position, running max m, p = 2^(s - m)
//   P   [128 x 128 keys] as two storage-type terms hi + lo, written to tensor
//       memory over the S columns it replaces
//   O  += P . V_tile   [128 x D]               (P from TMEM, V from shared memory,
//                                              O accumulated in TMEM)
//
// The running max is raised only when a tile's max exceeds it by more than 8
// (a factor 2^8): then O (in TMEM) and the row sum are rescaled by
// 2^(m_old - m_new) before the tile's product; otherwise p may reach 2^8, which
// fp32 sums and the hi + lo terms carry exactly as well.  The final division by
// the row sum makes the result independent of which max was used.
//
// Roles (576 threads): warp 0 issues TMA (Q once, then K(t) before V(t-1) into a
// ring of 32 KB stages), warp 1 issues tcgen05.mma, warps 2-17 run the softmax,
// four warps per row (32 keys and 32 output columns each).  Every wait is bounded.
#include <math_constants.h>

#include <mutex>

#include "pa_common.cuh"
#include "pa_sm100.cuh"

namespace pa {
namespace {

using namespace sm100;

constexpr int kD = 128;
constexpr int kRows = 128;                  // query rows per tile (M)
constexpr int kKeys = 128;                  // keys per KV tile (N of S, K of P.V)
constexpr int kSlab = 128 * 128;            // 128 rows x 128 bytes
constexpr int kTile = 2 * kSlab;            // 128 rows x 256 bytes (D = 128, 16-bit)
constexpr int kQOff = 0;
constexpr int kRingOff = kQOff + kTile;
constexpr int kSoftWarps = 16;               // four per TMEM lane quarter
constexpr int kThreads = 64 + 32 * kSoftWarps;  // producer, MMA, softmax
constexpr float kRescaleLog2 = 8.f;          // raise the running max only past this
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr int kSmemBudget = 232448 - 1024;  // per-block limit minus alignment slack
constexpr int kTailBytes = 8192;
constexpr int kStages = (kSmemBudget - kRingOff - kTailBytes) / kTile > 6
                            ? 6 : (kSmemBudget - kRingOff - kTailBytes) / kTile;
// TMEM: S/P[2] at columns 0 / 128 (P overwrites the S it was computed from),
// O at 256 (allocation is a power of two)
constexpr uint32_t kTmemCols = 512;

struct Tail {
  uint64_t full[kStages], empty[kStages];
  uint64_t q_full;
  uint64_t s_full[2], s_empty[2];
  uint64_t p_full;
  uint64_t pv_done;
  uint64_t drain;
  uint64_t red_bar[2][4], sum_bar[4];          // the four warps of a lane quarter
  float red_max[2][4][128];                    // [tile parity][column quarter][row]
  float red_sum[4][128];
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
  int B, total_q, Hq, Hkv, bs, max_blocks, num_blocks, max_q_len, n_qtiles;
  float scale_log2;
  int32_t* status_dev;
};

// Ring positions in the MMA's consumption order K(0), K(1), V(0), K(2), V(1), ...,
// V(last): S(t) is issued before P(t-1).V(t-1) so the softmax of tile t can start
// while the previous product runs.
__device__ __forceinline__ int pos_k(int t) { return t == 0 ? 0 : 2 * t - 1; }
__device__ __forceinline__ int pos_v(int t, int last) { return t < last ? 2 * t + 2 : 2 * t + 1; }

template <int DT, int G>
__global__ void __launch_bounds__(kThreads, 1)
prefill_tc_kernel(const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_q, const PrefillParams p) {
  constexpr int TQ = kRows / G;                 // query tokens per tile
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
  Tail* tl = reinterpret_cast<Tail*>(smem + kTailOff);
  volatile int* abort_flag = &tl->abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  allow_next_grid();
  wait_prior_grid();               // q, the pools and the tables may come from the previous kernel
  // blockIdx.x walks the query tiles of one (sequence, KV head), longest causal
  // work first, so the CTAs resident together read the same K/V from L2
  const int b = blockIdx.y / p.Hkv, h = blockIdx.y - b * p.Hkv;
  const int qt = p.n_qtiles - 1 - (int)blockIdx.x;
  const int qs = p.q_start[b];
  const int n = p.q_start[b + 1] - qs;
  const int L = p.seq_lens[b];
  if (n < 0 || n > L || n > p.max_q_len || L > p.max_blocks * p.bs || qs < 0 ||
      qs + n > p.total_q) {
    if (threadIdx.x == 0 && h == 0 && qt == 0) report(p.status_dev, PA_ERR_BAD_BLOCK_ID);
    return;
  }
  const int q0 = qt * TQ;
  if (q0 >= n) return;                          // uniform: no rows in this tile
  const int pos_last = L - n + min(q0 + TQ, n) - 1;
  const int n_kv = pos_last / kKeys + 1;        // KV tiles covering keys 0 .. pos_last
  const int last = n_kv - 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&tl->full[s], 1);
      mbar_init(&tl->empty[s], 1);
    }
    mbar_init(&tl->q_full, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&tl->s_full[i], 1);
      mbar_init(&tl->s_empty[i], 1);
      for (int w = 0; w < 4; ++w) mbar_init(&tl->red_bar[i][w], 4);
    }
    for (int w = 0; w < 4; ++w) mbar_init(&tl->sum_bar[w], 4);
    mbar_init(&tl->p_full, kSoftWarps);
    mbar_init(&tl->pv_done, 1);
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
    if (lane == 0) {
      mbar_arrive_expect_tx(&tl->q_full, kTile);
      tma_load_3d_hint(smem + kQOff, &tm_q, &tl->q_full, 0, h * G, qs + q0, q_policy);
      tma_load_3d_hint(smem + kQOff + kSlab, &tm_q, &tl->q_full, 64, h * G, qs + q0, q_policy);
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
    for (int t = 0; t <= last && ok; ++t) {
      ok = issue(&tm_k, t);
      if (ok && t > 0) ok = issue(&tm_v, t - 1);
    }
    if (ok) ok = issue(&tm_v, last);
    if (*abort_flag && lane == 0) {            // let copies in flight land before exit
      for (int s = 0; s < kStages; ++s)
        if (issued[s] >= 0) mbar_wait_drain(&tl->full[s], issued[s], kWaitNs);
      if (q_issued) mbar_wait_drain(&tl->q_full, 0, kWaitNs);
    }
  }
  else if (warp == 1) {
    // -------------------------------------------------------------- MMA issue --
    constexpr uint32_t ab = DT == PA_BFLOAT16 ? 1u : 0u;
    constexpr uint32_t idesc_s = idesc_f16(ab, 0, 0, kRows, kKeys);   // Q, K both K-major
    constexpr uint32_t idesc_o = idesc_f16(ab, 0, 1, kRows, kD);      // P (TMEM), V MN-major
    const uint32_t ring = smem_addr(smem + kRingOff);
    const uint32_t qaddr = smem_addr(smem + kQOff);
    bool ok = true, committed = false;
    // O += (P_hi + P_lo) . V_u.  P sits in S buffer u & 1: 16-key group k occupies
    // columns 16k .. 16k+7 (hi) and 16k+8 .. 16k+15 (lo).
    auto issue_pv = [&](int u) -> bool {
      const int vs = pos_v(u, last) % kStages, vph = (pos_v(u, last) / kStages) & 1;
      if (!mbar_wait(&tl->full[vs], vph, abort_flag, kWaitNs)) return false;
      if (!mbar_wait(&tl->p_full, u & 1, abort_flag, kWaitNs)) return false;
      tc_fence_after();
      const uint32_t vaddr = ring + vs * kTile;
      const uint32_t pcol = tmem + (u & 1) * kKeys;
#pragma unroll
      for (int kk = 0; kk < kKeys / 16; ++kk) {
        const uint64_t bd = smem_desc_sw128(vaddr + kk * 16 * 128, kSlab, 1024);
#pragma unroll
        for (int term = 0; term < 2; ++term)
          mma_f16_ts(tmem + 256, pcol + kk * 16 + term * 8, bd, idesc_o, (u | kk | term) != 0);
      }
      mma_commit(&tl->empty[vs]);
      mma_commit(&tl->s_empty[u & 1]);      // S/P buffer free for S(u + 2)
      mma_commit(&tl->pv_done);
      return true;
    };
    if (lane == 0) {
      ok = mbar_wait(&tl->q_full, 0, abort_flag, kWaitNs);
      for (int t = 0; t <= last && ok; ++t) {
        const int ks = pos_k(t) % kStages, kph = (pos_k(t) / kStages) & 1;
        ok = mbar_wait(&tl->full[ks], kph, abort_flag, kWaitNs) &&
             mbar_wait(&tl->s_empty[t & 1], ((t >> 1) & 1) ^ 1, abort_flag, kWaitNs);
        if (!ok) break;
        tc_fence_after();
        const uint32_t kaddr = ring + ks * kTile;
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kSlab + (kk & 3) * 32;
          mma_f16(tmem + (t & 1) * kKeys, smem_desc_sw128(qaddr + off, 16, 1024),
                  smem_desc_sw128(kaddr + off, 16, 1024), idesc_s, kk > 0);
        }
        mma_commit(&tl->empty[ks]);
        mma_commit(&tl->s_full[t & 1]);
        committed = true;
        if (t > 0) ok = issue_pv(t - 1);
      }
      if (ok) ok = issue_pv(last);
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
    // Four warps per TMEM lane quarter; column quarter j takes keys 32j .. 32j+31
    // of each S tile and output columns 32j .. 32j+31; the four exchange row maxima.
    const int wq = warp & 3;                     // TMEM lane quarter of this warp
    const int j = (warp - 2) >> 2;               // column quarter
    const int r = wq * 32 + lane;                // tile row = query token r / G, head r % G
    const int cb = j * 32;
    const uint32_t lane_base = (uint32_t)(wq * 32) << 16;
    const int i = q0 + r / G;                    // query token within the sequence's queries
    const bool row_valid = i < n;
    const int pos = row_valid ? L - n + i : -1;  // keys 0 .. pos are visible
    const uint32_t ocol = tmem + lane_base + 256 + cb;
    float m_run = -CUDART_INF_F, l_run = 0.f;
    bool ok = true;
    auto wait_all = [&](uint64_t* bar, int parity) -> bool {
      const bool w = mbar_wait(bar, parity, abort_flag, kWaitNs);
      return __all_sync(0xFFFFFFFFu, w);
    };
    const float sl2 = p.scale_log2;
    for (int t = 0; t <= last && ok; ++t) {
      const int sb = t & 1;
      if (!wait_all(&tl->s_full[sb], (t >> 1) & 1)) { ok = false; break; }
      tc_fence_after();
      const int kc = t * kKeys + cb;             // key of this thread's first column
      const bool partial = kc + 31 > pos;        // some of its keys lie past the row
      const uint32_t sadr = tmem + lane_base + sb * kKeys + cb;
      float sv[32];
      tmem_ld32(sadr, sv);
      // the tile's maximum of the visible raw scores (scale > 0 commutes with max)
      float mt = -CUDART_INF_F;
      if (!partial) {
#pragma unroll
        for (int e = 0; e < 32; ++e) mt = fmaxf(mt, sv[e]);
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) mt = fmaxf(mt, kc + e <= pos ? sv[e] : -CUDART_INF_F);
      }
      {   // over the row's four column quarters
        const int rb = t & 1;
        tl->red_max[rb][j][r] = mt;
        __syncwarp();
        if (lane == 0) mbar_arrive(&tl->red_bar[rb][wq]);
        if (!wait_all(&tl->red_bar[rb][wq], (t >> 1) & 1)) { ok = false; break; }
        mt = fmaxf(fmaxf(tl->red_max[rb][0][r], tl->red_max[rb][1][r]),
                   fmaxf(tl->red_max[rb][2][r], tl->red_max[rb][3][r]));
      }
      const float m_tile = mt * sl2;
      // Rows whose max grows by more than 2^8 raise it; O (complete up to tile
      // t-1) and l scale by 2^(m_old - m_new).  TMEM access is warp-wide, so the
      // warp rescales when any of its rows needs it (the others by 1).
      const bool raise = m_run != -CUDART_INF_F && m_tile > m_run + kRescaleLog2;
      if (__any_sync(0xFFFFFFFFu, raise)) {
        const float alpha = raise ? ex2_approx(m_run - m_tile) : 1.f;
        if (!wait_all(&tl->pv_done, (t - 1) & 1)) { ok = false; break; }
        tc_fence_after();
        float o[32];
        tmem_ld32(ocol, o);
        uint32_t ow[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) ow[e] = __float_as_uint(o[e] * alpha);
        tmem_st32(ocol, ow);
        l_run *= alpha;
      }
      if (m_run == -CUDART_INF_F || raise) m_run = m_tile;   // first visible tile, or raised
      const float neg_m = m_run == -CUDART_INF_F ? 0.f : -m_run;
      // p = 2^(s * scale * log2 e - m), written back over the S columns as
      // hi / lo storage-type pairs (see issue_pv)
      float ls = 0.f;
#pragma unroll
      for (int g = 0; g < 32; g += 16) {         // one 16-key group: 8 hi words, 8 lo words
        uint32_t pw[16];
#pragma unroll
        for (int e = 0; e < 16; e += 2) {
          float pa_ = ex2_approx(fmaf(sv[g + e], sl2, neg_m));
          float pb_ = ex2_approx(fmaf(sv[g + e + 1], sl2, neg_m));
          if (partial) {
            pa_ = kc + g + e <= pos ? pa_ : 0.f;
            pb_ = kc + g + e + 1 <= pos ? pb_ : 0.f;
          }
          ls += pa_ + pb_;
          if (DT == PA_BFLOAT16) {
            // hi = the top 16 bits (truncation), lo = the rest rounded: hi + lo
            // carries ~16 significant bits either way
            const uint32_t ua = __float_as_uint(pa_), ub = __float_as_uint(pb_);
            pw[e >> 1] = __byte_perm(ua, ub, 0x7632);
            pw[8 + (e >> 1)] = narrow2<DT>(pa_ - __uint_as_float(ua & 0xFFFF0000u),
                                           pb_ - __uint_as_float(ub & 0xFFFF0000u));
          } else {
            const uint32_t h2 = narrow2<DT>(pa_, pb_);
            const float2 hf = widen2<DT>(h2);
            pw[e >> 1] = h2;
            pw[8 + (e >> 1)] = narrow2<DT>(pa_ - hf.x, pb_ - hf.y);
          }
        }
        tmem_st16(sadr + g, pw);                 // over S columns already read
      }
      l_run += ls;
      // keys at or past L: their V rows hold whatever the slot or an earlier tile
      // left (0 * NaN must not reach O), so zero them before P.V reads the tile
      const int k0 = t * kKeys;
      if (k0 + kKeys > L) {
        const int u = pos_v(t, last);
        const int vs = u % kStages, vph = (u / kStages) & 1;
        if (!wait_all(&tl->full[vs], vph)) { ok = false; break; }
        if (k0 + r >= L) {                       // V row r: this warp zeroes 32 of its 128 columns
          uint4* v0 = reinterpret_cast<uint4*>(smem + kRingOff + vs * kTile + (j >> 1) * kSlab +
                                               r * 128 + (j & 1) * 64);
#pragma unroll
          for (int e = 0; e < 4; ++e) v0[e] = make_uint4(0, 0, 0, 0);
        }
      }
      // consume P.V(t-1)'s completion before P(t) is released, so the barrier
      // cannot run two phases ahead of any waiting warp
      if (t > 0 && !wait_all(&tl->pv_done, (t - 1) & 1)) { ok = false; break; }
      tc_fence_before();
      fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tl->p_full);
    }
    if (ok) ok = wait_all(&tl->pv_done, last & 1);
    if (ok) {   // row sum over the four column quarters
      tl->red_sum[j][r] = l_run;
      __syncwarp();
      if (lane == 0) mbar_arrive(&tl->sum_bar[wq]);
      ok = wait_all(&tl->sum_bar[wq], 0);
    }
    if (!ok) {
      if (lane == 0) set_abort();
    } else {
      tc_fence_after();
      float o[32];
      tmem_ld32(ocol, o);
      if (row_valid) {
        const float inv = 1.f / (tl->red_sum[0][r] + tl->red_sum[1][r] + tl->red_sum[2][r] +
                                 tl->red_sum[3][r]);
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.out) +
                                              ((int64_t)(qs + i) * p.Hq + h * G + r % G) * kD + cb);
#pragma unroll
        for (int c = 0; c < 4; ++c)
          dst[c] = make_uint4(narrow2<DT>(o[8 * c] * inv, o[8 * c + 1] * inv),
                              narrow2<DT>(o[8 * c + 2] * inv, o[8 * c + 3] * inv),
                              narrow2<DT>(o[8 * c + 4] * inv, o[8 * c + 5] * inv),
                              narrow2<DT>(o[8 * c + 6] * inv, o[8 * c + 7] * inv));
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
  const dim3 grid((unsigned)p.n_qtiles, (unsigned)(p.Hkv * p.B));
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
    case 4: return launch_g<DT, 4>(p, k, v, q, stream);
    case 8: return launch_g<DT, 8>(p, k, v, q, stream);
    case 16: return launch_g<DT, 16>(p, k, v, q, stream);
    default: return PA_ERR_UNSUPPORTED;
  }
}

bool aligned16(const void* ptr) { return ((uintptr_t)ptr & 15u) == 0; }

}  // namespace
}  // namespace pa

using namespace pa;

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
  if (head_dim != kD || (G != 1 && G != 2 && G != 4 && G != 8 && G != 16) ||
      (block_size != 8 && block_size != 16 && block_size != 32 && block_size != 64) ||
      (dtype != PA_FLOAT16 && dtype != PA_BFLOAT16))
    return PA_ERR_UNSUPPORTED;
  if (num_seqs == 0 || total_q == 0 || max_q_len == 0) return PA_OK;
  if (!out || !q || !k_pool || !v_pool || !block_tables || !seq_lens || !q_start)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(out) || !aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool))
    return PA_ERR_INVALID_ARG;
  if ((int64_t)num_blocks * block_size >= (1ll << 31) ||
      (int64_t)total_q * num_q_heads >= (1ll << 31))
    return PA_ERR_INVALID_ARG;
  const int TQ = kRows / G;
  const int64_t n_qtiles = ((int64_t)max_q_len + TQ - 1) / TQ;
  if ((int64_t)num_seqs * num_kv_heads > 65535) return PA_ERR_INVALID_ARG;   // grid y
  EncodeTiledFn enc = encode_fn();
  if (!enc) return PA_ERR_UNSUPPORTED;

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
  p.n_qtiles = (int)n_qtiles;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status_dev = status_dev;
  return dtype == PA_BFLOAT16 ? launch_dt<PA_BFLOAT16>(G, p, tk, tv, tq, stream)
                              : launch_dt<PA_FLOAT16>(G, p, tk, tv, tq, stream);
}
