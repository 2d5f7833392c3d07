// Prefill forward: exact attention, one fused kernel per call, sm_103a.
//
// Schedule (the FA-2 loop of "FlashAttention and GPU Data Movement", section 2): one thread
// block owns one 128-row query tile of one (batch, query head); it streams the 128-key K/V
// tiles of the matching key/value head through shared memory and keeps the online-softmax
// state on chip, writing O and the log-sum-exp once at the end.
//
// Roles inside a thread block (384 threads):
//   warps 0-7  softmax, two warpgroups taking alternate K/V tiles (0-3 the even ones, 4-7 the
//              odd ones); thread r of a warpgroup owns query row r.  Reads S_j from tensor
//              memory, applies the scale, the causal/ragged mask and the online-softmax update
//              ("FlashAttention and GPU Data Movement", section 3.1), writes P_j back to tensor
//              memory as 16-bit pairs, rescales the accumulator when the row maximum moved, and
//              runs the epilogue O = a / l, L = m + ln l (each warpgroup half of the columns).
//   warp 8     TMA producer: Q once, then K_j into a STAGES-deep ring.
//   warp 11    TMA producer: V_j into its own STAGES-deep ring.
//   warp 9     tcgen05 issuer of S_j = Q K_j^T (both operands in shared memory, fp32 result in
//              tensor memory); allocates and frees the 512 tensor-memory columns.
//   warp 10    tcgen05 issuer of O += P_j V_j (P from tensor memory, V from shared memory, fp32
//              accumulator in tensor memory).
// Tensor memory: S buffers at columns 0 and 128 (double-buffered so Q K_{j+1}^T runs while the
// softmax of tile j runs), the output accumulator at column 256, two P buffers after it.  A
// softmax releases its S buffer as soon as it has read it, so the score MMAs run ahead.
//
// Departures from the pages' kernels (prior art for A100/H100/B200): accumulators live in tensor
// memory instead of registers, P is handed to the second MMA through tensor memory instead of
// shared memory or registers, exponentials are base 2 with the scale folded into one FMA, and the
// accumulator is rescaled only when a row maximum rises by more than 2^8 (the final division uses
// the same stale maximum in l, so the result is unchanged: "FlashAttention Explained", section on
// FlashAttention-4, conditional rescaling).
#include <cstdio>

#include "internal.h"
#include "ptx.cuh"

namespace attn {

// Optional per-tile timestamps for schedule analysis; compiled in only when ATTN_FWD_TRACE is
// defined (never in the library build).
#ifdef ATTN_FWD_TRACE
__device__ unsigned long long g_fwd_trace[8][80][16];
#define FWD_TRACE(j, ev)                                                                      \
  do {                                                                                        \
    if (trace_slot >= 0 && (j) < 80) {                                                        \
      unsigned long long t_;                                                                  \
      asm volatile("mov.u64 %0, %%clock64;" : "=l"(t_));                                      \
      g_fwd_trace[trace_slot][(j)][(ev)] = t_;                                                \
    }                                                                                         \
  } while (0)
#else
#define FWD_TRACE(j, ev) \
  do {                   \
  } while (0)
#endif

constexpr int kBlockM = 128;
constexpr int kBlockN = 128;
constexpr int kFwdThreads = 384;  // warps 0-7 softmax, 8 and 11 TMA, 9-10 MMA issue
constexpr int kSoftmaxThreads = 128;  // one softmax warpgroup (thread = query row)
constexpr int kProducerWarp = 8, kQkWarp = 9, kPvWarp = 10, kVProducerWarp = 11;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256;
// P buffers follow O: columns 256 + d and 256 + d + 64 (16-bit pairs, 64 columns each).
template <int D>
struct PCols {
  static constexpr uint32_t kP0 = kColO + D, kP1 = kColO + D + 64;
  static_assert(kP1 + 64 <= kTmemCols, "tensor memory budget");
};
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale only if the max rises by > 2^8
constexpr uint32_t kSubTile = 128 * 128;   // bytes of one 64-column, 128-row swizzled sub-tile
constexpr uint64_t kDrainLimitNs = 100000000ull;

struct FwdParams {
  float* lse;
  int* status;
  int Hq, Hkv, N_q, N_kv;
  int n_qtiles, group, causal;
  float sl2;  // scale * log2(e)
};

template <int D, int STAGES>
struct FwdLayout {
  static constexpr uint32_t kQBytes = kBlockM * D * 2;
  static constexpr uint32_t kKVBytes = kBlockN * D * 2;
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK = kQ + kQBytes;
  static constexpr uint32_t kV = kK + STAGES * kKVBytes;
  static constexpr uint32_t kBar = kV + STAGES * kKVBytes;
  // q_full, k_full[S], v_full[S], k_empty[S], v_empty[S], s_full[2], s_free[2], p_ready[2],
  // o_done[2], drain, m_ready[2]  (the [2] barriers belong to the two S and P buffers, i.e.
  // to the even and the odd tiles)
  static constexpr uint32_t kNumBars = 1 + 4 * STAGES + 2 + 2 + 2 + 2 + 1 + 2;
  static constexpr uint32_t kMisc = kBar + kNumBars * 8;  // tmem slot, abort flag
  // running row maxima handed from one softmax warpgroup to the other: [tile parity][row], and
  // the odd warpgroup's row sums for the epilogue: [row]
  static constexpr uint32_t kMrow = kMisc + 16;
  static constexpr uint32_t kLsum = kMrow + 2 * kBlockM * 4;
  static constexpr uint32_t kBytes = kLsum + kBlockM * 4 + 1024;  // + alignment slack
  static_assert(kBytes <= 232448, "shared memory per block");
};

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          int* status) {
  const bool ok = wait_bounded(bar, parity, abort, status);
  return __all_sync(0xffffffffu, ok);
}

template <int D, bool BF16, int STAGES>
__global__ void __launch_bounds__(kFwdThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_o, const FwdParams p) {
  using L = FwdLayout<D, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);

  const uint32_t sQ = base + L::kQ;
  const uint32_t sK = base + L::kK;
  const uint32_t sV = base + L::kV;
  const uint32_t bars = base + L::kBar;
  const uint32_t bar_q = bars;
#define BAR_K(s) (bars + 8u * (1u + (s)))
#define BAR_V(s) (bars + 8u * (1u + STAGES + (s)))
#define BAR_KE(s) (bars + 8u * (1u + 2u * STAGES + (s)))
#define BAR_VE(s) (bars + 8u * (1u + 3u * STAGES + (s)))
#define BAR_S(b) (bars + 8u * (1u + 4u * STAGES + (b)))
#define BAR_SF(b) (bars + 8u * (3u + 4u * STAGES + (b)))
#define BAR_P(b) (bars + 8u * (5u + 4u * STAGES + (b)))
#define BAR_O(b) (bars + 8u * (7u + 4u * STAGES + (b)))
  const uint32_t bar_drain = bars + 8u * (9u + 4u * STAGES);
#define BAR_M(b) (bars + 8u * (10u + 4u * STAGES + (b)))
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L::kMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Work item: query heads of one key/value head are adjacent and, inside a head, the
  // query tiles run longest first (they carry the most K/V tiles under the causal mask).
  const int bh = blockIdx.x / p.n_qtiles;
  const int qt = p.n_qtiles - 1 - static_cast<int>(blockIdx.x % p.n_qtiles);
  const int h = bh % p.Hq;
  const int b = bh / p.Hq;
  const int kv_plane = b * p.Hkv + h / p.group;
  const int q0 = qt * kBlockM;
  int n_tiles, first_masked;
  kv_tile_range(qt, kBlockM, kBlockN, p.N_q, p.N_kv, p.causal, n_tiles, first_masked);
#ifdef ATTN_FWD_TRACE
  int trace_slot = -1;
  {
    const int ids[8] = {0, 1, 2, 3, 600, 1200, 2000, 4000};
    for (int i = 0; i < 8; ++i)
      if (static_cast<int>(blockIdx.x) == ids[i]) trace_slot = i;
  }
#endif

  if (threadIdx.x == 0) FWD_TRACE(79, 0);
  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(BAR_K(s), 1);
      mbar_init(BAR_V(s), 1);
      mbar_init(BAR_KE(s), 1);
      mbar_init(BAR_VE(s), 1);
    }
    mbar_init(BAR_S(0), 1);
    mbar_init(BAR_S(1), 1);
    mbar_init(BAR_SF(0), kSoftmaxThreads);
    mbar_init(BAR_SF(1), kSoftmaxThreads);
    mbar_init(BAR_P(0), kSoftmaxThreads);
    mbar_init(BAR_P(1), kSoftmaxThreads);
    mbar_init(BAR_O(0), 1);
    mbar_init(BAR_O(1), 1);
    mbar_init(bar_drain, 2);  // one commit from each issuer
    mbar_init(BAR_M(0), kSoftmaxThreads);
    mbar_init(BAR_M(1), kSoftmaxThreads);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kQkWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kProducerWarp || warp == kVProducerWarp) {
    // ----------------------------------------------------------------- TMA producers
    // Warp 8 loads Q and the K ring, warp 11 the V ring (separate warps, so neither waits on
    // the other's spin): a K slot is refilled as soon as its Q K^T finished, a V slot once its
    // P V finished.
    if (lane == 0 && n_tiles > 0) {
      const bool is_k = (warp == kProducerWarp);
      const CUtensorMap* tm = is_k ? &tm_k : &tm_v;
      const uint32_t ring = is_k ? sK : sV;
      if (is_k) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        mbar_arrive_expect_tx(bar_q, L::kQBytes);
#pragma unroll
        for (int sub = 0; sub < D / 64; ++sub)
          tma_load_3d(sQ + sub * kSubTile, &tm_q, bar_q, sub * 64, q0, bh);
      } else {
        prefetch_tmap(&tm_v);
      }
      int issued = 0;
      for (int j = 0; j < n_tiles; ++j) {
        const int s = j % STAGES;
        const uint32_t empty = is_k ? BAR_KE(s) : BAR_VE(s);
        const uint32_t full = is_k ? BAR_K(s) : BAR_V(s);
        if (j >= STAGES && !wait_bounded(empty, ((j / STAGES) - 1) & 1, abort_flag, p.status))
          break;
        mbar_arrive_expect_tx(full, L::kKVBytes);
#pragma unroll
        for (int sub = 0; sub < D / 64; ++sub)
          tma_load_3d(ring + s * L::kKVBytes + sub * kSubTile, tm, full, sub * 64, j * kBlockN,
                      kv_plane);
        issued = j + 1;
      }
      // Every load this thread issued lands before the block may exit.
      if (is_k) wait_bounded(bar_q, 0, nullptr, p.status, kDrainLimitNs);
      for (int j = (issued > STAGES ? issued - STAGES : 0); j < issued; ++j)
        wait_bounded(is_k ? BAR_K(j % STAGES) : BAR_V(j % STAGES), (j / STAGES) & 1, nullptr,
                     p.status, kDrainLimitNs);
    }
  } else if (warp == kQkWarp || warp == kPvWarp) {
    // ----------------------------------------------------------------- tcgen05 issuers
    // Warp 5 issues the score MMAs, warp 6 the P V MMAs.  The two streams touch disjoint tensor
    // memory (S buffers / O and P buffers) and disjoint shared memory (Q, K / V), so they need no
    // ordering between them beyond the barriers below, and each issuer's waits overlap the other
    // issuer's MMAs.
    if (lane == 0 && n_tiles > 0) {
      const bool qk_issuer = (warp == kQkWarp);
      constexpr uint32_t idesc_qk = make_idesc_f16(BF16, kBlockM, kBlockN, false);
      constexpr uint32_t idesc_pv = make_idesc_f16(BF16, kBlockM, D, true);
      bool ok = qk_issuer ? wait_bounded(bar_q, 0, abort_flag, p.status) : true;
      // S_t = Q K_t^T into S buffer t % 2, once the softmax of tile t - 2 has read that buffer.
      auto issue_qk = [&](int t) -> bool {
        FWD_TRACE(t, 8);
        const int s = t % STAGES;
        if (t >= 2 && !wait_bounded(BAR_SF(t & 1), ((t >> 1) - 1) & 1, abort_flag, p.status))
          return false;
        if (!wait_bounded(BAR_K(s), (t / STAGES) & 1, abort_flag, p.status)) return false;
        FWD_TRACE(t, 9);
        tc_fence_after();
        const uint32_t s_col = tmem + ((t & 1) ? kColS1 : kColS0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          // Q and K are K-major (d contiguous): 16 elements = 32 bytes per MMA inside the
          // 128-byte swizzle row; SBO = 1024 B between 8-row groups.
          const uint32_t off = (kk >> 2) * kSubTile + (kk & 3) * 32;
          const uint64_t adesc = make_sdesc_sw128(sQ + off, 16, 1024);
          const uint64_t bdesc = make_sdesc_sw128(sK + s * L::kKVBytes + off, 16, 1024);
          mma_ss(s_col, adesc, bdesc, idesc_qk, kk > 0 ? 1u : 0u);
        }
        mma_commit(BAR_S(t & 1));
        mma_commit(BAR_KE(s));  // K slot free
        FWD_TRACE(t, 10);
        return true;
      };
      // O += P_t V_t (P_t in P buffer t % 2, V_t in ring slot t % STAGES).
      auto issue_pv = [&](int t) -> bool {
        FWD_TRACE(t, 11);
        if (!wait_bounded(BAR_P(t & 1), (t >> 1) & 1, abort_flag, p.status)) return false;
        FWD_TRACE(t, 12);
        const int s = t % STAGES;
        if (!wait_bounded(BAR_V(s), (t / STAGES) & 1, abort_flag, p.status)) return false;
        FWD_TRACE(t, 13);
        tc_fence_after();
        const uint32_t p_col = tmem + ((t & 1) ? PCols<D>::kP1 : PCols<D>::kP0);
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk) {
          // V is [keys, d] with d contiguous: the B operand is MN-major.  16 keys per MMA
          // (two 8-row groups, SBO = 1024 B apart); the two 64-column halves of d are
          // separate swizzled sub-tiles (LBO = one sub-tile).
          const uint64_t bdesc = make_sdesc_sw128(sV + s * L::kKVBytes + kk * 16 * 128,
                                                  kSubTile, 1024);
          mma_ts(tmem + kColO, p_col + kk * 8, bdesc, idesc_pv, (t > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(BAR_O(t & 1));
        mma_commit(BAR_VE(s));  // V slot free
        FWD_TRACE(t, 14);
        return true;
      };
      // The score issuer runs up to two tiles ahead of the softmax (two S buffers); the P V
      // issuer follows the softmax tile by tile.
      for (int j = 0; ok && j < n_tiles; ++j) ok = qk_issuer ? issue_qk(j) : issue_pv(j);
      // Every MMA this thread issued completes before the block frees tensor memory.
      mma_commit(bar_drain);
      wait_bounded(bar_drain, 0, nullptr, p.status, kDrainLimitNs);
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------------------- softmax + epilogue
    // Two warpgroups share the rows: warps 0-3 take the even K/V tiles (S0, P0), warps 4-7 the
    // odd ones (S1, P1); in both, thread r owns query row r and warp % 4 is its tensor-memory
    // lane quarter.  The running maximum is the only state carried from tile to tile: the
    // warpgroup of tile j publishes m_j as soon as its row maxima are known (BAR_M), and the
    // other warpgroup, on tile j + 1, waits for it before its exponentials.  Each warpgroup keeps
    // its own partial row sum, rescaled whenever the maximum moves; the two are added at the end.
    const int wg = warp >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const bool tracer = (threadIdx.x & 127) == 0;
    const uint32_t row_tmem = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const int row = q0 + r;
    const int off = p.N_kv - p.N_q;
    const float sl2 = p.sl2;
    float* mrow = reinterpret_cast<float*>(gbase + L::kMrow);  // [tile parity][row]
    float* lsum = reinterpret_cast<float*>(gbase + L::kLsum);  // [row]
    const uint32_t s_col = wg ? kColS1 : kColS0;
    const uint32_t p_col = wg ? PCols<D>::kP1 : PCols<D>::kP0;
    float m_own = -INFINITY;  // maximum (log2 units) this warpgroup's partial sum refers to
    float l = 0.0f;           // this warpgroup's partial sum of 2^(x - m_own)
    bool ok = true;
    bool s_ready = false;  // S of this warpgroup's next tile already seen complete
    for (int j = wg; j < n_tiles; j += 2) {
      const int u = j >> 1;  // use index of this warpgroup's S and P buffers
      if (tracer) FWD_TRACE(j, 0);
      if (!__all_sync(0xffffffffu, s_ready) &&
          !warp_wait(BAR_S(wg), u & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      if (tracer) FWD_TRACE(j, 1);
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(row_tmem + s_col + c * 32, sr[c]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(BAR_SF(wg));  // S buffer free for Q K_{j+2}^T
      if (tracer) FWD_TRACE(j, 2);
      // Early, non-blocking test of the barrier needed before P is written (P V_{j-2} read
      // this P buffer); its latency hides under the work below.
      const bool p_free = (j < 2) || mbar_test_wait(BAR_O(wg), (u - 1) & 1);
      float x[kBlockN];
#pragma unroll
      for (int c = 0; c < 4; ++c)
#pragma unroll
        for (int e = 0; e < 32; ++e) x[c * 32 + e] = __uint_as_float(sr[c][e]);
      if (j >= first_masked) {
        int lim = p.causal ? row + off : p.N_kv - 1;  // last visible key of this row
        if (lim > p.N_kv - 1) lim = p.N_kv - 1;
        const int rel = lim - j * kBlockN;
#pragma unroll
        for (int c = 0; c < kBlockN; ++c)
          if (c > rel) x[c] = -INFINITY;
      }
      // Row maximum of the tile: three-input max, eight independent chains.
      float mx[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx[e] = fmaxf(x[e], x[8 + e]);
#pragma unroll
      for (int c = 16; c < kBlockN; c += 16)
#pragma unroll
        for (int e = 0; e < 8; ++e) mx[e] = max3f(mx[e], x[c + e], x[c + 8 + e]);
      const float tile_max = max3f(max3f(mx[0], mx[1], mx[2]), max3f(mx[3], mx[4], mx[5]),
                                   fmaxf(mx[6], mx[7]));
      // Running maximum after tile j - 1, from the other warpgroup.
      float m_prev = -INFINITY;
      if (j > 0) {
        if (!warp_wait(BAR_M(wg ^ 1), ((j - 1) >> 1) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        m_prev = mrow[(wg ^ 1) * kBlockM + r];
      }
      // The maximum moves only when it rises by more than 2^8 (also for the first finite one).
      float m_j = m_prev;
      float alpha = 1.0f;  // rescale of the accumulator O for this tile
      const float m_new = fmaxf(m_prev, tile_max * sl2);
      if (m_new - m_prev > kRescaleThreshold) {
        alpha = ex2(m_prev - m_new);
        m_j = m_new;
      }
      mrow[wg * kBlockM + r] = m_j;
      mbar_arrive(BAR_M(wg));  // m_j published for tile j + 1
      if (m_j != m_own) {
        l = (m_own == -INFINITY) ? 0.0f : l * ex2(m_own - m_j);
        m_own = m_j;
      }
      const float neg_mu = (m_j == -INFINITY) ? 0.0f : -m_j;
      // p = 2^(x * scale * log2(e) - m): one packed FMA per pair of scores, MUFU ex2, a packed
      // add into four pair-accumulators for the row sum, and the 16-bit pack for P.
      float ps[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      uint32_t pk[2][32];
#pragma unroll
      for (int c = 0; c < kBlockN; c += 2) {
        float a0, a1;
        fma2(a0, a1, x[c], x[c + 1], sl2, sl2, neg_mu, neg_mu);
        const float p0 = ex2(a0);
        const float p1 = ex2(a1);
        const int k2 = ((c >> 1) & 3) * 2;
        add2(ps[k2], ps[k2 + 1], p0, p1);
        pk[c >> 6][(c >> 1) & 31] = pack2<BF16>(p0, p1);
      }
      l += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
      s_ready = (j + 2 < n_tiles) && mbar_test_wait(BAR_S(wg), (u + 1) & 1);
      if (tracer) FWD_TRACE(j, 3);
      if (j >= 2) {
        if (!__all_sync(0xffffffffu, p_free) &&
            !warp_wait(BAR_O(wg), (u - 1) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();  // order the P store after the MMA that read the buffer
      }
      if (tracer) FWD_TRACE(j, 4);
      tmem_st32(row_tmem + p_col, pk[0]);
      tmem_st32(row_tmem + p_col + 32, pk[1]);
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
        // Rescaling the accumulator needs P V_{j-1} finished; P V_j waits for this tile's
        // p_ready and P V_{j+1} comes after it, so nothing else touches O meanwhile.
        if (!warp_wait(BAR_O(wg ^ 1), ((j - 1) >> 1) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(row_tmem + kColO + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
          tmem_st32(row_tmem + kColO + c * 32, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(BAR_P(wg));
      if (tracer) FWD_TRACE(j, 5);
    }
    // ------------------------------------------------------------- epilogue
    // The final maximum is the one after the last tile; the warpgroup that did not process
    // that tile reads it from the exchange.
    const int last = n_tiles - 1;
    float m_fin = m_own;
    if (ok && n_tiles > 0 && (last & 1) != wg) {
      if (warp_wait(BAR_M(last & 1), (last >> 1) & 1, abort_flag, p.status))
        m_fin = mrow[(last & 1) * kBlockM + r];
      else
        ok = false;
    }
    if (ok && n_tiles > 0) {
      // MMAs complete in issue order: the last P V done means every MMA is done.
      ok = warp_wait(BAR_O(last & 1), (last >> 1) & 1, abort_flag, p.status);
      tc_fence_after();
    }
    // Both partial sums onto the final maximum, then added (the odd warpgroup's through lsum,
    // the total handed back through mrow once nobody reads the maxima any more).
    if (m_own != m_fin) l = (m_own == -INFINITY) ? 0.0f : l * ex2(m_own - m_fin);
    named_bar_sync(1, 2 * kSoftmaxThreads);
    if (wg == 1) lsum[r] = l;
    named_bar_sync(1, 2 * kSoftmaxThreads);
    if (wg == 0) {
      l += lsum[r];
      mrow[r] = l;
    }
    named_bar_sync(1, 2 * kSoftmaxThreads);
    const float l_row = (wg == 0) ? l : mrow[r];
    const bool have = ok && n_tiles > 0;
    const float inv_l = (l_row > 0.0f) ? 1.0f / l_row : 0.0f;
    // Each warpgroup normalises and stores half of the output columns.
    if (have) {
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        uint32_t o[32];
        tmem_ld32(row_tmem + kColO + wg * (D / 2) + c * 32, o);
        tmem_wait_ld();
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint4 w;
          w.x = pack2<BF16>(__uint_as_float(o[q4 * 8 + 0]) * inv_l, __uint_as_float(o[q4 * 8 + 1]) * inv_l);
          w.y = pack2<BF16>(__uint_as_float(o[q4 * 8 + 2]) * inv_l, __uint_as_float(o[q4 * 8 + 3]) * inv_l);
          w.z = pack2<BF16>(__uint_as_float(o[q4 * 8 + 4]) * inv_l, __uint_as_float(o[q4 * 8 + 5]) * inv_l);
          w.w = pack2<BF16>(__uint_as_float(o[q4 * 8 + 6]) * inv_l, __uint_as_float(o[q4 * 8 + 7]) * inv_l);
          const uint32_t chunk = wg * (D / 16) + c * 4 + q4;  // 16-byte chunk of the row
          uint8_t* dst = gbase + L::kQ + (chunk >> 3) * kSubTile + sw128(r, chunk & 7);
          *reinterpret_cast<uint4*>(dst) = w;
        }
      }
    } else if (ok) {
      // No key visible to any row of this tile: O = 0.
      for (int c = 0; c < D / 16; ++c) {
        const int chunk = wg * (D / 16) + c;
        uint8_t* dst = gbase + L::kQ + (chunk >> 3) * kSubTile + sw128(r, chunk & 7);
        *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
      }
    }
    fence_proxy_async_smem();
    named_bar_sync(1, 2 * kSoftmaxThreads);
    if (ok && threadIdx.x == 0 && *abort_flag == 0) {
#pragma unroll
      for (int sub = 0; sub < D / 64; ++sub) tma_store_3d(&tm_o, sQ + sub * kSubTile, sub * 64, q0, bh);
      tma_store_commit();
      tma_store_wait_read0();
    }
    if (ok && wg == 0 && row < p.N_q) {
      const float mu = (m_fin == -INFINITY) ? 0.0f : m_fin;
      p.lse[static_cast<size_t>(bh) * p.N_q + row] =
          (l_row > 0.0f) ? (mu + lg2(l_row)) * 0.69314718055994531f : -INFINITY;
    }
  }
#undef BAR_K
#undef BAR_V
#undef BAR_KE
#undef BAR_VE
#undef BAR_S
#undef BAR_SF
#undef BAR_P
#undef BAR_O
#undef BAR_M
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0) FWD_TRACE(79, 1);
  if (warp == kQkWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// O = 0 and L = -inf for every row (used when there is no key at all).
template <bool BF16>
__global__ void attn_empty_rows_kernel(uint16_t* o, float* lse, size_t rows, int d) {
  const size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
  if (i < rows * d) o[i] = 0;
  if (i < rows) lse[i] = -INFINITY;
}

template <int D, bool BF16, int STAGES>
static int launch_fwd_variant(const FwdArgs& a, cudaStream_t stream) {
  using L = FwdLayout<D, STAGES>;
  CUtensorMap tq, tk, tv, to;
  const uint64_t bhq = static_cast<uint64_t>(a.B) * a.Hq;
  const uint64_t bhk = static_cast<uint64_t>(a.B) * a.Hkv;
  const uint64_t rq = static_cast<uint64_t>(D) * 2, rk = rq;
  if (!make_tmap_3d(&tq, a.q, BF16, D, a.N_q, bhq, rq, rq * a.N_q, 64, kBlockM, 1) ||
      !make_tmap_3d(&tk, a.k, BF16, D, a.N_kv, bhk, rk, rk * a.N_kv, 64, kBlockN, 1) ||
      !make_tmap_3d(&tv, a.v, BF16, D, a.N_kv, bhk, rk, rk * a.N_kv, 64, kBlockN, 1) ||
      !make_tmap_3d(&to, a.o, BF16, D, a.N_q, bhq, rq, rq * a.N_q, 64, kBlockM, 1))
    return -5;
  FwdParams p;
  p.lse = a.lse;
  p.status = device_status_ptr();
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.N_q = a.N_q;
  p.N_kv = a.N_kv;
  p.n_qtiles = (a.N_q + kBlockM - 1) / kBlockM;
  p.group = a.Hq / a.Hkv;
  p.causal = a.causal;
  p.sl2 = a.scale * 1.4426950408889634f;
  if (!p.status) return -5;
  auto kern = attn_fwd_kernel<D, BF16, STAGES>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes) !=
      cudaSuccess)
    return -5;
  const uint64_t blocks = static_cast<uint64_t>(p.n_qtiles) * bhq;
  if (blocks > 0x7fffffffull) return -2;
  kern<<<static_cast<unsigned>(blocks), kFwdThreads, L::kBytes, stream>>>(tq, tk, tv, to, p);
  return cudaGetLastError() == cudaSuccess ? 0 : -5;
}

#ifdef ATTN_FWD_TRACE
}  // namespace attn
extern "C" int attn_fwd_trace_copy(void* dst) {
  return static_cast<int>(cudaMemcpyFromSymbol(dst, attn::g_fwd_trace, sizeof(attn::g_fwd_trace)));
}
namespace attn {
#endif

int launch_attn_fwd(const FwdArgs& a, cudaStream_t stream) {
  if (a.B == 0 || a.N_q == 0) return 0;
  if (a.N_kv == 0) {
    const size_t rows = static_cast<size_t>(a.B) * a.Hq * a.N_q;
    const size_t n = rows * a.d;
    const unsigned blocks = static_cast<unsigned>((n + 255) / 256);
    if (a.bf16)
      attn_empty_rows_kernel<true><<<blocks, 256, 0, stream>>>(static_cast<uint16_t*>(a.o), a.lse, rows, a.d);
    else
      attn_empty_rows_kernel<false><<<blocks, 256, 0, stream>>>(static_cast<uint16_t*>(a.o), a.lse, rows, a.d);
    return cudaGetLastError() == cudaSuccess ? 0 : -5;
  }
  if (a.d == 64)
    return a.bf16 ? launch_fwd_variant<64, true, 4>(a, stream) : launch_fwd_variant<64, false, 4>(a, stream);
  if (a.d == 128)
    return a.bf16 ? launch_fwd_variant<128, true, 3>(a, stream) : launch_fwd_variant<128, false, 3>(a, stream);
  return -2;
}

}  // namespace attn
