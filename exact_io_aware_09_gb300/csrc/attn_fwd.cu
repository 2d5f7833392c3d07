// Prefill forward: exact attention, one fused persistent kernel per call, sm_103a.
//
// Schedule (the FA-2 loop of "FlashAttention and GPU Data Movement", section 2): a work item is
// one 128-row query tile of one (batch, query head); its 128-key K/V tiles stream through shared
// memory and the online-softmax state stays on chip until O and the log-sum-exp are written once
// at the end.  The grid has one block per work item, but only one block fits on an SM: a running
// block takes over the items of blocks that have not started yet (cluster launch control), so
// each SM runs one long-lived block whose pipelines run on from one item into the next — the
// next item's Q/K/V loads and first score MMAs overlap the current item's last tiles and
// epilogue.  Items are taken in launch order: the query heads of one key/value head adjacent (the
// K/V tiles they share stay in L2) and, inside a head, the longest query tiles first (under the
// causal mask a tile's key range grows with its row index), which keeps the tail of the grid short.
//
// Roles inside a thread block (384 threads):
//   warps 0-7  softmax, two warpgroups taking alternate K/V tiles of the block's tile sequence;
//              thread r of a warpgroup owns query row r.  Reads S_j from tensor memory, applies
//              the scale, the causal/ragged mask and the online-softmax update ("FlashAttention
//              and GPU Data Movement", section 3.1), writes P_j back to tensor memory as 16-bit
//              pairs and rescales the accumulator when the row maximum moved.  The warpgroup that
//              ran an item's last tile runs its epilogue O = a / l, L = m + ln l, with the other
//              warpgroup's partial row sum handed over through shared memory.
//   warp 8     work scheduler (cluster launch control) and TMA producer of Q and the K ring.
//   warp 11    TMA producer of the V ring.
//   warp 9     tcgen05 issuer of S_j = Q K_j^T (both operands in shared memory, fp32 result in
//              tensor memory); allocates and frees the 512 tensor-memory columns.
//   warp 10    tcgen05 issuer of O += P_j V_j (P from tensor memory, V from shared memory, fp32
//              accumulator in tensor memory).
// Tensor memory: S buffers at columns 0 and 128 (double-buffered so Q K_{j+1}^T runs while the
// softmax of tile j runs), the output accumulator at column 256, two P buffers after it.  A
// softmax releases its S buffer as soon as it has read it, so the score MMAs run ahead.
//
// Every barrier phase is counted over the block's whole tile sequence (all items), so the rings,
// buffers and hand-offs need no reset between items.
//
// Departures from the pages' kernels (prior art for A100/H100/B200): accumulators live in tensor
// memory instead of registers, P is handed to the second MMA through tensor memory instead of
// shared memory or registers, exponentials are base 2 with the scale folded into one FMA, and the
// accumulator is rescaled only when a row maximum rises by more than 2^8 (the final division uses
// the same stale maximum in l, so the result is unchanged: "FlashAttention Explained", section on
// FlashAttention-4, conditional rescaling).
#include <atomic>
#include <cstdio>

#include "internal.h"
#include "ptx.cuh"

namespace attn {

// Optional per-tile timestamps for schedule analysis; compiled in only when ATTN_FWD_TRACE is
// defined (never in the library build).
#ifdef ATTN_FWD_TRACE
__device__ unsigned long long g_fwd_trace[8][80][28];
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
// Readers of the work-item ring: lane 0 of warps 9, 10, 11 and of each softmax warp.
constexpr uint32_t kItemReaders = 3 + 8;
constexpr uint32_t kTmemCols = 512;
// Registers per thread after the rebalancing at the role split (launched with 168).
constexpr uint32_t kRegsSoftmax = 184, kRegsIssue = 136;
static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsIssue <= kFwdThreads * 168, "register split");
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256;
// P buffers follow O: columns 256 + d and 256 + d + 64 (16-bit pairs, 64 columns each).
template <int D>
struct PCols {
  static constexpr uint32_t kP0 = kColO + D, kP1 = kColO + D + 64;
  static_assert(kP1 + 64 <= kTmemCols, "tensor memory budget");
};
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale only if the max rises by > 2^8
// FP8: P enters the P V product as 2^kPShift8 P in E4M3.  The maximum moves whenever it rises by
// more than 2^kRescaleThreshold8, so P <= 2^3.8 and 2^5 P <= 2^8.8 < 448, inside E4M3's range;
// the row sum carries the same factor, which the epilogue removes.  (A lower threshold keeps
// more of P's small values out of E4M3's subnormal range but makes the rescale of O, which
// waits for the previous P V, frequent: on N(0,1) inputs a warp of 32 rows rescales on 43% of
// its tiles at 2^1 and on 0.3% at 2^3.8.)
constexpr float kRescaleThreshold8 = 3.8f;
constexpr int kPShift8 = 5;
constexpr uint32_t kSubTile = 128 * 128;   // bytes of one 64-column, 128-row swizzled sub-tile
constexpr uint64_t kDrainLimitNs = 100000000ull;

struct FwdParams {
  void* o;
  float* lse;
  int* status;
  int Hq, Hkv, N_q, N_kv;
  int n_qtiles, group, causal;
  int BH;           // batch * Hq
  int head_group;   // query heads walked together, longest query tiles first (see decode_item)
  int window;       // sliding window, keys behind the diagonal (-1: none)
  int n_kvtiles;    // key tiles of the sequence (row length of block_mask)
  const uint8_t* block_mask;  // [query tile][key tile], nonzero = compute; null: every tile
  // FP8 operands: E4M3 block scales of Q [B*Hq][query tile], K [B*Hkv][key tile], V [B*Hkv]
  const float* q_scale;
  const float* k_scale;
  const float* v_scale;
  float sl2;  // scale * log2(e)
};

// Barriers (8 bytes each), in this order after the K/V rings.
enum FwdBar : uint32_t {
  kBarQFull = 0,       // Q tile landed (TMA)
  kBarQEmpty = 1,      // the item's last score MMA finished: Q may be replaced
  kBarS = 2,           // [2] S buffer written (MMA commit)
  kBarSFree = 4,       // [2] S buffer read by the softmax (128 arrivals)
  kBarP = 6,           // [2] P buffer written, O rescaled (128 arrivals)
  kBarO = 8,           // [2] P V of a tile of that parity finished (MMA commit)
  kBarM = 10,          // [2][4] running maximum of a tile of that parity published, one barrier
                       // per warp (lane quarter): its 32 rows are all the partner warp needs
  kBarLFull = 18,      // [2] partial row sum handed to the epilogue (128 arrivals), by item parity
  kBarLEmpty = 20,     // [2] ... and read (128 arrivals)
  kBarItemFull = 22,   // [2] work-item ring slot written
  kBarItemEmpty = 24,  // [2] ... and read by every role (kItemReaders arrivals)
  kBarOStageFull = 26, // O of an item written to the staging buffer (128 arrivals)
  kBarClc = 27,        // cluster-launch-control answer landed
  kBarDrain = 28,      // both issuers' MMAs finished (two commits)
  kBarOStage = 29,     // the TMA store of the previous epilogue has read the O staging buffer
  kNumFixedBars = 30
};

template <int D, int KS, int VS, bool FP8 = false>
struct FwdLayout {
  static constexpr uint32_t kElem = FP8 ? 1 : 2;  // bytes per Q/K/V element
  static constexpr uint32_t kQBytes = kBlockM * D * kElem;
  static constexpr uint32_t kKVBytes = kBlockN * D * kElem;
  static constexpr uint32_t kOBytes = kBlockM * D * 2;  // O is written in 16 bits
  static constexpr uint32_t kQ = 0;
  static constexpr uint32_t kK = kQ + kQBytes;          // K ring, KS slots
  static constexpr uint32_t kV = kK + KS * kKVBytes;    // V ring, VS slots
  static constexpr uint32_t kOst = kV + VS * kKVBytes;  // O staging for the TMA store
  // k_full[KS], k_empty[KS], v_full[VS], v_empty[VS], then the FwdBar barriers
  static constexpr uint32_t kBar = kOst + kOBytes;
  static constexpr uint32_t kFixedBar = kBar + 2 * (KS + VS) * 8;
  static constexpr uint32_t kMisc = kFixedBar + kNumFixedBars * 8;  // tmem slot, abort, ring[2]
  static constexpr uint32_t kClc = (kMisc + 16 + 15) & ~15u;        // 16-byte answer
  // running row maximum handed from one softmax warpgroup to the other: [row]
  static constexpr uint32_t kMrow = kClc + 16;
  // partial row sums handed to the epilogue warpgroup: [item parity][row]
  static constexpr uint32_t kLpart = kMrow + kBlockM * 4;
  // per softmax warp: the owed epilogue's item index, first row, (batch, head), last tile
  static constexpr uint32_t kEpState = kLpart + 2 * kBlockM * 4;
  static constexpr uint32_t kBytes = kEpState + 8 * 4 * 4 + 1024;  // + alignment slack
  static_assert(kBytes <= 232448, "shared memory per block");
};

// One work item: a 128-row query tile of one (batch, query head).
struct FwdItem {
  int bh;            // batch * Hq + query head
  int q0;            // first query row
  int kv_plane;      // batch * Hkv + key/value head
  int n_tiles;       // K/V tiles the rows of this tile see (those of the block pattern)
  int j_begin;       // first key tile of the span
  int lo_masked;     // key tiles below this need the window's lower-edge mask
  int first_masked;  // key tiles from this on need the causal or ragged-edge mask
  const uint8_t* pattern;  // this query tile's row of the block pattern, or null
};

// Key tiles of an item in order: j_begin, j_begin + 1, ... skipping those the block pattern
// leaves out.  Every role walks the same sequence.
__device__ __forceinline__ int next_kv_tile(const FwdItem& it, int j) {
  if (it.pattern)
    while (!it.pattern[j]) ++j;
  return j;
}

// Work item `id` in launch order.  The (batch, query head) pairs are cut into groups of
// head_group consecutive ones (the query heads of one key/value head are consecutive, and
// head_group is a multiple of their number) whose K/V planes fill about half of L2; a group's
// items run longest query tile first across all its heads (under the causal mask a tile's key
// range grows with its row index), so that the last items of the grid are short ones while the
// K/V tiles in use stay in L2.
__device__ __forceinline__ FwdItem decode_item(int id, const FwdParams& p) {
  FwdItem it;
  const int span = p.head_group * p.n_qtiles;  // items per group
  const int g = id / span;
  const int r = id - g * span;
  const int h0 = g * p.head_group;
  const int gh = min(p.head_group, p.BH - h0);  // heads in this group (the last may be short)
  const int qt = p.n_qtiles - 1 - r / gh;
  it.bh = h0 + r % gh;
  it.q0 = qt * kBlockM;
  const int h = it.bh % p.Hq;
  const int b = it.bh / p.Hq;
  it.kv_plane = b * p.Hkv + h / p.group;
  int j_end;
  kv_tile_span(qt, kBlockM, kBlockN, p.N_q, p.N_kv, p.causal, p.window, it.j_begin, j_end,
               it.lo_masked, it.first_masked);
  it.pattern = nullptr;
  it.n_tiles = j_end - it.j_begin;
  if (p.block_mask) {
    it.pattern = p.block_mask + static_cast<size_t>(qt) * p.n_kvtiles;
    int n = 0;
    for (int j = it.j_begin; j < j_end; ++j) n += it.pattern[j] ? 1 : 0;
    it.n_tiles = n;
  }
  return it;
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          int* status) {
  const bool ok = wait_bounded(bar, parity, abort, status);
  return __all_sync(0xffffffffu, ok);
}

// Epilogue of one item for the softmax thread of row r (its warpgroup did not run the item's
// last tile; that P V has finished): adds the partial sum handed over by the other warpgroup to
// its own, writes O = a / l (the accumulator row read from tensor memory 32 columns at a time)
// to the staging buffer of the TMA store (128-byte-swizzled sub-tiles of 64 columns), and
// L = m + ln l to global memory.  m_fin is the item's final maximum and (l_own, m_own) this
// warpgroup's partial sum and the maximum it refers to.
template <int D, bool BF16, bool FP8 = false>
__device__ __forceinline__ bool run_epilogue(uint32_t o_tmem, float m_fin, float l_own,
                                             float m_own, int item, int q0, int bh, int r,
                                             uint32_t fbars, const float* lpart, uint8_t* staging,
                                             const FwdParams& p, volatile int* abort_flag) {
  // Handover slot item % 2; this is its (item / 2)-th use.
  const uint32_t slot = item & 1;
  if (!warp_wait(fbars + 8u * (kBarLFull + slot), (item >> 1) & 1, abort_flag, p.status))
    return false;
  float l_row = lpart[slot * kBlockM + r];
  mbar_arrive(fbars + 8u * (kBarLEmpty + slot));
  if (m_own != -INFINITY) l_row += l_own * ex2(m_own - m_fin);
  // FP8: the accumulator holds sum_j (2^5 p_j)_E4M3 v8_j with V = v8 * v_scale
  float out_scale = 1.0f;
  if constexpr (FP8) out_scale = p.v_scale[(bh / p.Hq) * p.Hkv + (bh % p.Hq) / p.group];
  const float inv_l = (l_row > 0.0f) ? out_scale / l_row : 0.0f;
  if (item >= 1 && !warp_wait(fbars + 8u * kBarOStage, (item - 1) & 1, abort_flag, p.status))
    return false;
#pragma unroll 1
  for (int c = 0; c < D / 32; ++c) {
    uint32_t o[32];
    tmem_ld32(o_tmem + c * 32, o);
    tmem_wait_ld();
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      uint4 w;
      w.x = pack2<BF16>(__uint_as_float(o[q4 * 8 + 0]) * inv_l,
                        __uint_as_float(o[q4 * 8 + 1]) * inv_l);
      w.y = pack2<BF16>(__uint_as_float(o[q4 * 8 + 2]) * inv_l,
                        __uint_as_float(o[q4 * 8 + 3]) * inv_l);
      w.z = pack2<BF16>(__uint_as_float(o[q4 * 8 + 4]) * inv_l,
                        __uint_as_float(o[q4 * 8 + 5]) * inv_l);
      w.w = pack2<BF16>(__uint_as_float(o[q4 * 8 + 6]) * inv_l,
                        __uint_as_float(o[q4 * 8 + 7]) * inv_l);
      const uint32_t chunk = c * 4 + q4;  // 16-byte chunk of the row
      *reinterpret_cast<uint4*>(staging + (chunk >> 3) * kSubTile + sw128(r, chunk & 7)) = w;
    }
  }
  fence_proxy_async_smem();
  mbar_arrive(fbars + 8u * kBarOStageFull);  // the P V issuer sends the TMA store
  const int row = q0 + r;
  if (row < p.N_q) {
    const float mu = (m_fin == -INFINITY) ? 0.0f : m_fin;
    const float shift = FP8 ? static_cast<float>(kPShift8) : 0.0f;
    p.lse[static_cast<size_t>(bh) * p.N_q + row] =
        (l_row > 0.0f) ? (mu + lg2(l_row) - shift) * 0.69314718055994531f : -INFINITY;
  }
  return true;
}

template <int D, bool BF16, int KS, int VS, bool FP8 = false>
__global__ void __launch_bounds__(kFwdThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                    const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v,
                    const __grid_constant__ CUtensorMap tm_o, const FwdParams p) {
  using L = FwdLayout<D, KS, VS, FP8>;
  // 128-byte swizzled column chunks of a Q/K tile row: 64 16-bit or 128 8-bit elements
  constexpr int kChunks = FP8 ? 1 : D / 64;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);

  const uint32_t sQ = base + L::kQ;
  const uint32_t sK = base + L::kK;
  const uint32_t sV = base + L::kV;
  const uint32_t sOst = base + L::kOst;
  const uint32_t bars = base + L::kBar;
  const uint32_t fbars = base + L::kFixedBar;
#define BAR_K(s) (bars + 8u * (s))
#define BAR_KE(s) (bars + 8u * (KS + (s)))
#define BAR_V(s) (bars + 8u * (2u * KS + (s)))
#define BAR_VE(s) (bars + 8u * (2u * KS + VS + (s)))
#define FBAR(i) (fbars + 8u * (i))
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L::kMisc + 4);
  volatile int* ring = reinterpret_cast<volatile int*>(gbase + L::kMisc + 8);  // [2] item ids
  const uint32_t clc_resp = base + L::kClc;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
#ifdef ATTN_FWD_TRACE
  const int trace_slot = (blockIdx.x < 8) ? static_cast<int>(blockIdx.x) : -1;
#endif

  if (threadIdx.x == 0) FWD_TRACE(79, 0);
  if (threadIdx.x == 0) {
    for (int s = 0; s < KS; ++s) {
      mbar_init(BAR_K(s), 1);
      mbar_init(BAR_KE(s), 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(BAR_V(s), 1);
      mbar_init(BAR_VE(s), 1);
    }
    mbar_init(FBAR(kBarQFull), 1);
    mbar_init(FBAR(kBarQEmpty), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(FBAR(kBarS + b), 1);
      mbar_init(FBAR(kBarSFree + b), kSoftmaxThreads);
      mbar_init(FBAR(kBarP + b), kSoftmaxThreads);
      mbar_init(FBAR(kBarO + b), 1);
      for (int q = 0; q < 4; ++q) mbar_init(FBAR(kBarM + b * 4 + q), 32);
      mbar_init(FBAR(kBarItemFull + b), 1);
      mbar_init(FBAR(kBarItemEmpty + b), kItemReaders);
      mbar_init(FBAR(kBarLFull + b), kSoftmaxThreads);
      mbar_init(FBAR(kBarLEmpty + b), kSoftmaxThreads);
    }
    mbar_init(FBAR(kBarOStageFull), kSoftmaxThreads);
    mbar_init(FBAR(kBarClc), 1);
    mbar_init(FBAR(kBarDrain), 2);  // one commit from each issuer
    mbar_init(FBAR(kBarOStage), 1);
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

  // Work item k of this block from the ring (single-thread readers; -1 = no more work).
  auto take_item = [&](int k, int& id) -> bool {
    if (!wait_bounded(FBAR(kBarItemFull + (k & 1)), (k >> 1) & 1, abort_flag, p.status))
      return false;
    id = ring[k & 1];
    mbar_arrive(FBAR(kBarItemEmpty + (k & 1)));
    return true;
  };

  if (warp >= kProducerWarp) {
    // Warps 8-11 (one warpgroup) need few registers; the softmax warpgroups take the rest of
    // the 168 per thread the block was launched with: 2 x 128 x 184 + 128 x 136 = 384 x 168.
    setmaxnreg_dec<kRegsIssue>();
  if (warp == kProducerWarp) {
    // ----------------------------------------------------------------- scheduler + Q/K producer
    // Publishes the block's work items (its own first, then those of pending blocks it cancels)
    // and loads, per item, K_0, Q and then K_1, K_2, ...: a K slot is refilled as soon as its
    // score MMA finished, and Q once the previous item's last score MMA finished.  The next
    // item is requested when an item starts; as soon as the answer is in, its Q tile is pulled
    // into L2, so that the Q load at the item boundary is short.
    if (lane == 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      int id = static_cast<int>(blockIdx.x);
      int next_id = -1;
      bool clc_live = true;     // no answer "nothing left" seen yet
      bool clc_pending = false;  // a request is in flight
      uint32_t clc_uses = 0;
      auto take_answer = [&]() {
        clc_pending = false;
        ++clc_uses;
        int x;
        if (clc_query(clc_resp, x)) {
          next_id = x;
          const FwdItem nx = decode_item(x, p);
          if (nx.n_tiles > 0) {
#pragma unroll
            for (int sub = 0; sub < kChunks; ++sub) tma_prefetch_l2_3d(&tm_q, sub * 64, nx.q0, nx.bh);
          }
        } else {
          next_id = -1;
          clc_live = false;
        }
      };
      int T = 0, kq = 0;  // K tiles and Q tiles loaded so far
      bool ok = true;
      for (int k = 0; ok; ++k) {
        if (k >= 2 &&
            !wait_bounded(FBAR(kBarItemEmpty + (k & 1)), ((k >> 1) - 1) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        ring[k & 1] = id;
        mbar_arrive(FBAR(kBarItemFull + (k & 1)));
        if (id < 0) break;
        // The following item is asked for with this item's last K load (a few tiles before the
        // softmax finishes this item): late enough that a block does not hold on to work other
        // blocks could start, early enough to pull the next Q tile into L2 in time.
        auto request_next = [&]() {
          if (clc_live) {
            mbar_arrive_expect_tx(FBAR(kBarClc), 16);
            clc_try_cancel(clc_resp, FBAR(kBarClc));
            clc_pending = true;
          }
        };
        next_id = -1;
        const FwdItem it = decode_item(id, p);
        if (it.n_tiles == 0) request_next();
        for (int j = 0, kt = it.j_begin; j < it.n_tiles; ++j, ++kt) {
          kt = next_kv_tile(it, kt);
          const int s = T % KS;
          if (T >= KS && !wait_bounded(BAR_KE(s), ((T / KS) - 1) & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(BAR_K(s), L::kKVBytes);
#pragma unroll
          for (int sub = 0; sub < kChunks; ++sub)
            tma_load_3d(sK + s * L::kKVBytes + sub * kSubTile, &tm_k, BAR_K(s), sub * 64,
                        kt * kBlockN, it.kv_plane);
          ++T;
          if (j == 0) {
            if (kq >= 1 && !wait_bounded(FBAR(kBarQEmpty), (kq - 1) & 1, abort_flag, p.status)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(FBAR(kBarQFull), L::kQBytes);
#pragma unroll
            for (int sub = 0; sub < kChunks; ++sub)
              tma_load_3d(sQ + sub * kSubTile, &tm_q, FBAR(kBarQFull), sub * 64, it.q0, it.bh);
            ++kq;
          }
          if (j == it.n_tiles - 1) request_next();
        }
        if (!ok) break;
        if (clc_pending) {
          if (!wait_bounded(FBAR(kBarClc), clc_uses & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          take_answer();
        }
        id = next_id;
      }
      // Every asynchronous write into this block's shared memory lands before it may exit.
      for (int t = (T > KS ? T - KS : 0); t < T; ++t)
        wait_bounded(BAR_K(t % KS), (t / KS) & 1, nullptr, p.status, kDrainLimitNs);
      if (kq >= 1)
        wait_bounded(FBAR(kBarQFull), (kq - 1) & 1, nullptr, p.status, kDrainLimitNs);
      if (clc_pending)
        wait_bounded(FBAR(kBarClc), clc_uses & 1, nullptr, p.status, kDrainLimitNs);
    }
    __syncwarp();
  } else if (warp == kVProducerWarp) {
    // ----------------------------------------------------------------- V producer
    if (lane == 0) {
      prefetch_tmap(&tm_v);
      int T = 0;
      bool ok = true;
      for (int k = 0; ok; ++k) {
        int id;
        if (!take_item(k, id)) break;
        if (id < 0) break;
        const FwdItem it = decode_item(id, p);
        for (int j = 0, kt = it.j_begin; j < it.n_tiles; ++j, ++kt) {
          kt = next_kv_tile(it, kt);
          const int s = T % VS;
          if (T >= VS && !wait_bounded(BAR_VE(s), ((T / VS) - 1) & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(BAR_V(s), L::kKVBytes);
          if constexpr (FP8) {
            // V^T tile: d rows of 128 keys (the K-major B operand of the 8-bit P V product)
            tma_load_3d(sV + s * L::kKVBytes, &tm_v, BAR_V(s), kt * kBlockN, 0, it.kv_plane);
          } else {
#pragma unroll
            for (int sub = 0; sub < D / 64; ++sub)
              tma_load_3d(sV + s * L::kKVBytes + sub * kSubTile, &tm_v, BAR_V(s), sub * 64,
                          kt * kBlockN, it.kv_plane);
          }
          ++T;
        }
      }
      for (int t = (T > VS ? T - VS : 0); t < T; ++t)
        wait_bounded(BAR_V(t % VS), (t / VS) & 1, nullptr, p.status, kDrainLimitNs);
    }
    __syncwarp();
  } else if (warp == kQkWarp || warp == kPvWarp) {
    // ----------------------------------------------------------------- tcgen05 issuers
    // Warp 9 issues the score MMAs, warp 10 the P V MMAs.  The two streams touch disjoint tensor
    // memory (S buffers / O and P buffers) and disjoint shared memory (Q, K / V), so they need no
    // ordering between them beyond the barriers below, and each issuer's waits overlap the other
    // issuer's MMAs.
    if (lane == 0) {
      const bool qk_issuer = (warp == kQkWarp);
      // (FP8: kind::f8f6f4 with format code 0 = E4M3 for A and B; V^T is K-major)
      constexpr uint32_t idesc_qk = make_idesc_f16(BF16 && !FP8, kBlockM, kBlockN, false);
      constexpr uint32_t idesc_pv = make_idesc_f16(BF16 && !FP8, kBlockM, D, !FP8);
      // S_t = Q K_t^T into S buffer t % 2, once the softmax of tile t - 2 has read that buffer.
      auto issue_qk = [&](int t) -> bool {
        FWD_TRACE(t, 8);
        const int s = t % KS;
        if (t >= 2 &&
            !wait_bounded(FBAR(kBarSFree + (t & 1)), ((t >> 1) - 1) & 1, abort_flag, p.status))
          return false;
        FWD_TRACE(t, 15);
        if (!wait_bounded(BAR_K(s), (t / KS) & 1, abort_flag, p.status)) return false;
        FWD_TRACE(t, 9);
        tc_fence_after();
        const uint32_t s_col = tmem + ((t & 1) ? kColS1 : kColS0);
        if constexpr (FP8) {
          // 8-bit Q and K, K-major: 32 elements = 32 bytes per MMA in the one 128-byte row
#pragma unroll
          for (int kk = 0; kk < D / 32; ++kk) {
            const uint64_t adesc = make_sdesc_sw128(sQ + kk * 32, 16, 1024);
            const uint64_t bdesc = make_sdesc_sw128(sK + s * L::kKVBytes + kk * 32, 16, 1024);
            mma_ss_f8(s_col, adesc, bdesc, idesc_qk, kk > 0 ? 1u : 0u);
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            // Q and K are K-major (d contiguous): 16 elements = 32 bytes per MMA inside the
            // 128-byte swizzle row; SBO = 1024 B between 8-row groups.
            const uint32_t off = (kk >> 2) * kSubTile + (kk & 3) * 32;
            const uint64_t adesc = make_sdesc_sw128(sQ + off, 16, 1024);
            const uint64_t bdesc = make_sdesc_sw128(sK + s * L::kKVBytes + off, 16, 1024);
            mma_ss(s_col, adesc, bdesc, idesc_qk, kk > 0 ? 1u : 0u);
          }
        }
        mma_commit(FBAR(kBarS + (t & 1)));
        mma_commit(BAR_KE(s));  // K slot free
        FWD_TRACE(t, 10);
        return true;
      };
      // O (+)= P_t V_t (P_t in P buffer t % 2, V_t in ring slot t % VS); the first tile of
      // an item overwrites the accumulator.
      auto issue_pv = [&](int t, bool first) -> bool {
        FWD_TRACE(t, 11);
        if (!wait_bounded(FBAR(kBarP + (t & 1)), (t >> 1) & 1, abort_flag, p.status)) return false;
        FWD_TRACE(t, 12);
        const int s = t % VS;
        if (!wait_bounded(BAR_V(s), (t / VS) & 1, abort_flag, p.status)) return false;
        FWD_TRACE(t, 13);
        tc_fence_after();
        const uint32_t p_col = tmem + ((t & 1) ? PCols<D>::kP1 : PCols<D>::kP0);
        if constexpr (FP8) {
          // P: E4M3 codes, four per tensor-memory column; V^T rows (d) of 128 keys, K-major:
          // 32 keys = 32 bytes per MMA in the 128-byte row
#pragma unroll
          for (int kk = 0; kk < kBlockN / 32; ++kk) {
            const uint64_t bdesc = make_sdesc_sw128(sV + s * L::kKVBytes + kk * 32, 16, 1024);
            mma_ts_f8(tmem + kColO, p_col + kk * 8, bdesc, idesc_pv, (!first || kk > 0) ? 1u : 0u);
          }
        } else {
#pragma unroll
          for (int kk = 0; kk < kBlockN / 16; ++kk) {
            // V is [keys, d] with d contiguous: the B operand is MN-major.  16 keys per MMA
            // (two 8-row groups, SBO = 1024 B apart); the two 64-column halves of d are
            // separate swizzled sub-tiles (LBO = one sub-tile).
            const uint64_t bdesc = make_sdesc_sw128(sV + s * L::kKVBytes + kk * 16 * 128,
                                                    kSubTile, 1024);
            mma_ts(tmem + kColO, p_col + kk * 8, bdesc, idesc_pv, (!first || kk > 0) ? 1u : 0u);
          }
        }
        mma_commit(FBAR(kBarO + (t & 1)));
        mma_commit(BAR_VE(s));  // V slot free
        FWD_TRACE(t, 14);
        return true;
      };
      // The score issuer runs up to two tiles ahead of the softmax (two S buffers), also into
      // the next item; the P V issuer follows the softmax tile by tile.  The P V issuer also
      // sends each item's O tile to global memory: the epilogue of item e fills the staging
      // buffer during the first tile of item e + 1, and the TMA store goes out from here while
      // item e + 1's MMAs run (at the latest after its last P V), so that no softmax warp ever
      // waits for a store.
      int T = 0, kq = 0;  // tiles and non-empty items issued so far
      int st_q0 = 0, st_bh = 0;  // the previous non-empty item, whose O is to be stored
      bool stored = true;        // ... and its store has been issued
      auto store_o = [&]() {
#pragma unroll
        for (int sub = 0; sub < D / 64; ++sub)
          tma_store_3d(&tm_o, sOst + sub * kSubTile, sub * 64, st_q0, st_bh);
        tma_store_commit();
        stored = true;
      };
      bool ok = true;
      for (int k = 0; ok; ++k) {
        int id;
        if (!take_item(k, id)) break;
        if (id < 0) break;
        const FwdItem it = decode_item(id, p);
        if (it.n_tiles == 0) continue;
        if (qk_issuer) {
          if (!wait_bounded(FBAR(kBarQFull), kq & 1, abort_flag, p.status)) break;
          for (int j = 0; ok && j < it.n_tiles; ++j) ok = issue_qk(T + j);
          if (ok) mma_commit(FBAR(kBarQEmpty));  // Q free once these MMAs finished
        } else {
          for (int j = 0; ok && j < it.n_tiles; ++j) {
            ok = issue_pv(T + j, j == 0);
            if (!stored && mbar_test_wait(FBAR(kBarOStageFull), (kq - 1) & 1)) store_o();
          }
          if (!ok) break;
          if (kq >= 1) {
            // The staging buffer is free again once the store has read it.
            if (!stored) {
              if (!wait_bounded(FBAR(kBarOStageFull), (kq - 1) & 1, abort_flag, p.status)) break;
              store_o();
            }
            tma_store_wait_read0();
            mbar_arrive(FBAR(kBarOStage));
          }
          st_q0 = it.q0;
          st_bh = it.bh;
          stored = false;
        }
        T += it.n_tiles;
        ++kq;
      }
      if (!qk_issuer && ok && kq >= 1 && !stored &&
          wait_bounded(FBAR(kBarOStageFull), (kq - 1) & 1, abort_flag, p.status))
        store_o();
      if (!qk_issuer) tma_store_wait_all();  // every O tile written before the block exits
      // Every MMA this thread issued completes before the block frees tensor memory.
      if (T > 0)
        mma_commit(FBAR(kBarDrain));
      else
        mbar_arrive(FBAR(kBarDrain));
      wait_bounded(FBAR(kBarDrain), 0, nullptr, p.status, kDrainLimitNs);
    }
    __syncwarp();
  }
    tc_fence_before();
    __syncthreads();  // every tensor-memory access and MMA of the block has finished
    if (warp == kQkWarp) {
      tc_fence_after();
      tmem_dealloc(tmem, kTmemCols);
    }
  } else {
    setmaxnreg_inc<kRegsSoftmax>();
    // ----------------------------------------------------------------- softmax + epilogue
    // Two warpgroups share the rows: warpgroup w takes the tiles t of the block's tile sequence
    // with t % 2 == w (S buffer w, P buffer w); in both, thread r owns query row r and warp % 4
    // is its tensor-memory lane quarter.  The running maximum is the only state carried from
    // tile to tile: the warpgroup of tile t publishes m_t as soon as its row maxima are known
    // (kBarM, one barrier per warp: warp q of one warpgroup and warp q of the other own the same
    // 32 rows), and the other warpgroup, on tile t + 1, waits for it before its exponentials.
    // Each warpgroup keeps its own partial row sum, rescaled whenever the maximum moves.
    //
    // Epilogue of an item whose last tile is t_e: the warpgroup of t_e hands its partial sum
    // (relative to the final maximum m_{t_e}) over through shared memory and goes on; the other
    // warpgroup finishes the item during its next tile t_e + 1 (the first tile of the next
    // item): it reads m_{t_e} with the running maximum, reads the accumulator out of tensor
    // memory between storing P_{t_e+1} and releasing it (so before P V_{t_e+1} overwrites the
    // accumulator), then writes O = a / l to the staging buffer for the TMA store and the
    // log-sum-exp to global memory.
    const int wg = warp >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t row_tmem = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    [[maybe_unused]] const bool tracer = (threadIdx.x & 127) == 0;  // timestamp hooks only
    const int off = p.N_kv - p.N_q;
    const float sl2 = p.sl2;
    // read once: the masked tiles' bounds (those tiles come once or twice an item, and their
    // parameter reads would otherwise be fetched cold)
    const int n_kv = p.N_kv, causal = p.causal, window = p.window;
    float* mrow = reinterpret_cast<float*>(gbase + L::kMrow);    // [row]
    float* lpart = reinterpret_cast<float*>(gbase + L::kLpart);  // [item parity][row]
    const uint32_t s_col = wg ? kColS1 : kColS0;
    const uint32_t p_col = wg ? PCols<D>::kP1 : PCols<D>::kP0;
    float m_own = -INFINITY;  // maximum (log2 units) this warpgroup's partial sum refers to
    float l = 0.0f;           // this warpgroup's partial sum of 2^(x - m_own)
    int T = 0;                // tiles of the block's sequence before the current item
    int kq = 0;               // items with at least one tile before the current one
    bool ok = true;
    bool s_ready = false;  // S of this warpgroup's next tile already seen complete
    // Epilogue this warpgroup owes: item index, first row, (batch, head), partial sum and
    // its maximum, and the item's last tile.
    // The owed epilogue's item data wait in shared memory (one copy per warp, written by its
    // lane 0 and read by the same warp), so that they take no registers across the
    // exponential loop.
    volatile int* ep_state = reinterpret_cast<volatile int*>(gbase + L::kEpState) + 4 * warp;
    bool ep_pending = false;
    float ep_l = 0.0f, ep_m = -INFINITY;

    for (int k = 0; ok; ++k) {
      if (tracer) FWD_TRACE(T, 16 + wg * 4);
      if (!warp_wait(FBAR(kBarItemFull + (k & 1)), (k >> 1) & 1, abort_flag, p.status)) break;
      if (tracer) FWD_TRACE(T, 17 + wg * 4);
      const int id = ring[k & 1];
      __syncwarp();
      if (lane == 0) mbar_arrive(FBAR(kBarItemEmpty + (k & 1)));
      if (id < 0) break;
      const FwdItem it = decode_item(id, p);
      if (tracer) FWD_TRACE(T, 18 + wg * 4);
      const int n = it.n_tiles;
      const int row = it.q0 + r;
      if (n == 0) {
        // No key visible to any row of this tile: O = 0, L = -inf.
        if (wg == 0 && row < p.N_q) {
          const size_t row_index = static_cast<size_t>(it.bh) * p.N_q + row;
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + row_index * D);
#pragma unroll
          for (int c = 0; c < D / 8; ++c) dst[c] = make_uint4(0, 0, 0, 0);
          p.lse[row_index] = -INFINITY;
        }
        continue;
      }
      const int T0 = T;
      const int T_last = T0 + n - 1;
      // FP8: the item's Q block scale (its K block scales are read per tile, before the wait
      // for the tile's scores, so that the loads are in flight during the wait)
      float q_sc = 1.0f;
      if constexpr (FP8) q_sc = p.q_scale[static_cast<size_t>(it.bh) * p.n_qtiles + it.q0 / kBlockM];
      for (int i = 0, j = it.j_begin; i < n; ++i, ++j) {
        j = next_kv_tile(it, j);  // key tile of the item's i-th tile
        const int t = T0 + i;
        if ((t & 1) != wg) continue;
        const int u = t >> 1;  // use index of this warpgroup's S and P buffers
        float k_sc = 1.0f;
        if constexpr (FP8) k_sc = p.k_scale[static_cast<size_t>(it.kv_plane) * p.n_kvtiles + j];
        if (tracer) FWD_TRACE(t, 0);
        if (!__all_sync(0xffffffffu, s_ready) &&
            !warp_wait(FBAR(kBarS + wg), u & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        if (tracer) FWD_TRACE(t, 1);
        tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(row_tmem + s_col + c * 32, sr[c]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(FBAR(kBarSFree + wg));  // S buffer free for Q K_{t+2}^T
        if (tracer) FWD_TRACE(t, 2);
        // Early, non-blocking test of the barrier needed before P is written (P V_{t-2} read
        // this P buffer); its latency hides under the work below.
        const bool p_free = (t < 2) || mbar_test_wait(FBAR(kBarO + wg), (u - 1) & 1);
        float x[kBlockN];
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) x[c * 32 + e] = __uint_as_float(sr[c][e]);
        if (j >= it.first_masked || j < it.lo_masked) {
          // Visible columns [lo, hi] of this row in this tile: hi from the causal bound or the
          // ragged end, lo from the sliding window.  One code path for every masked tile, as
          // four 32-column bit masks and one test per column: masked tiles come once or twice
          // an item, so their code is fetched cold, and a short path costs less.
          int hi = kBlockN - 1, lo = 0;
          if (j >= it.first_masked) {
            int lim = causal ? row + off : n_kv - 1;  // last visible key of this row
            if (lim > n_kv - 1) lim = n_kv - 1;
            hi = min(lim - j * kBlockN, kBlockN - 1);
          }
          if (j < it.lo_masked) lo = max(row + off - window - j * kBlockN, 0);
          uint32_t vis[kBlockN / 32];
#pragma unroll
          for (int g = 0; g < kBlockN / 32; ++g) {
            const int a = max(lo - 32 * g, 0), bb = min(hi - 32 * g, 31);
            vis[g] = (a > bb) ? 0u : ((0xffffffffu >> (31 - bb)) & (0xffffffffu << a));
          }
          // x + 0 where visible, x + (-inf) where not: integer arithmetic, no per-column
          // condition (each of which could otherwise become a divergent branch)
#pragma unroll
          for (int c = 0; c < kBlockN; ++c)
            x[c] += __uint_as_float((((vis[c >> 5] >> (c & 31)) & 1u) - 1u) & 0xff800000u);
        }
        // Row maximum of the tile: three-input max, sixteen independent chains.
        float mx[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) mx[e] = fmaxf(x[e], x[16 + e]);
#pragma unroll
        for (int c = 32; c < kBlockN; c += 32)
#pragma unroll
          for (int e = 0; e < 16; ++e) mx[e] = max3f(mx[e], x[c + e], x[c + 16 + e]);
#pragma unroll
        for (int e = 0; e < 8; ++e) mx[e] = fmaxf(mx[e], mx[e + 8]);
        const float tile_max = max3f(max3f(mx[0], mx[1], mx[2]), max3f(mx[3], mx[4], mx[5]),
                                     fmaxf(mx[6], mx[7]));
        // Running maximum after tile t - 1, from the other warpgroup (on the first tile of an
        // item: the previous item's final maximum, which an owed epilogue needs).  The wait also
        // orders this tile's write of mrow after the other warpgroup's read of it.
        float m_read = -INFINITY;
        if (tracer) FWD_TRACE(t, 24);
        if (t > 0) {
          if (!warp_wait(FBAR(kBarM + (wg ^ 1) * 4 + quarter), ((t - 1) >> 1) & 1, abort_flag,
                         p.status)) {
            ok = false;
            break;
          }
          m_read = mrow[r];
        }
        const float m_prev = (i > 0) ? m_read : -INFINITY;
        // Score scale of this tile: scale * log2(e), times the E4M3 block scales for FP8.
        float tsc = sl2;
        if constexpr (FP8) tsc = sl2 * q_sc * k_sc;
        // The maximum moves only when it rises by more than 2^8 (also for the first finite one);
        // FP8: by more than 2^3.8.
        float m_j = m_prev;
        float alpha = 1.0f;  // rescale of the accumulator O for this tile
        const float m_new = fmaxf(m_prev, tile_max * tsc);
        if (m_new - m_prev > (FP8 ? kRescaleThreshold8 : kRescaleThreshold)) {
          alpha = ex2(m_prev - m_new);
          m_j = m_new;
        }
        mrow[r] = m_j;
        mbar_arrive(FBAR(kBarM + wg * 4 + quarter));  // m_t published for tile t + 1
        if (tracer) FWD_TRACE(t, 25);
        if (m_j != m_own) {
          l = (m_own == -INFINITY) ? 0.0f : l * ex2(m_own - m_j);
          m_own = m_j;
        }
        const float neg_mu = ((m_j == -INFINITY) ? 0.0f : -m_j) + (FP8 ? kPShift8 : 0);
        // p = 2^(x * scale * log2(e) - m): one packed FMA per pair of scores and MUFU ex2, all
        // of them first (in place, so that consecutive ex2 depend on nothing but their own FMA),
        // then a packed add into four pair-accumulators for the row sum and the 16-bit pack for
        // P (FP8: 2^5 p, four E4M3 codes per word).
#pragma unroll
        for (int c = 0; c < kBlockN; c += 2) {
          float a0, a1;
          fma2(a0, a1, x[c], x[c + 1], tsc, tsc, neg_mu, neg_mu);
          x[c] = ex2(a0);
          x[c + 1] = ex2(a1);
        }
        float ps[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        uint32_t pk[2][32];
#pragma unroll
        for (int c = 0; c < kBlockN; c += 4) {
          const float p0 = x[c], p1 = x[c + 1], p2 = x[c + 2], p3 = x[c + 3];
          const int k2 = ((c >> 1) & 3) * 2;
          add2(ps[k2], ps[k2 + 1], p0, p1);
          add2(ps[k2 + 2], ps[k2 + 3], p2, p3);
          if constexpr (FP8) {
            pk[0][c >> 2] = pack4_e4m3(p0, p1, p2, p3);
          } else {
            pk[c >> 6][(c >> 1) & 31] = pack2<BF16>(p0, p1);
            pk[c >> 6][((c >> 1) & 31) + 1] = pack2<BF16>(p2, p3);
          }
        }
        l += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
        // Tile t + 2 is this warpgroup's next one, in this item or the next.
        s_ready = mbar_test_wait(FBAR(kBarS + wg), (u + 1) & 1);
        if (tracer) FWD_TRACE(t, 3);
        if (t >= 2) {
          if (!__all_sync(0xffffffffu, p_free) &&
              !warp_wait(FBAR(kBarO + wg), (u - 1) & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();  // order the P store after the MMA that read the buffer
        }
        if (tracer) FWD_TRACE(t, 4);
        tmem_st32(row_tmem + p_col, pk[0]);
        if constexpr (!FP8) tmem_st32(row_tmem + p_col + 32, pk[1]);
        // Both cases below need P V_{t-1} finished: P V_t waits for this tile's P and P V_{t+1}
        // comes after it, so nothing else touches the accumulator meanwhile.
        const bool rescale = i > 0 && __any_sync(0xffffffffu, alpha != 1.0f);
        if (rescale || ep_pending) {
          if (!warp_wait(FBAR(kBarO + (wg ^ 1)), ((t - 1) >> 1) & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        if (rescale) {
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
        if (ep_pending) {
          // The first tile after the owed item's last one: its accumulator is read out before
          // this tile's P is released to P V_t, which overwrites it.
          if (tracer) FWD_TRACE(ep_state[3], 6);
          if (!run_epilogue<D, BF16, FP8>(row_tmem + kColO, m_read, ep_l, ep_m, ep_state[0],
                                     ep_state[1], ep_state[2], r,
                                     fbars, lpart, gbase + L::kOst, p, abort_flag)) {
            ok = false;
            break;
          }
          ep_pending = false;
          if (tracer) FWD_TRACE(ep_state[3], 7);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(FBAR(kBarP + wg));
        if (tracer) FWD_TRACE(t, 5);
      }
      if (!ok) break;
      if (tracer) FWD_TRACE(T, 19 + wg * 4);
      // ------------------------------------------------------------- end of the item
      if ((T_last & 1) == wg) {
        // This warpgroup ran the last tile: its partial sum refers to the final maximum.  The
        // other warpgroup finishes the item.
        // Handover slot kq % 2, free once item kq - 2's epilogue has read it.
        const int slot = kq & 1;
        if (kq >= 2 &&
            !warp_wait(FBAR(kBarLEmpty + slot), ((kq >> 1) - 1) & 1, abort_flag, p.status))
          break;
        lpart[slot * kBlockM + r] = l;
        mbar_arrive(FBAR(kBarLFull + slot));
      } else {
        ep_pending = true;
        if (lane == 0) {
          ep_state[0] = kq;
          ep_state[1] = it.q0;
          ep_state[2] = it.bh;
          ep_state[3] = T_last;
        }
        __syncwarp();
        ep_l = l;
        ep_m = m_own;
      }
      l = 0.0f;
      m_own = -INFINITY;
      T += n;
      ++kq;
    }
    if (ok && ep_pending) {
      // No tile follows the block's last item: finish it here.  A parity wait is only sound
      // while its barrier is at most one phase behind or ahead of the awaited one: tile t_e - 1
      // was this warpgroup's (its P-buffer wait saw P V_{t_e-3} finish), so P V_{t_e-1} is
      // awaited first on this warpgroup's barrier, which makes P V_{t_e-2} finished too and
      // P V_{t_e} the next phase of the other barrier.
      const int t_e = ep_state[3];
      bool done = true;
      if (t_e >= 1)
        done = warp_wait(FBAR(kBarO + ((t_e - 1) & 1)), ((t_e - 1) >> 1) & 1, abort_flag, p.status);
      done = done && warp_wait(FBAR(kBarO + (t_e & 1)), (t_e >> 1) & 1, abort_flag, p.status);
      if (done && warp_wait(FBAR(kBarM + (t_e & 1) * 4 + quarter), (t_e >> 1) & 1, abort_flag,
                            p.status)) {
        tc_fence_after();
        run_epilogue<D, BF16, FP8>(row_tmem + kColO, mrow[r], ep_l, ep_m, ep_state[0], ep_state[1],
                              ep_state[2], r, fbars,
                              lpart, gbase + L::kOst, p, abort_flag);
      }
    }
    tc_fence_before();
    __syncthreads();  // the other warpgroup's matching barrier ends its branch
    if (threadIdx.x == 0) FWD_TRACE(79, 1);
  }
#undef BAR_K
#undef BAR_V
#undef BAR_KE
#undef BAR_VE
#undef FBAR
}

// O = 0 and L = -inf for every row (used when there is no key at all).
template <bool BF16>
__global__ void attn_empty_rows_kernel(uint16_t* o, float* lse, size_t rows, int d) {
  const size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x;
  if (i < rows * d) o[i] = 0;
  if (i < rows) lse[i] = -INFINITY;
}

template <int D, bool BF16, int KS, int VS, bool FP8 = false>
static int launch_fwd_variant(const FwdArgs& a, cudaStream_t stream) {
  using L = FwdLayout<D, KS, VS, FP8>;
  CUtensorMap tq, tk, tv, to;
  const uint64_t bhq = static_cast<uint64_t>(a.B) * a.Hq;
  const uint64_t bhk = static_cast<uint64_t>(a.B) * a.Hkv;
  const uint64_t rq = static_cast<uint64_t>(D) * 2, rk = rq;
  if constexpr (FP8) {
    // E4M3 codes: Q and K rows of d bytes (one 128-byte swizzle chunk at d = 128); V^T rows of
    // nkvp keys, loaded as d x 128-key tiles
    if (!make_tmap_3d_u8(&tq, a.q8, D, a.N_q, bhq, D, static_cast<uint64_t>(D) * a.N_q, D, kBlockM, 1) ||
        !make_tmap_3d_u8(&tk, a.k8, D, a.N_kv, bhk, D, static_cast<uint64_t>(D) * a.N_kv, D, kBlockN, 1) ||
        !make_tmap_3d_u8(&tv, a.vt8, a.nkvp, D, bhk, a.nkvp, static_cast<uint64_t>(a.nkvp) * D,
                         kBlockN, D, 1))
      return -5;
  } else {
    if (!make_tmap_3d(&tq, a.q, BF16, D, a.N_q, bhq, rq, rq * a.N_q, 64, kBlockM, 1) ||
        !make_tmap_3d(&tk, a.k, BF16, D, a.N_kv, bhk, rk, rk * a.N_kv, 64, kBlockN, 1) ||
        !make_tmap_3d(&tv, a.v, BF16, D, a.N_kv, bhk, rk, rk * a.N_kv, 64, kBlockN, 1))
      return -5;
  }
  if (!make_tmap_3d(&to, a.o, BF16, D, a.N_q, bhq, rq, rq * a.N_q, 64, kBlockM, 1)) return -5;
  FwdParams p;
  p.o = a.o;
  p.lse = a.lse;
  p.status = device_status_ptr();
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.N_q = a.N_q;
  p.N_kv = a.N_kv;
  p.n_qtiles = (a.N_q + kBlockM - 1) / kBlockM;
  p.group = a.Hq / a.Hkv;
  p.causal = (a.causal || a.window >= 0) ? 1 : 0;
  p.window = a.window;
  p.n_kvtiles = (a.N_kv + kBlockN - 1) / kBlockN;
  p.block_mask = a.block_mask;
  p.q_scale = a.q_scale;
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
  p.BH = static_cast<int>(bhq);
  {
    // Query heads whose K/V planes fill about half of L2, a multiple of the heads sharing one
    // key/value plane.
    static int l2_bytes = -1;
    if (l2_bytes < 0) {
      int dev = 0, v = 0;
      if (cudaGetDevice(&dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev) != cudaSuccess || v <= 0)
        v = 64 << 20;
      l2_bytes = v;
    }
    const uint64_t plane_bytes = 2ull * a.N_kv * D * L::kElem;
    uint64_t planes = (static_cast<uint64_t>(l2_bytes) / 2) / plane_bytes;
    if (planes < 1) planes = 1;
    uint64_t heads = planes * static_cast<uint64_t>(a.Hq / a.Hkv);
    if (heads > bhq) heads = bhq;
    p.head_group = static_cast<int>(heads);
  }
  p.sl2 = a.scale * 1.4426950408889634f;
  if (!p.status) return -5;
  auto kern = attn_fwd_kernel<D, BF16, KS, VS, FP8>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes) !=
      cudaSuccess)
    return -5;
  // One block per work item; the running blocks take over the items of the others.
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

static std::atomic<int> g_d64_mode{0};

int set_d64_kernel(int mode) {
  if (mode < 0 || mode > 2) return -1;
  return g_d64_mode.exchange(mode);
}

int launch_attn_fwd_fp8_kernel(const FwdArgs& a, cudaStream_t stream) {
  if (a.d != 128) return -2;
  return a.bf16 ? launch_fwd_variant<128, true, 4, 4, true>(a, stream)
                : launch_fwd_variant<128, false, 4, 4, true>(a, stream);
}

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
  if (a.d == 64) {
    // Two query tiles per item when there are more query tiles than SMs (so that the pairs
    // still cover every SM), else one.
    const int mode = g_d64_mode.load();
    bool pair = (mode == 1);
    if (mode == 0) {
      const uint64_t tiles = static_cast<uint64_t>(a.B) * a.Hq * ((a.N_q + kBlockM - 1) / kBlockM);
      int dev = 0, n_sm = 0;
      if (cudaGetDevice(&dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return -5;
      pair = tiles > static_cast<uint64_t>(n_sm);
    }
    if (pair) return launch_attn_fwd_pair(a, stream);
    return a.bf16 ? launch_fwd_variant<64, true, 4, 4>(a, stream)
                  : launch_fwd_variant<64, false, 4, 4>(a, stream);
  }
  if (a.d == 128)
    return a.bf16 ? launch_fwd_variant<128, true, 3, 2>(a, stream)
                  : launch_fwd_variant<128, false, 3, 2>(a, stream);
  return -2;
}

}  // namespace attn
