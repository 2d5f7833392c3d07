// Prefill forward for head dimension 64: two query tiles per work item, sm_103a.
//
// The structure of FlashAttention-4 ("FlashAttention Explained", section on FlashAttention-4:
// two query tiles ping-ponged in tensor memory): a work item is a pair of 128-row query tiles
// that read the same key/value plane, and each K/V tile that lands in shared memory serves
// both.  Softmax warpgroup w owns query tile w of the pair outright: its S buffer, its P
// buffer, its accumulator O_w and its running (m, l), so the two warpgroups never wait for
// each other.  At d = 64 tensor memory holds all of it with P in its own columns: S_0 and S_1
// at columns 0 and 128, O_0 and O_1 at 256 and 320, P_0 and P_1 at 384 and 448.  (At d = 128
// the two accumulators leave no room for P beside S, and P written over S puts the next score
// MMA behind the previous P V on every tile; that kernel keeps one query tile per item.)
//
// Pairs: with grouped-query heads, two query heads of one key/value head at the same query
// tile (identical key ranges and masks); otherwise two consecutive query tiles of one head
// (under the causal mask the upper tile sees one key tile more).  Items run longest first over
// groups of pairs whose K/V planes fill about half of L2, as in the d = 128 kernel; a running
// block takes over the items of blocks not yet started (cluster launch control), so each SM
// runs one long-lived block whose pipelines run on from one item into the next.
//
// Roles (384 threads): warps 0-3 and 4-7 the softmax warpgroups of query tiles 0 and 1
// (thread = query row); warp 8 the scheduler and the TMA producer of Q (double-buffered by item
// parity) and of the K and V rings; warp 9 issues S_w = Q_w K^T for both tiles (and owns tensor
// memory); warps 10 and 11 issue O_0 += P_0 V and O_1 += P_1 V, one each, so that neither tile's
// P V queues behind the other's (a thread pushing eight MMAs through the pipe's short queue
// is busy for hundreds of cycles).  The online-softmax step, the conditional rescale (only when
// the row maximum rises by more than 2^8) and the epilogue O = a / l, L = m + ln l are those of
// the d = 128 kernel ("FlashAttention and GPU Data Movement", section 3.1).
#include <atomic>

#include "internal.h"
#include "ptx.cuh"

namespace attn {

namespace {

constexpr int kD = 64;
constexpr int kTm = 128;  // query rows of a tile
constexpr int kTn = 128;  // keys of a key tile
constexpr int kThreads = 384;
constexpr int kSoftmaxThreads = 128;
constexpr int kProducerWarp = 8, kQkWarp = 9, kPvWarp0 = 10, kPvWarp1 = 11;
constexpr uint32_t kItemReaders = 3 + 8;  // lane 0 of warps 9, 10, 11 and of each softmax warp
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kRegsSoftmax = 184, kRegsIssue = 136;
static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsIssue <= kThreads * 168, "register split");
constexpr uint32_t kColS = 0, kColO = 256, kColP = 384;  // + 128 w, + 64 w, + 64 w
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr uint32_t kTile = kTm * kD * 2;   // bytes of a Q, K or V tile (one swizzled sub-tile)
constexpr int KS = 4, VS = 4;              // K and V ring slots
static_assert(KS == VS, "one producer loop fills both rings slot by slot");
constexpr uint64_t kDrainLimitNs = 100000000ull;

struct PairParams {
  void* o;
  float* lse;
  int* status;
  int Hq, Hkv, N_q, N_kv, G, n_qtiles, causal, window, n_kvtiles;
  const uint8_t* block_mask;  // [query tile][key tile], nonzero = compute; null: every tile
  int pair_heads;  // 1: two query heads of a key/value head; 0: two query tiles of one head
  int Gp;          // head pairs per key/value head (pair_heads)
  int n_lanes;     // (batch, key/value head, head pair) or (batch, query head)
  int n_depth;     // query tiles, or query-tile pairs, per lane
  int lane_group;  // lanes walked together, longest items first
  float sl2;       // scale * log2(e)
};

// Barriers (8 bytes each) after the K/V rings; [2] = per query tile w or per item parity.
enum PairBar : uint32_t {
  kBarQFull = 0,      // [2] an item's Q tiles landed, by item parity
  kBarQEmpty = 2,     // [2] the item's last score MMA finished
  kBarSFull = 4,      // [2] S_w written (MMA commit)
  kBarSFree = 6,      // [2] S_w read (128 arrivals)
  kBarPReady = 8,     // [2] P_w written, O_w rescaled (128 arrivals)
  kBarPDone = 10,     // [2] P_w V finished (MMA commit): P_w free, O_w up to date
  kBarODrained = 12,  // [2] O_w read out by the item's epilogue (128 arrivals)
  kBarItemFull = 14,  // [2] work-item ring slot written
  kBarItemEmpty = 16, // [2] ... and read by every role
  kBarClc = 18,       // cluster-launch-control answer landed
  kBarDrain = 19,     // the three issuers' MMAs finished (three commits)
  kNumFixedBars = 20
};

struct PairLayout {
  static constexpr uint32_t kQ = 0;                      // [item parity][w] Q tiles
  static constexpr uint32_t kK = kQ + 4 * kTile;         // K ring
  static constexpr uint32_t kV = kK + KS * kTile;        // V ring
  static constexpr uint32_t kBar = kV + VS * kTile;      // k_full, k_empty, v_full, v_empty
  static constexpr uint32_t kFixedBar = kBar + 2 * (KS + VS) * 8;
  static constexpr uint32_t kMisc = kFixedBar + kNumFixedBars * 8;  // tmem slot, abort, ring[2]
  static constexpr uint32_t kClc = (kMisc + 16 + 15) & ~15u;
  static constexpr uint32_t kBytes = kClc + 16 + 1024;  // + alignment slack
  static_assert(kBytes <= 232448, "shared memory per block");
};

// One query tile of a work item.
struct PairTile {
  int bh;            // batch * Hq + query head
  int q0;            // first query row
  int j0, j1;        // key tiles [j0, j1) hold every key this tile's rows see
  int lo_masked;     // key tiles below this need the window's lower-edge mask
  int first_masked;  // key tiles from this on need the causal or ragged-edge mask
  const uint8_t* pattern;  // this query tile's row of the block pattern, or null
  bool valid;        // the pair has this tile (an odd tail leaves the second one out)
};

struct PairItem {
  int kv_plane;
  int u0, u1;  // key tiles [u0, u1) span both tiles' ranges
  PairTile t[2];
};

__device__ __forceinline__ bool tile_sees(const PairTile& t, int j) {
  return j >= t.j0 && j < t.j1 && (!t.pattern || t.pattern[j]);
}

__device__ __forceinline__ bool pair_sees(const PairItem& it, int j) {
  return tile_sees(it.t[0], j) || tile_sees(it.t[1], j);
}

// Work item `id` in launch order: lanes are cut into groups of lane_group; a group's items run
// longest first across its lanes (under the causal mask a query tile's key range grows with its
// row index).
__device__ __forceinline__ PairItem decode_pair(int id, const PairParams& p) {
  PairItem it;
  const int span = p.lane_group * p.n_depth;
  const int g = id / span;
  const int r = id - g * span;
  const int l0 = g * p.lane_group;
  const int gl = min(p.lane_group, p.n_lanes - l0);
  const int depth = p.n_depth - 1 - r / gl;
  const int lane = l0 + r % gl;
  int bh[2], qt[2];
  bool valid[2];
  if (p.pair_heads) {
    const int bkv = lane / p.Gp;
    const int m = lane - bkv * p.Gp;
    const int b = bkv / p.Hkv, hk = bkv % p.Hkv;
    bh[0] = b * p.Hq + hk * p.G + 2 * m;
    bh[1] = bh[0] + 1;
    qt[0] = qt[1] = depth;
    valid[0] = true;
    valid[1] = 2 * m + 1 < p.G;
    it.kv_plane = bkv;
  } else {
    bh[0] = bh[1] = lane;
    qt[0] = 2 * depth;
    qt[1] = 2 * depth + 1;
    valid[0] = true;
    valid[1] = qt[1] < p.n_qtiles;
    it.kv_plane = (lane / p.Hq) * p.Hkv + (lane % p.Hq) / p.G;
  }
  it.u0 = 0x7fffffff;
  it.u1 = 0;
#pragma unroll
  for (int w = 0; w < 2; ++w) {
    PairTile& t = it.t[w];
    t.bh = bh[w];
    t.q0 = qt[w] * kTm;
    t.valid = valid[w];
    t.pattern = nullptr;
    if (valid[w]) {
      kv_tile_span(qt[w], kTm, kTn, p.N_q, p.N_kv, p.causal, p.window, t.j0, t.j1, t.lo_masked,
                   t.first_masked);
      if (p.block_mask) t.pattern = p.block_mask + static_cast<size_t>(qt[w]) * p.n_kvtiles;
    } else {
      t.j0 = t.j1 = t.lo_masked = t.first_masked = 0;
    }
    if (t.j0 < t.j1) {
      it.u0 = min(it.u0, t.j0);
      it.u1 = max(it.u1, t.j1);
    }
  }
  if (it.u1 == 0) it.u0 = 0;
  return it;
}

// The last key tile of the item's sequence (-1: the item has none).
__device__ __forceinline__ int last_pair_tile(const PairItem& it) {
  for (int j = it.u1 - 1; j >= it.u0; --j)
    if (pair_sees(it, j)) return j;
  return -1;
}

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                          int* status) {
  const bool ok = wait_bounded(bar, parity, abort, status);
  return __all_sync(0xffffffffu, ok);
}

template <bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_pair_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const PairParams p) {
  using L = PairLayout;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t sQ = base + L::kQ;
  const uint32_t sK = base + L::kK;
  const uint32_t sV = base + L::kV;
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

  if (threadIdx.x == 0) {
    for (int s = 0; s < KS; ++s) {
      mbar_init(BAR_K(s), 1);
      mbar_init(BAR_KE(s), 1);
    }
    for (int s = 0; s < VS; ++s) {
      mbar_init(BAR_V(s), 1);
      mbar_init(BAR_VE(s), 2);  // both P V issuers
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(FBAR(kBarQFull + b), 1);
      mbar_init(FBAR(kBarQEmpty + b), 1);
      mbar_init(FBAR(kBarSFull + b), 1);
      mbar_init(FBAR(kBarSFree + b), kSoftmaxThreads);
      mbar_init(FBAR(kBarPReady + b), kSoftmaxThreads);
      mbar_init(FBAR(kBarPDone + b), 1);
      mbar_init(FBAR(kBarODrained + b), kSoftmaxThreads);
      mbar_init(FBAR(kBarItemFull + b), 1);
      mbar_init(FBAR(kBarItemEmpty + b), kItemReaders);
    }
    mbar_init(FBAR(kBarClc), 1);
    mbar_init(FBAR(kBarDrain), 3);
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

  auto take_item = [&](int k, int& id) -> bool {
    if (!wait_bounded(FBAR(kBarItemFull + (k & 1)), (k >> 1) & 1, abort_flag, p.status))
      return false;
    id = ring[k & 1];
    mbar_arrive(FBAR(kBarItemEmpty + (k & 1)));
    return true;
  };

  if (warp >= kProducerWarp) {
    setmaxnreg_dec<kRegsIssue>();
    if (warp == kProducerWarp) {
      // ------------------------------------------------------------- scheduler + producer
      // Publishes the block's work items (its own first, then those of pending blocks it
      // cancels) and loads, per item, the K and V tiles of its sequence, with the item's Q
      // tiles after its first K tile (Q buffer by item parity, refilled once the score MMAs of
      // the item two back finished).  The next item is asked for with the item's last K load;
      // as soon as the answer is in, its Q tiles are pulled into L2.
      if (lane == 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        int id = static_cast<int>(blockIdx.x);
        int next_id = -1;
        bool clc_live = true, clc_pending = false;
        uint32_t clc_uses = 0;
        auto request_next = [&]() {
          if (clc_live) {
            mbar_arrive_expect_tx(FBAR(kBarClc), 16);
            clc_try_cancel(clc_resp, FBAR(kBarClc));
            clc_pending = true;
          }
        };
        auto take_answer = [&]() {
          clc_pending = false;
          ++clc_uses;
          int x;
          if (clc_query(clc_resp, x)) {
            next_id = x;
            const PairItem nx = decode_pair(x, p);
#pragma unroll
            for (int w = 0; w < 2; ++w)
              if (nx.t[w].valid && nx.t[w].j0 < nx.t[w].j1)
                tma_prefetch_l2_3d(&tm_q, 0, nx.t[w].q0, nx.t[w].bh);
          } else {
            next_id = -1;
            clc_live = false;
          }
        };
        int T = 0, kq = 0;  // K tiles loaded, items with tiles loaded
        bool ok = true;
        for (int k = 0; ok; ++k) {
          if (k >= 2 && !wait_bounded(FBAR(kBarItemEmpty + (k & 1)), ((k >> 1) - 1) & 1,
                                      abort_flag, p.status)) {
            ok = false;
            break;
          }
          ring[k & 1] = id;
          mbar_arrive(FBAR(kBarItemFull + (k & 1)));
          if (id < 0) break;
          next_id = -1;
          const PairItem it = decode_pair(id, p);
          const int j_last = last_pair_tile(it);
          if (j_last < 0) request_next();
          bool first = true;
          for (int j = it.u0; j_last >= 0 && j <= j_last; ++j) {
            if (!pair_sees(it, j)) continue;
            // slot s of both rings (they have the same depth): K once the score products of its
            // previous tile finished, V once both P V products of its previous tile did; both
            // waits come before either load, so that a wait that runs out leaves no copy that
            // the drain below would miss
            const int s = T % KS;
            if (T >= KS && (!wait_bounded(BAR_KE(s), ((T / KS) - 1) & 1, abort_flag, p.status) ||
                            !wait_bounded(BAR_VE(s), ((T / VS) - 1) & 1, abort_flag, p.status))) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(BAR_K(s), kTile);
            tma_load_3d(sK + s * kTile, &tm_k, BAR_K(s), 0, j * kTn, it.kv_plane);
            mbar_arrive_expect_tx(BAR_V(s), kTile);
            tma_load_3d(sV + s * kTile, &tm_v, BAR_V(s), 0, j * kTn, it.kv_plane);
            ++T;
            if (first) {
              first = false;
              const int qb = kq & 1;
              if (kq >= 2 &&
                  !wait_bounded(FBAR(kBarQEmpty + qb), ((kq >> 1) - 1) & 1, abort_flag, p.status)) {
                ok = false;
                break;
              }
              const uint32_t bytes = (it.t[1].valid ? 2u : 1u) * kTile;
              mbar_arrive_expect_tx(FBAR(kBarQFull + qb), bytes);
#pragma unroll
              for (int w = 0; w < 2; ++w)
                if (it.t[w].valid)
                  tma_load_3d(sQ + (qb * 2 + w) * kTile, &tm_q, FBAR(kBarQFull + qb), 0, it.t[w].q0,
                              it.t[w].bh);
              ++kq;
            }
            if (j == j_last) request_next();
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
        // every asynchronous write into this block's shared memory lands before it may exit
        for (int t = (T > KS ? T - KS : 0); t < T; ++t) {
          wait_bounded(BAR_K(t % KS), (t / KS) & 1, nullptr, p.status, kDrainLimitNs);
          wait_bounded(BAR_V(t % VS), (t / VS) & 1, nullptr, p.status, kDrainLimitNs);
        }
        for (int q = (kq > 2 ? kq - 2 : 0); q < kq; ++q)
          wait_bounded(FBAR(kBarQFull + (q & 1)), (q >> 1) & 1, nullptr, p.status, kDrainLimitNs);
        if (clc_pending)
          wait_bounded(FBAR(kBarClc), clc_uses & 1, nullptr, p.status, kDrainLimitNs);
      }
      __syncwarp();
    } else {
      // ------------------------------------------------------------- tcgen05 issuers
      // Warp 9: for each key tile of an item, S_w = Q_w K^T for the tiles w that see it, each
      // once warpgroup w has read its previous S.  Warp 10 + w: O_w (+)= P_w V for the key
      // tiles query tile w sees, each once P_w is stored; the first of an item overwrites O_w,
      // after the previous item's epilogue has read it out.  Each P V issuer arrives on every
      // V slot's release once per key tile of the sequence, after seeing that slot's load (so
      // that its arrival never counts toward the slot's previous use).
      if (lane == 0) {
        const bool qk_issuer = (warp == kQkWarp);
        static_assert(kPvWarp1 == kPvWarp0 + 1, "P V issuers of query tiles 0 and 1");
        const int pw = qk_issuer ? 0 : warp - kPvWarp0;  // the P V issuer's query tile
        constexpr uint32_t idesc_qk = make_idesc_f16(BF16, kTm, kTn, false);
        constexpr uint32_t idesc_pv = make_idesc_f16(BF16, kTm, kD, true);
        int T = 0, kq = 0;
        int used[2] = {0, 0};  // score products issued per query tile w (score issuer)
        int pv_used = 0;       // P V products issued (P V issuer)
        int pv_items = 0;      // items in which the issuer's query tile had a key tile
        bool ok = true;
        for (int k = 0; ok; ++k) {
          int id;
          if (!take_item(k, id)) break;
          if (id < 0) break;
          const PairItem it = decode_pair(id, p);
          const int j_last = last_pair_tile(it);
          if (j_last < 0) continue;
          const PairTile mine = pw ? it.t[1] : it.t[0];  // the P V issuer's query tile
          const int qb = kq & 1;
          if (qk_issuer && !wait_bounded(FBAR(kBarQFull + qb), (kq >> 1) & 1, abort_flag, p.status))
            break;
          bool pv_first = true;
          for (int j = it.u0; ok && j <= j_last; ++j) {
            if (!pair_sees(it, j)) continue;
            if (qk_issuer) {
              const int s = T % KS;
              bool waited = false;
#pragma unroll
              for (int w = 0; w < 2; ++w) {
                if (!tile_sees(it.t[w], j)) continue;
                if (used[w] >= 1 && !wait_bounded(FBAR(kBarSFree + w), (used[w] - 1) & 1,
                                                  abort_flag, p.status)) {
                  ok = false;
                  break;
                }
                if (!waited) {
                  if (!wait_bounded(BAR_K(s), (T / KS) & 1, abort_flag, p.status)) {
                    ok = false;
                    break;
                  }
                  waited = true;
                }
                tc_fence_after();
                const uint32_t q_tile = sQ + (qb * 2 + w) * kTile;
#pragma unroll
                for (int kk = 0; kk < kD / 16; ++kk) {
                  const uint64_t adesc = make_sdesc_sw128(q_tile + kk * 32, 16, 1024);
                  const uint64_t bdesc = make_sdesc_sw128(sK + s * kTile + kk * 32, 16, 1024);
                  mma_ss(tmem + kColS + 128u * w, adesc, bdesc, idesc_qk, kk > 0 ? 1u : 0u);
                }
                mma_commit(FBAR(kBarSFull + w));
                ++used[w];
              }
              if (!ok) break;
              mma_commit(BAR_KE(s));  // K slot free
            } else {
              const int s = T % VS;
              if (!wait_bounded(BAR_V(s), (T / VS) & 1, abort_flag, p.status)) {
                ok = false;
                break;
              }
              if (!tile_sees(mine, j)) {
                mbar_arrive(BAR_VE(s));  // nothing of this issuer reads the slot
              } else {
                if (!wait_bounded(FBAR(kBarPReady + pw), pv_used & 1, abort_flag, p.status) ||
                    (pv_first && pv_items >= 1 &&
                     !wait_bounded(FBAR(kBarODrained + pw), (pv_items - 1) & 1, abort_flag,
                                   p.status))) {
                  ok = false;
                  break;
                }
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kTn / 16; ++kk) {
                  // V [keys, d], d contiguous: the MN-major B operand, 16 keys per MMA
                  const uint64_t bdesc =
                      make_sdesc_sw128(sV + s * kTile + kk * 16 * 128, 128 * 128, 1024);
                  mma_ts(tmem + kColO + 64u * pw, tmem + kColP + 64u * pw + kk * 8, bdesc,
                         idesc_pv, (!pv_first || kk > 0) ? 1u : 0u);
                }
                mma_commit(FBAR(kBarPDone + pw));
                mma_commit(BAR_VE(s));  // this issuer's reads of the V slot done
                pv_first = false;
                ++pv_used;
              }
            }
            ++T;
          }
          if (!ok) break;
          if (qk_issuer) {
            mma_commit(FBAR(kBarQEmpty + qb));  // Q buffer free once these MMAs finished
          } else if (!pv_first) {
            ++pv_items;
          }
          ++kq;
        }
        // every MMA this thread issued completes before the block frees tensor memory
        if (T > 0 && (qk_issuer || pv_used > 0))
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
    // ------------------------------------------------------------- softmax + epilogue
    // Warpgroup w takes query tile w of every item; thread r owns row r (warp % 4 is its
    // tensor-memory lane quarter).  Per key tile: read S_w and release it (the next score MMA
    // may overwrite it), the mask, the row maximum, the running maximum (moved only when it
    // rises by more than 2^8), p = 2^(x scale log2(e) - m), the row sum, P_w, and the rescale of
    // O_w when the maximum moved.  Per item: O = a / l and L = m + ln l.
    const int w = warp >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t row_tmem = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t s_tmem = row_tmem + kColS + 128u * w;
    const uint32_t o_tmem = row_tmem + kColO + 64u * w;
    const uint32_t p_tmem = row_tmem + kColP + 64u * w;
    const int off = p.N_kv - p.N_q;
    const float sl2 = p.sl2;
    const int n_kv = p.N_kv, causal = p.causal, window = p.window;
    int used = 0;  // key tiles this warpgroup has processed
    bool ok = true;
    for (int k = 0; ok; ++k) {
      if (!warp_wait(FBAR(kBarItemFull + (k & 1)), (k >> 1) & 1, abort_flag, p.status)) break;
      const int id = ring[k & 1];
      __syncwarp();
      if (lane == 0) mbar_arrive(FBAR(kBarItemEmpty + (k & 1)));
      if (id < 0) break;
      const PairItem it = decode_pair(id, p);
      const PairTile tt = w ? it.t[1] : it.t[0];  // (a select keeps it out of local memory)
      if (!tt.valid) continue;
      const int row = tt.q0 + r;
      float m_run = -INFINITY;  // running maximum (log2 units) of this row
      float l = 0.0f;           // sum of 2^(x - m_run)
      int i = 0;                // key tiles of this item processed
      for (int j = tt.j0; j < tt.j1; ++j) {
        if (tt.pattern && !tt.pattern[j]) continue;
        if (!warp_wait(FBAR(kBarSFull + w), used & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(s_tmem + c * 32, sr[c]);
        tmem_wait_ld();
        tc_fence_before();
        mbar_arrive(FBAR(kBarSFree + w));  // S_w free for the next score MMA
        float x[kTn];
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int e = 0; e < 32; ++e) x[c * 32 + e] = __uint_as_float(sr[c][e]);
        if (j >= tt.first_masked || j < tt.lo_masked) {
          // visible columns [lo, hi] of this row in this tile, as four 32-column bit masks
          int hi = kTn - 1, lo = 0;
          if (j >= tt.first_masked) {
            int lim = causal ? row + off : n_kv - 1;
            if (lim > n_kv - 1) lim = n_kv - 1;
            hi = min(lim - j * kTn, kTn - 1);
          }
          if (j < tt.lo_masked) lo = max(row + off - window - j * kTn, 0);
          uint32_t vis[kTn / 32];
#pragma unroll
          for (int g = 0; g < kTn / 32; ++g) {
            const int a = max(lo - 32 * g, 0), bb = min(hi - 32 * g, 31);
            vis[g] = (a > bb) ? 0u : ((0xffffffffu >> (31 - bb)) & (0xffffffffu << a));
          }
#pragma unroll
          for (int c = 0; c < kTn; ++c)
            x[c] += __uint_as_float((((vis[c >> 5] >> (c & 31)) & 1u) - 1u) & 0xff800000u);
        }
        float mx[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) mx[e] = fmaxf(x[e], x[16 + e]);
#pragma unroll
        for (int c = 32; c < kTn; c += 32)
#pragma unroll
          for (int e = 0; e < 16; ++e) mx[e] = max3f(mx[e], x[c + e], x[c + 16 + e]);
#pragma unroll
        for (int e = 0; e < 8; ++e) mx[e] = fmaxf(mx[e], mx[e + 8]);
        const float tile_max = max3f(max3f(mx[0], mx[1], mx[2]), max3f(mx[3], mx[4], mx[5]),
                                     fmaxf(mx[6], mx[7]));
        float alpha = 1.0f;
        const float m_new = fmaxf(m_run, tile_max * sl2);
        if (m_new - m_run > kRescaleThreshold) {
          alpha = ex2(m_run - m_new);
          l *= alpha;  // (0 while m_run is -inf)
          m_run = m_new;
        }
        const float neg_mu = (m_run == -INFINITY) ? 0.0f : -m_run;
#pragma unroll
        for (int c = 0; c < kTn; c += 2) {
          float a0, a1;
          fma2(a0, a1, x[c], x[c + 1], sl2, sl2, neg_mu, neg_mu);
          x[c] = ex2(a0);
          x[c + 1] = ex2(a1);
        }
        float ps[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        uint32_t pk[2][32];
#pragma unroll
        for (int c = 0; c < kTn; c += 4) {
          const float p0 = x[c], p1 = x[c + 1], p2 = x[c + 2], p3 = x[c + 3];
          const int k2 = ((c >> 1) & 3) * 2;
          add2(ps[k2], ps[k2 + 1], p0, p1);
          add2(ps[k2 + 2], ps[k2 + 3], p2, p3);
          pk[c >> 6][(c >> 1) & 31] = pack2<BF16>(p0, p1);
          pk[c >> 6][((c >> 1) & 31) + 1] = pack2<BF16>(p2, p3);
        }
        l += ((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7]));
        // P_w V of the previous key tile has finished: P_w is free and O_w up to date
        if (used >= 1 &&
            !warp_wait(FBAR(kBarPDone + w), (used - 1) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        tmem_st32(p_tmem, pk[0]);
        tmem_st32(p_tmem + 32, pk[1]);
        if (i > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll 1
          for (int c = 0; c < kD / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(o_tmem + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(o_tmem + c * 32, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(FBAR(kBarPReady + w));
        ++used;
        ++i;
      }
      if (!ok) break;
      uint16_t* orow = static_cast<uint16_t*>(p.o) + (static_cast<size_t>(tt.bh) * p.N_q + row) * kD;
      float* lrow = p.lse + static_cast<size_t>(tt.bh) * p.N_q + row;
      if (i == 0) {
        // no key visible to any row of this tile: O = 0, L = -inf
        if (row < p.N_q) {
#pragma unroll
          for (int c = 0; c < kD / 8; ++c) reinterpret_cast<uint4*>(orow)[c] = make_uint4(0, 0, 0, 0);
          *lrow = -INFINITY;
        }
        continue;
      }
      // epilogue: the last P_w V has finished; the accumulator out, then O = a / l
      if (!warp_wait(FBAR(kBarPDone + w), (used - 1) & 1, abort_flag, p.status)) break;
      tc_fence_after();
      uint32_t oa[2][32];
      tmem_ld32(o_tmem, oa[0]);
      tmem_ld32(o_tmem + 32, oa[1]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(FBAR(kBarODrained + w));  // the next item's first P_w V may overwrite O_w
      if (row < p.N_q) {
        const float inv_l = (l > 0.0f) ? 1.0f / l : 0.0f;
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint4 v4;
            v4.x = pack2<BF16>(__uint_as_float(oa[c][q4 * 8 + 0]) * inv_l,
                               __uint_as_float(oa[c][q4 * 8 + 1]) * inv_l);
            v4.y = pack2<BF16>(__uint_as_float(oa[c][q4 * 8 + 2]) * inv_l,
                               __uint_as_float(oa[c][q4 * 8 + 3]) * inv_l);
            v4.z = pack2<BF16>(__uint_as_float(oa[c][q4 * 8 + 4]) * inv_l,
                               __uint_as_float(oa[c][q4 * 8 + 5]) * inv_l);
            v4.w = pack2<BF16>(__uint_as_float(oa[c][q4 * 8 + 6]) * inv_l,
                               __uint_as_float(oa[c][q4 * 8 + 7]) * inv_l);
            reinterpret_cast<uint4*>(orow)[c * 4 + q4] = v4;
          }
        const float mu = (m_run == -INFINITY) ? 0.0f : m_run;
        *lrow = (l > 0.0f) ? (mu + lg2(l)) * 0.69314718055994531f : -INFINITY;
      }
    }
    tc_fence_before();
    __syncthreads();  // the producer warpgroup's matching barrier ends its branch
  }
#undef BAR_K
#undef BAR_KE
#undef BAR_V
#undef BAR_VE
#undef FBAR
}

template <bool BF16>
int launch_pair(const FwdArgs& a, cudaStream_t stream) {
  using L = PairLayout;
  CUtensorMap tq, tk, tv;
  const uint64_t bhq = static_cast<uint64_t>(a.B) * a.Hq;
  const uint64_t bhk = static_cast<uint64_t>(a.B) * a.Hkv;
  const uint64_t rb = static_cast<uint64_t>(kD) * 2;
  if (!make_tmap_3d(&tq, a.q, BF16, kD, a.N_q, bhq, rb, rb * a.N_q, 64, kTm, 1) ||
      !make_tmap_3d(&tk, a.k, BF16, kD, a.N_kv, bhk, rb, rb * a.N_kv, 64, kTn, 1) ||
      !make_tmap_3d(&tv, a.v, BF16, kD, a.N_kv, bhk, rb, rb * a.N_kv, 64, kTn, 1))
    return -5;
  PairParams p;
  p.o = a.o;
  p.lse = a.lse;
  p.status = device_status_ptr();
  if (!p.status) return -5;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.N_q = a.N_q;
  p.N_kv = a.N_kv;
  p.G = a.Hq / a.Hkv;
  p.n_qtiles = (a.N_q + kTm - 1) / kTm;
  p.causal = (a.causal || a.window >= 0) ? 1 : 0;
  p.window = a.window;
  p.n_kvtiles = (a.N_kv + kTn - 1) / kTn;
  p.block_mask = a.block_mask;
  p.pair_heads = p.G >= 2 ? 1 : 0;
  p.Gp = (p.G + 1) / 2;
  const uint64_t lanes = p.pair_heads ? bhk * p.Gp : bhq;
  const uint64_t depth = p.pair_heads ? p.n_qtiles : (p.n_qtiles + 1) / 2;
  if (lanes * depth > 0x7fffffffull) return -2;
  p.n_lanes = static_cast<int>(lanes);
  p.n_depth = static_cast<int>(depth);
  {
    // lanes whose K/V planes fill about half of L2 (every lane of a plane together)
    static std::atomic<int> l2_bytes{-1};
    if (l2_bytes.load() < 0) {
      int dev = 0, v = 0;
      if (cudaGetDevice(&dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&v, cudaDevAttrL2CacheSize, dev) != cudaSuccess || v <= 0)
        v = 64 << 20;
      l2_bytes.store(v);
    }
    const uint64_t plane_bytes = 2ull * a.N_kv * kD * 2;
    uint64_t planes = (static_cast<uint64_t>(l2_bytes.load()) / 2) / plane_bytes;
    if (planes < 1) planes = 1;
    uint64_t lg = planes * (p.pair_heads ? static_cast<uint64_t>(p.Gp) : 1ull);
    if (lg > lanes) lg = lanes;
    p.lane_group = static_cast<int>(lg);
  }
  p.sl2 = a.scale * 1.4426950408889634f;
  auto kern = attn_fwd_pair_kernel<BF16>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes) !=
      cudaSuccess)
    return -5;
  // one block per work item; the running blocks take over the items of the others
  kern<<<static_cast<unsigned>(lanes * depth), kThreads, L::kBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? 0 : -5;
}

}  // namespace

int launch_attn_fwd_pair(const FwdArgs& a, cudaStream_t stream) {
  if (a.d != kD) return -2;
  return a.bf16 ? launch_pair<true>(a, stream) : launch_pair<false>(a, stream);
}

}  // namespace attn
