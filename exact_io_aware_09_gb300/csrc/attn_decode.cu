// Split-KV decode: one new query token per sequence attends to its whole packed KV cache.
//
// "FlashAttention Explained", section "Decoding, Paged and Split-KV Variants", and "FlashAttention
// and GPU Data Movement", section 6.1: with one query row the query axis gives no parallelism, so
// the key/value sequence is split into chunks processed by separate thread blocks; each chunk
// yields a partial state (m, l, o) and the partial states are merged exactly with the block-merge
// rule of "How FlashAttention Reduces HBM Traffic Exactly", section "Why softmax does not prevent
// tiling".
//
// Kernel 1 (split): block (split s, key/value head hk, sequence b).  A producer warp streams the
// chunk's K and V rows of head hk through a ring of 64-token stages with TMA (the cache is
// [tokens, Hkv, d], so one stage is 64 strided 2*d-byte rows per tensor).  Four compute warps
// each take 16 tokens of every stage and run the online softmax for the G = Hq/Hkv query heads
// that share hk.  The per-token work is tiny (8 FLOP per cache byte) and the kernel is bound by
// HBM, so the two small products run on warp-level mma.sync tiles (m16n8k16, query heads padded
// to 16 rows) straight from the swizzled stage buffers.  The four warps' states are merged in
// shared memory and the chunk's normalised (m, l, o) is written to the workspace.
// Kernel 2 (merge): one block per (sequence, query head) merges that row's chunk states.
//
// Paged cache ("FlashAttention Explained", section "Decoding, Paged and Split-KV Variants": the
// cache in fixed-size non-contiguous blocks addressed through a block table, read by a split-KV
// kernel): the same kernels with the producer reading each stage through the block table -- one
// TMA box per stage when a page holds a whole 64-token stage, one box per page otherwise -- and
// the sequence length taken from seqlens.  The cache is seen by TMA as a 4-D tensor {64
// channels, token, channel half, head}, so that one box brings both 64-channel halves of its
// rows: a stage holds R-row boxes (R = min(page size, 64); 64 for the packed cache) laid out
// [box][half][R rows][128 B], and a 16-token page costs one TMA operation per tensor instead of
// two.
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace attn {

constexpr int kDecTok = 64;      // tokens per ring stage
constexpr int kDecWarps = 4;     // compute warps, 16 tokens of each stage apiece
constexpr int kDecThreads = 160;  // + one producer warp
constexpr int kDecStages = 3;
constexpr int kMaxGroup = 16;    // query heads per key/value head (rows of the m16 tile)

struct DecParams {
  const uint16_t* q;   // [B, Hq, D]
  const int32_t* cu;   // [B + 1] (packed cache)
  const int32_t* block_table;  // [B, max_pages] (paged cache) or null
  const int32_t* seqlens;      // [B] (paged cache)
  int page_size, page_log2, max_pages, num_pages;
  int box_log2;        // log2 of the rows of one TMA box: min(page_size, 64); 64 when packed
  float* ws_o;         // [B * Hq * max_splits, D]  normalised partial outputs
  float* ws_ml;        // [B * Hq * max_splits, 2]  (m in log2 units, l)
  int* status;
  int Hq, Hkv, G, capacity, max_seqlen, split, max_splits;
  float sl2;
};

template <int D>
struct DecLayout {
  static constexpr uint32_t kHalf = kDecTok * 128;             // one 64-column half of a stage
  static constexpr uint32_t kTensor = (D / 64) * kHalf;         // K or V of one stage
  static constexpr uint32_t kStage = 2 * kTensor;
  static constexpr uint32_t kRing = kDecStages * kStage;
  static constexpr uint32_t kRed = kDecWarps * kMaxGroup * (D + 2) * 4;  // reuses the ring
  static_assert(kRed <= kRing, "merge scratch must fit in the ring");
  static constexpr uint32_t kBar = kRing;                        // full[S], empty[S]
  static constexpr uint32_t kMisc = kBar + 2 * kDecStages * 8;   // abort flag
  // paged cache: first cache row of every page of the split (-1: not loaded)
  static constexpr uint32_t kPages = kMisc + 16;
  static constexpr int kMaxSplitPages = 8192 / 16;
  static constexpr uint32_t kBytes = kPages + kMaxSplitPages * 4 + 1024;
};

__device__ __forceinline__ bool dec_warp_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                              int* status) {
  const bool ok = wait_bounded(bar, parity, abort, status);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ bool lengths_ok(const DecParams& p, int t_start, int t_stop) {
  const int len = t_stop - t_start;
  return t_start >= 0 && len >= 0 && len <= p.max_seqlen && t_stop <= p.capacity;
}

// Sequence b's tokens: rows [t_start, t_stop) of the packed cache, or logical positions
// [0, seqlens[b]) of a paged one.  False for lengths the caller's bounds do not allow.
__device__ __forceinline__ bool seq_bounds(const DecParams& p, int b, int& t_start, int& t_stop) {
  if (p.block_table) {
    t_start = 0;
    t_stop = p.seqlens[b];
    return t_stop >= 0 && t_stop <= p.max_seqlen &&
           ((t_stop + p.page_size - 1) >> p.page_log2) <= p.max_pages;
  }
  t_start = p.cu[b];
  t_stop = p.cu[b + 1];
  return lengths_ok(p, t_start, t_stop);
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kDecThreads)
    attn_decode_split_kernel(const __grid_constant__ CUtensorMap tm_k,
                             const __grid_constant__ CUtensorMap tm_v, const DecParams p) {
  using L = DecLayout<D>;
  const int split = blockIdx.x;
  const int hk = blockIdx.y;
  const int b = blockIdx.z;
  // the merge kernel may be scheduled once every block of this grid has started (it waits for
  // this grid's completion before reading anything)
  if (threadIdx.x == 0) griddep_launch_dependents();
  int t_start, t_stop;
  if (!seq_bounds(p, b, t_start, t_stop)) {
    if (split == 0 && hk == 0 && threadIdx.x == 0) latch_status(p.status, kStatusBadLengths);
    return;
  }
  const int len = t_stop - t_start;
  const int n_splits = (len + p.split - 1) / p.split;
  if (split >= n_splits) return;
  const int t0 = t_start + split * p.split;
  const int n_tok = min(p.split, t_stop - t0);
  const int n_stages = (n_tok + kDecTok - 1) / kDecTok;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bars = base + L::kBar;
#define FULL(s) (bars + 8u * (s))
#define EMPTY(s) (bars + 8u * (kDecStages + (s)))
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L::kMisc);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kDecStages; ++s) {
      mbar_init(FULL(s), 1);
      mbar_init(EMPTY(s), kDecWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == kDecWarps) {
    // ------------------------------------------------------------------ TMA producer
    int* page_row = reinterpret_cast<int*>(gbase + L::kPages);
    if (p.block_table) {
      // The split's block-table entries, read once by the whole warp: the first cache row of
      // each page that holds tokens of the split, or -1 for an entry outside the pool (reported).
      const int32_t* tbl = p.block_table + static_cast<size_t>(b) * p.max_pages;
      const int first = t0 >> p.page_log2;
      const int n_pg = ((t0 + n_tok - 1) >> p.page_log2) - first + 1;
      for (int i = lane; i < n_pg; i += 32) {
        const int pg = tbl[first + i];
        const bool good = pg >= 0 && pg < p.num_pages;
        if (!good) latch_status(p.status, kStatusBadLengths);
        page_row[i] = good ? pg * p.page_size : -1;
      }
      __syncwarp();
    }
    // The cache is streamed once: its lines go first out of L2, so that the partial states this
    // grid writes are still there when the merge reads them.
    const uint64_t stream_policy = l2_policy_evict_first();
    if (!p.block_table) {
      if (lane == 0) {
        int issued = 0;
        for (int st = 0; st < n_stages; ++st) {
          const int s = st % kDecStages;
          if (st >= kDecStages &&
              !wait_bounded(EMPTY(s), ((st / kDecStages) - 1) & 1, abort_flag, p.status))
            break;
          const uint32_t kbuf = base + s * L::kStage;
          const uint32_t vbuf = kbuf + L::kTensor;
          const int tl = t0 + st * kDecTok;  // first token of the stage
          mbar_arrive_expect_tx(FULL(s), 2 * L::kTensor);
          tma_load_4d_hint(kbuf, &tm_k, FULL(s), 0, tl, 0, hk, stream_policy);
          tma_load_4d_hint(vbuf, &tm_v, FULL(s), 0, tl, 0, hk, stream_policy);
          issued = st + 1;
        }
        for (int st = (issued > kDecStages ? issued - kDecStages : 0); st < issued; ++st)
          wait_bounded(FULL(st % kDecStages), (st / kDecStages) & 1, nullptr, p.status,
                       100000000ull);
      }
    } else {
      // Pages of a stage that hold tokens of the sequence: one when a page spans the whole
      // stage (its rows tl .. tl + 63 lie in one page), else 64 / page_size pages loaded to
      // consecutive row blocks of the stage, each by its own lane (lane i: page i of the stage),
      // so that the copies of small pages go out side by side.  Lane 0 waits for the ring slot
      // and arms its barrier with the stage's bytes first.  Rows past the sequence end are
      // masked by the compute warps; a block-table entry outside the page pool is reported and
      // its load skipped.
      const int rows = min(p.page_size, kDecTok);
      const int n_pg = kDecTok / rows;
      const int first = t0 >> p.page_log2;
      const uint32_t page_bytes = 2u * (D / 64) * rows * 128u;  // K and V, both channel halves
      int issued = 0;
      for (int st = 0; st < n_stages; ++st) {
        const int s = st % kDecStages;
        bool ok = true;
        if (lane == 0 && st >= kDecStages)
          ok = wait_bounded(EMPTY(s), ((st / kDecStages) - 1) & 1, abort_flag, p.status);
        if (!__shfl_sync(0xffffffffu, ok, 0)) break;
        const uint32_t kbuf = base + s * L::kStage;
        const uint32_t vbuf = kbuf + L::kTensor;
        const int tl = t0 + st * kDecTok;  // first token of the stage
        int phys = -1;
        if (lane < n_pg) {
          const int t = tl + lane * rows;
          if (t < t_stop) {
            const int r0 = page_row[(t >> p.page_log2) - first];
            if (r0 >= 0) phys = r0 + (t & (p.page_size - 1));
          }
        }
        const uint32_t n_loads = __popc(__ballot_sync(0xffffffffu, phys >= 0));
        if (lane == 0) mbar_arrive_expect_tx(FULL(s), n_loads * page_bytes);
        __syncwarp();
        if (phys >= 0) {
          const uint32_t box_off = static_cast<uint32_t>(lane) * (D / 64) * rows * 128u;
          tma_load_4d_hint(kbuf + box_off, &tm_k, FULL(s), 0, phys, 0, hk, stream_policy);
          tma_load_4d_hint(vbuf + box_off, &tm_v, FULL(s), 0, phys, 0, hk, stream_policy);
        }
        issued = st + 1;
      }
      if (lane == 0)
        for (int st = (issued > kDecStages ? issued - kDecStages : 0); st < issued; ++st)
          wait_bounded(FULL(st % kDecStages), (st / kDecStages) & 1, nullptr, p.status,
                       100000000ull);
    }
    return;  // the producer takes no part in the reduction below
  }

  // -------------------------------------------------------------------- compute warps
  const int g = lane >> 2;  // accumulator row (query head inside the group) and +8
  const int c = lane & 3;
  const int hq0 = hk * p.G;
  const bool row0 = g < p.G, row1 = g + 8 < p.G;
  const uint16_t* qb = p.q + (static_cast<size_t>(b) * p.Hq + hq0) * D;
  uint32_t qa[D / 16][4];
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const int col = ks * 16 + 2 * c;
    qa[ks][0] = row0 ? *reinterpret_cast<const uint32_t*>(qb + g * D + col) : 0u;
    qa[ks][1] = row1 ? *reinterpret_cast<const uint32_t*>(qb + (g + 8) * D + col) : 0u;
    qa[ks][2] = row0 ? *reinterpret_cast<const uint32_t*>(qb + g * D + col + 8) : 0u;
    qa[ks][3] = row1 ? *reinterpret_cast<const uint32_t*>(qb + (g + 8) * D + col + 8) : 0u;
  }
  float m[2] = {-INFINITY, -INFINITY};
  float l[2] = {0.f, 0.f};  // partial over this thread's columns
  float o[D / 8][4];
#pragma unroll
  for (int nd = 0; nd < D / 8; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
  // Byte offset of (row, 64-channel half) in a stage of R = 2^box_log2-row boxes laid out
  // [box][half][R rows][128 B]; the 128-byte swizzle's row phase is row % 8 in every layout.
  const int bl2 = p.box_log2;
  auto stage_off = [&](int row, int half) -> uint32_t {
    return (static_cast<uint32_t>((row >> bl2) * (D / 64) + half) << (bl2 + 7)) +
           (static_cast<uint32_t>(row & ((1 << bl2) - 1)) << 7);
  };
  // this lane's ldmatrix rows: K (scores) and V (the transposed P V operand)
  uint32_t k_row[D / 64], v_row[D / 64];
#pragma unroll
  for (int h = 0; h < D / 64; ++h) {
    k_row[h] = stage_off(warp * 16 + ((lane >> 4) << 3) + (lane & 7), h);
    v_row[h] = stage_off(warp * 16 + (((lane >> 3) & 1) << 3) + (lane & 7), h);
  }

  bool ok = true;
  for (int st = 0; st < n_stages; ++st) {
    const int s = st % kDecStages;
    if (!dec_warp_wait(FULL(s), (st / kDecStages) & 1, abort_flag, p.status)) {
      ok = false;
      break;
    }
    const uint32_t kbuf = base + s * L::kStage;
    const uint32_t vbuf = kbuf + L::kTensor;
    const int key0 = st * kDecTok + warp * 16;  // first token of this warp, chunk-relative
    const int valid = n_tok - key0;             // tokens of this warp that belong to the chunk
    if (valid > 0) {
      if (valid < 16) {
        // Rows past the chunk hold other sequences' (or unwritten) cache rows: zero their V so
        // 0 * V stays 0 even for non-finite garbage.
        for (int i = lane; i < (16 - valid) * (D / 8); i += 32) {
          const int rr = warp * 16 + valid + i / (D / 8);
          const int ch = i % (D / 8);
          *reinterpret_cast<uint4*>(gbase + (vbuf - base) + stage_off(rr, ch >> 3) +
                                    (((ch & 7) ^ (rr & 7)) << 4)) = make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
      }
      // S = Q K^T for this warp's 16 tokens: two n8 tiles.
      float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int chunk = ks * 2 + ((lane >> 3) & 1);
        const int key = warp * 16 + ((lane >> 4) << 3) + (lane & 7);
        uint32_t b00, b01, b10, b11;
        ldmatrix_x4(kbuf + k_row[chunk >> 3] + (((chunk & 7) ^ (key & 7)) << 4), b00, b01, b10, b11);
        mma_m16n8k16<BF16>(sc[0], qa[ks], b00, b01);
        mma_m16n8k16<BF16>(sc[1], qa[ks], b10, b11);
      }
      // Online softmax for rows g and g + 8 over the 16 tokens ("FlashAttention and GPU Data
      // Movement", section 3.1), base 2 with the scale folded in.
      float x[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int kidx = nt * 8 + 2 * c + (e & 1);
          x[nt][e] = (kidx < valid) ? sc[nt][e] * p.sl2 : -INFINITY;
        }
      float mx0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
      float mx1 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
      const float a0 = (m[0] == -INFINITY) ? 0.f : ex2(m[0] - mn0);
      const float a1 = (m[1] == -INFINITY) ? 0.f : ex2(m[1] - mn1);
      const float mu0 = (mn0 == -INFINITY) ? 0.f : mn0;
      const float mu1 = (mn1 == -INFINITY) ? 0.f : mn1;
      m[0] = mn0;
      m[1] = mn1;
      float pr[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        pr[nt][0] = ex2(x[nt][0] - mu0);
        pr[nt][1] = ex2(x[nt][1] - mu0);
        pr[nt][2] = ex2(x[nt][2] - mu1);
        pr[nt][3] = ex2(x[nt][3] - mu1);
      }
      l[0] = l[0] * a0 + (pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]);
      l[1] = l[1] * a1 + (pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]);
#pragma unroll
      for (int nd = 0; nd < D / 8; ++nd) {
        o[nd][0] *= a0;
        o[nd][1] *= a0;
        o[nd][2] *= a1;
        o[nd][3] *= a1;
      }
      // O += P V: P (16 rows x 16 tokens) comes straight from the score fragments.
      uint32_t pa[4];
      pa[0] = pack2<BF16>(pr[0][0], pr[0][1]);
      pa[1] = pack2<BF16>(pr[0][2], pr[0][3]);
      pa[2] = pack2<BF16>(pr[1][0], pr[1][1]);
      pa[3] = pack2<BF16>(pr[1][2], pr[1][3]);
#pragma unroll
      for (int nd2 = 0; nd2 < D / 16; ++nd2) {
        const int key = warp * 16 + (((lane >> 3) & 1) << 3) + (lane & 7);
        const int chunk = nd2 * 2 + (lane >> 4);
        uint32_t v0, v1, v2, v3;
        ldmatrix_x4_trans(vbuf + v_row[chunk >> 3] + (((chunk & 7) ^ (key & 7)) << 4), v0, v1, v2,
                          v3);
        mma_m16n8k16<BF16>(o[2 * nd2], pa, v0, v1);
        mma_m16n8k16<BF16>(o[2 * nd2 + 1], pa, v2, v3);
      }
      if (valid < 16) fence_proxy_async_smem();  // generic zeros before the next TMA write
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(EMPTY(s));
  }

  // ---------------------------------------------------- merge the four warps' states
  l[0] += __shfl_xor_sync(0xffffffffu, l[0], 1);
  l[0] += __shfl_xor_sync(0xffffffffu, l[0], 2);
  l[1] += __shfl_xor_sync(0xffffffffu, l[1], 1);
  l[1] += __shfl_xor_sync(0xffffffffu, l[1], 2);
  named_bar_sync(1, kDecWarps * 32);  // every warp is done with the ring
  ok = ok && (*abort_flag == 0);
  float* red = reinterpret_cast<float*>(gbase);  // [warp][row][D + 2]
  constexpr int kRow = D + 2;
  if (ok) {
    float* rw = red + warp * kMaxGroup * kRow;
#pragma unroll
    for (int nd = 0; nd < D / 8; ++nd) {
      if (row0) {
        rw[g * kRow + nd * 8 + 2 * c] = o[nd][0];
        rw[g * kRow + nd * 8 + 2 * c + 1] = o[nd][1];
      }
      if (row1) {
        rw[(g + 8) * kRow + nd * 8 + 2 * c] = o[nd][2];
        rw[(g + 8) * kRow + nd * 8 + 2 * c + 1] = o[nd][3];
      }
    }
    if (c == 0) {
      if (row0) {
        rw[g * kRow + D] = m[0];
        rw[g * kRow + D + 1] = l[0];
      }
      if (row1) {
        rw[(g + 8) * kRow + D] = m[1];
        rw[(g + 8) * kRow + D + 1] = l[1];
      }
    }
  }
  named_bar_sync(1, kDecWarps * 32);
  if (ok) {
    const size_t part0 = (static_cast<size_t>(b) * p.Hq + hq0) * p.max_splits + split;
    for (int i = threadIdx.x; i < p.G * D; i += kDecWarps * 32) {
      const int row = i / D, col = i % D;
      float mm = -INFINITY;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) mm = fmaxf(mm, red[(w * kMaxGroup + row) * kRow + D]);
      float ll = 0.f, acc = 0.f;
#pragma unroll
      for (int w = 0; w < kDecWarps; ++w) {
        const float mw = red[(w * kMaxGroup + row) * kRow + D];
        const float wgt = (mw == -INFINITY) ? 0.f : ex2(mw - mm);
        ll += wgt * red[(w * kMaxGroup + row) * kRow + D + 1];
        acc += wgt * red[(w * kMaxGroup + row) * kRow + col];
      }
      const size_t part = part0 + static_cast<size_t>(row) * p.max_splits;
      p.ws_o[part * D + col] = acc / ll;
      if (col == 0) {
        p.ws_ml[part * 2] = mm;
        p.ws_ml[part * 2 + 1] = ll;
      }
    }
  }
#undef FULL
#undef EMPTY
}

// Merge the chunk states of one (sequence, query head) row:
//   m = max_s m_s,  w_s = 2^(m_s - m) l_s,  l = sum_s w_s,  o = sum_s w_s o_s / l,
//   L = ln 2 * (m + log2 l).
// One warp finds m over the row's splits (its lanes striding over them) and the block writes
// the weights w_s of up to kMergeChunk splits at a time to shared memory; then every thread sums
// its channel over those splits with sixteen independent loads in flight, in split order.  A row
// has up to max_seqlen / split splits (64 for 32k tokens at 512): walked one after the other,
// each load would wait a full memory latency.
constexpr int kMergeChunk = 256;

template <int D, bool BF16>
__global__ void __launch_bounds__(D)
    attn_decode_merge_kernel(const DecParams p, uint16_t* out, float* lse) {
  __shared__ float w_s[kMergeChunk];
  __shared__ float row_max;
  // launched as a programmatic dependent of the split kernel: its partial states are complete
  // and visible once this returns
  griddep_wait();
  const int hq = blockIdx.x;
  const int b = blockIdx.y;
  const int col = threadIdx.x;
  int t_start, t_stop;
  if (!seq_bounds(p, b, t_start, t_stop)) return;
  const int n_splits = (t_stop - t_start + p.split - 1) / p.split;
  const size_t row = static_cast<size_t>(b) * p.Hq + hq;
  if (n_splits == 0) {
    out[row * D + col] = 0;
    if (col == 0) lse[row] = -INFINITY;
    return;
  }
  const size_t part0 = row * p.max_splits;
  const float2* ml = reinterpret_cast<const float2*>(p.ws_ml) + part0;  // (m, l) per split
  if (threadIdx.x < 32) {
    float m = -INFINITY;
    for (int s = threadIdx.x; s < n_splits; s += 32) m = fmaxf(m, ml[s].x);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if (threadIdx.x == 0) row_max = m;
  }
  __syncthreads();
  const float mm = row_max;
  float ll = 0.f, acc = 0.f;
  for (int c0 = 0; c0 < n_splits; c0 += kMergeChunk) {
    const int nc = min(kMergeChunk, n_splits - c0);
    for (int s = threadIdx.x; s < nc; s += D) {
      const float2 v = ml[c0 + s];
      w_s[s] = ex2(v.x - mm) * v.y;
    }
    __syncthreads();
    const float* o = p.ws_o + (part0 + c0) * D + col;
    int s = 0;
    for (; s + 16 <= nc; s += 16) {
      float v[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) v[u] = o[static_cast<size_t>(s + u) * D];
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const float w = w_s[s + u];
        ll += w;
        acc += w * v[u];
      }
    }
    for (; s < nc; ++s) {
      const float w = w_s[s];
      ll += w;
      acc += w * o[static_cast<size_t>(s) * D];
    }
    __syncthreads();  // every thread has read this chunk's weights
  }
  const float v = acc / ll;
  uint32_t pk = pack2<BF16>(v, 0.f);
  out[row * D + col] = static_cast<uint16_t>(pk & 0xffffu);
  if (col == 0) lse[row] = (mm + lg2(ll)) * 0.69314718055994531f;
}

size_t decode_workspace_bytes(int B, int Hq, int max_seqlen, int split, int d) {
  if (B <= 0 || Hq <= 0 || max_seqlen < 0 || split <= 0 || d <= 0) return 0;
  const size_t max_splits = (static_cast<size_t>(max_seqlen) + split - 1) / split;
  const size_t parts = static_cast<size_t>(B) * Hq * (max_splits > 0 ? max_splits : 1);
  const size_t o_bytes = (parts * d * 4 + 255) & ~static_cast<size_t>(255);
  return o_bytes + parts * 2 * 4;
}

template <int D, bool BF16>
static int launch_decode_variant(const DecodeArgs& a, cudaStream_t stream) {
  using L = DecLayout<D>;
  const int max_splits = (a.max_seqlen + a.split - 1) / a.split;
  const bool any_keys = a.kv_capacity > 0 && max_splits > 0;
  CUtensorMap tk, tv;
  const uint64_t row = static_cast<uint64_t>(D) * 2;
  const bool paged = a.block_table != nullptr;
  // the token axis: the packed cache, or every page of the pool end to end
  const uint64_t tokens = paged ? static_cast<uint64_t>(a.num_pages) * a.page_size
                                : static_cast<uint64_t>(a.kv_capacity);
  const uint32_t box_rows = paged ? static_cast<uint32_t>(min(a.page_size, kDecTok)) : kDecTok;
  // {64 channels, token, channel half, head}: one box = box_rows tokens x both halves of d
  const uint64_t dims[4] = {64, tokens, D / 64, static_cast<uint64_t>(a.Hkv)};
  const uint64_t strides[3] = {row * a.Hkv, 128, row};
  const uint32_t box[4] = {64, box_rows, D / 64, 1};
  if (any_keys && (!make_tmap_4d(&tk, a.k_cache, BF16, dims, strides, box) ||
                   !make_tmap_4d(&tv, a.v_cache, BF16, dims, strides, box)))
    return -5;
  DecParams p;
  p.q = static_cast<const uint16_t*>(a.q);
  p.cu = a.cu_seqlens;
  p.block_table = a.block_table;
  p.seqlens = a.seqlens;
  p.page_size = a.page_size;
  p.page_log2 = 0;
  while (paged && (1 << p.page_log2) < a.page_size) ++p.page_log2;
  p.box_log2 = 0;
  while ((1u << p.box_log2) < box_rows) ++p.box_log2;
  p.max_pages = a.max_pages;
  p.num_pages = a.num_pages;
  const size_t parts = static_cast<size_t>(a.B) * a.Hq * (max_splits > 0 ? max_splits : 1);
  p.ws_o = static_cast<float*>(a.workspace);
  p.ws_ml = reinterpret_cast<float*>(static_cast<char*>(a.workspace) +
                                     ((parts * D * 4 + 255) & ~static_cast<size_t>(255)));
  p.status = device_status_ptr();
  if (!p.status) return -5;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.G = a.Hq / a.Hkv;
  p.capacity = a.kv_capacity;
  p.max_seqlen = a.max_seqlen;
  p.split = a.split;
  p.max_splits = max_splits > 0 ? max_splits : 1;
  p.sl2 = a.scale * 1.4426950408889634f;
  auto kern = attn_decode_split_kernel<D, BF16>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes) !=
      cudaSuccess)
    return -5;
  if (any_keys) {
    dim3 grid(max_splits, a.Hkv, a.B);
    kern<<<grid, kDecThreads, L::kBytes, stream>>>(tk, tv, p);
    if (cudaGetLastError() != cudaSuccess) return -5;
  }
  // The merge goes out as a programmatic dependent of the kernel before it (the split kernel,
  // or whatever the stream ran last): its blocks are scheduled early and wait at their start
  // (griddepcontrol.wait) until that grid has completed, which hides the launch gap.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.Hq, a.B);
  cfg.blockDim = dim3(D);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, attn_decode_merge_kernel<D, BF16>, p, static_cast<uint16_t*>(a.o),
                         a.lse) != cudaSuccess)
    return -5;
  return cudaGetLastError() == cudaSuccess ? 0 : -5;
}

// ------------------------------------------------------------------------------------------
// Scratch for callers that cannot allocate device memory.
//
// Some callers have no way to hand the decode a workspace: a serving loop that may not call
// cudaMalloc in its step (the call can synchronise the whole device), a host that runs under a
// fixed device-memory budget owned by another allocator it has no handle to, or an embedding
// that lends the library only its input and output buffers.  For them the partial states live
// in this fixed array, which every GPU that loads the library keeps until the process exits.  All calls share it: two such
// calls running at the same time on the GPU would overwrite each other's partial states, so
// they must be ordered (same stream, or synchronised).  Nothing in it needs to start at zero:
// every partial state is written before it is read.
// ------------------------------------------------------------------------------------------
constexpr size_t kStaticScratchBytes = size_t(32) << 20;  // 32 MiB
static __device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

int static_decode_scratch(void** ptr, size_t* bytes) {
  static void* per_device[64];
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -7;
  std::lock_guard<std::mutex> lock(mu);
  if (!per_device[dev]) {
    // Host code cannot use g_decode_scratch as a device address; ask the runtime for this
    // device's copy (first call on each device, with that device current).
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return -5;
    per_device[dev] = p;
  }
  *ptr = per_device[dev];
  *bytes = kStaticScratchBytes;
  return 0;
}

int launch_attn_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (a.d == 64)
    return a.bf16 ? launch_decode_variant<64, true>(a, stream) : launch_decode_variant<64, false>(a, stream);
  if (a.d == 128)
    return a.bf16 ? launch_decode_variant<128, true>(a, stream) : launch_decode_variant<128, false>(a, stream);
  return -2;
}

}  // namespace attn
