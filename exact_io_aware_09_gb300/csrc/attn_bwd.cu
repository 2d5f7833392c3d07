// Backward pass of exact attention by recomputation, sm_103a.
//
// "FlashAttention Explained", section "Backward Pass: Recomputation Beats Storage": the forward
// pass saves O and one log-sum-exp L per row; the backward pass recomputes the score and
// probability tiles from Q, K and L (P = exp(S - L)) and forms
//     dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D) with D_i = rowsum(dO_i o O_i),
//     dQ = scale dS K,  dK = scale dS^T Q.
// The pages note that accumulating dQ across key tiles with atomic adds makes the result
// nondeterministic.  Here every gradient is owned by exactly one thread block, so the result is
// deterministic by construction:
//   kernel 0  D and L log2(e) per query row (padded to whole 128-row tiles);
//   kernel 1  one block per 128-key tile of one (batch, key/value head): loops over the query
//             tiles of every query head that shares the key/value head and keeps dK and dV in
//             tensor memory (four MMAs per step: S^T, dP^T, dV += P^T dO, dK += dS^T Q);
//   kernel 2  one block per 128-row query tile: loops over the key tiles and keeps dQ in
//             tensor memory (three MMAs per step: S, dP, dQ += dS K).
// S and dP are recomputed in both kernels (seven MMAs per tile pair instead of five): the price
// of owning every output without atomics.
//
// The dK/dV kernel steps through 64 queries at a time (S^T and dP^T as 128 x 64 products,
// double-buffered, so one step's elementwise work overlaps the next step's products); the dQ
// kernel takes whole 128 x 128 tiles with single S and dP buffers that are released as soon as
// they have been read.  The two elementwise warpgroups take alternate steps in kernel 1 and
// split each tile's keys in kernel 2.  Probabilities and dS go back to tensor memory as 16-bit
// pairs (over the fp32 columns they came from, or into a buffer of their own) and feed the
// accumulating MMAs as their A operand.
//
// Roles inside a thread block (384 threads): warps 0-3 and 4-7 the elementwise warpgroups
// (thread = one row of the tensor-memory tiles: a key in kernel 1, a query in kernel 2), warp 8
// the TMA producer, warp 9 the issuer of the score products (S^T or S; it owns the
// tensor-memory allocation), warp 11 the issuer of dP^T or dP, warp 10 the issuer of the
// accumulations (dV and dK, or dQ).  Each issuing thread commits its own products; the
// hand-offs between them run through the elementwise warps' barriers.  Every wait on a barrier
// is bounded.
#include <algorithm>
#include <map>
#include <memory>
#include <mutex>
#include <queue>
#include <tuple>
#include <vector>

#include "internal.h"
#include "ptx.cuh"

namespace attn {

namespace {

constexpr int kBT = 128;            // rows of a query tile and keys of a key tile
constexpr int kKvThreads = 384;    // three issuing warps in either kernel
constexpr int kQThreads = 384;
constexpr int kEwThreads = 128;     // one elementwise warpgroup (two of them: warps 0-3, 4-7)
// warp 9 issues the score products S^T or S (and owns the tensor-memory allocation), warp 11
// the dP^T or dP products, warp 10 the gradient accumulations.  Several issuing threads keep
// the tensor pipe's short queue fed while one of them waits on a barrier.
constexpr int kBwdProducerWarp = 8, kBwdIssuerWarp = 9, kBwdAccWarp = 10, kBwdDpWarp = 11;
constexpr uint32_t kBwdTmemCols = 512;
constexpr uint32_t kSub = 128 * 128;  // bytes of one 64-column, 128-row swizzled sub-tile
constexpr uint64_t kBwdDrainNs = 100000000ull;

struct BwdParams {
  const float* lse2;  // [B*Hq, nqp]  -L * log2(e); -inf on padding rows
  const float* dvec;  // [B*Hq, nqp]  -scale * D; 0 on padding rows
  const uint16_t* q;     // [B, Hq, N_q, d]
  const uint16_t* k;     // [B, Hkv, N_kv, d]
  const uint16_t* v;
  const uint16_t* dout;  // [B, Hq, N_q, d]
  uint16_t* dq;       // [B, Hq, N_q, d]
  uint16_t* dk;       // [B, Hkv, N_kv, d]
  uint16_t* dv;
  int* status;
  int Hq, Hkv, G, N_q, N_kv, n_qtiles, n_kvtiles, nqp, causal;
  float sl2;    // scale * log2(e)
  float scale;
};

template <bool BF16>
__device__ __forceinline__ float half_to_f32(uint32_t h) {
  if constexpr (BF16) {
    return __uint_as_float(h << 16);
  } else {
    float f;
    asm("{\n\t.reg .f16 t;\n\tmov.b16 t, %1;\n\tcvt.f32.f16 %0, t;\n\t}" : "=f"(f) : "h"(static_cast<uint16_t>(h)));
    return f;
  }
}

__device__ __forceinline__ bool ew_wait(uint32_t bar, uint32_t parity, volatile int* abort,
                                        int* status) {
  const bool ok = wait_bounded(bar, parity, abort, status);
  return __all_sync(0xffffffffu, ok);
}

// One 128 x D tile row r of a tensor-memory accumulator -> 16-bit values of global row `dst`.
template <int D, bool BF16>
__device__ __forceinline__ void store_acc_row(uint32_t row_tmem_col, uint16_t* dst, bool store) {
#pragma unroll 1
  for (int c = 0; c < D / 32; ++c) {
    uint32_t a[32];
    tmem_ld32(row_tmem_col + c * 32, a);
    tmem_wait_ld();
    if (store) {
      uint4* out = reinterpret_cast<uint4*>(dst + c * 32);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4)
        out[q4] = make_uint4(pack2<BF16>(__uint_as_float(a[8 * q4 + 0]), __uint_as_float(a[8 * q4 + 1])),
                             pack2<BF16>(__uint_as_float(a[8 * q4 + 2]), __uint_as_float(a[8 * q4 + 3])),
                             pack2<BF16>(__uint_as_float(a[8 * q4 + 4]), __uint_as_float(a[8 * q4 + 5])),
                             pack2<BF16>(__uint_as_float(a[8 * q4 + 6]), __uint_as_float(a[8 * q4 + 7])));
    }
  }
}

template <int D>
__device__ __forceinline__ void store_zero_row(uint16_t* dst) {
  uint4* out = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int c = 0; c < D / 8; ++c) out[c] = make_uint4(0, 0, 0, 0);
}

}  // namespace

// ------------------------------------------------------------------------------------------
// kernel 0: -scale D = -scale rowsum(dO o O) and -L log2(e), d / 8 lanes per (padded) query row
// ------------------------------------------------------------------------------------------
template <int D, bool BF16>
__global__ void attn_bwd_pre_kernel(const uint16_t* o, const uint16_t* dout, const float* lse,
                                    float* lse2, float* dvec, int N_q, int nqp, long long rows,
                                    float scale) {
  // D / 8 lanes per row, 16-byte loads of O and dO; 32 / (D / 8) rows per warp
  constexpr int kLanes = D / 8;
  const long long w = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) / kLanes;
  const int lane = threadIdx.x % kLanes;
  const bool in = w < rows;
  const long long bh = in ? w / nqp : 0;
  const int i = in ? static_cast<int>(w - bh * nqp) : 0;
  float acc = 0.0f;
  if (in && i < N_q) {
    const size_t base = (static_cast<size_t>(bh) * N_q + i) * D + lane * 8;
    const uint4 a = *reinterpret_cast<const uint4*>(o + base);
    const uint4 b = *reinterpret_cast<const uint4*>(dout + base);
    const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      acc = fmaf(half_to_f32<BF16>(av[c] & 0xffffu), half_to_f32<BF16>(bv[c] & 0xffffu), acc);
      acc = fmaf(half_to_f32<BF16>(av[c] >> 16), half_to_f32<BF16>(bv[c] >> 16), acc);
    }
  }
#pragma unroll
  for (int sh = kLanes / 2; sh > 0; sh >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, sh);
  if (in && lane == 0) {
    // stored negated (and D times the scale), so that the elementwise steps are single FMAs:
    // s * scale log2(e) + (-L log2(e)) and dP * scale + (-scale D)
    dvec[w] = (i < N_q) ? -scale * acc : 0.0f;
    lse2[w] = (i < N_q) ? -lse[bh * N_q + i] * 1.4426950408889634f : -INFINITY;
  }
}

// ------------------------------------------------------------------------------------------
// kernel 1: dK, dV of one 128-key tile
// ------------------------------------------------------------------------------------------
// The query tiles stream through a ring of shared-memory stages of 64 queries (Q, dO, and their
// L log2(e) and D), taken one stage per step: S^T and dP^T (128 keys x 64 queries) are
// double-buffered in tensor memory, and elementwise warpgroup w takes the steps of buffer w, so
// that the MMAs of one step run while the elementwise step of the other is computed.  Tensor
// memory: S^T[2] 0-127, dP^T[2] 128-255, dV 256-(256+d), dK after it; P^T and dS^T go back as
// 16-bit pairs over the first 32 columns of the buffers they came from.
constexpr int kStepQ = 64;  // queries per step of the dK/dV kernel

// Dispatch order of the dK/dV kernel's blocks.  A block's work grows with the query tiles that
// see its key tile, and under the causal mask the longest blocks are long against a GPU's share
// of the whole (a 128-key tile of an 8192-token sequence with eight query heads: 1,024 64-query
// steps, against about 1,750 per SM): started longest first, the blocks leave a tail of about 7%.
// The launcher packs the blocks into one bin per SM (largest first, each into the fullest bin
// that stays under the average load) and lists them in the order in which SMs that free up in
// turn would take them; block i of the launch then runs job order.job[i].  n = 0: the default
// order (key tile major, job = block index).
constexpr int kMaxKvOrder = 2048;
struct KvOrder {
  int n;
  uint16_t job[kMaxKvOrder];
};

template <int D, int QS>
struct KvLayout {
  static constexpr uint32_t kTile = kBT * D * 2;             // K or V: 128 rows
  static constexpr uint32_t kHalf = kStepQ * D * 2;          // Q or dO: 64 rows
  static constexpr uint32_t kHalfSub = kStepQ * 128;         // one 64-column sub-tile of it
  static constexpr uint32_t kStage = (2 * kHalf + 512 + 1023) / 1024 * 1024;
  static constexpr uint32_t kK = 0;
  static constexpr uint32_t kV = kTile;
  static constexpr uint32_t kStages = 2 * kTile;
  static constexpr uint32_t kBar = kStages + QS * kStage;
  // kv_full, st_full[QS], st_empty[QS], s_full[2], dp_full[2], p_ready[2], drain,
  // p_free[2], ds_free[2], drain of the S^T issuer, ds_ready[2], drain of the dP^T issuer
  static constexpr uint32_t kNumBars = 1 + 2 * QS + 15;
  static constexpr uint32_t kMisc = kBar + kNumBars * 8;  // tmem slot, abort flag
  static constexpr uint32_t kBytes = kMisc + 16 + 1024;
  static constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
  static_assert(kTile % 1024 == 0 && kHalf % 1024 == 0, "tile alignment");
  static_assert(kBytes <= 232448, "shared memory per block");
};

// K-major A (128 rows x D, 64-column sub-tiles A_SUB bytes apart) x K-major B^T (N rows x D,
// sub-tiles B_SUB apart): D[128 x N] = A B^T, from the descriptors of the operands' first K
// step: a descriptor's start address field counts 16-byte units, so a later K step's
// descriptor is the first one plus a constant (the issuing thread builds two descriptors per
// product instead of two per MMA).
template <int D, uint32_t A_SUB, uint32_t B_SUB>
__device__ __forceinline__ void mma_rows_rows_d(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk)
    mma_ss(d_tmem, a_desc + (((kk >> 2) * A_SUB + (kk & 3) * 32) >> 4),
           b_desc + (((kk >> 2) * B_SUB + (kk & 3) * 32) >> 4), idesc, kk > 0 ? 1u : 0u);
}

// A [128 x K] in tensor memory as 16-bit pairs (K / 2 columns from a_tmem) times B [K rows x D]
// in shared memory read MN-major, from the descriptor of its first 16 rows: D[128 x D] (+)= A B.
template <int K>
__device__ __forceinline__ void mma_tmem_rows_d(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                uint32_t idesc, bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < K / 16; ++kk)
    mma_ts(d_tmem, a_tmem + kk * 8, b_desc + ((kk * 16 * 128) >> 4), idesc,
           (accumulate || kk > 0) ? 1u : 0u);
}

template <int D, bool BF16, int QS>
__global__ void __launch_bounds__(kKvThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q,
                         const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_do, const BwdParams p,
                         const __grid_constant__ KvOrder order) {
  using L = KvLayout<D, QS>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bars = base + L::kBar;
  const uint32_t bar_kv = bars;
#define ST_FULL(s) (bars + 8u * (1 + (s)))
#define ST_EMPTY(s) (bars + 8u * (1 + QS + (s)))
  const uint32_t bar_b = bars + 8u * (1 + 2 * QS);
#define S_FULL(b) (bar_b + 8u * (b))           // S^T of buffer b written (MMA commit)
#define DP_FULL(b) (bar_b + 8u * (2 + (b)))     // dP^T of buffer b written (MMA commit)
#define P_READY(b) (bar_b + 8u * (4 + (b)))     // P^T of buffer b stored (128 arrivals)
#define DS_READY(b) (bar_b + 8u * (12 + (b)))   // dS^T of buffer b stored (128 arrivals)
#define P_FREE(b) (bar_b + 8u * (7 + (b)))      // dV product of buffer b done: S^T columns free
#define DS_FREE(b) (bar_b + 8u * (9 + (b)))     // dK product of buffer b done: dP^T columns free
  const uint32_t bar_drain = bar_b + 8u * 6;
  const uint32_t bar_drain_s = bar_b + 8u * 11;
  const uint32_t bar_drain_dp = bar_b + 8u * 14;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L::kMisc + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // The dQ kernel needs nothing this one writes: its blocks may take the SMs this grid's
  // blocks leave, as soon as every block of this grid has started.
  if (threadIdx.x == 0) griddep_launch_dependents();

  // job: key tile kt of (batch, key/value head) bkv, numbered key tile major; the launch order
  // is the packed one of KvOrder when the launcher gives one
  const int n_planes = static_cast<int>(gridDim.x / p.n_kvtiles);
  const int job = order.n ? static_cast<int>(order.job[blockIdx.x]) : static_cast<int>(blockIdx.x);
  const int kt = job / n_planes;
  const int bkv = job % n_planes;
  const int b = bkv / p.Hkv;
  const int hk = bkv % p.Hkv;
  const int off = p.N_kv - p.N_q;
  int qt_lo = 0;
  if (p.causal) {
    const int first_row = kt * kBT - off;  // first query row that sees key kt * 128
    qt_lo = first_row > 0 ? first_row / kBT : 0;
  }
  const int nq_per = p.n_qtiles - qt_lo;  // query tiles per query head
  const int n = nq_per > 0 ? p.G * nq_per : 0;
  const int n_steps = 2 * n;              // two 64-query steps per query tile

  if (threadIdx.x == 0) {
    mbar_init(bar_kv, 1);
    for (int s = 0; s < QS; ++s) {
      mbar_init(ST_FULL(s), 1);
      mbar_init(ST_EMPTY(s), 1);
    }
    for (int bb = 0; bb < 2; ++bb) {
      mbar_init(S_FULL(bb), 1);
      mbar_init(DP_FULL(bb), 1);
      mbar_init(P_READY(bb), kEwThreads);
      mbar_init(DS_READY(bb), kEwThreads);
      mbar_init(P_FREE(bb), 1);
      mbar_init(DS_FREE(bb), 1);
    }
    mbar_init(bar_drain, 1);
    mbar_init(bar_drain_s, 1);
    mbar_init(bar_drain_dp, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kBwdIssuerWarp) {
    tmem_alloc(smem_u32(tmem_slot), kBwdTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kBwdProducerWarp) {
    if (lane == 0 && n > 0) {
      prefetch_tmap(&tm_q);
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      prefetch_tmap(&tm_do);
      mbar_arrive_expect_tx(bar_kv, 2 * L::kTile);
#pragma unroll
      for (int sub = 0; sub < D / 64; ++sub) {
        tma_load_3d(base + L::kK + sub * kSub, &tm_k, bar_kv, sub * 64, kt * kBT, bkv);
        tma_load_3d(base + L::kV + sub * kSub, &tm_v, bar_kv, sub * 64, kt * kBT, bkv);
      }
      int issued = 0;
      for (int i = 0; i < n_steps; ++i) {
        const int s = i % QS;
        if (i >= QS && !wait_bounded(ST_EMPTY(s), ((i / QS) - 1) & 1, abort_flag, p.status)) break;
        const int tile = i >> 1;
        const int g = tile / nq_per;
        const int q0 = (qt_lo + tile % nq_per) * kBT + (i & 1) * kStepQ;
        const int bhq = b * p.Hq + hk * p.G + g;
        const uint32_t st = base + L::kStages + s * L::kStage;
        mbar_arrive_expect_tx(ST_FULL(s), 2 * L::kHalf + 512);
#pragma unroll
        for (int sub = 0; sub < D / 64; ++sub) {
          tma_load_3d(st + sub * L::kHalfSub, &tm_q, ST_FULL(s), sub * 64, q0, bhq);
          tma_load_3d(st + L::kHalf + sub * L::kHalfSub, &tm_do, ST_FULL(s), sub * 64, q0, bhq);
        }
        const size_t vec = static_cast<size_t>(bhq) * p.nqp + static_cast<size_t>(q0);
        bulk_load(st + 2 * L::kHalf, p.lse2 + vec, kStepQ * 4, ST_FULL(s));
        bulk_load(st + 2 * L::kHalf + 256, p.dvec + vec, kStepQ * 4, ST_FULL(s));
        issued = i + 1;
      }
      wait_bounded(bar_kv, 0, nullptr, p.status, kBwdDrainNs);
      for (int i = (issued > QS ? issued - QS : 0); i < issued; ++i)
        wait_bounded(ST_FULL(i % QS), (i / QS) & 1, nullptr, p.status, kBwdDrainNs);
    }
    __syncwarp();
  } else if (warp == kBwdIssuerWarp || warp == kBwdDpWarp) {
    if (lane == 0 && n > 0) {
      // Step i in buffer i % 2.  Warp 9: S^T_i = K Q_i^T once step i - 2's dV product (which
      // reads P^T from the same columns) is done.  Warp 11: dP^T_i = V dO_i^T once step i - 2's
      // dK product (dS^T) is done.  Waiting for each product separately lets step i's products
      // start while step i - 2's are still in the pipe, and the two threads' waits overlap
      // each other's issue.
      const bool is_s = (warp == kBwdIssuerWarp);
      constexpr uint32_t idesc_s = make_idesc_f16(BF16, kBT, kStepQ, false);
      const uint64_t a_desc = make_sdesc_sw128(base + (is_s ? L::kK : L::kV), 16, 1024);
      const uint32_t col0 = is_s ? L::kColS : L::kColDP;
      const uint32_t b_off = is_s ? 0u : L::kHalf;  // Q or dO of the stage
      bool ok = wait_bounded(bar_kv, 0, abort_flag, p.status);
      for (int i = 0; ok && i < n_steps; ++i) {
        const int s = i % QS, bb = i & 1;
        if (!wait_bounded(ST_FULL(s), (i / QS) & 1, abort_flag, p.status)) break;
        if (i >= 2 && !wait_bounded(is_s ? P_FREE(bb) : DS_FREE(bb), ((i >> 1) - 1) & 1,
                                    abort_flag, p.status))
          break;
        tc_fence_after();
        const uint32_t st = base + L::kStages + s * L::kStage;
        mma_rows_rows_d<D, kSub, L::kHalfSub>(tmem + col0 + bb * kStepQ, a_desc,
                                               make_sdesc_sw128(st + b_off, 16, 1024), idesc_s);
        mma_commit(is_s ? S_FULL(bb) : DP_FULL(bb));
      }
      // this thread's products are complete before the block ends (after an abort as well)
      const uint32_t drain = is_s ? bar_drain_s : bar_drain_dp;
      mma_commit(drain);
      wait_bounded(drain, 0, nullptr, p.status, kBwdDrainNs);
    }
    __syncwarp();
  } else if (warp == kBwdAccWarp) {
    if (lane == 0 && n > 0) {
      // Once P^T_i is stored: dV += P^T_i dO_i (its commit frees the S^T columns); once dS^T_i
      // is stored: dK += dS^T_i Q_i (its commit frees the dP^T columns and the stage: step i's
      // score products are complete, the elementwise warps waited for them before storing).
      constexpr uint32_t idesc_acc = make_idesc_f16(BF16, kBT, D, true);
      for (int i = 0; i < n_steps; ++i) {
        const int s = i % QS, bb = i & 1;
        const uint32_t st = base + L::kStages + s * L::kStage;
        if (!wait_bounded(P_READY(bb), (i >> 1) & 1, abort_flag, p.status)) break;
        tc_fence_after();
        mma_tmem_rows_d<kStepQ>(tmem + L::kColDV, tmem + L::kColS + bb * kStepQ,
                                make_sdesc_sw128(st + L::kHalf, L::kHalfSub, 1024), idesc_acc,
                                i > 0);  // dV += P^T dO
        mma_commit(P_FREE(bb));
        if (!wait_bounded(DS_READY(bb), (i >> 1) & 1, abort_flag, p.status)) break;
        tc_fence_after();
        mma_tmem_rows_d<kStepQ>(tmem + L::kColDK, tmem + L::kColDP + bb * kStepQ,
                                make_sdesc_sw128(st, L::kHalfSub, 1024), idesc_acc,
                                i > 0);  // dK += dS^T Q
        mma_commit(ST_EMPTY(s));
        mma_commit(DS_FREE(bb));
      }
      mma_commit(bar_drain);
      wait_bounded(bar_drain, 0, nullptr, p.status, kBwdDrainNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ elementwise (thread = key)
    // Warpgroup w takes the steps of buffer w; thread r owns key row r (warp % 4 is its
    // tensor-memory lane quarter).
    const int wg = warp >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int kr = kt * kBT + r;  // this thread's key
    const uint32_t row_tmem = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl2 = p.sl2, scale = p.scale;
    const int q_first_visible = kr - off;  // the smallest query row that sees this key
    const uint32_t s_col = L::kColS + wg * kStepQ, dp_col = L::kColDP + wg * kStepQ;
    bool ok = true;
    for (int i = wg; i < n_steps; i += 2) {
      const int s = i % QS;
      const int tile = i >> 1;
      const int q0 = (qt_lo + tile % nq_per) * kBT + (i & 1) * kStepQ;
      const float* lv = reinterpret_cast<const float*>(gbase + L::kStages + s * L::kStage +
                                                       2 * L::kHalf);
      const float* dvv = lv + kStepQ;
      if (!ew_wait(S_FULL(wg), (i >> 1) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // P^T row of this key over the step's 64 queries, kept in registers for dS^T:
      // p = 2^(s scale log2(e) - L log2(e)), one packed FMA per pair; the causal test only
      // where some query of the 64 precedes this key
      float pv[kStepQ];
      uint32_t pp[kStepQ / 2];
      {
        uint32_t sv[2][32];
        tmem_ld32(row_tmem + s_col, sv[0]);
        tmem_ld32(row_tmem + s_col + 32, sv[1]);
        tmem_wait_ld();
        const bool full = !p.causal || q0 >= q_first_visible;
        const bool all_full = __all_sync(0xffffffffu, full);
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const int col = h * 32 + e;
            const float4 l4 = *reinterpret_cast<const float4*>(lv + col);
            float a0, a1, a2, a3;
            fma2(a0, a1, __uint_as_float(sv[h][e]), __uint_as_float(sv[h][e + 1]), sl2, sl2, l4.x, l4.y);
            fma2(a2, a3, __uint_as_float(sv[h][e + 2]), __uint_as_float(sv[h][e + 3]), sl2, sl2, l4.z,
                 l4.w);
            if (!all_full) {
              const int rel = q_first_visible - (q0 + col);  // columns below rel precede the key
              a0 = (0 >= rel) ? a0 : -INFINITY;
              a1 = (1 >= rel) ? a1 : -INFINITY;
              a2 = (2 >= rel) ? a2 : -INFINITY;
              a3 = (3 >= rel) ? a3 : -INFINITY;
            }
            pv[col] = ex2(a0);
            pv[col + 1] = ex2(a1);
            pv[col + 2] = ex2(a2);
            pv[col + 3] = ex2(a3);
            pp[col >> 1] = pack2<BF16>(pv[col], pv[col + 1]);
            pp[(col >> 1) + 1] = pack2<BF16>(pv[col + 2], pv[col + 3]);
          }
      }
      tmem_st32(row_tmem + s_col, pp);  // P^T over the S^T columns already read
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(P_READY(wg));  // dV += P^T dO may start while dS^T is formed
      if (!ew_wait(DP_FULL(wg), (i >> 1) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t dpv[2][32];
      tmem_ld32(row_tmem + dp_col, dpv[0]);
      tmem_ld32(row_tmem + dp_col + 32, dpv[1]);
      tmem_wait_ld();
      // dS^T = P^T o (dP^T - D) scale = P^T o (dP^T scale + (-scale D)): two packed FMAs a pair
      uint32_t dd[kStepQ / 2];
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const int col = h * 32 + e;
          const float4 d4 = *reinterpret_cast<const float4*>(dvv + col);
          float u0, u1, u2, u3, g0, g1, g2, g3;
          fma2(u0, u1, __uint_as_float(dpv[h][e]), __uint_as_float(dpv[h][e + 1]), scale, scale, d4.x, d4.y);
          fma2(u2, u3, __uint_as_float(dpv[h][e + 2]), __uint_as_float(dpv[h][e + 3]), scale, scale, d4.z,
               d4.w);
          fma2(g0, g1, pv[col], pv[col + 1], u0, u1, 0.0f, 0.0f);
          fma2(g2, g3, pv[col + 2], pv[col + 3], u2, u3, 0.0f, 0.0f);
          dd[col >> 1] = pack2<BF16>(g0, g1);
          dd[(col >> 1) + 1] = pack2<BF16>(g2, g3);
        }
      tmem_st32(row_tmem + dp_col, dd);  // dS^T over the dP^T columns already read
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(DS_READY(wg));
    }
    // epilogue: warpgroup 0 stores dV, warpgroup 1 dK, once the last MMA has finished
    if (ok && n > 0) ok = ew_wait(bar_drain, 0, abort_flag, p.status);
    if (ok) {
      tc_fence_after();
      const bool store = kr < p.N_kv;
      const size_t grow = (static_cast<size_t>(bkv) * p.N_kv + (store ? kr : 0)) * D;
      uint16_t* dst = (wg ? p.dk : p.dv) + grow;
      if (n > 0)
        store_acc_row<D, BF16>(row_tmem + (wg ? L::kColDK : L::kColDV), dst, store);
      else if (store)
        store_zero_row<D>(dst);
    }
  }
#undef ST_FULL
#undef ST_EMPTY
#undef S_FULL
#undef DP_FULL
#undef P_READY
#undef DS_READY
#undef P_FREE
#undef DS_FREE
  tc_fence_before();
  __syncthreads();
  if (warp == kBwdIssuerWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kBwdTmemCols);
  }
}

// ------------------------------------------------------------------------------------------
// kernel 2: dQ of one 128-row query tile
// ------------------------------------------------------------------------------------------
// Q stays in tensor memory as the A operand of S = Q K^T; dO (shared memory) is that of
// dP = dO V^T.  Tensor memory: Q 0-63, S 64-191, dP 192-319, dS 320-383, dQ 384-.  The two
// elementwise warpgroups split each tile's 128 keys and release S and dP as soon as they have
// read them, and dS has its own buffer, so that the tensor pipe takes, per tile, S_{t+1} and
// dP_{t+1} (issued while tile t's elementwise step runs) and then dQ += dS_t K_t: no product
// waits for another tile's dS.
template <int D, int KR, int VR>
struct QLayout {
  static constexpr uint32_t kTile = kBT * D * 2;
  static constexpr uint32_t kDO = 0;                 // dO tile
  static constexpr uint32_t kK = kTile;              // K ring, KR slots
  static constexpr uint32_t kV = kK + KR * kTile;    // V ring, VR slots
  static constexpr uint32_t kBar = kV + VR * kTile;
  // k_full[KR], k_empty[KR], v_full[VR], v_empty[VR], q_ready, do_full, s_full, s_free,
  // drain of the S issuer, dp_free, ds_ready[2], drain, ds_free[2], drain of the dP issuer;
  // dP written is the V slot's release barrier
  static constexpr uint32_t kNumBars = 2 * KR + 2 * VR + 12;
  static constexpr uint32_t kMisc = kBar + kNumBars * 8;
  static constexpr uint32_t kBytes = kMisc + 16 + 1024;
  static constexpr uint32_t kColQ = 0, kColS = 64, kColDP = 192, kColDS = 320, kColDQ = 384;
  static_assert(kBytes <= 232448, "shared memory per block");
};

// Half h of A [128 x 128] B: A in tensor memory as 16-bit pairs (64 columns), B [128 rows x D]
// in shared memory read MN-major; the product over A's columns and B's rows 64h .. 64h + 63:
// D[128 x D] (+)= A[:, 64h:64h+64] B[64h:64h+64, :].
__device__ __forceinline__ void mma_tmem_kt_half(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_smem,
                                                 uint32_t idesc, int h, bool accumulate) {
  const uint64_t b_desc = make_sdesc_sw128(b_smem, kSub, 1024);
#pragma unroll
  for (int k4 = 0; k4 < kBT / 32; ++k4) {
    const int kk = h * (kBT / 32) + k4;
    mma_ts(d_tmem, a_tmem + kk * 8, b_desc + ((kk * 16 * 128) >> 4), idesc,
           (accumulate || k4 > 0) ? 1u : 0u);
  }
}

// A [128 x D] in tensor memory as 16-bit pairs (D / 2 columns) times B^T, B [128 rows x D]
// K-major in shared memory (64-column sub-tiles kSub apart): D[128 x 128] = A B^T.
template <int D>
__device__ __forceinline__ void mma_tmem_rows_t(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_smem,
                                                uint32_t idesc) {
  const uint64_t b_desc = make_sdesc_sw128(b_smem, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk)
    mma_ts(d_tmem, a_tmem + kk * 8, b_desc + (((kk >> 2) * kSub + (kk & 3) * 32) >> 4), idesc,
           kk > 0 ? 1u : 0u);
}

// One row of a contiguous 16-bit [rows, D] tensor as D / 2 32-bit words (zeros for a row past
// the end), and those words into tensor memory, thread = lane row: two elements a column with
// the lower-indexed one in the low half (the A operand layout of tcgen05.mma kind::f16).  The
// load is issued before the block's setup, the store after it, so that the setup hides the
// load's latency.
template <int D>
__device__ __forceinline__ void row_load(const uint16_t* src, bool valid, uint4 (&w)[D / 8]) {
#pragma unroll
  for (int i = 0; i < D / 8; ++i)
    w[i] = valid ? reinterpret_cast<const uint4*>(src)[i] : make_uint4(0, 0, 0, 0);
}

template <int D>
__device__ __forceinline__ void row_to_tmem(uint32_t taddr, const uint4 (&w)[D / 8]) {
#pragma unroll
  for (int c = 0; c < D / 64; ++c) {
    uint32_t v[32];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      v[4 * i] = w[c * 8 + i].x;
      v[4 * i + 1] = w[c * 8 + i].y;
      v[4 * i + 2] = w[c * 8 + i].z;
      v[4 * i + 3] = w[c * 8 + i].w;
    }
    tmem_st32(taddr + c * 32, v);
  }
}

template <int D, bool BF16, int KR, int VR>
__global__ void __launch_bounds__(kQThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_do, const BwdParams p) {
  using L = QLayout<D, KR, VR>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t bars = base + L::kBar;
#define K_FULL(s) (bars + 8u * (s))
#define K_EMPTY(s) (bars + 8u * (KR + (s)))
#define V_FULL(s) (bars + 8u * (2 * KR + (s)))
#define V_EMPTY(s) (bars + 8u * (2 * KR + VR + (s)))
  const uint32_t bar_q = bars + 8u * (2 * KR + 2 * VR);  // Q rows in tensor memory (128)
  const uint32_t bar_do = bar_q + 8;         // dO tile landed (TMA)
  const uint32_t bar_sfull = bar_q + 16;     // S_t written (MMA commit)
  const uint32_t bar_sfree = bar_q + 24;     // S_t read (256 arrivals)
  const uint32_t bar_drain_s = bar_q + 32;   // S issuer's products done (commit)
  const uint32_t bar_drain_dp = bar_q + 88;  // dP issuer's products done (commit)
  const uint32_t bar_dpfree = bar_q + 40;    // dP_t read (256 arrivals)
#define DS_READY(w) (bar_q + 48 + 8u * (w))       // warpgroup w's half of dS_t stored (128)
#define DS_FREE(w) (bar_q + 72 + 8u * (w))        // dQ's product over that half done (commit)
  const uint32_t bar_drain = bar_q + 64;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + L::kMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + L::kMisc + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // item: query tile qt of (batch, query head) bh.  Query-tile major, last tile first: under
  // the causal mask the longest items of every head start first and the grid ends on one-tile
  // items; the heads of one key/value head run side by side and share its K/V tiles in L2.
  const int n_bh = static_cast<int>(gridDim.x) / p.n_qtiles;
  const int qt = p.n_qtiles - 1 - static_cast<int>(blockIdx.x) / n_bh;
  const int bh = static_cast<int>(blockIdx.x) % n_bh;
  const int kv_plane = (bh / p.Hq) * p.Hkv + (bh % p.Hq) / p.G;
  int n, first_masked;
  kv_tile_range(qt, kBT, kBT, p.N_q, p.N_kv, p.causal, n, first_masked);
  // warpgroup 0 (thread = query row) starts loading the tile's Q rows now
  uint4 q_row[D / 8];
  if (n > 0 && threadIdx.x < kEwThreads) {
    const int qr = qt * kBT + static_cast<int>(threadIdx.x);
    row_load<D>(p.q + (static_cast<size_t>(bh) * p.N_q + (qr < p.N_q ? qr : 0)) * D, qr < p.N_q,
                q_row);
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < KR; ++s) {
      mbar_init(K_FULL(s), 1);
      mbar_init(K_EMPTY(s), 1);
    }
    for (int s = 0; s < VR; ++s) {
      mbar_init(V_FULL(s), 1);
      mbar_init(V_EMPTY(s), 1);
    }
    mbar_init(bar_q, kEwThreads);
    mbar_init(bar_do, 1);
    mbar_init(bar_sfull, 1);
    mbar_init(bar_sfree, 2 * kEwThreads);
    mbar_init(bar_dpfree, 2 * kEwThreads);
    for (int w = 0; w < 2; ++w) {
      mbar_init(DS_READY(w), kEwThreads);
      mbar_init(DS_FREE(w), 1);
    }
    mbar_init(bar_drain, 1);
    mbar_init(bar_drain_s, 1);
    mbar_init(bar_drain_dp, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == kBwdIssuerWarp) {
    tmem_alloc(smem_u32(tmem_slot), kBwdTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kBwdProducerWarp) {
    if (lane == 0 && n > 0) {
      prefetch_tmap(&tm_k);
      prefetch_tmap(&tm_v);
      prefetch_tmap(&tm_do);
      mbar_arrive_expect_tx(bar_do, L::kTile);
#pragma unroll
      for (int sub = 0; sub < D / 64; ++sub)
        tma_load_3d(base + L::kDO + sub * kSub, &tm_do, bar_do, sub * 64, qt * kBT, bh);
      int issued_k = 0, issued_v = 0;
      for (int t = 0; t < n; ++t) {
        const int sk = t % KR, sv = t % VR;
        if (t >= KR && !wait_bounded(K_EMPTY(sk), ((t / KR) - 1) & 1, abort_flag, p.status)) break;
        mbar_arrive_expect_tx(K_FULL(sk), L::kTile);
#pragma unroll
        for (int sub = 0; sub < D / 64; ++sub)
          tma_load_3d(base + L::kK + sk * L::kTile + sub * kSub, &tm_k, K_FULL(sk), sub * 64,
                      t * kBT, kv_plane);
        issued_k = t + 1;
        if (t >= VR && !wait_bounded(V_EMPTY(sv), ((t / VR) - 1) & 1, abort_flag, p.status)) break;
        mbar_arrive_expect_tx(V_FULL(sv), L::kTile);
#pragma unroll
        for (int sub = 0; sub < D / 64; ++sub)
          tma_load_3d(base + L::kV + sv * L::kTile + sub * kSub, &tm_v, V_FULL(sv), sub * 64,
                      t * kBT, kv_plane);
        issued_v = t + 1;
      }
      wait_bounded(bar_do, 0, nullptr, p.status, kBwdDrainNs);
      for (int t = (issued_k > KR ? issued_k - KR : 0); t < issued_k; ++t)
        wait_bounded(K_FULL(t % KR), (t / KR) & 1, nullptr, p.status, kBwdDrainNs);
      for (int t = (issued_v > VR ? issued_v - VR : 0); t < issued_v; ++t)
        wait_bounded(V_FULL(t % VR), (t / VR) & 1, nullptr, p.status, kBwdDrainNs);
    }
    __syncwarp();
  } else if (warp == kBwdIssuerWarp) {
    if (lane == 0 && n > 0) {
      // S_t = Q K_t^T once S_{t-1} has been read
      constexpr uint32_t idesc_rr = make_idesc_f16(BF16, kBT, kBT, false);
      bool ok = wait_bounded(bar_q, 0, abort_flag, p.status);
      for (int t = 0; ok && t < n; ++t) {
        const int sk = t % KR;
        if (t > 0 && !wait_bounded(bar_sfree, (t - 1) & 1, abort_flag, p.status)) break;
        if (!wait_bounded(K_FULL(sk), (t / KR) & 1, abort_flag, p.status)) break;
        tc_fence_after();
        mma_tmem_rows_t<D>(tmem + L::kColS, tmem + L::kColQ, base + L::kK + sk * L::kTile, idesc_rr);
        mma_commit(bar_sfull);
      }
      // this thread's products are complete before the block ends (after an abort as well)
      mma_commit(bar_drain_s);
      wait_bounded(bar_drain_s, 0, nullptr, p.status, kBwdDrainNs);
    }
    __syncwarp();
  } else if (warp == kBwdDpWarp) {
    if (lane == 0 && n > 0) {
      // dP_t = dO V_t^T once dP_{t-1} has been read
      constexpr uint32_t idesc_rr = make_idesc_f16(BF16, kBT, kBT, false);
      const uint64_t do_desc = make_sdesc_sw128(base + L::kDO, 16, 1024);
      bool ok = wait_bounded(bar_do, 0, abort_flag, p.status);
      for (int t = 0; ok && t < n; ++t) {
        const int sv = t % VR;
        if (t > 0 && !wait_bounded(bar_dpfree, (t - 1) & 1, abort_flag, p.status)) break;
        if (!wait_bounded(V_FULL(sv), (t / VR) & 1, abort_flag, p.status)) break;
        tc_fence_after();
        mma_rows_rows_d<D, kSub, kSub>(tmem + L::kColDP, do_desc,
                                       make_sdesc_sw128(base + L::kV + sv * L::kTile, 16, 1024),
                                       idesc_rr);
        // one commit for both readers: the elementwise warps (dP_t written) and the producer
        // (V slot free) wait on the V slot's barrier
        mma_commit(V_EMPTY(sv));
      }
      mma_commit(bar_drain_dp);
      wait_bounded(bar_drain_dp, 0, nullptr, p.status, kBwdDrainNs);
    }
    __syncwarp();
  } else if (warp == kBwdAccWarp) {
    if (lane == 0 && n > 0) {
      // dQ += dS_t K_t in two halves over the keys, each once its warpgroup has stored its
      // half of dS_t; each half's commit frees that half of the dS buffer.  After both, the K
      // slot is free (S_t, read by the elementwise warps before they stored dS_t, is complete).
      constexpr uint32_t idesc_q = make_idesc_f16(BF16, kBT, D, true);
      bool ok = true;
      for (int t = 0; ok && t < n; ++t) {
        const uint32_t kslot = base + L::kK + (t % KR) * L::kTile;
        for (int w = 0; w < 2; ++w) {
          if (!wait_bounded(DS_READY(w), t & 1, abort_flag, p.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          mma_tmem_kt_half(tmem + L::kColDQ, tmem + L::kColDS, kslot, idesc_q, w,
                           t > 0 || w > 0);  // dQ += dS K over keys 64w .. 64w + 63
          mma_commit(DS_FREE(w));
        }
        if (ok) mma_commit(K_EMPTY(t % KR));
      }
      mma_commit(bar_drain);
      wait_bounded(bar_drain, 0, nullptr, p.status, kBwdDrainNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ elementwise (thread = query)
    // Warpgroup w takes keys c0 = 64w .. c0+63 of every key tile; thread r owns query row r.
    const int wg = warp >> 2;
    const int c0 = wg * 64;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const int row = qt * kBT + r;
    const uint32_t row_tmem = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const size_t vec = static_cast<size_t>(bh) * p.nqp + row;
    const float nl2 = p.lse2[vec];  // -L log2(e)
    const float nsd = p.dvec[vec];  // -scale D
    const float sl2 = p.sl2, scale = p.scale;
    int lim = p.causal ? row + (p.N_kv - p.N_q) : p.N_kv - 1;  // last visible key of this row
    if (lim > p.N_kv - 1) lim = p.N_kv - 1;
    bool ok = true;
    if (n > 0 && wg == 0) {
      // warpgroup 0 writes the Q rows it loaded before the setup
      row_to_tmem<D>(row_tmem + L::kColQ, q_row);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_q);
    }
    const uint32_t s_col = L::kColS + c0, dp_col = L::kColDP + c0, ds_col = L::kColDS + wg * 32;
    for (int t = 0; t < n; ++t) {
      const bool masked = t >= first_masked;
      const int rel = lim - (t * kBT + c0);  // last visible key, relative to this half tile
      if (!ew_wait(bar_sfull, t & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sv[2][32];
      tmem_ld32(row_tmem + s_col, sv[0]);
      tmem_ld32(row_tmem + s_col + 32, sv[1]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar_sfree);  // S_{t+1} may overwrite
      // p = 2^(s scale log2(e) - L log2(e)), one packed FMA a pair; the mask only on the tiles
      // that need it (the same for every row of the tile)
      float pv[64];
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int col = h * 32 + e;
          float a0, a1;
          fma2(a0, a1, __uint_as_float(sv[h][e]), __uint_as_float(sv[h][e + 1]), sl2, sl2, nl2, nl2);
          if (masked) {
            a0 = (col <= rel) ? a0 : -INFINITY;
            a1 = (col + 1 <= rel) ? a1 : -INFINITY;
          }
          pv[col] = ex2(a0);
          pv[col + 1] = ex2(a1);
        }
      // dP_t written: the commit that also frees V slot t % VR (its (t / VR)-th phase); the
      // next phase needs dP_{t+VR}, which waits for this warpgroup's read of dP_{t+VR-1}
      if (!ew_wait(V_EMPTY(t % VR), (t / VR) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t dpv[2][32];
      tmem_ld32(row_tmem + dp_col, dpv[0]);
      tmem_ld32(row_tmem + dp_col + 32, dpv[1]);
      tmem_wait_ld();
      tc_fence_before();
      mbar_arrive(bar_dpfree);  // dP_{t+1} may overwrite
      // dS = P o (dP scale + (-scale D)): two packed FMAs a pair
      uint32_t dd[32];
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int col = h * 32 + e;
          float u0, u1, g0, g1;
          fma2(u0, u1, __uint_as_float(dpv[h][e]), __uint_as_float(dpv[h][e + 1]), scale, scale, nsd, nsd);
          fma2(g0, g1, pv[col], pv[col + 1], u0, u1, 0.0f, 0.0f);
          dd[col >> 1] = pack2<BF16>(g0, g1);
        }
      // this warpgroup's half of the dS buffer: free once dQ's product over it for tile t - 1
      // has finished
      if (t > 0 && !ew_wait(DS_FREE(wg), (t - 1) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      tmem_st32(row_tmem + ds_col, dd);  // keys c0 .. c0+63 as 16-bit pairs
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(DS_READY(wg));
    }
    if (ok && n > 0) ok = ew_wait(bar_drain, 0, abort_flag, p.status);
    if (ok && wg == 0) {
      tc_fence_after();
      const bool store = row < p.N_q;
      const size_t grow = (static_cast<size_t>(bh) * p.N_q + (store ? row : 0)) * D;
      if (n > 0)
        store_acc_row<D, BF16>(row_tmem + L::kColDQ, p.dq + grow, store);
      else if (store)
        store_zero_row<D>(p.dq + grow);
    }
  }
#undef K_FULL
#undef K_EMPTY
#undef V_FULL
#undef V_EMPTY
#undef DS_READY
#undef DS_FREE
  tc_fence_before();
  __syncthreads();
  if (warp == kBwdIssuerWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kBwdTmemCols);
  }
  // This grid may have started while the dK/dV kernel was still running; no block of it
  // finishes before that kernel has, so that whatever follows on the stream sees dK and dV
  // complete.
  if (threadIdx.x == 0) griddep_wait();
}

// ------------------------------------------------------------------------------------------
// launcher
// ------------------------------------------------------------------------------------------
size_t bwd_workspace_bytes(int B, int Hq, int N_q) {
  if (B <= 0 || Hq <= 0 || N_q <= 0) return 0;
  const size_t nqp = (static_cast<size_t>(N_q) + kBT - 1) / kBT * kBT;
  return static_cast<size_t>(B) * Hq * nqp * 8;  // L log2(e) and D, fp32
}

// 64-query steps of the dK/dV job for key tile kt (as the kernel counts them).
static int kv_job_steps(int kt, int n_qtiles, int G, int causal, int off) {
  int qt_lo = 0;
  if (causal) {
    const int first_row = kt * kBT - off;
    qt_lo = first_row > 0 ? first_row / kBT : 0;
  }
  const int nq_per = n_qtiles - qt_lo;
  return nq_per > 0 ? 2 * G * nq_per : 0;
}

// The packed dispatch order for a grid of n_planes x n_kvtiles jobs on n_sm SMs: writes the job
// of every block to job[0 .. n) and returns n, or 0 when the default order stands (no causal
// mask: equal jobs; no more jobs than SMs; more than `cap` jobs).
int bwd_kv_order(int n_planes, int n_kvtiles, int n_qtiles, int G, int causal, int off, int n_sm,
                 uint16_t* job, int cap) {
  const long long n_jobs_ll = static_cast<long long>(n_planes) * n_kvtiles;
  if (!causal || n_sm <= 0 || n_jobs_ll <= n_sm || n_jobs_ll > cap || n_jobs_ll > 65536) return 0;
  const int n_jobs = static_cast<int>(n_jobs_ll);
  // job weights: its steps plus a block's fixed cost (about four steps: setup, K/V load,
  // pipeline fill, dK/dV store)
  std::vector<long long> w(n_jobs);
  long long total = 0;
  for (int j = 0; j < n_jobs; ++j) {
    w[j] = kv_job_steps(j / n_planes, n_qtiles, G, causal, off) + 4;
    total += w[j];
  }
  std::vector<int> by_size(n_jobs);
  for (int j = 0; j < n_jobs; ++j) by_size[j] = j;
  std::stable_sort(by_size.begin(), by_size.end(), [&](int x, int y) { return w[x] > w[y]; });
  // best fit under a cap a little above the average load; of a few caps, the plan whose
  // fullest bin is lowest
  const long long avg = (total + n_sm - 1) / n_sm;
  std::vector<std::vector<int>> bins;
  long long best_max = -1;
  for (int step = 0; step <= 12; ++step) {
    const long long bin_cap = avg + avg * step / 400;  // up to 3% above the average
    std::vector<std::vector<int>> trial(n_sm);
    std::vector<long long> load(n_sm, 0);
    for (int j : by_size) {
      int best = -1, emptiest = 0;
      for (int b = 0; b < n_sm; ++b) {
        if (load[b] + w[j] <= bin_cap && (best < 0 || load[b] > load[best])) best = b;
        if (load[b] < load[emptiest]) emptiest = b;
      }
      const int b = best >= 0 ? best : emptiest;
      trial[b].push_back(j);  // largest first within a bin
      load[b] += w[j];
    }
    const long long mx = *std::max_element(load.begin(), load.end());
    if (best_max < 0 || mx < best_max) {
      best_max = mx;
      bins.swap(trial);
    }
  }
  // the order in which SMs that free up in turn take the bins' jobs
  int n = 0;
  using Slot = std::pair<long long, int>;  // (time the SM frees up, bin)
  std::priority_queue<Slot, std::vector<Slot>, std::greater<Slot>> free_at;
  std::vector<size_t> next(n_sm, 0);
  for (int b = 0; b < n_sm; ++b) free_at.push({0, b});
  while (!free_at.empty()) {
    const Slot sl = free_at.top();
    free_at.pop();
    const int b = sl.second;
    if (next[b] < bins[b].size()) {
      const int j = bins[b][next[b]++];
      job[n++] = static_cast<uint16_t>(j);
      free_at.push({sl.first + w[j], b});
    }
  }
  return n == n_jobs ? n : 0;
}

// The packed dispatch order (KvOrder) for one shape on the current device, computed once and
// kept.
static const KvOrder* kv_order(int n_planes, int n_kvtiles, int n_qtiles, int G, int causal,
                               int off) {
  static const KvOrder kDefault = {0, {}};
  int dev = 0, n_sm = 0;
  if (!causal || cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return &kDefault;
  using Key = std::tuple<int, int, int, int, int, int>;
  static std::map<Key, std::unique_ptr<KvOrder>> cache;
  static std::mutex mu;
  const Key key{n_planes, n_kvtiles, n_qtiles, G, off, n_sm};
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(key);
  if (it != cache.end()) return it->second.get();
  auto order = std::make_unique<KvOrder>();
  order->n = bwd_kv_order(n_planes, n_kvtiles, n_qtiles, G, causal, off, n_sm, order->job,
                          kMaxKvOrder);
  const KvOrder* out = order.get();
  cache.emplace(key, std::move(order));
  return out;
}

template <int D, bool BF16>
static int launch_bwd_variant(const BwdArgs& a, cudaStream_t stream) {
  constexpr int QS = (D == 128) ? 4 : 6;  // 64-query stages of the dK/dV kernel
  constexpr int KR = (D == 128) ? 3 : 6;  // K slots of the dQ kernel
  constexpr int VR = (D == 128) ? 3 : 6;  // V slots of the dQ kernel (dO takes one tile too)
  using LK = KvLayout<D, QS>;
  using LQ = QLayout<D, KR, VR>;
  const uint64_t bhq = static_cast<uint64_t>(a.B) * a.Hq;
  const uint64_t bhk = static_cast<uint64_t>(a.B) * a.Hkv;
  const uint64_t rb = static_cast<uint64_t>(D) * 2;
  CUtensorMap tk, tv, tdo;
  CUtensorMap tq64, tdo64;  // 64-row boxes: the stages of the dK/dV kernel
  if (!make_tmap_3d(&tq64, a.q, BF16, D, a.N_q, bhq, rb, rb * a.N_q, 64, kStepQ, 1) ||
      !make_tmap_3d(&tdo64, a.dout, BF16, D, a.N_q, bhq, rb, rb * a.N_q, 64, kStepQ, 1))
    return -5;
  if (!make_tmap_3d(&tdo, a.dout, BF16, D, a.N_q, bhq, rb, rb * a.N_q, 64, kBT, 1) ||
      !make_tmap_3d(&tk, a.k, BF16, D, a.N_kv, bhk, rb, rb * a.N_kv, 64, kBT, 1) ||
      !make_tmap_3d(&tv, a.v, BF16, D, a.N_kv, bhk, rb, rb * a.N_kv, 64, kBT, 1))
    return -5;
  BwdParams p;
  const int n_qtiles = (a.N_q + kBT - 1) / kBT;
  const int nqp = n_qtiles * kBT;
  p.lse2 = static_cast<const float*>(a.workspace);
  p.dvec = p.lse2 + bhq * nqp;
  p.q = static_cast<const uint16_t*>(a.q);
  p.k = static_cast<const uint16_t*>(a.k);
  p.v = static_cast<const uint16_t*>(a.v);
  p.dout = static_cast<const uint16_t*>(a.dout);
  p.dq = static_cast<uint16_t*>(a.dq);
  p.dk = static_cast<uint16_t*>(a.dk);
  p.dv = static_cast<uint16_t*>(a.dv);
  p.status = device_status_ptr();
  if (!p.status) return -5;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.G = a.Hq / a.Hkv;
  p.N_q = a.N_q;
  p.N_kv = a.N_kv;
  p.n_qtiles = n_qtiles;
  p.n_kvtiles = (a.N_kv + kBT - 1) / kBT;
  p.nqp = nqp;
  p.causal = a.causal;
  p.scale = a.scale;
  p.sl2 = a.scale * 1.4426950408889634f;
  const long long rows = static_cast<long long>(bhq) * nqp;
  attn_bwd_pre_kernel<D, BF16><<<static_cast<unsigned>((rows * (D / 8) + 255) / 256), 256, 0, stream>>>(
      static_cast<const uint16_t*>(a.o), static_cast<const uint16_t*>(a.dout), a.lse,
      const_cast<float*>(p.lse2), const_cast<float*>(p.dvec), a.N_q, nqp, rows, a.scale);
  if (cudaGetLastError() != cudaSuccess) return -5;
  auto kkv = attn_bwd_dkdv_kernel<D, BF16, QS>;
  auto kq = attn_bwd_dq_kernel<D, BF16, KR, VR>;
  if (cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, LK::kBytes) != cudaSuccess ||
      cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, LQ::kBytes) != cudaSuccess)
    return -5;
  const uint64_t kv_blocks = bhk * p.n_kvtiles;
  const uint64_t q_blocks = bhq * n_qtiles;
  if (kv_blocks > 0x7fffffffull || q_blocks > 0x7fffffffull) return -2;
  const KvOrder* order = kv_order(static_cast<int>(bhk), p.n_kvtiles, n_qtiles, p.G, a.causal,
                                  a.N_kv - a.N_q);
  kkv<<<static_cast<unsigned>(kv_blocks), kKvThreads, LK::kBytes, stream>>>(tq64, tk, tv, tdo64, p,
                                                                            *order);
  if (cudaGetLastError() != cudaSuccess) return -5;
  // dQ as a programmatic dependent of dK/dV: its blocks fill the SMs of dK/dV's tail.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(q_blocks));
  cfg.blockDim = dim3(kQThreads);
  cfg.dynamicSmemBytes = LQ::kBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kq, tk, tv, tdo, p) != cudaSuccess) return -5;
  return cudaGetLastError() == cudaSuccess ? 0 : -5;
}

int launch_attn_bwd(const BwdArgs& a, cudaStream_t stream) {
  if (a.d == 64)
    return a.bf16 ? launch_bwd_variant<64, true>(a, stream) : launch_bwd_variant<64, false>(a, stream);
  if (a.d == 128)
    return a.bf16 ? launch_bwd_variant<128, true>(a, stream) : launch_bwd_variant<128, false>(a, stream);
  return -2;
}

}  // namespace attn
