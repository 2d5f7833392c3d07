// Prefill forward: exact attention, one fused kernel per call, sm_103a.
//
// Schedule (the FA-2 loop of "FlashAttention and GPU Data Movement", section 2): one thread
// block owns one 128-row query tile of one (batch, query head); it streams the 128-key K/V
// tiles of the matching key/value head through shared memory and keeps the online-softmax
// state on chip, writing O and the log-sum-exp once at the end.
//
// Roles inside a thread block (192 threads):
//   warps 0-3  softmax: thread r owns query row r.  Reads S_j from tensor memory, applies the
//              scale, the causal/ragged mask and the online-softmax update ("FlashAttention and
//              GPU Data Movement", section 3.1), writes P_j back to tensor memory as 16-bit
//              pairs, rescales the accumulator when the row maximum moved, and runs the
//              epilogue O = a / l, L = m + ln l.
//   warp 4     TMA producers: lane 0 loads Q once and K_j into a STAGES-deep ring, lane 1
//              loads V_j into its own ring.
//   warp 5     tcgen05 issuer: S_j = Q K_j^T (both operands in shared memory) and
//              O += P_j V_j (P from tensor memory, V from shared memory), fp32 accumulators in
//              tensor memory; allocates and frees the 512 tensor-memory columns.
// Tensor memory: S buffers at columns 0 and 128 (double-buffered so Q K_{j+1}^T runs while the
// softmax of tile j runs), the output accumulator at column 256.
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

constexpr int kBlockM = 128;
constexpr int kBlockN = 128;
constexpr int kFwdThreads = 192;
constexpr int kSoftmaxThreads = 128;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256;
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
  // q_full, k_full[S], v_full[S], k_empty[S], v_empty[S], s_full[2], p_ready, o_done, drain
  static constexpr uint32_t kNumBars = 1 + 4 * STAGES + 2 + 3;
  static constexpr uint32_t kMisc = kBar + kNumBars * 8;  // tmem slot, abort flag
  static constexpr uint32_t kBytes = kMisc + 16 + 1024;   // + alignment slack
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
  const uint32_t bar_p = bars + 8u * (3u + 4u * STAGES);
  const uint32_t bar_o = bars + 8u * (4u + 4u * STAGES);
  const uint32_t bar_drain = bars + 8u * (5u + 4u * STAGES);
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
    mbar_init(bar_p, kSoftmaxThreads);
    mbar_init(bar_o, 1);
    mbar_init(bar_drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 4) {
    // ----------------------------------------------------------------- TMA producers
    // Lane 0 loads Q and the K ring, lane 1 the V ring: a K slot is refilled as soon as its
    // Q K^T finished, a V slot once its P V finished, without one ring waiting on the other.
    if (lane < 2 && n_tiles > 0) {
      const bool is_k = (lane == 0);
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
  } else if (warp == 5) {
    // ----------------------------------------------------------------- tcgen05 issuer
    if (lane == 0 && n_tiles > 0) {
      constexpr uint32_t idesc_qk = make_idesc_f16(BF16, kBlockM, kBlockN, false);
      constexpr uint32_t idesc_pv = make_idesc_f16(BF16, kBlockM, D, true);
      bool ok = wait_bounded(bar_q, 0, abort_flag, p.status);
      // O += P_t V_t for tile t (P_t in the S buffer of tile t, V_t in ring slot t % STAGES).
      auto issue_pv = [&](int t) -> bool {
        if (!wait_bounded(bar_p, t & 1, abort_flag, p.status)) return false;
        const int s = t % STAGES;
        if (!wait_bounded(BAR_V(s), (t / STAGES) & 1, abort_flag, p.status)) return false;
        tc_fence_after();
        const uint32_t p_col = tmem + ((t & 1) ? kColS1 : kColS0);
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk) {
          // V is [keys, d] with d contiguous: the B operand is MN-major.  16 keys per MMA
          // (two 8-row groups, SBO = 1024 B apart); the two 64-column halves of d are
          // separate swizzled sub-tiles (LBO = one sub-tile).
          const uint64_t bdesc = make_sdesc_sw128(sV + s * L::kKVBytes + kk * 16 * 128,
                                                  kSubTile, 1024);
          mma_ts(tmem + kColO, p_col + kk * 8, bdesc, idesc_pv, (t > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar_o);
        mma_commit(BAR_VE(s));  // V slot free
        return true;
      };
      for (int j = 0; ok && j < n_tiles; ++j) {
        const int s = j % STAGES;
        if (!wait_bounded(BAR_K(s), (j / STAGES) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t s_col = tmem + ((j & 1) ? kColS1 : kColS0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          // Q and K are K-major (d contiguous): 16 elements = 32 bytes per MMA inside the
          // 128-byte swizzle row; SBO = 1024 B between 8-row groups.
          const uint32_t off = (kk >> 2) * kSubTile + (kk & 3) * 32;
          const uint64_t adesc = make_sdesc_sw128(sQ + off, 16, 1024);
          const uint64_t bdesc = make_sdesc_sw128(sK + s * L::kKVBytes + off, 16, 1024);
          mma_ss(s_col, adesc, bdesc, idesc_qk, kk > 0 ? 1u : 0u);
        }
        mma_commit(BAR_S(j & 1));
        mma_commit(BAR_KE(s));  // K slot free
        if (j > 0 && !issue_pv(j - 1)) ok = false;
      }
      if (ok) issue_pv(n_tiles - 1);
      // Every MMA this thread issued completes before the block frees tensor memory.
      mma_commit(bar_drain);
      wait_bounded(bar_drain, 0, nullptr, p.status, kDrainLimitNs);
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------------------- softmax + epilogue
    const int r = threadIdx.x;  // query row inside the tile; lane quarter = warp
    const uint32_t row_tmem = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    const int row = q0 + r;
    const int off = p.N_kv - p.N_q;
    const float sl2 = p.sl2;
    float m = -INFINITY;  // running max of the scaled scores, log2 units
    float l = 0.0f;       // running sum of 2^(x - m)
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const uint32_t s_col = (j & 1) ? kColS1 : kColS0;
      if (!warp_wait(BAR_S(j & 1), (j >> 1) & 1, abort_flag, p.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t sr[4][32];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(row_tmem + s_col + c * 32, sr[c]);
      tmem_wait_ld();
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
      float mx[8];
#pragma unroll
      for (int e = 0; e < 8; ++e) mx[e] = x[e];
#pragma unroll
      for (int c = 8; c < kBlockN; c += 8)
#pragma unroll
        for (int e = 0; e < 8; ++e) mx[e] = fmaxf(mx[e], x[c + e]);
      const float tile_max =
          fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      const float m_new = fmaxf(m, tile_max * sl2);
      float alpha = 1.0f;
      if (m_new - m > kRescaleThreshold) {  // also true for the first finite maximum
        alpha = ex2(m - m_new);
        m = m_new;
      }
      const float neg_mu = (m == -INFINITY) ? 0.0f : -m;
      float ps[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      uint32_t pk[2][32];
#pragma unroll
      for (int c = 0; c < kBlockN; c += 2) {
        const float p0 = ex2(fmaf(x[c], sl2, neg_mu));
        const float p1 = ex2(fmaf(x[c + 1], sl2, neg_mu));
        ps[(c >> 1) & 7] += p0 + p1;
        pk[c >> 6][(c >> 1) & 31] = pack2<BF16>(p0, p1);
      }
      l = l * alpha + (((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7])));
      tmem_st32(row_tmem + s_col, pk[0]);
      tmem_st32(row_tmem + s_col + 32, pk[1]);
      if (j > 0) {
        // The previous P V has to finish before the accumulator is touched (and before this
        // tile's P is published, which keeps the p_ready phases in step with the issuer).
        if (!warp_wait(bar_o, (j - 1) & 1, abort_flag, p.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.0f)) {
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
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_p);
    }
    // ------------------------------------------------------------- epilogue
    if (ok && n_tiles > 0) {
      ok = warp_wait(bar_o, (n_tiles - 1) & 1, abort_flag, p.status);
      tc_fence_after();
    }
    const bool have = ok && n_tiles > 0;
    const float inv_l = (l > 0.0f) ? 1.0f / l : 0.0f;
    if (have) {
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(row_tmem + kColO + c * 32, o);
        tmem_wait_ld();
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) {
          uint4 w;
          w.x = pack2<BF16>(__uint_as_float(o[q4 * 8 + 0]) * inv_l, __uint_as_float(o[q4 * 8 + 1]) * inv_l);
          w.y = pack2<BF16>(__uint_as_float(o[q4 * 8 + 2]) * inv_l, __uint_as_float(o[q4 * 8 + 3]) * inv_l);
          w.z = pack2<BF16>(__uint_as_float(o[q4 * 8 + 4]) * inv_l, __uint_as_float(o[q4 * 8 + 5]) * inv_l);
          w.w = pack2<BF16>(__uint_as_float(o[q4 * 8 + 6]) * inv_l, __uint_as_float(o[q4 * 8 + 7]) * inv_l);
          const uint32_t chunk = c * 4 + q4;  // 16-byte chunk of the row (8 elements)
          uint8_t* dst = gbase + L::kQ + (chunk >> 3) * kSubTile + sw128(r, chunk & 7);
          *reinterpret_cast<uint4*>(dst) = w;
        }
      }
    } else if (ok) {
      // No key visible to any row of this tile: O = 0.
      for (int chunk = 0; chunk < D / 8; ++chunk) {
        uint8_t* dst = gbase + L::kQ + (chunk >> 3) * kSubTile + sw128(r, chunk & 7);
        *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
      }
    }
    fence_proxy_async_smem();
    named_bar_sync(1, kSoftmaxThreads);
    if (ok && r == 0 && *abort_flag == 0) {
#pragma unroll
      for (int sub = 0; sub < D / 64; ++sub) tma_store_3d(&tm_o, sQ + sub * kSubTile, sub * 64, q0, bh);
      tma_store_commit();
      tma_store_wait_read0();
    }
    if (ok && row < p.N_q) {
      const float mu = (m == -INFINITY) ? 0.0f : m;
      p.lse[static_cast<size_t>(bh) * p.N_q + row] =
          (l > 0.0f) ? (mu + lg2(l)) * 0.69314718055994531f : -INFINITY;
    }
  }
#undef BAR_K
#undef BAR_V
#undef BAR_KE
#undef BAR_VE
#undef BAR_S
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
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
