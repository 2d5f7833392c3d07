// FP8 forward with incoherent processing: the preparation of the 8-bit operands.
//
// "FlashAttention Explained", section "FP8 Attention and Incoherent Processing": Q and K are
// multiplied by the same random orthogonal matrix M = H diag(s) / sqrt(d) (a Hadamard transform
// with random sign flips) before quantisation, so that (Q M)(K M)^T = Q K^T while outlier
// channels spread over all channels, and the operands are quantised to E4M3 with per-block
// scaling factors.  This file writes, from the 16-bit inputs:
//   Q8, K8   E4M3 codes of the rotated rows, [planes, N, d], one scale per 128-row tile;
//   V^T8     E4M3 codes of V (not rotated), transposed to [planes, d, nkvp] (the K-major B
//            operand of the 8-bit P V product), one scale per plane;
// then runs the FP8 variant of the prefill kernel on them.  A block's scale is a power of two:
// the smallest 2^e with amax <= 448 * 2^e (448 is E4M3's largest value), so that the codes
// E4M3(x * 2^-e) (nearest even, saturating) come from an exact multiply instead of a division.
// The rotation runs in fp32 with the fast Walsh-Hadamard butterflies in a fixed order (stage
// h = 1, 2, ..., d/2: (a, b) -> (a + b, a - b)), then one multiply by the fp32 value of
// 1/sqrt(d).
#include <atomic>
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace attn {

namespace {

constexpr int kT = 128;        // rows of a tile
constexpr int kPrepThreads = 256;
constexpr int kPrepWarps = kPrepThreads / 32;

// Eight consecutive 16-bit values (16 bytes) as floats.
template <bool BF16>
__device__ __forceinline__ void load8(const uint16_t* p, float v[8]) {
  const uint4 w = *reinterpret_cast<const uint4*>(p);
  const uint32_t h[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (BF16) {
      v[2 * i] = __uint_as_float(h[i] << 16);
      v[2 * i + 1] = __uint_as_float(h[i] & 0xffff0000u);
    } else {
      float lo, hi;
      asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\t"
          "cvt.f32.f16 %1, b;\n\t}"
          : "=f"(lo), "=f"(hi)
          : "r"(h[i]));
      v[2 * i] = lo;
      v[2 * i + 1] = hi;
    }
  }
}

// Eight 16-bit values already loaded (16 bytes) as floats.
template <bool BF16>
__device__ __forceinline__ void load8_words(const uint4 w, float v[8]) {
  const uint32_t h[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (BF16) {
      v[2 * i] = __uint_as_float(h[i] << 16);
      v[2 * i + 1] = __uint_as_float(h[i] & 0xffff0000u);
    } else {
      float lo, hi;
      asm("{\n\t.reg .f16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\t"
          "cvt.f32.f16 %1, b;\n\t}"
          : "=f"(lo), "=f"(hi)
          : "r"(h[i]));
      v[2 * i] = lo;
      v[2 * i + 1] = hi;
    }
  }
}

__device__ __forceinline__ float block_max(float v, float* red) {
  for (int sh = 16; sh > 0; sh >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, sh));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float m = red[0];
  for (int w = 1; w < static_cast<int>(blockDim.x >> 5); ++w) m = fmaxf(m, red[w]);
  __syncthreads();
  return m;
}

// Exponent e of a block's scale 2^e: the smallest with amax <= 448 * 2^e, at least -126 so
// that 2^e and 2^-e are normal fp32 values; 0 for an all-zero block.  With amax = (1 + M/2^23)
// 2^(E-127), amax <= 1.75 * 2^(8+e) holds from e = E - 135 when the mantissa is at most 0.75
// (1.75 = 448 / 2^8), from e = E - 134 otherwise.
__device__ __forceinline__ int scale_exp(float amax) {
  if (!(amax > 0.0f)) return 0;
  const uint32_t b = __float_as_uint(amax);
  const int E = static_cast<int>((b >> 23) & 0xffu);
  const int e = ((b & 0x7fffffu) <= 0x600000u) ? E - 135 : E - 134;
  return e < -126 ? -126 : e;
}

__device__ __forceinline__ float exp2i(int e) {  // 2^e for -126 <= e <= 127
  return __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
}

}  // namespace

// Rotation and quantisation of Q and K in one persistent launch: the (plane, 128-row tile)
// tiles of Q and then those of K, numbered in that order, go round-robin over the blocks.  A
// tile's two 64-channel halves come in by TMA (128-byte swizzle) into a four-deep ring, so
// that the next three tiles load while this one is computed (one block per SM); threads 2r and 2r + 1 take channels
// 0-63 and 64-127 of row r (reading their 16-byte chunks at the swizzled positions, free of
// bank conflicts), apply the sign flips, run the butterfly stages h = 1 .. 32 in registers in
// the plain order and stage h = 64 across the thread pair (the lower keeps a + b, the upper
// computes a - b from the value it receives: the same fp32 operations), then x fp32(1/sqrt(d)),
// the tile amax by a block reduction, the power-of-two scale and the codes by an exact multiply.
// The codes go to a swizzled staging buffer (two, alternating by tile) and out by one TMA store.
constexpr int kRotThreads = 2 * kT;
constexpr int kRotStages = 4;
constexpr uint32_t kRotHalf = kT * 64 * 2;        // one 64-channel half of a 16-bit tile
constexpr uint32_t kRotIn = 2 * kRotHalf;          // a 16-bit tile (two halves)
constexpr uint32_t kRotCodes = kT * 128;           // a tile of codes
constexpr uint32_t kRotBars = kRotStages * kRotIn + 2 * kRotCodes;
constexpr uint32_t kRotSmem = kRotBars + kRotStages * 8 + 2 * 8 * 4 + 1024;  // + alignment

template <int D, bool BF16>
__global__ void __launch_bounds__(kRotThreads, 1)
    fp8_rotate_quantize_kernel(const __grid_constant__ CUtensorMap tm_q,
                               const __grid_constant__ CUtensorMap tm_k,
                               const __grid_constant__ CUtensorMap tm_q8,
                               const __grid_constant__ CUtensorMap tm_k8, const int8_t* signs,
                               float inv_sqrt_d, float* sq, float* sk, int nqt, int nkt,
                               int q_tiles, int n_tiles, int* status) {
  static_assert(D == 128, "two 64-channel halves per row");
  constexpr int kH = D / 2;  // channels per thread
  extern __shared__ uint8_t rot_smem[];
  const uint32_t raw = smem_u32(rot_smem);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = rot_smem + (base - raw);
  const uint32_t bars = base + kRotBars;
  float* red = reinterpret_cast<float*>(gbase + kRotBars + kRotStages * 8);  // [2][8]
  const int my_row = threadIdx.x >> 1, half = threadIdx.x & 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // this block's tiles: blockIdx.x, blockIdx.x + gridDim.x, ...
  const int my_tiles =
      static_cast<int>(blockIdx.x) < n_tiles ? (n_tiles - 1 - static_cast<int>(blockIdx.x)) / gridDim.x + 1 : 0;
  auto load_tile = [&](int i) {  // this block's i-th tile into stage i % kRotStages
    const int t = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
    const bool is_q = t < q_tiles;
    const int b = is_q ? t : t - q_tiles;
    const int nt = is_q ? nqt : nkt;
    const uint32_t st = base + (i % kRotStages) * kRotIn;
    const uint32_t bar = bars + 8u * (i % kRotStages);
    mbar_arrive_expect_tx(bar, kRotIn);
#pragma unroll
    for (int h = 0; h < 2; ++h)
      tma_load_3d(st + h * kRotHalf, is_q ? &tm_q : &tm_k, bar, h * 64, (b % nt) * kT, b / nt);
  };
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRotStages; ++s) mbar_init(bars + 8u * s, 1);
    fence_barrier_init();
  }
  __syncthreads();
  int issued = 0;  // tiles whose loads thread 0 has issued
  if (threadIdx.x == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    for (; issued < kRotStages && issued < my_tiles; ++issued) load_tile(issued);
  }
  // signs of this thread's 64 channels as two 32-bit masks (bit c set: channel negated)
  uint32_t neg[kH / 32] = {};
  if (signs) {
    uint32_t all[D / 32];
#pragma unroll
    for (int q = 0; q < D / 32; ++q) all[q] = __ballot_sync(0xffffffffu, signs[q * 32 + lane] < 0);
#pragma unroll
    for (int q = 0; q < kH / 32; ++q) neg[q] = half ? all[kH / 32 + q] : all[q];
  }
  bool ok = true;
  int consumed = 0;  // tiles whose loads every thread has seen land
  for (int i = 0; i < my_tiles; ++i) {
    const int t = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
    const bool is_q = t < q_tiles;
    const int b = is_q ? t : t - q_tiles;
    const int nt = is_q ? nqt : nkt;
    const int s = i % kRotStages;
    const bool landed = wait_bounded(bars + 8u * s, (i / kRotStages) & 1, nullptr, status);
    if (!__syncthreads_and(landed)) {
      ok = false;
      break;
    }
    consumed = i + 1;
    // 1. this thread's half row (16-byte chunk c of the row sits at chunk c ^ (row % 8))
    const uint8_t* src = gbase + s * kRotIn + half * kRotHalf;
    float v[kH];
#pragma unroll
    for (int c = 0; c < kH / 8; ++c) {
      const uint4 w = *reinterpret_cast<const uint4*>(src + sw128(my_row, c));
      float f[8];
      load8_words<BF16>(w, f);
#pragma unroll
      for (int e = 0; e < 8; ++e) v[c * 8 + e] = f[e];
    }
    if (signs) {
#pragma unroll
      for (int c = 0; c < kH; ++c)
        v[c] = __int_as_float(__float_as_int(v[c]) ^ (((neg[c >> 5] >> (c & 31)) & 1u) << 31));
#pragma unroll
      for (int h = 1; h < kH; h <<= 1)
#pragma unroll
        for (int j = 0; j < kH; ++j)
          if ((j & h) == 0) {
            const float a = v[j], c = v[j + h];
            v[j] = a + c;
            v[j + h] = a - c;
          }
      // h = 64: element j of the lower half with element j of the upper half
#pragma unroll
      for (int j = 0; j < kH; ++j) {
        const float other = __shfl_xor_sync(0xffffffffu, v[j], 1);
        v[j] = half ? other - v[j] : v[j] + other;
      }
#pragma unroll
      for (int c = 0; c < kH; ++c) v[c] = v[c] * inv_sqrt_d;
    }
    float amax = 0.0f;
#pragma unroll
    for (int c = 0; c < kH; ++c) amax = fmaxf(amax, fabsf(v[c]));
    // 2. tile amax (reduction slots alternate by tile); the block barrier also ends every read
    // of stage s and, through thread 0's wait before it, the store that last read this tile's
    // staging buffer
    for (int sh = 16; sh > 0; sh >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, sh));
    if (lane == 0) red[(i & 1) * 8 + warp] = amax;
    if (threadIdx.x == 0) tma_store_wait_read1();
    __syncthreads();
    if (threadIdx.x == 0 && issued < my_tiles) load_tile(issued++);
    float m = red[(i & 1) * 8];
#pragma unroll
    for (int w = 1; w < kRotThreads / 32; ++w) m = fmaxf(m, red[(i & 1) * 8 + w]);
    const int e = scale_exp(m);
    if (threadIdx.x == 0) (is_q ? sq : sk)[b] = exp2i(e);
    const float inv = exp2i(-e);
    // 3. codes: row r's 128 bytes, chunk c at chunk c ^ (r % 8) of staging buffer i % 2
    uint8_t* codes = gbase + kRotStages * kRotIn + (i & 1) * kRotCodes;
#pragma unroll
    for (int c = 0; c < kH; c += 16) {
      uint4 w;
      w.x = pack4_e4m3(v[c + 0] * inv, v[c + 1] * inv, v[c + 2] * inv, v[c + 3] * inv);
      w.y = pack4_e4m3(v[c + 4] * inv, v[c + 5] * inv, v[c + 6] * inv, v[c + 7] * inv);
      w.z = pack4_e4m3(v[c + 8] * inv, v[c + 9] * inv, v[c + 10] * inv, v[c + 11] * inv);
      w.w = pack4_e4m3(v[c + 12] * inv, v[c + 13] * inv, v[c + 14] * inv, v[c + 15] * inv);
      *reinterpret_cast<uint4*>(codes + sw128(my_row, half * 4 + c / 16)) = w;
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (threadIdx.x == 0) {
      tma_store_3d(is_q ? &tm_q8 : &tm_k8, smem_u32(codes), 0, (b % nt) * kT, b / nt);
      tma_store_commit();
    }
  }
  if (threadIdx.x == 0) {
    tma_store_wait_all();  // every code tile written before the block exits
    // loads issued but not consumed (after a time-out) land before the shared memory goes away
    for (int j = consumed; j < issued; ++j)
      wait_bounded(bars + 8u * (j % kRotStages), (j / kRotStages) & 1, nullptr, status,
                   100000000ull);
  }
}

// Per-plane amax of V over 128-row tiles, 16-byte loads (non-negative floats order as their bit
// patterns, so an integer atomicMax takes the maximum).
template <int D, bool BF16>
__global__ void __launch_bounds__(kPrepThreads)
    fp8_plane_amax_kernel(const uint16_t* x, unsigned* amax_bits, int N, int n_tiles) {
  __shared__ float red[kPrepWarps];
  const int plane = blockIdx.x / n_tiles, tile = blockIdx.x % n_tiles;
  const int rows = min(kT, N - tile * kT);
  const uint16_t* src = x + (static_cast<size_t>(plane) * N + static_cast<size_t>(tile) * kT) * D;
  float m = 0.0f;
  for (int c = threadIdx.x; c < rows * (D / 8); c += kPrepThreads) {
    float v[8];
    load8<BF16>(src + static_cast<size_t>(c) * 8, v);
#pragma unroll
    for (int e = 0; e < 8; ++e) m = fmaxf(m, fabsf(v[e]));
  }
  m = block_max(m, red);
  if (threadIdx.x == 0) atomicMax(amax_bits + plane, __float_as_uint(m));
}

// V -> E4M3 codes transposed to [plane, d, nkvp]; one block per (plane, 128-key tile); keys past
// N get code 0.  A thread converts four keys x eight channels (four 16-byte loads, sixteen lanes
// covering a row), regroups the codes into one 4-key word per channel and stores the words into
// a shared [d][128 + 4]-byte tile; the tile's rows then go out as 128-byte coalesced rows.
template <int D, bool BF16>
__global__ void __launch_bounds__(kPrepThreads)
    fp8_v_transpose_kernel(const uint16_t* x, const unsigned* amax_bits, float* scales,
                           uint8_t* vt, int N, int n_tiles, int nkvp) {
  constexpr int kPitch = kT + 4;  // bytes per channel row in shared memory
  __shared__ __align__(16) uint8_t tile[D * kPitch];
  const int plane = blockIdx.x / n_tiles, kt = blockIdx.x % n_tiles;
  const int e = scale_exp(__uint_as_float(amax_bits[plane]));
  if (kt == 0 && threadIdx.x == 0) scales[plane] = exp2i(e);
  const float inv = exp2i(-e);
  const uint16_t* src = x + static_cast<size_t>(plane) * N * D;
  constexpr int kChunks = D / 8;                 // 8-channel chunks of a row
  constexpr int kUnits = (kT / 4) * kChunks;     // (key quad, chunk) pairs
  for (int u = threadIdx.x; u < kUnits; u += kPrepThreads) {
    const int chunk = u % kChunks, quad = u / kChunks;
    uint32_t w[4][2];  // codes of key kq*4 + r, channels 8 chunk .. +7
#pragma unroll
    for (int r = 0; r < 4; ++r) {
      const int key = kt * kT + quad * 4 + r;
      if (key < N) {
        float v[8];
        load8<BF16>(src + static_cast<size_t>(key) * D + chunk * 8, v);
        w[r][0] = pack4_e4m3(v[0] * inv, v[1] * inv, v[2] * inv, v[3] * inv);
        w[r][1] = pack4_e4m3(v[4] * inv, v[5] * inv, v[6] * inv, v[7] * inv);
      } else {
        w[r][0] = w[r][1] = 0u;
      }
    }
    // channel e of the chunk: byte e % 4 of word e / 4 of each key -> one word of four keys
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int h = e >> 2, sh = (e & 3) * 8;
      const uint32_t word = ((w[0][h] >> sh) & 0xffu) | (((w[1][h] >> sh) & 0xffu) << 8) |
                            (((w[2][h] >> sh) & 0xffu) << 16) | (((w[3][h] >> sh) & 0xffu) << 24);
      *reinterpret_cast<uint32_t*>(tile + (chunk * 8 + e) * kPitch + quad * 4) = word;
    }
  }
  __syncthreads();
  for (int u = threadIdx.x; u < D * (kT / 4); u += kPrepThreads) {
    const int c = u / (kT / 4), word = u % (kT / 4);
    *reinterpret_cast<uint32_t*>(vt + (static_cast<size_t>(plane) * D + c) * nkvp + kt * kT +
                                 word * 4) = *reinterpret_cast<const uint32_t*>(tile + c * kPitch + word * 4);
  }
}

// ------------------------------------------------------------------------------------------
// workspace and launch
// ------------------------------------------------------------------------------------------
static size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

size_t fp8_workspace_layout(int B, int Hq, int Hkv, int N_q, int N_kv, int d, size_t off[7]) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || N_q <= 0 || N_kv <= 0 || d <= 0) return 0;
  const size_t pq = static_cast<size_t>(B) * Hq, pk = static_cast<size_t>(B) * Hkv;
  const size_t nqt = (static_cast<size_t>(N_q) + kT - 1) / kT;
  const size_t nkt = (static_cast<size_t>(N_kv) + kT - 1) / kT;
  const size_t nkvp = nkt * kT;
  size_t o = 0;
  off[0] = o; o = align256(o + pq * N_q * d);     // Q8
  off[1] = o; o = align256(o + pk * N_kv * d);    // K8
  off[2] = o; o = align256(o + pk * d * nkvp);    // V^T8
  off[3] = o; o = align256(o + pq * nqt * 4);     // Q scales
  off[4] = o; o = align256(o + pk * nkt * 4);     // K scales
  off[5] = o; o = align256(o + pk * 4);           // V scales
  off[6] = o; o = align256(o + pk * 4);           // V amax scratch
  return o;
}

int launch_attn_fwd_fp8(const FwdArgs& a, const int8_t* signs, void* workspace,
                        cudaStream_t stream) {
  if (a.d != 128) return -2;
  constexpr int D = 128;
  size_t off[7];
  if (fp8_workspace_layout(a.B, a.Hq, a.Hkv, a.N_q, a.N_kv, a.d, off) == 0) return -1;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int pq = a.B * a.Hq, pk = a.B * a.Hkv;
  const int nqt = (a.N_q + kT - 1) / kT, nkt = (a.N_kv + kT - 1) / kT;
  // the fp32 value of 1/sqrt(d), as an fp32 division of fp32 values
  const float inv_sqrt_d = 1.0f / sqrtf(static_cast<float>(D));
  FwdArgs f = a;
  f.q8 = ws + off[0];
  f.k8 = ws + off[1];
  f.vt8 = ws + off[2];
  f.q_scale = reinterpret_cast<float*>(ws + off[3]);
  f.k_scale = reinterpret_cast<float*>(ws + off[4]);
  f.v_scale = reinterpret_cast<float*>(ws + off[5]);
  f.nkvp = nkt * kT;
  unsigned* amax = reinterpret_cast<unsigned*>(ws + off[6]);
  if (cudaMemsetAsync(amax, 0, static_cast<size_t>(pk) * 4, stream) != cudaSuccess) return -5;
  auto run = [&](auto bf16_tag) -> int {
    constexpr bool BF = decltype(bf16_tag)::value;
    const uint16_t* v16 = static_cast<const uint16_t*>(a.v);
    CUtensorMap tq, tk, tq8, tk8;
    const uint64_t rb = static_cast<uint64_t>(D) * 2;
    if (!make_tmap_3d(&tq, a.q, BF, D, a.N_q, pq, rb, rb * a.N_q, 64, kT, 1) ||
        !make_tmap_3d(&tk, a.k, BF, D, a.N_kv, pk, rb, rb * a.N_kv, 64, kT, 1) ||
        !make_tmap_3d_u8(&tq8, f.q8, D, a.N_q, pq, D, static_cast<uint64_t>(D) * a.N_q, D, kT, 1) ||
        !make_tmap_3d_u8(&tk8, f.k8, D, a.N_kv, pk, D, static_cast<uint64_t>(D) * a.N_kv, D, kT, 1))
      return -5;
    int* status = device_status_ptr();
    if (!status) return -5;
    auto kern = fp8_rotate_quantize_kernel<D, BF>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kRotSmem) !=
        cudaSuccess)
      return -5;
    static std::atomic<int> n_sm{0};
    if (n_sm.load() == 0) {
      int dev = 0, v = 0;
      if (cudaGetDevice(&dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
        return -5;
      n_sm.store(v);
    }
    const int tiles = pq * nqt + pk * nkt;
    const int grid = tiles < n_sm.load() ? tiles : n_sm.load();  // one block per SM
    kern<<<grid, kRotThreads, kRotSmem, stream>>>(
        tq, tk, tq8, tk8, signs, inv_sqrt_d, const_cast<float*>(f.q_scale),
        const_cast<float*>(f.k_scale), nqt, nkt, pq * nqt, tiles, status);
    fp8_plane_amax_kernel<D, BF><<<pk * nkt, kPrepThreads, 0, stream>>>(v16, amax, a.N_kv, nkt);
    fp8_v_transpose_kernel<D, BF><<<pk * nkt, kPrepThreads, 0, stream>>>(
        v16, amax, const_cast<float*>(f.v_scale), static_cast<uint8_t*>(const_cast<void*>(f.vt8)),
        a.N_kv, nkt, f.nkvp);
    return cudaGetLastError() == cudaSuccess ? 0 : -5;
  };
  const int st = a.bf16 ? run(std::true_type{}) : run(std::false_type{});
  if (st != 0) return st;
  return launch_attn_fwd_fp8_kernel(f, stream);
}

}  // namespace attn
