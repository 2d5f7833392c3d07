// FP8 forward with incoherent processing: the preparation of the 8-bit operands.
//
// "FlashAttention Explained", section "FP8 Attention and Incoherent Processing": Q and K are
// multiplied by the same random orthogonal matrix M = H diag(s) / sqrt(d) (a Hadamard transform
// with random sign flips) before quantisation, so that (Q M)(K M)^T = Q K^T while outlier
// channels spread over all channels, and the operands are quantised to E4M3 with per-block
// scaling factors.  This file writes, from the 16-bit inputs:
//   Q8, K8   E4M3 codes of the rotated rows, [planes, N, d], one scale per 128-row tile
//            (amax of the rotated tile / 448);
//   V^T8     E4M3 codes of V (not rotated), transposed to [planes, d, nkvp] (the K-major B
//            operand of the 8-bit P V product), one scale per plane;
// then runs the FP8 variant of the prefill kernel on them.  The rotation runs in fp32 with the
// fast Walsh-Hadamard butterflies in a fixed order (stage h = 1, 2, ..., d/2: (a, b) ->
// (a + b, a - b)), then one multiply by the fp32 value of 1/sqrt(d); the codes are
// E4M3(x / scale) with an IEEE division, nearest even, saturating.
#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace attn {

namespace {

constexpr int kT = 128;  // rows of a tile

template <bool BF16>
__device__ __forceinline__ float load_half(const uint16_t* p) {
  const uint32_t h = *p;
  if constexpr (BF16) {
    return __uint_as_float(h << 16);
  } else {
    float f;
    asm("{\n\t.reg .f16 t;\n\tmov.b16 t, %1;\n\tcvt.f32.f16 %0, t;\n\t}" : "=f"(f) : "h"(static_cast<uint16_t>(h)));
    return f;
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

}  // namespace

// One block per (plane, 128-row tile), thread = row: rotate (optional), tile amax, quantise.
template <int D, bool BF16>
__global__ void __launch_bounds__(kT)
    fp8_rotate_quantize_kernel(const uint16_t* x, const int8_t* signs, float inv_sqrt_d,
                               uint8_t* codes, float* scales, int N, int n_tiles) {
  __shared__ float red[kT / 32];
  const int plane = blockIdx.x / n_tiles;
  const int tile = blockIdx.x % n_tiles;
  const int row = tile * kT + threadIdx.x;
  const bool live = row < N;
  float v[D];
  const uint16_t* src = x + (static_cast<size_t>(plane) * N + (live ? row : 0)) * D;
#pragma unroll
  for (int c = 0; c < D; ++c) v[c] = live ? load_half<BF16>(src + c) : 0.0f;
  if (signs) {
#pragma unroll
    for (int c = 0; c < D; ++c) v[c] = signs[c] < 0 ? -v[c] : v[c];
#pragma unroll
    for (int h = 1; h < D; h <<= 1)
#pragma unroll
      for (int j = 0; j < D; ++j)
        if ((j & h) == 0) {
          const float a = v[j], b = v[j + h];
          v[j] = a + b;
          v[j + h] = a - b;
        }
#pragma unroll
    for (int c = 0; c < D; ++c) v[c] = v[c] * inv_sqrt_d;
  }
  float amax = 0.0f;
#pragma unroll
  for (int c = 0; c < D; ++c) amax = fmaxf(amax, fabsf(v[c]));
  amax = block_max(amax, red);
  const float scale = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  if (threadIdx.x == 0) scales[blockIdx.x] = scale;
  if (!live) return;
  uint4* dst = reinterpret_cast<uint4*>(codes + (static_cast<size_t>(plane) * N + row) * D);
#pragma unroll
  for (int c = 0; c < D; c += 16) {
    uint4 w;
    w.x = pack4_e4m3(__fdiv_rn(v[c + 0], scale), __fdiv_rn(v[c + 1], scale),
                     __fdiv_rn(v[c + 2], scale), __fdiv_rn(v[c + 3], scale));
    w.y = pack4_e4m3(__fdiv_rn(v[c + 4], scale), __fdiv_rn(v[c + 5], scale),
                     __fdiv_rn(v[c + 6], scale), __fdiv_rn(v[c + 7], scale));
    w.z = pack4_e4m3(__fdiv_rn(v[c + 8], scale), __fdiv_rn(v[c + 9], scale),
                     __fdiv_rn(v[c + 10], scale), __fdiv_rn(v[c + 11], scale));
    w.w = pack4_e4m3(__fdiv_rn(v[c + 12], scale), __fdiv_rn(v[c + 13], scale),
                     __fdiv_rn(v[c + 14], scale), __fdiv_rn(v[c + 15], scale));
    dst[c / 16] = w;
  }
}

// Per-plane amax of V (non-negative floats order as their bit patterns).
template <int D, bool BF16>
__global__ void fp8_plane_amax_kernel(const uint16_t* x, unsigned* amax_bits, int N, int n_tiles) {
  __shared__ float red[kT / 32];
  const int plane = blockIdx.x / n_tiles;
  const int row = (blockIdx.x % n_tiles) * kT + threadIdx.x;
  float m = 0.0f;
  if (row < N) {
    const uint16_t* src = x + (static_cast<size_t>(plane) * N + row) * D;
#pragma unroll 8
    for (int c = 0; c < D; ++c) m = fmaxf(m, fabsf(load_half<BF16>(src + c)));
  }
  m = block_max(m, red);
  if (threadIdx.x == 0) atomicMax(amax_bits + plane, __float_as_uint(m));
}

// V -> E4M3 codes transposed to [plane, d, nkvp]; one block per (plane, 128-key tile), thread =
// key; keys past N get code 0.  The block's 128 keys x d codes pass through shared memory so
// that each output row (one channel, 128 keys) is written with 16-byte stores.
template <int D, bool BF16>
__global__ void __launch_bounds__(kT)
    fp8_v_transpose_kernel(const uint16_t* x, const unsigned* amax_bits, float* scales,
                           uint8_t* vt, int N, int n_tiles, int nkvp) {
  __shared__ __align__(16) uint8_t tile[D][kT];
  const int plane = blockIdx.x / n_tiles;
  const int kt = blockIdx.x % n_tiles;
  const int key = kt * kT + threadIdx.x;
  const float amax = __uint_as_float(amax_bits[plane]);
  const float scale = amax > 0.0f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  if (kt == 0 && threadIdx.x == 0) scales[plane] = scale;
  const uint16_t* src = x + (static_cast<size_t>(plane) * N + (key < N ? key : 0)) * D;
#pragma unroll 4
  for (int c = 0; c < D; c += 4) {
    uint32_t w = 0;
    if (key < N)
      w = pack4_e4m3(__fdiv_rn(load_half<BF16>(src + c), scale),
                     __fdiv_rn(load_half<BF16>(src + c + 1), scale),
                     __fdiv_rn(load_half<BF16>(src + c + 2), scale),
                     __fdiv_rn(load_half<BF16>(src + c + 3), scale));
    tile[c][threadIdx.x] = w & 0xff;
    tile[c + 1][threadIdx.x] = (w >> 8) & 0xff;
    tile[c + 2][threadIdx.x] = (w >> 16) & 0xff;
    tile[c + 3][threadIdx.x] = w >> 24;
  }
  __syncthreads();
  for (int i = threadIdx.x; i < D * (kT / 16); i += kT) {
    const int c = i / (kT / 16), part = i % (kT / 16);
    *reinterpret_cast<uint4*>(vt + (static_cast<size_t>(plane) * D + c) * nkvp + kt * kT + part * 16) =
        *reinterpret_cast<const uint4*>(&tile[c][part * 16]);
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
    fp8_rotate_quantize_kernel<D, BF><<<pq * nqt, kT, 0, stream>>>(
        static_cast<const uint16_t*>(a.q), signs, inv_sqrt_d, static_cast<uint8_t*>(const_cast<void*>(f.q8)),
        const_cast<float*>(f.q_scale), a.N_q, nqt);
    fp8_rotate_quantize_kernel<D, BF><<<pk * nkt, kT, 0, stream>>>(
        static_cast<const uint16_t*>(a.k), signs, inv_sqrt_d, static_cast<uint8_t*>(const_cast<void*>(f.k8)),
        const_cast<float*>(f.k_scale), a.N_kv, nkt);
    fp8_plane_amax_kernel<D, BF><<<pk * nkt, kT, 0, stream>>>(static_cast<const uint16_t*>(a.v), amax,
                                                              a.N_kv, nkt);
    fp8_v_transpose_kernel<D, BF><<<pk * nkt, kT, 0, stream>>>(
        static_cast<const uint16_t*>(a.v), amax, const_cast<float*>(f.v_scale),
        static_cast<uint8_t*>(const_cast<void*>(f.vt8)), a.N_kv, nkt, f.nkvp);
    return cudaGetLastError() == cudaSuccess ? 0 : -5;
  };
  const int st = a.bf16 ? run(std::true_type{}) : run(std::false_type{});
  if (st != 0) return st;
  return launch_attn_fwd_fp8_kernel(f, stream);
}

}  // namespace attn
