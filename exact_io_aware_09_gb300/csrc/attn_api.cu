// C ABI of libattn_gb300.so: argument checks, TMA descriptors, the device status word and the
// timeout self-test.  The kernels live in attn_fwd.cu and attn_decode.cu.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/attn.h"
#include "internal.h"
#include "ptx.cuh"

namespace attn {

__device__ int g_status;  // first device-side error since the last attn_poll_status

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices];
std::mutex g_status_mu;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The kernels use tcgen05 and are built for sm_103a only.  `data` (one of the call's buffers,
// or null) must not be another GPU's memory: the launch goes to the current device, whose
// kernels could not reach it.  Host memory the GPU can address is left to the caller.
int check_device(const void* data) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_DEVICE;
  static std::atomic<int> checked[kMaxDevices];  // 0 unknown, 1 ok, 2 not usable
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_DEVICE;
  int known = checked[dev].load(std::memory_order_relaxed);
  if (known == 0) {
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return ATTN_ERR_DEVICE;
    known = (prop.major == 10 && prop.minor == 3) ? 1 : 2;
    checked[dev].store(known, std::memory_order_relaxed);
  }
  if (known != 1) return ATTN_ERR_DEVICE;
  if (data) {
    cudaPointerAttributes pa;
    if (cudaPointerGetAttributes(&pa, data) != cudaSuccess) {
      (void)cudaGetLastError();
      return ATTN_ERR_INVALID_ARG;
    }
    if (pa.type == cudaMemoryTypeDevice && pa.device != dev) return ATTN_ERR_INVALID_ARG;
  }
  return ATTN_OK;
}

}  // namespace

bool make_tmap_3d(CUtensorMap* map, const void* base, bool bf16, uint64_t dim0, uint64_t dim1,
                  uint64_t dim2, uint64_t stride1, uint64_t stride2, uint32_t box0,
                  uint32_t box1, uint32_t box2) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || dim0 == 0 || dim1 == 0 || dim2 == 0) return false;
  const cuuint64_t dims[3] = {dim0, dim1, dim2};
  const cuuint64_t strides[2] = {stride1, stride2};
  const cuuint32_t box[3] = {box0, box1, box2};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r =
      fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
         const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_4d(CUtensorMap* map, const void* base, bool bf16, const uint64_t dims[4],
                  const uint64_t strides[3], const uint32_t box[4]) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || dims[0] == 0 || dims[1] == 0 || dims[2] == 0 || dims[3] == 0) return false;
  const cuuint64_t d[4] = {dims[0], dims[1], dims[2], dims[3]};
  const cuuint64_t st[3] = {strides[0], strides[1], strides[2]};
  const cuuint32_t bx[4] = {box[0], box[1], box[2], box[3]};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r =
      fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
         const_cast<void*>(base), d, st, bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool make_tmap_3d_u8(CUtensorMap* map, const void* base, uint64_t dim0, uint64_t dim1,
                     uint64_t dim2, uint64_t stride1, uint64_t stride2, uint32_t box0,
                     uint32_t box1, uint32_t box2) {
  EncodeTiledFn fn = encode_fn();
  if (!fn || dim0 == 0 || dim1 == 0 || dim2 == 0) return false;
  const cuuint64_t dims[3] = {dim0, dim1, dim2};
  const cuuint64_t strides[2] = {stride1, stride2};
  const cuuint32_t box[3] = {box0, box1, box2};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

int* device_status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_status_mu);
  if (!g_status_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<int*>(p);
  }
  return g_status_ptr[dev];
}

// Waits on a barrier no one arrives at, for `limit_ns`, then latches the time-out status.
__global__ void selftest_timeout_kernel(int* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_barrier_init();
  }
  __syncthreads();
  wait_bounded(smem_u32(&bar), 0, nullptr, status, limit_ns);
}

// Dispatch order of the dK/dV kernel's blocks (attn_bwd.cu): job of every block in job[0 .. n),
// n returned; 0 = the default order.
int bwd_kv_order(int n_planes, int n_kvtiles, int n_qtiles, int G, int causal, int off, int n_sm,
                 uint16_t* job, int cap);

}  // namespace attn

using namespace attn;

extern "C" {

// The three prefill entry points share their checks and the kernel.
static int fwd_common(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int Hq, int Hkv, int N_q, int N_kv, int d, int causal, int window,
                      const uint8_t* block_mask, float scale, attn_stream_t stream,
                      attn_dtype_t dtype) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || N_q < 0 || N_kv < 0 || Hq % Hkv != 0)
    return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.0f)) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (B == 0 || N_q == 0) return ATTN_OK;
  if (!q || !o || !lse || (N_kv > 0 && (!k || !v))) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(o) || !aligned16(lse) ||
      (N_kv > 0 && (!aligned16(k) || !aligned16(v))))
    return ATTN_ERR_MISALIGNED;
  const int dev_ok = check_device(q);
  if (dev_ok != ATTN_OK) return dev_ok;
  FwdArgs a{q, k, v, o, lse, B, Hq, Hkv, N_q, N_kv, d, causal ? 1 : 0, scale,
            dtype == ATTN_BF16, window, block_mask};
  return launch_attn_fwd(a, reinterpret_cast<cudaStream_t>(stream));
}

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
             int Hkv, int N_q, int N_kv, int d, int causal, float scale, attn_stream_t stream,
             attn_dtype_t dtype) {
  return fwd_common(q, k, v, o, lse, B, Hq, Hkv, N_q, N_kv, d, causal, -1, nullptr, scale,
                    stream, dtype);
}

int attn_fwd_window(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                    int Hq, int Hkv, int N_q, int N_kv, int d, int window, float scale,
                    attn_stream_t stream, attn_dtype_t dtype) {
  if (window < 0) return ATTN_ERR_INVALID_ARG;
  return fwd_common(q, k, v, o, lse, B, Hq, Hkv, N_q, N_kv, d, 1, window, nullptr, scale,
                    stream, dtype);
}

int attn_fwd_block_sparse(const void* q, const void* k, const void* v, void* o, float* lse,
                          int B, int Hq, int Hkv, int N_q, int N_kv, int d, int causal,
                          const uint8_t* block_mask, float scale, attn_stream_t stream,
                          attn_dtype_t dtype) {
  if (!block_mask) return ATTN_ERR_INVALID_ARG;
  return fwd_common(q, k, v, o, lse, B, Hq, Hkv, N_q, N_kv, d, causal, -1, block_mask, scale,
                    stream, dtype);
}

size_t attn_fwd_fp8_workspace_bytes(int B, int Hq, int Hkv, int N_q, int N_kv, int d) {
  size_t off[7];
  return fp8_workspace_layout(B, Hq, Hkv, N_q, N_kv, d, off);
}

int attn_fwd_fp8_workspace_offsets(int B, int Hq, int Hkv, int N_q, int N_kv, int d,
                                   size_t* offsets) {
  if (!offsets) return ATTN_ERR_INVALID_ARG;
  return fp8_workspace_layout(B, Hq, Hkv, N_q, N_kv, d, offsets) ? ATTN_OK : ATTN_ERR_INVALID_ARG;
}

int attn_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B, int Hq,
                 int Hkv, int N_q, int N_kv, int d, int causal, float scale, const int8_t* signs,
                 void* workspace, size_t workspace_bytes, attn_stream_t stream,
                 attn_dtype_t dtype) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || N_q < 0 || N_kv < 0 || Hq % Hkv != 0)
    return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.0f)) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (d != 128) return ATTN_ERR_UNSUPPORTED;
  if (B == 0 || N_q == 0) return ATTN_OK;
  if (N_kv == 0)  // nothing to quantise: O = 0, L = -inf as in attn_fwd
    return fwd_common(q, k, v, o, lse, B, Hq, Hkv, N_q, N_kv, d, causal, -1, nullptr, scale,
                      stream, dtype);
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) ||
      !aligned16(workspace))
    return ATTN_ERR_MISALIGNED;
  if (!workspace || workspace_bytes < attn_fwd_fp8_workspace_bytes(B, Hq, Hkv, N_q, N_kv, d))
    return ATTN_ERR_WORKSPACE;
  const int dev_ok = check_device(q);
  if (dev_ok != ATTN_OK) return dev_ok;
  FwdArgs a{q, k, v, o, lse, B, Hq, Hkv, N_q, N_kv, d, causal ? 1 : 0, scale,
            dtype == ATTN_BF16, -1, nullptr};
  return launch_attn_fwd_fp8(a, signs, workspace, reinterpret_cast<cudaStream_t>(stream));
}

int attn_fwd_kv_span(int q_tile, int block_m, int block_n, int N_q, int N_kv, int causal,
                     int window, int* j_begin, int* j_end, int* lo_masked, int* hi_masked) {
  if (q_tile < 0 || block_m <= 0 || block_n <= 0 || N_q < 0 || N_kv < 0 || window < -1 ||
      !j_begin || !j_end || !lo_masked || !hi_masked)
    return ATTN_ERR_INVALID_ARG;
  kv_tile_span(q_tile, block_m, block_n, N_q, N_kv, causal ? 1 : 0, window, *j_begin, *j_end,
               *lo_masked, *hi_masked);
  return ATTN_OK;
}

size_t attn_bwd_workspace_bytes(int B, int Hq, int N_q) { return bwd_workspace_bytes(B, Hq, N_q); }

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
             const float* lse, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N_q,
             int N_kv, int d, int causal, float scale, attn_dtype_t dtype, void* workspace,
             size_t workspace_bytes, attn_stream_t stream) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || N_q < 0 || N_kv < 0 || Hq % Hkv != 0)
    return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.0f)) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (B == 0 || (N_q == 0 && N_kv == 0)) return ATTN_OK;
  if ((N_q > 0 && (!q || !o || !dout || !lse || !dq)) || (N_kv > 0 && (!k || !v || !dk || !dv)))
    return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv) || !aligned16(workspace) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return ATTN_ERR_MISALIGNED;
  const int dev_ok = check_device(N_q > 0 ? q : k);
  if (dev_ok != ATTN_OK) return dev_ok;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (N_q == 0 || N_kv == 0) {
    // no (query, key) pair: every gradient is zero
    if (N_q > 0 && cudaMemsetAsync(dq, 0, static_cast<size_t>(B) * Hq * N_q * d * 2, st) != cudaSuccess)
      return ATTN_ERR_LAUNCH;
    if (N_kv > 0 &&
        (cudaMemsetAsync(dk, 0, static_cast<size_t>(B) * Hkv * N_kv * d * 2, st) != cudaSuccess ||
         cudaMemsetAsync(dv, 0, static_cast<size_t>(B) * Hkv * N_kv * d * 2, st) != cudaSuccess))
      return ATTN_ERR_LAUNCH;
    return ATTN_OK;
  }
  if (!workspace || workspace_bytes < bwd_workspace_bytes(B, Hq, N_q)) return ATTN_ERR_WORKSPACE;
  BwdArgs a{q, k, v, o, dout, lse, dq, dk, dv, B, Hq, Hkv, N_q, N_kv, d, causal ? 1 : 0, scale,
            dtype == ATTN_BF16, workspace};
  return launch_attn_bwd(a, st);
}

size_t attn_decode_workspace_bytes(int B, int Hq, int max_seqlen_k, int split_size, int d) {
  return decode_workspace_bytes(B, Hq, max_seqlen_k, split_size, d);
}

// The decode kernels index sequences by a grid's second or third dimension (at most 65,535).
constexpr int kMaxDecodeBatch = 65535;

int attn_decode_splitkv(const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* cu_seqlens_k, int kv_capacity, int max_seqlen_k, void* o,
                        float* lse, int B, int Hq, int Hkv, int d, int split_size, float scale,
                        attn_dtype_t dtype, void* workspace, size_t workspace_bytes,
                        attn_stream_t stream) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || kv_capacity < 0 || max_seqlen_k < 0)
    return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.0f)) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (split_size < 64 || split_size > 8192 || split_size % 64 != 0) return ATTN_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (Hq / Hkv > 16) return ATTN_ERR_UNSUPPORTED;
  if (B > kMaxDecodeBatch) return ATTN_ERR_UNSUPPORTED;
  if (B == 0) return ATTN_OK;
  if (!q || !o || !lse || !cu_seqlens_k) return ATTN_ERR_INVALID_ARG;
  if (max_seqlen_k > 0 && kv_capacity > 0 && (!k_cache || !v_cache)) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(o) || !aligned16(k_cache) || !aligned16(v_cache) ||
      !aligned16(workspace) || (reinterpret_cast<uintptr_t>(cu_seqlens_k) & 3u))
    return ATTN_ERR_MISALIGNED;
  const size_t need = decode_workspace_bytes(B, Hq, max_seqlen_k, split_size, d);
  if (!workspace || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
  const int dev_ok = check_device(q);
  if (dev_ok != ATTN_OK) return dev_ok;
  DecodeArgs a{q, k_cache, v_cache, cu_seqlens_k, kv_capacity, max_seqlen_k, o, lse, B,
               Hq, Hkv, d, split_size, scale, dtype == ATTN_BF16, workspace};
  return launch_attn_decode(a, reinterpret_cast<cudaStream_t>(stream));
}

int attn_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                      const int32_t* block_table, const int32_t* seqlens_k, int num_pages,
                      int page_size, int max_pages_per_seq, int max_seqlen_k, void* o, float* lse,
                      int B, int Hq, int Hkv, int d, int split_size, float scale,
                      attn_dtype_t dtype, void* workspace, size_t workspace_bytes,
                      attn_stream_t stream) {
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || num_pages < 0 || max_pages_per_seq < 0 ||
      max_seqlen_k < 0)
    return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.0f)) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (page_size < 16 || page_size > (1 << 16) || (page_size & (page_size - 1)) != 0)
    return ATTN_ERR_UNSUPPORTED;
  if (split_size < 64 || split_size > 8192 || split_size % 64 != 0) return ATTN_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (Hq / Hkv > 16) return ATTN_ERR_UNSUPPORTED;
  if (B > kMaxDecodeBatch) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(num_pages) * page_size > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(max_pages_per_seq) * page_size < max_seqlen_k)
    return ATTN_ERR_INVALID_ARG;
  if (B == 0) return ATTN_OK;
  if (!q || !o || !lse || !block_table || !seqlens_k) return ATTN_ERR_INVALID_ARG;
  if (max_seqlen_k > 0 && (num_pages == 0 || !k_pages || !v_pages)) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(o) || !aligned16(k_pages) || !aligned16(v_pages) ||
      !aligned16(workspace) || (reinterpret_cast<uintptr_t>(block_table) & 3u) ||
      (reinterpret_cast<uintptr_t>(seqlens_k) & 3u))
    return ATTN_ERR_MISALIGNED;
  const size_t need = decode_workspace_bytes(B, Hq, max_seqlen_k, split_size, d);
  if (!workspace || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
  const int dev_ok = check_device(q);
  if (dev_ok != ATTN_OK) return dev_ok;
  DecodeArgs a{q, k_pages, v_pages, nullptr, num_pages * page_size, max_seqlen_k, o, lse, B,
               Hq, Hkv, d, split_size, scale, dtype == ATTN_BF16, workspace};
  a.block_table = block_table;
  a.seqlens = seqlens_k;
  a.page_size = page_size;
  a.max_pages = max_pages_per_seq;
  a.num_pages = num_pages;
  return launch_attn_decode(a, reinterpret_cast<cudaStream_t>(stream));
}

int attn_decode_splitkv_static(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* cu_seqlens_k, int kv_capacity, int max_seqlen_k,
                               void* o, float* lse, int B, int Hq, int Hkv, int d, int split_size,
                               float scale, attn_dtype_t dtype, attn_stream_t stream) {
  // Same checks as attn_decode_splitkv, except that the partial states go to the library's own
  // fixed scratch instead of a caller workspace.  Nothing here allocates.
  if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || kv_capacity < 0 || max_seqlen_k < 0)
    return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.0f)) return ATTN_ERR_INVALID_ARG;
  if (dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_INVALID_ARG;
  if (split_size < 64 || split_size > 8192 || split_size % 64 != 0) return ATTN_ERR_UNSUPPORTED;
  if (d != 64 && d != 128) return ATTN_ERR_UNSUPPORTED;
  if (Hq / Hkv > 16) return ATTN_ERR_UNSUPPORTED;
  if (B > kMaxDecodeBatch) return ATTN_ERR_UNSUPPORTED;
  if (B == 0) return ATTN_OK;
  if (!q || !o || !lse || !cu_seqlens_k) return ATTN_ERR_INVALID_ARG;
  if (max_seqlen_k > 0 && kv_capacity > 0 && (!k_cache || !v_cache)) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(o) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(cu_seqlens_k) & 3u))
    return ATTN_ERR_MISALIGNED;
  const size_t need = decode_workspace_bytes(B, Hq, max_seqlen_k, split_size, d);
  if (need > attn_decode_static_scratch_bytes()) return ATTN_ERR_WORKSPACE;
  const int dev_ok = check_device(q);
  if (dev_ok != ATTN_OK) return dev_ok;
  void* scratch = nullptr;
  size_t scratch_bytes = 0;
  const int st = static_decode_scratch(&scratch, &scratch_bytes);
  if (st != 0) return st;
  if (need > scratch_bytes) return ATTN_ERR_WORKSPACE;
  DecodeArgs a{q, k_cache, v_cache, cu_seqlens_k, kv_capacity, max_seqlen_k, o, lse, B,
               Hq, Hkv, d, split_size, scale, dtype == ATTN_BF16, scratch};
  return launch_attn_decode(a, reinterpret_cast<cudaStream_t>(stream));
}

size_t attn_decode_static_scratch_bytes(void) { return size_t(32) << 20; }

int attn_poll_status(attn_stream_t stream) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_ERR_LAUNCH;
  int* dp = device_status_ptr();
  if (!dp) return ATTN_ERR_LAUNCH;
  int st = 0;
  if (cudaMemcpy(&st, dp, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ERR_LAUNCH;
  if (st != 0) {
    const int zero = 0;
    if (cudaMemcpy(dp, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return ATTN_ERR_LAUNCH;
  }
  return st;
}

const char* attn_status_string(int status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported shape or type";
    case ATTN_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case ATTN_ERR_LAUNCH: return "kernel launch or tensor map failed";
    case ATTN_ERR_TIMEOUT: return "a bounded wait inside a kernel timed out";
    case ATTN_ERR_DEVICE: return "no usable sm_103 device";
    case ATTN_ERR_BAD_LENGTHS: return "a sequence length exceeds max_seqlen_k or kv_capacity";
    default: return "unknown status";
  }
}

int attn_fwd_set_d64_kernel(int mode) {
  const int prev = attn::set_d64_kernel(mode);
  return prev < 0 ? ATTN_ERR_INVALID_ARG : prev;
}

int attn_fwd_kv_tiles(int q_tile, int block_m, int block_n, int N_q, int N_kv, int causal,
                      int* n_tiles, int* first_masked) {
  if (q_tile < 0 || block_m <= 0 || block_n <= 0 || N_q < 0 || N_kv < 0 || !n_tiles ||
      !first_masked)
    return ATTN_ERR_INVALID_ARG;
  int n = 0, fm = 0;
  kv_tile_range(q_tile, block_m, block_n, N_q, N_kv, causal ? 1 : 0, n, fm);
  *n_tiles = n;
  *first_masked = fm;
  return ATTN_OK;
}

int attn_bwd_kv_order(int B, int Hq, int Hkv, int N_q, int N_kv, int causal, int n_sm,
                      uint16_t* job, int cap, int* n) {
  if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || N_q < 0 || N_kv < 0 || n_sm <= 0 || !n ||
      cap < 0 || (cap > 0 && !job))
    return ATTN_ERR_INVALID_ARG;
  const int n_qtiles = (N_q + 127) / 128, n_kvtiles = (N_kv + 127) / 128;
  *n = bwd_kv_order(B * Hkv, n_kvtiles, n_qtiles, Hq / Hkv, causal ? 1 : 0, N_kv - N_q, n_sm, job,
                    cap);
  return ATTN_OK;
}

int attn_selftest_timeout(int limit_us, attn_stream_t stream) {
  if (limit_us < 1 || limit_us > 1000000) return ATTN_ERR_INVALID_ARG;
  const int dev_ok = check_device(nullptr);
  if (dev_ok != ATTN_OK) return dev_ok;
  int* st = device_status_ptr();
  if (!st) return ATTN_ERR_LAUNCH;
  selftest_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      st, static_cast<uint64_t>(limit_us) * 1000ull);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

const char* attn_version(void) { return "attn_gb300 0.1 (sm_103a; tcgen05 prefill, split-KV decode)"; }

}  // extern "C"
