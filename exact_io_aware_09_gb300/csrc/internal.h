// Host-side declarations shared by the translation units of libattn_gb300.so.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace attn {

// Encode a 3-D tiled TMA descriptor over a contiguous 16-bit tensor with dimensions
// {dim0 (innermost, elements), dim1, dim2}, byte strides {stride1, stride2}, a box of
// {box0, box1, box2} elements and the 128-byte swizzle.  Returns false on failure.
bool make_tmap_3d(CUtensorMap* map, const void* base, bool bf16, uint64_t dim0, uint64_t dim1,
                  uint64_t dim2, uint64_t stride1, uint64_t stride2, uint32_t box0,
                  uint32_t box1, uint32_t box2);

// A 4-D tiled TMA descriptor over a 16-bit tensor: dims {dim0 (innermost, elements), dim1,
// dim2, dim3}, byte strides of dims 1-3 (in any order of size), box {box0 .. box3}, 128-byte
// swizzle.  Returns false on failure.
bool make_tmap_4d(CUtensorMap* map, const void* base, bool bf16, const uint64_t dims[4],
                  const uint64_t strides[3], const uint32_t box[4]);

// The same over a contiguous 8-bit tensor (E4M3 codes).
bool make_tmap_3d_u8(CUtensorMap* map, const void* base, uint64_t dim0, uint64_t dim1,
                     uint64_t dim2, uint64_t stride1, uint64_t stride2, uint32_t box0,
                     uint32_t box1, uint32_t box2);

// Device address of the status word of the current device (nullptr on failure).
int* device_status_ptr();

// Query tile range of the prefill schedule (also exported through the C ABI).
__host__ __device__ inline void kv_tile_range(int qt, int bm, int bn, int n_q, int n_kv,
                                              int causal, int& n_tiles, int& first_masked) {
  const long long n_all = (static_cast<long long>(n_kv) + bn - 1) / bn;
  const long long ragged_last = (n_kv % bn) ? n_all - 1 : n_all;
  if (!causal) {
    n_tiles = static_cast<int>(n_all);
    first_masked = static_cast<int>(ragged_last);
    return;
  }
  const long long off = static_cast<long long>(n_kv) - n_q;
  const long long r_first = static_cast<long long>(qt) * bm;
  long long r_last = static_cast<long long>(qt + 1) * bm;
  if (r_last > n_q) r_last = n_q;
  r_last -= 1;
  const long long kmax = r_last + off;  // last key the last row of the tile may see
  if (kmax < 0 || n_all == 0) {
    n_tiles = 0;
    first_masked = 0;
    return;
  }
  long long n = kmax / bn + 1;
  if (n > n_all) n = n_all;
  const long long kmin = r_first + off;  // last key the first row of the tile may see
  long long fm = (kmin + 1 >= 0) ? (kmin + 1) / bn : 0;  // tiles every row sees in full
  if (fm > ragged_last) fm = ragged_last;
  if (fm > n) fm = n;
  n_tiles = static_cast<int>(n);
  first_masked = static_cast<int>(fm);
}

// Key-tile span of query tile qt (tiles of bm rows and bn keys) under the causal bound and an
// optional sliding window of `window` keys behind the diagonal (window < 0: none; a window
// implies the causal bound): the tiles [j_begin, j_end) hold every visible key; tiles below
// lo_masked need the window's lower-edge mask and tiles from hi_masked on the upper
// (causal or ragged-edge) mask.  An empty span has j_begin == j_end.
__host__ __device__ inline void kv_tile_span(int qt, int bm, int bn, int n_q, int n_kv,
                                             int causal, int window, int& j_begin, int& j_end,
                                             int& lo_masked, int& hi_masked) {
  int n = 0, fm = 0;
  kv_tile_range(qt, bm, bn, n_q, n_kv, (causal || window >= 0) ? 1 : 0, n, fm);
  j_begin = 0;
  j_end = n;
  lo_masked = 0;
  hi_masked = fm;
  if (window < 0 || n == 0) return;
  const long long off = static_cast<long long>(n_kv) - n_q;
  const long long r_first = static_cast<long long>(qt) * bm;
  long long r_last = static_cast<long long>(qt + 1) * bm;
  if (r_last > n_q) r_last = n_q;
  r_last -= 1;
  const long long lo_first = r_first + off - window;  // lowest key the first row sees
  const long long lo_last = r_last + off - window;    // lowest key the last row sees
  long long jb = lo_first > 0 ? lo_first / bn : 0;
  long long lm = lo_last > 0 ? (lo_last + bn - 1) / bn : 0;  // tiles below see a cut
  if (jb > n) jb = n;
  if (lm < jb) lm = jb;
  if (lm > n) lm = n;
  j_begin = static_cast<int>(jb);
  lo_masked = static_cast<int>(lm);
  if (hi_masked < j_begin) hi_masked = j_begin;
}

struct FwdArgs {
  const void* q;
  const void* k;
  const void* v;
  void* o;
  float* lse;
  int B, Hq, Hkv, N_q, N_kv, d, causal;
  float scale;
  bool bf16;
  int window;                 // sliding window (keys behind the diagonal); -1 = none
  const uint8_t* block_mask;  // [ceil(N_q/128)][ceil(N_kv/128)] tiles to compute; null = all
  // FP8 operands (set by the FP8 entry point after its preparation): E4M3 codes of the rotated
  // Q [B*Hq, N_q, d] and K [B*Hkv, N_kv, d], of V transposed [B*Hkv, d, nkvp], and their scales
  const void* q8 = nullptr;
  const void* k8 = nullptr;
  const void* vt8 = nullptr;
  const float* q_scale = nullptr;
  const float* k_scale = nullptr;
  const float* v_scale = nullptr;
  int nkvp = 0;
};

struct DecodeArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* cu_seqlens;
  int kv_capacity, max_seqlen;
  void* o;
  float* lse;
  int B, Hq, Hkv, d, split;
  float scale;
  bool bf16;
  void* workspace;
  // paged cache (block_table != null): k_cache/v_cache are [num_pages, page_size, Hkv, d],
  // sequence b's token t is row t % page_size of page block_table[b * max_pages + t / page_size],
  // and seqlens[b] replaces cu_seqlens
  const int32_t* block_table = nullptr;
  const int32_t* seqlens = nullptr;
  int page_size = 0, max_pages = 0, num_pages = 0;
};

struct BwdArgs {
  const void* q;
  const void* k;
  const void* v;
  const void* o;
  const void* dout;
  const float* lse;
  void* dq;
  void* dk;
  void* dv;
  int B, Hq, Hkv, N_q, N_kv, d, causal;
  float scale;
  bool bf16;
  void* workspace;
};

// Launchers (return an attn_status_t value).
int launch_attn_fwd(const FwdArgs& a, cudaStream_t stream);
// d = 64: two query tiles per work item (attn_fwd_pair.cu)
int launch_attn_fwd_pair(const FwdArgs& a, cudaStream_t stream);
// The d = 64 kernel choice: 0 automatic, 1 two query tiles per item, 2 one (attn_fwd.cu).
int set_d64_kernel(int mode);
int launch_attn_fwd_fp8_kernel(const FwdArgs& a, cudaStream_t stream);
// FP8 forward: prepares the rotated, quantised operands in `workspace` (layout from
// fp8_workspace_layout: Q8, K8, V^T8, Q scales, K scales, V scales, V amax) and runs the kernel.
int launch_attn_fwd_fp8(const FwdArgs& a, const int8_t* signs, void* workspace,
                        cudaStream_t stream);
size_t fp8_workspace_layout(int B, int Hq, int Hkv, int N_q, int N_kv, int d, size_t off[7]);
int launch_attn_decode(const DecodeArgs& a, cudaStream_t stream);
int launch_attn_bwd(const BwdArgs& a, cudaStream_t stream);
size_t bwd_workspace_bytes(int B, int Hq, int N_q);
size_t decode_workspace_bytes(int B, int Hq, int max_seqlen, int split, int d);
// Device address and size of the library-owned decode scratch of the current device
// (set up on the first call per device).  Returns 0 or an attn_status_t value.
int static_decode_scratch(void** ptr, size_t* bytes);

}  // namespace attn
