/*
 * attn.h -- C ABI of the GB300 (sm_103a) exact-attention library libattn_gb300.so.
 *
 * The library computes exact scaled dot-product attention
 *
 *     O = softmax(Q K^T * scale + mask) V,     L = rowwise log-sum-exp of (Q K^T * scale + mask)
 *
 * in tiles with an online softmax, so the N x N score and probability matrices never reach
 * device memory ("FlashAttention and GPU Data Movement", sections 2 and 3.1; "How
 * FlashAttention Reduces HBM Traffic Exactly", section "FlashAttention's core move").
 *
 * Conventions shared by every entry point
 *  - Pointers named q, k, v, o, lse, k_cache, v_cache, cu_seqlens_k and workspace are DEVICE
 *    pointers into memory the caller allocated and owns.  The library allocates no device
 *    memory in any call and keeps no pointer after a call returns.
 *  - All work is enqueued on `stream` (a cudaStream_t; NULL = the legacy default stream),
 *    which must belong to the current device, and the buffers must be that device's memory:
 *    a call whose q (or first buffer) lives on another GPU returns ATTN_ERR_INVALID_ARG.
 *    Calls return without synchronising.  Results are valid once the stream reaches them.
 *  - Tensors are contiguous, without strides.  Base pointers must be 16-byte aligned (the
 *    tiles are moved by the Tensor Memory Accelerator).
 *  - Element type: one `attn_dtype_t` applies to q, k, v and o alike.  Scores, the running
 *    max and sum, and the output accumulator are fp32; O is rounded to the element type
 *    (nearest-even); lse is fp32, natural log.
 *  - Errors: argument errors return a negative `attn_status_t` before anything is launched.
 *    A failed launch returns ATTN_ERR_LAUNCH.  Errors found on the device (a bounded wait that
 *    timed out, a sequence length past the promised maximum) are latched in a per-device
 *    status word that `attn_poll_status` returns.  There is no fallback path: an unsupported
 *    shape or type is refused, never computed another way.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st *attn_stream_t; /* same type as cudaStream_t */

typedef enum {
    ATTN_F16 = 0,  /* IEEE binary16 */
    ATTN_BF16 = 1  /* bfloat16 */
} attn_dtype_t;

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = -1, /* null pointer, negative size, Hq % Hkv != 0, bad scale,
                                  q in another GPU's memory than the current device ...   */
    ATTN_ERR_UNSUPPORTED = -2, /* valid request outside what the kernels implement (e.g. d)  */
    ATTN_ERR_MISALIGNED = -3,  /* a base pointer is not 16-byte aligned                       */
    ATTN_ERR_WORKSPACE = -4,   /* workspace missing or smaller than attn_decode_workspace_bytes */
    ATTN_ERR_LAUNCH = -5,      /* the CUDA runtime refused a launch or a tensor map            */
    ATTN_ERR_TIMEOUT = -6,     /* a bounded wait inside a kernel expired (device status word)  */
    ATTN_ERR_DEVICE = -7,      /* no usable sm_103 device, or a device-side argument check     */
    ATTN_ERR_BAD_LENGTHS = -8  /* device-side: a sequence is longer than max_seqlen_k or runs
                                  past kv_capacity (its rows of o and lse are not written)     */
} attn_status_t;

/*
 * attn_fwd -- exact attention forward (prefill), one fused kernel.
 *
 * Defined by: the three-step materialising definition S = Q K^T * scale, P = softmax(S),
 * O = P V ("How FlashAttention Reduces HBM Traffic Exactly", section "The performance problem
 * is data movement"), computed by the FA-2 loop -- one query tile per thread block, K/V tiles
 * streamed through on-chip memory, online softmax with an unnormalised accumulator divided
 * once at the end ("FlashAttention and GPU Data Movement", sections 2 and 3.1) -- with causal
 * tiles past the diagonal skipped and the diagonal tiles masked (same page, section 2.1), and
 * the log-sum-exp exported ("FlashAttention Explained", section "Why the statistics are cheap
 * to store").
 *
 *   q   [B, Hq,  N_q,  d]  element type `dtype`
 *   k   [B, Hkv, N_kv, d]
 *   v   [B, Hkv, N_kv, d]
 *   o   [B, Hq,  N_q,  d]  output, element type `dtype`
 *   lse [B, Hq,  N_q]      output, fp32, L = m + ln(l) in units of the scaled scores;
 *                          -inf for a row that sees no key
 *   Grouped-query attention: query head h reads key/value head h / (Hq / Hkv).
 *   causal != 0: key j is visible to query i iff j <= i + (N_kv - N_q) (bottom-right aligned;
 *   plain "j <= i" when N_q == N_kv).  A row that sees no key gets O = 0 and L = -inf.
 *   scale: multiplies the fp32 dot products (1/sqrt(d) in the usual case); must be finite
 *   and > 0.
 *
 * Supported: d in {64, 128}; dtype F16 or BF16; Hq % Hkv == 0; B, Hq, Hkv >= 1;
 * N_q, N_kv >= 0 (B == 0 or N_q == 0 is a no-op; N_kv == 0 gives O = 0, L = -inf).
 * Returns ATTN_OK or a negative attn_status_t.  Requires one sm_103 GPU (tcgen05 tensor cores).
 */
int attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
             int Hkv, int N_q, int N_kv, int d, int causal, float scale, attn_stream_t stream,
             attn_dtype_t dtype);

/*
 * attn_bwd_workspace_bytes -- bytes of the workspace attn_bwd needs: two fp32 values (L log2 e
 * and D) per query row, rounded up to whole 128-row tiles.  0 for invalid arguments.
 */
size_t attn_bwd_workspace_bytes(int B, int Hq, int N_q);

/*
 * attn_bwd -- gradients of attn_fwd by recomputation ("FlashAttention Explained", section
 * "Backward Pass: Recomputation Beats Storage"): with P = exp(scale Q K^T + mask - L),
 *   dV = P^T dO,  dP = dO V^T,  dS = P o (dP - D) with D_i = rowsum(dO_i o O_i),
 *   dQ = scale dS K,  dK = scale dS^T Q
 * (grouped-query heads: dK, dV of a key/value head sum over its query heads).
 *
 *   q, o, dout   [B, Hq, N_q, d] device, contiguous, 16-bit (`dtype`): the forward's inputs, its
 *                output O and the incoming gradient dO
 *   k, v         [B, Hkv, N_kv, d] device
 *   lse          [B, Hq, N_q] fp32 device: the forward's L (natural log), as attn_fwd returns it
 *   dq           [B, Hq, N_q, d] out;  dk, dv [B, Hkv, N_kv, d] out; 16-bit `dtype`, written in
 *                full (no accumulation into them)
 *   causal, scale, dtype, d (64 or 128)   as the forward call
 *   workspace    device, >= attn_bwd_workspace_bytes(B, Hq, N_q) bytes, caller-owned scratch
 * Deterministic: every output element is written by one thread block, without atomics.
 * Enqueued on `stream`; returns ATTN_OK or a negative attn_status_t.
 */
int attn_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout,
             const float *lse, void *dq, void *dk, void *dv, int B, int Hq, int Hkv, int N_q,
             int N_kv, int d, int causal, float scale, attn_dtype_t dtype, void *workspace,
             size_t workspace_bytes, attn_stream_t stream);

/*
 * attn_fwd_fp8 -- prefill attention on FP8 tensor cores with incoherent processing ("FlashAttention
 * Explained", section "FP8 Attention and Incoherent Processing": Q and K multiplied by the same
 * random orthogonal matrix M -- a Hadamard transform with random sign flips -- before
 * quantisation, so (Q M)(K M)^T = Q K^T while outlier channels spread over all channels;
 * E4M3 operands with per-block scaling factors).  An approximation of attn_fwd: it changes the
 * numerics and needs an accuracy gate, as the pages say.
 *
 * Arguments as attn_fwd (d must be 128), plus
 *   signs      device int8 [d] of +-1, the random sign flips of M (caller-drawn); null: no
 *              rotation (plain block-scaled FP8)
 *   workspace  device, >= attn_fwd_fp8_workspace_bytes(...) bytes, caller-owned; receives the
 *              E4M3 operands and their scales (layout: attn_fwd_fp8_workspace_offsets)
 * Q and K rows are rotated (fp32, fast Walsh-Hadamard butterflies) and quantised with one scale
 * per 128-row tile; V is quantised with one scale per (batch, key/value head) and stored
 * transposed.  Each scale is a power of two, the smallest 2^e with amax <= 448 * 2^e (448: the
 * largest E4M3 value; 1 for an all-zero block), and the codes are E4M3(x * 2^-e), nearest even.
 * P enters the P V product as E4M3.  O is written in `dtype`, L in fp32 as
 * attn_fwd.  Returns ATTN_OK or a negative attn_status_t.
 */
size_t attn_fwd_fp8_workspace_bytes(int B, int Hq, int Hkv, int N_q, int N_kv, int d);

/* attn_fwd_fp8_workspace_offsets -- byte offsets in that workspace of: Q codes [B*Hq, N_q, d],
 * K codes [B*Hkv, N_kv, d], V^T codes [B*Hkv, d, nkvp] (nkvp = N_kv rounded up to 128), Q scales
 * [B*Hq, ceil(N_q/128)], K scales [B*Hkv, ceil(N_kv/128)], V scales [B*Hkv] (fp32), scratch. */
int attn_fwd_fp8_workspace_offsets(int B, int Hq, int Hkv, int N_q, int N_kv, int d,
                                   size_t *offsets /* [7] */);

int attn_fwd_fp8(const void *q, const void *k, const void *v, void *o, float *lse, int B, int Hq,
                 int Hkv, int N_q, int N_kv, int d, int causal, float scale, const int8_t *signs,
                 void *workspace, size_t workspace_bytes, attn_stream_t stream,
                 attn_dtype_t dtype);

/*
 * attn_fwd_window -- prefill attention with a sliding window, the mask that changes the
 * operator ("FlashAttention Explained", FlexAttention section, sliding_causal: key kv is visible
 * to query q iff q >= kv and q - kv <= W; "FlashAttention, annotated", section on causal masks
 * and windows: key tiles outside the window are skipped, not masked).
 *
 * Arguments as attn_fwd, with `causal` replaced by
 *   window   W >= 0: key j is visible to query row i iff 0 <= (i + N_kv - N_q) - j <= W
 *            (bottom-right aligned as attn_fwd's causal mask, which W >= N_kv reproduces).
 * Only the key tiles a query tile can see are loaded; the tiles cut by the window's lower edge
 * or the diagonal are masked element by element.  A row with no visible key gets O = 0,
 * L = -inf.  Returns ATTN_OK, ATTN_ERR_INVALID_ARG (W < 0) or another attn_status_t.
 */
int attn_fwd_window(const void *q, const void *k, const void *v, void *o, float *lse, int B,
                    int Hq, int Hkv, int N_q, int N_kv, int d, int window, float scale,
                    attn_stream_t stream, attn_dtype_t dtype);

/*
 * attn_fwd_block_sparse -- prefill attention restricted to a pattern of (query tile, key
 * tile) blocks ("FlashAttention, annotated", section 3.3, block-sparse FlashAttention: a fixed
 * pattern of tiles to compute and skip; the BlockMask of "FlashAttention Explained", one
 * pattern shared by every batch and head).
 *
 * Arguments as attn_fwd, plus
 *   block_mask  device pointer, uint8 [ceil(N_q / 128)][ceil(N_kv / 128)], row-major: nonzero
 *               = compute query tile r (rows 128 r .. 128 r + 127) against key tile c (keys
 *               128 c .. 128 c + 127).  Read-only; owned by the caller; read while the call
 *               runs on `stream`.
 * Keys outside listed blocks are invisible; inside a listed block the causal rule (if
 * `causal`) still applies.  Unlisted blocks are neither loaded nor computed.  A row with no
 * visible key gets O = 0, L = -inf.  Returns ATTN_OK, ATTN_ERR_INVALID_ARG (null pattern) or
 * another attn_status_t.
 */
int attn_fwd_block_sparse(const void *q, const void *k, const void *v, void *o, float *lse,
                          int B, int Hq, int Hkv, int N_q, int N_kv, int d, int causal,
                          const uint8_t *block_mask, float scale, attn_stream_t stream,
                          attn_dtype_t dtype);

/*
 * attn_decode_workspace_bytes -- device workspace attn_decode_splitkv needs.
 *
 * The split-KV decode writes one partial state (m, l, o[d]) per (sequence, query head,
 * split) before merging them; this returns the bytes for B sequences of at most
 * max_seqlen_k tokens cut into split_size-token splits.  Returns 0 for invalid arguments.
 */
size_t attn_decode_workspace_bytes(int B, int Hq, int max_seqlen_k, int split_size, int d);

/*
 * attn_decode_splitkv -- one decode step: one new query token per sequence against its
 * whole KV cache, split along the keys and merged exactly.
 *
 * Defined by: the same attention definition with a 1 x n score row ("FlashAttention and Why
 * Attention Is a Memory-Traffic Problem", section "Prefill versus decode"); the key/value
 * sequence is split into split_size-token chunks, each chunk produces a partial state
 * (m, l, o) with the online softmax, and the partial states are merged with the block-merge
 * rule m = max(m1, m2), l = e^(m1-m) l1 + e^(m2-m) l2, o = (e^(m1-m) l1 o1 + e^(m2-m) l2 o2)/l
 * ("How FlashAttention Reduces HBM Traffic Exactly", section "Why softmax does not prevent
 * tiling"; "FlashAttention Explained", section "Decoding, Paged and Split-KV Variants";
 * "FlashAttention and GPU Data Movement", section 6.1).
 *
 *   q            [B, Hq, d]                  element type `dtype`
 *   k_cache      [kv_capacity, Hkv, d]       packed (varlen) cache: sequence b owns token rows
 *   v_cache      [kv_capacity, Hkv, d]       cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1
 *   cu_seqlens_k [B + 1] int32, DEVICE, non-decreasing, cu_seqlens_k[0] = 0 is not required
 *   kv_capacity  token rows allocated in each cache
 *   max_seqlen_k upper bound on every sequence length (sizes the grid and the workspace);
 *                a longer sequence is reported as ATTN_ERR_BAD_LENGTHS by attn_poll_status
 *   o            [B, Hq, d] output, element type `dtype`
 *   lse          [B, Hq] output fp32 (natural log, scaled scores); -inf for an empty sequence
 *   split_size   tokens per split: a multiple of 64 in [64, 8192] (512 in the usual case)
 *   workspace    device scratch of at least attn_decode_workspace_bytes(B, Hq, max_seqlen_k,
 *                split_size, d) bytes, 16-byte aligned; its contents need no initialisation
 *   Query head h reads key/value head h / (Hq / Hkv); Hq / Hkv must be <= 16.
 *
 * Supported: d in {64, 128}; dtype F16 or BF16; B <= 65535 (the kernels index sequences by a
 * grid dimension of that size; a larger batch returns ATTN_ERR_UNSUPPORTED before any launch:
 * split it into several calls).  Returns ATTN_OK or a negative attn_status_t.
 * Calls that share a workspace must not overlap on the device.
 */
int attn_decode_splitkv(const void *q, const void *k_cache, const void *v_cache,
                        const int32_t *cu_seqlens_k, int kv_capacity, int max_seqlen_k,
                        void *o, float *lse, int B, int Hq, int Hkv, int d, int split_size,
                        float scale, attn_dtype_t dtype, void *workspace,
                        size_t workspace_bytes, attn_stream_t stream);

/*
 * attn_decode_splitkv_static -- attn_decode_splitkv for callers that cannot allocate.
 *
 * No counterpart on the pages: this is a library convenience.  Some callers cannot obtain
 * device memory at the point where they decode -- a serving loop that may not call cudaMalloc
 * inside its step (the call can synchronise the whole device), a process whose device memory
 * belongs to another allocator it has no handle to, or an embedding that lends the library only
 * its input and output buffers.  This
 * entry point takes the same inputs and outputs as attn_decode_splitkv (see there) but no
 * workspace: the partial states go to a fixed scratch array inside the library (a file-scope
 * __device__ array of the decode module), which the CUDA runtime places on a GPU when it loads
 * that module there and keeps until the process exits.  With the runtime's default lazy module
 * loading that happens at the first decode call of either kind on the device (this entry point
 * or attn_decode_splitkv / attn_decode_paged, which share the module), so every process that
 * decodes on a GPU holds the 32 MiB there.  No call allocates anything else.
 *
 *  - Limit: attn_decode_workspace_bytes(B, Hq, max_seqlen_k, split_size, d) must not exceed
 *    attn_decode_static_scratch_bytes() (32 MiB, e.g. 15 sequences x 64 heads x 32k tokens at
 *    512-token splits, d = 128); larger requests return ATTN_ERR_WORKSPACE before any launch.
 *  - The first call on each device looks up that device's copy of the scratch array (with the
 *    device current), which may load the decode module and commit its memory; make that first
 *    call before any stream capture.
 *  - Every call shares the one array and it keeps the last call's contents.  Nothing in it
 *    needs to start at zero, but two calls that overlap on the GPU (different streams without
 *    ordering, or two threads) race on it: order them.
 * Returns ATTN_OK or a negative attn_status_t.
 */
int attn_decode_splitkv_static(const void *q, const void *k_cache, const void *v_cache,
                               const int32_t *cu_seqlens_k, int kv_capacity, int max_seqlen_k,
                               void *o, float *lse, int B, int Hq, int Hkv, int d,
                               int split_size, float scale, attn_dtype_t dtype,
                               attn_stream_t stream);

/*
 * attn_decode_paged -- the split-KV decode step over a paged KV cache ("FlashAttention
 * Explained", section "Decoding, Paged and Split-KV Variants": PagedAttention stores the cache
 * in fixed-size non-contiguous blocks addressed through a block table; production engines run
 * split-KV decoding over it).
 *
 *   q             [B, Hq, d] device, contiguous, the new token of every sequence
 *   k_pages,
 *   v_pages       [num_pages, page_size, Hkv, d] device, contiguous: the page pool
 *   block_table   [B, max_pages_per_seq] int32 device: sequence b's token t is row
 *                 t % page_size of page block_table[b * max_pages_per_seq + t / page_size];
 *                 entries past the sequence's last page are not read
 *   seqlens_k     [B] int32 device: cached tokens of each sequence (0 allowed: O = 0, L = -inf)
 *   num_pages     pages in the pool; page_size a power of two from 16 to 65536
 *   max_seqlen_k  upper bound of seqlens_k (<= max_pages_per_seq * page_size), sizes the grid
 *   o, lse, B, Hq, Hkv, d, split_size, scale, dtype, workspace, workspace_bytes, stream
 *                 as attn_decode_splitkv (the workspace size is attn_decode_workspace_bytes;
 *                 B <= 65535)
 * The result equals attn_decode_splitkv on the gathered packed cache.  A length above
 * max_seqlen_k or a block-table entry outside [0, num_pages) is reported as
 * ATTN_ERR_BAD_LENGTHS by attn_poll_status (that sequence's output is then undefined).
 * Returns ATTN_OK or a negative attn_status_t.
 */
int attn_decode_paged(const void *q, const void *k_pages, const void *v_pages,
                      const int32_t *block_table, const int32_t *seqlens_k, int num_pages,
                      int page_size, int max_pages_per_seq, int max_seqlen_k, void *o, float *lse,
                      int B, int Hq, int Hkv, int d, int split_size, float scale,
                      attn_dtype_t dtype, void *workspace, size_t workspace_bytes,
                      attn_stream_t stream);

/* attn_decode_static_scratch_bytes -- size of the scratch attn_decode_splitkv_static uses. */
size_t attn_decode_static_scratch_bytes(void);

/*
 * attn_poll_status -- synchronise `stream`, then read and clear the status word of the
 * current device.  Returns ATTN_OK, the first device-side error latched since the last poll
 * (ATTN_ERR_TIMEOUT, ATTN_ERR_BAD_LENGTHS), or ATTN_ERR_LAUNCH if the synchronisation failed.
 */
int attn_poll_status(attn_stream_t stream);

/* attn_status_string -- static text for a status code. */
const char *attn_status_string(int status);

/*
 * attn_fwd_kv_tiles -- host-side copy of the tile range the prefill kernel walks for one
 * query tile (the causal skip bound and the first tile needing the element mask, "FlashAttention
 * and GPU Data Movement", section 2.1), exposed so the schedule can be checked without a GPU.
 *
 *   q_tile   0-based query tile (rows q_tile*block_m .. q_tile*block_m + block_m - 1)
 *   block_m, block_n   query rows per tile, keys per K/V tile (the kernel uses 128, 128)
 *   *n_tiles       number of K/V tiles loaded (tiles 0 .. n_tiles-1)
 *   *first_masked  first K/V tile that needs the element mask (causal diagonal or the ragged
 *                  end of the keys); == *n_tiles when none does
 * Returns ATTN_OK or ATTN_ERR_INVALID_ARG.
 */
int attn_fwd_kv_tiles(int q_tile, int block_m, int block_n, int N_q, int N_kv, int causal,
                      int *n_tiles, int *first_masked);

/*
 * attn_fwd_kv_span -- host-side copy of the key-tile span the prefill kernel walks for one
 * query tile under a sliding window (window >= 0, which implies the causal bound) or none
 * (window == -1): tiles *j_begin .. *j_end - 1 are loaded; tiles below *lo_masked need the
 * window's lower-edge mask, tiles from *hi_masked on the diagonal or ragged-end mask.
 * Returns ATTN_OK or ATTN_ERR_INVALID_ARG.
 */
int attn_fwd_kv_span(int q_tile, int block_m, int block_n, int N_q, int N_kv, int causal,
                     int window, int *j_begin, int *j_end, int *lo_masked, int *hi_masked);

/*
 * attn_bwd_kv_order -- host-side copy of the order in which attn_bwd launches the blocks of its
 * dK/dV kernel (one block per 128-key tile of each (batch, key/value head)), exposed so the
 * schedule can be checked without a GPU.  Under the causal mask a block's work grows with the
 * query tiles that see its key tile; the blocks are packed into one bin per SM (largest first,
 * each into the fullest bin that stays under the average load) and listed in the order in which
 * SMs that free up in turn would take them.  Jobs are numbered key tile major:
 * job = key_tile * (B * Hkv) + b * Hkv + h.
 *
 *   n_sm   SMs the grid runs on
 *   job    [cap] out: the job of launch block i, i < *n
 *   *n     entries written; 0 when the launch keeps the default order (job = block index: no
 *          causal mask, no more blocks than SMs, or more than `cap` blocks; attn_bwd itself
 *          uses cap = 2048)
 * Returns ATTN_OK or ATTN_ERR_INVALID_ARG.
 */
int attn_bwd_kv_order(int B, int Hq, int Hkv, int N_q, int N_kv, int causal, int n_sm,
                      uint16_t *job, int cap, int *n);

/*
 * attn_fwd_set_d64_kernel -- choose the prefill kernel for head dimension 64 (every later call
 * of attn_fwd, attn_fwd_window and attn_fwd_block_sparse in this process, on every device):
 *   ATTN_D64_AUTO (0, the default): two query tiles per work item, which share each K/V tile
 *     ("FlashAttention Explained", section on FlashAttention-4: two query tiles per thread
 *     block), when the call has more 128-row query tiles (B * Hq * ceil(N_q / 128)) than the
 *     device has SMs; else one query tile per item, which spreads a small call over more SMs;
 *   ATTN_D64_PAIR (1), ATTN_D64_SINGLE (2): always that kernel.
 * Both compute the same operator within the same rounding.  Returns the previous mode, or
 * ATTN_ERR_INVALID_ARG for any other value (the mode is then unchanged).  Thread-safe.
 */
enum { ATTN_D64_AUTO = 0, ATTN_D64_PAIR = 1, ATTN_D64_SINGLE = 2 };
int attn_fwd_set_d64_kernel(int mode);

/*
 * attn_selftest_timeout -- launch one tiny kernel that waits on a barrier nothing ever
 * arrives at, with a limit of `limit_us` microseconds (1 .. 1000000), then records
 * ATTN_ERR_TIMEOUT in the status word and returns.  Used to check, on a GPU, that a wait which
 * runs out leaves the context usable and reports through attn_poll_status.
 */
int attn_selftest_timeout(int limit_us, attn_stream_t stream);

/* attn_version -- library version string. */
const char *attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
