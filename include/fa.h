/*
 * fa.h -- C ABI of the exact IO-aware attention library for GB300 (sm_103a).
 *
 * What the library computes (one head = one (b, h) pair, all heads at once):
 *
 *   S   = scale * Q K^T                          (N x N, never stored)
 *   P   = softmax_row(S) over the allowed keys   (never stored)
 *   O   = P V
 *   LSE = per-row natural log-sum-exp of the allowed scaled scores
 *
 * Source: page "FlashAttention" (aiwiki), section "Attention and the memory
 * bottleneck" (the scaled dot-product formula and its masks), section
 * "Tiling and online normalization" (the running max / running sum /
 * rescaled accumulator recurrence the forward kernel evaluates tile by
 * tile), and page "FlashAttention IO-aware explained", section
 * "Recomputation and IO complexity" (the backward pass rebuilds score tiles
 * from stored row statistics instead of storing P).  Block-sparse skipping:
 * page "Fast and Memory Efficient Exact Attention", "Summary & Methodology
 * Analysis" (zero blocks of a predefined block-sparsity mask are skipped).
 *
 * Which (query i, key j) pairs are allowed, for batch element b:
 *     (!causal || j <= i)
 *  && (block_mask == NULL || block_mask[(i/128)*T + j/128] != 0)
 *  && (kv_len == NULL     || j < kv_len[b])              (kv_len clamped to [0, N])
 *  && (window_left  < 0   || j >= i - window_left)       (fa_mask calls only)
 *  && (window_right < 0   || j <= i + window_right)      (fa_mask calls only)
 * with T = ceil(N/128).  A query row with no allowed key gets O = 0 and
 * LSE = -inf, and contributes nothing to the gradients.  The sliding window
 * follows page "FlashAttention" (aiwiki), section "Software integration and
 * limitations", which lists causal and sliding-window masks among the
 * method's interfaces; (w, 0) with causal is the usual causal window of the
 * last w+1 keys.
 *
 * Common conventions
 *  - Tensors are dense, row-major, on the current CUDA device:
 *      Q, K, V, O, dO, dQ, dK, dV : bf16 [B, H, N, d], d in {64, 128},
 *                                   base pointers 16-byte aligned;
 *      LSE, D                     : fp32 [B, H, N];
 *      block_mask                 : uint8 [T, T] (shared by every (b, h)) or NULL;
 *      kv_len                     : int32 [B] or NULL.
 *  - Every pointer is a DEVICE pointer unless stated otherwise.  The caller
 *    owns every buffer; the library allocates no device memory on these
 *    calls and keeps no pointer after a call returns.
 *  - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream) and never synchronises, except fa_last_device_status.
 *  - Errors are status codes; the library never aborts.  Arguments are
 *    validated on the host before anything is launched; on an invalid
 *    argument nothing is launched and no output is written.
 *  - Outputs are written in bf16 (round to nearest even) except LSE and D.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size, overflow   */
  FA_ERR_UNSUPPORTED = 2, /* head dimension other than 64 or 128          */
  FA_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed          */
  FA_ERR_TIMEOUT = 4      /* a bounded in-kernel wait gave up (see below)  */
} fa_status;

/* Human-readable name of a status code (static storage, never NULL). */
FA_API const char* fa_status_string(int status);

/*
 * Every mask option in one place (the fa_*_masked calls take a pointer to
 * it; NULL = no mask).  Fields as in the allowed-pair rule above:
 *   causal        nonzero = j <= i
 *   window_left   >= 0: j >= i - window_left;  < 0: unbounded
 *   window_right  >= 0: j <= i + window_right; < 0: unbounded
 *   block_mask    uint8 [T, T] device or NULL (zero tiles are skipped)
 *   kv_len        int32 [B] device or NULL
 *   dropout_p     probability of dropping each element of P, in [0, 1),
 *                 used in steps of 1/256 (p8 = round(256 p), at most 255);
 *                 0 = no dropout.  O = ((P o Z) / (1 - p8/256)) V with Z the
 *                 keep mask; LSE is that of P (unaffected).
 *   dropout_seed, dropout_offset
 *                 the generator state: Z(b, h, i, j) = [u >= p8] with u byte
 *                 j % 16 of Philox4x32-10(counter (j/16, i, b*H + h,
 *                 dropout_offset), key (seed mod 2^32, seed >> 32)), i, j
 *                 positions within the head (within the sequence when
 *                 packed).  The backward regenerates Z from the same state,
 *                 so pass the forward's values (page "FlashAttention: Fast
 *                 and Memory-Efficient Exact Attention with IO-Awareness",
 *                 claims on the backward pass: the mask is not stored).
 * A window side of N or more is the same as unbounded.  Dropout is not
 * offered by the plain (non-_masked) calls.
 */
typedef struct fa_mask {
  int causal;
  int window_left;
  int window_right;
  const uint8_t* block_mask;
  const int32_t* kv_len;
  float dropout_p;
  uint64_t dropout_seed;
  uint32_t dropout_offset;
} fa_mask;

/*
 * Forward pass: O and LSE.
 *   q, k, v    : bf16 [B,H,N,d], read only.
 *   o          : bf16 [B,H,N,d], written.
 *   lse        : fp32 [B,H,N], written (natural log; -inf on fully masked rows).
 *   scale      : multiplies Q K^T (usually 1/sqrt(d)); any finite value, of
 *                either sign (0 gives uniform weights over the allowed keys).
 *   causal     : nonzero = causal mask j <= i.
 *   block_mask : see above; its zero tiles are never loaded or computed.
 *   kv_len     : see above.
 * Requires B, H, N >= 1, B*H <= 2^31-1, B*H*N*d < 2^62, d in {64,128}.
 */
FA_API int fa_forward(const void* q, const void* k, const void* v, void* o, float* lse,
               int B, int H, int N, int d, float scale, int causal,
               const uint8_t* block_mask, const int32_t* kv_len, void* stream);

/* fa_forward with the full mask description (sliding windows included). */
FA_API int fa_forward_masked(const void* q, const void* k, const void* v, void* o, float* lse,
                             int B, int H, int N, int d, float scale, const fa_mask* mask,
                             void* stream);

/*
 * Bytes of device workspace fa_backward needs: LSE*log2(e) and D
 * (fp32 [B*H][Np] each, Np = N rounded up to a multiple of 128) followed by
 * the fp32 dQ accumulator [B,H,N,d] and 256 bytes for the dK/dV kernel's
 * work-item counter, each part 256-byte aligned.
 * O(B*H*N*d): linear in N (no N x N buffer).  Returns 0 for invalid sizes.
 */
FA_API size_t fa_backward_workspace_bytes(int B, int H, int N, int d);

/*
 * Workspace for a backward call with `mask` (NULL = no mask).  With a block
 * mask (and N <= 131,072, B*H*ceil(N/128)*4 < 2^31) this adds room for
 * spreading the work of a key tile over up to 4 CTAs: a key tile with many
 * live query tiles (a global column, say) otherwise walks all of them in one
 * CTA while the GPU idles.  The extra part holds a work plan
 * (16 * 4 * ceil(N/128) bytes plus 256) and 32 fp32 slots of 2 x 128 x d
 * values per head (1 KiB x d each), about B*H*d*32 KiB in all.  Given a
 * workspace of at least this size, fa_backward_masked / fa_backward /
 * fa_backward_dkdv launch a small planning kernel before the dK/dV kernel
 * and split heavy key tiles (each part of a split key tile stores its fp32
 * dK, dV rows in its slot, and a join kernel after the dK/dV kernel adds
 * them in part order and writes the bf16 rows); with only
 * fa_backward_workspace_bytes() they do not split.  Results agree up to the
 * order of fp32 additions.  Returns 0 for invalid sizes.
 */
FA_API size_t fa_backward_workspace_bytes_masked(int B, int H, int N, int d,
                                                 const fa_mask* mask);

/*
 * Backward pass: dQ, dK, dV of L = sum(O * dO), recomputing P tile by tile
 * from Q, K and the forward's LSE (P is never stored).
 *   q, k, v, o : forward inputs and output, bf16 [B,H,N,d].
 *   lse        : forward's LSE, fp32 [B,H,N].
 *   dout       : dO, bf16 [B,H,N,d].
 *   dq, dk, dv : bf16 [B,H,N,d], written.
 *   workspace  : device buffer of at least fa_backward_workspace_bytes(),
 *                256-byte aligned, owned by the caller; its contents on
 *                entry are ignored and on exit are unspecified.
 *   Other arguments as in fa_forward and equal to the forward call's.
 *   dq, dk, dv and the workspace must not overlap each other or any input.
 * Launches, in order on `stream`: the D = rowsum(dO * O) preprocess (which
 * also clears the dQ accumulator), the dK/dV kernel (which also adds each
 * tile's dS K into the dQ accumulator), and the dQ conversion; with a split
 * (below), its plan kernel first.  Each kernel after the first is launched
 * with programmatic dependent launch: it may start, and do the set-up that
 * needs no result of the kernel before it, while that kernel finishes; it
 * waits for that kernel's results before it reads them.  No kernel starts
 * before all work enqueued ahead of the call has completed.
 */
FA_API int fa_backward(const void* q, const void* k, const void* v, const void* o,
                const float* lse, const void* dout, void* dq, void* dk, void* dv,
                int B, int H, int N, int d, float scale, int causal,
                const uint8_t* block_mask, const int32_t* kv_len,
                void* workspace, size_t workspace_bytes, void* stream);

/* fa_backward with the full mask description; the mask must be the one the
 * forward was called with. */
FA_API int fa_backward_masked(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dout, void* dq, void* dk, void* dv,
                              int B, int H, int N, int d, float scale, const fa_mask* mask,
                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * The three launches of fa_backward, exposed one by one so a caller can
 * time or overlap them; calling them in this order on one stream with the
 * same workspace computes exactly what fa_backward computes (fa_backward
 * also starts the dK/dV kernel's set-up during the preprocess's tail, which
 * the separate calls do not).  Arguments mean what they mean in
 * fa_backward; each validates its own arguments and none reads memory that
 * work enqueued ahead of it may still be writing.
 *
 * fa_backward_preprocess: D = rowsum(dO * O) and LSE*log2(e) into the
 *   workspace (padding rows and rows without an allowed key get +inf, so
 *   their probabilities rebuild as 0) and clears the workspace's fp32 dQ
 *   accumulator [B,H,N,d].
 * fa_backward_dkdv: for every live 128-key tile, recomputes P and dS from
 *   Q, K, V, dO and the workspace's LSE and D, writes dK (times scale) and
 *   dV, and adds dS K into the workspace's dQ accumulator.  Needs its own
 *   preprocess call first (which also resets the work counter it takes its
 *   key tiles from at d = 64).  With a block mask and a workspace of
 *   fa_backward_workspace_bytes_masked() it is three launches (the split
 *   plan, the kernel, the join of the split key tiles).
 * fa_backward_dq_convert: dQ = scale * accumulator, rounded to bf16.
 */
FA_API int fa_backward_preprocess(const void* o, const void* dout, const float* lse, int B,
                                  int H, int N, int d, void* workspace,
                                  size_t workspace_bytes, void* stream);
FA_API int fa_backward_dkdv(const void* q, const void* k, const void* v, const void* dout,
                            void* dk, void* dv, int B, int H, int N, int d, float scale,
                            int causal, const uint8_t* block_mask, const int32_t* kv_len,
                            void* workspace, size_t workspace_bytes, void* stream);
FA_API int fa_backward_dq_convert(void* dq, int B, int H, int N, int d, float scale,
                                  const void* workspace, size_t workspace_bytes,
                                  void* stream);

/*
 * Backward pass for callers that cannot allocate device memory.  (No
 * counterpart in the method's description: an interface convenience.)
 *
 * Who needs it: code embedded in a host framework that owns every device
 * allocation (its own pool or memory budget) and forbids raw cudaMalloc from
 * plug-ins, and latency-critical callers that must keep cudaMalloc/cudaFree
 * (which can synchronise the whole device) off their hot path -- callers
 * that therefore cannot hand fa_backward a workspace.
 *
 * Same arguments and results as fa_backward, minus the workspace: the
 * library uses a fixed array of FA_NOALLOC_SCRATCH_BYTES of device memory
 * that is part of the library image, reserved on every GPU that loads the
 * library and held until the process exits.  Nothing is allocated.
 *  - Problems whose fa_backward_workspace_bytes() exceeds
 *    FA_NOALLOC_SCRATCH_BYTES are rejected with FA_ERR_INVALID_ARG before
 *    any CUDA call.  That size is 2 * r(4*B*H*Np) + r(4*B*H*N*d) + 256 bytes,
 *    with Np = N rounded up to a multiple of 128 and r() rounding up to a
 *    multiple of 256; call fa_backward_workspace_bytes() to test a shape
 *    (e.g. B*H = 16, N = 8192, d = 64 needs 33.0 MiB and is rejected; at
 *    N = 7680 it needs 30.9 MiB and fits).
 *  - With a block mask the spare room of the array beyond that size, when
 *    there is enough of it, lets the backward split heavy key tiles over
 *    several CTAs exactly as fa_backward does given
 *    fa_backward_workspace_bytes_masked() bytes; otherwise it runs unsplit.
 *    The results agree either way.
 *  - The first call on a device looks up the array's device address on that
 *    device (the current device) and caches it; make that first call before
 *    any stream capture.
 *  - Every call on a device shares the one array.  Each call rewrites every
 *    part of it that it reads (the dQ accumulator is cleared first), but
 *    calls whose work overlaps on the GPU (other streams, other host
 *    threads) race on it: serialise them.
 */
#define FA_NOALLOC_SCRATCH_BYTES (32u << 20)
FA_API int fa_backward_noalloc(const void* q, const void* k, const void* v, const void* o,
                               const float* lse, const void* dout, void* dq, void* dk,
                               void* dv, int B, int H, int N, int d, float scale, int causal,
                               const uint8_t* block_mask, const int32_t* kv_len, void* stream);

/*
 * Tile schedule of one batch element, as the kernels enumerate it: every
 * live (query tile, key tile) pair of 128x128 tiles, i.e. every tile pair
 * holding at least one allowed (i, j), in query-tile-major order, with a
 * flag that is 1 when some in-range pair of the tile is disallowed (the
 * kernel masks elements there) and 0 when the tile is fully allowed.
 *   b          : batch element whose kv_len applies (ignored if kv_len NULL).
 *   row_ptr    : int32 [T+1] device, written (CSR offsets by query tile).
 *   col_idx    : int32 [T*T] device, written (key tile of each live pair).
 *   partial    : uint8 [T*T] device, written.
 * Entries of col_idx / partial past row_ptr[T] are left untouched.
 */
FA_API int fa_tile_schedule(int N, int causal, const uint8_t* block_mask,
                     const int32_t* kv_len, int b, int32_t* row_ptr,
                     int32_t* col_idx, uint8_t* partial, void* stream);

/* fa_tile_schedule with the full mask description. */
FA_API int fa_tile_schedule_masked(int N, const fa_mask* mask, int b, int32_t* row_ptr,
                                   int32_t* col_idx, uint8_t* partial, void* stream);

/*
 * Packed variable-length sequences (page "FlashAttention" (aiwiki), section
 * "Software integration and limitations": variable-length sequences are
 * among the method's interfaces).  The B sequences lie back to back along
 * the token axis:
 *   q, k, v, o, dout, dq, dk, dv : bf16 [total, H, d] (token-major), 16-byte
 *                                  aligned;
 *   lse                          : fp32 [H, total];
 *   cu_seqlens                   : int32 [B+1] device; sequence b is tokens
 *                                  cu_seqlens[b] .. cu_seqlens[b+1]-1,
 *                                  normally cu_seqlens[0] = 0 and
 *                                  cu_seqlens[B] = total;
 *   max_seqlen                   : at least every sequence's length (sizes
 *                                  the grid; <= 8,388,480).
 * Each sequence attends only within itself, exactly as a batch element of
 * its own length would under fa_forward_masked: token t = cu_seqlens[b] + i
 * is query/key i of sequence b.  mask may give causal and the sliding
 * window; block_mask and kv_len must be NULL (FA_ERR_UNSUPPORTED otherwise).
 * Offsets out of order, out of [0, total] or longer than max_seqlen are
 * clamped in the kernels, which then record FA_ERR_INVALID_ARG in the error
 * word read by fa_last_device_status.  O, LSE, dK and dV of tokens outside
 * every sequence are not written; their dQ is 0.
 */
FA_API int fa_forward_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                             const int32_t* cu_seqlens, int B, int H, int total,
                             int max_seqlen, int d, float scale, const fa_mask* mask,
                             void* stream);

/* Workspace of fa_backward_varlen: LSE*log2(e) and D per sequence row, padded
 * (fp32 [B*H][ceil(max_seqlen/128)*128] each), then the fp32 dQ accumulator
 * [H, total, d] (head-major); each part 256-byte aligned.  0 for invalid
 * sizes. */
FA_API size_t fa_varlen_workspace_bytes(int B, int H, int total, int max_seqlen, int d);

/* Backward of fa_forward_varlen (same sequences, mask and scale); launches
 * the packed preprocess, the dK/dV/dQ kernel and the dQ conversion. */
FA_API int fa_backward_varlen(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dout, void* dq, void* dk, void* dv,
                              const int32_t* cu_seqlens, int B, int H, int total,
                              int max_seqlen, int d, float scale, const fa_mask* mask,
                              void* workspace, size_t workspace_bytes, void* stream);

/*
 * Reads and clears the library's device error word on the current device
 * after synchronising `stream`.  Kernels that wait on an mbarrier give up
 * after a bounded number of polls, record FA_ERR_TIMEOUT there and exit,
 * so a lost signal surfaces here instead of hanging the GPU.
 * Returns FA_OK, FA_ERR_TIMEOUT, or FA_ERR_CUDA if synchronisation failed.
 */
FA_API int fa_last_device_status(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
