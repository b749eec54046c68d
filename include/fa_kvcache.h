/*
 * fa_kvcache.h -- C ABI of attention against a key/value cache, split over
 * the keys, and of the merge of partial attention results.  Part of the
 * library declared in fa.h (same status codes and conventions).
 *
 * What it computes (page "FlashAttention", aiwiki): section "Software
 * integration and limitations" names inference with cached keys and values
 * among the method's interfaces; the arithmetic is the scaled dot-product
 * formula of section "Attention and the memory bottleneck":
 *
 *   for each (b, h) and query row r < Nq, with L = cache_len[b] (clamped
 *   to [0, Nk]; L = Nk when cache_len is NULL):
 *     allowed(r, j) = j < L && (!causal || j <= L - Nq + r)
 *     O[r]   = sum_j softmax_j(scale * q_r . k_j over allowed j) v_j
 *     LSE[r] = natural log-sum-exp of the allowed scaled scores
 *
 * i.e. the Nq query rows are the last Nq tokens of a sequence whose first L
 * tokens are in the cache.  A row with no allowed key gets O = 0 and
 * LSE = -inf.
 *
 * Key splitting and merging (section "Tiling and online normalization"):
 * the allowed key range of every (b, h) is cut into num_splits parts that
 * run on different CTAs; each yields a normalised partial output O_s and
 * its LSE_s, and the parts are folded with the running-max / running-sum /
 * rescaled-accumulator update, treating (O_s, LSE_s) as the state
 * m = LSE_s, l = 1, u = O_s (the kernel evaluates the fold in its closed
 * form LSE = log sum_s e^{LSE_s}, O = sum_s e^{LSE_s - LSE} O_s).  The
 * result equals the unsplit one up to floating-point rounding.
 *
 * Layouts (row-major, device memory, caller-owned):
 *   q, o              : bf16 [B, H, Nq, d], 16-byte aligned
 *   k_cache, v_cache  : bf16 [B, H, Nk, d], 16-byte aligned
 *   lse               : fp32 [B, H, Nq]
 *   cache_len         : int32 [B] or NULL
 *   d in {64, 128}.
 */
#ifndef FA_GB300_KVCACHE_H
#define FA_GB300_KVCACHE_H

#include "fa.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Largest accepted num_splits. */
#define FA_KVCACHE_MAX_SPLITS 256

/*
 * The number of key splits fa_forward_kvcache uses when called with
 * num_splits = 0, for a GPU with num_sms multiprocessors (num_sms <= 0: the
 * current device's count).  A pure host function when num_sms > 0.
 * Returns 0 for invalid sizes (or when the device cannot be queried).
 */
FA_API int fa_kvcache_num_splits(int B, int H, int Nq, int Nk, int d, int num_sms);

/*
 * Bytes of device workspace fa_forward_kvcache needs for this num_splits
 * (0 = the automatic choice on the current device): the partial outputs,
 * fp32 [S][B*H*Nq][d], then the partial LSEs, fp32 [S][B*H*Nq], each part
 * 256-byte aligned.  0 when S = 1 (no workspace is used) and for invalid
 * sizes.
 */
FA_API size_t fa_kvcache_workspace_bytes(int B, int H, int Nq, int Nk, int d, int num_splits);

/*
 * O and LSE of Nq query rows per head against the cache (see above).
 *   scale      : multiplies q . k (usually 1/sqrt(d)); finite.
 *   causal     : nonzero = row r sees keys j <= L - Nq + r.
 *   num_splits : 0 = automatic, else 1 .. FA_KVCACHE_MAX_SPLITS.
 *   workspace  : used only when the split count S > 1; then at least
 *                fa_kvcache_workspace_bytes(.., S) bytes, 256-byte aligned;
 *                contents on entry ignored, on exit unspecified.
 * Requires B, H, Nq, Nk >= 1, B*H <= 2^31-1.  Launches the split kernel
 * and, when S > 1, the merge (fa_combine), both on `stream`.  Cache slots
 * j >= L are never read into the result (they may hold anything).
 */
FA_API int fa_forward_kvcache(const void* q, const void* k_cache, const void* v_cache,
                              void* o, float* lse, int B, int H, int Nq, int Nk, int d,
                              float scale, int causal, const int32_t* cache_len,
                              int num_splits, void* workspace, size_t workspace_bytes,
                              void* stream);

/*
 * Merge of partial attention results over disjoint key sets:
 *   o_parts   : fp32 [num_parts][rows][d], normalised partial outputs,
 *               16-byte aligned;
 *   lse_parts : fp32 [num_parts][rows], their natural-log LSEs; -inf marks
 *               a part with no allowed key (its o_parts row is ignored);
 *   o         : bf16 [rows][d], written, 8-byte aligned;
 *   lse       : fp32 [rows], written.
 * A row whose parts are all empty gets O = 0, LSE = -inf.  Requires
 * num_parts >= 1, rows >= 1, d a multiple of 4 in [4, 1024].
 */
FA_API int fa_combine(const float* o_parts, const float* lse_parts, int num_parts,
                      long long rows, int d, void* o, float* lse, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_KVCACHE_H */
