/*
 * fa_fp8.h -- C ABI of the FP8 (e4m3) attention forward with block
 * quantisation.  Part of the library declared in fa.h (same status codes and
 * conventions).  Inexact by design: page "FlashAttention" (aiwiki), section
 * "Development across generations", describes an FP8 path with block
 * quantisation to reduce quantisation error and asks that such low-precision
 * execution be told apart from exact attention.
 *
 * What is computed, per (b, h), d = 128:
 *   Q, K: per block of 128 rows, scale s = amax / 448 (fp32; 1 for an
 *         all-zero block), code = e4m3(x / s) (fp32 division, round to
 *         nearest even, saturating);
 *   V:    one scale for the whole head, codes likewise, stored transposed;
 *   S = scale * (Q8 K8^T) * sq * sk,  P = the online softmax of S with its
 *   probabilities rounded to e4m3 for the P V product, O = (P8 V8) * sv / l
 *   with l the row sum of the unrounded probabilities, LSE of S.
 * Masks: causal or none (no block mask, key padding or window).
 *
 * Workspace layout (caller-owned, 256-byte aligned, each part 256-byte
 * aligned in this order): q8 e4m3 [B*H][N][128], k8 e4m3 [B*H][N][128],
 * vt8 e4m3 [B*H][128][Np] (Np = ceil(N/128)*128, codes of keys >= N are 0),
 * q scales fp32 [B*H][ceil(N/128)], k scales likewise, v scales fp32 [B*H],
 * then fp32 [B*H][ceil(N/128)] scratch.
 */
#ifndef FA_GB300_FP8_H
#define FA_GB300_FP8_H

#include "fa.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Bytes of workspace of the calls below; 0 for invalid sizes (d != 128 included). */
FA_API size_t fa_fp8_workspace_bytes(int B, int H, int N, int d);

/* Quantise bf16 q, k, v [B,H,N,d] into the workspace (four launches). */
FA_API int fa_fp8_quantize(const void* q, const void* k, const void* v, int B, int H, int N,
                           int d, void* workspace, size_t workspace_bytes, void* stream);

/* Attention on operands already quantised into `workspace` by
 * fa_fp8_quantize (e.g. K and V reused across calls): o bf16 [B,H,N,d],
 * lse fp32 [B,H,N]. */
FA_API int fa_forward_fp8_quantized(const void* workspace, void* o, float* lse, int B, int H,
                                    int N, int d, float scale, int causal, void* stream);

/* fa_fp8_quantize followed by fa_forward_fp8_quantized. */
FA_API int fa_forward_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                          int H, int N, int d, float scale, int causal, void* workspace,
                          size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_FP8_H */
