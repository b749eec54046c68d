/*
 * fa_selftest.h -- tensor-core self-test of the attention library.
 *
 * Not part of the attention method: a check of the sm_103a building blocks
 * the attention kernels are assembled from, on one 128-row tile, so that a
 * wrong operand layout is caught in isolation.  All pointers are device
 * pointers; the call is asynchronous on `stream`.
 *
 *   a : bf16 [128][128] row-major.
 *   b : mode 0: bf16 [128][128] row-major (one row per output column);
 *       modes 1-4: bf16 [128][n] row-major.
 *   c : fp32 [128][n] row-major output (n = 128 in mode 0).
 *   mode 0: c = a * b^T  (both operands K-major in shared memory via TMA;
 *           the S = Q K^T path).
 *   mode 1: c = a * b    (a K-major via TMA, b MN-major via TMA; the
 *           O += P V path with P in shared memory).
 *   mode 2: c = a * b    (a written to tensor memory by tcgen05.st, b
 *           MN-major via TMA; the O += P V path with P in tensor memory).
 *   mode 3: c = a * b    (a written to shared memory by threads in the
 *           128-byte-swizzled layout, b MN-major via TMA).
 *   mode 4: c = a^T * b (a MN-major via TMA, i.e. the M index runs along
 *           a's rows in memory; b MN-major via TMA; the dQ^T = K^T dS^T
 *           path of the backward).
 *   mode 5: c = a * b^T with a, b e4m3 (8-bit float) [128][128] row-major,
 *           both K-major via TMA (the FP8 S = Q K^T and O += P V paths).
 *   mode 6: c = a[:, :16] * b[:, :16]^T with b bf16 [n][128] row-major: one
 *           MMA of depth 16, both operands K-major with the 32-byte swizzle,
 *           a written to shared memory by threads, b via TMA (the row
 *           statistic operand of the backward).
 *   mode 7: as mode 6 with a also via TMA.
 *   n    : 64 or 128 (modes 1-4, 6, 7).
 * Returns 0 on success, 1 on a bad argument, 3 on a CUDA error.  A bounded
 * wait that gives up is reported by fa_last_device_status().
 */
#ifndef FA_GB300_SELFTEST_H
#define FA_GB300_SELFTEST_H

#include "fa.h"

#ifdef __cplusplus
extern "C" {
#endif

FA_API int fa_selftest_mma(int mode, const void* a, const void* b, float* c, int n,
                           void* stream);

/*
 * Self-test of the bounded waits (failure detection without a GPU fault).
 * Every mbarrier wait in the attention kernels gives up after a time limit,
 * records FA_ERR_TIMEOUT in the library's device error word, makes the other
 * warps of its CTA stop, lets the CTA's copies and tensor-core work in
 * flight finish (again with bounded waits), frees its tensor memory and
 * exits, so a lost signal cannot hang the GPU.  These two entry points run
 * that path on purpose: the same arguments as fa_forward / fa_backward (no
 * block mask or key lengths; d = 128 or 64, the forward's d = 64 kernel
 * being the one-query-tile one with P in TMEM columns of its own and the
 * backward's the persistent one; FA_ERR_UNSUPPORTED for other d), but one
 * warp of each CTA withholds one arrival (the
 * forward's first softmax warp its P-ready signal for its first key tile;
 * the backward's first element-wise warp its signal for the CTA's first
 * query step) and the waits give up after 1 ms instead of 2 s.  The call returns FA_OK at
 * launch; fa_last_device_status() then returns FA_ERR_TIMEOUT (and clears
 * it), the outputs are unspecified, and the device stays usable.
 */
FA_API int fa_selftest_forward_lost_signal(const void* q, const void* k, const void* v, void* o,
                                           float* lse, int B, int H, int N, int d, float scale,
                                           int causal, void* stream);
FA_API int fa_selftest_backward_lost_signal(const void* q, const void* k, const void* v,
                                            const void* o, const float* lse, const void* dout,
                                            void* dq, void* dk, void* dv, int B, int H, int N,
                                            int d, float scale, int causal, void* workspace,
                                            size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_SELFTEST_H */
