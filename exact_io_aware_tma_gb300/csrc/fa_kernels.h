// Internal launch entry points of the attention kernels (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>

#include "fa_common.cuh"

namespace fa {

cudaError_t launch_fwd_tc(const Problem& p, const void* q, const void* k, const void* v,
                          void* o, float* lse, cudaStream_t st);

int* status_word();

// split != nullptr (padded layout with a block mask): the work of key tiles
// with many live query tiles is spread over several CTAs by a plan kernel
// launched first (BwdSplit in fa_common.cuh).
cudaError_t launch_bwd_tc(const Problem& p, const void* q, const void* k, const void* v,
                          const void* dout, const float* lse2, const float* dvec, float* dq_acc,
                          void* dk, void* dv, int npad, const BwdSplit* split, cudaStream_t st);

// Self-test launches of the d = 128 forward (tile-pair CTAs) and dK/dV
// kernels in which one warp withholds one arrival and waits give up after
// 1 ms: the bounded-wait abort path, reached on purpose (padded layout, no
// dropout; cudaErrorInvalidValue otherwise).
cudaError_t launch_fwd_tc_lost_signal(const Problem& p, const void* q, const void* k,
                                      const void* v, void* o, float* lse, cudaStream_t st);
cudaError_t launch_bwd_tc_lost_signal(const Problem& p, const void* q, const void* k,
                                      const void* v, const void* dout, const float* lse2,
                                      const float* dvec, float* dq_acc, void* dk, void* dv,
                                      int npad, cudaStream_t st);

// e4m3 forward (d = 128) on quantised operands: q8, k8 [B*H][N][128],
// vt8 [B*H][128][ceil(N/128)*128], q/k scales [B*H][T], v scale [B*H].
cudaError_t launch_fwd_fp8(const Problem& p, const void* q8, const void* k8, const void* vt8,
                           const float* q_scale, const float* k_scale, const float* v_scale,
                           void* o, float* lse, cudaStream_t st);

}  // namespace fa
