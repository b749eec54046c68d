// Internal launch entry points of the attention kernels (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>

#include "fa_common.cuh"

namespace fa {

cudaError_t launch_fwd_tc(const Problem& p, const void* q, const void* k, const void* v,
                          void* o, float* lse, cudaStream_t st);

int* status_word();

cudaError_t launch_bwd_tc(const Problem& p, const void* q, const void* k, const void* v,
                          const void* dout, const float* lse2, const float* dvec, float* dq_acc,
                          void* dk, void* dv, int npad, cudaStream_t st);

}  // namespace fa
