// Internal launch entry points of the attention kernels (not part of the C ABI).
#pragma once

#include <cuda_runtime.h>

#include "fa_common.cuh"

namespace fa {

// Launch of `kern` on `st`; with `early`, the programmatic stream-serialisation
// attribute lets it start before the previous kernel in the stream ends (the
// kernel then calls griddep_wait() before it touches that kernel's output).
template <class... Params, class... Args>
cudaError_t launch_k(bool early, void (*kern)(Params...), dim3 grid, dim3 block, size_t smem,
                     cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = early ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Params>(args)...);
}

cudaError_t launch_fwd_tc(const Problem& p, const void* q, const void* k, const void* v,
                          void* o, float* lse, cudaStream_t st);

int* status_word();

// split != nullptr (padded layout with a block mask): the work of key tiles
// with many live query tiles is spread over several CTAs by a plan kernel
// (BwdSplit in fa_common.cuh), launched first unless `early`.  early: the
// call comes straight after the preprocess kernel's launch, and the plan (for
// a split) was launched before that preprocess; the dK/dV kernel may then
// start while the preprocess runs.  next_item: the work-item counter of the
// persistent d = 64 kernel (padded layout, no dropout), cleared by the
// preprocess; nullptr for the other forms.
cudaError_t launch_bwd_tc(const Problem& p, const void* q, const void* k, const void* v,
                          const void* dout, const float* lse2, const float* dvec, float* dq_acc,
                          void* dk, void* dv, int npad, const BwdSplit* split,
                          unsigned long long* next_item, bool early, cudaStream_t st);
cudaError_t launch_bwd_plan(const Problem& p, const BwdSplit& split, cudaStream_t st);

// The persistent dK/dV kernel of d = 64 (padded layout, no dropout): one CTA
// per SM taking work items from `next_item` (cleared by the preprocess).
// p.hgroup set by the caller; split: the plan's items, or nullptr.  lose:
// the self-test instantiation that withholds one arrival (no split).
cudaError_t launch_bwd_persist(const Problem& p, const void* q, const void* k, const void* v,
                               const void* dout, const float* lse2, const float* dvec,
                               float* dq_acc, void* dk, void* dv, int npad,
                               const BwdSplit* split, unsigned long long* next_item, bool early,
                               cudaStream_t st, bool lose = false);

// Self-test launches of the d = 128 forward (tile-pair CTAs) and of the
// dK/dV kernels (d = 128, and the persistent d = 64 kernel, which takes the
// workspace's work counter) in which one warp withholds one arrival and
// waits give up after 1 ms: the bounded-wait abort path, reached on purpose
// (padded layout, no dropout; cudaErrorInvalidValue otherwise).
cudaError_t launch_fwd_tc_lost_signal(const Problem& p, const void* q, const void* k,
                                      const void* v, void* o, float* lse, cudaStream_t st);
cudaError_t launch_bwd_tc_lost_signal(const Problem& p, const void* q, const void* k,
                                      const void* v, const void* dout, const float* lse2,
                                      const float* dvec, float* dq_acc, void* dk, void* dv,
                                      int npad, unsigned long long* next_item, cudaStream_t st);

// e4m3 forward (d = 128) on quantised operands: q8, k8 [B*H][N][128],
// vt8 [B*H][128][ceil(N/128)*128], q/k scales [B*H][T], v scale [B*H].
cudaError_t launch_fwd_fp8(const Problem& p, const void* q8, const void* k8, const void* vt8,
                           const float* q_scale, const float* k_scale, const float* v_scale,
                           void* o, float* lse, cudaStream_t st);

}  // namespace fa
