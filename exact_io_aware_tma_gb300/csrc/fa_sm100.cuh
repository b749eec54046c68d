// Blackwell (sm_100 family, built for sm_103a) device primitives in inline
// PTX: mbarriers with bounded waits, TMA tensor copies, and the tcgen05
// tensor-core instructions (TMEM allocation, MMA, commit, TMEM load/store).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {
namespace sm100 {

// A wait that has not completed after this long (ns) is treated as lost: the
// waiter records FA_ERR_TIMEOUT and the CTA winds down instead of hanging.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
// The limit of the self-test instantiations that withhold one arrival on
// purpose (so that a wait runs out quickly).
constexpr uint64_t kShortWaitLimitNs = 1000000ull;
constexpr int kStatusTimeout = 4;  // FA_ERR_TIMEOUT

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// The same test, but the thread may stay suspended until the phase completes
// or up to `hint_ns` nanoseconds have passed (instead of the hardware's own,
// short, limit), so a waiting thread does not keep re-issuing the test and
// take issue slots from the other warps of its SM sub-partition.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity,
                                                    uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Non-blocking test of the same condition (no suspend window).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Shared abort word of a CTA plus the global status word.
struct Abort {
  volatile int* flag;                 // shared memory
  int* status;                        // global
  uint64_t limit_ns = kWaitLimitNs;   // how long a wait may take
};

// Suspension hints (ns) of the two kinds of waits.  Latency-critical waiters
// (MMA issuers, softmax / element-wise warps) poll (hint 0: the hardware's
// own short suspension), since a thread sleeping in the barrier resumes up
// to about a microsecond after the phase completes.  Background waiters (the
// TMA producer, the dQ warps) sleep in the barrier, so that they do not take
// issue slots from the critical warps of their SM sub-partition; the abort
// flag and the time limit are re-checked at least this often.
constexpr uint32_t kPollHintNs = 0;
constexpr uint32_t kSleepHintNs = 20000;

// Waits until the phase of `bar` with parity `parity` has completed.  Returns
// false (and raises the CTA's abort flag and the global status) on timeout,
// or false at once if another warp of the CTA already aborted.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const Abort& ab,
                                          uint32_t hint_ns = kPollHintNs) {
  if (mbar_test(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (hint_ns != 0 ? mbar_try_wait_sleep(bar, parity, hint_ns) : mbar_try_wait(bar, parity))
      return true;
    if (*ab.flag) return false;
    if (globaltimer() - t0 > ab.limit_ns) {
      *ab.flag = 1;
      atomicExch(ab.status, kStatusTimeout);
      return false;
    }
  }
}

// ------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int c0, int c1,
                                             int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// Plain (untensored) bulk copy global -> shared; both addresses 16-byte
// aligned, size a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// Element-wise add of a shared-memory tile into the global tensor of `map`
// (a reduce-add performed by the TMA unit); elements outside the tensor are
// skipped.  The innermost coordinate times the element size must be a
// multiple of 16 bytes, and no coordinate may be negative.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, uint32_t src, int c0,
                                                  int c1, int c2) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group"
      " [%0, {%2, %3, %4}], [%1];" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(src), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}
// Waits until at most one committed bulk group still reads shared memory.
__device__ __forceinline__ void bulk_wait_read_1() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
__device__ __forceinline__ void tma_store_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void tma_store_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Makes generic-proxy shared-memory writes visible to the async proxy (TMA
// store, tcgen05.mma operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void named_barrier(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// ------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem desc]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc], 8-bit floating-point operands
// (kind::f8f6f4; K = 32 per instruction), fp32 accumulation.
__device__ __forceinline__ void mma_ss_f8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when every tcgen05 operation this thread issued so far
// has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

// Instruction descriptor of kind::f16 with bf16 A/B and fp32 accumulation.
// Bit fields: [4,6) D format (1 = f32), [7,10) A format (1 = bf16),
// [10,13) B format (1 = bf16), 15 A MN-major, 16 B MN-major,
// [17,23) N >> 3, [24,29) M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor of kind::f8f6f4 with e4m3 A and B (format code 0
// in both fields), fp32 accumulation, both operands K-major.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor for a 128-byte-swizzled operand tile.
// [0,14) start >> 4, [16,30) leading-dim byte offset >> 4, [32,46) stride-dim
// byte offset >> 4, [46,48) version 1, [61,64) layout 2 = 128B swizzle.
// K-major tiles: rows of 128 bytes, 8-row groups 1024 bytes apart (SBO).
// MN-major tiles: LBO = distance between 64-element column blocks, SBO =
// distance between 8-row groups along K.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// The same descriptor for a 32-byte-swizzled K-major operand (layout 6):
// rows of 32 bytes (K = 16 bf16, one MMA's depth), 8-row groups `sbo` bytes
// apart; within a group the two 16-byte halves of rows 4-7 trade places.
__device__ __forceinline__ uint64_t sdesc_sw32(uint32_t saddr, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | (1ull << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (6ull << 61);
}

// Byte offset of 16-byte half `c` (0 or 1) of row r in a 32-byte-swizzled
// K-major tile whose 8-row groups are 256 bytes apart.
__host__ __device__ constexpr uint32_t sw32_offset(int r, int c) {
  return (uint32_t)r * 32u + ((uint32_t)(c ^ ((r >> 2) & 1)) << 4);
}


// ---- GEMMs issued as one instruction sequence each (descriptor offsets
// folded into immediates; the first MMA honours `acc`, the rest accumulate).

// K = 128 (8 MMAs), both operands K-major in 16 KB column halves.
__device__ __forceinline__ void mma_ss_kmajor_k128_h16k(uint32_t d, uint64_t a, uint64_t b, uint32_t id,
                                      uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p, t;\n .reg .b64 a, b;\n"
      " setp.ne.b32 p, %4, 0;\n setp.eq.u32 t, 1, 1;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
      " add.s64 a, %1, 2;\n add.s64 b, %2, 2;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      " add.s64 a, %1, 4;\n add.s64 b, %2, 4;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      " add.s64 a, %1, 6;\n add.s64 b, %2, 6;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      " add.s64 a, %1, 1024;\n add.s64 b, %2, 1024;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      " add.s64 a, %1, 1026;\n add.s64 b, %2, 1026;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      " add.s64 a, %1, 1028;\n add.s64 b, %2, 1028;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      " add.s64 a, %1, 1030;\n add.s64 b, %2, 1030;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      "}\n" ::"r"(d), "l"(a), "l"(b), "r"(id), "r"(acc)
      : "memory");
}

// K = 64 (4 MMAs), both operands K-major (one 64-column half).
__device__ __forceinline__ void mma_ss_kmajor_k64(uint32_t d, uint64_t a, uint64_t b, uint32_t id,
                                      uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p, t;\n .reg .b64 a, b;\n"
      " setp.ne.b32 p, %4, 0;\n setp.eq.u32 t, 1, 1;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
      " add.s64 a, %1, 2;\n add.s64 b, %2, 2;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      " add.s64 a, %1, 4;\n add.s64 b, %2, 4;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      " add.s64 a, %1, 6;\n add.s64 b, %2, 6;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      "}\n" ::"r"(d), "l"(a), "l"(b), "r"(id), "r"(acc)
      : "memory");
}

// K = 128 (8 MMAs): A from TMEM (8 columns per K step), B MN-major (16 rows = 2048 B per step).
__device__ __forceinline__ void mma_ts_mn_k128(uint32_t d, uint32_t a, uint64_t b, uint32_t id,
                                      uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p, t;\n .reg .b32 a;\n .reg .b64 b;\n"
      " setp.ne.b32 p, %4, 0;\n setp.eq.u32 t, 1, 1;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n"
      " add.u32 a, %1, 8;\n add.s64 b, %2, 128;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, t;\n"
      " add.u32 a, %1, 16;\n add.s64 b, %2, 256;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, t;\n"
      " add.u32 a, %1, 24;\n add.s64 b, %2, 384;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, t;\n"
      " add.u32 a, %1, 32;\n add.s64 b, %2, 512;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, t;\n"
      " add.u32 a, %1, 40;\n add.s64 b, %2, 640;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, t;\n"
      " add.u32 a, %1, 48;\n add.s64 b, %2, 768;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, t;\n"
      " add.u32 a, %1, 56;\n add.s64 b, %2, 896;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, t;\n"
      "}\n" ::"r"(d), "r"(a), "l"(b), "r"(id), "r"(acc)
      : "memory");
}


// ---- backward GEMM patterns (same convention as above)

// K = 128 (8 MMAs): A K-major in 16 KB halves, B K-major in 8 KB halves.
__device__ __forceinline__ void mma_ss_kmajor_k128_a16k_b8k(uint32_t d, uint64_t a, uint64_t b, uint32_t id,
                                      uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p, t;\n .reg .b64 a, b;\n"
      " setp.ne.b32 p, %4, 0;\n setp.eq.u32 t, 1, 1;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
      " add.s64 a, %1, 2;\n add.s64 b, %2, 2;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      " add.s64 a, %1, 4;\n add.s64 b, %2, 4;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      " add.s64 a, %1, 6;\n add.s64 b, %2, 6;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      " add.s64 a, %1, 1024;\n add.s64 b, %2, 512;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      " add.s64 a, %1, 1026;\n add.s64 b, %2, 514;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      " add.s64 a, %1, 1028;\n add.s64 b, %2, 516;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      " add.s64 a, %1, 1030;\n add.s64 b, %2, 518;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      "}\n" ::"r"(d), "l"(a), "l"(b), "r"(id), "r"(acc)
      : "memory");
}

// K = 64 (4 MMAs): A and B K-major (one 64-column half each).
__device__ __forceinline__ void mma_ss_kmajor_k64_a16k_b8k(uint32_t d, uint64_t a, uint64_t b, uint32_t id,
                                      uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p, t;\n .reg .b64 a, b;\n"
      " setp.ne.b32 p, %4, 0;\n setp.eq.u32 t, 1, 1;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
      " add.s64 a, %1, 2;\n add.s64 b, %2, 2;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      " add.s64 a, %1, 4;\n add.s64 b, %2, 4;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      " add.s64 a, %1, 6;\n add.s64 b, %2, 6;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      "}\n" ::"r"(d), "l"(a), "l"(b), "r"(id), "r"(acc)
      : "memory");
}

// K = 64 (4 MMAs): A from TMEM, B MN-major.
__device__ __forceinline__ void mma_ts_mn_k64(uint32_t d, uint32_t a, uint64_t b, uint32_t id,
                                      uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p, t;\n .reg .b32 a;\n .reg .b64 b;\n"
      " setp.ne.b32 p, %4, 0;\n setp.eq.u32 t, 1, 1;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n"
      " add.u32 a, %1, 8;\n add.s64 b, %2, 128;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, t;\n"
      " add.u32 a, %1, 16;\n add.s64 b, %2, 256;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, t;\n"
      " add.u32 a, %1, 24;\n add.s64 b, %2, 384;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, t;\n"
      "}\n" ::"r"(d), "r"(a), "l"(b), "r"(id), "r"(acc)
      : "memory");
}

// K = 64 (4 MMAs): A from TMEM in two 16-column halves 32 columns apart
// (columns 0-15 and 32-47), B MN-major.
__device__ __forceinline__ void mma_ts_mn_k64_gap32(uint32_t d, uint32_t a, uint64_t b, uint32_t id,
                                      uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p, t;\n .reg .b32 a;\n .reg .b64 b;\n"
      " setp.ne.b32 p, %4, 0;\n setp.eq.u32 t, 1, 1;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n"
      " add.u32 a, %1, 8;\n add.s64 b, %2, 128;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, t;\n"
      " add.u32 a, %1, 32;\n add.s64 b, %2, 256;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, t;\n"
      " add.u32 a, %1, 40;\n add.s64 b, %2, 384;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [a], b, %3, t;\n"
      "}\n" ::"r"(d), "r"(a), "l"(b), "r"(id), "r"(acc)
      : "memory");
}

// K = 64 (4 MMAs): A K-major within one 128-byte row, B MN-major.
__device__ __forceinline__ void mma_ss_kmajor_mn_k64(uint32_t d, uint64_t a, uint64_t b, uint32_t id,
                                      uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p, t;\n .reg .b64 a, b;\n"
      " setp.ne.b32 p, %4, 0;\n setp.eq.u32 t, 1, 1;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
      " add.s64 a, %1, 2;\n add.s64 b, %2, 128;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      " add.s64 a, %1, 4;\n add.s64 b, %2, 256;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      " add.s64 a, %1, 6;\n add.s64 b, %2, 384;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      "}\n" ::"r"(d), "l"(a), "l"(b), "r"(id), "r"(acc)
      : "memory");
}

// K = 128 (8 MMAs): A and B both MN-major.
__device__ __forceinline__ void mma_ss_mn_mn_k128(uint32_t d, uint64_t a, uint64_t b, uint32_t id,
                                      uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p, t;\n .reg .b64 a, b;\n"
      " setp.ne.b32 p, %4, 0;\n setp.eq.u32 t, 1, 1;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n"
      " add.s64 a, %1, 128;\n add.s64 b, %2, 128;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      " add.s64 a, %1, 256;\n add.s64 b, %2, 256;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      " add.s64 a, %1, 384;\n add.s64 b, %2, 384;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      " add.s64 a, %1, 512;\n add.s64 b, %2, 512;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      " add.s64 a, %1, 640;\n add.s64 b, %2, 640;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      " add.s64 a, %1, 768;\n add.s64 b, %2, 768;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      " add.s64 a, %1, 896;\n add.s64 b, %2, 896;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, t;\n"
      "}\n" ::"r"(d), "l"(a), "l"(b), "r"(id), "r"(acc)
      : "memory");
}


// TMEM -> registers: 32 lanes x 32 consecutive 32-bit columns; thread t of
// the warp receives lane (warp's lane base + t).  Waits for completion.
#define FA_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), \
                 "=r"(r[i + 4]), "=r"(r[i + 5]), "=r"(r[i + 6]), "=r"(r[i + 7])
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : FA_R8(0), FA_R8(8), FA_R8(16), FA_R8(24)
      : "r"(taddr)
      : "memory");
}
#undef FA_R8


// TMEM -> registers, 32 lanes x 128 consecutive columns in one instruction,
// then one completion wait.
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%128];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr)
      : "memory");
}

// TMEM -> registers: 32 lanes x 64 columns, one completion wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n"
      "tcgen05.wait::ld.sync.aligned;\n"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
}



// ---- packed fp32 arithmetic (two lanes per instruction) and 3-input max
__device__ __forceinline__ void fma2(float& d0, float& d1, float a0, float a1, float b0, float b1,
                                     float c0, float c1) {
  asm("{\n .reg .b64 x, y, z, w;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %5};\n"
      " mov.b64 z, {%6, %7};\n fma.rn.f32x2 w, x, y, z;\n mov.b64 {%0, %1}, w;\n}\n"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}
__device__ __forceinline__ void add2(float& d0, float& d1, float a0, float a1, float b0, float b1) {
  asm("{\n .reg .b64 x, y, w;\n mov.b64 x, {%2, %3};\n mov.b64 y, {%4, %5};\n"
      " add.rn.f32x2 w, x, y;\n mov.b64 {%0, %1}, w;\n}\n"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b0), "f"(b1));
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

#define FA_W8(i) "r"(r[i]), "r"(r[i + 1]), "r"(r[i + 2]), "r"(r[i + 3]), \
                 "r"(r[i + 4]), "r"(r[i + 5]), "r"(r[i + 6]), "r"(r[i + 7])
// registers -> TMEM, 32 lanes x 32 columns (no wait; see tmem_st_wait).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n" ::"r"(taddr),
      FA_W8(0), FA_W8(8), FA_W8(16), FA_W8(24)
      : "memory");
}
// registers -> TMEM, 32 lanes x 16 columns.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n" ::"r"(taddr),
      FA_W8(0), FA_W8(8)
      : "memory");
}
#undef FA_W8
__device__ __forceinline__ void tmem_st_wait() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}


}  // namespace sm100
}  // namespace fa
