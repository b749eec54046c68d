// Single-tile tensor-core self-test: exercises, one at a time, the operand
// paths the attention kernels are built from (TMA with the 128- and 32-byte swizzles,
// K-major and MN-major shared-memory descriptors, A staged in TMEM, TMEM
// loads) on one 128-row tile, so a layout mistake shows up as a wrong
// product here rather than as a wrong attention output.
#include <cuda_bf16.h>

#include "../../include/fa_selftest.h"
#include "fa_common.cuh"
#include "fa_kernels.h"
#include "fa_sm100.cuh"
#include "fa_tma_host.h"

namespace fa {
using namespace sm100;

constexpr int kHalf = 128 * 128;  // bytes of one 128-row x 64-column bf16 box

__global__ void __launch_bounds__(128, 1)
    selftest_kernel(const __grid_constant__ CUtensorMap tm_a,
                    const __grid_constant__ CUtensorMap tm_b, const __nv_bfloat16* a_glob,
                    float* c, int mode, int n, int* status) {
  extern __shared__ uint8_t smem_raw[];
  // An offset (not an integer round trip) keeps the pointer visibly in shared
  // memory, so C++ accesses through it compile to shared-memory instructions.
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sA = smem_u32(smem);
  const uint32_t sB = sA + 2 * kHalf;
  const uint32_t bars = sB + 2 * kHalf;  // [0] tma, [1] mma
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 4 * kHalf + 64);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + 4 * kHalf + 128);
  const Abort ab{abort_flag, status};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int r = threadIdx.x;  // tile row owned by this thread

  if (threadIdx.x == 0) {
    mbar_init(bars, 1);
    mbar_init(bars + 8, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int b_halves = (mode == 0) ? 2 : n / 64;
  if (threadIdx.x == 0) {
    if (mode >= 6) {
      // K = 16: one 32-byte-swizzled box of 16 columns per operand
      mbar_expect_tx(bars, (mode == 7 ? 128 * 32 : 0) + n * 32);
      if (mode == 7) tma_load_3d(sA, &tm_a, bars, 0, 0, 0);
      tma_load_3d(sB, &tm_b, bars, 0, 0, 0);
    } else if (mode == 5) {
      // 8-bit: one 128-byte-wide box of 128 rows per operand
      mbar_expect_tx(bars, 2 * kHalf);
      tma_load_3d(sA, &tm_a, bars, 0, 0, 0);
      tma_load_3d(sB, &tm_b, bars, 0, 0, 0);
    } else {
      const bool a_by_tma = (mode == 0 || mode == 1 || mode == 4);
      mbar_expect_tx(bars, (a_by_tma ? 2 * kHalf : 0) + b_halves * kHalf);
      if (a_by_tma)
        for (int h = 0; h < 2; ++h) tma_load_3d(sA + h * kHalf, &tm_a, bars, h * 64, 0, 0);
      for (int h = 0; h < b_halves; ++h) tma_load_3d(sB + h * kHalf, &tm_b, bars, h * 64, 0, 0);
    }
  }
  if (mode == 2) {
    // A row r -> TMEM lane r, columns 128..191 (two bf16 per 32-bit column)
    uint32_t v[32];
    const uint32_t* src = reinterpret_cast<const uint32_t*>(a_glob + r * 128);
    for (int h = 0; h < 2; ++h) {
      for (int j = 0; j < 32; ++j) v[j] = src[h * 32 + j];
      tmem_st32(tmem + ((uint32_t)(warp * 32) << 16) + 128 + h * 32, v);
    }
    tmem_st_wait();
  }
  if (mode == 3) {
    // A row r written by this thread into the 128-byte-swizzled K-major layout
    const uint4* src = reinterpret_cast<const uint4*>(a_glob + r * 128);
    for (int ch = 0; ch < 16; ++ch) {
      const int h = ch >> 3, w = ch & 7;
      *reinterpret_cast<uint4*>(smem + h * kHalf + r * 128 + ((w ^ (r & 7)) << 4)) = src[ch];
    }
    fence_proxy_async_smem();
  }
  if (mode == 6) {
    // A row r (first 16 columns) written by this thread in the 32-byte-swizzled layout
    const uint4* src = reinterpret_cast<const uint4*>(a_glob + r * 128);
    for (int ch = 0; ch < 2; ++ch) *reinterpret_cast<uint4*>(smem + sw32_offset(r, ch)) = src[ch];
    fence_proxy_async_smem();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  bool ok = mbar_wait(bars, 0, ab);
  if (ok && threadIdx.x == 0) {
    tc_fence_after();
    if (mode >= 6) {
      // c = a[:, :16] b[:, :16]^T: one MMA of depth 16, both operands K-major
      // with the 32-byte swizzle (8-row groups 256 bytes apart)
      mma_ss(tmem, sdesc_sw32(sA, 256), sdesc_sw32(sB, 256), idesc_bf16(128, n, false, false), 0);
    } else if (mode == 5) {
      // c = a b^T with e4m3 operands, both K-major: K = 128 in four steps of
      // 32 elements (32 bytes) along the swizzled rows
      const uint32_t id = idesc_e4m3(128, 128);
      for (int kk = 0; kk < 4; ++kk)
        mma_ss_f8(tmem, sdesc_sw128(sA + kk * 32, 16, 1024), sdesc_sw128(sB + kk * 32, 16, 1024),
                  id, kk > 0);
    } else if (mode == 4) {
      // c = a^T b: A operand MN-major (M = columns of a, K = rows of a)
      const uint32_t id = idesc_bf16(128, n, true, true);
      for (int kk = 0; kk < 8; ++kk)
        mma_ss(tmem, sdesc_sw128(sA + kk * 2048, kHalf, 1024),
               sdesc_sw128(sB + kk * 2048, kHalf, 1024), id, kk > 0);
    } else if (mode == 0) {
      const uint32_t id = idesc_bf16(128, 128, false, false);
      for (int kk = 0; kk < 8; ++kk) {
        const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
        mma_ss(tmem, sdesc_sw128(sA + off, 16, 1024), sdesc_sw128(sB + off, 16, 1024), id, kk > 0);
      }
    } else {
      const uint32_t id = idesc_bf16(128, n, false, true);
      for (int kk = 0; kk < 8; ++kk) {
        const uint64_t bd = sdesc_sw128(sB + kk * 2048, kHalf, 1024);
        if (mode == 2) {
          mma_ts(tmem, tmem + 128 + kk * 8, bd, id, kk > 0);
        } else {
          const uint32_t off = (kk >> 2) * kHalf + (kk & 3) * 32;
          mma_ss(tmem, sdesc_sw128(sA + off, 16, 1024), bd, id, kk > 0);
        }
      }
    }
    mma_commit(bars + 8);
  }
  __syncwarp();
  ok = ok && mbar_wait(bars + 8, 0, ab);
  tc_fence_after();
  if (ok) {
    const int ncols = (mode == 0 || mode == 5) ? 128 : n;
    for (int c0 = 0; c0 < ncols; c0 += 32) {
      uint32_t v[32];
      tmem_ld32(tmem + ((uint32_t)(warp * 32) << 16) + c0, v);
      for (int j = 0; j < 32; ++j) c[r * ncols + c0 + j] = __uint_as_float(v[j]);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

}  // namespace fa

using namespace fa;

extern "C" int fa_selftest_mma(int mode, const void* a, const void* b, float* c, int n,
                               void* stream) {
  if (mode < 0 || mode > 7 || !a || !b || !c) return 1;
  if (mode != 0 && mode != 5 && n != 64 && n != 128) return 1;
  CUtensorMap ta, tb;
  if (mode >= 6) {
    if (!make_bf16_map_sw32(&ta, a, 128, 128, 1, 128) || !make_bf16_map_sw32(&tb, b, 128, n, 1, n))
      return 3;
  } else if (mode == 5) {
    if (!make_u8_map_3d(&ta, a, 128, 128, 1, 128) || !make_u8_map_3d(&tb, b, 128, 128, 1, 128))
      return 3;
  } else {
    if (!make_bf16_map_3d(&ta, a, 128, 128, 1, 128)) return 3;
    if (!make_bf16_map_3d(&tb, b, mode == 0 ? 128 : n, 128, 1, 128)) return 3;
  }
  const int smem = 4 * kHalf + 1024 + 256;
  if (cudaFuncSetAttribute(selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return 3;
  int* st = status_word();
  if (st == nullptr) return 3;
  selftest_kernel<<<1, 128, smem, static_cast<cudaStream_t>(stream)>>>(
      ta, tb, static_cast<const __nv_bfloat16*>(a), c, mode, n, st);
  return cudaGetLastError() == cudaSuccess ? 0 : 3;
}
