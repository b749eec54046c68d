// Shared device helpers of the attention kernels: the allowed-pair predicate,
// the live-tile walk, bf16 packing and the warp-level tensor-core fragments.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

constexpr int kTile = 128;  // block-mask tile side (queries and keys)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Arguments every kernel shares.  Pointers are device pointers.
struct Problem {
  int B, H, N, d;
  int T;                  // ceil(N / 128)
  float scale;            // multiplies Q K^T
  float scale_log2;       // scale * log2(e): scores are kept in log2 units
  int causal;
  const uint8_t* block_mask;  // [T, T] or nullptr
  const int32_t* kv_len;      // [B] or nullptr
  int* status;                // device error word (bounded waits record here)
};

// Valid-key bound of batch element b: min(N, max(0, kv_len[b])).
__device__ __forceinline__ int key_limit(const Problem& p, int b) {
  if (p.kv_len == nullptr) return p.N;
  int l = __ldg(p.kv_len + b);
  return l < 0 ? 0 : (l > p.N ? p.N : l);
}

// A (query tile, key tile) pair is live when some (i, j) in it is allowed.
// With equal query and key lengths the causal rule keeps kt <= qt.
__device__ __forceinline__ bool tile_live(const Problem& p, int qt, int kt,
                                          int klim) {
  if (p.causal && kt > qt) return false;
  if (kt * kTile >= klim) return false;
  if (p.block_mask != nullptr && __ldg(p.block_mask + (size_t)qt * p.T + kt) == 0)
    return false;
  return true;
}

// A live tile needs element masking when some in-range (i, j) of it is not
// allowed: the causal diagonal tile, or a tile crossing the key limit.
__device__ __forceinline__ bool tile_partial(const Problem& p, int qt, int kt,
                                             int klim) {
  // Causal diagonal tile: some j > i exists once it holds two rows in range.
  if (p.causal && kt == qt && p.N - qt * kTile > 1) return true;
  // Key limit inside the tile's in-range columns.
  return klim < min(p.N, (kt + 1) * kTile);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- Ampere-style async copy, ldmatrix and mma.sync (warp-level path) ----

__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, bool valid) {
  int n = valid ? 16 : 0;  // zero-fill when the source row is out of range
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst),
               "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;\n" ::);
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                        uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                          uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D(16x8 fp32) += A(16x16 bf16, row) * B(16x8 bf16, col)
__device__ __forceinline__ void mma_bf16(float* c, const uint32_t* a, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Byte offset of 16-byte chunk `c` of row `r` in a row-major bf16 tile whose
// rows hold `chunks` chunks (a power of two), with the chunk index XOR-
// swizzled by the row so that eight rows read at one column hit different
// bank groups.
__device__ __forceinline__ uint32_t swz(int r, int c, int chunks) {
  int m = chunks >= 8 ? 7 : chunks - 1;
  return (uint32_t)((r * chunks + (c ^ (r & m))) * 16);
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace fa
