// FP8 (e4m3) forward with block quantisation: the quantisation kernels and
// the C ABI.  The attention kernel itself is in fa_fwd_fp8.cu.
//
// What is computed (page "FlashAttention" (aiwiki), section "Development
// across generations": an FP8 path with block quantisation to reduce
// quantisation error, to be told apart from exact attention): Q and K are
// quantised per block of 128 rows of one (b, h) -- scale s = amax / 448,
// code = e4m3(x / s), round to nearest even, saturating -- and V per head;
// attention runs on the codes with the scales applied to the scores and the
// output.  V is written transposed ([d][keys]) so that every tensor-core
// operand of the attention kernel is K-major.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include <cmath>
#include <cstdint>

#include "../../include/fa.h"
#include "../../include/fa_fp8.h"
#include "fa_common.cuh"
#include "fa_kernels.h"
#include "fa_sm100.cuh"

namespace fa {
namespace fp8 {

constexpr float kE4m3Max = 448.f;

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  const int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  float m = 0.f;
  for (int i = 0; i < nw; ++i) m = fmaxf(m, red[i]);
  __syncthreads();
  return m;
}

__device__ __forceinline__ uint8_t to_e4m3(float x) {
  return (uint8_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}

// x / s rounded to nearest even, from y = 1/s rounded to nearest: q = x*y is
// within an ulp of the quotient, the remainder x - q*s is exact in one fused
// multiply-add, and q + (x - q*s)*y rounds to the correctly rounded quotient
// (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Dev. 34(1), 1990) -- for quotients and
// s in the normal range, which the callers ensure (|x| <= 448 s, s >= 2^-126;
// otherwise they divide).  An exact quotient keeps q (and its sign).
__device__ __forceinline__ float div_by_scale(float x, float s, float y) {
  const float q = x * y;
  const float r = fmaf(-q, s, x);
  return r == 0.f ? q : fmaf(r, y, q);
}

// Brings one 128-row block (rows x 256 bytes, contiguous) of a bf16
// [BH][N][128] tensor into shared memory with a single bulk copy.  Returns
// false if the copy did not land within the wait limit (the library's device
// status then says so); the CTA then waits once more for the copy before it
// may exit.
__device__ __forceinline__ bool stage_block(uint8_t* tile, uint64_t* bar, volatile int* abort,
                                            const void* src, int bytes, int* status) {
  using namespace sm100;
  const uint32_t b = smem_u32(bar);
  if (threadIdx.x == 0) {
    *abort = 0;
    mbar_init(b, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_expect_tx(b, (uint32_t)bytes);
    bulk_load(smem_u32(tile), src, (uint32_t)bytes, b);
  }
  const Abort ab{abort, status};
  if (mbar_wait(b, 0, ab)) return true;
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(b, 0) && globaltimer() - t0 < kWaitLimitNs) {
  }
  return false;
}

// One CTA per (b, h) and 128-row block of a bf16 [BH][N][128] tensor; grid
// (B*H, T, 3): z = 0 quantises Q, z = 1 K (the block's scale and its e4m3
// codes, same layout), z = 2 only records V's block maximum (V last, so
// that it is the most recent data in L2 when its codes are made).  The
// block is staged in shared memory by one bulk copy, then each thread takes
// eight 16-byte chunks (consecutive threads on consecutive chunks), once for
// the maximum and once for the codes.
__global__ void __launch_bounds__(256)
    quant_qk_amax_kernel(const __nv_bfloat16* __restrict__ q, const __nv_bfloat16* __restrict__ k,
                         const __nv_bfloat16* __restrict__ v, uint8_t* __restrict__ q8,
                         uint8_t* __restrict__ k8, float* __restrict__ qs,
                         float* __restrict__ ks, float* __restrict__ vamax, int N, int T,
                         int* status) {
  __shared__ __align__(128) uint8_t tile[128 * 256];
  __shared__ uint64_t bar;
  __shared__ int abort;
  __shared__ float red[8];
  const long long bh = blockIdx.x;
  const int t = blockIdx.y, z = blockIdx.z;
  const __nv_bfloat16* x = z == 0 ? q : (z == 1 ? k : v);
  const int rows = min(128, N - t * 128);
  const long long base = (bh * N + (long long)t * 128) * 128;  // element offset of the block
  const bool ok = stage_block(tile, &bar, &abort, x + base, rows * 256, status);
  auto chunk = [&](int i) {  // chunk i: row i / 16, columns 8 * (i % 16) ..
    return ok && (i >> 4) < rows ? reinterpret_cast<const uint4*>(tile)[i]
                                 : make_uint4(0u, 0u, 0u, 0u);
  };
  float m = 0.f;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const uint4 w = chunk(threadIdx.x + 256 * u);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h[e]);
      m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
  const float amax = block_max(m, red);
  if (z == 2) {
    if (threadIdx.x == 0) vamax[bh * T + t] = amax;
    return;
  }
  const float sc = amax > 0.f ? __fdiv_rn(amax, kE4m3Max) : 1.f;
  if (threadIdx.x == 0) (z == 0 ? qs : ks)[bh * T + t] = sc;
  uint8_t* codes = z == 0 ? q8 : k8;
  const bool by_rcp = sc >= 0x1p-126f;  // (a block of tiny values divides)
  const float rc = __frcp_rn(sc);
  auto quot = [&](float f) { return by_rcp ? div_by_scale(f, sc, rc) : __fdiv_rn(f, sc); };
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int i = threadIdx.x + 256 * u;
    if ((i >> 4) >= rows) continue;
    const uint4 w = chunk(i);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
    uint32_t word[2] = {0u, 0u};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h[e]);
      const uint32_t pair = (uint32_t)to_e4m3(quot(f.x)) | ((uint32_t)to_e4m3(quot(f.y)) << 8);
      word[e >> 1] |= pair << (16 * (e & 1));
    }
    *reinterpret_cast<uint2*>(codes + base + (long long)i * 8) = make_uint2(word[0], word[1]);
  }
}

// V codes, transposed: one CTA per 128-key block of one (b, h).  The head's
// scale is the largest of its block maxima over 448.  The block's
// [128 keys][128] bf16 is staged in shared memory by one bulk copy; each
// thread then converts 16 consecutive keys of one column (a warp: 32
// adjacent columns of one key at a time, 64 contiguous bytes, so the column
// reads are conflict-free) and stores them as one 16-byte chunk of Vt
// [BH][128][Np] (keys past N as zero codes).
__global__ void __launch_bounds__(256)
    quant_vt_kernel(const __nv_bfloat16* __restrict__ v, const float* __restrict__ amax,
                    uint8_t* __restrict__ vt, float* __restrict__ vscale, int N, int T, int Np,
                    int* status) {
  __shared__ __align__(128) uint8_t tile[128 * 256];
  __shared__ uint64_t bar;
  __shared__ int abort;
  __shared__ float red[8];
  const long long bh = blockIdx.x;
  const int t = blockIdx.y;
  const int rows = min(128, N - t * 128);
  const bool ok = stage_block(tile, &bar, &abort, v + (bh * N + (long long)t * 128) * 128,
                              rows * 256, status);
  float m = 0.f;
  for (int i = threadIdx.x; i < T; i += blockDim.x) m = fmaxf(m, amax[bh * T + i]);
  m = block_max(m, red);
  const float sc = m > 0.f ? __fdiv_rn(m, kE4m3Max) : 1.f;
  if (t == 0 && threadIdx.x == 0) vscale[bh] = sc;
  const bool by_rcp = sc >= 0x1p-126f;
  const float rc = __frcp_rn(sc);
  uint8_t* dst = vt + bh * 128 * (long long)Np + (long long)t * 128;
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    const int id = threadIdx.x + 256 * u, col = id & 127, k0 = (id >> 7) * 16;
    uint32_t word[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      uint32_t acc = 0u;
#pragma unroll
      for (int b = 0; b < 4; ++b) {
        const int key = k0 + 4 * e + b;
        if (ok && key < rows) {
          const float f = __bfloat162float(
              *reinterpret_cast<const __nv_bfloat16*>(tile + key * 256 + col * 2));
          const float qv = by_rcp ? div_by_scale(f, sc, rc) : __fdiv_rn(f, sc);
          acc |= (uint32_t)to_e4m3(qv) << (8 * b);
        }
      }
      word[e] = acc;
    }
    *reinterpret_cast<uint4*>(dst + (long long)col * Np + k0) =
        make_uint4(word[0], word[1], word[2], word[3]);
  }
}

struct Layout {
  size_t q8, k8, vt8, qs, ks, vs, amax, total;
};

static size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static Layout layout(long long bh, int N) {
  const int T = (N + 127) / 128;
  const long long Np = (long long)T * 128;
  Layout L;
  size_t off = 0;
  L.q8 = off;
  off += round_up((size_t)bh * N * 128, 256);
  L.k8 = off;
  off += round_up((size_t)bh * N * 128, 256);
  L.vt8 = off;
  off += round_up((size_t)bh * 128 * Np, 256);
  L.qs = off;
  off += round_up((size_t)bh * T * 4, 256);
  L.ks = off;
  off += round_up((size_t)bh * T * 4, 256);
  L.vs = off;
  off += round_up((size_t)bh * 4, 256);
  L.amax = off;
  off += round_up((size_t)bh * T * 4, 256);
  L.total = off;
  return L;
}

static bool aligned(const void* ptr, size_t a) {
  return (reinterpret_cast<uintptr_t>(ptr) % a) == 0;
}

static int check(int B, int H, int N, int d, float scale) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (d != 128) return FA_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  const long long bh = (long long)B * H;
  if (bh > 2147483647LL) return FA_ERR_INVALID_ARG;
  if ((N + 127) / 128 > 65535) return FA_ERR_INVALID_ARG;  // grid.y: 128-row blocks
  if (bh * ((N + 127) / 128) > 2147483647LL) return FA_ERR_INVALID_ARG;
  if ((double)bh * N * d > 4.0e18) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

}  // namespace fp8
}  // namespace fa

using namespace fa;
using namespace fa::fp8;

extern "C" {

size_t fa_fp8_workspace_bytes(int B, int H, int N, int d) {
  if (check(B, H, N, d, 1.f) != FA_OK) return 0;
  return layout((long long)B * H, N).total;
}

int fa_fp8_quantize(const void* q, const void* k, const void* v, int B, int H, int N, int d,
                    void* workspace, size_t workspace_bytes, void* stream) {
  int st = check(B, H, N, d, 1.f);
  if (st != FA_OK) return st;
  if (!q || !k || !v || !aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16))
    return FA_ERR_INVALID_ARG;
  const long long bh = (long long)B * H;
  const Layout L = layout(bh, N);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < L.total)
    return FA_ERR_INVALID_ARG;
  char* ws = static_cast<char*>(workspace);
  const int T = (N + 127) / 128;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* st_word = status_word();
  if (st_word == nullptr) return FA_ERR_CUDA;
  quant_qk_amax_kernel<<<dim3((unsigned)bh, (unsigned)T, 3), 256, 0, s>>>(
      static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
      static_cast<const __nv_bfloat16*>(v), reinterpret_cast<uint8_t*>(ws + L.q8),
      reinterpret_cast<uint8_t*>(ws + L.k8), reinterpret_cast<float*>(ws + L.qs),
      reinterpret_cast<float*>(ws + L.ks), reinterpret_cast<float*>(ws + L.amax), N, T, st_word);
  dim3 grid((unsigned)bh, (unsigned)T);
  quant_vt_kernel<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(v),
                                       reinterpret_cast<const float*>(ws + L.amax),
                                       reinterpret_cast<uint8_t*>(ws + L.vt8),
                                       reinterpret_cast<float*>(ws + L.vs), N, T, T * 128,
                                       st_word);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_forward_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                   int H, int N, int d, float scale, int causal, void* workspace,
                   size_t workspace_bytes, void* stream) {
  int st = check(B, H, N, d, scale);
  if (st != FA_OK) return st;
  if (!o || !lse || !aligned(o, 16) || !aligned(lse, 4)) return FA_ERR_INVALID_ARG;
  st = fa_fp8_quantize(q, k, v, B, H, N, d, workspace, workspace_bytes, stream);
  if (st != FA_OK) return st;
  return fa_forward_fp8_quantized(workspace, o, lse, B, H, N, d, scale, causal, stream);
}

int fa_forward_fp8_quantized(const void* workspace, void* o, float* lse, int B, int H, int N,
                             int d, float scale, int causal, void* stream) {
  int st = check(B, H, N, d, scale);
  if (st != FA_OK) return st;
  if (!workspace || !aligned(workspace, 256) || !o || !lse || !aligned(o, 16) ||
      !aligned(lse, 4))
    return FA_ERR_INVALID_ARG;
  const long long bh = (long long)B * H;
  const Layout L = layout(bh, N);
  const char* ws = static_cast<const char*>(workspace);
  Problem p = {};
  p.B = B;
  p.H = H;
  p.N = N;
  p.d = d;
  p.T = (N + 127) / 128;
  p.scale = scale;
  p.scale_log2 = scale * kLog2e;
  p.causal = causal ? 1 : 0;
  p.wl = p.wr = -1;
  p.drop_scale = 1.f;
  p.status = status_word();
  if (p.status == nullptr) return FA_ERR_CUDA;
  cudaError_t e = launch_fwd_fp8(p, ws + L.q8, ws + L.k8, ws + L.vt8,
                                 reinterpret_cast<const float*>(ws + L.qs),
                                 reinterpret_cast<const float*>(ws + L.ks),
                                 reinterpret_cast<const float*>(ws + L.vs), o, lse,
                                 static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // extern "C"
