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

// One CTA per (b, h) and 128-row block (grid (B*H, T)) of a bf16 [BH][N][d]
// tensor: the
// block's scale and its e4m3 codes (same layout).  d = 128: 16 bf16 per
// thread-row chunk; 256 threads walk the 128 x 128 block twice (max, codes).
__global__ void __launch_bounds__(256)
    quant_rows_kernel(const __nv_bfloat16* __restrict__ x, uint8_t* __restrict__ codes,
                      float* __restrict__ scales, int N, int T) {
  __shared__ float red[8];
  const long long bh = blockIdx.x;
  const int t = blockIdx.y;
  const int rows = min(128, N - t * 128);
  const long long base = (bh * N + (long long)t * 128) * 128;  // element offset of the block
  const int n8 = rows * 16;  // 8-element chunks in the block
  float m = 0.f;
  for (int i = threadIdx.x; i < n8; i += blockDim.x) {
    const uint4 w = *reinterpret_cast<const uint4*>(x + base + (long long)i * 8);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h[e]);
      m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
  const float amax = block_max(m, red);
  const float s = amax > 0.f ? __fdiv_rn(amax, kE4m3Max) : 1.f;
  if (threadIdx.x == 0) scales[bh * T + t] = s;
  for (int i = threadIdx.x; i < n8; i += blockDim.x) {
    const uint4 w = *reinterpret_cast<const uint4*>(x + base + (long long)i * 8);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h[e]);
      const uint32_t pair = (uint32_t)to_e4m3(__fdiv_rn(f.x, s)) |
                            ((uint32_t)to_e4m3(__fdiv_rn(f.y, s)) << 8);
      if (e < 2)
        lo |= pair << (16 * e);
      else
        hi |= pair << (16 * (e - 2));
    }
    *reinterpret_cast<uint2*>(codes + base + (long long)i * 8) = make_uint2(lo, hi);
  }
}

// Largest |v| of each 128-row block of V (one CTA per block).
__global__ void __launch_bounds__(256)
    amax_rows_kernel(const __nv_bfloat16* __restrict__ x, float* __restrict__ amax, int N,
                     int T) {
  __shared__ float red[8];
  const long long bh = blockIdx.x;
  const int t = blockIdx.y;
  const int rows = min(128, N - t * 128);
  const long long base = (bh * N + (long long)t * 128) * 128;
  float m = 0.f;
  for (int i = threadIdx.x; i < rows * 16; i += blockDim.x) {
    const uint4 w = *reinterpret_cast<const uint4*>(x + base + (long long)i * 8);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h[e]);
      m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
    }
  }
  m = block_max(m, red);
  if (threadIdx.x == 0) amax[bh * T + t] = m;
}

// V codes, transposed: one CTA per 128-key block of one (b, h) reads the
// [128 keys][128] bf16 block in 16-byte chunks (8 values of one key),
// scales by the head's scale (max over the head's block maxima), writes the
// codes transposed into a padded shared tile, and stores [128][128 keys]
// e4m3 rows of Vt [BH][128][Np] in 16-byte chunks (keys past N as zero codes).
__global__ void __launch_bounds__(256)
    quant_vt_kernel(const __nv_bfloat16* __restrict__ v, const float* __restrict__ amax,
                    uint8_t* __restrict__ vt, float* __restrict__ vscale, int N, int T, int Np) {
  constexpr int LD = 128 + 16;  // row pitch of the transposed tile (bytes)
  __shared__ __align__(16) uint8_t tile[128 * LD];
  __shared__ float red[8];
  const long long bh = blockIdx.x;
  const int t = blockIdx.y;
  float m = 0.f;
  for (int i = threadIdx.x; i < T; i += blockDim.x) m = fmaxf(m, amax[bh * T + i]);
  m = block_max(m, red);
  const float s = m > 0.f ? __fdiv_rn(m, kE4m3Max) : 1.f;
  if (t == 0 && threadIdx.x == 0) vscale[bh] = s;
  const int rows = min(128, N - t * 128);
  const __nv_bfloat16* src = v + (bh * N + (long long)t * 128) * 128;
  // 2048 chunks: chunk c = key (c / 16), columns 8 * (c % 16) .. +7
  for (int c = threadIdx.x; c < 2048; c += blockDim.x) {
    const int key = c >> 4, col0 = (c & 15) * 8;
    uint4 w = make_uint4(0, 0, 0, 0);
    if (key < rows) w = *reinterpret_cast<const uint4*>(src + key * 128 + col0);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(h[e]);
      tile[(col0 + 2 * e) * LD + key] = key < rows ? to_e4m3(__fdiv_rn(f.x, s)) : 0;
      tile[(col0 + 2 * e + 1) * LD + key] = key < rows ? to_e4m3(__fdiv_rn(f.y, s)) : 0;
    }
  }
  __syncthreads();
  // 1024 chunks of 16 codes: chunk c = column (c / 8), keys 16 * (c % 8) .. +15
  uint8_t* dst = vt + bh * 128 * (long long)Np + (long long)t * 128;
  for (int c = threadIdx.x; c < 1024; c += blockDim.x) {
    const int col = c >> 3, k0 = (c & 7) * 16;
    *reinterpret_cast<uint4*>(dst + (long long)col * Np + k0) =
        *reinterpret_cast<const uint4*>(&tile[col * LD + k0]);
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
  dim3 grid((unsigned)bh, (unsigned)T);
  quant_rows_kernel<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(q),
                                         reinterpret_cast<uint8_t*>(ws + L.q8),
                                         reinterpret_cast<float*>(ws + L.qs), N, T);
  quant_rows_kernel<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(k),
                                         reinterpret_cast<uint8_t*>(ws + L.k8),
                                         reinterpret_cast<float*>(ws + L.ks), N, T);
  amax_rows_kernel<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(v),
                                        reinterpret_cast<float*>(ws + L.amax), N, T);
  quant_vt_kernel<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(v),
                                       reinterpret_cast<const float*>(ws + L.amax),
                                       reinterpret_cast<uint8_t*>(ws + L.vt8),
                                       reinterpret_cast<float*>(ws + L.vs), N, T, T * 128);
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
