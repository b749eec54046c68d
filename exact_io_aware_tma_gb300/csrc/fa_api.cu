// C ABI of the attention library: host-side validation, the small
// memory-bound kernels (backward preprocess, dQ conversion, tile schedule)
// and the launches of the tiled kernels, all asynchronous on the caller's
// stream.  See include/fa.h for the contract of each entry point.
#include <cmath>
#include <cstdint>

#include "../../include/fa.h"
#include "../../include/fa_selftest.h"
#include "fa_common.cuh"
#include "fa_kernels.h"

namespace fa {

// Device error word: kernels with bounded waits record FA_ERR_TIMEOUT here.
__device__ int g_fa_status = 0;

// ---------------------------------------------------------------------------
// Backward preprocess.  Per query row (padded per head to a multiple of 128
// rows): D_i = sum_c dO_ic * O_ic and L_i = LSE_i * log2(e), written as +inf
// for rows without an allowed key and for padding rows (so every
// probability the backward rebuilds for them is 2^-inf = 0), D = 0 there;
// also clears the fp32 dQ accumulator.  One thread per 16-byte chunk (8 bf16)
// of a row; the CH chunks of a row are adjacent lanes and reduce by shuffles.
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(256)
    bwd_preprocess_kernel(const __nv_bfloat16* __restrict__ o,
                          const __nv_bfloat16* __restrict__ dout, const float* __restrict__ lse,
                          float* __restrict__ lse2, float* __restrict__ dvec,
                          float* __restrict__ dq_acc, unsigned long long* __restrict__ next_item,
                          long long heads, int N, int npad) {
  constexpr int CH = D / 8;
  const long long n = heads * npad * CH;
  griddep_wait();
  griddep_release();
  if (blockIdx.x == 0 && threadIdx.x == 0) *next_item = 0;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i - (threadIdx.x & 31) < n;
       i += (long long)gridDim.x * blockDim.x) {
    float acc = 0.f;
    const bool in = i < n;
    const long long prow = i / CH;  // padded row index
    const long long bh = prow / npad;
    const int row = (int)(prow % npad);
    const bool live = in && row < N;
    if (live) {
      const long long e = ((bh * N + row) * CH + (i % CH)) * 8;
      uint4 a = *reinterpret_cast<const uint4*>(o + e);
      uint4 b = *reinterpret_cast<const uint4*>(dout + e);
      const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float2 x = __bfloat1622float2(pa[j]);
        float2 y = __bfloat1622float2(pb[j]);
        acc = fmaf(x.x, y.x, acc);
        acc = fmaf(x.y, y.y, acc);
      }
      float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
      reinterpret_cast<float4*>(dq_acc + e)[0] = z;
      reinterpret_cast<float4*>(dq_acc + e)[1] = z;
    }
#pragma unroll
    for (int off = CH / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (in && (i % CH) == 0) {
      dvec[prow] = live ? acc : 0.f;
      const float l = live ? lse[bh * N + row] : -INFINITY;
      lse2[prow] = l == -INFINITY ? INFINITY : l * kLog2e;
    }
  }
}

// The same preprocess for the packed variable-length layout: row `row` of
// (b, h) is token cu_seqlens[b] + row of [total][H][d] (rows at or past the
// sequence's length are padding); LSE is [H][total].  The fp32 dQ
// accumulator [H][total][d] is cleared in full, so tokens outside every
// sequence end with dQ = 0.
template <int D>
__global__ void __launch_bounds__(256)
    bwd_preprocess_packed_kernel(const __nv_bfloat16* __restrict__ o,
                                 const __nv_bfloat16* __restrict__ dout,
                                 const float* __restrict__ lse, float* __restrict__ lse2,
                                 float* __restrict__ dvec, float* __restrict__ dq_acc,
                                 const int32_t* __restrict__ cu, int H, long long heads, int total,
                                 int maxlen, int npad) {
  constexpr int CH = D / 8;
  const long long n = heads * npad * CH;
  const long long stride = (long long)gridDim.x * blockDim.x;
  griddep_wait();
  griddep_release();
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i - (threadIdx.x & 31) < n;
       i += stride) {
    float acc = 0.f;
    const bool in = i < n;
    const long long prow = i / CH;  // padded row index
    const long long bh = prow / npad;
    const int row = (int)(prow % npad);
    int start = 0, len = 0;
    if (in) {
      const int b = (int)(bh / H);
      int s0 = __ldg(cu + b), e0 = __ldg(cu + b + 1);
      s0 = min(max(s0, 0), total);
      e0 = min(max(e0, s0), total);
      start = s0;
      len = min(e0 - s0, maxlen);
    }
    const int h = (int)(bh % H);
    const bool live = in && row < len;
    if (live) {
      const long long e = (((long long)(start + row) * H + h) * CH + (i % CH)) * 8;
      uint4 a = *reinterpret_cast<const uint4*>(o + e);
      uint4 b4 = *reinterpret_cast<const uint4*>(dout + e);
      const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&a);
      const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&b4);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        float2 x = __bfloat1622float2(pa[j]);
        float2 y = __bfloat1622float2(pb[j]);
        acc = fmaf(x.x, y.x, acc);
        acc = fmaf(x.y, y.y, acc);
      }
    }
#pragma unroll
    for (int off = CH / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (in && (i % CH) == 0) {
      dvec[prow] = live ? acc : 0.f;
      const float l = live ? lse[(long long)h * total + start + row] : -INFINITY;
      lse2[prow] = l == -INFINITY ? INFINITY : l * kLog2e;
    }
  }
  const long long nz = (long long)total * H * D / 4;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < nz; i += stride)
    reinterpret_cast<float4*>(dq_acc)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// Packed layout: dQ [total][H][d] = scale * dQacc [H][total][d], fp32 ->
// bf16, 8 elements per thread (consecutive threads: consecutive chunks of
// one token's heads, so the bf16 writes are contiguous).
__global__ void __launch_bounds__(256)
    dq_convert_packed_kernel(const float* __restrict__ dq_acc, __nv_bfloat16* __restrict__ dq,
                             float scale, int H, int total, int d) {
  const long long chunks = (long long)total * H * (d / 8);
  griddep_wait();
  griddep_release();
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < chunks;
       i += (long long)gridDim.x * blockDim.x) {
    const long long e = i * 8;  // element of dq [total][H][d]
    const int c = (int)(e % d);
    const long long th = e / d;
    const int h = (int)(th % H);
    const long long t = th / H;
    const float* src = dq_acc + ((long long)h * total + t) * d + c;
    const float4 a = reinterpret_cast<const float4*>(src)[0];
    const float4 b = reinterpret_cast<const float4*>(src)[1];
    uint4 r;
    r.x = pack_bf16(a.x * scale, a.y * scale);
    r.y = pack_bf16(a.z * scale, a.w * scale);
    r.z = pack_bf16(b.x * scale, b.y * scale);
    r.w = pack_bf16(b.z * scale, b.w * scale);
    *reinterpret_cast<uint4*>(dq + e) = r;
  }
}

// dQ = scale * dQacc, fp32 -> bf16, 8 elements per thread.
__global__ void __launch_bounds__(256)
    dq_convert_kernel(const float* __restrict__ dq_acc, __nv_bfloat16* __restrict__ dq,
                      float scale, long long chunks) {
  griddep_wait();
  griddep_release();
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < chunks;
       i += (long long)gridDim.x * blockDim.x) {
    float4 a = reinterpret_cast<const float4*>(dq_acc + i * 8)[0];
    float4 b = reinterpret_cast<const float4*>(dq_acc + i * 8)[1];
    uint4 r;
    r.x = pack_bf16(a.x * scale, a.y * scale);
    r.y = pack_bf16(a.z * scale, a.w * scale);
    r.z = pack_bf16(b.x * scale, b.y * scale);
    r.w = pack_bf16(b.z * scale, b.w * scale);
    *reinterpret_cast<uint4*>(dq + i * 8) = r;
  }
}

// Tile schedule of one batch element (one CTA): CSR over query tiles of the
// live key tiles, with the element-mask flag.  Uses the same predicates as
// the attention kernels.
__global__ void __launch_bounds__(1024)
    tile_schedule_kernel(Problem p, int b, int32_t* row_ptr, int32_t* col_idx,
                         uint8_t* partial) {
  __shared__ int s_cnt[1024];
  __shared__ int s_carry;
  const int klim = key_limit(p, b);
  if (threadIdx.x == 0) {
    s_carry = 0;
    row_ptr[0] = 0;
  }
  __syncthreads();
  for (int base = 0; base < p.T; base += blockDim.x) {
    const int qt = base + threadIdx.x;
    int c = 0;
    if (qt < p.T)
      for (int kt = 0; kt < p.T; ++kt) c += tile_live(p, qt, kt, klim) ? 1 : 0;
    s_cnt[threadIdx.x] = c;
    __syncthreads();
    // inclusive scan (Hillis-Steele)
    for (int off = 1; off < (int)blockDim.x; off <<= 1) {
      int x = threadIdx.x >= (unsigned)off ? s_cnt[threadIdx.x - off] : 0;
      __syncthreads();
      s_cnt[threadIdx.x] += x;
      __syncthreads();
    }
    const int carry = s_carry;
    if (qt < p.T) {
      int pos = carry + s_cnt[threadIdx.x] - c;
      row_ptr[qt + 1] = carry + s_cnt[threadIdx.x];
      for (int kt = 0; kt < p.T; ++kt) {
        if (tile_live(p, qt, kt, klim)) {
          col_idx[pos] = kt;
          partial[pos] = tile_partial(p, qt, kt, klim) ? 1 : 0;
          ++pos;
        }
      }
    }
    __syncthreads();
    if (threadIdx.x == blockDim.x - 1) s_carry = carry + s_cnt[threadIdx.x];
    __syncthreads();
  }
}

int* status_word() {
  int* ptr = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_fa_status) != cudaSuccess)
    return nullptr;
  return ptr;
}

static bool aligned(const void* ptr, size_t a) {
  return (reinterpret_cast<uintptr_t>(ptr) % a) == 0;
}

// Shared size checks.  Fills `p` on success.  Window sides of N or more
// allow every key on that side and are stored as unbounded (-1), which also
// keeps i + wr within int range.  A scale whose scale*log2(e) is zero or
// subnormal is held at +-1e-30 in log2 units: the scores it produces are
// still 0 to within fp32 rounding (uniform attention), while a masked score
// (+-inf) still maps to -inf, where 0 * inf would give NaN.
static int check_sizes(int B, int H, int N, int d, float scale, const fa_mask* m, Problem* p) {
  if (B < 1 || H < 1 || N < 1) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  const long long bh = (long long)B * H;
  if (bh > 2147483647LL) return FA_ERR_INVALID_ARG;
  const long long T = ((long long)N + kTile - 1) / kTile;
  if (T > 65535) return FA_ERR_INVALID_ARG;  // N <= 8,388,480
  if (bh * T > 2147483647LL) return FA_ERR_INVALID_ARG;  // one CTA per (head, tile)
  // B*H*N*d elements must stay far from int64 overflow
  if ((double)bh * N * d > 4.0e18) return FA_ERR_INVALID_ARG;
  p->B = B;
  p->H = H;
  p->N = N;
  p->d = d;
  p->T = (int)T;
  p->scale = scale;
  float sl = scale * kLog2e;
  if (std::fabs(sl) < 1e-30f) sl = sl < 0.f ? -1e-30f : 1e-30f;
  p->scale_log2 = sl;
  p->causal = (m != nullptr && m->causal) ? 1 : 0;
  p->wl = (m != nullptr && m->window_left >= 0 && m->window_left < N) ? m->window_left : -1;
  p->wr = (m != nullptr && m->window_right >= 0 && m->window_right < N) ? m->window_right : -1;
  p->block_mask = m != nullptr ? m->block_mask : nullptr;
  p->kv_len = m != nullptr ? m->kv_len : nullptr;
  p->status = nullptr;
  p->cu_seqlens = nullptr;
  p->total = 0;
  p->drop_p8 = 0;
  p->seed_lo = p->seed_hi = p->drop_offset = 0;
  p->drop_scale = 1.f;
  if (m != nullptr && m->dropout_p != 0.f) {
    // dropout probability in steps of 1/256, below 1
    if (!(m->dropout_p > 0.f && m->dropout_p < 1.f)) return FA_ERR_INVALID_ARG;
    int p8 = (int)std::lround((double)m->dropout_p * 256.0);
    p8 = p8 > 255 ? 255 : p8;
    p->drop_p8 = (uint32_t)p8;
    p->seed_lo = (uint32_t)(m->dropout_seed & 0xffffffffull);
    p->seed_hi = (uint32_t)(m->dropout_seed >> 32);
    p->drop_offset = m->dropout_offset;
    p->drop_scale = (float)(1.0 / (1.0 - p8 / 256.0));
  }
  return FA_OK;
}

static fa_mask plain_mask(int causal, const uint8_t* block_mask, const int32_t* kv_len) {
  fa_mask m = {};
  m.causal = causal;
  m.window_left = -1;
  m.window_right = -1;
  m.block_mask = block_mask;
  m.kv_len = kv_len;
  return m;
}

static size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
static int padded_rows(int N) { return (N + kTile - 1) / kTile * kTile; }

}  // namespace fa

using namespace fa;

extern "C" {

const char* fa_status_string(int s) {
  switch (s) {
    case FA_OK: return "FA_OK";
    case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
    case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
    case FA_ERR_CUDA: return "FA_ERR_CUDA";
    case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
    default: return "FA_ERR_UNKNOWN";
  }
}

int fa_forward_masked(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                      int H, int N, int d, float scale, const fa_mask* mask, void* stream) {
  Problem p;
  int st = check_sizes(B, H, N, d, scale, mask, &p);
  if (st != FA_OK) return st;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(lse, 4) || !aligned(p.kv_len, 4))
    return FA_ERR_INVALID_ARG;
  p.status = status_word();
  if (p.status == nullptr) return FA_ERR_CUDA;
  cudaError_t e = launch_fwd_tc(p, q, k, v, o, lse, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_forward(const void* q, const void* k, const void* v, void* o, float* lse, int B,
               int H, int N, int d, float scale, int causal, const uint8_t* block_mask,
               const int32_t* kv_len, void* stream) {
  const fa_mask m = plain_mask(causal, block_mask, kv_len);
  return fa_forward_masked(q, k, v, o, lse, B, H, N, d, scale, &m, stream);
}

size_t fa_backward_workspace_bytes(int B, int H, int N, int d) {
  Problem p;
  if (check_sizes(B, H, N, d, 1.0f, nullptr, &p) != FA_OK) return 0;
  const size_t vec = round_up((size_t)B * H * padded_rows(N) * sizeof(float), 256);
  // LSE*log2(e), D, the fp32 dQ accumulator, the dK/dV kernel's work counter
  return 2 * vec + round_up((size_t)B * H * N * d * sizeof(float), 256) + 256;
}

// Extra workspace of the split backward (block masks): the plan's items and
// split list (256 bytes) and the fp32 slots; 0 where it does not apply.
static size_t split_bytes(const Problem& p) {
  const long long heads = (long long)p.B * p.H;
  if (p.block_mask == nullptr || p.T > kPlanMaxTiles ||
      heads * p.T * kSplitMax > 2147483647LL)
    return 0;
  return round_up((size_t)p.T * kSplitMax * sizeof(int4), 256) + 256 +
         (size_t)heads * kSplitSlots * 2 * 128 * p.d * sizeof(float);
}

size_t fa_backward_workspace_bytes_masked(int B, int H, int N, int d, const fa_mask* mask) {
  Problem p;
  if (check_sizes(B, H, N, d, 1.0f, mask, &p) != FA_OK) return 0;
  return fa_backward_workspace_bytes(B, H, N, d) + split_bytes(p);
}

static int check_workspace(int B, int H, int N, int d, const void* ws, size_t wsb) {
  if (!ws || !aligned(ws, 256)) return FA_ERR_INVALID_ARG;
  if (wsb < fa_backward_workspace_bytes(B, H, N, d)) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

// Workspace: L = LSE*log2(e) [B*H][Np], D [B*H][Np] (Np = N rounded up to
// 128), then the fp32 dQ accumulator [B*H][N][d].
static size_t ws_vec_bytes(long long heads, int N) {
  return round_up((size_t)heads * padded_rows(N) * sizeof(float), 256);
}
static float* ws_lse2(void* ws) { return static_cast<float*>(ws); }
static float* ws_dvec(void* ws, long long heads, int N) {
  return reinterpret_cast<float*>(static_cast<char*>(ws) + ws_vec_bytes(heads, N));
}
static float* ws_dq_acc(void* ws, long long heads, int N) {
  return reinterpret_cast<float*>(static_cast<char*>(ws) + 2 * ws_vec_bytes(heads, N));
}
// work-item counter of the persistent dK/dV kernel (cleared by the preprocess)
static unsigned long long* ws_counter(void* ws, long long heads, int N, int d) {
  return reinterpret_cast<unsigned long long*>(
      static_cast<char*>(ws) + 2 * ws_vec_bytes(heads, N) +
      round_up((size_t)heads * N * d * sizeof(float), 256));
}

// Elementwise kernels: enough CTAs for every chunk, capped at a few waves.
static unsigned elementwise_blocks(long long chunks) {
  long long nblk = (chunks + 255) / 256;
  if (nblk > 152LL * 32) nblk = 152LL * 32;
  return (unsigned)(nblk < 1 ? 1 : nblk);
}

int fa_backward_preprocess(const void* o, const void* dout, const float* lse, int B, int H,
                           int N, int d, void* workspace, size_t workspace_bytes, void* stream) {
  Problem p;
  int st = check_sizes(B, H, N, d, 1.0f, nullptr, &p);
  if (st != FA_OK) return st;
  if (!o || !dout || !lse || !aligned(o, 16) || !aligned(dout, 16) || !aligned(lse, 4))
    return FA_ERR_INVALID_ARG;
  st = check_workspace(B, H, N, d, workspace, workspace_bytes);
  if (st != FA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const long long heads = (long long)B * H;
  const int npad = padded_rows(N);
  const unsigned nblk = elementwise_blocks(heads * npad * (d / 8));
  auto ob = static_cast<const __nv_bfloat16*>(o);
  auto db = static_cast<const __nv_bfloat16*>(dout);
  const cudaError_t e = launch_k(
      true, d == 64 ? bwd_preprocess_kernel<64> : bwd_preprocess_kernel<128>, dim3(nblk),
      dim3(256), 0, s, ob, db, lse, ws_lse2(workspace), ws_dvec(workspace, heads, N),
      ws_dq_acc(workspace, heads, N), ws_counter(workspace, heads, N, d), heads, N, npad);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

// The dK/dV call's problem and, with a block mask and room for the split's
// extra workspace, its split (key tiles with many live query tiles spread
// over several CTAs).
static int dkdv_problem(const void* q, const void* k, const void* v, const void* dout,
                        const void* dk, const void* dv, int B, int H, int N, int d, float scale,
                        const fa_mask* mask, void* workspace, size_t workspace_bytes,
                        Problem* p, BwdSplit* split, bool* use_split) {
  int st = check_sizes(B, H, N, d, scale, mask, p);
  if (st != FA_OK) return st;
  if (!q || !k || !v || !dout || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(dout, 16) ||
      !aligned(dk, 16) || !aligned(dv, 16) || !aligned(p->kv_len, 4))
    return FA_ERR_INVALID_ARG;
  st = check_workspace(B, H, N, d, workspace, workspace_bytes);
  if (st != FA_OK) return st;
  p->status = status_word();
  if (p->status == nullptr) return FA_ERR_CUDA;
  *split = BwdSplit{};
  const size_t base = fa_backward_workspace_bytes(B, H, N, d), extra = split_bytes(*p);
  *use_split = extra != 0 && workspace_bytes >= base + extra;
  if (*use_split) {
    char* w = static_cast<char*>(workspace) + base;
    split->items = reinterpret_cast<const int4*>(w);
    w += round_up((size_t)p->T * kSplitMax * sizeof(int4), 256);
    split->nitems = reinterpret_cast<const int*>(w);
    w += 256;
    split->slots = reinterpret_cast<float*>(w);
  }
  return FA_OK;
}

// early: called straight after the preprocess's launch, with the split's
// plan (if any) launched before that preprocess.
static int backward_dkdv(const void* q, const void* k, const void* v, const void* dout, void* dk,
                         void* dv, int B, int H, int N, int d, float scale, const fa_mask* mask,
                         void* workspace, size_t workspace_bytes, void* stream, bool early) {
  Problem p;
  BwdSplit split;
  bool use_split;
  int st = dkdv_problem(q, k, v, dout, dk, dv, B, H, N, d, scale, mask, workspace,
                        workspace_bytes, &p, &split, &use_split);
  if (st != FA_OK) return st;
  const long long heads = (long long)B * H;
  cudaError_t e = launch_bwd_tc(p, q, k, v, dout, ws_lse2(workspace),
                                ws_dvec(workspace, heads, N), ws_dq_acc(workspace, heads, N),
                                dk, dv, padded_rows(N), use_split ? &split : nullptr,
                                ws_counter(workspace, heads, N, d), early,
                                static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_backward_dkdv(const void* q, const void* k, const void* v, const void* dout, void* dk,
                     void* dv, int B, int H, int N, int d, float scale, int causal,
                     const uint8_t* block_mask, const int32_t* kv_len, void* workspace,
                     size_t workspace_bytes, void* stream) {
  const fa_mask m = plain_mask(causal, block_mask, kv_len);
  return backward_dkdv(q, k, v, dout, dk, dv, B, H, N, d, scale, &m, workspace, workspace_bytes,
                       stream, false);
}

int fa_backward_dq_convert(void* dq, int B, int H, int N, int d, float scale,
                           const void* workspace, size_t workspace_bytes, void* stream) {
  Problem p;
  int st = check_sizes(B, H, N, d, scale, nullptr, &p);
  if (st != FA_OK) return st;
  if (!dq || !aligned(dq, 16)) return FA_ERR_INVALID_ARG;
  st = check_workspace(B, H, N, d, workspace, workspace_bytes);
  if (st != FA_OK) return st;
  const long long heads = (long long)B * H;
  const long long chunks = heads * N * (d / 8);
  const cudaError_t e =
      launch_k(true, dq_convert_kernel, dim3(elementwise_blocks(chunks)), dim3(256), 0,
               static_cast<cudaStream_t>(stream), ws_dq_acc(const_cast<void*>(workspace), heads, N),
               static_cast<__nv_bfloat16*>(dq), scale, chunks);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_backward_masked(const void* q, const void* k, const void* v, const void* o,
                       const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                       int H, int N, int d, float scale, const fa_mask* mask, void* workspace,
                       size_t workspace_bytes, void* stream) {
  Problem p;
  int st = check_sizes(B, H, N, d, scale, mask, &p);
  if (st != FA_OK) return st;
  // Validate every argument before the first launch, so a rejected call
  // writes nothing.
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
      !aligned(lse, 4) || !aligned(p.kv_len, 4))
    return FA_ERR_INVALID_ARG;
  st = check_workspace(B, H, N, d, workspace, workspace_bytes);
  if (st != FA_OK) return st;
  // The split's plan (block mask) goes first and the preprocess waits for
  // it, so the dK/dV kernel can start while the preprocess runs.
  {
    Problem pd;
    BwdSplit split;
    bool use_split;
    st = dkdv_problem(q, k, v, dout, dk, dv, B, H, N, d, scale, mask, workspace, workspace_bytes,
                      &pd, &split, &use_split);
    if (st != FA_OK) return st;
    if (use_split && launch_bwd_plan(pd, split, static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return FA_ERR_CUDA;
  }
  st = fa_backward_preprocess(o, dout, lse, B, H, N, d, workspace, workspace_bytes, stream);
  if (st != FA_OK) return st;
  st = backward_dkdv(q, k, v, dout, dk, dv, B, H, N, d, scale, mask, workspace, workspace_bytes,
                     stream, true);
  if (st != FA_OK) return st;
  return fa_backward_dq_convert(dq, B, H, N, d, scale, workspace, workspace_bytes, stream);
}

int fa_backward(const void* q, const void* k, const void* v, const void* o,
                const float* lse, const void* dout, void* dq, void* dk, void* dv, int B,
                int H, int N, int d, float scale, int causal, const uint8_t* block_mask,
                const int32_t* kv_len, void* workspace, size_t workspace_bytes,
                void* stream) {
  const fa_mask m = plain_mask(causal, block_mask, kv_len);
  return fa_backward_masked(q, k, v, o, lse, dout, dq, dk, dv, B, H, N, d, scale, &m, workspace,
                            workspace_bytes, stream);
}

int fa_tile_schedule_masked(int N, const fa_mask* mask, int b, int32_t* row_ptr,
                            int32_t* col_idx, uint8_t* partial, void* stream) {
  Problem p;
  int st = check_sizes(1, 1, N, 64, 1.0f, mask, &p);
  if (st != FA_OK) return st;
  if (!row_ptr || !col_idx || !partial || b < 0) return FA_ERR_INVALID_ARG;
  if (!aligned(row_ptr, 4) || !aligned(col_idx, 4) || !aligned(p.kv_len, 4))
    return FA_ERR_INVALID_ARG;
  tile_schedule_kernel<<<1, 1024, 0, static_cast<cudaStream_t>(stream)>>>(p, b, row_ptr,
                                                                          col_idx, partial);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_tile_schedule(int N, int causal, const uint8_t* block_mask, const int32_t* kv_len,
                     int b, int32_t* row_ptr, int32_t* col_idx, uint8_t* partial,
                     void* stream) {
  const fa_mask m = plain_mask(causal, block_mask, kv_len);
  return fa_tile_schedule_masked(N, &m, b, row_ptr, col_idx, partial, stream);
}

// ---------------------------------------------------------------- packed
// Variable-length sequences in the packed layout (include/fa.h): the grid is
// sized by max_seqlen and each CTA takes its own sequence's span.

static int check_varlen(int B, int H, int total, int max_seqlen, int d, float scale,
                        const fa_mask* mask, const int32_t* cu, Problem* p) {
  if (B < 1 || H < 1 || total < 1 || max_seqlen < 1) return FA_ERR_INVALID_ARG;
  if (mask != nullptr && (mask->block_mask != nullptr || mask->kv_len != nullptr))
    return FA_ERR_UNSUPPORTED;
  if (cu == nullptr || !aligned(cu, 4)) return FA_ERR_INVALID_ARG;
  if ((long long)B * H > 2147483647LL) return FA_ERR_INVALID_ARG;
  if ((double)total * H * d > 4.0e18) return FA_ERR_INVALID_ARG;
  int st = check_sizes(B, H, max_seqlen, d, scale, mask, p);
  if (st != FA_OK) return st;
  p->cu_seqlens = cu;
  p->total = total;
  return FA_OK;
}

size_t fa_varlen_workspace_bytes(int B, int H, int total, int max_seqlen, int d) {
  Problem p;
  int dummy = 0;
  if (check_varlen(B, H, total, max_seqlen, d, 1.0f, nullptr, &dummy, &p) != FA_OK) return 0;
  const size_t vec = round_up((size_t)B * H * padded_rows(max_seqlen) * sizeof(float), 256);
  return 2 * vec + round_up((size_t)total * H * d * sizeof(float), 256);
}

int fa_forward_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                      const int32_t* cu_seqlens, int B, int H, int total, int max_seqlen, int d,
                      float scale, const fa_mask* mask, void* stream) {
  Problem p;
  int st = check_varlen(B, H, total, max_seqlen, d, scale, mask, cu_seqlens, &p);
  if (st != FA_OK) return st;
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(lse, 4))
    return FA_ERR_INVALID_ARG;
  p.status = status_word();
  if (p.status == nullptr) return FA_ERR_CUDA;
  cudaError_t e = launch_fwd_tc(p, q, k, v, o, lse, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_backward_varlen(const void* q, const void* k, const void* v, const void* o,
                       const float* lse, const void* dout, void* dq, void* dk, void* dv,
                       const int32_t* cu_seqlens, int B, int H, int total, int max_seqlen, int d,
                       float scale, const fa_mask* mask, void* workspace,
                       size_t workspace_bytes, void* stream) {
  Problem p;
  int st = check_varlen(B, H, total, max_seqlen, d, scale, mask, cu_seqlens, &p);
  if (st != FA_OK) return st;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
      !aligned(lse, 4))
    return FA_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256) ||
      workspace_bytes < fa_varlen_workspace_bytes(B, H, total, max_seqlen, d))
    return FA_ERR_INVALID_ARG;
  p.status = status_word();
  if (p.status == nullptr) return FA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const long long heads = (long long)B * H;
  const int npad = padded_rows(max_seqlen);
  const size_t vec = round_up((size_t)heads * npad * sizeof(float), 256);
  float* lse2 = static_cast<float*>(workspace);
  float* dvec = reinterpret_cast<float*>(static_cast<char*>(workspace) + vec);
  float* dq_acc = reinterpret_cast<float*>(static_cast<char*>(workspace) + 2 * vec);
  const unsigned nblk = elementwise_blocks(heads * npad * (d / 8));
  auto ob = static_cast<const __nv_bfloat16*>(o);
  auto db = static_cast<const __nv_bfloat16*>(dout);
  cudaError_t e = launch_k(
      true, d == 64 ? bwd_preprocess_packed_kernel<64> : bwd_preprocess_packed_kernel<128>,
      dim3(nblk), dim3(256), 0, s, ob, db, lse, lse2, dvec, dq_acc, cu_seqlens, H, heads, total,
      max_seqlen, npad);
  if (e != cudaSuccess) return FA_ERR_CUDA;
  e = launch_bwd_tc(p, q, k, v, dout, lse2, dvec, dq_acc, dk, dv, npad, nullptr, nullptr, true,
                    s);
  if (e != cudaSuccess) return FA_ERR_CUDA;
  const long long chunks = (long long)total * H * (d / 8);
  e = launch_k(true, dq_convert_packed_kernel, dim3(elementwise_blocks(chunks)), dim3(256), 0, s,
               (const float*)dq_acc, static_cast<__nv_bfloat16*>(dq), scale, H, total, d);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_selftest_forward_lost_signal(const void* q, const void* k, const void* v, void* o,
                                    float* lse, int B, int H, int N, int d, float scale,
                                    int causal, void* stream) {
  const fa_mask m = plain_mask(causal, nullptr, nullptr);
  Problem p;
  int st = check_sizes(B, H, N, d, scale, &m, &p);
  if (st != FA_OK) return st;
  if (d != 128 && d != 64) return FA_ERR_UNSUPPORTED;
  if (!q || !k || !v || !o || !lse || !aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) ||
      !aligned(o, 16) || !aligned(lse, 4))
    return FA_ERR_INVALID_ARG;
  p.status = status_word();
  if (p.status == nullptr) return FA_ERR_CUDA;
  cudaError_t e = launch_fwd_tc_lost_signal(p, q, k, v, o, lse, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_selftest_backward_lost_signal(const void* q, const void* k, const void* v, const void* o,
                                     const float* lse, const void* dout, void* dq, void* dk,
                                     void* dv, int B, int H, int N, int d, float scale,
                                     int causal, void* workspace, size_t workspace_bytes,
                                     void* stream) {
  const fa_mask m = plain_mask(causal, nullptr, nullptr);
  Problem p;
  int st = check_sizes(B, H, N, d, scale, &m, &p);
  if (st != FA_OK) return st;
  if (d != 128 && d != 64) return FA_ERR_UNSUPPORTED;
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
      !aligned(lse, 4))
    return FA_ERR_INVALID_ARG;
  st = check_workspace(B, H, N, d, workspace, workspace_bytes);
  if (st != FA_OK) return st;
  p.status = status_word();
  if (p.status == nullptr) return FA_ERR_CUDA;
  st = fa_backward_preprocess(o, dout, lse, B, H, N, d, workspace, workspace_bytes, stream);
  if (st != FA_OK) return st;
  const long long heads = (long long)B * H;
  cudaError_t e = launch_bwd_tc_lost_signal(
      p, q, k, v, dout, ws_lse2(workspace), ws_dvec(workspace, heads, N),
      ws_dq_acc(workspace, heads, N), dk, dv, padded_rows(N), ws_counter(workspace, heads, N, d),
      static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return FA_ERR_CUDA;
  return fa_backward_dq_convert(dq, B, H, N, d, scale, workspace, workspace_bytes, stream);
}

int fa_last_device_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FA_ERR_CUDA;
  int h = 0;
  if (cudaMemcpyFromSymbol(&h, g_fa_status, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
  if (h != 0) {
    int z = 0;
    if (cudaMemcpyToSymbol(g_fa_status, &z, sizeof(int)) != cudaSuccess) return FA_ERR_CUDA;
  }
  return h;
}

}  // extern "C"
