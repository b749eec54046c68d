// Warp-level (mma.sync) tiled attention forward.
//
// One CTA owns 128 query rows of one (b, h); 8 warps own 16 rows each.  The
// CTA walks the live 128-key tiles of its query tile (block mask, causal
// rule and key limit; dead tiles are never loaded) in 64-key steps, with
// K/V double-buffered in shared memory by cp.async, and evaluates the
// online-softmax recurrence of page "FlashAttention" (aiwiki), section
// "Tiling and online normalization", in log2 units:
//     m' = max(m, max_j s_j),  l' = 2^(m-m') l + sum_j 2^(s_j-m'),
//     u' = 2^(m-m') u + sum_j 2^(s_j-m') v_j,      O = u / l,
// with s_j = scale * log2(e) * q.k_j.  O and LSE = ln2 * (m + log2 l) are
// written once.  The N x N score matrix never leaves registers.
#include "fa_common.cuh"
#include "fa_kernels.h"

namespace fa {

template <int D>
struct FwdMma {
  static constexpr int BM = 128, BN = 64, WARPS = 8, THREADS = WARPS * 32;
  static constexpr int CH = D / 8;  // 16-byte chunks per row
  static constexpr int Q_BYTES = BM * D * 2;
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int SMEM = Q_BYTES + 4 * KV_BYTES;  // Q, K[2], V[2]
};

// Next live 64-key block after (kt, sub); false when the walk is done.
__device__ __forceinline__ bool next_key_block(const Problem& p, int qt, int klim,
                                               int& kt, int& sub) {
  ++sub;
  if (sub == 2 || kt * kTile + sub * 64 >= klim) {
    sub = 0;
    ++kt;
    while (kt < p.T && !tile_live(p, qt, kt, klim)) ++kt;
    if (kt >= p.T) return false;
  }
  return true;
}

template <int D>
__global__ void __launch_bounds__(FwdMma<D>::THREADS, 1)
    fwd_mma_kernel(Problem p, const __nv_bfloat16* __restrict__ q,
                   const __nv_bfloat16* __restrict__ k,
                   const __nv_bfloat16* __restrict__ v, __nv_bfloat16* __restrict__ o,
                   float* __restrict__ lse) {
  using C = FwdMma<D>;
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t sQ = smem_u32(smem);
  const uint32_t sK0 = sQ + C::Q_BYTES;
  const uint32_t sV0 = sK0 + 2 * C::KV_BYTES;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const long long bh = blockIdx.x;
  const int qt = p.T - 1 - (int)blockIdx.y;  // heaviest causal tiles first
  const int b = (int)(bh / p.H);
  const int q0 = qt * C::BM;
  const int klim = key_limit(p, b);
  const size_t head = (size_t)bh * p.N * D;

  // ---- Q tile ----
  for (int i = tid; i < C::BM * C::CH; i += C::THREADS) {
    int r = i / C::CH, c = i % C::CH;
    int row = q0 + r;
    bool ok = row < p.N;
    cp_async_16(sQ + swz(r, c, C::CH), q + head + (size_t)(ok ? row : 0) * D + c * 8, ok);
  }
  auto load_kv = [&](int stage, int kbase) {
    for (int i = tid; i < C::BN * C::CH; i += C::THREADS) {
      int r = i / C::CH, c = i % C::CH;
      int row = kbase + r;
      bool ok = row < p.N;
      size_t off = head + (size_t)(ok ? row : 0) * D + c * 8;
      cp_async_16(sK0 + stage * C::KV_BYTES + swz(r, c, C::CH), k + off, ok);
      cp_async_16(sV0 + stage * C::KV_BYTES + swz(r, c, C::CH), v + off, ok);
    }
  };

  int kt = -1, sub = 1;
  bool have = next_key_block(p, qt, klim, kt, sub);
  if (have) load_kv(0, kt * kTile + sub * 64);
  cp_async_commit();

  float acc[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  uint32_t qa[D / 16][4];
  bool q_loaded = false;

  int stage = 0;
  while (have) {
    const int cur_kt = kt, cur_kbase = kt * kTile + sub * 64;
    have = next_key_block(p, qt, klim, kt, sub);
    if (have) load_kv(stage ^ 1, kt * kTile + sub * 64);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();

    if (!q_loaded) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        int r = warp * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        int c = kk * 2 + (lane >> 4);
        ldsm_x4(sQ + swz(r, c, C::CH), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
      }
      q_loaded = true;
    }

    // ---- S = Q K^T for this warp's 16 rows x 64 keys ----
    float s[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
    const uint32_t sK = sK0 + stage * C::KV_BYTES;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
      for (int np = 0; np < 4; ++np) {
        int r = np * 16 + (lane & 7) + ((lane >> 4) << 3);
        int c = kk * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(sK + swz(r, c, C::CH), b0, b1, b2, b3);
        mma_bf16(s[2 * np], qa[kk], b0, b1);
        mma_bf16(s[2 * np + 1], qa[kk], b2, b3);
      }
    }

    // ---- scale to log2 units, mask partial blocks ----
    const bool need_mask = (p.causal && cur_kt == qt) || (cur_kbase + 64 > klim);
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float x = s[nt][e] * p.scale_log2;
        if (need_mask) {
          int i = q0 + warp * 16 + g + ((e >> 1) << 3);
          int j = cur_kbase + nt * 8 + 2 * t4 + (e & 1);
          if (j >= klim || (p.causal && j > i)) x = -INFINITY;
        }
        s[nt][e] = x;
      }
    }

    // ---- online softmax update ----
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      float mx = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) mx = fmaxf(mx, fmaxf(s[nt][2 * r], s[nt][2 * r + 1]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run[r], mx);
      const float ref = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = fast_exp2(m_run[r] - ref);  // 0 while nothing seen
      float sum = 0.f;
#pragma unroll
      for (int nt = 0; nt < 8; ++nt) {
        float p0 = fast_exp2(s[nt][2 * r] - ref);
        float p1 = fast_exp2(s[nt][2 * r + 1] - ref);
        s[nt][2 * r] = p0;
        s[nt][2 * r + 1] = p1;
        sum += p0 + p1;
      }
      l_run[r] = l_run[r] * alpha + sum;
      m_run[r] = m_new;
#pragma unroll
      for (int dt = 0; dt < D / 8; ++dt) {
        acc[dt][2 * r] *= alpha;
        acc[dt][2 * r + 1] *= alpha;
      }
    }

    // ---- O += P V ----
    const uint32_t sV = sV0 + stage * C::KV_BYTES;
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      uint32_t pa[4];
      pa[0] = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
      pa[1] = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
      pa[2] = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      pa[3] = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        int r = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        int c = dp * 2 + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(sV + swz(r, c, C::CH), b0, b1, b2, b3);
        mma_bf16(acc[2 * dp], pa, b0, b1);
        mma_bf16(acc[2 * dp + 1], pa, b2, b3);
      }
    }
    __syncthreads();
    stage ^= 1;
  }
  cp_async_wait<0>();
  __syncthreads();

  // ---- epilogue: O = u / l (bf16), LSE = ln2 * (m + log2 l) ----
  uint8_t* sO = smem;  // reuse the Q tile
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    float l = l_run[r];
    l += __shfl_xor_sync(0xffffffffu, l, 1);
    l += __shfl_xor_sync(0xffffffffu, l, 2);
    const float inv = l > 0.f ? 1.f / l : 0.f;
    const int rl = warp * 16 + g + r * 8;
#pragma unroll
    for (int dt = 0; dt < D / 8; ++dt) {
      int col = dt * 8 + 2 * t4;
      *reinterpret_cast<uint32_t*>(sO + swz(rl, col >> 3, C::CH) + (col & 7) * 2) =
          pack_bf16(acc[dt][2 * r] * inv, acc[dt][2 * r + 1] * inv);
    }
    if (t4 == 0 && q0 + rl < p.N)
      lse[(size_t)bh * p.N + q0 + rl] =
          l > 0.f ? (m_run[r] + log2f(l)) * kLn2 : -INFINITY;
  }
  __syncthreads();
  for (int i = tid; i < C::BM * C::CH; i += C::THREADS) {
    int r = i / C::CH, c = i % C::CH;
    if (q0 + r < p.N)
      *reinterpret_cast<uint4*>(o + head + (size_t)(q0 + r) * D + c * 8) =
          *reinterpret_cast<const uint4*>(sO + swz(r, c, C::CH));
  }
}

template <int D>
cudaError_t launch_fwd_mma_t(const Problem& p, const void* q, const void* k,
                             const void* v, void* o, float* lse, cudaStream_t st) {
  using C = FwdMma<D>;
  auto kern = fwd_mma_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((long long)p.B * p.H), (unsigned)p.T);
  kern<<<grid, C::THREADS, C::SMEM, st>>>(
      p, static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
      static_cast<const __nv_bfloat16*>(v), static_cast<__nv_bfloat16*>(o), lse);
  return cudaGetLastError();
}

cudaError_t launch_fwd_mma(const Problem& p, const void* q, const void* k, const void* v,
                           void* o, float* lse, cudaStream_t st) {
  return p.d == 64 ? launch_fwd_mma_t<64>(p, q, k, v, o, lse, st)
                   : launch_fwd_mma_t<128>(p, q, k, v, o, lse, st);
}

}  // namespace fa
