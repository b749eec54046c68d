// Warp-level (mma.sync) attention backward with recomputation.
//
// One CTA owns 128 keys of one (b, h); 8 warps own 16 key rows each.  K and
// V are loaded once; the CTA walks the live query tiles of its key tile in
// BM-row steps (Q, dO, LSE, D double-buffered by cp.async) and, per step,
// rebuilds the probabilities from the stored row statistic instead of
// reading a stored P (page "FlashAttention IO-aware explained", section
// "Recomputation and IO complexity"):
//     S^T  = scale K Q^T,     P^T = exp(S^T - LSE)
//     dV  += P^T dO
//     dP^T = V dO^T,          dS^T = P^T * (dP^T - D)
//     dK  += dS^T Q           (scaled by `scale` at the end)
//     dQacc += dS K           (fp32 atomics into the workspace; the
//                              conversion kernel applies `scale`)
// K and V are read from HBM once; Q, dO and the dQ accumulator are passed
// over once per live key tile, the pattern of Theorem 5's proof (page
// "FlashAttention: Fast and Memory-Efficient Exact Attention with
// IO-Awareness", "C Proofs").
#include "fa_common.cuh"
#include "fa_kernels.h"

namespace fa {

template <int D>
struct BwdMma {
  static constexpr int BN = 128, WARPS = 8, THREADS = WARPS * 32;
  static constexpr int BM = D == 64 ? 64 : 32;  // query rows per step
  static constexpr int CH = D / 8;
  static constexpr int DSCH = BM / 8;  // 16-byte chunks per dS^T row
  static constexpr int KV_BYTES = BN * D * 2;
  static constexpr int QB_BYTES = BM * D * 2;
  static constexpr int DS_BYTES = BN * BM * 2;
  // K, V, Q[2], dO[2], dS^T, lse2[2][BM], Dv[2][BM]
  static constexpr int OFF_V = KV_BYTES;
  static constexpr int OFF_Q = 2 * KV_BYTES;
  static constexpr int OFF_DO = OFF_Q + 2 * QB_BYTES;
  static constexpr int OFF_DS = OFF_DO + 2 * QB_BYTES;
  static constexpr int OFF_L = OFF_DS + DS_BYTES;
  static constexpr int OFF_D = OFF_L + 2 * BM * 4;
  static constexpr int SMEM = OFF_D + 2 * BM * 4;
};

// Next live BM-row query block after (qt, q0) for key tile kt.
template <int BM>
__device__ __forceinline__ bool next_query_block(const Problem& p, int kt, int klim,
                                                 int& qt, int& q0) {
  q0 += BM;
  if (qt < 0 || q0 >= (qt + 1) * kTile || q0 >= p.N) {
    ++qt;
    while (qt < p.T && !tile_live(p, qt, kt, klim)) ++qt;
    if (qt >= p.T) return false;
    q0 = qt * kTile;
  }
  return true;
}

template <int D>
__global__ void __launch_bounds__(BwdMma<D>::THREADS)
    bwd_mma_kernel(Problem p, const __nv_bfloat16* __restrict__ q,
                   const __nv_bfloat16* __restrict__ k,
                   const __nv_bfloat16* __restrict__ v,
                   const __nv_bfloat16* __restrict__ dout,
                   const float* __restrict__ lse, const float* __restrict__ dvec,
                   float* __restrict__ dq_acc, __nv_bfloat16* __restrict__ dk,
                   __nv_bfloat16* __restrict__ dv) {
  using C = BwdMma<D>;
  constexpr int BM = C::BM, NT = BM / 8;  // n-tiles of 8 queries per step
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t s0 = smem_u32(smem);
  const uint32_t sK = s0, sV = s0 + C::OFF_V;
  float* sL = reinterpret_cast<float*>(smem + C::OFF_L);
  float* sD = reinterpret_cast<float*>(smem + C::OFF_D);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, t4 = lane & 3;
  const long long bh = blockIdx.x;
  const int kt = blockIdx.y;
  const int b = (int)(bh / p.H);
  const int k0 = kt * C::BN;
  const int klim = key_limit(p, b);
  const size_t head = (size_t)bh * p.N * D;
  const size_t rowh = (size_t)bh * p.N;

  for (int i = tid; i < C::BN * C::CH; i += C::THREADS) {
    int r = i / C::CH, c = i % C::CH;
    int row = k0 + r;
    bool ok = row < p.N;
    size_t off = head + (size_t)(ok ? row : 0) * D + c * 8;
    cp_async_16(sK + swz(r, c, C::CH), k + off, ok);
    cp_async_16(sV + swz(r, c, C::CH), v + off, ok);
  }
  auto load_q = [&](int st, int qb) {
    const uint32_t sQ = s0 + C::OFF_Q + st * C::QB_BYTES;
    const uint32_t sO = s0 + C::OFF_DO + st * C::QB_BYTES;
    for (int i = tid; i < BM * C::CH; i += C::THREADS) {
      int r = i / C::CH, c = i % C::CH;
      int row = qb + r;
      bool ok = row < p.N;
      size_t off = head + (size_t)(ok ? row : 0) * D + c * 8;
      cp_async_16(sQ + swz(r, c, C::CH), q + off, ok);
      cp_async_16(sO + swz(r, c, C::CH), dout + off, ok);
    }
    for (int i = tid; i < BM; i += C::THREADS) {
      int row = qb + i;
      float l = row < p.N ? lse[rowh + row] : -INFINITY;
      // +inf turns every probability of a dead or out-of-range row into 0.
      sL[st * BM + i] = l == -INFINITY ? INFINITY : l * kLog2e;
      sD[st * BM + i] = row < p.N ? dvec[rowh + row] : 0.f;
    }
  };

  int qt = -1, q0 = 0;
  bool have = next_query_block<BM>(p, kt, klim, qt, q0);
  if (have) load_q(0, q0);
  cp_async_commit();

  float dva[D / 8][4], dka[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i)
#pragma unroll
    for (int e = 0; e < 4; ++e) dva[i][e] = dka[i][e] = 0.f;

  int st = 0;
  while (have) {
    const int cur_qt = qt, cur_q0 = q0;
    have = next_query_block<BM>(p, kt, klim, qt, q0);
    if (have) load_q(st ^ 1, q0);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();

    const uint32_t sQ = s0 + C::OFF_Q + st * C::QB_BYTES;
    const uint32_t sO = s0 + C::OFF_DO + st * C::QB_BYTES;
    const float* L = sL + st * BM;
    const float* Dv = sD + st * BM;

    // ---- S^T = K Q^T and dP^T = V dO^T (16 keys x BM queries per warp) ----
    float sT[NT][4], dpT[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) sT[i][e] = dpT[i][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
      uint32_t ka[4], va[4];
      {
        int r = warp * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        int c = kk * 2 + (lane >> 4);
        ldsm_x4(sK + swz(r, c, C::CH), ka[0], ka[1], ka[2], ka[3]);
        ldsm_x4(sV + swz(r, c, C::CH), va[0], va[1], va[2], va[3]);
      }
#pragma unroll
      for (int np = 0; np < NT / 2; ++np) {
        int r = np * 16 + (lane & 7) + ((lane >> 4) << 3);
        int c = kk * 2 + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(sQ + swz(r, c, C::CH), b0, b1, b2, b3);
        mma_bf16(sT[2 * np], ka, b0, b1);
        mma_bf16(sT[2 * np + 1], ka, b2, b3);
        ldsm_x4(sO + swz(r, c, C::CH), b0, b1, b2, b3);
        mma_bf16(dpT[2 * np], va, b0, b1);
        mma_bf16(dpT[2 * np + 1], va, b2, b3);
      }
    }

    // ---- P^T = 2^(scale*log2e*S^T - LSE*log2e); dS^T = P^T (dP^T - D) ----
    const bool need_mask = (p.causal && cur_qt == kt) || (k0 + C::BN > klim);
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        int jl = warp * 16 + g + ((e >> 1) << 3);  // key row in tile
        int il = nt * 8 + 2 * t4 + (e & 1);         // query column in step
        float pr = fast_exp2(sT[nt][e] * p.scale_log2 - L[il]);
        if (need_mask) {
          int j = k0 + jl, i = cur_q0 + il;
          if (j >= klim || (p.causal && j > i)) pr = 0.f;
        }
        sT[nt][e] = pr;
        dpT[nt][e] = pr * (dpT[nt][e] - Dv[il]);
      }
    }

    // ---- dV += P^T dO ; dK += dS^T Q ----
#pragma unroll
    for (int kk = 0; kk < BM / 16; ++kk) {
      uint32_t pa[4], da[4];
      pa[0] = pack_bf16(sT[2 * kk][0], sT[2 * kk][1]);
      pa[1] = pack_bf16(sT[2 * kk][2], sT[2 * kk][3]);
      pa[2] = pack_bf16(sT[2 * kk + 1][0], sT[2 * kk + 1][1]);
      pa[3] = pack_bf16(sT[2 * kk + 1][2], sT[2 * kk + 1][3]);
      da[0] = pack_bf16(dpT[2 * kk][0], dpT[2 * kk][1]);
      da[1] = pack_bf16(dpT[2 * kk][2], dpT[2 * kk][3]);
      da[2] = pack_bf16(dpT[2 * kk + 1][0], dpT[2 * kk + 1][1]);
      da[3] = pack_bf16(dpT[2 * kk + 1][2], dpT[2 * kk + 1][3]);
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        int r = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
        int c = dp * 2 + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(sO + swz(r, c, C::CH), b0, b1, b2, b3);
        mma_bf16(dva[2 * dp], pa, b0, b1);
        mma_bf16(dva[2 * dp + 1], pa, b2, b3);
        ldsm_x4_t(sQ + swz(r, c, C::CH), b0, b1, b2, b3);
        mma_bf16(dka[2 * dp], da, b0, b1);
        mma_bf16(dka[2 * dp + 1], da, b2, b3);
      }
    }

    // ---- dS^T to shared memory (bf16, [key][query]) ----
    uint8_t* sDS = smem + C::OFF_DS;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        int jl = warp * 16 + g + h * 8;
        int il = nt * 8 + 2 * t4;  // queries il, il+1 are adjacent in a row
        *reinterpret_cast<uint32_t*>(sDS + swz(jl, il >> 3, C::DSCH) + (il & 7) * 2) =
            pack_bf16(dpT[nt][2 * h], dpT[nt][2 * h + 1]);
      }
    }
    __syncthreads();

    // ---- dQacc[BM x D] += dS K : warp tile = 16 query rows x (D / WPC) cols ----
    {
      constexpr int RG = BM / 16;         // row groups
      constexpr int WPC = C::WARPS / RG;  // warps per row group
      constexpr int COLS = D / WPC;       // output columns per warp
      const int rg = warp / WPC, cg = warp % WPC;
      float qa[COLS / 8][4];
#pragma unroll
      for (int i = 0; i < COLS / 8; ++i) qa[i][0] = qa[i][1] = qa[i][2] = qa[i][3] = 0.f;
      const uint32_t sDSa = s0 + C::OFF_DS;
#pragma unroll
      for (int kk = 0; kk < C::BN / 16; ++kk) {
        uint32_t a[4];
        {
          // A = dS (query rows x keys) read transposed from dS^T [key][query]
          int r = kk * 16 + (lane & 7) + ((lane >> 4) << 3);
          int c = rg * 2 + ((lane >> 3) & 1);
          ldsm_x4_t(sDSa + swz(r, c, C::DSCH), a[0], a[1], a[2], a[3]);
        }
#pragma unroll
        for (int dp = 0; dp < COLS / 16; ++dp) {
          int r = kk * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
          int c = (cg * COLS) / 8 + dp * 2 + (lane >> 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(sK + swz(r, c, C::CH), b0, b1, b2, b3);
          mma_bf16(qa[2 * dp], a, b0, b1);
          mma_bf16(qa[2 * dp + 1], a, b2, b3);
        }
      }
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        int i = cur_q0 + rg * 16 + g + h * 8;
        if (i < p.N) {
          float* dst = dq_acc + (head + (size_t)i * D) + cg * COLS + 2 * t4;
#pragma unroll
          for (int nt = 0; nt < COLS / 8; ++nt) {
            atomicAdd(dst + nt * 8, qa[nt][2 * h]);
            atomicAdd(dst + nt * 8 + 1, qa[nt][2 * h + 1]);
          }
        }
      }
    }
    __syncthreads();
    st ^= 1;
  }
  cp_async_wait<0>();
  __syncthreads();

  // ---- dK = scale * dK, dV: stage through shared memory, coalesced store ----
  uint8_t* sKb = smem;
  uint8_t* sVb = smem + C::OFF_V;
#pragma unroll
  for (int dt = 0; dt < D / 8; ++dt) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      int r = warp * 16 + g + h * 8, col = dt * 8 + 2 * t4;
      uint32_t off = swz(r, col >> 3, C::CH) + (col & 7) * 2;
      *reinterpret_cast<uint32_t*>(sKb + off) =
          pack_bf16(dka[dt][2 * h] * p.scale, dka[dt][2 * h + 1] * p.scale);
      *reinterpret_cast<uint32_t*>(sVb + off) = pack_bf16(dva[dt][2 * h], dva[dt][2 * h + 1]);
    }
  }
  __syncthreads();
  for (int i = tid; i < C::BN * C::CH; i += C::THREADS) {
    int r = i / C::CH, c = i % C::CH;
    if (k0 + r < p.N) {
      size_t off = head + (size_t)(k0 + r) * D + c * 8;
      *reinterpret_cast<uint4*>(dk + off) =
          *reinterpret_cast<const uint4*>(sKb + swz(r, c, C::CH));
      *reinterpret_cast<uint4*>(dv + off) =
          *reinterpret_cast<const uint4*>(sVb + swz(r, c, C::CH));
    }
  }
}

template <int D>
cudaError_t launch_bwd_mma_t(const Problem& p, const void* q, const void* k,
                             const void* v, const void* dout, const float* lse,
                             const float* dvec, float* dq_acc, void* dk, void* dv,
                             cudaStream_t s) {
  using C = BwdMma<D>;
  auto kern = bwd_mma_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       C::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)((long long)p.B * p.H), (unsigned)p.T);
  kern<<<grid, C::THREADS, C::SMEM, s>>>(
      p, static_cast<const __nv_bfloat16*>(q), static_cast<const __nv_bfloat16*>(k),
      static_cast<const __nv_bfloat16*>(v), static_cast<const __nv_bfloat16*>(dout), lse,
      dvec, dq_acc, static_cast<__nv_bfloat16*>(dk), static_cast<__nv_bfloat16*>(dv));
  return cudaGetLastError();
}

cudaError_t launch_bwd_mma(const Problem& p, const void* q, const void* k, const void* v,
                           const void* dout, const float* lse, const float* dvec,
                           float* dq_acc, void* dk, void* dv, cudaStream_t s) {
  return p.d == 64 ? launch_bwd_mma_t<64>(p, q, k, v, dout, lse, dvec, dq_acc, dk, dv, s)
                   : launch_bwd_mma_t<128>(p, q, k, v, dout, lse, dvec, dq_acc, dk, dv, s);
}

}  // namespace fa
