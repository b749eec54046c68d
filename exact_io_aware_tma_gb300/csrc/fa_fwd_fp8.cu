// FP8 (e4m3) tensor-core attention forward for sm_103a, d = 128.
//
// The structure of the bf16 forward (two 128-row query tiles per CTA, a TMA
// producer, one MMA-issuing thread, two softmax warpgroups, the lazily moved
// reference of the online softmax of page "FlashAttention" (aiwiki), section
// "Tiling and online normalization") with block-quantised operands:
//   S_i = (Q8_i K8_j^T) * qs[qt] * ks[kt]     (kind::f8f6f4, K = 4 x 32)
//   P_i = 2^(S_i * scale * log2(e) - m)   rounded to e4m3 (P <= 2^8 < 448)
//   O_i += P8_i Vt8_j^T                       (kind::f8f6f4; Vt8 = V^T codes)
//   O = O * vs / l,  l the row sum of the unrounded P.
// Every operand is K-major with the 128-byte swizzle: Q8 / K8 rows hold 128
// codes (one 128-byte row), V is stored transposed ([d][keys]) by the
// quantisation pass, and P is written by the softmax threads into shared
// memory (one 128-byte row per query row) instead of tensor memory.
//
// Shared memory: Q0 | P0 | Q1 | P1 (16 KB each; O of tile i is staged in
// Q_i + P_i, 32 KB, once every MMA has completed), then a ring of 8 K/Vt
// slots of 16 KB.  TMEM: S0, S1, O0, O1 = 512 columns.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "fa_common.cuh"
#include "fa_kernels.h"
#include "fa_sm100.cuh"
#include "fa_tma_host.h"

namespace fa {
using namespace sm100;

struct Fp8Cfg {
  static constexpr int THREADS = 384;
  static constexpr int NSLOT = 8;
  static constexpr int TILE = 128 * 128;  // one 8-bit 128 x 128 tile
  static constexpr int HALF = 128 * 128;  // one bf16 128-row x 64-column box (O staging)
  static constexpr int OFF_Q0 = 0, OFF_P0 = TILE, OFF_Q1 = 2 * TILE, OFF_P1 = 3 * TILE;
  static constexpr int OFF_KV = 4 * TILE;
  static constexpr int OFF_BAR = OFF_KV + NSLOT * TILE;
  static constexpr int B_Q = 0, B_FULL = 1, B_EMPTY = 1 + NSLOT, B_S = 1 + 2 * NSLOT,
                       B_P = B_S + 2, B_O = B_P + 2, B_DRAIN = B_O + 2, NBAR = B_DRAIN + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_MISC + 64 + 1024;
  static constexpr int COL_S0 = 0, COL_S1 = 128, COL_O0 = 256, COL_O1 = 384;
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(SMEM <= 232448, "shared memory budget");
};

// Next live key tile after kt within [first, last] (no block mask here).
__device__ __forceinline__ int fp8_next_tile(int first, int last, int kt, int T) {
  kt = kt + 1 < first ? first : kt + 1;
  return kt <= last ? kt : T;
}

// Four values rounded to e4m3 (nearest even, saturating), a in the lowest
// byte: consecutive keys in consecutive bytes of the K-major P row.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  return (uint32_t)__nv_cvt_float_to_fp8(a, __NV_SATFINITE, __NV_E4M3) |
         ((uint32_t)__nv_cvt_float_to_fp8(b, __NV_SATFINITE, __NV_E4M3) << 8) |
         ((uint32_t)__nv_cvt_float_to_fp8(c, __NV_SATFINITE, __NV_E4M3) << 16) |
         ((uint32_t)__nv_cvt_float_to_fp8(d, __NV_SATFINITE, __NV_E4M3) << 24);
}

__global__ void __launch_bounds__(Fp8Cfg::THREADS, 1)
    fwd_fp8_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_vt, const __grid_constant__ CUtensorMap tm_o,
                   Problem p, const float* __restrict__ q_scale, const float* __restrict__ k_scale,
                   const float* __restrict__ v_scale, float* __restrict__ lse) {
  using C = Fp8Cfg;
  extern __shared__ uint8_t smem_raw[];
  // An offset (not an integer round trip) keeps the pointer visibly in shared
  // memory, so C++ accesses through it compile to shared-memory instructions.
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t s0 = smem_u32(smem);
  const uint32_t bar0 = s0 + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 16);
  const Abort ab{abort_flag, p.status};

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Grid: grouped order (heaviest pairs first across a group of heads whose
  // K and V stay in L2).
  const int npairs = (p.T + 1) / 2;
  long long bh;
  int yi;
  grouped_cta(p, blockIdx.x, npairs, bh, yi);
  const int pair = npairs - 1 - yi;
  const int qt0 = 2 * pair;
  const int qt1 = (2 * pair + 1 < p.T) ? 2 * pair + 1 : -1;
  const int klim = p.N;
  int first0, last0, first1 = 0, last1 = -1;
  qtile_key_tiles(p, qt0, klim, first0, last0);
  if (qt1 >= 0) qtile_key_tiles(p, qt1, klim, first1, last1);
  const int ufirst = first0 <= last0 ? first0 : first1;
  const int ulast = max(last0, last1);

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NBAR; ++i)
      mbar_init(bar(i), (i == C::B_P || i == C::B_P + 1) ? 4 : 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_vt);
    prefetch_tensormap(&tm_o);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_expect_tx(bar(C::B_Q), (qt1 >= 0 ? 2 : 1) * C::TILE);
      tma_load_3d(s0 + C::OFF_Q0, &tm_q, bar(C::B_Q), 0, qt0 * 128, (int)bh);
      if (qt1 >= 0) tma_load_3d(s0 + C::OFF_Q1, &tm_q, bar(C::B_Q), 0, qt1 * 128, (int)bh);
      int slot = 0, round = 0;
      bool ok = true;
      for (int kt = fp8_next_tile(ufirst, ulast, -1, p.T); kt < p.T && ok;
           kt = fp8_next_tile(ufirst, ulast, kt, p.T)) {
        for (int which = 0; which < 2; ++which) {
          if (!mbar_wait(bar(C::B_EMPTY + slot), (round & 1) ^ 1, ab)) {
            ok = false;
            break;
          }
          const uint32_t dst = s0 + C::OFF_KV + slot * C::TILE;
          mbar_expect_tx(bar(C::B_FULL + slot), C::TILE);
          if (which == 0)
            tma_load_3d(dst, &tm_k, bar(C::B_FULL + slot), 0, kt * 128, (int)bh);
          else
            tma_load_3d(dst, &tm_vt, bar(C::B_FULL + slot), kt * 128, 0, (int)bh);
          if (++slot == C::NSLOT) {
            slot = 0;
            ++round;
          }
        }
      }
      // Drain: every load issued lands before shared memory is released.
      for (int s = 0; s < C::NSLOT; ++s) {
        const int last = round - (s >= slot ? 1 : 0);
        if (last >= 0) {
          const uint64_t t0 = globaltimer();
          while (!mbar_try_wait(bar(C::B_FULL + s), last & 1) &&
                 globaltimer() - t0 < kWaitLimitNs) {
          }
        }
      }
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(bar(C::B_Q), 0) && globaltimer() - t0 < kWaitLimitNs) {
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t id = idesc_e4m3(128, 128);
      constexpr uint32_t slot_step = C::TILE >> 4;
      const uint64_t dq0 = sdesc_sw128(s0 + C::OFF_Q0, 16, 1024);
      const uint64_t dq1 = sdesc_sw128(s0 + C::OFF_Q1, 16, 1024);
      const uint64_t dp0 = sdesc_sw128(s0 + C::OFF_P0, 16, 1024);
      const uint64_t dp1 = sdesc_sw128(s0 + C::OFF_P1, 16, 1024);
      const uint64_t dkv = sdesc_sw128(s0 + C::OFF_KV, 16, 1024);
      const uint32_t t_s0 = tmem + C::COL_S0, t_s1 = tmem + C::COL_S1;
      const uint32_t t_o0 = tmem + C::COL_O0, t_o1 = tmem + C::COL_O1;
      // K = 128 codes per row in four 32-code (32-byte) steps
      auto gemm = [&](uint32_t d, uint64_t a, uint64_t b, bool acc) {
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss_f8(d, a + (uint64_t)(2 * kk), b + (uint64_t)(2 * kk), id, (acc || kk > 0) ? 1u : 0u);
      };
      auto live0 = [&](int kt) { return kt >= first0 && kt <= last0; };
      auto live1 = [&](int kt) { return kt >= first1 && kt <= last1; };
      int slot = 0, phase = 0;
      bool ok = mbar_wait(bar(C::B_Q), 0, ab);
      tc_fence_after();
      int cur = fp8_next_tile(ufirst, ulast, -1, p.T);
      int npv0 = 0, npv1 = 0;
      if (ok && cur < p.T) {
        ok = mbar_wait(bar(C::B_FULL + slot), phase, ab);
        tc_fence_after();
        if (ok) {
          const uint64_t dk = dkv + (uint64_t)(slot * slot_step);
          if (live0(cur)) {
            gemm(t_s0, dq0, dk, false);
            mma_commit(bar(C::B_S + 0));
          }
          if (live1(cur)) {
            gemm(t_s1, dq1, dk, false);
            mma_commit(bar(C::B_S + 1));
          }
          mma_commit(bar(C::B_EMPTY + slot));
        }
        if (++slot == C::NSLOT) { slot = 0; phase ^= 1; }
      }
      while (ok && cur < p.T) {
        const bool l0 = live0(cur), l1 = live1(cur);
        const int vslot = slot, vphase = phase;
        if (++slot == C::NSLOT) { slot = 0; phase ^= 1; }
        const int nxt = fp8_next_tile(ufirst, ulast, cur, p.T);
        const bool has_next = nxt < p.T;
        const bool n0 = has_next && live0(nxt), n1 = has_next && live1(nxt);
        const int kslot = slot, kphase = phase;
        if (has_next && ++slot == C::NSLOT) { slot = 0; phase ^= 1; }
        const uint64_t dv = dkv + (uint64_t)(vslot * slot_step);
        const uint64_t dk = dkv + (uint64_t)(kslot * slot_step);
        if (!(ok = mbar_wait(bar(C::B_FULL + vslot), vphase, ab))) break;
        if (has_next && !(ok = mbar_wait(bar(C::B_FULL + kslot), kphase, ab))) break;
        tc_fence_after();
        if (l0) {
          if (!(ok = mbar_wait(bar(C::B_P + 0), npv0 & 1, ab))) break;
          tc_fence_after();
          gemm(t_o0, dp0, dv, npv0 > 0);
          ++npv0;
        }
        if (n0) {
          gemm(t_s0, dq0, dk, false);
          mma_commit(bar(C::B_S + 0));
        }
        if (l1) {
          if (!(ok = mbar_wait(bar(C::B_P + 1), npv1 & 1, ab))) break;
          tc_fence_after();
          gemm(t_o1, dp1, dv, npv1 > 0);
          ++npv1;
        }
        mma_commit(bar(C::B_EMPTY + vslot));
        if (has_next) {
          if (n1) {
            gemm(t_s1, dq1, dk, false);
            mma_commit(bar(C::B_S + 1));
          }
          mma_commit(bar(C::B_EMPTY + kslot));
        }
        cur = nxt;
      }
      mma_commit(bar(C::B_O + 0));
      mma_commit(bar(C::B_O + 1));
      mma_commit(bar(C::B_DRAIN));
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(bar(C::B_DRAIN), 0) && globaltimer() - t0 < kWaitLimitNs) {
      }
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax
    const int i = (warp - 4) >> 2;  // query tile of this warpgroup
    const int qt = i == 0 ? qt0 : qt1;
    if (qt >= 0) {
      const int r = ((warp & 3) << 5) + lane;
      const int row = qt * 128 + r;
      const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
      const uint32_t col_s = i == 0 ? C::COL_S0 : C::COL_S1;
      const uint32_t col_o = i == 0 ? C::COL_O0 : C::COL_O1;
      uint8_t* prow = smem + (i == 0 ? C::OFF_P0 : C::OFF_P1) + r * 128;
      const float qs = __ldg(q_scale + bh * p.T + qt);
      const int myfirst = i == 0 ? first0 : first1, mylast = i == 0 ? last0 : last1;
      float m_ref = -INFINITY, l = 0.f;
      int n = 0;
      bool ok = true;
      for (int kt = fp8_next_tile(ufirst, ulast, -1, p.T); kt < p.T;
           kt = fp8_next_tile(ufirst, ulast, kt, p.T)) {
        if (kt < myfirst || kt > mylast) continue;
        // per-tile score multiplier: scale * log2(e) * qs * ks (kept off zero
        // so that a masked +-inf never meets 0 * inf)
        float cl2 = p.scale_log2 * qs * __ldg(k_scale + bh * p.T + kt);
        if (fabsf(cl2) < 1e-30f) cl2 = cl2 < 0.f ? -1e-30f : 1e-30f;
        if (!(ok = mbar_wait(bar(C::B_S + i), n & 1, ab))) break;
        tc_fence_after();
        float s[128];
        {
          uint32_t raw[128];
          tmem_ld128(lane_base + col_s, raw);
#pragma unroll
          for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(raw[c]);
        }
        {
          const int k0 = kt * 128;
          const int hi = row_key_hi(p, row, klim) + 1 - k0;
          if (hi < 128) {
            const float fill = cl2 >= 0.f ? -INFINITY : INFINITY;
#pragma unroll
            for (int c = 0; c < 128; ++c)
              if (c >= hi) s[c] = fill;
          }
        }
        float mx;
        if (cl2 >= 0.f) {
          float m4[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
          for (int c = 4; c + 8 <= 124; c += 8)
#pragma unroll
            for (int e = 0; e < 4; ++e) m4[e] = max3f(m4[e], s[c + e], s[c + 4 + e]);
#pragma unroll
          for (int e = 0; e < 4; ++e) m4[e] = fmaxf(m4[e], s[124 + e]);
          mx = max3f(m4[0], m4[1], fmaxf(m4[2], m4[3]));
        } else {
          float m4[4] = {INFINITY, INFINITY, INFINITY, INFINITY};
#pragma unroll
          for (int c = 0; c < 128; ++c) m4[c & 3] = fminf(m4[c & 3], s[c]);
          const float mn = fminf(fminf(m4[0], m4[1]), fminf(m4[2], m4[3]));
          mx = mn == INFINITY ? -INFINITY : mn;
        }
        const float m_tile = mx == -INFINITY ? -INFINITY : mx * cl2;
        float alpha = 1.f;
        if (m_tile > m_ref + 8.f) {
          alpha = fast_exp2(m_ref - m_tile);
          m_ref = m_tile;
        }
        const float nref = m_ref == -INFINITY ? 0.f : -m_ref;
        // P (<= 2^8) rounded to e4m3 into the K-major swizzled P buffer:
        // row r, 16-byte chunk c (keys 16c .. 16c+15) at (c ^ (r & 7)) * 16
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t w[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            float x0, x1, x2, x3;
            const int b = 16 * c + 4 * q;
            fma2(x0, x1, s[b], s[b + 1], cl2, cl2, nref, nref);
            fma2(x2, x3, s[b + 2], s[b + 3], cl2, cl2, nref, nref);
            const float p0 = fast_exp2(x0), p1 = fast_exp2(x1), p2 = fast_exp2(x2),
                        p3 = fast_exp2(x3);
            add2(sa[q], sb[q], sa[q], sb[q], p0, p1);
            add2(sa[q], sb[q], sa[q], sb[q], p2, p3);
            w[q] = e4m3x4(p0, p1, p2, p3);
          }
          *reinterpret_cast<uint4*>(prow + ((c ^ (r & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
        }
        const float sum = ((sa[0] + sb[0]) + (sa[1] + sb[1])) + ((sa[2] + sb[2]) + (sa[3] + sb[3]));
        l = l * alpha + sum;
        if (n > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t o[32];
            tmem_ld32(lane_base + col_o + 32 * c, o);
#pragma unroll
            for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
            tmem_st32(lane_base + col_o + 32 * c, o);
          }
        }
        fence_proxy_async_smem();
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_P + i));
        ++n;
      }
      // ---- epilogue: O * vs / l -> bf16 -> shared (swizzled, Q_i + P_i) -> TMA store
      if (ok) ok = mbar_wait(bar(C::B_O + i), 0, ab);
      tc_fence_after();
      uint8_t* stage = smem + (i == 0 ? C::OFF_Q0 : C::OFF_Q1);
      const float inv = l > 0.f ? __ldg(v_scale + bh) / l : 0.f;
      if (ok) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          tmem_ld32(lane_base + col_o + 32 * c, o);
          uint32_t pk[16];
#pragma unroll
          for (int j = 0; j < 16; ++j)
            pk[j] = pack_bf16(__uint_as_float(o[2 * j]) * inv, __uint_as_float(o[2 * j + 1]) * inv);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int cc = 4 * c + q;
            uint8_t* dst = stage + (cc >> 3) * C::HALF + r * 128 + (((cc & 7) ^ (r & 7)) << 4);
            *reinterpret_cast<uint4*>(dst) =
                make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          }
        }
        if (row < p.N)
          lse[(size_t)bh * p.N + row] = l > 0.f ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
      }
      fence_proxy_async_smem();
      named_barrier(1 + i, 128);
      if (ok && r == 0) {
        for (int h = 0; h < 2; ++h)
          tma_store_3d(&tm_o, smem_u32(stage) + h * C::HALF, h * 64, qt * 128, (int)bh);
        tma_store_commit();
        tma_store_wait_read();  // shared memory read out; the writes finish with the grid
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

cudaError_t launch_fwd_fp8(const Problem& pin, const void* q8, const void* k8, const void* vt8,
                           const float* q_scale, const float* k_scale, const float* v_scale,
                           void* o, float* lse, cudaStream_t st) {
  using C = Fp8Cfg;
  // Heads per CTA group: e4m3 K and V of a group within about 64 MB.
  Problem p = pin;
  {
    const long long heads = (long long)p.B * p.H;
    long long g = (64ll << 20) / ((long long)p.N * 128 * 2);
    p.hgroup = (int)(g < 1 ? 1 : (g > heads ? heads : g));
  }
  const long long bh = (long long)p.B * p.H;
  CUtensorMap tq, tk, tvt, to;
  if (!make_u8_map_3d(&tq, q8, 128, p.N, bh, 128) || !make_u8_map_3d(&tk, k8, 128, p.N, bh, 128) ||
      !make_u8_map_3d(&tvt, vt8, p.T * 128, 128, bh, 128) ||
      !make_bf16_map_3d(&to, o, 128, p.N, bh, 128))
    return cudaErrorInvalidValue;
  cudaError_t e =
      cudaFuncSetAttribute(fwd_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)(bh * ((p.T + 1) / 2)));
  fwd_fp8_kernel<<<grid, C::THREADS, C::SMEM, st>>>(tq, tk, tvt, to, p, q_scale, k_scale, v_scale,
                                                    lse);
  return cudaGetLastError();
}

}  // namespace fa
