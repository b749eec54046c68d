// Attention of a few query rows against a key/value cache, split over the
// keys, and the merge of partial results.
//
// What is computed (page "FlashAttention", aiwiki): the scaled dot-product
// formula of section "Attention and the memory bottleneck" for Nq query rows
// against the cache_len[b] valid slots of an Nk-slot cache (the inference-
// with-cached-keys interface of section "Software integration and
// limitations"); the key range of every head is cut into `S` splits that
// run on different CTAs, each producing a normalised partial output and its
// log-sum-exp, and the partials are folded together with the running-max /
// running-sum / rescaled-accumulator update of section "Tiling and online
// normalization" (a partial (O_s, LSE_s) is the state m = LSE_s, l = 1,
// u = O_s).
//
// Why CUDA cores and not the tensor cores: with at most 4 rows per pass the
// kernel does 2*Nq*d multiply-adds per 4*d bytes of K and V it streams, far
// below the ridge point of the machine; the limit is HBM bandwidth.  The
// design therefore aims at streaming: a TMA producer warp keeps three (d=128)
// or six (d=64) 32/16 KB K+V stages in flight per CTA, two CTAs per SM, and
// four consumer warps turn each stage into scores and an output update with
// packed fp32 FMAs fast enough to stay behind the copies.
//
// Rows per pass: Nq query rows are taken in groups of RQ = 1, 2 or 4 that
// share one walk over the keys.  The group's rows come from the producer in
// a two-slot ring (bulk copy plus the item's key range), so the consumers
// never wait on a global load at an item boundary; they hold the rows in
// registers, or, for four rows of d = 128, as an fp32 copy in shared memory
// (registers would leave room for only one CTA per SM).
//
// Consumer layout, per 64-key stage: consumer warp w owns keys 16w..16w+15.
//   scores:  8 lanes per key (lane group g = lane/8 takes keys 4p+g of its
//            16 in pass p = 0..3); lane li = lane%8 holds 16-byte chunk li of
//            each 64-column box of the query rows in registers (pre-scaled by
//            scale*log2(e)) and reads the same chunk of the key row; the 8
//            partial dot products reduce by three xor-shuffles.
//   softmax: per row, the max over the warp's 16 keys (two more shuffles),
//            p = 2^(s - m) with the running max m, a per-lane partial row sum.
//   output:  lane owns d/32 consecutive columns; p goes through a small
//            per-warp shared buffer and is read back as a broadcast.
// Each warp thus keeps its own online-softmax state; at the end of an item
// the four states are merged through shared memory with the same update.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/fa.h"
#include "../../include/fa_kvcache.h"
#include "fa_common.cuh"
#include "fa_kernels.h"
#include "fa_sm100.cuh"
#include "fa_tma_host.h"

namespace fa {
namespace kvc {

using namespace sm100;

constexpr int KT = 64;                // keys per stage
constexpr int NCW = 4;                // consumer warps
constexpr int THREADS = 32 * (1 + NCW);
constexpr int KPW = KT / NCW;         // keys per consumer warp per stage
constexpr int RQ_MAX = 4;             // query rows per pass
template <int D, int RQ>
struct Cfg {
  // One-row passes need few registers: three CTAs per SM (more warps to hide
  // the latency of each CTA's dependent steps), 64 KB of stages each;
  // otherwise two CTAs with 96 KB.  Either way about 192 KB per SM in flight.
  static constexpr int CTAS = RQ == 1 ? 3 : 2;
  static constexpr int STAGE_BUDGET = CTAS == 3 ? 64 * 1024 : 96 * 1024;
  static constexpr int NB = D / 64;              // 64-column boxes per row
  static constexpr int BOX = KT * 128;           // one box: 64 rows x 128 B
  static constexpr int TILE = NB * BOX;          // K or V of one stage
  static constexpr int STAGE = 2 * TILE;
  static constexpr int NS = STAGE_BUDGET / STAGE;
  static constexpr int NC = D / 32;              // output columns per lane
  // Query rows live in registers (RQ*NB*8 floats per lane) unless that would
  // cost two CTAs per SM; then in an fp32 shared copy read per use.
  static constexpr bool QREG = RQ * NB <= 4;
  static constexpr int QSLOT = RQ * D * 2 + 16;  // bf16 rows + item header
  static constexpr int OFF_Q = NS * STAGE;       // q ring: 2 slots
  static constexpr int OFF_Q32 = OFF_Q + 2 * QSLOT;            // fp32 [RQ][D] (if !QREG)
  static constexpr int OFF_P = OFF_Q32 + (QREG ? 0 : RQ * D * 4);  // p: [NCW][KPW] x float4
  static constexpr int OFF_ML = OFF_P + NCW * KPW * 16;  // m, l: [2][NCW][RQ_MAX]
  static constexpr int OFF_U = OFF_ML + 2 * NCW * RQ_MAX * 4;  // u: [NCW][RQ][D]
  // full[NS], empty[NS], qfull[2], qempty[2]
  static constexpr int OFF_BAR = OFF_U + NCW * RQ * D * 4;
  static constexpr int OFF_FLAG = OFF_BAR + (2 * NS + 4) * 8;
  static constexpr int SMEM = OFF_FLAG + 16 + 1024;  // + slack to align the base to 1024
  static_assert(NS >= 2, "need at least two stages");
  static_assert(RQ <= NCW, "one merging warp per query row");
  static_assert(QSLOT % 16 == 0 && OFF_Q32 % 16 == 0, "16-byte aligned q buffers");
};

struct Params {
  int B, H, Nq, Nk;
  long long BH;           // B*H
  int S;                  // key splits per (head, query group)
  int QG;                 // query groups of RQ rows
  long long items;        // B*H*S*QG
  float scale_log2;       // scale * log2(e)
  int causal;
  const int32_t* cache_len;   // [B] or nullptr
  const __nv_bfloat16* q;     // [B,H,Nq,D]
  __nv_bfloat16* o;           // [B,H,Nq,D]   (S == 1)
  float* lse;                 // [B,H,Nq]     (S == 1)
  float* o_part;              // [S][B*H*Nq][D]  (S > 1)
  float* lse_part;            // [S][B*H*Nq]     (S > 1)
  int* status;
};

// Geometry of one work item: head bh, split s, query group qg, its rows
// [r0, r0+nr) -- pure arithmetic on the item index -- and, from the cache
// length L of its batch row, the first row's key limit kmin and its key
// tiles [t0, t1).  The producer derives all of it and hands L, kmin, t0, t1
// to the consumers in the item's query slot.
struct Item {
  long long bh;
  int s, r0, nr, L, kmin, t0, t1;
};

template <int RQ>
__device__ __forceinline__ Item item_rows(const Params& p, long long it) {
  Item x;
  const int qg = (int)(it % p.QG);
  x.s = (int)((it / p.QG) % p.S);
  x.bh = it / ((long long)p.QG * p.S);
  x.r0 = qg * RQ;
  x.nr = min(RQ, p.Nq - x.r0);
  return x;
}

template <int RQ>
__device__ __forceinline__ Item item_at(const Params& p, long long it) {
  Item x = item_rows<RQ>(p, it);
  const int b = (int)(x.bh / p.H);
  int L = p.Nk;
  if (p.cache_len != nullptr) {
    L = __ldg(p.cache_len + b);
    L = L < 0 ? 0 : (L > p.Nk ? p.Nk : L);
  }
  x.L = L;
  // Row r (absolute) sits at position L - Nq + r and, when causal, sees keys
  // j <= L - Nq + r.  The group needs keys below kend, its last row's limit.
  int kend = p.causal ? min(L, L - p.Nq + x.r0 + x.nr) : L;
  x.kmin = p.causal ? min(L, L - p.Nq + x.r0 + 1) : L;
  if (kend < 0) kend = 0;
  const int nt = (kend + KT - 1) / KT;
  x.t0 = (int)((long long)x.s * nt / p.S);
  x.t1 = (int)((long long)(x.s + 1) * nt / p.S);
  return x;
}

// Bounded wait that ignores the CTA's abort flag: used only to let copies
// already issued land before the CTA exits.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
  if (mbar_test(bar, parity)) return;
  const uint64_t t0 = globaltimer();
  while (!mbar_try_wait(bar, parity))
    if (globaltimer() - t0 > kWaitLimitNs) return;
}

__device__ __forceinline__ float2 bf16x2_to_f2(uint32_t w) {
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

template <int D, int RQ>
__global__ void __launch_bounds__(THREADS, Cfg<D, RQ>::CTAS)
    kvcache_split_kernel(const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, Params p) {
  using C = Cfg<D, RQ>;
  extern __shared__ uint8_t smem_raw[];
  // Offset (not an integer round trip) keeps the pointer visibly in shared
  // memory, so the accesses below compile to shared-memory loads and stores.
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_full = sbase + C::OFF_BAR;
  const uint32_t bar_empty = bar_full + C::NS * 8;
  const uint32_t bar_qfull = bar_empty + C::NS * 8;
  const uint32_t bar_qempty = bar_qfull + 2 * 8;
  volatile int* flag = reinterpret_cast<volatile int*>(smem + C::OFF_FLAG);
  const Abort ab{flag, p.status};
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::NS; ++i) {
      mbar_init(bar_full + 8 * i, 1);
      mbar_init(bar_empty + 8 * i, NCW);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_qfull + 8 * i, 1);
      mbar_init(bar_qempty + 8 * i, NCW);
    }
    *flag = 0;
    fence_barrier_init();
  }
  __syncthreads();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensormap(&tm_k);
      prefetch_tensormap(&tm_v);
      int slot = 0, qs = 0;
      uint32_t phase = 0, qph = 0;
      long long issued = 0, qissued = 0;
      bool ok = true;
      for (long long it = blockIdx.x; it < p.items && ok; it += gridDim.x) {
        const Item x = item_at<RQ>(p, it);
        // The item's query rows and header into query slot qs.
        if (!mbar_wait(bar_qempty + 8 * qs, qph ^ 1, ab)) break;
        uint8_t* qslot = smem + C::OFF_Q + qs * C::QSLOT;
        int* hdr = reinterpret_cast<int*>(qslot + RQ * D * 2);
        hdr[0] = x.L;
        hdr[1] = x.kmin;
        hdr[2] = x.t0;
        hdr[3] = x.t1;
        const uint32_t qbytes = (uint32_t)x.nr * D * 2;
        mbar_expect_tx(bar_qfull + 8 * qs, qbytes);
        bulk_load(smem_u32(qslot), p.q + (x.bh * p.Nq + x.r0) * D, qbytes, bar_qfull + 8 * qs);
        ++qissued;
        if (++qs == 2) {
          qs = 0;
          qph ^= 1;
        }
        for (int t = x.t0; t < x.t1; ++t) {
          if (!mbar_wait(bar_empty + 8 * slot, phase ^ 1, ab)) {
            ok = false;
            break;
          }
          const uint32_t full = bar_full + 8 * slot;
          const uint32_t dst = sbase + slot * C::STAGE;
          mbar_expect_tx(full, C::STAGE);
#pragma unroll
          for (int c = 0; c < C::NB; ++c) {
            tma_load_3d(dst + c * C::BOX, &tm_k, full, c * 64, t * KT, (int)x.bh);
            tma_load_3d(dst + C::TILE + c * C::BOX, &tm_v, full, c * 64, t * KT, (int)x.bh);
          }
          ++issued;
          if (++slot == C::NS) {
            slot = 0;
            phase ^= 1;
          }
        }
      }
      // Let every copy issued land before the CTA may exit: the last
      // min(NS, issued) stages and min(2, qissued) query slots, newest first.
      for (int i = 0; i < C::NS && i < issued; ++i) {
        if (--slot < 0) {
          slot = C::NS - 1;
          phase ^= 1;
        }
        drain_wait(bar_full + 8 * slot, phase);
      }
      for (int i = 0; i < 2 && i < qissued; ++i) {
        if (--qs < 0) {
          qs = 1;
          qph ^= 1;
        }
        drain_wait(bar_qfull + 8 * qs, qph);
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int cw = warp - 1;
  const int g = lane >> 3;
  const int li = lane & 7;
  float* s_p = reinterpret_cast<float*>(smem + C::OFF_P) + cw * KPW * 4;
  float* s_m = reinterpret_cast<float*>(smem + C::OFF_ML);
  float* s_l = s_m + NCW * RQ_MAX;
  float* s_u = reinterpret_cast<float*>(smem + C::OFF_U);
  const uint32_t q32_base = sbase + C::OFF_Q32;
  int slot = 0, qs = 0;
  uint32_t phase = 0, qph = 0;
  bool ok = true;

  for (long long it = blockIdx.x; it < p.items; it += gridDim.x) {
    Item x = item_rows<RQ>(p, it);
    x.L = 0;
    x.kmin = 0;
    x.t0 = x.t1 = 0;

    // Query rows r0..r0+nr-1 (zero past nr), in log2 units: chunk li of each
    // box in registers, or the whole group as fp32 in shared memory.
    float2 qf[C::QREG ? RQ : 1][C::NB][4];
    if (ok && mbar_wait(bar_qfull + 8 * qs, qph, ab)) {
      const uint8_t* qslot = smem + C::OFF_Q + qs * C::QSLOT;
      const int* hdr = reinterpret_cast<const int*>(qslot + RQ * D * 2);
      x.L = hdr[0];
      x.kmin = hdr[1];
      x.t0 = hdr[2];
      x.t1 = hdr[3];
      if constexpr (C::QREG) {
#pragma unroll
        for (int r = 0; r < RQ; ++r) {
#pragma unroll
          for (int c = 0; c < C::NB; ++c) {
            uint4 w = make_uint4(0, 0, 0, 0);
            if (r < x.nr)
              w = *reinterpret_cast<const uint4*>(qslot + r * D * 2 + c * 128 + li * 16);
            const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 f = bf16x2_to_f2(ws[e]);
              qf[r][c][e] = make_float2(f.x * p.scale_log2, f.y * p.scale_log2);
            }
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_qempty + 8 * qs);
      } else {
        // 128 consumer threads convert RQ*D values, 4 each per round.
        float* q32 = reinterpret_cast<float*>(smem + C::OFF_Q32);
        for (int i = (threadIdx.x - 32) * 4; i < RQ * D; i += 32 * NCW * 4) {
          const int r = i / D;
          float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
          if (r < x.nr) {
            const uint2 w = *reinterpret_cast<const uint2*>(qslot + i * 2);
            const float2 a = bf16x2_to_f2(w.x), b2 = bf16x2_to_f2(w.y);
            f = make_float4(a.x * p.scale_log2, a.y * p.scale_log2, b2.x * p.scale_log2,
                            b2.y * p.scale_log2);
          }
          *reinterpret_cast<float4*>(q32 + i) = f;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_qempty + 8 * qs);
      }
    } else {
      ok = false;
    }
    if (++qs == 2) {
      qs = 0;
      qph ^= 1;
    }
    if constexpr (!C::QREG) named_barrier(1, 32 * NCW);  // q32 complete

    float m[RQ], l[RQ];
    float2 u[RQ][C::NC / 2];
#pragma unroll
    for (int r = 0; r < RQ; ++r) {
      m[r] = -INFINITY;
      l[r] = 0.f;
#pragma unroll
      for (int e = 0; e < C::NC / 2; ++e) u[r][e] = make_float2(0.f, 0.f);
    }

    for (int t = x.t0; t < x.t1 && ok; ++t) {
      if (!mbar_wait(bar_full + 8 * slot, phase, ab)) {
        ok = false;
        break;
      }
      const uint8_t* kb = smem + slot * C::STAGE;
      const uint8_t* vb = kb + C::TILE;

      // Scores of keys 16cw + 4pp + g, rows 0..RQ-1.
      float s[4][RQ];
#pragma unroll
      for (int pp = 0; pp < 4; ++pp) {
        const int j = cw * KPW + pp * 4 + g;
        float2 acc[RQ];
#pragma unroll
        for (int r = 0; r < RQ; ++r) acc[r] = make_float2(0.f, 0.f);
#pragma unroll
        for (int c = 0; c < C::NB; ++c) {
          const uint4 w = *reinterpret_cast<const uint4*>(
              kb + c * C::BOX + j * 128 + ((li ^ (j & 7)) << 4));
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
          if constexpr (C::QREG) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float2 kf = bf16x2_to_f2(ws[e]);
#pragma unroll
              for (int r = 0; r < RQ; ++r)
                fma2(acc[r].x, acc[r].y, qf[r][c][e].x, qf[r][c][e].y, kf.x, kf.y, acc[r].x,
                     acc[r].y);
            }
          } else {
            float2 kf[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) kf[e] = bf16x2_to_f2(ws[e]);
#pragma unroll
            for (int r = 0; r < RQ; ++r) {
              // volatile: read per use, not hoisted into registers for the tile
              float4 qa, qb;
              const uint32_t qa_addr = q32_base + (uint32_t)((r * D + c * 64 + li * 8) * 4);
              asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                           : "=f"(qa.x), "=f"(qa.y), "=f"(qa.z), "=f"(qa.w)
                           : "r"(qa_addr));
              asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];"
                           : "=f"(qb.x), "=f"(qb.y), "=f"(qb.z), "=f"(qb.w)
                           : "r"(qa_addr + 16));
              fma2(acc[r].x, acc[r].y, qa.x, qa.y, kf[0].x, kf[0].y, acc[r].x, acc[r].y);
              fma2(acc[r].x, acc[r].y, qa.z, qa.w, kf[1].x, kf[1].y, acc[r].x, acc[r].y);
              fma2(acc[r].x, acc[r].y, qb.x, qb.y, kf[2].x, kf[2].y, acc[r].x, acc[r].y);
              fma2(acc[r].x, acc[r].y, qb.z, qb.w, kf[3].x, kf[3].y, acc[r].x, acc[r].y);
            }
          }
        }
#pragma unroll
        for (int r = 0; r < RQ; ++r) {
          float v = acc[r].x + acc[r].y;
          v += __shfl_xor_sync(0xffffffffu, v, 1);
          v += __shfl_xor_sync(0xffffffffu, v, 2);
          v += __shfl_xor_sync(0xffffffffu, v, 4);
          s[pp][r] = v;
        }
      }
      // Element mask where the stage reaches past the first row's limit.
      if ((t + 1) * KT > x.kmin) {
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
          const int jg = t * KT + cw * KPW + pp * 4 + g;
#pragma unroll
          for (int r = 0; r < RQ; ++r) {
            const int lim = p.causal ? min(x.L, x.L - p.Nq + x.r0 + r + 1) : x.L;
            if (jg >= lim) s[pp][r] = -INFINITY;
          }
        }
      }
      // Online softmax over the warp's 16 keys; s becomes p in place.  The
      // reference m moves lazily, as in the forward kernel: only when some
      // score exceeds it by more than 8 (log2 units) is the warp max taken
      // and u, l rescaled; otherwise p = 2^(s - m) <= 2^8 with the old m,
      // which leaves u / l unchanged.  A row that has seen no allowed key
      // keeps m = -inf and gets p = 0; exp2(-inf - (-inf)) is never formed.
#pragma unroll
      for (int r = 0; r < RQ; ++r) {
        float mx = fmaxf(fmaxf(s[0][r], s[1][r]), fmaxf(s[2][r], s[3][r]));
        if (__any_sync(0xffffffffu, mx > m[r] + 8.f)) {
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float alpha = fast_exp2(m[r] - mx);  // 0 while m = -inf
          m[r] = mx;
          l[r] *= alpha;
#pragma unroll
          for (int e = 0; e < C::NC / 2; ++e) {
            u[r][e].x *= alpha;
            u[r][e].y *= alpha;
          }
        }
        const float ref = m[r] == -INFINITY ? 0.f : m[r];
        float sum = 0.f;
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
          s[pp][r] = fast_exp2(s[pp][r] - ref);
          sum += s[pp][r];
        }
        l[r] += sum;
      }
      // p of the warp's 16 keys to shared memory, one float4 of rows per key.
      __syncwarp();
      if (li == 0) {
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
          float4 v;
          v.x = s[pp][0];
          v.y = RQ > 1 ? s[pp][RQ > 1 ? 1 : 0] : 0.f;
          v.z = RQ > 2 ? s[pp][RQ > 2 ? 2 : 0] : 0.f;
          v.w = RQ > 3 ? s[pp][RQ > 3 ? 3 : 0] : 0.f;
          reinterpret_cast<float4*>(s_p)[pp * 4 + g] = v;
        }
      }
      __syncwarp();
      // u += p V over the warp's 16 keys; lane owns columns NC*lane .. +NC-1.
      // Slots at or past L are read but replaced by 0 before use (p is 0
      // there too): they may hold anything, including non-finite values.
      // A select rather than a loop exit lets all 16 keys' loads issue at
      // once instead of one dependent round trip per key.
      const int nvalid = min(KPW, max(0, x.L - (t * KT + cw * KPW)));
#pragma unroll
      for (int kk = 0; kk < KPW; ++kk) {
        const bool live = kk < nvalid;
        const int j = cw * KPW + kk;
        const float4 pv = reinterpret_cast<const float4*>(s_p)[kk];
        const float pa[4] = {pv.x, pv.y, pv.z, pv.w};
        if constexpr (D == 128) {
          // columns 4*lane..+3: box lane/16, chunk (lane%16)/2, half lane%2
          uint2 w = *reinterpret_cast<const uint2*>(
              vb + (lane >> 4) * C::BOX + j * 128 + ((((lane & 15) >> 1) ^ (j & 7)) << 4) +
              ((lane & 1) << 3));
          if (!live) w = make_uint2(0u, 0u);
          const float2 v0 = bf16x2_to_f2(w.x), v1 = bf16x2_to_f2(w.y);
#pragma unroll
          for (int r = 0; r < RQ; ++r) {
            fma2(u[r][0].x, u[r][0].y, pa[r], pa[r], v0.x, v0.y, u[r][0].x, u[r][0].y);
            fma2(u[r][1].x, u[r][1].y, pa[r], pa[r], v1.x, v1.y, u[r][1].x, u[r][1].y);
          }
        } else {
          // columns 2*lane, 2*lane+1: chunk lane/4, quarter lane%4
          uint32_t w0 = *reinterpret_cast<const uint32_t*>(
              vb + j * 128 + (((lane >> 2) ^ (j & 7)) << 4) + ((lane & 3) << 2));
          if (!live) w0 = 0u;
          const float2 v0 = bf16x2_to_f2(w0);
#pragma unroll
          for (int r = 0; r < RQ; ++r)
            fma2(u[r][0].x, u[r][0].y, pa[r], pa[r], v0.x, v0.y, u[r][0].x, u[r][0].y);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + 8 * slot);
      if (++slot == C::NS) {
        slot = 0;
        phase ^= 1;
      }
    }

    // ---- merge the four warps' states; warp r writes query row r.
#pragma unroll
    for (int r = 0; r < RQ; ++r) {
      // lanes of a group hold copies of one partial sum: add the 4 groups
      l[r] += __shfl_xor_sync(0xffffffffu, l[r], 8);
      l[r] += __shfl_xor_sync(0xffffffffu, l[r], 16);
      if (lane == 0) {
        s_m[cw * RQ_MAX + r] = m[r];
        s_l[cw * RQ_MAX + r] = l[r];
      }
      float* dst = s_u + (cw * RQ + r) * D + lane * C::NC;
#pragma unroll
      for (int e = 0; e < C::NC / 2; ++e) reinterpret_cast<float2*>(dst)[e] = u[r][e];
    }
    named_barrier(1, 32 * NCW);
    if (cw < x.nr) {
      const int r = cw;
      float mm = -INFINITY;
#pragma unroll
      for (int w = 0; w < NCW; ++w) mm = fmaxf(mm, s_m[w * RQ_MAX + r]);
      float o[C::NC];
#pragma unroll
      for (int e = 0; e < C::NC; ++e) o[e] = 0.f;
      float lse = -INFINITY;
      if (mm != -INFINITY) {
        float lt = 0.f;
#pragma unroll
        for (int w = 0; w < NCW; ++w) {
          const float wt = fast_exp2(s_m[w * RQ_MAX + r] - mm);
          lt = fmaf(wt, s_l[w * RQ_MAX + r], lt);
          const float* src = s_u + (w * RQ + r) * D + lane * C::NC;
#pragma unroll
          for (int e = 0; e < C::NC; ++e) o[e] = fmaf(wt, src[e], o[e]);
        }
        const float inv = 1.f / lt;
#pragma unroll
        for (int e = 0; e < C::NC; ++e) o[e] *= inv;
        lse = (mm + log2f(lt)) * kLn2;
      }
      const long long row = x.bh * p.Nq + x.r0 + r;
      if (p.S == 1) {
        if constexpr (C::NC == 4) {
          uint2 w = make_uint2(pack_bf16(o[0], o[1]), pack_bf16(o[2], o[3]));
          *reinterpret_cast<uint2*>(p.o + row * D + lane * 4) = w;
        } else {
          *reinterpret_cast<uint32_t*>(p.o + row * D + lane * 2) = pack_bf16(o[0], o[1]);
        }
        if (lane == 0) p.lse[row] = lse;
      } else {
        const long long prow = (long long)x.s * p.BH * p.Nq + row;
        float* dst = p.o_part + prow * D + lane * C::NC;
        if constexpr (C::NC == 4)
          *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
        else
          *reinterpret_cast<float2*>(dst) = make_float2(o[0], o[1]);
        if (lane == 0) p.lse_part[prow] = lse;
      }
    }
    named_barrier(1, 32 * NCW);
  }
}

// Merge of S partial results per row: o_part [S][rows][d] fp32 (normalised),
// lse_part [S][rows] (natural log, -inf = empty part) -> o bf16 [rows][d],
// lse fp32 [rows].  One warp per row; every lane carries the running
// (m, l) of the row and the running u of its columns 4*lane + 128*i.  Parts
// are taken eight at a time: all eight LSEs and output rows are loaded
// before any arithmetic (the kernel is bound by memory latency, not
// bandwidth), then the group is folded in with the online-normalisation
// update -- its largest LSE as the group maximum, each part weighted by
// 2^(LSE_s - m).  An empty part has weight 0 and is dropped by a select, so
// whatever its output row holds never reaches the result.
__global__ void __launch_bounds__(256)
    combine_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part, int S,
                   long long rows, int d, __nv_bfloat16* __restrict__ o,
                   float* __restrict__ lse) {
  constexpr int MAXV = 8;  // d <= 1024: up to 8 float4 per lane
  constexpr int G = 8;     // parts per group
  const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const int nv = d / 4;  // float4 per row
  float m = -INFINITY, l = 0.f;
  float4 u[MAXV];
#pragma unroll
  for (int i = 0; i < MAXV; ++i) u[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < S; s0 += G) {
    const int n = min(G, S - s0);
    float ls[G];
#pragma unroll
    for (int g = 0; g < G; ++g)
      ls[g] = g < n ? __ldg(lse_part + (long long)(s0 + g) * rows + row) * kLog2e : -INFINITY;
    if (nv <= 32) {
      // d <= 128: one float4 per lane and part -- load the whole group first
      float4 x[G];
#pragma unroll
      for (int g = 0; g < G; ++g)
        x[g] = (g < n && lane < nv)
                   ? __ldg(reinterpret_cast<const float4*>(
                               o_part + ((long long)(s0 + g) * rows + row) * d) + lane)
                   : make_float4(0.f, 0.f, 0.f, 0.f);
      float mg = m;
#pragma unroll
      for (int g = 0; g < G; ++g) mg = fmaxf(mg, ls[g]);
      if (mg == -INFINITY) continue;  // nothing folded yet and the group is empty
      const float a = fast_exp2(m - mg);  // 0 while m = -inf
      l *= a;
      u[0].x *= a; u[0].y *= a; u[0].z *= a; u[0].w *= a;
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float w = fast_exp2(ls[g] - mg);  // 0 for an empty part
        l += w;
        u[0].x += w != 0.f ? w * x[g].x : 0.f;
        u[0].y += w != 0.f ? w * x[g].y : 0.f;
        u[0].z += w != 0.f ? w * x[g].z : 0.f;
        u[0].w += w != 0.f ? w * x[g].w : 0.f;
      }
      m = mg;
    } else {
      float mg = m;
#pragma unroll
      for (int g = 0; g < G; ++g) mg = fmaxf(mg, ls[g]);
      if (mg == -INFINITY) continue;
      const float a = fast_exp2(m - mg);
      l *= a;
#pragma unroll
      for (int i = 0; i < MAXV; ++i) {
        u[i].x *= a; u[i].y *= a; u[i].z *= a; u[i].w *= a;
      }
      for (int g = 0; g < n; ++g) {
        const float w = fast_exp2(ls[g] - mg);
        l += w;
        if (w == 0.f) continue;  // warp-uniform
        const float4* src =
            reinterpret_cast<const float4*>(o_part + ((long long)(s0 + g) * rows + row) * d);
#pragma unroll
        for (int i = 0; i < MAXV; ++i) {
          const int c = lane + 32 * i;
          if (c < nv) {
            const float4 x = __ldg(src + c);
            u[i].x = fmaf(w, x.x, u[i].x);
            u[i].y = fmaf(w, x.y, u[i].y);
            u[i].z = fmaf(w, x.z, u[i].z);
            u[i].w = fmaf(w, x.w, u[i].w);
          }
        }
      }
      m = mg;
    }
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
  for (int i = 0; i < MAXV; ++i) {
    const int c = lane + 32 * i;
    if (c < nv) {
      uint2 w = make_uint2(pack_bf16(u[i].x * inv, u[i].y * inv),
                           pack_bf16(u[i].z * inv, u[i].w * inv));
      *reinterpret_cast<uint2*>(o + row * d + 4 * c) = w;
    }
  }
  if (lane == 0) lse[row] = l > 0.f ? (m + log2f(l)) * kLn2 : -INFINITY;
}

// ------------------------------------------------------------------ host

// Query rows per pass: 1, 2 or 4 (a fifth row starts a second group that
// re-reads the same K/V tiles, from L2 while the groups run side by side).
static int rows_per_pass(int Nq) { return Nq >= 4 ? 4 : (Nq >= 2 ? 2 : 1); }

template <int D, int RQ>
static cudaError_t launch_split(const Params& p, const void* k, const void* v, int nsm,
                                cudaStream_t st) {
  using C = Cfg<D, RQ>;
  auto kern = kvcache_split_kernel<D, RQ>;
  static std::once_flag once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(once, [&] {
    attr_err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  });
  if (attr_err != cudaSuccess) return attr_err;
  CUtensorMap tk, tv;
  const long long heads = (long long)p.B * p.H;
  if (!make_bf16_map_3d(&tk, k, D, p.Nk, heads, KT) ||
      !make_bf16_map_3d(&tv, v, D, p.Nk, heads, KT))
    return cudaErrorInvalidValue;
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, THREADS, C::SMEM);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  long long grid = (long long)per_sm * nsm;
  if (grid > p.items) grid = p.items;
  kern<<<(unsigned)grid, THREADS, C::SMEM, st>>>(tk, tv, p);
  return cudaGetLastError();
}

template <int D>
static cudaError_t launch_split_d(const Params& p, int rq, const void* k, const void* v,
                                  int nsm, cudaStream_t st) {
  switch (rq) {
    case 1: return launch_split<D, 1>(p, k, v, nsm, st);
    case 2: return launch_split<D, 2>(p, k, v, nsm, st);
    default: return launch_split<D, 4>(p, k, v, nsm, st);
  }
}

static int device_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

static size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

static bool aligned(const void* ptr, size_t a) {
  return (reinterpret_cast<uintptr_t>(ptr) % a) == 0;
}

static int check_sizes(int B, int H, int Nq, int Nk, int d) {
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED;
  const long long bh = (long long)B * H;
  if (bh > 2147483647LL) return FA_ERR_INVALID_ARG;
  if ((double)bh * (Nq > Nk ? Nq : Nk) * d > 4.0e18) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

}  // namespace kvc
}  // namespace fa

using namespace fa;
using namespace fa::kvc;

extern "C" {

int fa_kvcache_num_splits(int B, int H, int Nq, int Nk, int d, int num_sms) {
  if (check_sizes(B, H, Nq, Nk, d) != FA_OK) return 0;
  if (num_sms <= 0) num_sms = device_sms();
  if (num_sms <= 0) return 0;
  const int rq = rows_per_pass(Nq);
  const long long units = (long long)B * H * ((Nq + rq - 1) / rq);
  const long long slots = (long long)(rq == 1 ? 3 : 2) * num_sms;  // resident CTAs
  // At most one split per 4 key tiles (256 keys), at most FA_KVCACHE_MAX_SPLITS.
  long long s_hi = ((long long)Nk + 4 * KT - 1) / (4 * KT);
  if (s_hi > FA_KVCACHE_MAX_SPLITS) s_hi = FA_KVCACHE_MAX_SPLITS;
  if (s_hi < 1) s_hi = 1;
  // Items per resident CTA: about 1.5 for one-row passes (each extra split
  // costs a partial write and a merge, and a little over one round already
  // keeps HBM busy), 8 for multi-row passes (longer per-tile work: many
  // smaller items balance better).  Measured on 128-384 head decode batches.
  const long long want = rq == 1 ? (3 * slots + 1) / 2 : 8 * slots;
  long long S = (want + units - 1) / units;
  if (S > s_hi) S = s_hi;
  if (S < 1) S = 1;
  return (int)S;
}

size_t fa_kvcache_workspace_bytes(int B, int H, int Nq, int Nk, int d, int num_splits) {
  if (check_sizes(B, H, Nq, Nk, d) != FA_OK) return 0;
  if (num_splits == 0) num_splits = fa_kvcache_num_splits(B, H, Nq, Nk, d, 0);
  if (num_splits < 1 || num_splits > FA_KVCACHE_MAX_SPLITS) return 0;
  if (num_splits == 1) return 0;
  const size_t rows = (size_t)B * H * Nq;
  return round_up((size_t)num_splits * rows * d * sizeof(float), 256) +
         round_up((size_t)num_splits * rows * sizeof(float), 256);
}

int fa_combine(const float* o_parts, const float* lse_parts, int num_parts, long long rows,
               int d, void* o, float* lse, void* stream) {
  if (num_parts < 1 || rows < 1 || d < 4 || d > 1024 || d % 4 != 0) return FA_ERR_INVALID_ARG;
  if (!o_parts || !lse_parts || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned(o_parts, 16) || !aligned(lse_parts, 4) || !aligned(o, 8) || !aligned(lse, 4))
    return FA_ERR_INVALID_ARG;
  if ((double)num_parts * rows * d > 4.0e18) return FA_ERR_INVALID_ARG;
  const long long blocks = (rows + 7) / 8;
  if (blocks > 2147483647LL) return FA_ERR_INVALID_ARG;
  combine_kernel<<<(unsigned)blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      o_parts, lse_parts, num_parts, rows, d, static_cast<__nv_bfloat16*>(o), lse);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

int fa_forward_kvcache(const void* q, const void* k_cache, const void* v_cache, void* o,
                       float* lse, int B, int H, int Nq, int Nk, int d, float scale,
                       int causal, const int32_t* cache_len, int num_splits, void* workspace,
                       size_t workspace_bytes, void* stream) {
  int st = check_sizes(B, H, Nq, Nk, d);
  if (st != FA_OK) return st;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (!q || !k_cache || !v_cache || !o || !lse) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(o, 16) ||
      !aligned(lse, 4) || !aligned(cache_len, 4))
    return FA_ERR_INVALID_ARG;
  if (num_splits < 0 || num_splits > FA_KVCACHE_MAX_SPLITS) return FA_ERR_INVALID_ARG;
  // With an explicit split count every argument is checked before any CUDA
  // call; the automatic choice needs the device's multiprocessor count.
  if (num_splits > 1) {
    if (!workspace || !aligned(workspace, 256)) return FA_ERR_INVALID_ARG;
    if (workspace_bytes < fa_kvcache_workspace_bytes(B, H, Nq, Nk, d, num_splits))
      return FA_ERR_INVALID_ARG;
  }
  const int nsm = device_sms();
  if (nsm <= 0) return FA_ERR_CUDA;
  const int S = num_splits == 0 ? fa_kvcache_num_splits(B, H, Nq, Nk, d, nsm) : num_splits;
  if (S < 1) return FA_ERR_INVALID_ARG;
  const size_t rows = (size_t)B * H * Nq;
  if (S > 1) {
    if (!workspace || !aligned(workspace, 256)) return FA_ERR_INVALID_ARG;
    if (workspace_bytes < fa_kvcache_workspace_bytes(B, H, Nq, Nk, d, S))
      return FA_ERR_INVALID_ARG;
  }
  Params p;
  p.B = B;
  p.H = H;
  p.Nq = Nq;
  p.Nk = Nk;
  p.BH = (long long)B * H;
  p.S = S;
  const int rq = rows_per_pass(Nq);
  p.QG = (Nq + rq - 1) / rq;
  p.items = (long long)B * H * S * p.QG;
  p.scale_log2 = scale * kLog2e;
  p.causal = causal ? 1 : 0;
  p.cache_len = cache_len;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.o = static_cast<__nv_bfloat16*>(o);
  p.lse = lse;
  p.o_part = S > 1 ? static_cast<float*>(workspace) : nullptr;
  p.lse_part = S > 1 ? reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                                round_up((size_t)S * rows * d * sizeof(float), 256))
                     : nullptr;
  p.status = status_word();
  if (p.status == nullptr) return FA_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = d == 64 ? launch_split_d<64>(p, rq, k_cache, v_cache, nsm, s)
                          : launch_split_d<128>(p, rq, k_cache, v_cache, nsm, s);
  if (e != cudaSuccess) return FA_ERR_CUDA;
  if (S == 1) return FA_OK;
  return fa_combine(p.o_part, p.lse_part, S, (long long)rows, d, o, lse, stream);
}

}  // extern "C"
