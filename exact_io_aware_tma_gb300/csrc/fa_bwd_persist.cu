// Persistent form of the attention backward's dK/dV kernel at d = 64 (padded
// layout, no dropout), sm_103a.
//
// The same per-step work as the one-CTA-per-key-tile kernel (fa_bwd_tc.cu:
// S^T = K Q^T, dP^T = V dO^T, P^T and dS^T rebuilt from the stored row
// statistics, dV += P^T dO, dK += dS^T Q, dQ^T = K^T dS^T added into the fp32
// dQ accumulator; page "FlashAttention IO-aware explained", section
// "Recomputation and IO complexity"), with the same warp roles, TMEM columns
// and step pipeline.  What differs is the schedule.  At d = 64 a key tile's
// work is short (2-16 steps of ~1 us for N <= 1024), and with one CTA per
// key tile each CTA paid its set-up (barriers, TMEM, the live bitmask), the
// ~1.2 us gap before the next CTA of the SM started, the latency of its
// first K, V, Q, dO loads and its epilogue in series with the work: about a
// quarter of the kernel.  Here one CTA per SM walks work items -- its first
// is its block index, later ones come from a counter in the workspace
// (cleared by the preprocess), in the same grouped, heaviest-first order the
// hardware gave the CTAs -- and:
//   - the producer warp publishes each item (key tile, head, split part and
//     its live bitmask) in one of two shared buffers as soon as it has
//     issued the previous item's loads, so every role finds it ready;
//   - K and V are double-buffered, so the next item's K, V and first steps
//     load while the current item runs; the ring of step stages and every
//     per-step barrier carry on across items (the roles count steps per CTA);
//   - dK and dV of an item leave through that item's K/V buffer (its
//     products are done by then), which the producer refills only after the
//     store has read it, and the next item's first dV, dK products wait only
//     until the epilogue has read the accumulators out of TMEM.
//
// Warp roles (512 threads): warp 0 producer (all lanes publish items, lane 0
// issues the loads); warps 1, 2 the two MMA issuers (warp 1 owns TMEM);
// warps 4-7 and 12-15 the element-wise groups (queries 0-31 and 32-63 of
// each step; group 0 also runs each item's epilogue); warps 8, 9 the dQ
// warps (TMEM lanes 0-63 = the head dimensions); warps 3, 10, 11 idle.
// TMEM columns: dV [0,64), dK [64,128), S[b] = 128 + 64b, dP[b] = 256 + 64b,
// dQ[b] = 384 + 64b.
#include <cuda_bf16.h>

#include "fa_common.cuh"
#include "fa_kernels.h"
#include "fa_sm100.cuh"
#include "fa_tma_host.h"

namespace fa {
using namespace sm100;

namespace {

struct PTc {
  static constexpr int D = 64;
  static constexpr int BQ = 64;                  // query rows per step
  static constexpr int QH = 32;                  // queries per element-wise group and step
  static constexpr int THREADS = 512;
  static constexpr int DQ_WARPS = 2;             // dQ warps holding TMEM lanes below d
  static constexpr int NS = 4;                   // step stages
  static constexpr int HALF_K = 128 * 128;       // [128 rows][64 cols] bf16 box
  static constexpr int HALF_Q = 64 * 128;        // [64 rows][64 cols] bf16 box
  static constexpr int KT = 128 * D * 2;         // K or V tile
  static constexpr int KVB = 2 * KT;             // K, V of one work item
  static constexpr int QB = BQ * D * 2;          // Q or dO block
  static constexpr int STAGE = 2 * QB;           // Q, dO of one step
  static constexpr int OFF_KV = 0;               // two K/V buffers
  static constexpr int OFF_ST = 2 * KVB;
  static constexpr int OFF_VEC = OFF_ST + NS * STAGE;  // [NS][LSE*log2e (64), D (64)]
  static constexpr int OFF_DS = (OFF_VEC + NS * 512 + 1023) / 1024 * 1024;
  static constexpr int DS = 128 * BQ * 2;        // dS^T [128 keys][64 q] bf16, x2
  static constexpr int OFF_BAR = OFF_DS + 2 * DS;
  // B_KV[b]: K/V buffer b loaded; B_FULL/B_EMPTY: the step ring (a step's
  // release, after its dK, also says that its dV has read P^T out of S
  // buffer b); B_S[b]: S^T, dP^T of buffer b computed; B_EW[b]: P^T, dS^T of
  // buffer b written; B_DQF/B_DQE[b]: dQ^T buffer b computed / read out
  // (dS^T buffer b is free once B_DQF[b] completes: dQ^T is its last
  // reader); B_FIN: an item's dK, dV complete; B_DRAIN: per issuer, its last
  // products done; B_ITEM[b]: item published in buffer b; B_ITEMF[b]: every
  // role done with it; B_KVF[b]: K/V buffer b free (its item's products and
  // dK/dV store done); B_ACCF: dK, dV read out of TMEM.
  static constexpr int B_KV = 0, B_FULL = 2, B_EMPTY = 2 + NS, B_S = 2 + 2 * NS, B_EW = B_S + 2,
                       B_DQF = B_EW + 2, B_DQE = B_DQF + 2, B_FIN = B_DQE + 2,
                       B_DRAIN = B_FIN + 1, B_ITEM = B_DRAIN + 2,
                       B_ITEMF = B_ITEM + 2, B_KVF = B_ITEMF + 2, B_ACCF = B_KVF + 2,
                       NBAR = B_ACCF + 1;
  // misc: TMEM address (+0), abort flag (+16), two PItem buffers (+64)
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  // live query tiles of an item's range under a block mask, one bit each,
  // one buffer per published item
  static constexpr int OFF_LIVE = (OFF_MISC + 128 + 127) / 128 * 128;
  static constexpr int LIVEB = 65536 / 8;
  // the step's dQ rows, [64 rows][32 columns] fp32 per dQ warp, two buffers,
  // added into the accumulator by TMA reduce-adds
  static constexpr int DQW = BQ * 32 * 4;
  static constexpr int DQS = 2 * DQW;
  static constexpr int OFF_DQS = (OFF_LIVE + 2 * LIVEB + 1023) / 1024 * 1024;
  static constexpr int SMEM = OFF_DQS + 2 * DQS + 1024;
  static constexpr int COL_DV = 0, COL_DK = D, COL_S = 2 * D, COL_DP = 2 * D + 128,
                       COL_DQ = 2 * D + 256;
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(COL_DQ + 128 <= 512, "TMEM columns");
  static_assert(SMEM <= 232448, "shared memory budget");
};

// A work item: key tile kt of head bh; a part of a split key tile covers
// query tiles [qa, qb] (meta: part | parts << 8 | first slot << 16).
// kt < 0: no more work.
struct PItem {
  int kt, bh, qa, qb, meta, pad[3];
};

// Work item w in the grouped, heaviest-first order (the order of the
// one-CTA-per-item grid); false for a split rank past the plan's item count.
template <bool SPLIT>
__device__ __forceinline__ bool decode_item(const Problem& p, long long w, const BwdSplit& sp,
                                            PItem& it) {
  long long bh;
  int r;
  if constexpr (SPLIT) {
    grouped_cta(p, w, p.T * kSplitMax, bh, r);
    if (r >= __ldg(sp.nitems)) return false;
    const int4 x = __ldg(sp.items + r);
    it.kt = x.x;
    it.qa = x.y;
    it.qb = x.z;
    it.meta = x.w;
  } else {
    grouped_cta(p, w, p.T, bh, r);
    it.kt = r;
    it.qa = 0;
    it.qb = -1;
    it.meta = 1 << 8;
  }
  it.bh = (int)bh;
  return true;
}

// Next 64-row query step after (qt, sub) of key tile kt: the live query
// tiles of its range in ascending order, two halves each, skipping halves
// past N; under a block mask from the item's bitmask `live` (bit t: query
// tile first + t).
__device__ __forceinline__ bool next_step(const Problem& p, int kt, int klim,
                                          const uint32_t* live, int& qt, int& sub) {
  if (qt >= 0 && sub == 0 && qt * 128 + 64 < p.N) {
    sub = 1;
    return true;
  }
  sub = 0;
  int qf, ql;
  ktile_query_tiles(p, kt, klim, qf, ql);
  qt = qt < 0 ? qf : qt + 1;
  if (p.block_mask == nullptr) return qt <= ql;
  while (qt <= ql) {
    const int t = qt - qf;
    const uint32_t w = live[t >> 5] >> (t & 31);  // bits past the range are 0
    if (w != 0) {
      qt += __ffs(w) - 1;
      return true;
    }
    qt += 32 - (t & 31);
  }
  return false;
}

// LOSE: self-test instantiation only (fa_selftest_backward_lost_signal at
// d = 64): warp 4 withholds its arrival for the CTA's first step and every
// wait gives up after 1 ms, so the gradient issuer's wait runs out and the
// abort, drain and status paths run.
template <bool SPLIT, bool LOSE = false>
__global__ void __launch_bounds__(PTc::THREADS, 1)
    bwd_persist_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_dk,
                       const __grid_constant__ CUtensorMap tm_dv,
                       const __grid_constant__ CUtensorMap tm_dq, const Problem p,
                       const float* __restrict__ lse2, const float* __restrict__ dvec, int npad,
                       const BwdSplit sp, unsigned long long* __restrict__ next_item) {
  using C = PTc;
  constexpr int D = C::D, QH = C::QH;
  PItem first;
  if (!decode_item<SPLIT>(p, blockIdx.x, sp, first)) first.kt = -1;  // fetch another
  extern __shared__ uint8_t smem_raw[];
  // An offset (not an integer round trip) keeps the pointer visibly in shared
  // memory, so C++ accesses through it compile to shared-memory instructions.
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t s0 = smem_u32(smem);
  const uint32_t bar0 = s0 + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 16);
  volatile PItem* info = reinterpret_cast<volatile PItem*>(smem + C::OFF_MISC + 64);
  const Abort ab{abort_flag, p.status, LOSE ? kShortWaitLimitNs : kWaitLimitNs};
  // item n's live bitmask and K/V buffer
  auto live_of = [&](int n) {
    return reinterpret_cast<const uint32_t*>(smem + C::OFF_LIVE + (n & 1) * C::LIVEB);
  };
  auto kv_of = [&](int n) { return s0 + C::OFF_KV + (n & 1) * C::KVB; };
  // Item n as the producer published it in buffer n % 2; false once there is
  // no more work (or on abort).
  auto get_item = [&](int n, PItem& it, bool& ok, uint32_t hint) -> bool {
    if (!(ok = mbar_wait(bar(C::B_ITEM + (n & 1)), (n >> 1) & 1, ab, hint))) return false;
    const volatile PItem& v = info[n & 1];
    it.kt = v.kt;
    it.bh = v.bh;
    it.qa = v.qa;
    it.qb = v.qb;
    it.meta = v.meta;
    return it.kt >= 0;
  };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (warp == 0) {
    // the barriers, one per lane of warp 0
    for (int i = lane; i < C::NBAR; i += 32) {
      int cnt = 1;
      if (i == C::B_EW || i == C::B_EW + 1) cnt = 8;
      if (i == C::B_DQE || i == C::B_DQE + 1) cnt = C::DQ_WARPS;
      if (i == C::B_ITEMF || i == C::B_ITEMF + 1) cnt = 2 + 8 + C::DQ_WARPS;
      if (i == C::B_KVF || i == C::B_KVF + 1) cnt = 2;
      if (i == C::B_ACCF) cnt = 4;
      mbar_init(bar(i), cnt);
    }
    fence_barrier_init();
    __syncwarp();
  }
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    // K and V of the first item, issued before the rest of the set-up
    if (first.kt >= 0) {
      mbar_expect_tx(bar(C::B_KV), 2 * C::KT);
      tma_load_3d(kv_of(0), &tm_k, bar(C::B_KV), 0, first.kt * 128, first.bh);
      tma_load_3d(kv_of(0) + C::KT, &tm_v, bar(C::B_KV), 0, first.kt * 128, first.bh);
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    prefetch_tensormap(&tm_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Every lane fetches and publishes the items (the live bitmask by
    // ballots); lane 0 issues their loads.
    griddep_wait();  // the preprocess's LSE, D rows and the counter it cleared
    if (lane == 0) griddep_release();
    const long long nwork = (long long)p.B * p.H * p.T * (SPLIT ? kSplitMax : 1);
    auto fetch = [&](PItem& it) {
      for (;;) {
        unsigned long long w = 0;
        if (lane == 0) w = gridDim.x + atomicAdd(next_item, 1ull);
        w = __shfl_sync(0xffffffffu, w, 0);
        if (w >= (unsigned long long)nwork) {
          it.kt = -1;
          return;
        }
        if (decode_item<SPLIT>(p, (long long)w, sp, it)) return;
      }
    };
    int slot = 0, round = 0;
    // K/V loads issued into buffers 0 and 1 (two scalars: an indexed array
    // would live in local memory)
    int kv_uses0 = first.kt >= 0 ? 1 : 0, kv_uses1 = 0;
    PItem it = first;
    bool ok = true;
    for (int n = 0; ok; ++n) {
      const int ib = n & 1;
      if (n > 0 || it.kt < 0) fetch(it);
      // buffer ib last held item n - 2: every role must be done with it
      if (n >= 2) {
        bool w_ok = true;
        if (lane == 0) w_ok = mbar_wait(bar(C::B_ITEMF + ib), ((n - 2) >> 1) & 1, ab, kSleepHintNs);
        if (!__shfl_sync(0xffffffffu, w_ok, 0)) break;
      }
      const int klim = it.kt >= 0 ? key_limit(p, it.bh / p.H) : 0;
      if (it.kt >= 0 && p.block_mask != nullptr) {
        int qf, ql;
        ktile_query_tiles(p, it.kt, klim, qf, ql);
        const int cnt = ql - qf + 1;
        uint32_t* lv = const_cast<uint32_t*>(live_of(n));
        for (int wi = 0; wi < ((cnt + 31) >> 5); ++wi) {
          const int t = (wi << 5) + lane;
          const bool in_part = !SPLIT || (qf + t >= it.qa && qf + t <= it.qb);
          const uint32_t bits =
              __ballot_sync(0xffffffffu, t < cnt && in_part && tile_live(p, qf + t, it.kt, klim));
          if (lane == 0) lv[wi] = bits;
        }
      }
      if (lane == 0) {
        info[ib].kt = it.kt;
        info[ib].bh = it.bh;
        info[ib].qa = it.qa;
        info[ib].qb = it.qb;
        info[ib].meta = it.meta;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_ITEM + ib));
      if (it.kt < 0) break;
      if (lane == 0) {
        const int kb = n & 1;
        if (n > 0 || kv_uses0 == 0) {
          // K/V buffer kb: its previous item's products and dK/dV store are
          // done with it
          const int uses = kb ? kv_uses1 : kv_uses0;
          if (uses > 0 && !mbar_wait(bar(C::B_KVF + kb), (uses - 1) & 1, ab, kSleepHintNs))
            ok = false;
          if (ok) {
            mbar_expect_tx(bar(C::B_KV + kb), 2 * C::KT);
            tma_load_3d(kv_of(n), &tm_k, bar(C::B_KV + kb), 0, it.kt * 128, it.bh);
            tma_load_3d(kv_of(n) + C::KT, &tm_v, bar(C::B_KV + kb), 0, it.kt * 128, it.bh);
            if (kb)
              ++kv_uses1;
            else
              ++kv_uses0;
          }
        }
        // Q, dO and the 64 LSE / D values of each step into the next stage
        const size_t vec_base = (size_t)it.bh * npad;
        int qt = -1, sub = 0;
        while (ok && next_step(p, it.kt, klim, live_of(n), qt, sub)) {
          const int q0 = qt * 128 + sub * 64;
          if (!(ok = mbar_wait(bar(C::B_EMPTY + slot), (round & 1) ^ 1, ab, kSleepHintNs))) break;
          const uint32_t st = s0 + C::OFF_ST + slot * C::STAGE;
          const uint32_t fb = bar(C::B_FULL + slot);
          const uint32_t vb = s0 + C::OFF_VEC + slot * 512;
          mbar_expect_tx(fb, 2 * C::QB + 512);
          tma_load_3d(st, &tm_q, fb, 0, q0, it.bh);
          tma_load_3d(st + C::QB, &tm_do, fb, 0, q0, it.bh);
          bulk_load(vb, lse2 + vec_base + q0, 256, fb);
          bulk_load(vb + 256, dvec + vec_base + q0, 256, fb);
          if (++slot == C::NS) {
            slot = 0;
            ++round;
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (lane == 0) {
      // Drain every load issued before shared memory is released.
      for (int s = 0; s < C::NS; ++s) {
        const int last = round - (s >= slot ? 1 : 0);
        if (last >= 0) {
          const uint64_t t0 = globaltimer();
          while (!mbar_try_wait(bar(C::B_FULL + s), last & 1) &&
                 globaltimer() - t0 < kWaitLimitNs) {
          }
        }
      }
      for (int kb = 0; kb < 2; ++kb) {
        const int uses = kb ? kv_uses1 : kv_uses0;
        if (uses > 0) {
          const uint64_t t0 = globaltimer();
          while (!mbar_try_wait(bar(C::B_KV + kb), (uses - 1) & 1) &&
                 globaltimer() - t0 < kWaitLimitNs) {
          }
        }
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    //   warp 1: S^T(j), dP^T(j) into buffer j % 2 (owns TMEM);
    //   warp 2: dV(i), dK(i), dQ^T(i) into dQ[i % 2].
    // S^T(j) waits until dV(j-2) has read P^T(j-2) from the same columns
    // (the release of step j-2's stage, committed after its dK, says so);
    // dQ^T(i) until the dQ warps have read dQ^T(i-2) out.  j, i count the
    // CTA's steps (across items); dV and dK accumulate from each item's
    // first step.
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(128, C::BQ, false, false);
      constexpr uint32_t id_kv = idesc_bf16(128, D, false, true);
      constexpr uint32_t id_q = idesc_bf16(128, C::BQ, true, true);
      constexpr uint32_t st_step = C::STAGE >> 4, qb_step = C::QB >> 4, ds_step = C::DS >> 4;
      const uint64_t dst_k = sdesc_sw128(s0 + C::OFF_ST, 16, 1024);          // stage 0 Q, K-major
      const uint64_t dst_mn = sdesc_sw128(s0 + C::OFF_ST, C::HALF_Q, 1024);  // stage 0 Q, MN-major
      const uint64_t dds = sdesc_sw128(s0 + C::OFF_DS, 16, 1024);            // dS^T buffer 0
      const uint32_t t_dv = tmem + C::COL_DV, t_dk = tmem + C::COL_DK;
      int J = 0;  // steps of the earlier items
      bool ok = true;
      PItem it;
      for (int n = 0; ok && get_item(n, it, ok, kPollHintNs); ++n) {
        const uint64_t dk_k = sdesc_sw128(kv_of(n), 16, 1024);            // K, K-major
        const uint64_t dv_k = sdesc_sw128(kv_of(n) + C::KT, 16, 1024);    // V, K-major
        const uint64_t dk_mn = sdesc_sw128(kv_of(n), C::HALF_K, 1024);    // K^T, MN-major
        // only the number of steps matters to the issuers, counted up front
        const int klim = key_limit(p, it.bh / p.H);
        int nsteps = 0;
        for (int qt = -1, sub = 0; next_step(p, it.kt, klim, live_of(n), qt, sub);) ++nsteps;
        mbar_arrive(bar(C::B_ITEMF + (n & 1)));
        if (!(ok = mbar_wait(bar(C::B_KV + (n & 1)), (n >> 1) & 1, ab))) break;
        tc_fence_after();
        if (warp == 1) {
          for (int jj = 0; ok && jj < nsteps; ++jj) {
            const int j = J + jj;
            const int bf = j & 1;
            const uint64_t sq = dst_k + (uint64_t)((j % C::NS) * st_step);
            if (!(ok = mbar_wait(bar(C::B_FULL + j % C::NS), (j / C::NS) & 1, ab))) break;
            if (j >= 2 &&
                !(ok = mbar_wait(bar(C::B_EMPTY + (j - 2) % C::NS), ((j - 2) / C::NS) & 1, ab)))
              break;
            tc_fence_after();
            mma_ss_kmajor_k64_a16k_b8k(tmem + C::COL_S + 64 * bf, dk_k, sq, id_s, 0);
            mma_ss_kmajor_k64_a16k_b8k(tmem + C::COL_DP + 64 * bf, dv_k, sq + qb_step, id_s, 0);
            mma_commit(bar(C::B_S + bf));
          }
        } else {
          // the epilogue has read the previous item's dK, dV out of TMEM
          if (n > 0) {
            if (!(ok = mbar_wait(bar(C::B_ACCF), (n - 1) & 1, ab))) break;
            tc_fence_after();
          }
          for (int ii = 0; ok && ii < nsteps; ++ii) {
            const int i = J + ii;
            const int bf = i & 1;
            const uint64_t sq_mn = dst_mn + (uint64_t)((i % C::NS) * st_step);
            const uint64_t ds = dds + (uint64_t)(bf * ds_step);
            if (!(ok = mbar_wait(bar(C::B_EW + bf), (i >> 1) & 1, ab))) break;
            tc_fence_after();
            // dV += P^T dO   (P^T: bf16 in TMEM over S[bf], the two groups'
            // halves 32 columns apart; dO as MN-major B)
            mma_ts_mn_k64_gap32(t_dv, tmem + C::COL_S + 64 * bf, sq_mn + qb_step, id_kv, ii > 0);
            // dK += dS^T Q
            mma_ss_kmajor_mn_k64(t_dk, ds, sq_mn, id_kv, ii > 0);
            mma_commit(bar(C::B_EMPTY + i % C::NS));
            // dQ^T = K^T dS^T into dQ[bf], once dQ^T(i-2) has been read out
            if (i >= 2) {
              if (!(ok = mbar_wait(bar(C::B_DQE + bf), ((i - 2) >> 1) & 1, ab))) break;
              tc_fence_after();
            }
            mma_ss_mn_mn_k128(tmem + C::COL_DQ + 64 * bf, dk_mn, ds, id_q, 0);
            mma_commit(bar(C::B_DQF + bf));
          }
          // dK and dV are complete once this thread's last products are (the
          // other issuer's finished before they could start), and so is
          // every read of the item's K/V buffer
          mma_commit(bar(C::B_FIN));
          mma_commit(bar(C::B_KVF + (n & 1)));
        }
        J += nsteps;
      }
      mma_commit(bar(C::B_DRAIN + warp - 1));
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(bar(C::B_DRAIN + warp - 1), 0) && globaltimer() - t0 < kWaitLimitNs) {
      }
    }
  } else if ((warp >= 4 && warp < 8) || warp >= 12) {
    // ------------------------------------------------------------ element-wise
    // group g (warps 4-7, 12-15) takes the step's queries qo .. qo + 31
    const int g = warp >= 12 ? 1 : 0;
    const int qo = g * QH;
    const int r = ((warp & 3) << 5) + lane;  // key row within the tile
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const float cl2 = p.scale_log2;
    int J = 0;  // steps of the earlier items
    bool ok = true;
    PItem it;
    for (int n = 0; ok && get_item(n, it, ok, kPollHintNs); ++n) {
      const int kt = it.kt, bh = it.bh;
      const int klim = key_limit(p, bh / p.H);
      const int j = kt * 128 + r;  // key index
      int qt = -1, sub = 0, i = 0;
      for (; next_step(p, kt, klim, live_of(n), qt, sub); ++i) {
        const int s = J + i;  // the CTA's step index
        const int bf = s & 1;
        const int q0 = qt * 128 + sub * 64;
        const uint8_t* vb = smem + C::OFF_VEC + (s % C::NS) * 512;
        const float* l2 = reinterpret_cast<const float*>(vb) + qo;
        const float* dv = reinterpret_cast<const float*>(vb + 256) + qo;
        if (!(ok = mbar_wait(bar(C::B_S + bf), (s >> 1) & 1, ab))) break;
        tc_fence_after();
        uint32_t sr[QH], pr[QH];
        tmem_ld32(lane_base + C::COL_S + 64 * bf + qo, sr);
        tmem_ld32(lane_base + C::COL_DP + 64 * bf + qo, pr);
        // queries c of the step allowed for this key: lo <= c < hi.  Only
        // whether the step has disallowed queries is kept through the loop;
        // they are zeroed in the packed words afterwards.
        auto q_range = [&](int& lo, int& hi) {
          lo = 64;
          hi = 64;
          if (j < klim) {
            lo = max(0, col_q_lo(p, j) - q0);
            hi = min(64, col_q_hi(p, j) + 1 - q0);
          }
        };
        bool edge;
        {
          int lo, hi;
          q_range(lo, hi);
          edge = lo > qo || hi < qo + QH;
        }
        uint32_t pk[QH / 2], dk[QH / 2];
#pragma unroll
        for (int c4 = 0; c4 < QH / 4; ++c4) {
          const float4 L = reinterpret_cast<const float4*>(l2)[c4];
          const float4 Dd = reinterpret_cast<const float4*>(dv)[c4];
          float x0, x1, x2, x3;
          fma2(x0, x1, __uint_as_float(sr[4 * c4]), __uint_as_float(sr[4 * c4 + 1]), cl2, cl2,
               -L.x, -L.y);
          fma2(x2, x3, __uint_as_float(sr[4 * c4 + 2]), __uint_as_float(sr[4 * c4 + 3]), cl2,
               cl2, -L.z, -L.w);
          const float p0 = fast_exp2(x0), p1 = fast_exp2(x1), p2 = fast_exp2(x2),
                      p3 = fast_exp2(x3);
          float e0, e1, e2, e3;
          add2(e0, e1, __uint_as_float(pr[4 * c4]), __uint_as_float(pr[4 * c4 + 1]), -Dd.x,
               -Dd.y);
          add2(e2, e3, __uint_as_float(pr[4 * c4 + 2]), __uint_as_float(pr[4 * c4 + 3]), -Dd.z,
               -Dd.w);
          pk[2 * c4] = pack_bf16(p0, p1);
          pk[2 * c4 + 1] = pack_bf16(p2, p3);
          dk[2 * c4] = pack_bf16(p0 * e0, p1 * e1);
          dk[2 * c4 + 1] = pack_bf16(p2 * e2, p3 * e3);
        }
        if (edge) {
          // disallowed queries: P and dS are 0 (the values computed for them
          // above, possibly non-finite, are discarded half-word by half-word)
          int lo, hi;
          q_range(lo, hi);
          lo -= qo;
          hi -= qo;
#pragma unroll
          for (int w = 0; w < QH / 2; ++w) {
            const uint32_t keep = ((2 * w >= lo && 2 * w < hi) ? 0x0000ffffu : 0u) |
                                  ((2 * w + 1 >= lo && 2 * w + 1 < hi) ? 0xffff0000u : 0u);
            pk[w] &= keep;
            dk[w] &= keep;
          }
        }
        // P^T (bf16 pairs) over the group's own S^T columns (0-15 and 32-47:
        // each group overwrites only columns it has already read)
        tmem_st16(lane_base + C::COL_S + 64 * bf + qo, pk);
        // dS^T row r into the 128-byte-swizzled buffer bf, once dK / dQ^T of
        // step s-2 (which read this buffer) have completed: the commit after
        // dQ^T, the last of them, covers both.
        if (s >= 2) {
          if (!(ok = mbar_wait(bar(C::B_DQF + bf), ((s - 2) >> 1) & 1, ab))) break;
        }
        uint8_t* dsb = smem + C::OFF_DS + bf * C::DS + r * 128;
#pragma unroll
        for (int c8 = 0; c8 < QH / 8; ++c8)
          *reinterpret_cast<uint4*>(dsb + (((c8 + qo / 8) ^ (r & 7)) << 4)) =
              make_uint4(dk[4 * c8], dk[4 * c8 + 1], dk[4 * c8 + 2], dk[4 * c8 + 3]);
        fence_proxy_async_smem();
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && !(LOSE && s == 0 && warp == 4)) mbar_arrive(bar(C::B_EW + bf));
      }
      if (g == 0) {
        // ---- epilogue: dK (x scale), dV out of TMEM; a part of a split key
        // tile stores its fp32 rows (0 if it ran no step) into its slot for
        // the join kernel, a whole key tile goes to bf16 through the item's
        // K/V buffer and a TMA store
        if (ok) ok = mbar_wait(bar(C::B_FIN), n & 1, ab);
        tc_fence_after();
        const bool have = i > 0 && ok;
        bool emit = true;
        if constexpr (SPLIT) {
          const int meta = info[n & 1].meta;  // the buffer is held until the arrival below
          if (((meta >> 8) & 0xff) > 1) {
            float* mine =
                sp.slots +
                (((size_t)bh * kSplitSlots + (meta >> 16) + (meta & 0xff)) * 2 * 128 + r) * D;
            for (int t = 0; t < 2; ++t) {
#pragma unroll 1
              for (int c = 0; c < D / 32; ++c) {
                uint32_t o[32];
                if (have) {
                  tmem_ld32(lane_base + (t == 0 ? C::COL_DK : C::COL_DV) + 32 * c, o);
                } else {
#pragma unroll
                  for (int e = 0; e < 32; ++e) o[e] = 0u;
                }
#pragma unroll
                for (int e = 0; e < 8; ++e)
                  reinterpret_cast<uint4*>(mine + t * 128 * D + 32 * c)[e] =
                      make_uint4(o[4 * e], o[4 * e + 1], o[4 * e + 2], o[4 * e + 3]);
              }
            }
            emit = false;
          }
        }
        uint8_t* stg = smem + (kv_of(n) - s0);  // dK tile, then dV tile
#pragma unroll
        for (int t = 0; t < 2 && emit; ++t) {
          const uint32_t col = t == 0 ? C::COL_DK : C::COL_DV;
          const float mul = t == 0 ? p.scale : 1.f;
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            if (have) {
              tmem_ld32(lane_base + col + 32 * c, o);
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) o[e] = 0u;
            }
            uint32_t pw[16];
#pragma unroll
            for (int e = 0; e < 16; ++e)
              pw[e] =
                  pack_bf16(__uint_as_float(o[2 * e]) * mul, __uint_as_float(o[2 * e + 1]) * mul);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int cc = 4 * c + q;
              uint8_t* dst = stg + t * C::KT + r * 128 + (((cc & 7) ^ (r & 7)) << 4);
              *reinterpret_cast<uint4*>(dst) =
                  make_uint4(pw[4 * q], pw[4 * q + 1], pw[4 * q + 2], pw[4 * q + 3]);
            }
          }
        }
        // dK, dV are out of TMEM: the next item's first products may
        // overwrite them
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_ACCF));
        fence_proxy_async_smem();
        named_barrier(1, 128);
        if (r == 0) {
          if (ok && emit) {
            tma_store_3d(&tm_dk, smem_u32(stg), 0, kt * 128, bh);
            tma_store_3d(&tm_dv, smem_u32(stg) + C::KT, 0, kt * 128, bh);
            tma_store_commit();
            tma_store_wait_read();  // shared memory read out; the writes finish with the grid
          }
          mbar_arrive(bar(C::B_KVF + (n & 1)));
        }
      }
      // done with item n's buffer (its bitmask, and the part word above)
      if (lane == 0) mbar_arrive(bar(C::B_ITEMF + (n & 1)));
      J += i;
    }
  } else if (warp == 8 || warp == 9) {
    // ------------------------------------------------------------ dQ
    // one head-dimension row per thread (TMEM lane = warp's quadrant + lane):
    // each warp stages its 32 head dimensions of the step's 64 query rows in
    // shared memory (a warp instruction stores 32 consecutive floats of one
    // row: conflict-free) and its lane 0 adds the tile into the accumulator
    // with one TMA reduce-add (rows outside the tensor are skipped).  The
    // buffer of step s is rewritten at step s + 2, once that reduce has read
    // it.
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    int J = 0;  // steps of the earlier items
    bool ok = true;
    griddep_wait();  // the accumulator the preprocess cleared
    PItem it;
    for (int n = 0; ok && get_item(n, it, ok, kSleepHintNs); ++n) {
      const int bh = it.bh;
      const int klim = key_limit(p, bh / p.H);
      int qt = -1, sub = 0, i = 0;
      for (; next_step(p, it.kt, klim, live_of(n), qt, sub); ++i) {
        const int s = J + i;  // the CTA's step index
        const int bf = s & 1;
        const int q0 = qt * 128 + sub * 64;
        if (!(ok = mbar_wait(bar(C::B_DQF + bf), (s >> 1) & 1, ab, kSleepHintNs))) break;
        tc_fence_after();
        uint32_t v[64];
        tmem_ld64(lane_base + C::COL_DQ + 64 * bf, v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(C::B_DQE + bf));
        float* stg =
            reinterpret_cast<float*>(smem + C::OFF_DQS + (s & 1) * C::DQS + (warp & 3) * C::DQW);
        if (lane == 0 && s >= 2) bulk_wait_read_1();
        __syncwarp();
#pragma unroll
        for (int q = 0; q < 64; ++q) stg[q * 32 + lane] = __uint_as_float(v[q]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_reduce_add_3d(&tm_dq, smem_u32(stg), 32 * (warp & 3), q0, bh);
          tma_store_commit();
        }
      }
      if (lane == 0) mbar_arrive(bar(C::B_ITEMF + (n & 1)));
      J += i;
    }
    // the reduce-adds of the last steps have read their shared memory
    if (lane == 0) tma_store_wait_read();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

}  // namespace

cudaError_t launch_bwd_persist(const Problem& p, const void* q, const void* k, const void* v,
                               const void* dout, const float* lse2, const float* dvec,
                               float* dq_acc, void* dk, void* dv, int npad,
                               const BwdSplit* split, unsigned long long* next_item, bool early,
                               cudaStream_t st, bool lose) {
  if (p.d != 64 || p.cu_seqlens != nullptr || p.drop_p8 != 0 || next_item == nullptr)
    return cudaErrorInvalidValue;
  const long long bh = (long long)p.B * p.H;
  CUtensorMap tq, tk, tv, tdo, tdk, tdv, tdq;
  if (!(make_bf16_map_3d(&tq, q, 64, p.N, bh, PTc::BQ) &&
        make_bf16_map_3d(&tk, k, 64, p.N, bh, 128) && make_bf16_map_3d(&tv, v, 64, p.N, bh, 128) &&
        make_bf16_map_3d(&tdo, dout, 64, p.N, bh, PTc::BQ) &&
        make_bf16_map_3d(&tdk, dk, 64, p.N, bh, 128) &&
        make_bf16_map_3d(&tdv, dv, 64, p.N, bh, 128) &&
        make_f32_map_3d(&tdq, dq_acc, 64, p.N, bh, PTc::BQ, 32)))
    return cudaErrorInvalidValue;
  int dev = 0, nsm = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  // one CTA per SM, at most one per work item
  long long ctas = bh * p.T * (split != nullptr ? kSplitMax : 1);
  if (ctas > nsm) ctas = nsm;
  const BwdSplit none{nullptr, nullptr, nullptr};
  auto kern = lose ? bwd_persist_kernel<false, true>
                   : split != nullptr ? bwd_persist_kernel<true> : bwd_persist_kernel<false>;
  if (lose && split != nullptr) return cudaErrorInvalidValue;
  if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, PTc::SMEM)) !=
      cudaSuccess)
    return e;
  return launch_k(early, kern, dim3((unsigned)ctas), dim3(PTc::THREADS), PTc::SMEM, st, tq, tk,
                  tv, tdo, tdk, tdv, tdq, p, lse2, dvec, npad, split != nullptr ? *split : none,
                  next_item);
}

}  // namespace fa
