// Tensor-core (tcgen05 + TMA) attention backward with recomputation, sm_103a.
//
// One CTA owns one 128-key tile of one (b, h).  K and V are loaded once; the
// CTA walks the live query tiles of its key tile in 64-row steps.  Per step
// i (queries q0 .. q0+63) it rebuilds the probabilities from the stored row
// statistic instead of reading a stored P (page "FlashAttention IO-aware
// explained", section "Recomputation and IO complexity"; Theorem 5's proof
// on page "FlashAttention: Fast and Memory-Efficient Exact Attention with
// IO-Awareness", "C Proofs": K, V read once, passes over Q, O, dO, dQ):
//     S^T  = K Q^T              (TMEM, 128 x 64)
//     dP^T = V dO^T             (TMEM, 128 x 64)
//     P^T  = 2^(scale*log2e*S^T - LSE*log2e)     (masked; bf16 back to TMEM)
//     dS^T = P^T * (dP^T - D)                    (bf16 to shared memory)
//     dV  += P^T dO             (A = P^T from TMEM)
//     dK  += dS^T Q             (scaled by `scale` in the epilogue)
//     dQ^T = K^T dS^T           (TMEM, d x 64; added into the fp32 dQ
//                                accumulator; the conversion kernel
//                                applies `scale`)
// with D = rowsum(dO * O) and LSE*log2e precomputed per query row.
//
// Warp roles (384 threads; 512 at d = 64 without dropout):
//   warp 0      TMA producer: K, V once; per step Q, dO (64 rows) and the
//               64 LSE / D values into a ring of stages.
//   warps 1, 2  MMA issuers (one thread each): warp 1 the recompute GEMMs
//               S^T, dP^T (and owns TMEM), warp 2 the gradient GEMMs dV, dK,
//               dQ^T.
//   warps 4-7   element-wise: P^T, dS^T (one key row per thread); at the
//               end dK, dV from TMEM to bf16 and a TMA store.  At d = 64
//               without dropout they take queries 0-31 of each step and
//               warps 12-15 queries 32-63.
//   warps 8-11  dQ: dQ^T from TMEM, one head-dim row per thread (warps whose
//               lanes lie at or above d idle).  d = 128: added into the fp32
//               accumulator with red.global.add from registers (coalesced
//               across the warp), so the dQ tile costs no shared-memory
//               traffic.  d = 64: each warp stages its 32 head dimensions
//               of the step's 64 query rows in shared memory and adds them
//               with one TMA reduce-add.
//
// TMEM columns: dV [0,d), dK [d,2d), S[b] = 2d + 64b, dP[b] = 2d + 128 + 64b
// for the two step buffers b.  At d = 64 dQ^T has two buffers of its own,
// dQ[b] = 384 + 64b, so the recompute GEMMs never wait for the dQ warps.
// At d = 128 the 512 columns are full: dQ^T of step i is written over
// dP[i % 2] once the element-wise warps have consumed dP^T(i) (it is the
// first gradient GEMM of the step, so that the dQ warps read it out early),
// and dP^T(i+2) waits until they have.  For d = 64 the dQ^T product is
// issued with M = 128 (the second 64 rows read the V tile and are
// discarded).
#include <cuda_bf16.h>

#include "fa_common.cuh"
#include "fa_kernels.h"
#include "fa_sm100.cuh"
#include "fa_tma_host.h"

namespace fa {
using namespace sm100;

// Element-wise warpgroups: at d = 64 (no dropout) two groups of four warps
// share each step, one per 32 queries, since there the element-wise work of
// a step outlasts its MMAs; otherwise one group of four takes all 64.
template <int D, bool DROP>
struct BwdEw {
  static constexpr int GROUPS = (D == 64 && !DROP) ? 2 : 1;
  static constexpr int QH = 64 / GROUPS;           // queries per thread and step
  static constexpr int THREADS = 256 + 128 * GROUPS;
};

template <int D>
struct BwdTc {
  static constexpr int BQ = 64;                 // query rows per step
  // dQ^T in TMEM buffers of its own and reduced through shared memory by
  // TMA reduce-adds (d = 64), or over dP^T and reduced by the dQ warps with
  // atomics from registers (d = 128, where TMEM and shared memory are full)
  static constexpr bool SEPQ = D == 64;
  // dQ warps holding TMEM lanes below d (the others have nothing to do)
  static constexpr int DQ_WARPS = D / 32;
  static constexpr int NS = D == 128 ? 3 : 4;   // step stages
  static constexpr int HALF_K = 128 * 128;      // [128 rows][64 cols] bf16 box
  static constexpr int HALF_Q = 64 * 128;       // [64 rows][64 cols] bf16 box
  static constexpr int KT = 128 * D * 2;        // K or V tile
  static constexpr int QB = BQ * D * 2;         // Q or dO block
  static constexpr int STAGE = 2 * QB;          // Q, dO of one step
  static constexpr int OFF_K = 0, OFF_V = KT, OFF_ST = 2 * KT;
  static constexpr int OFF_VEC = OFF_ST + NS * STAGE;  // [NS][LSE*log2e (64), D (64)]
  static constexpr int OFF_DS = (OFF_VEC + NS * 512 + 1023) / 1024 * 1024;
  static constexpr int DS = 128 * BQ * 2;             // dS^T [128 keys][64 q] bf16, x2
  static constexpr int OFF_BAR = OFF_DS + 2 * DS;
  // B_DSF[b]: the gradient GEMMs that read dS^T buffer b have completed
  // (d = 128; at d = 64 dQ^T is their last and B_DQF[b] says so)
  static constexpr int B_KV = 0, B_FULL = 1, B_EMPTY = 1 + NS, B_S = 1 + 2 * NS, B_EW = B_S + 2,
                       B_DQF = B_EW + 2, B_DQE = B_DQF + 2, B_SF = B_DQE + 2, B_FIN = B_SF + 2,
                       B_DRAIN = B_FIN + 1, B_DSF = B_DRAIN + 2, NBAR = B_DSF + 2;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  // misc: TMEM address (+0), abort flag (+16) and the split item's part
  // word (+44)
  // dropout keep bytes of a step, [64 queries][128 keys], two buffers
  static constexpr int OFF_DROP = (OFF_MISC + 64 + 127) / 128 * 128;
  static constexpr int DROPB = BQ * 128;
  // live query tiles of the key tile's range under a block mask, one bit each
  static constexpr int OFF_LIVE = OFF_DROP + 2 * DROPB;
  static constexpr int LIVEB = 65536 / 8;
  // d = 64: the step's dQ rows, [64 rows][32 columns] fp32 per dQ warp (two
  // warps), two buffers, added into the accumulator by TMA reduce-adds
  static constexpr int DQW = BQ * 32 * 4;
  static constexpr int DQS = 2 * DQW;
  static constexpr int OFF_DQS = (OFF_LIVE + LIVEB + 1023) / 1024 * 1024;
  static constexpr int SMEM = (SEPQ ? OFF_DQS + 2 * DQS : OFF_LIVE + LIVEB) + 1024;
  static constexpr int COL_DV = 0, COL_DK = D, COL_S = 2 * D, COL_DP = 2 * D + 128;
  static constexpr int COL_DQ = SEPQ ? 2 * D + 256 : COL_DP;
  static_assert(!SEPQ || COL_DQ + 128 <= 512, "TMEM columns");
  static constexpr uint32_t TMEM_COLS = 512;
  static_assert(2 * KT <= NS * STAGE, "dK/dV staging must fit in the stage ring");
  static_assert(SMEM <= 232448, "shared memory budget");
};

// Next 64-row query step after (qt, sub) for key tile kt: live query tiles
// in ascending order within the key tile's query-tile range (exact without a
// block mask; recomputed here from the constant parameters rather than kept
// live in registers across the roles' loops), two halves each, skipping
// halves past N.  Under a block mask the live tiles come from `live`, bit t
// for query tile first + t, built once per CTA: the mask's column of a key
// tile is one byte per 128-byte line, so testing it per step from global
// memory put a cache miss on every role's loop.
// (A CTA of the split variant runs one part of a key tile's live tiles: the
// bitmask then holds only that part's bits.)
template <int D>
__device__ __forceinline__ bool next_q_step(const Problem& p, int kt, int klim,
                                            const uint8_t* smem, int& qt, int& sub) {
  if (qt >= 0 && sub == 0 && qt * 128 + 64 < p.N) {
    sub = 1;
    return true;
  }
  sub = 0;
  int qf, ql;
  ktile_query_tiles(p, kt, klim, qf, ql);
  qt = qt < 0 ? qf : qt + 1;
  if (p.block_mask == nullptr) return qt <= ql;
  const uint32_t* live = reinterpret_cast<const uint32_t*>(smem + BwdTc<D>::OFF_LIVE);
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

// LOSE: self-test instantiation only (fa_selftest_backward_lost_signal): the
// first element-wise warp withholds its arrival for the first query step
// and every wait gives up after 1 ms, so the gradient issuer's wait runs out
// and the abort, drain and status paths run.
template <int D, bool PACKED, bool DROP, bool SPLIT, bool LOSE = false>
__global__ void __launch_bounds__(BwdEw<D, DROP>::THREADS, 1)
    bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                  const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                  const __grid_constant__ CUtensorMap tm_dq, const Problem pin, const float* __restrict__ lse2, const float* __restrict__ dvec,
                  float* __restrict__ dq_acc, int npad, __nv_bfloat16* __restrict__ dk_rows,
                  __nv_bfloat16* __restrict__ dv_rows, const BwdSplit sp) {
  using C = BwdTc<D>;
  using EW = BwdEw<D, DROP>;
  // Geometry of this CTA's (b, h): padded layout [B*H][N][d] (TMA coordinates
  // (x, row, bh)), or one sequence of the packed layout [total][H][d]
  // (coordinates (x, h, start + row)), whose length then plays the role of N.
  // Grid: one CTA per (head, key tile) in the grouped order -- small key
  // tiles carry the most causal work: first, across a group of heads whose
  // Q, dO and dQ accumulator stay in L2.
  // Split variant: CTA rank r of a head runs work item r of the plan (key
  // tile, part [qa, qb] of its query range, part k of n), heaviest first.
  long long bh;
  int kt;
  int4 item = make_int4(0, 0, -1, 1 << 8);
  if constexpr (SPLIT) {
    int r;
    grouped_cta(pin, blockIdx.x, pin.T * kSplitMax, bh, r);
    if (r >= __ldg(sp.nitems)) return;
    item = __ldg(sp.items + r);
    kt = item.x;
  } else {
    grouped_cta(pin, blockIdx.x, pin.T, bh, kt);
  }
  const int b = (int)(bh / pin.H);
  const int head = (int)(bh % pin.H);
  Problem p = pin;
  int start = 0;
  if constexpr (PACKED) {
    int len;
    seq_span(pin, b, start, len);
    p.N = len;
    p.T = (len + kTile - 1) / kTile;
  }
  if (kt >= p.T) return;  // packed: past this sequence's key tiles
  auto cy = [&](int row) { return PACKED ? head : row; };
  auto cz = [&](int row) { return PACKED ? start + row : (int)bh; };
  extern __shared__ uint8_t smem_raw[];
  // An offset (not an integer round trip) keeps the pointer visibly in shared
  // memory, so C++ accesses through it compile to shared-memory instructions.
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t s0 = smem_u32(smem);
  const uint32_t bar0 = s0 + C::OFF_BAR;
  auto bar = [&](int i) { return bar0 + 8u * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 16);
  const Abort ab{abort_flag, p.status, LOSE ? kShortWaitLimitNs : kWaitLimitNs};
  // Suspension hint of the latency-critical waits (issuers, element-wise
  // warps): at d = 128, where each step's MMAs take long enough to absorb a
  // late wake-up, a short sleep in the barrier (fewer polls taking issue
  // slots from the element-wise warps) measured 1% faster; at d = 64 polling.
  constexpr uint32_t crit_hint = D == 128 ? 200u : kPollHintNs;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int klim = key_limit(p, b);

  if (warp == 0) {
    // the barriers, one per lane of warp 0
    for (int i = lane; i < C::NBAR; i += 32) {
      const bool ew = i == C::B_EW || i == C::B_EW + 1;
      const bool dqe = i == C::B_DQE || i == C::B_DQE + 1;
      mbar_init(bar(i), ew ? 4 * EW::GROUPS : dqe ? C::DQ_WARPS : 1);
    }
    fence_barrier_init();
    __syncwarp();
  }
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    // K and V of the tile, issued by the producer thread before the rest of
    // the set-up (TMEM, the live bitmask, the CTA barrier) so that their
    // latency overlaps it
    mbar_expect_tx(bar(C::B_KV), 2 * C::KT);
    for (int h = 0; h < D / 64; ++h) {
      tma_load_3d(s0 + C::OFF_K + h * C::HALF_K, &tm_k, bar(C::B_KV), h * 64, cy(kt * 128),
                  cz(kt * 128));
      tma_load_3d(s0 + C::OFF_V + h * C::HALF_K, &tm_v, bar(C::B_KV), h * 64, cy(kt * 128),
                  cz(kt * 128));
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  if (p.block_mask != nullptr) {
    // the range's liveness, 32 query tiles per warp and word, all warps at once
    int qf, ql;
    ktile_query_tiles(p, kt, klim, qf, ql);
    if constexpr (SPLIT) {
      if (threadIdx.x == 0) reinterpret_cast<int*>(smem + C::OFF_MISC)[11] = item.w;
    }
    const int n = ql - qf + 1;
    for (int wi = warp; wi < ((n + 31) >> 5); wi += EW::THREADS / 32) {
      const int t = (wi << 5) + lane;
      const bool in_part = !SPLIT || (qf + t >= item.y && qf + t <= item.z);
      const uint32_t bits =
          __ballot_sync(0xffffffffu, t < n && in_part && tile_live(p, qf + t, kt, klim));
      if (lane == 0) reinterpret_cast<uint32_t*>(smem + C::OFF_LIVE)[wi] = bits;
    }
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
  const size_t vec_base = (size_t)bh * npad;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      // the preprocess's LSE and D rows are read from here on
      griddep_wait();
      griddep_release();
      int qt = -1, sub = 0, slot = 0, round = 0;
      while (next_q_step<D>(p, kt, klim, smem, qt, sub)) {
        const int q0 = qt * 128 + sub * 64;
        if (!mbar_wait(bar(C::B_EMPTY + slot), (round & 1) ^ 1, ab, kSleepHintNs)) break;
        const uint32_t st = s0 + C::OFF_ST + slot * C::STAGE;
        const uint32_t fb = bar(C::B_FULL + slot);
        const uint32_t vb = s0 + C::OFF_VEC + slot * 512;
        mbar_expect_tx(fb, 2 * C::QB + 512);
        for (int h = 0; h < D / 64; ++h) {
          tma_load_3d(st + h * C::HALF_Q, &tm_q, fb, h * 64, cy(q0), cz(q0));
          tma_load_3d(st + C::QB + h * C::HALF_Q, &tm_do, fb, h * 64, cy(q0), cz(q0));
        }
        bulk_load(vb, lse2 + vec_base + q0, 256, fb);
        bulk_load(vb + 256, dvec + vec_base + q0, 256, fb);
        if (++slot == C::NS) {
          slot = 0;
          ++round;
        }
      }
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
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(bar(C::B_KV), 0) && globaltimer() - t0 < kWaitLimitNs) {
      }
    }
  } else if (warp == 1 || warp == 2) {
    // ------------------------------------------------------------ MMA issuers
    // Two issuing threads: issuing one tcgen05.mma costs a thread about as
    // long as a narrow MMA takes to run, so one thread cannot feed the tensor
    // core with all five GEMMs of a step and its barrier polls.
    //   warp 1: S^T(j), dP^T(j) into buffer j % 2 (owns TMEM);
    //   warp 2: d = 64: dV(i), dK(i), dQ^T(i) into dQ[i % 2];
    //           d = 128: dQ^T(i) over dP[i % 2], dV(i), dK(i).
    // S^T(j) waits until dV(j-2) has read P^T(j-2) from the same columns
    // (s_free at d = 128; at d = 64 the release of step j-2's Q, dO stage,
    // committed after its dK); at d = 128 dP^T(j) waits until the dQ warps
    // have read dQ^T(j-2) out, at d = 64 dQ^T(i) waits for that instead.
    if (lane == 0) {
      constexpr uint32_t id_s = idesc_bf16(128, C::BQ, false, false);
      constexpr uint32_t id_kv = idesc_bf16(128, D, false, true);
      constexpr uint32_t id_q = idesc_bf16(128, C::BQ, true, true);
      constexpr uint32_t st_step = C::STAGE >> 4, qb_step = C::QB >> 4, ds_step = C::DS >> 4;
      const uint64_t dk_k = sdesc_sw128(s0 + C::OFF_K, 16, 1024);       // K, K-major
      const uint64_t dv_k = sdesc_sw128(s0 + C::OFF_V, 16, 1024);       // V, K-major
      const uint64_t dk_mn = sdesc_sw128(s0 + C::OFF_K, C::HALF_K, 1024);  // K^T, MN-major
      const uint64_t dst_k = sdesc_sw128(s0 + C::OFF_ST, 16, 1024);     // stage 0 Q, K-major
      const uint64_t dst_mn = sdesc_sw128(s0 + C::OFF_ST, C::HALF_Q, 1024);  // stage 0 Q, MN-major
      const uint64_t dds = sdesc_sw128(s0 + C::OFF_DS, 16, 1024);       // dS^T buffer 0
      const uint32_t t_dv = tmem + C::COL_DV, t_dk = tmem + C::COL_DK;
      // The issuers need only the number of steps (descriptors depend on the
      // step index alone), so the walk is counted once up front.
      int nsteps = 0;
      for (int qt = -1, sub = 0; next_q_step<D>(p, kt, klim, smem, qt, sub);) ++nsteps;
      bool ok = mbar_wait(bar(C::B_KV), 0, ab);
      tc_fence_after();
      if (warp == 1) {
        for (int j = 0; ok && j < nsteps; ++j) {
          const int bf = j & 1;
          const uint64_t sq = dst_k + (uint64_t)((j % C::NS) * st_step);
          if (!(ok = mbar_wait(bar(C::B_FULL + j % C::NS), (j / C::NS) & 1, ab, crit_hint))) break;
          // d = 64: the release of step j-2's Q, dO stage (after its dK,
          // which follows its dV) says that dV has read P^T(j-2)
          if (j >= 2 && !(ok = mbar_wait(C::SEPQ ? bar(C::B_EMPTY + (j - 2) % C::NS)
                                                 : bar(C::B_SF + bf),
                                         C::SEPQ ? ((j - 2) / C::NS) & 1 : ((j - 2) >> 1) & 1,
                                         ab, crit_hint)))
            break;
          tc_fence_after();
          if (D == 128)
            mma_ss_kmajor_k128_a16k_b8k(tmem + C::COL_S + 64 * bf, dk_k, sq, id_s, 0);
          else
            mma_ss_kmajor_k64_a16k_b8k(tmem + C::COL_S + 64 * bf, dk_k, sq, id_s, 0);
          if (!C::SEPQ && j >= 2) {
            if (!(ok = mbar_wait(bar(C::B_DQE + bf), ((j - 2) >> 1) & 1, ab, crit_hint))) break;
            tc_fence_after();
          }
          if (D == 128)
            mma_ss_kmajor_k128_a16k_b8k(tmem + C::COL_DP + 64 * bf, dv_k, sq + qb_step, id_s, 0);
          else
            mma_ss_kmajor_k64_a16k_b8k(tmem + C::COL_DP + 64 * bf, dv_k, sq + qb_step, id_s, 0);
          mma_commit(bar(C::B_S + bf));
        }
      } else {
        for (int i = 0; ok && i < nsteps; ++i) {
          const int bf = i & 1;
          const uint64_t sq_mn = dst_mn + (uint64_t)((i % C::NS) * st_step);
          const uint64_t ds = dds + (uint64_t)(bf * ds_step);
          if (!(ok = mbar_wait(bar(C::B_EW + bf), (i >> 1) & 1, ab, crit_hint))) break;
          tc_fence_after();
          if constexpr (!C::SEPQ) {
            // dQ^T = K^T dS^T over dP[bf] (dP^T(i) is in the element-wise
            // warps' registers by now)
            mma_ss_mn_mn_k128(tmem + C::COL_DQ + 64 * bf, dk_mn, ds, id_q, 0);
            mma_commit(bar(C::B_DQF + bf));
          }
          // dV += P^T dO   (P^T: bf16 in TMEM over S[bf], in two halves 32
          // columns apart with two element-wise groups; dO as MN-major B)
          if constexpr (EW::GROUPS == 2)
            mma_ts_mn_k64_gap32(t_dv, tmem + C::COL_S + 64 * bf, sq_mn + qb_step, id_kv, i > 0);
          else
            mma_ts_mn_k64(t_dv, tmem + C::COL_S + 64 * bf, sq_mn + qb_step, id_kv, i > 0);
          if constexpr (!C::SEPQ) mma_commit(bar(C::B_SF + bf));
          // dK += dS^T Q
          mma_ss_kmajor_mn_k64(t_dk, ds, sq_mn, id_kv, i > 0);
          mma_commit(bar(C::B_EMPTY + i % C::NS));
          if constexpr (C::SEPQ) {
            // dQ^T = K^T dS^T into dQ[bf], once dQ^T(i-2) has been read out
            if (i >= 2) {
              if (!(ok = mbar_wait(bar(C::B_DQE + bf), ((i - 2) >> 1) & 1, ab, crit_hint))) break;
              tc_fence_after();
            }
            mma_ss_mn_mn_k128(tmem + C::COL_DQ + 64 * bf, dk_mn, ds, id_q, 0);
            mma_commit(bar(C::B_DQF + bf));
          }
          if constexpr (!C::SEPQ) mma_commit(bar(C::B_DSF + bf));
        }
        // dK and dV are complete once this thread's last MMAs are (the other
        // issuer's work for the last step finished before it could start)
        mma_commit(bar(C::B_FIN));
      }
      mma_commit(bar(C::B_DRAIN + warp - 1));
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(bar(C::B_DRAIN + warp - 1), 0) && globaltimer() - t0 < kWaitLimitNs) {
      }
    }
  } else if ((warp >= 4 && warp < 8) || warp >= 12) {
    // ------------------------------------------------------------ element-wise
    // group g (warps 4-7, or 12-15 with two groups) takes the step's queries
    // qo .. qo + QH - 1
    constexpr int QH = EW::QH;
    const int g = warp >= 12 ? 1 : 0;
    const int qo = g * QH;
    const int r = ((warp & 3) << 5) + lane;  // key row within the tile
    const int j = kt * 128 + r;              // key index
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const float cl2 = p.scale_log2;
    int qt = -1, sub = 0, i = 0;
    bool ok = true;
    for (; next_q_step<D>(p, kt, klim, smem, qt, sub); ++i) {
      const int bf = i & 1;
      const int q0 = qt * 128 + sub * 64;
      const uint8_t* vb = smem + C::OFF_VEC + (i % C::NS) * 512;
      const float* l2 = reinterpret_cast<const float*>(vb) + qo;
      const float* dv = reinterpret_cast<const float*>(vb + 256) + qo;
      // Dropout: the step's 64 x 128 keep bytes, generated by the four warps
      // together (four generator calls per thread, each 16 keys of one
      // query) while the tensor core computes S^T and dP^T, stored with the
      // 16-byte chunk index XOR-swizzled by the query row; double-buffered,
      // so one barrier per step keeps writers behind readers.
      const uint8_t* drop_buf = smem + C::OFF_DROP + (i & 1) * C::DROPB;
      if constexpr (DROP) {
        const int c = r & 63, kh = (r >> 6) * 4;
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const int kb = kh + kk;
          const uint4 w = dropout_bytes(p, bh, q0 + c, kt * 8 + kb);
          *reinterpret_cast<uint4*>(const_cast<uint8_t*>(drop_buf) + c * 128 +
                                    ((kb ^ (c & 7)) << 4)) = w;
        }
        named_barrier(2, 128);
      }
      if (!(ok = mbar_wait(bar(C::B_S + bf), (i >> 1) & 1, ab, crit_hint))) break;
      tc_fence_after();
      uint32_t sr[QH], pr[QH];
      if constexpr (QH == 64) {
        tmem_ld64(lane_base + C::COL_S + 64 * bf, sr);
        tmem_ld64(lane_base + C::COL_DP + 64 * bf, pr);
      } else {
        tmem_ld32(lane_base + C::COL_S + 64 * bf + qo, sr);
        tmem_ld32(lane_base + C::COL_DP + 64 * bf + qo, pr);
      }
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
        fma2(x0, x1, __uint_as_float(sr[4 * c4]), __uint_as_float(sr[4 * c4 + 1]), cl2, cl2, -L.x,
             -L.y);
        fma2(x2, x3, __uint_as_float(sr[4 * c4 + 2]), __uint_as_float(sr[4 * c4 + 3]), cl2, cl2,
             -L.z, -L.w);
        const float p0 = fast_exp2(x0), p1 = fast_exp2(x1), p2 = fast_exp2(x2),
                    p3 = fast_exp2(x3);
        float e0, e1, e2, e3;
        if constexpr (DROP) {
          // P o Z / (1 - p) feeds dV; dP = (dO V^T) o Z / (1 - p) feeds dS
          float z[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int c = 4 * c4 + e;
            const uint8_t u = drop_buf[c * 128 + (((r >> 4) ^ (c & 7)) << 4) + (r & 15)];
            z[e] = u >= p.drop_p8 ? p.drop_scale : 0.f;
          }
          fma2(e0, e1, __uint_as_float(pr[4 * c4]), __uint_as_float(pr[4 * c4 + 1]), z[0], z[1],
               -Dd.x, -Dd.y);
          fma2(e2, e3, __uint_as_float(pr[4 * c4 + 2]), __uint_as_float(pr[4 * c4 + 3]), z[2],
               z[3], -Dd.z, -Dd.w);
          pk[2 * c4] = pack_bf16(p0 * z[0], p1 * z[1]);
          pk[2 * c4 + 1] = pack_bf16(p2 * z[2], p3 * z[3]);
        } else {
          add2(e0, e1, __uint_as_float(pr[4 * c4]), __uint_as_float(pr[4 * c4 + 1]), -Dd.x,
               -Dd.y);
          add2(e2, e3, __uint_as_float(pr[4 * c4 + 2]), __uint_as_float(pr[4 * c4 + 3]), -Dd.z,
               -Dd.w);
          pk[2 * c4] = pack_bf16(p0, p1);
          pk[2 * c4 + 1] = pack_bf16(p2, p3);
        }
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
      // P^T (bf16 pairs) over the group's own S^T columns: columns 0-31
      // with one group; 0-15 and 32-47 with two (each group overwrites only
      // columns it has already read)
      if constexpr (QH == 64)
        tmem_st32(lane_base + C::COL_S + 64 * bf, pk);
      else
        tmem_st16(lane_base + C::COL_S + 64 * bf + qo, pk);
      // dS^T row r into the 128-byte-swizzled buffer bf, once dK / dQ^T of
      // step i-2 (which read this buffer) have completed (at d = 64 the
      // commit after dQ^T, the last of them, covers both).
      if (i >= 2) {
        const uint32_t fb = bar((C::SEPQ ? C::B_DQF : C::B_DSF) + bf);
        if (!(ok = mbar_wait(fb, ((i - 2) >> 1) & 1, ab, crit_hint))) break;
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
      if (lane == 0 && !(LOSE && i == 0 && warp == 4)) mbar_arrive(bar(C::B_EW + bf));
    }
    // ---- epilogue (group 0): dK (x scale), dV -> bf16 -> shared (swizzled) -> TMA store;
    // in the packed layout a key tile that ends past its sequence is written
    // row by row instead (a whole-tile store would overwrite the next
    // sequence's first rows).
    if (g == 0) {
    if (ok) ok = mbar_wait(bar(C::B_FIN), 0, ab);
    tc_fence_after();
    // A part of a split key tile stores its fp32 dK, dV rows (0 if it ran no
    // step) into its own slot; the join kernel adds the parts afterwards.
    bool emit = true;
    const bool have = i > 0 && ok;
    if constexpr (SPLIT) {
      // the item's part word, kept in shared memory through the loops
      const int meta = reinterpret_cast<const volatile int*>(smem + C::OFF_MISC)[11];
      if (((meta >> 8) & 0xff) > 1) {
        float* mine = sp.slots +
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
    uint8_t* stg = smem + C::OFF_ST;  // dK tile, then dV tile
    const bool direct = PACKED && (kt + 1) * 128 > p.N;
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
          pw[e] = pack_bf16(__uint_as_float(o[2 * e]) * mul, __uint_as_float(o[2 * e + 1]) * mul);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int cc = 4 * c + q;
          const uint4 w = make_uint4(pw[4 * q], pw[4 * q + 1], pw[4 * q + 2], pw[4 * q + 3]);
          if (direct) {
            if (ok && j < p.N)
              reinterpret_cast<uint4*>((t == 0 ? dk_rows : dv_rows) +
                                       ((size_t)(start + j) * p.H + head) * D)[cc] = w;
          } else {
            uint8_t* dst = stg + t * C::KT + (cc >> 3) * C::HALF_K + r * 128 +
                           (((cc & 7) ^ (r & 7)) << 4);
            *reinterpret_cast<uint4*>(dst) = w;
          }
        }
      }
    }
    fence_proxy_async_smem();
    named_barrier(1, 128);
    if (ok && emit && r == 0 && !direct) {
      for (int h = 0; h < D / 64; ++h) {
        tma_store_3d(&tm_dk, smem_u32(stg) + h * C::HALF_K, h * 64, cy(kt * 128), cz(kt * 128));
        tma_store_3d(&tm_dv, smem_u32(stg) + C::KT + h * C::HALF_K, h * 64, cy(kt * 128),
                     cz(kt * 128));
      }
      tma_store_commit();
      tma_store_wait_read();  // shared memory read out; the writes finish with the grid
    }
    }
  } else if (warp >= 8 && warp < 12) {
    // ------------------------------------------------------------ dQ
    const int c = ((warp & 3) << 5) + lane;  // head-dim index = TMEM lane
    const bool valid = c < D;                 // the same for the whole warp
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    int qt = -1, sub = 0;
    bool ok = true;
    if (valid) griddep_wait();  // the accumulator the preprocess cleared
    for (int i = 0; valid && next_q_step<D>(p, kt, klim, smem, qt, sub); ++i) {
      const int bf = i & 1;
      const int q0 = qt * 128 + sub * 64;
      if (!(ok = mbar_wait(bar(C::B_DQF + bf), (i >> 1) & 1, ab, kSleepHintNs))) break;
      tc_fence_after();
      uint32_t v[64];
      if (valid) tmem_ld64(lane_base + C::COL_DQ + 64 * bf, v);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(C::B_DQE + bf));
      // padded: [B*H][N][d]; packed: [H][total][d] (head-major, so a head's
      // rows are contiguous and the reductions do not collide in L2 the way
      // rows H*d apart do)
      const int rows = min(64, p.N - q0);
      float* dst_rows = PACKED ? dq_acc + ((size_t)head * p.total + start + q0) * D
                               : dq_acc + ((size_t)bh * p.N + q0) * D;
      if constexpr (C::SEPQ) {
        // d = 64: each dQ warp writes its 32 columns of the step's rows to
        // its own shared buffer (a warp instruction stores 32 consecutive
        // floats of one row: conflict-free) and its lane 0 adds the tile
        // into the accumulator with a TMA reduce-add (rows outside the
        // tensor are skipped; in the packed layout the rows past this
        // sequence carry exact zeros, since their dS is masked to 0).  The
        // buffer of step i is rewritten at step i + 2, once that reduce has
        // read it.
        if (valid) {
          float* stg = reinterpret_cast<float*>(smem + C::OFF_DQS + (i & 1) * C::DQS +
                                                (warp & 3) * C::DQW);
          if (lane == 0 && i >= 2) bulk_wait_read_1();
          __syncwarp();
#pragma unroll
          for (int q = 0; q < 64; ++q) stg[q * 32 + lane] = __uint_as_float(v[q]);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (PACKED)
              tma_reduce_add_3d(&tm_dq, smem_u32(stg), 32 * (warp & 3), start + q0, head);
            else
              tma_reduce_add_3d(&tm_dq, smem_u32(stg), 32 * (warp & 3), q0, (int)bh);
            tma_store_commit();
          }
        }
      } else {
        // d = 128: straight from registers: for each query the warp's 32
        // lanes add 32 consecutive floats of its row.  (Vector reductions
        // after a 4 x 4 shuffle transpose measured 16% slower here.)
        float* dst = dst_rows + c;
#pragma unroll
        for (int q = 0; q < 64; ++q)
          if (q < rows) atomicAdd(dst + (size_t)q * D, __uint_as_float(v[q]));
      }
    }
    // the reduce-adds of the last steps have read their shared memory
    if (C::SEPQ && valid && lane == 0) tma_store_wait_read();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// Work plan of the split backward, one CTA.  Per key tile, c = its live
// query tiles (block mask, causal rule, window; the per-batch key limit is
// left to the kernel, which only drops tiles from a part), counted from a
// row-major (coalesced) pass over the mask.  With a = the average work per
// SM, max(2, ceil(B*H*sum(c) / nsm)), a key tile with c > a runs as
// n = min(kSplitMax, ceil(c / a)) parts of consecutive live tiles (a doubles
// until the split tiles' parts fit kSplitSlots slots per head); part k
// starts at the query tile holding live tile k*c/n, found by one warp per
// split key tile.  Items are ordered by their number of live tiles,
// heaviest first.  plan[0] = the item count, plan[1] = the number of split
// key tiles, then (key tile, first slot, parts) for each of them.
__global__ void __launch_bounds__(1024)
    bwd_plan_kernel(const Problem p, int nsm, long long heads, int4* __restrict__ items,
                    int* __restrict__ plan) {
  __shared__ int cnt[kPlanMaxTiles];
  __shared__ int meta[kPlanMaxTiles];  // n | slot base << 16
  __shared__ int hist[kPlanMaxTiles + 2];
  __shared__ int start[kSplitSlots];  // first query tile of each part of a split key tile
  __shared__ int split_kt[kSplitSlots];
  __shared__ unsigned long long tot;
  __shared__ int slots, next_base, nsplit;
  const int T = p.T, tid = threadIdx.x, nth = blockDim.x;
  const int warp = tid >> 5, lane = tid & 31;
  griddep_wait();
  griddep_release();
  if (tid == 0) {
    tot = 0;
    next_base = 0;
    nsplit = 0;
  }
  for (int w = tid; w < T; w += nth) cnt[w] = 0;
  for (int w = tid; w <= T + 1; w += nth) hist[w] = 0;
  __syncthreads();
  for (int qt = warp; qt < T; qt += nth / 32)
    for (int kt = lane; kt < T; kt += 32)
      if (tile_live(p, qt, kt, p.N)) atomicAdd(&cnt[kt], 1);
  __syncthreads();
  for (int kt = tid; kt < T; kt += nth) atomicAdd(&tot, (unsigned long long)cnt[kt]);
  __syncthreads();
  long long a = ((long long)tot * heads + nsm - 1) / nsm;
  if (a < 2) a = 2;
  auto parts = [&](int c) {
    return c > a ? (int)min((long long)kSplitMax, (c + a - 1) / a) : 1;
  };
  for (;;) {
    if (tid == 0) slots = 0;
    __syncthreads();
    for (int kt = tid; kt < T; kt += nth) {
      const int n = parts(cnt[kt]);
      if (n > 1) atomicAdd(&slots, n);
    }
    __syncthreads();
    const bool fits = slots <= kSplitSlots;
    __syncthreads();
    if (fits) break;
    a *= 2;
  }
  for (int kt = tid; kt < T; kt += nth) {
    const int c = cnt[kt], n = parts(c);
    int base = 0;
    if (n > 1) {
      base = atomicAdd(&next_base, n);
      split_kt[atomicAdd(&nsplit, 1)] = kt;
    }
    meta[kt] = n | (base << 16);
    for (int k = 0; k < n; ++k) atomicAdd(&hist[(k + 1) * c / n - k * c / n], 1);
  }
  __syncthreads();
  // part starts of the split key tiles: warp w scans key tile split_kt[w]'s
  // column 32 query tiles at a time, counting live tiles with ballots
  for (int sk = warp; sk < nsplit; sk += nth / 32) {
    const int kt = split_kt[sk], c = cnt[kt], n = meta[kt] & 0xffff, base = meta[kt] >> 16;
    int k = 1, seen = 0;
    for (int q0 = 0; q0 < T && k < n; q0 += 32) {
      const uint32_t bits = __ballot_sync(0xffffffffu, q0 + lane < T && tile_live(p, q0 + lane, kt, p.N));
      const int nb = __popc(bits);
      while (k < n && seen + nb > k * c / n) {
        // the (k*c/n - seen)-th set bit of this chunk
        uint32_t b = bits;
        for (int skip = k * c / n - seen; skip > 0; --skip) b &= b - 1;
        if (lane == 0) start[base + k] = q0 + __ffs(b) - 1;
        ++k;
      }
      seen += nb;
    }
  }
  if (tid == 0) {  // first position of each weight, heaviest first
    int pos = 0;
    for (int w = T; w >= 0; --w) {
      const int h = hist[w];
      hist[w] = pos;
      pos += h;
    }
    plan[0] = pos;
    plan[1] = nsplit;
  }
  __syncthreads();
  // items: the whole range [0, T-1] for an unsplit key tile (the kernel
  // walks its live tiles), consecutive query-tile ranges for the parts
  for (int kt = tid; kt < T; kt += nth) {
    const int c = cnt[kt], n = meta[kt] & 0xffff, base = meta[kt] >> 16;
    for (int k = 0; k < n; ++k) {
      const int qa = k == 0 ? 0 : start[base + k];
      const int qb = k == n - 1 ? T - 1 : start[base + k + 1] - 1;
      const int w = (k + 1) * c / n - k * c / n;
      items[atomicAdd(&hist[w], 1)] = make_int4(kt, qa, qb, k | (n << 8) | (base << 16));
    }
  }
  for (int sk = tid; sk < nsplit; sk += nth) {
    const int kt = split_kt[sk];
    plan[2 + 3 * sk] = kt;
    plan[3 + 3 * sk] = meta[kt] >> 16;
    plan[4 + 3 * sk] = meta[kt] & 0xffff;
  }
}

// Join of the split key tiles: block (j, bh) adds the fp32 parts of split
// key tile j of head bh in part order, scales dK, rounds both to bf16 and
// writes the tile's rows below N.  Eight consecutive values per thread step.
template <int D>
__global__ void __launch_bounds__(256)
    bwd_split_join_kernel(const Problem p, long long heads, const int* __restrict__ plan,
                          const float* __restrict__ slots, __nv_bfloat16* __restrict__ dk,
                          __nv_bfloat16* __restrict__ dv) {
  const int j = blockIdx.x;
  griddep_wait();
  griddep_release();
  if (j >= __ldg(plan + 1)) return;
  const int kt = __ldg(plan + 2 + 3 * j), base = __ldg(plan + 3 + 3 * j),
            n = __ldg(plan + 4 + 3 * j);
  constexpr int kPart = 2 * 128 * D;  // floats of one part: dK rows, then dV rows
  for (long long bh = blockIdx.y; bh < heads; bh += gridDim.y) {
    const float* src = slots + ((size_t)bh * kSplitSlots + base) * kPart;
    for (int e = threadIdx.x * 8; e < kPart; e += 256 * 8) {
      float acc[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) acc[u] = 0.f;
      for (int k = 0; k < n; ++k) {
        const float4 x0 = __ldg(reinterpret_cast<const float4*>(src + (size_t)k * kPart + e));
        const float4 x1 = __ldg(reinterpret_cast<const float4*>(src + (size_t)k * kPart + e + 4));
        acc[0] += x0.x, acc[1] += x0.y, acc[2] += x0.z, acc[3] += x0.w;
        acc[4] += x1.x, acc[5] += x1.y, acc[6] += x1.z, acc[7] += x1.w;
      }
      const int t = e / (128 * D), r = (e / D) & 127, c = e % D;
      const int row = kt * 128 + r;
      if (row >= p.N) continue;
      const float mul = t == 0 ? p.scale : 1.f;
      const uint4 w = make_uint4(pack_bf16(acc[0] * mul, acc[1] * mul),
                                 pack_bf16(acc[2] * mul, acc[3] * mul),
                                 pack_bf16(acc[4] * mul, acc[5] * mul),
                                 pack_bf16(acc[6] * mul, acc[7] * mul));
      *reinterpret_cast<uint4*>((t == 0 ? dk : dv) + ((size_t)bh * p.N + row) * D + c) = w;
    }
  }
}

cudaError_t launch_bwd_plan(const Problem& p, const BwdSplit& split, cudaStream_t st) {
  // the current device's SM count, asked on every call (a few hundred
  // nanoseconds; a process-wide cache would be wrong across devices and
  // racy across host threads)
  int dev = 0, nsm = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
    return e;
  return launch_k(true, bwd_plan_kernel, dim3(1), dim3(1024), 0, st, p, nsm,
                  (long long)p.B * p.H, const_cast<int4*>(split.items),
                  const_cast<int*>(split.nitems));
}

// early: launched straight after the preprocess kernel, which waited for the
// split plan (launched before it); the kernel may then start while the
// preprocess is still running.
template <int D, bool PACKED, bool DROP, bool SPLIT, bool LOSE = false>
static cudaError_t launch_bwd_tc_t(const Problem& pin, const void* q, const void* k,
                                   const void* v, const void* dout, const float* lse2,
                                   const float* dvec, float* dq_acc, void* dk, void* dv, int npad,
                                   const BwdSplit& split, unsigned long long* next_item,
                                   bool early, cudaStream_t st) {
  using C = BwdTc<D>;
  // Heads per CTA group: Q, dO (bf16) and the fp32 dQ accumulator of a group
  // within about 64 MB (half of L2).
  Problem p = pin;
  {
    const long long heads = (long long)p.B * p.H;
    long long g = (64ll << 20) / ((long long)p.N * D * 8);
    p.hgroup = (int)(g < 1 ? 1 : (g > heads ? heads : g));
  }
  const long long bh = (long long)p.B * p.H;
  cudaError_t e;
  if constexpr (SPLIT) {
    if (!early && (e = launch_bwd_plan(p, split, st)) != cudaSuccess) return e;
  }
  if constexpr (D == 64 && !PACKED && !DROP) {
    // d = 64: the persistent kernel (fa_bwd_persist.cu)
    e = launch_bwd_persist(p, q, k, v, dout, lse2, dvec, dq_acc, dk, dv, npad,
                           SPLIT ? &split : nullptr, next_item, early, st, LOSE);
  } else {
    CUtensorMap tq, tk, tv, tdo, tdk, tdv, tdq;
    bool maps;
    if constexpr (PACKED)
      maps = make_bf16_map_packed(&tq, q, D, p.H, p.total, C::BQ) &&
             make_bf16_map_packed(&tk, k, D, p.H, p.total, 128) &&
             make_bf16_map_packed(&tv, v, D, p.H, p.total, 128) &&
             make_bf16_map_packed(&tdo, dout, D, p.H, p.total, C::BQ) &&
             make_bf16_map_packed(&tdk, dk, D, p.H, p.total, 128) &&
             make_bf16_map_packed(&tdv, dv, D, p.H, p.total, 128) &&
             make_f32_map_3d(&tdq, dq_acc, D, p.total, p.H, C::BQ, 32);
    else
      maps = make_bf16_map_3d(&tq, q, D, p.N, bh, C::BQ) &&
             make_bf16_map_3d(&tk, k, D, p.N, bh, 128) &&
             make_bf16_map_3d(&tv, v, D, p.N, bh, 128) &&
             make_bf16_map_3d(&tdo, dout, D, p.N, bh, C::BQ) &&
             make_bf16_map_3d(&tdk, dk, D, p.N, bh, 128) &&
             make_bf16_map_3d(&tdv, dv, D, p.N, bh, 128) &&
             make_f32_map_3d(&tdq, dq_acc, D, p.N, bh, C::BQ, 32);
    if (!maps) return cudaErrorInvalidValue;
    auto kern = bwd_tc_kernel<D, PACKED, DROP, SPLIT, LOSE>;
    constexpr int threads = BwdEw<D, DROP>::THREADS;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(bh * p.T * (SPLIT ? kSplitMax : 1)));
    e = launch_k(early, kern, grid, dim3(threads), C::SMEM, st, tq, tk, tv, tdo, tdk, tdv, tdq, p,
                 lse2, dvec, dq_acc, npad, static_cast<__nv_bfloat16*>(dk),
                 static_cast<__nv_bfloat16*>(dv), split);
  }
  if constexpr (SPLIT) {
    if (e != cudaSuccess) return e;
    dim3 jgrid(kSplitSlots / 2, (unsigned)(bh < 65535 ? bh : 65535));
    e = launch_k(true, bwd_split_join_kernel<D>, jgrid, dim3(256), 0, st, p, bh,
                 (const int*)split.nitems, (const float*)split.slots,
                 static_cast<__nv_bfloat16*>(dk), static_cast<__nv_bfloat16*>(dv));
  }
  return e;
}

template <bool PACKED, bool DROP, bool SPLIT>
static cudaError_t launch_bwd_tc_d(const Problem& p, const void* q, const void* k, const void* v,
                                   const void* dout, const float* lse2, const float* dvec,
                                   float* dq_acc, void* dk, void* dv, int npad,
                                   const BwdSplit& split, unsigned long long* next_item,
                                   bool early, cudaStream_t st) {
  return p.d == 64 ? launch_bwd_tc_t<64, PACKED, DROP, SPLIT>(p, q, k, v, dout, lse2, dvec,
                                                              dq_acc, dk, dv, npad, split,
                                                              next_item, early, st)
                   : launch_bwd_tc_t<128, PACKED, DROP, SPLIT>(p, q, k, v, dout, lse2, dvec,
                                                               dq_acc, dk, dv, npad, split,
                                                               next_item, early, st);
}

cudaError_t launch_bwd_tc_lost_signal(const Problem& p, const void* q, const void* k,
                                      const void* v, const void* dout, const float* lse2,
                                      const float* dvec, float* dq_acc, void* dk, void* dv,
                                      int npad, unsigned long long* next_item, cudaStream_t st) {
  if ((p.d != 128 && p.d != 64) || p.cu_seqlens != nullptr || p.drop_p8 != 0)
    return cudaErrorInvalidValue;
  const BwdSplit none{nullptr, nullptr, nullptr};
  return p.d == 128 ? launch_bwd_tc_t<128, false, false, false, true>(
                          p, q, k, v, dout, lse2, dvec, dq_acc, dk, dv, npad, none, nullptr,
                          false, st)
                    : launch_bwd_tc_t<64, false, false, false, true>(
                          p, q, k, v, dout, lse2, dvec, dq_acc, dk, dv, npad, none, next_item,
                          false, st);
}

cudaError_t launch_bwd_tc(const Problem& p, const void* q, const void* k, const void* v,
                          const void* dout, const float* lse2, const float* dvec, float* dq_acc,
                          void* dk, void* dv, int npad, const BwdSplit* split,
                          unsigned long long* next_item, bool early, cudaStream_t st) {
  const bool packed = p.cu_seqlens != nullptr, drop = p.drop_p8 != 0;
  const BwdSplit none{nullptr, nullptr, nullptr};
  if (packed)
    return drop ? launch_bwd_tc_d<true, true, false>(p, q, k, v, dout, lse2, dvec, dq_acc, dk, dv,
                                                     npad, none, next_item, early, st)
                : launch_bwd_tc_d<true, false, false>(p, q, k, v, dout, lse2, dvec, dq_acc, dk,
                                                      dv, npad, none, next_item, early, st);
  if (split != nullptr)
    return drop ? launch_bwd_tc_d<false, true, true>(p, q, k, v, dout, lse2, dvec, dq_acc, dk, dv,
                                                     npad, *split, next_item, early, st)
                : launch_bwd_tc_d<false, false, true>(p, q, k, v, dout, lse2, dvec, dq_acc, dk,
                                                      dv, npad, *split, next_item, early, st);
  return drop ? launch_bwd_tc_d<false, true, false>(p, q, k, v, dout, lse2, dvec, dq_acc, dk, dv,
                                                    npad, none, next_item, early, st)
              : launch_bwd_tc_d<false, false, false>(p, q, k, v, dout, lse2, dvec, dq_acc, dk, dv,
                                                     npad, none, next_item, early, st);
}

}  // namespace fa
