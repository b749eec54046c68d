// Tensor-core (tcgen05 + TMA) tiled attention forward for sm_103a.
//
// One CTA owns two 128-row query tiles of one (b, h) (tiles 2p and 2p+1) and
// streams the union of their live 128-key tiles (block mask, causal rule,
// key limit; dead tiles are never loaded) through a ring of shared-memory
// slots filled by TMA, in stages of {V_j, K_(j+1)} (one full and one empty
// barrier per key tile).  The SOLO instantiation owns one query tile (warps
// 2-5 do its softmax, TMEM columns S [0,128), O [128,128+d)) and runs two
// CTAs per SM; at d = 64 it keeps P in columns of its own, otherwise (P over
// S) its ring is of single K and V tiles.
// The online-softmax recurrence of page
// "FlashAttention" (aiwiki), section "Tiling and online normalization", is
// evaluated per query row in log2 units with a lazily moved reference:
//     m' = max over the tile of scale*log2(e)*q.k_j
//     if m' > m + 8:  alpha = 2^(m - m'),  m = m'          (else alpha = 1)
//     p_j = 2^(scale*log2(e)*q.k_j - m),  l = alpha*l + sum_j p_j,
//     u = alpha*u + sum_j p_j v_j,        O = u / l,  LSE = ln2*(m + log2 l)
// Keeping m below the running max by at most 8 bounds p_j by 2^8 and leaves
// u / l unchanged (the reference cancels), so the result is exact up to
// rounding; it saves most rescalings of the accumulator.
//
// Warp roles (384 threads):
//   warp 0      TMA producer: Q tiles once, then V_j and K_(j+1) into a stage.
//   warp 1      MMA issuer (one thread): S_i = Q_i K_j^T into TMEM, then
//               O_i += P_i V_j with P_i read from TMEM; owns TMEM.
//   warps 4-7   softmax for query tile 0 (TMEM lanes 0-127, one row per thread)
//   warps 8-11  softmax for query tile 1
// The softmax warps read S from TMEM, write P (bf16) back over it, rescale
// O in TMEM when the reference moves, and finally normalise O, store it
// through shared memory with a TMA store, and write LSE.
//
// TMEM columns: S0 [0,128), S1 [128,256), O0 [256,256+d), O1 [256+d,256+2d).
// MMA order per key tile j:  PV0(j), S0(j+1), PV1(j), S1(j+1); tcgen05 ops of
// one thread execute in issue order, so S_i(j+1) overwrites P_i(j) only after
// PV_i(j) has read it, and the commit that signals S_i(j+1) also covers
// PV_i(j) (the softmax warps may then touch O_i).
#include <cuda_bf16.h>

#include "fa_common.cuh"
#include "fa_kernels.h"
#include "fa_sm100.cuh"
#include "fa_tma_host.h"

namespace fa {
using namespace sm100;

// Words of the per-CTA key-tile bitmask of one query tile (up to 65536 tiles).
constexpr int kFwdLiveWords = 65536 / 32;

// SOLO: one query tile per CTA (192 threads: producer, MMA issuer, four
// softmax warps; 256 TMEM columns; a shallower ring) so that two CTAs share
// an SM -- for short sequences, where a CTA's fixed costs (set-up, first
// tile, epilogue) are a large part of its time and two CTAs hide each
// other's.
template <int D, bool SOLO = false>
struct FwdTc {
  static constexpr int THREADS = SOLO ? 192 : 384;
  static constexpr int WARP_SM = SOLO ? 2 : 4;   // first softmax warp
  static constexpr int NQ = SOLO ? 1 : 2;        // query tiles per CTA
  static constexpr int NSLOT = SOLO ? (D == 64 ? 4 : 2) : (D == 64 ? 8 : 4);  // K/V ring slots
  static constexpr int HALF = 128 * 128;         // one 128-row x 64-col bf16 box
  static constexpr int TILE = 128 * D * 2;       // one 128-row tile
  static constexpr int OFF_Q = 0;                // Q0, Q1 (reused for O staging)
  static constexpr int OFF_KV = NQ * TILE;
  static constexpr int OFF_BAR = OFF_KV + NSLOT * TILE;
  // barriers: q_full, kv_full[NSLOT], kv_empty[NSLOT] (one per slot, or
  // one per stage of two slots in the staged ring, which uses the first
  // NSLOT / 2 of each), s_full[2], p_ready[2], o_done[2], drain
  static constexpr int B_Q = 0, B_FULL = 1, B_EMPTY = 1 + NSLOT, B_S = 1 + 2 * NSLOT,
                       B_P = B_S + 2, B_O = B_P + 2, B_DRAIN = B_O + 2, NBAR = B_DRAIN + 1;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  // live key tiles of the union's range under a block mask, one bit each,
  // for query tile 0 and query tile 1
  static constexpr int OFF_LIVE = (OFF_MISC + 64 + 127) / 128 * 128;
  static constexpr int SMEM = OFF_LIVE + NQ * kFwdLiveWords * 4 + 1024;  // + slack for 1024-byte alignment
  static_assert(SMEM <= (SOLO ? 232448 / 2 - 1024 : 232448), "shared memory budget");
  static constexpr int COL_S0 = 0, COL_S1 = 128, COL_O0 = SOLO ? 128 : 256, COL_O1 = 256 + D;
  static constexpr uint32_t TMEM_COLS = SOLO ? 256 : 512;
  // One-tile CTAs at d = 64 (SEPP): P has TMEM columns of its own (S 0-127,
  // O 128-191, P 192-255), so S of the next key tile is computed as soon as
  // the softmax has read this one into registers, while it still works on
  // it.  The second tile's barriers serve as s_free (the softmax warps have
  // read S) and p_free (the P . V that read P has completed).
  static constexpr bool SEPP = SOLO && D == 64;  // used by the kernel without dropout
  static constexpr int COL_P = 192, B_SFREE = B_S + 1, B_PFREE = B_P + 1;
};

// Next key tile after kt that is live for query tile q0 or q1, within the
// union's range [first, last] (the union of two adjacent tiles' ranges is one
// range: query tile q0 + 1 starts at most one tile later than q0 ends).
// Under a block mask the liveness comes from `live` (bit t of word block 0 /
// 1: key tile first + t for query tile q0 / q1), built once per CTA rather
// than read from the mask in every role's loop.
template <bool SOLO = false>
__device__ __forceinline__ int next_union_tile(const Problem& p, const uint32_t* live, int first,
                                               int last, int kt) {
  kt = kt + 1 < first ? first : kt + 1;
  if (p.block_mask == nullptr) return kt <= last ? kt : p.T;
  while (kt <= last) {
    const int t = kt - first;
    const uint32_t w =
        (live[t >> 5] | (SOLO ? 0u : live[kFwdLiveWords + (t >> 5)])) >> (t & 31);
    if (w != 0) return kt + __ffs(w) - 1;  // bits past the range are 0
    kt += 32 - (t & 31);
  }
  return p.T;
}

// Whether key tile kt (within [first, last]) is live for query tile i of the
// CTA, from the bitmask above.
__device__ __forceinline__ bool live_bit(const uint32_t* live, int i, int first, int kt) {
  const int t = kt - first;
  return (live[i * kFwdLiveWords + (t >> 5)] >> (t & 31)) & 1u;
}

// One key tile of the online softmax for one query row (TMEM lane =
// thread): S from TMEM columns col_s, the row's mask, the lazily moved
// reference m_ref and the running sum l (O at col_o rescaled when the
// reference moves and `rescale_o`), P as bf16 written to columns col_p
// (over S, or columns of its own).  after_load() runs once S is in
// registers, before_store() before P or O is written.  The caller waits for
// the TMEM stores before signalling P.
template <int D, bool DROP, class AfterLoad, class BeforeStore>
__device__ __forceinline__ void softmax_tile(const Problem& p, long long bh, int row, int kt,
                                             int klim, uint32_t lane_base, uint32_t col_s,
                                             uint32_t col_o, uint32_t col_p, bool rescale_o,
                                             float& m_ref, float& l, AfterLoad after_load,
                                             BeforeStore before_store) {
  const float cl2 = p.scale_log2;
  float s[128];
  {
    uint32_t raw[128];
    tmem_ld128(lane_base + col_s, raw);
#pragma unroll
    for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(raw[c]);
  }
  after_load();
  // This row's allowed keys in the tile: columns [lo, hi).  Masked
  // scores get the value that the scale sends to -inf (and that the
  // row max / min below ignores), so p = 2^-inf = 0 for either sign.
  {
    const int k0 = kt * 128;
    const int lo = row_key_lo(p, row) - k0;
    const int hi = row_key_hi(p, row, klim) + 1 - k0;
    if (lo > 0 || hi < 128) {
      const float fill = cl2 >= 0.f ? -INFINITY : INFINITY;
#pragma unroll
      for (int c = 0; c < 128; ++c)
        if (c < lo || c >= hi) s[c] = fill;
    }
  }
  // row max (row min for a negative scale): 4 independent chains of
  // 3-input max
  float mx;
  if (cl2 >= 0.f) {
    // s[0..3] seed the chains; 15 steps cover s[4..123]; s[124..127] last
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
    alpha = fast_exp2(m_ref - m_tile);  // 0 when m_ref = -inf
    m_ref = m_tile;
  }
  const float nref = m_ref == -INFINITY ? 0.f : -m_ref;
  before_store();
  // p = 2^(s * scale*log2e - m): argument by packed FMA, exp2 on MUFU,
  // row sum by packed adds over four independent pairs
  float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    // dropout: keep bits of the chunk's 32 keys (two generator calls of
    // 16 keys each); dropped probabilities still count in the row sum
    uint32_t keep = 0xffffffffu;
    if constexpr (DROP) {
      const uint4 a = dropout_bytes(p, bh, row, kt * 8 + 2 * c);
      const uint4 b2 = dropout_bytes(p, bh, row, kt * 8 + 2 * c + 1);
      keep = keep4(a.x, p.drop_p8) | keep4(a.y, p.drop_p8) << 4 |
             keep4(a.z, p.drop_p8) << 8 | keep4(a.w, p.drop_p8) << 12 |
             keep4(b2.x, p.drop_p8) << 16 | keep4(b2.y, p.drop_p8) << 20 |
             keep4(b2.z, p.drop_p8) << 24 | keep4(b2.w, p.drop_p8) << 28;
    }
    uint32_t pk[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      float x0, x1;
      fma2(x0, x1, s[32 * c + 2 * j], s[32 * c + 2 * j + 1], cl2, cl2, nref, nref);
      const float p0 = fast_exp2(x0);
      const float p1 = fast_exp2(x1);
      add2(sa[j & 3], sb[j & 3], sa[j & 3], sb[j & 3], p0, p1);
      if constexpr (DROP)
        pk[j] = pack_bf16((keep >> (2 * j)) & 1u ? p0 : 0.f,
                          (keep >> (2 * j + 1)) & 1u ? p1 : 0.f);
      else
        pk[j] = pack_bf16(p0, p1);
    }
    tmem_st16(lane_base + col_p + 16 * c, pk);
  }
  const float sum = ((sa[0] + sb[0]) + (sa[1] + sb[1])) + ((sa[2] + sb[2]) + (sa[3] + sb[3]));
  l = l * alpha + sum;
  if (rescale_o && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      tmem_ld32(lane_base + col_o + 32 * c, o);
#pragma unroll
      for (int j = 0; j < 32; ++j) o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha);
      tmem_st32(lane_base + col_o + 32 * c, o);
    }
  }
}

// LOSE: self-test instantiation only (fa_selftest_forward_lost_signal): the
// first softmax warp withholds its P-ready arrival for the first key tile
// and every wait gives up after 1 ms, so the MMA issuer's wait runs out and
// the abort, drain and status paths run.
template <int D, bool PACKED, bool DROP, bool SOLO, bool LOSE = false>
__global__ void __launch_bounds__(FwdTc<D, SOLO>::THREADS, SOLO ? 2 : 1)
    fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const Problem pin, float* __restrict__ lse, __nv_bfloat16* __restrict__ o_rows) {
  using C = FwdTc<D, SOLO>;
  // P in columns of its own (one-tile CTAs at d = 64; with dropout the
  // extra waits cost registers the Philox rounds need, so P stays over S)
  constexpr bool SEPP = C::SEPP && !DROP;
  // the staged K/V ring (below) everywhere but the one-tile kernel with P over S
  constexpr bool STAGED = SEPP || !SOLO;
  // Geometry of this CTA's (b, h): padded layout [B*H][N][d] (TMA coordinates
  // (x, row, bh)), or one sequence of the packed layout [total][H][d]
  // (coordinates (x, h, start + row)), whose length then plays the role of N.
  // Grid: one CTA per (head, query-tile pair) in the grouped order
  // (heaviest pairs first across a group of heads whose K and V stay in L2);
  // SOLO: one CTA per (head, query tile), in the same order.
  const int npairs_grid = SOLO ? pin.T : (pin.T + 1) / 2;
  long long bh;
  int yi;
  grouped_cta(pin, blockIdx.x, npairs_grid, bh, yi);
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
  const int npairs = SOLO ? p.T : (p.T + 1) / 2;
  if (yi >= npairs) return;  // packed: past this sequence's tiles
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

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = npairs - 1 - yi;  // heaviest causal pairs first
  const int qt0 = SOLO ? pair : 2 * pair;
  const int qt1 = (!SOLO && 2 * pair + 1 < p.T) ? 2 * pair + 1 : -1;
  const int klim = key_limit(p, b);
  // Live key tiles of each query tile (exact without a block mask, a bound
  // with one) and of their union.
  int first0, last0, first1 = 0, last1 = -1;
  qtile_key_tiles(p, qt0, klim, first0, last0);
  if (qt1 >= 0) qtile_key_tiles(p, qt1, klim, first1, last1);
  const int ufirst = first0 <= last0 ? first0 : first1;
  const int ulast = max(last0, last1);

  if (warp == 0) {
    // the barriers, one per lane of warp 0
    for (int i = lane; i < C::NBAR; i += 32)
      mbar_init(bar(i), (i == C::B_P || (i == C::B_P + 1 && !SEPP) || (i == C::B_SFREE && SEPP))
                            ? 4
                            : 1);
    fence_barrier_init();
    __syncwarp();
  }
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    // the query tiles, issued by the producer thread before the rest of the
    // set-up (TMEM, the live bitmask, the CTA barrier) so that their latency
    // overlaps it
    mbar_expect_tx(bar(C::B_Q), (qt1 >= 0 ? 2 : 1) * C::TILE);
    for (int h = 0; h < D / 64; ++h) {
      tma_load_3d(s0 + C::OFF_Q + h * C::HALF, &tm_q, bar(C::B_Q), h * 64, cy(qt0 * 128),
                  cz(qt0 * 128));
      if (qt1 >= 0)
        tma_load_3d(s0 + C::OFF_Q + C::TILE + h * C::HALF, &tm_q, bar(C::B_Q), h * 64,
                    cy(qt1 * 128), cz(qt1 * 128));
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  const uint32_t* live = reinterpret_cast<const uint32_t*>(smem + C::OFF_LIVE);
  if (p.block_mask != nullptr) {
    // liveness over the union's range, 32 key tiles per warp and word
    const int n = ulast - ufirst + 1;
    for (int wi = warp; wi < ((n + 31) >> 5); wi += C::THREADS / 32) {
      const int t = (wi << 5) + lane, kt = ufirst + t;
      const uint32_t b0 = __ballot_sync(0xffffffffu, t < n && tile_live(p, qt0, kt, klim));
      const uint32_t b1 =
          __ballot_sync(0xffffffffu, t < n && qt1 >= 0 && tile_live(p, qt1, kt, klim));
      if (lane == 0) {
        reinterpret_cast<uint32_t*>(smem + C::OFF_LIVE)[wi] = b0;
        if constexpr (!SOLO) reinterpret_cast<uint32_t*>(smem + C::OFF_LIVE)[kFwdLiveWords + wi] = b1;
      }
    }
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tm_q);
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_v);
    prefetch_tensormap(&tm_o);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (STAGED && warp <= 1) {
    // Staged ring (two-tile CTAs, and one-tile CTAs at d = 64 without
    // dropout): NSTAGE stages of two slots, stage t holding V of the t-th
    // live key tile of the union and K of the next one (slots 2s and 2s + 1,
    // s = t mod NSTAGE) on one full and one empty barrier, so that a key
    // tile costs the issuer one load wait and one release.  K of the first
    // tile goes to the last stage's K slot ahead of that stage's first use.
    constexpr int NSTAGE = C::NSLOT / 2, LAST = NSTAGE - 1;
    constexpr uint32_t slot_step = C::TILE >> 4;  // descriptor units per ring slot
    if (warp == 0 && lane == 0) {
      // ---------------------------------------------------------- producer
      auto load_tile = [&](const CUtensorMap* map, int slot, uint32_t fb, int kt) {
        for (int h = 0; h < D / 64; ++h)
          tma_load_3d(s0 + C::OFF_KV + slot * C::TILE + h * C::HALF, map, fb, h * 64,
                      cy(kt * 128), cz(kt * 128));
      };
      bool ok = true;
      int kt = next_union_tile<SOLO>(p, live, ufirst, ulast, -1);
      int t = 0;  // stages issued
      const int first_k = kt < p.T ? 1 : 0;
      if (first_k) {
        mbar_expect_tx(bar(C::B_FULL + LAST), C::TILE);
        load_tile(&tm_k, 2 * LAST + 1, bar(C::B_FULL + LAST), kt);
      }
      while (ok && kt < p.T) {
        const int nxt = next_union_tile<SOLO>(p, live, ufirst, ulast, kt);
        const int s = t % NSTAGE;
        // stage t reuses the slots of stage t - NSTAGE, released by the
        // issuer after key tile t - NSTAGE; the last stage's first use waits
        // for the first S instead (its K slot held the first K)
        if (s == LAST || t >= NSTAGE) {
          const int ph = s == LAST ? t / NSTAGE : t / NSTAGE - 1;
          if (!(ok = mbar_wait(bar(C::B_EMPTY + s), ph & 1, ab, kSleepHintNs))) break;
        }
        const uint32_t fb = bar(C::B_FULL + s);
        mbar_expect_tx(fb, (nxt < p.T ? 2 : 1) * C::TILE);
        load_tile(&tm_v, 2 * s, fb, kt);
        if (nxt < p.T) load_tile(&tm_k, 2 * s + 1, fb, nxt);
        ++t;
        kt = nxt;
      }
      // Drain (matters only after an abort): the last phase issued on each
      // full barrier (stages s, s + NSTAGE, ...; the first K too on the
      // last one) and the query tiles.
      for (int s = 0; s < NSTAGE; ++s) {
        const int nph = (t > s ? (t - s - 1) / NSTAGE + 1 : 0) + (s == LAST ? first_k : 0);
        if (nph == 0) continue;
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(bar(C::B_FULL + s), (nph - 1) & 1) &&
               globaltimer() - t0 < kWaitLimitNs) {
        }
      }
      {
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(bar(C::B_Q), 0) && globaltimer() - t0 < kWaitLimitNs) {
        }
      }
    } else if (warp == 1 && lane == 0) {
      // ------------------------------------------------------- MMA issuer
      constexpr uint32_t id_qk = idesc_bf16(128, 128, false, false);
      constexpr uint32_t id_pv = idesc_bf16(128, D, false, true);
      const uint64_t dq0 = sdesc_sw128(s0 + C::OFF_Q, 16, 1024);
      const uint64_t dq1 = sdesc_sw128(s0 + C::OFF_Q + C::TILE, 16, 1024);
      const uint64_t dk0 = sdesc_sw128(s0 + C::OFF_KV, 16, 1024);      // K operand of slot 0
      const uint64_t dv0 = sdesc_sw128(s0 + C::OFF_KV, C::HALF, 1024);  // V operand of slot 0
      const uint32_t t_s0 = tmem + C::COL_S0, t_s1 = tmem + C::COL_S1;
      const uint32_t t_o0 = tmem + C::COL_O0, t_o1 = tmem + C::COL_O1;
      auto qk = [&](uint32_t t_s, uint64_t dq, int slot) {
        if (D == 128)
          mma_ss_kmajor_k128_h16k(t_s, dq, dk0 + (uint64_t)(slot * slot_step), id_qk, 0);
        else
          mma_ss_kmajor_k64(t_s, dq, dk0 + (uint64_t)(slot * slot_step), id_qk, 0);
      };
      const bool masked = p.block_mask != nullptr;
      auto live0 = [&](int kt) {
        return masked ? live_bit(live, 0, ufirst, kt) : (kt >= first0 && kt <= last0);
      };
      auto live1 = [&](int kt) {
        if constexpr (SOLO) return false;
        return masked ? live_bit(live, 1, ufirst, kt) : (kt >= first1 && kt <= last1);
      };
      bool ok = mbar_wait(bar(C::B_Q), 0, ab);
      tc_fence_after();
      int kt = next_union_tile<SOLO>(p, live, ufirst, ulast, -1);
      int ns0 = 0;  // S of query tile 0 issued (one-tile d = 64: for s_free)
      if (ok && kt < p.T) {
        ok = mbar_wait(bar(C::B_FULL + LAST), 0, ab);
        tc_fence_after();
        if (ok) {
          if (SOLO || live0(kt)) {
            qk(t_s0, dq0, 2 * LAST + 1);
            mma_commit(bar(C::B_S + 0));
            ++ns0;
          }
          if (live1(kt)) {
            qk(t_s1, dq1, 2 * LAST + 1);
            mma_commit(bar(C::B_S + 1));
          }
          mma_commit(bar(C::B_EMPTY + LAST));
        }
      }
      int npv0 = 0, npv1 = 0;
      for (int j = 0; ok && kt < p.T; ++j) {
        const int nxt = next_union_tile<SOLO>(p, live, ufirst, ulast, kt);
        const int s = j % NSTAGE;
        // a one-tile CTA's union is its own tiles: every tile is live
        const bool l0 = SOLO || live0(kt), l1 = live1(kt);
        const bool n0 = nxt < p.T && (SOLO || live0(nxt)), n1 = nxt < p.T && live1(nxt);
        const uint64_t dv = dv0 + (uint64_t)(2 * s * slot_step);
        // stage j is phase j / NSTAGE of its full barrier (one more on the
        // last barrier, which first carried the first K)
        const int ph = s == LAST ? j / NSTAGE + 1 : j / NSTAGE;
        if (!(ok = mbar_wait(bar(C::B_FULL + s), ph & 1, ab))) break;
        tc_fence_after();
        if constexpr (SEPP) {
          // the next S as soon as the softmax has read this one (P has
          // columns of its own), then P . V once P is ready
          if (n0) {
            if (!(ok = mbar_wait(bar(C::B_SFREE), (ns0 - 1) & 1, ab))) break;
            tc_fence_after();
            qk(t_s0, dq0, 2 * s + 1);
            mma_commit(bar(C::B_S + 0));
            ++ns0;
          }
          if (l0) {
            if (!(ok = mbar_wait(bar(C::B_P + 0), npv0 & 1, ab))) break;
            tc_fence_after();
            mma_ts_mn_k128(t_o0, tmem + C::COL_P, dv, id_pv, npv0 > 0);
            mma_commit(bar(C::B_PFREE));
            ++npv0;
          }
        } else {
          // P over S: S_i of the next tile after P_i . V has read P_i
          if (l0) {
            if (!(ok = mbar_wait(bar(C::B_P + 0), npv0 & 1, ab))) break;
            tc_fence_after();
            mma_ts_mn_k128(t_o0, t_s0, dv, id_pv, npv0 > 0);
            ++npv0;
          }
          if (n0) {
            qk(t_s0, dq0, 2 * s + 1);
            mma_commit(bar(C::B_S + 0));
          }
          if (l1) {
            if (!(ok = mbar_wait(bar(C::B_P + 1), npv1 & 1, ab))) break;
            tc_fence_after();
            mma_ts_mn_k128(t_o1, t_s1, dv, id_pv, npv1 > 0);
            ++npv1;
          }
          if (n1) {
            qk(t_s1, dq1, 2 * s + 1);
            mma_commit(bar(C::B_S + 1));
          }
        }
        mma_commit(bar(C::B_EMPTY + s));
        kt = nxt;
      }
      mma_commit(bar(C::B_O + 0));
      if constexpr (!SOLO) mma_commit(bar(C::B_O + 1));
      // Drain all issued tensor-core work before TMEM can be released.
      mma_commit(bar(C::B_DRAIN));
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(bar(C::B_DRAIN), 0) && globaltimer() - t0 < kWaitLimitNs) {
      }
    }
  } else if (warp == 0) {
    // ------------------------------------------------------------ producer
    // (unstaged: the one-tile kernel with P over S -- d = 128, or dropout --
    // whose two slots hold one key tile's K and V, each released on its own)
    if (lane == 0) {
      int slot = 0, round = 0;
      // per-slot count of loads issued, for the final drain
      bool ok = true;
      for (int kt = next_union_tile<SOLO>(p, live, ufirst, ulast, -1); kt < p.T && ok;
           kt = next_union_tile<SOLO>(p, live, ufirst, ulast, kt)) {
        for (int which = 0; which < 2; ++which) {
          if (!mbar_wait(bar(C::B_EMPTY + slot), (round & 1) ^ 1, ab, kSleepHintNs)) {
            ok = false;
            break;
          }
          const uint32_t dst = s0 + C::OFF_KV + slot * C::TILE;
          mbar_expect_tx(bar(C::B_FULL + slot), C::TILE);
          for (int h = 0; h < D / 64; ++h)
            tma_load_3d(dst + h * C::HALF, which == 0 ? &tm_k : &tm_v, bar(C::B_FULL + slot),
                        h * 64, cy(kt * 128), cz(kt * 128));
          if (++slot == C::NSLOT) {
            slot = 0;
            ++round;
          }
        }
      }
      // Drain: every load issued must have landed before shared memory is
      // released (matters only after an abort; otherwise these phases have
      // completed already).  Slot s was last filled in round
      // round - (s >= slot ? 1 : 0).
      for (int s = 0; s < C::NSLOT; ++s) {
        const int last = round - (s >= slot ? 1 : 0);
        if (last >= 0) {
          const uint64_t t0 = globaltimer();
          while (!mbar_try_wait(bar(C::B_FULL + s), last & 1) &&
                 globaltimer() - t0 < kWaitLimitNs) {
          }
        }
      }
      {
        const uint64_t t0 = globaltimer();
        while (!mbar_try_wait(bar(C::B_Q), 0) && globaltimer() - t0 < kWaitLimitNs) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // (unstaged, as the producer above; the second query tile's branches are
    // compiled out there.)  Kept lean: one thread issues every GEMM as a
    // single instruction sequence from precomputed descriptors, so the
    // tensor core is not left waiting on this thread's bookkeeping.
    if (lane == 0) {
      constexpr uint32_t id_qk = idesc_bf16(128, 128, false, false);
      constexpr uint32_t id_pv = idesc_bf16(128, D, false, true);
      constexpr uint32_t slot_step = C::TILE >> 4;  // descriptor units per ring slot
      const uint64_t dq0 = sdesc_sw128(s0 + C::OFF_Q, 16, 1024);
      const uint64_t dq1 = sdesc_sw128(s0 + C::OFF_Q + C::TILE, 16, 1024);
      const uint64_t dk0 = sdesc_sw128(s0 + C::OFF_KV, 16, 1024);      // K operand of slot 0
      const uint64_t dv0 = sdesc_sw128(s0 + C::OFF_KV, C::HALF, 1024);  // V operand of slot 0
      const uint32_t t_s0 = tmem + C::COL_S0, t_s1 = tmem + C::COL_S1;
      const uint32_t t_o0 = tmem + C::COL_O0, t_o1 = tmem + C::COL_O1;
      auto qk = [&](uint32_t t_s, uint64_t dq, int slot) {
        if (D == 128)
          mma_ss_kmajor_k128_h16k(t_s, dq, dk0 + (uint64_t)(slot * slot_step), id_qk, 0);
        else
          mma_ss_kmajor_k64(t_s, dq, dk0 + (uint64_t)(slot * slot_step), id_qk, 0);
      };
      // Liveness of key tile kt for query tile 0 / 1: without a block mask
      // it is first_i <= kt <= last_i, so the loop needs no predicate calls.
      const bool masked = p.block_mask != nullptr;
      auto live0 = [&](int kt) {
        return masked ? live_bit(live, 0, ufirst, kt) : (kt >= first0 && kt <= last0);
      };
      auto live1 = [&](int kt) {
        if constexpr (SOLO) return false;
        return masked ? live_bit(live, 1, ufirst, kt) : (kt >= first1 && kt <= last1);
      };
      int slot = 0, phase = 0;  // next ring slot to consume and its phase parity
      bool ok = mbar_wait(bar(C::B_Q), 0, ab);
      tc_fence_after();
      int cur = next_union_tile<SOLO>(p, live, ufirst, ulast, -1);
      int npv0 = 0, npv1 = 0;
      if (ok && cur < p.T) {
        ok = mbar_wait(bar(C::B_FULL + slot), phase, ab);
        tc_fence_after();
        if (ok) {
          if (live0(cur)) {
            qk(t_s0, dq0, slot);
            mma_commit(bar(C::B_S + 0));
          }
          if (live1(cur)) {
            qk(t_s1, dq1, slot);
            mma_commit(bar(C::B_S + 1));
          }
          mma_commit(bar(C::B_EMPTY + slot));
        }
        if (++slot == C::NSLOT) { slot = 0; phase ^= 1; }
      }
      while (ok && cur < p.T) {
        const bool l0 = live0(cur);
        const bool l1 = live1(cur);
        const int vslot = slot, vphase = phase;
        if (++slot == C::NSLOT) { slot = 0; phase ^= 1; }
        const int nxt = next_union_tile<SOLO>(p, live, ufirst, ulast, cur);
        const bool has_next = nxt < p.T;
        const bool n0 = has_next && live0(nxt);
        const bool n1 = has_next && live1(nxt);
        const int kslot = slot, kphase = phase;
        if (has_next && ++slot == C::NSLOT) { slot = 0; phase ^= 1; }
        const uint64_t dv = dv0 + (uint64_t)(vslot * slot_step);
        if (!(ok = mbar_wait(bar(C::B_FULL + vslot), vphase, ab))) break;
        if (has_next && !(ok = mbar_wait(bar(C::B_FULL + kslot), kphase, ab))) break;
        tc_fence_after();
        if (l0) {
          if (!(ok = mbar_wait(bar(C::B_P + 0), npv0 & 1, ab))) break;
          tc_fence_after();
          mma_ts_mn_k128(t_o0, t_s0, dv, id_pv, npv0 > 0);
          ++npv0;
        }
        if (n0) {
          qk(t_s0, dq0, kslot);
          mma_commit(bar(C::B_S + 0));
        }
        if (l1) {
          if (!(ok = mbar_wait(bar(C::B_P + 1), npv1 & 1, ab))) break;
          tc_fence_after();
          mma_ts_mn_k128(t_o1, t_s1, dv, id_pv, npv1 > 0);
          ++npv1;
        }
        mma_commit(bar(C::B_EMPTY + vslot));
        if (has_next) {
          if (n1) {
            qk(t_s1, dq1, kslot);
            mma_commit(bar(C::B_S + 1));
          }
          mma_commit(bar(C::B_EMPTY + kslot));
        }
        cur = nxt;
      }
      mma_commit(bar(C::B_O + 0));
      mma_commit(bar(C::B_O + 1));
      // Drain all issued tensor-core work before TMEM can be released.
      mma_commit(bar(C::B_DRAIN));
      const uint64_t t0 = globaltimer();
      while (!mbar_try_wait(bar(C::B_DRAIN), 0) && globaltimer() - t0 < kWaitLimitNs) {
      }
    }
  } else if (warp >= C::WARP_SM) {
    // ------------------------------------------------------------ softmax
    const int i = (warp - C::WARP_SM) >> 2;  // query tile of this warpgroup
    const int qt = i == 0 ? qt0 : qt1;
    if (qt >= 0) {
      const int r = ((warp & 3) << 5) + lane;  // row within the tile = TMEM lane
      const int row = qt * 128 + r;
      const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
      const uint32_t col_s = i == 0 ? C::COL_S0 : C::COL_S1;
      const uint32_t col_o = i == 0 ? C::COL_O0 : C::COL_O1;
      float m_ref = -INFINITY, l = 0.f;
      int n = 0;
      bool ok = true;
      const int myfirst = i == 0 ? first0 : first1, mylast = i == 0 ? last0 : last1;
      const bool bmask = p.block_mask != nullptr;
      for (int kt = next_union_tile<SOLO>(p, live, ufirst, ulast, -1); kt < p.T;
           kt = next_union_tile<SOLO>(p, live, ufirst, ulast, kt)) {
        if (bmask ? !live_bit(live, i, ufirst, kt) : (kt < myfirst || kt > mylast)) continue;
        if (!(ok = mbar_wait(bar(C::B_S + i), n & 1, ab))) break;
        tc_fence_after();
        // SEPP: S read -> the issuer may compute the next S into these
        // columns; P and O are written only once the previous P . V (which
        // read P and added into O) has completed
        auto after_load = [&]() {
          if constexpr (SEPP) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(C::B_SFREE));
          }
        };
        auto before_store = [&]() {
          if constexpr (SEPP) {
            if (n > 0 && ok) ok = mbar_wait(bar(C::B_PFREE), (n - 1) & 1, ab);
            tc_fence_after();
          }
        };
        softmax_tile<D, DROP>(p, bh, row, kt, klim, lane_base, col_s, col_o,
                              SEPP ? C::COL_P : col_s, n > 0, m_ref, l, after_load,
                              before_store);
        if (!ok) break;
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0 && !(LOSE && n == 0 && warp == C::WARP_SM)) mbar_arrive(bar(C::B_P + i));
        ++n;
      }
      // ---- epilogue: O = u / l -> bf16 -> shared (swizzled) -> TMA store;
      // in the packed layout a tile that ends past its sequence is written
      // row by row instead (a whole-tile store would overwrite the next
      // sequence's first rows).
      if (ok) ok = mbar_wait(bar(C::B_O + i), 0, ab);
      tc_fence_after();
      uint8_t* stage = smem + C::OFF_Q + i * C::TILE;
      // O = u / l, times 1 / (1 - p) for the kept elements under dropout
      const float inv = l > 0.f ? (DROP ? p.drop_scale : 1.f) / l : 0.f;
      const bool direct = PACKED && (qt + 1) * 128 > p.N;
      if (ok) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(lane_base + col_o + 32 * c, o);
          uint32_t pk[16];
          // a row without an allowed key never had O written: 0, not stale * 0
#pragma unroll
          for (int j = 0; j < 16; ++j)
            pk[j] = l > 0.f ? pack_bf16(__uint_as_float(o[2 * j]) * inv,
                                        __uint_as_float(o[2 * j + 1]) * inv)
                            : 0u;
          // 32 columns = four 16-byte chunks, chunk index cc = 4c + q
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int cc = 4 * c + q;
            const uint4 w = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
            if (direct) {
              if (row < p.N)
                reinterpret_cast<uint4*>(o_rows + ((size_t)(start + row) * p.H + head) * D)[cc] = w;
            } else {
              uint8_t* dst = stage + (cc >> 3) * C::HALF + r * 128 + (((cc & 7) ^ (r & 7)) << 4);
              *reinterpret_cast<uint4*>(dst) = w;
            }
          }
        }
        if (row < p.N) {
          const size_t li = PACKED ? (size_t)head * p.total + start + row : (size_t)bh * p.N + row;
          lse[li] = l > 0.f ? (m_ref + __log2f(l)) * kLn2 : -INFINITY;
        }
      }
      fence_proxy_async_smem();
      named_barrier(1 + i, 128);
      if (ok && r == 0 && !direct) {
        for (int h = 0; h < D / 64; ++h)
          tma_store_3d(&tm_o, smem_u32(stage) + h * C::HALF, h * 64, cy(qt * 128), cz(qt * 128));
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

// Heads per CTA group: K and V of a group within about 64 MB (half of L2).
static int heads_per_group(long long heads, long long bytes_per_head) {
  long long g = (64ll << 20) / (bytes_per_head > 0 ? bytes_per_head : 1);
  if (g < 1) g = 1;
  if (g > heads) g = heads;
  return (int)g;
}

template <int D, bool PACKED, bool DROP, bool SOLO, bool LOSE = false>
static cudaError_t launch_fwd_tc_t(const Problem& pin, const void* q, const void* k,
                                   const void* v, void* o, float* lse, cudaStream_t st) {
  using C = FwdTc<D, SOLO>;
  Problem p = pin;
  p.hgroup = heads_per_group((long long)p.B * p.H, (long long)p.N * D * 4);
  const long long bh = (long long)p.B * p.H;
  CUtensorMap tq, tk, tv, to;
  bool maps;
  if constexpr (PACKED)
    maps = make_bf16_map_packed(&tq, q, D, p.H, p.total, 128) &&
           make_bf16_map_packed(&tk, k, D, p.H, p.total, 128) &&
           make_bf16_map_packed(&tv, v, D, p.H, p.total, 128) &&
           make_bf16_map_packed(&to, o, D, p.H, p.total, 128);
  else
    maps = make_bf16_map_3d(&tq, q, D, p.N, bh, 128) && make_bf16_map_3d(&tk, k, D, p.N, bh, 128) &&
           make_bf16_map_3d(&tv, v, D, p.N, bh, 128) && make_bf16_map_3d(&to, o, D, p.N, bh, 128);
  if (!maps) return cudaErrorInvalidValue;
  auto kern = fwd_tc_kernel<D, PACKED, DROP, SOLO, LOSE>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
  if (e != cudaSuccess) return e;
  dim3 grid((unsigned)(bh * (SOLO ? p.T : (p.T + 1) / 2)));
  kern<<<grid, C::THREADS, C::SMEM, st>>>(tq, tk, tv, to, p, lse,
                                          static_cast<__nv_bfloat16*>(o));
  return cudaGetLastError();
}

// One query tile per CTA, two CTAs per SM, where it measured faster than
// the tile pair (same bits out):
//  - d = 64, padded, no dropout: always (1.01-1.10x on causal and full masks
//    of N = 1024-8192, 1.2x on a band-plus-global block mask), since a
//    pair's fixed costs weigh most against its short MMAs;
//  - d = 64 with dropout or packed sequences: up to 2048 rows (1.12x with
//    dropout at N = 1024, 1.04x for 16 sequences of 512-2048), not beyond
//    (0.95x with dropout at N = 8192, 0.93x for sequences up to 8192);
//  - d = 128 (padded, no dropout): only under a sliding window narrower than
//    2048 keys on each side (1.07x at a 1024-key causal window); other
//    d = 128 work runs faster as pairs, which share each K/V tile between
//    two query tiles (0.87x-1.0x as one-tile CTAs).
static bool use_solo(const Problem& p) {
  if (p.d == 64) return (p.drop_p8 == 0 && p.cu_seqlens == nullptr) || p.N <= 2048;
  if (p.cu_seqlens != nullptr || p.drop_p8 != 0) return false;
  const bool narrow_left = p.wl >= 0 && p.wl < 2048;
  const bool narrow_right = p.causal || (p.wr >= 0 && p.wr < 2048);
  return narrow_left && narrow_right;
}

template <bool PACKED, bool DROP>
static cudaError_t launch_fwd_tc_d(const Problem& p, const void* q, const void* k, const void* v,
                                   void* o, float* lse, cudaStream_t st) {
  if (p.d == 64) {
    // padded without dropout use_solo() always holds at d = 64: no pair
    // instantiation is built for it
    if constexpr (!PACKED && !DROP)
      return launch_fwd_tc_t<64, false, false, true>(p, q, k, v, o, lse, st);
    else
      return use_solo(p) ? launch_fwd_tc_t<64, PACKED, DROP, true>(p, q, k, v, o, lse, st)
                         : launch_fwd_tc_t<64, PACKED, DROP, false>(p, q, k, v, o, lse, st);
  }
  if constexpr (!PACKED && !DROP)
    if (use_solo(p)) return launch_fwd_tc_t<128, false, false, true>(p, q, k, v, o, lse, st);
  return launch_fwd_tc_t<128, PACKED, DROP, false>(p, q, k, v, o, lse, st);
}

cudaError_t launch_fwd_tc_lost_signal(const Problem& p, const void* q, const void* k,
                                      const void* v, void* o, float* lse, cudaStream_t st) {
  if ((p.d != 128 && p.d != 64) || p.cu_seqlens != nullptr || p.drop_p8 != 0)
    return cudaErrorInvalidValue;
  // d = 64: the one-tile kernel (P apart, two-stage ring)
  if (p.d == 64) return launch_fwd_tc_t<64, false, false, true, true>(p, q, k, v, o, lse, st);
  return launch_fwd_tc_t<128, false, false, false, true>(p, q, k, v, o, lse, st);
}

cudaError_t launch_fwd_tc(const Problem& p, const void* q, const void* k, const void* v, void* o,
                          float* lse, cudaStream_t st) {
  const bool packed = p.cu_seqlens != nullptr, drop = p.drop_p8 != 0;
  if (packed)
    return drop ? launch_fwd_tc_d<true, true>(p, q, k, v, o, lse, st)
                : launch_fwd_tc_d<true, false>(p, q, k, v, o, lse, st);
  return drop ? launch_fwd_tc_d<false, true>(p, q, k, v, o, lse, st)
              : launch_fwd_tc_d<false, false>(p, q, k, v, o, lse, st);
}

}  // namespace fa
