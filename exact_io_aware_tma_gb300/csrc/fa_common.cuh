// Shared device helpers of the attention kernels: the allowed-pair predicate,
// the live-tile walk, bf16 packing and the exp2 used by every softmax.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

constexpr int kTile = 128;  // block-mask tile side (queries and keys)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Arguments every kernel shares.  Pointers are device pointers.
struct Problem {
  int B, H, N, d;
  int T;                  // ceil(N / 128)
  float scale;            // multiplies Q K^T
  float scale_log2;       // scale * log2(e): scores are kept in log2 units
  int causal;
  int wl, wr;             // sliding window: j >= i - wl (wl >= 0), j <= i + wr
                          // (wr >= 0); -1 = unbounded on that side
  const uint8_t* block_mask;  // [T, T] or nullptr
  const int32_t* kv_len;      // [B] or nullptr
  int* status;                // device error word (bounded waits record here)
  // Packed variable-length layout (kernels instantiated for it only): the B
  // sequences lie back to back in [total, H, d]; sequence b is tokens
  // cu_seqlens[b] .. cu_seqlens[b+1]-1, and N above is the longest length
  // (it sizes the grid; each CTA takes its own sequence's length as N).
  const int32_t* cu_seqlens;
  int total;
  // CTA order: heads go in groups of hgroup (sized by the host so that a
  // group's working set fits in about half of L2); within a group the CTAs
  // walk the tiles heaviest first, cycling over the group's heads.
  int hgroup;
  // Dropout on P (kernels instantiated for it only): element (i, j) of head
  // bh is kept iff byte j % 16 of Philox4x32-10(counter (j/16, i, bh,
  // drop_offset), key (seed_lo, seed_hi)) is >= drop_p8; kept probabilities
  // are scaled by drop_scale = 1 / (1 - drop_p8 / 256).
  uint32_t drop_p8;
  uint32_t seed_lo, seed_hi, drop_offset;
  float drop_scale;
};

// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
// easy as 1, 2, 3", SC'11), written from its published definition: ten
// rounds, each multiplying counter words 0 and 2 by two odd constants and
// crossing the products' high halves with words 1, 3 and the key, the key
// advancing by two Weyl constants between rounds.
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const uint32_t lo0 = c.x * 0xD2511F53u, hi0 = __umulhi(c.x, 0xD2511F53u);
    const uint32_t lo1 = c.z * 0xCD9E8D57u, hi1 = __umulhi(c.z, 0xCD9E8D57u);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c;
}

// The 16 keep bytes of keys 16*jb .. 16*jb+15 of query row i: byte t of the
// result (word t/4, bits 8*(t%4)) is the uniform byte of key 16*jb + t.
__device__ __forceinline__ uint4 dropout_bytes(const Problem& p, long long bh, int i, int jb) {
  return philox4x32_10(make_uint4((uint32_t)jb, (uint32_t)i, (uint32_t)bh, p.drop_offset),
                       p.seed_lo, p.seed_hi);
}

// Keep bits of four uniform bytes (bit t = byte t >= p8).
__device__ __forceinline__ uint32_t keep4(uint32_t w, uint32_t p8) {
  return ((w & 0xffu) >= p8 ? 1u : 0u) | (((w >> 8) & 0xffu) >= p8 ? 2u : 0u) |
         (((w >> 16) & 0xffu) >= p8 ? 4u : 0u) | ((w >> 24) >= p8 ? 8u : 0u);
}

// Backward work split of key tiles with many live query tiles (block
// masks): up to kSplitMax parts per key tile, kSplitSlots part slots per
// head, planned for at most kPlanMaxTiles key tiles.
constexpr int kSplitMax = 4;
constexpr int kSplitSlots = 32;
constexpr int kPlanMaxTiles = 1024;
// The plan and the slots a split backward reads and writes (device
// pointers into the caller's workspace).
struct BwdSplit {
  const int4* items;  // [T * kSplitMax] work items, heaviest first
  const int* nitems;  // [0]: number of items; [1]: number of split key
                      // tiles; [2 + 3j ..]: split key tile j (tile, first
                      // slot, parts)
  float* slots;       // [B*H][kSplitSlots][2][128][d] fp32 partial dK, dV rows
};

// Head and tile rank of CTA `cta` of a grid of B*H x ntiles CTAs in the
// grouped order above (the last group may hold fewer heads).
__device__ __forceinline__ void grouped_cta(const Problem& p, long long cta, int ntiles,
                                            long long& bh, int& rank) {
  const long long heads = (long long)p.B * p.H;
  const long long per_group = (long long)p.hgroup * ntiles;
  const long long g = cta / per_group;
  const long long j = cta - g * per_group;
  const long long first = g * p.hgroup;
  const int gsize = (int)min((long long)p.hgroup, heads - first);
  rank = (int)(j / gsize);
  bh = first + j % gsize;
}

// Token span of sequence b in the packed layout.  Offsets that are out of
// order, out of range or longer than N are clamped (the call then records
// FA_ERR_INVALID_ARG in the status word).
__device__ __forceinline__ void seq_span(const Problem& p, int b, int& start, int& len) {
  int s = __ldg(p.cu_seqlens + b), e = __ldg(p.cu_seqlens + b + 1);
  const bool bad = s < 0 || e < s || e > p.total || e - s > p.N;
  s = min(max(s, 0), p.total);
  e = min(max(e, s), p.total);
  start = s;
  len = min(e - s, p.N);
  if (bad && threadIdx.x == 0 && p.status != nullptr) atomicExch(p.status, 1);
}

// Valid-key bound of batch element b: min(N, max(0, kv_len[b])).
__device__ __forceinline__ int key_limit(const Problem& p, int b) {
  if (p.kv_len == nullptr) return p.N;
  int l = __ldg(p.kv_len + b);
  return l < 0 ? 0 : (l > p.N ? p.N : l);
}

// The keys query row i may attend form one interval [row_key_lo, row_key_hi]
// (empty when lo > hi), and the queries key column j (< klim) serves form
// [col_q_lo, col_q_hi]; all four ends are nondecreasing in the row/column.
__device__ __forceinline__ int row_key_lo(const Problem& p, int i) {
  return p.wl >= 0 ? max(0, i - p.wl) : 0;
}
__device__ __forceinline__ int row_key_hi(const Problem& p, int i, int klim) {
  int h = klim - 1;
  if (p.causal) h = min(h, i);
  if (p.wr >= 0) h = min(h, i + p.wr);
  return h;
}
__device__ __forceinline__ int col_q_lo(const Problem& p, int j) {
  int l = p.causal ? j : 0;
  if (p.wr >= 0) l = max(l, j - p.wr);
  return l;
}
__device__ __forceinline__ int col_q_hi(const Problem& p, int j) {
  return p.wl >= 0 ? min(p.N - 1, j + p.wl) : p.N - 1;
}

// A (query tile, key tile) pair is live when some allowed (i, j) lies in it:
// some row i of the tile has keys in the tile's key range.  By the
// monotonicity above that is: the rows i with row_key_lo(i) <= jmax (i.e.
// i <= jmax + wl) and row_key_hi(i) >= jmin (i.e. i >= col_q_lo(jmin), given
// jmin < klim) include one of the tile.  With equal query and key lengths
// the causal rule alone keeps kt <= qt.
__device__ __forceinline__ bool tile_live(const Problem& p, int qt, int kt, int klim) {
  const int jmin = kt * kTile;
  if (jmin >= klim) return false;
  if (p.causal && kt > qt) return false;
  if (p.wl >= 0 || p.wr >= 0) {
    const int imin = qt * kTile, imax = min(p.N, imin + kTile) - 1;
    const int jmax = min(klim, jmin + kTile) - 1;
    const int ilo = max(imin, col_q_lo(p, jmin));
    const int ihi = p.wl >= 0 ? min(imax, jmax + p.wl) : imax;
    if (ilo > ihi) return false;
  }
  if (p.block_mask != nullptr && __ldg(p.block_mask + (size_t)qt * p.T + kt) == 0)
    return false;
  return true;
}

// A live tile needs element masking when some in-range (i, j) of it is not
// allowed: its last row's interval starts after the first key, or its first
// row's interval ends before the last in-range key (the causal diagonal tile,
// a tile crossing the key limit, the edges of a window).
__device__ __forceinline__ bool tile_partial(const Problem& p, int qt, int kt, int klim) {
  const int imin = qt * kTile, imax = min(p.N, imin + kTile) - 1;
  const int jmin = kt * kTile, jn = min(p.N, jmin + kTile) - 1;
  if (row_key_lo(p, imax) > jmin) return true;
  return row_key_hi(p, imin, klim) < jn;
}

// Without a block mask the live key tiles of query tile qt are exactly
// [first, last] (first > last: none): rows with no key are only ever the
// last rows of a tile, so the union of the rows' intervals runs from the
// first row's start to the last row's end.
__device__ __forceinline__ void qtile_key_tiles(const Problem& p, int qt, int klim, int& first,
                                                int& last) {
  const int imin = qt * kTile, imax = min(p.N, imin + kTile) - 1;
  const int lo = row_key_lo(p, imin), hi = row_key_hi(p, imax, klim);
  if (lo > hi) {
    first = 0;
    last = -1;
  } else {
    first = lo / kTile;
    last = hi / kTile;
  }
}

// Likewise the live query tiles of key tile kt without a block mask.
__device__ __forceinline__ void ktile_query_tiles(const Problem& p, int kt, int klim, int& first,
                                                  int& last) {
  const int jmin = kt * kTile;
  if (jmin >= klim) {
    first = 0;
    last = -1;
    return;
  }
  const int jmax = min(klim, jmin + kTile) - 1;
  first = col_q_lo(p, jmin) / kTile;
  last = col_q_hi(p, jmax) / kTile;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Programmatic dependent launch.  A kernel launched with the programmatic
// stream-serialisation attribute may start while the kernel before it in the
// stream is still running; griddep_wait() returns once that kernel has
// completed and its writes are visible (at once for a kernel launched the
// ordinary way).  griddep_release() lets the next kernel so launched be
// scheduled.  Every kernel here releases only after its own wait, so a kernel
// that starts early still finds all work before its predecessor complete:
// only what the predecessor itself writes needs the wait.
__device__ __forceinline__ void griddep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_release() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace fa
