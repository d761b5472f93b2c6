// Sparse causal attention engine for sm_103a (A-shape, Vertical-Slash and
// Block-Sparse heads in one kernel).
//
// What it computes (MInference page, eq.(1)-(2) restricted to N_h(i), with
// the online-softmax merge of eq.(7)-(8)): for every query row i of a work
// item, o_i = Σ_{j in N(i)} e^{s_ij} v_j / Σ_{j in N(i)} e^{s_ij}.
//
// One CTA processes one item: two 128-row query tiles ("sub-items" X = 0, 1,
// each of two 64-row halves) that read the same KV head, against one stream of
// 128-key tiles holding every key either sub-item needs.  Sharing the K/V
// stream doubles the tensor work per loaded byte.
//   warp 8     planner: merges the sub-items' key sets into tiles of two
//              64-key segments (or, for Vertical-Slash, eight 16-key
//              segments holding attended keys) and writes
//              each tile's descriptor (segments, per-half validity masks,
//              per-sub-item activity and A-shape row rules) into a ring; a
//              terminating descriptor ends the item;
//   warp 10    loader: TMA-loads both Q tiles once, then K(j) and V(j) of
//              every tile into a four-slot ring (K in slots 0/2, V in 1/3);
//   warps 9/11 MMA issuers (one thread each, one per sub-item X): per tile,
//              O_X += P_X V of the previous tile, then S_X = Q_X K^T.  While
//              one sub-item's softmax runs, the tensor core works for the
//              other, and neither issuer waits for the other's P;
//   warps 0-7  softmax: warps 4X..4X+3 own sub-item X; thread r is query row r
//              (TMEM lane r) with all 128 keys of a tile.  Per-row masks
//              (causal, A-shape sink and window) are applied before the max; O_X
//              is rescaled in TMEM only when the max grows by more than 2^8; P
//              (bf16 pairs) overwrites the first 64 columns of S_X.
// In Vertical-Slash tiles, the keys that a whole 64-row half does not attend
// are masked by the tensor core: such a tile gets one more K-step in
// S_X = Q_X K^T, a one-hot 16-wide row selector per half (Q side, fixed)
// against a per-key column of 0 or -BIG per half (K side, written by the
// loader), so masked scores arrive as -BIG (exactly 0 after the exponential)
// and attended scores unchanged.  (Range tiles mask whole 64-key words in the
// softmax, where the extra K-step costs more than it saves.)
// Every (i, j) pair enters the softmax at most once: a key lies in one tile
// of the item, and masks drop what lies outside N(i) (MInference page §3.2
// and §5.1 "boundary masks": set to -inf before the max).
// Every launch runs a kernel compiled for one pattern (the others' planner,
// loader and mask code left out); a layer with several patterns launches each
// pattern in its own kernel on forked streams (launch_attention).  The kernel
// that holds all three is the fallback when the side streams cannot be made.
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>
#include <vector>

#include "internal.h"
#include "ptx.cuh"

namespace msa {

namespace {

constexpr int kSoftWarps = 8;
constexpr int kPlannerWarp = 8;
constexpr int kMmaWarp0 = 9;    // MMA issuer of sub-item 0
constexpr int kLoaderWarp = 10;
constexpr int kMmaWarp1 = 11;   // MMA issuer of sub-item 1
constexpr int kThreads = 32 * (kSoftWarps + 4);
constexpr int kSlots = 4;  // K(j) in slot 2j mod 4, V(j) in slot 2j+1 mod 4
constexpr int kDescSlots = 8;
constexpr int kDescReaders = kSoftWarps + 3;  // softmax warps, two MMA warps, loader warp
constexpr int kMaxStagedBlocks = 512;         // Block-Sparse list entries staged per half
constexpr uint32_t kTmemCols = 512;
// TMEM columns: S of sub-item X at 128 X (P over its first 64 columns), O of
// sub-item X at 256 + 128 X
constexpr uint32_t kColS = 0, kColO = 256;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr uint32_t kIdleNs = 256;          // poll interval of the planner's and loader's waits
// P columns per TMEM store: small stores keep few packed values live next to
// the 128 scores, which is what keeps the softmax free of register spills
constexpr int kPChunk = 4;
constexpr bool kTurnLock = true;            // sub-items take turns on each SMSP's softmax section
constexpr uint16_t kBf16NegBig = 0xFF7Fu;   // -3.3895e38, the most negative finite bf16
constexpr float kMaskedBelow = -1e30f;      // a raw score below this is a masked one


// kTileRange: two 64-key segments (seg[0], seg[1]); kTileRange16: eight 16-key
// segments (seg[0..7], non-decreasing; seg_hi = the last attended one).
enum TileKind : int32_t { kTileRange = 0, kTileRange16 = 1, kTileEnd = 2 };

struct TileDesc {
  int32_t seg[8];       // first key of each segment
  int32_t seg_hi;
  int32_t kind;         // TileKind (kTileEnd: no more tiles in this item)
  uint8_t rule[2][2];   // A-shape row rule per [sub-item][segment]: bit0 j < sink, bit1 j > i - window
  uint8_t active[2];    // sub-item X attends some key of this tile
  uint8_t bias;         // some existing half leaves a key of this tile out: the masking K-step runs
  uint8_t pad;
  uint32_t mask[4][4];  // per half 2X+h: bit k = key k of the tile may be attended
};

// A half of an active sub-item that exists and leaves out some key of the
// tile: that tile's scores need the masking K-step.
__device__ __forceinline__ uint8_t tile_needs_bias(const TileDesc& d, const int* ex) {
  uint32_t all = ~0u;
  for (int hh = 0; hh < 4; ++hh)
    if (ex[hh] && d.active[hh >> 1])
      all &= d.mask[hh][0] & d.mask[hh][1] & d.mask[hh][2] & d.mask[hh][3];
  return all != ~0u ? 1 : 0;
}

enum {
  kBarQ = 0,
  kBarFull = 1,
  kBarEmpty = kBarFull + kSlots,
  kBarSFull = kBarEmpty + kSlots,  // per sub-item: S of its latest tile is in TMEM
  kBarPFull = kBarSFull + 2,       // per sub-item: P of its latest tile is in TMEM
  kBarODone = kBarPFull + 2,       // per sub-item: every MMA of its issuer has completed
  kBarDFull = kBarODone + 2,
  kBarDEmpty = kBarDFull + kDescSlots,
  kNumBars = kBarDEmpty + kDescSlots
};

template <int D>
struct Layout {
  static constexpr int kTile = 128 * D * 2;  // 128 rows of d_h bf16
  static constexpr int kQ = 0;               // the two Q tiles
  static constexpr int kRing = kQ + 2 * kTile;
  static constexpr int kDesc = kRing + kSlots * kTile;
  static constexpr int kBlk = kDesc + kDescSlots * (int)sizeof(TileDesc);  // Block-Sparse lists
  // masking K-step operands (128 rows x 16 bf16, unswizzled core matrices, 4 KB
  // each): the two sub-items' row selectors, then two key-mask slots
  static constexpr int kAug = kBlk + 4 * kMaxStagedBlocks * 4;
  static constexpr int kBars = kAug + 4 * 4096;
  static constexpr int kMisc = kBars + kNumBars * 8;
  static constexpr int kTotal = kMisc + 64;  // misc words: [0] TMEM base, [2] abort, [8..11] softmax turns
  // > 113 KB keeps one CTA per SM, so the 512-column TMEM allocation never waits.
  static constexpr int kAlloc = (kTotal + 1024) > 120 * 1024 ? (kTotal + 1024) : 120 * 1024;
  static_assert(kAlloc <= 227 * 1024, "shared memory budget");
};

__device__ __forceinline__ void set_error(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Two fp32 values in one 64-bit register pair, for the packed f32x2 instructions.
__device__ __forceinline__ uint64_t pk2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ void up2(uint64_t v, float& a, float& b) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t low_mask64(int c) {  // bits [0, c), c clamped to [0, 64]
  c = c < 0 ? 0 : (c > 64 ? 64 : c);
  return c >= 64 ? ~0ull : ((1ull << c) - 1ull);
}

__device__ __forceinline__ uint32_t low_mask32(int c) {
  c = c < 0 ? 0 : (c > 32 ? 32 : c);
  return c >= 32 ? 0xFFFFFFFFu : ((1u << c) - 1u);
}

__device__ __forceinline__ uint32_t keys_below(int base, int limit) {  // bits k with base + k < limit
  return low_mask32(limit - base);
}

// 32 bits of an nw-word map starting at bit p >= 0 (bits past the end read 0).
__device__ __forceinline__ uint32_t bits_window32(const uint32_t* bits, int nw, int p) {
  const int w = p >> 5, sh = p & 31;
  const uint32_t lo = w < nw ? __ldg(bits + w) : 0u;
  const uint32_t hi = (w + 1) < nw ? __ldg(bits + w + 1) : 0u;
  return __funnelshift_r(lo, hi, sh);
}

// ------------------------------------------------------------------ item geometry
// The four halves of an item are hh = 2X + h (sub-item X, half h).
struct Geo {
  int row0[4];    // first query row of each half
  int ex[4];      // half has at least one row < n
  int e[4];       // last row of each half's query block (clipped to n-1)
  int sub_ex[2];  // sub-item has a half with rows
  int hi_key[2];  // last key sub-item X may attend
};

__device__ __forceinline__ Geo make_geo(const Unit& U, int t, int n, int nqt) {
  Geo G;
  for (int X = 0; X < 2; ++X) {
    const SubUnit& S = U.sub[X];
    const int tq = t * S.stride + S.offset;
    const bool live = (X == 0 || U.has1) && tq < nqt;
    G.sub_ex[X] = 0;
    G.hi_key[X] = -1;
    for (int h = 0; h < 2; ++h) {
      const int hh = 2 * X + h;
      G.row0[hh] = 128 * tq + S.row_off[h];
      G.ex[hh] = live && G.row0[hh] < n;
      const int e = G.row0[hh] + 63;
      G.e[hh] = e < n - 1 ? e : n - 1;
      if (G.ex[hh]) {
        G.sub_ex[X] = 1;
        G.hi_key[X] = max(G.hi_key[X], G.e[hh]);
      }
    }
  }
  return G;
}

// ------------------------------------------------------------------ A-shape segments
// MInference page eq.(3): rows i attend j < g or i-w < j <= i.  Per sub-item
// X, the key ranges [0, g) (slot 2X) and [a0-w+1, last row] (slot 2X+1), or
// one range [0, last row] when they touch, become intervals of 64-key
// segments with a row rule; the union over both sub-items is walked in
// ascending order.  Lane 0 runs it; unused slots have lo > hi.
struct AshapeSeg {
  int lo[4], hi[4], rule[4];
  int cur;
  __device__ void init(const Unit& U, const Geo& G, int n) {
    cur = 0;
#pragma unroll
    for (int X = 0; X < 2; ++X) {
      lo[2 * X] = lo[2 * X + 1] = 1;
      hi[2 * X] = hi[2 * X + 1] = 0;
      rule[2 * X] = 1;
      rule[2 * X + 1] = 2;
      if (!G.sub_ex[X]) continue;
      const int g = U.sub[X].sink, w = U.sub[X].window;
      const int a0 = min(G.row0[2 * X], G.row0[2 * X + 1]);
      const int hk = G.hi_key[X];
      const int sw = max(0, a0 - w + 1);
      if (sw <= g) {
        lo[2 * X] = 0; hi[2 * X] = hk >> 6; rule[2 * X] = 3;
      } else {
        if (g > 0) { lo[2 * X] = 0; hi[2 * X] = (min(g, n) - 1) >> 6; }
        lo[2 * X + 1] = sw >> 6; hi[2 * X + 1] = hk >> 6;
      }
    }
  }
  // Next segment of the union with each sub-item's rule (0: not attended).
  __device__ bool next(int& seg, int (&r)[2]) {
    int best = 0x7FFFFFFF;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (hi[q] >= cur && lo[q] <= hi[q]) best = min(best, max(lo[q], cur));
    if (best == 0x7FFFFFFF) return false;
    seg = best;
    r[0] = r[1] = 0;
#pragma unroll
    for (int q = 0; q < 4; ++q)
      if (lo[q] <= best && best <= hi[q]) r[q >> 1] |= rule[q];
    cur = best + 1;
    return true;
  }
};

// ------------------------------------------------------------------ Block-Sparse segments
// MInference page eq.(6): half hh (query block u_hh) attends the key blocks
// J_{u_hh}.  The four halves' ascending lists are staged in shared memory
// (lists longer than the staging buffer are read from global memory) and
// merged; each union block is one segment with its membership bits.  Lane 0
// runs the merge.
struct BlockSeg {
  const int32_t* L[4];
  int cnt[4], u[4], p[4];
  int last;
  int pend[4], pendb[4];  // per class (1: sub-item 0 only, 2: sub-item 1 only, 3: both): a block waiting for a partner
  __device__ void init(const Unit& U, const Geo& G, const AttnArgs& a, const SeqInfo& S, int lane, int* sblk) {
    bool fits = true;
    const int nbs = n_blocks(S.n);
    const int64_t base = (int64_t)a.bs_nslots * S.nb0;
    for (int hh = 0; hh < 4; ++hh) {
      const int X = hh >> 1, h = hh & 1;
      u[hh] = G.row0[hh] / 64;
      cnt[hh] = 0;
      L[hh] = nullptr;
      p[hh] = 0;
      if (G.ex[hh]) {
        const int64_t off = base + (int64_t)U.sub[X].slot[h] * nbs + u[hh];
        L[hh] = a.bs_idx + off * a.bs_topk;
        const int c = __ldg(a.bs_cnt + off);
        cnt[hh] = c < 0 ? 0 : (c > a.bs_topk ? a.bs_topk : c);
        fits = fits && cnt[hh] <= kMaxStagedBlocks;
      }
    }
    if (fits) {
      for (int hh = 0; hh < 4; ++hh) {
        for (int x = lane; x < cnt[hh]; x += 32) sblk[hh * kMaxStagedBlocks + x] = __ldg(L[hh] + x);
        L[hh] = sblk + hh * kMaxStagedBlocks;
      }
      __syncwarp();
    }
    last = -1;
    for (int c = 0; c < 4; ++c) pend[c] = pendb[c] = -1;
  }
  // Next union block and the halves that hold it; bits = -1 flags a list
  // that is not strictly ascending.
  __device__ bool next(int& v, int& bits) {
    int best = 0x7FFFFFFF;
    int val[4];
    for (int hh = 0; hh < 4; ++hh) {
      val[hh] = p[hh] < cnt[hh] ? L[hh][p[hh]] : 0x7FFFFFFF;
      best = min(best, val[hh]);
    }
    if (best == 0x7FFFFFFF) return false;
    v = best;
    bits = 0;
    for (int hh = 0; hh < 4; ++hh)
      if (val[hh] == best) { bits |= 1 << hh; ++p[hh]; }
    if (v <= last) bits = -1;
    else last = v;
    return true;
  }
};

// ------------------------------------------------------------------ Vertical-Slash segments
// Physical set of row i in query block [a, e] (MInference page §2.1 and §4.1):
// keys covered by some slash tile [a-δ, e-δ] (δ in D), plus the vertical
// columns C, restricted to j <= i.  For a full block, key j is covered iff bit
// n-1-a+j of the dilated coverage map is set, so a 32-key mask word is a
// 32-bit window of that map; a ragged last block (fewer than 64 rows) is
// dilated exactly from D.  Every 16-key segment holding a key that one of the
// item's four halves attends (slash-covered or a vertical) is loaded whole;
// eight such segments, ascending, make a tile.  Against 64-key segments this
// drops about an eighth of the Vertical-Slash tiles (isolated slash runs and
// verticals occupy a fraction of a 64-key block).
//
// The whole warp runs it: lane l evaluates key block grp + l of a group of 32
// (all loads of a group in flight at once); the segments are then placed in
// ascending order from a warp prefix sum.

// Bits [p, p+32) of an n-bit map held in nw words (zeros outside the map).
__device__ __forceinline__ uint32_t bits32_at(const uint32_t* bits, int nw, int p) {
  const int w = p >> 5, sh = p & 31;  // floor division for negative p
  const uint32_t lo = (w >= 0 && w < nw) ? __ldg(bits + w) : 0u;
  const uint32_t hi = (w + 1 >= 0 && w + 1 < nw) ? __ldg(bits + w + 1) : 0u;
  return __funnelshift_r(lo, hi, sh);
}

// Bit k set iff the n-bit map D has a bit in [A-k, A-k+L-1] (1 <= L <= 64):
// key base+k is covered by the slash tiles of the L-row block starting at
// row base+A.
__device__ __forceinline__ uint32_t exact_cover32(const uint32_t* dbits, int nw, int A, int L) {
  const int lo = A - 31;  // δ held in bit 0 of the window
  unsigned __int128 v = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) v |= (unsigned __int128)bits32_at(dbits, nw, lo + 32 * q) << (32 * q);
  // e bit p = OR of v bits [p, p+L-1]
  unsigned __int128 e = v;
  int span = 1;
  while (2 * span <= L) {
    e |= e >> span;
    span *= 2;
  }
  if (span < L) e |= e >> (L - span);
  return __brev((uint32_t)e);  // bit k = e bit 31-k
}

struct VSSeg {
  const uint32_t* cbits[2];
  const uint32_t* dbits[2];
  const uint32_t* cover[2];
  int cw, nw, NB, hi_key, two;
  int a[4], e[4], L[4], ex[4];
  int grp;           // first block of the current 32-block group
  uint32_t m[4][2];  // this lane's block: attend masks per half
  uint32_t qm;       // this lane's block: 16-key quarters with attended keys, not yet placed
  __device__ void init(const Unit& U, const Geo& G, const AttnArgs& A, const SeqInfo& S) {
    cw = n_cover_words(S.n);
    nw = n_words(S.n);
    const int64_t wbase = (int64_t)A.vs_nslots * S.word0, cbase = (int64_t)A.vs_nslots * S.cword0;
#pragma unroll
    for (int X = 0; X < 2; ++X) {
      const int slot = U.sub[X].slot[0];
      dbits[X] = A.vs_dbits + wbase + (int64_t)slot * nw;
      cbits[X] = A.vs_cbits + wbase + (int64_t)slot * nw;
      cover[X] = A.vs_cover + cbase + (int64_t)slot * cw;
    }
    two = U.has1 && U.sub[1].slot[0] != U.sub[0].slot[0];
    hi_key = max(G.hi_key[0], G.hi_key[1]);
    NB = hi_key < 0 ? 0 : hi_key / 64 + 1;
#pragma unroll
    for (int hh = 0; hh < 4; ++hh) {
      a[hh] = G.row0[hh];
      e[hh] = G.e[hh];
      ex[hh] = G.ex[hh];
      L[hh] = e[hh] - a[hh] + 1;
    }
    grp = -32;
    qm = 0u;
  }
  // Masks of the 32 blocks of the next group, one lane per 64-key block.
  __device__ void load_group(int lane, int n) {
    grp += 32;
    const int b = grp + lane;
    uint32_t un[2] = {0u, 0u};
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      const int base = 64 * b + 32 * w;
      const uint32_t kin = keys_below(base, hi_key + 1);
      const uint32_t c0 = (b < NB && base <= hi_key) ? __ldg(cbits[0] + (base >> 5)) & kin : 0u;
      const uint32_t c1 = two ? ((b < NB && base <= hi_key) ? __ldg(cbits[1] + (base >> 5)) & kin : 0u) : c0;
#pragma unroll
      for (int hh = 0; hh < 4; ++hh) {
        uint32_t s = 0u;
        if (b < NB && ex[hh] && base <= e[hh]) {
          s = L[hh] == 64 ? bits_window32(cover[hh >> 1], cw, n - 1 - a[hh] + base)
                          : exact_cover32(dbits[hh >> 1], nw, a[hh] - base, L[hh]);
          s = (s | (hh < 2 ? c0 : c1)) & keys_below(base, e[hh] + 1);
        }
        m[hh][w] = s;
        un[w] |= s;
      }
    }
    qm = ((un[0] & 0xFFFFu) ? 1u : 0u) | ((un[0] >> 16) ? 2u : 0u) | ((un[1] & 0xFFFFu) ? 4u : 0u) |
         ((un[1] >> 16) ? 8u : 0u);
  }
  // Produce the next tile into d: the next (up to) eight 16-key segments that
  // hold attended keys, ascending; false when the item has no more tiles.
  // Positions come from a warp prefix sum over the lanes' quarter counts, so
  // the lanes place their segments (and 16-bit mask pieces) in parallel.
  __device__ bool emit(int lane, int n, TileDesc& d) {
    uint16_t* m16 = reinterpret_cast<uint16_t*>(&d.mask[0][0]);  // [half][segment]
    if (lane < 16) d.mask[lane >> 2][lane & 3] = 0u;
    __syncwarp();
    int f = 0, hi = -1;
    uint32_t act = 0u;  // bit X: sub-item X attends a key of this tile (this lane's pieces)
    for (;;) {
      if (__ballot_sync(0xFFFFFFFFu, qm != 0u) == 0u) {
        if (grp + 32 >= NB) break;
        load_group(lane, n);
        continue;
      }
      const int c = __popc(qm);
      int incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      int pos = f + incl - c;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (!((qm >> q) & 1u)) continue;
        if (pos < 8) {
          const int key0 = 64 * (grp + lane) + 16 * q;
          d.seg[pos] = key0;
          hi = max(hi, key0);
#pragma unroll
          for (int hh = 0; hh < 4; ++hh) {
            const uint32_t bits = (m[hh][q >> 1] >> (16 * (q & 1))) & 0xFFFFu;
            if (bits) {
              m16[hh * 8 + pos] = (uint16_t)bits;
              act |= 1u << (hh >> 1);
            }
          }
          qm &= ~(1u << q);
        }
        ++pos;
      }
      f = min(8, f + __shfl_sync(0xFFFFFFFFu, incl, 31));
      if (f == 8) break;
    }
    if (f == 0) return false;
    hi = __reduce_max_sync(0xFFFFFFFFu, hi);
    act = __reduce_or_sync(0xFFFFFFFFu, act);
    __syncwarp();  // d.seg[0 .. f) and the mask pieces written
    if (lane == 0) {
      for (int x = f; x < 8; ++x) d.seg[x] = hi;  // reload a valid segment, masked (starts stay ascending)
      d.seg_hi = hi;
      d.kind = kTileRange16;
      d.active[0] = act & 1u;
      d.active[1] = (act >> 1) & 1u;
      d.rule[0][0] = d.rule[0][1] = d.rule[1][0] = d.rule[1][1] = 0;
      d.bias = tile_needs_bias(d, ex);
    }
    return true;
  }
};

// ------------------------------------------------------------------ kernel
// kPat: the unit patterns a launch holds (bit 1 << UnitPattern); a launch of
// one pattern compiles only that pattern's planner, loader and softmax paths.
constexpr int kPatA = 1 << kUnitAshape, kPatV = 1 << kUnitVS, kPatB = 1 << kUnitBlock;
constexpr int kPatAll = kPatA | kPatV | kPatB;

template <int D, bool kCount, int kPat>
__global__ void __launch_bounds__(kThreads, 1)
    sparse_attn_kernel(const __grid_constant__ AttnMaps M, const AttnArgs A,
                       const __grid_constant__ UnitTable UT, const __grid_constant__ SeqTable ST) {
  using Ly = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Ly::kBars);
  TileDesc* descs = reinterpret_cast<TileDesc*>(sm + Ly::kDesc);
  int* sblk = reinterpret_cast<int*>(sm + Ly::kBlk);
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(sm + Ly::kMisc);  // [0] tmem, [2] abort

  constexpr bool kHasA = (kPat & kPatA) != 0, kHasV = (kPat & kPatV) != 0, kHasB = (kPat & kPatB) != 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // sequence of this item (entries ordered by their first item), then band, t and unit within it
  const SeqInfo& SI = ST.s[seq_search(ST.count, [&](int x) { return ST.s[x].item0; }, (int64_t)blockIdx.x)];
  int rem = (int)blockIdx.x - SI.item0, band = 0;
  while (band + 1 < A.n_bands && rem >= (UT.band[band + 1] - UT.band[band]) * SI.T) {
    rem -= (UT.band[band + 1] - UT.band[band]) * SI.T;
    ++band;
  }
  const int band_units = UT.band[band + 1] - UT.band[band];
  const int t = SI.T - 1 - rem / band_units;
  const Unit& U = UT.u[UT.band[band] + rem % band_units];
  const bool is_vs = kPat == kPatV || (kHasV && U.pattern == kUnitVS);
  const bool is_block = kPat == kPatB || (kHasB && U.pattern == kUnitBlock);
  const bool is_ashape = kPat == kPatA || (kHasA && U.pattern == kUnitAshape);
  const int n = SI.n;
  const Geo G = make_geo(U, t, n, n_tiles(n));
  // rows of the [rows, d] views: token i of head h of this sequence is row H * tok0 + h * n + i
  const int32_t qrow0 = A.Hq * SI.tok0, krow0 = A.Hkv * SI.tok0 + U.kvh * n;
  {  // a row range (chunked attention) skips the items outside it; the whole CTA agrees
    bool in_range = false;
#pragma unroll
    for (int hh = 0; hh < 4; ++hh) in_range = in_range || (G.ex[hh] && G.row0[hh] >= A.row_lo && G.row0[hh] < A.row_hi);
    if (!in_range) return;
  }

  if (warp == 0) {
    tmem_alloc(const_cast<uint32_t*>(&misc[0]), kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 32 * kMmaWarp0) {
    mbar_init(&bars[kBarQ], 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(&bars[kBarFull + s], 1);
      mbar_init(&bars[kBarEmpty + s], 2);  // one release per MMA issuer
    }
    for (int X = 0; X < 2; ++X) {
      mbar_init(&bars[kBarSFull + X], 1);
      mbar_init(&bars[kBarPFull + X], 4);
      mbar_init(&bars[kBarODone + X], 1);
    }
    for (int s = 0; s < kDescSlots; ++s) {
      mbar_init(&bars[kBarDFull + s], 1);
      mbar_init(&bars[kBarDEmpty + s], kDescReaders);
    }
    misc[2] = 0;
    for (int q = 0; q < 4; ++q) misc[8 + q] = 0;  // softmax turns (one per SMSP)
    fence_mbar_init();
  }
  // masking K-step operands: row selectors (row r of sub-item X has 1.0 in
  // column 2X + r / 64), key-mask slots zeroed (their columns 0-3 are written per tile)
  if (is_vs) {
    for (int x = threadIdx.x; x < 4 * 128; x += kThreads) {
      const int op = x >> 7, r = x & 127;
      uint8_t* row = sm + Ly::kAug + op * 4096 + (r >> 3) * 256 + (r & 7) * 16;
      uint32_t w[2] = {0u, 0u};
      if (op < 2) {
        const int col = 2 * op + (r >> 6);
        w[col >> 1] = 0x3F80u << (16 * (col & 1));  // bf16 1.0
      }
      *reinterpret_cast<uint4*>(row) = make_uint4(w[0], w[1], 0u, 0u);     // columns 0-7
      *reinterpret_cast<uint4*>(row + 128) = make_uint4(0u, 0u, 0u, 0u);  // columns 8-15
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];

  uint8_t* sQ = sm + Ly::kQ;
  uint8_t* sR = sm + Ly::kRing;
  auto desc_full = [&](int j) { return mbar_wait(&bars[kBarDFull + j % kDescSlots], (j / kDescSlots) & 1); };
  auto desc_release = [&](int j) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[kBarDEmpty + j % kDescSlots]);
  };

  if (warp == kPlannerWarp) {
    // ------------------------------------------------------------ planner
    AshapeSeg as;
    BlockSeg bs;
    VSSeg vw;
    if (is_ashape) as.init(U, G, n);
    else if (is_block) bs.init(U, G, A, SI, lane, sblk);
    else if (kHasV) vw.init(U, G, A, SI);
    bool ok = true;
    for (int j = 0;; ++j) {
      if (misc[2]) { ok = false; break; }
      const int slot = j % kDescSlots;
      if (!mbar_wait_idle(&bars[kBarDEmpty + slot], ((j / kDescSlots) & 1) ^ 1, kIdleNs)) { ok = false; break; }
      TileDesc& d = descs[slot];
      bool more;
      if (is_vs) {
        more = vw.emit(lane, n, d);
      } else {
        // lane 0 takes up to two segments of the union
        int sg[2] = {0, 0}, rl[2][2] = {{0, 0}, {0, 0}}, bits[2] = {0, 0};
        int got = 0;
        if (kHasA && lane == 0 && is_ashape) {
          for (; got < 2; ++got) {
            int s = 0, r2[2] = {0, 0};
            if (!as.next(s, r2)) break;
            sg[got] = s;
            rl[0][got] = r2[0];
            rl[1][got] = r2[1];
            bits[got] = (r2[0] ? 3 : 0) | (r2[1] ? 12 : 0);
          }
        } else if (kHasB && lane == 0) {
          // Block-Sparse: the two blocks of a tile are taken from the same class
          // (kept by sub-item 0 only, by sub-item 1 only, or by both), so that a
          // sub-item skips the tiles it does not attend; a block waits in
          // pend[class] for its partner, and the leftovers close the item.
          for (;;) {
            int s = 0, b = 0;
            const bool has = bs.next(s, b);
            if (!has) {
              for (int c = 1; c < 4 && got < 2; ++c)
                if (bs.pend[c] >= 0) { sg[got] = bs.pend[c]; bits[got] = bs.pendb[c]; bs.pend[c] = -1; ++got; }
              break;
            }
            if (b < 0) { b = 0; set_error(A.err, kErrIndex); }
            for (int hh = 0; hh < 4; ++hh)  // a block must be causal for each half that keeps it
              if (((b >> hh) & 1) && (s < 0 || s > bs.u[hh])) { b &= ~(1 << hh); set_error(A.err, kErrIndex); }
            if (s < 0 || 64 * s >= n) b = 0;
            const int c = ((b & 3) ? 1 : 0) | ((b & 12) ? 2 : 0);
            if (c == 0) continue;  // kept by no half
            if (bs.pend[c] >= 0) {
              sg[0] = bs.pend[c]; bits[0] = bs.pendb[c];
              sg[1] = s; bits[1] = b;
              got = 2;
              bs.pend[c] = -1;
              break;
            }
            bs.pend[c] = s;
            bs.pendb[c] = b;
          }
        }
        got = __shfl_sync(0xFFFFFFFFu, got, 0);
        more = got > 0;
        if (more && lane == 0) {
          if (got == 1) { sg[1] = sg[0]; bits[1] = 0; rl[0][1] = rl[1][1] = 0; }  // reload a valid segment, masked
          d.kind = kTileRange;
          for (int s = 0; s < 2; ++s) {
            d.seg[s] = 64 * sg[s];
            for (int w = 0; w < 2; ++w) {
              const uint32_t m = keys_below(64 * sg[s] + 32 * w, n);
              for (int hh = 0; hh < 4; ++hh) d.mask[hh][2 * s + w] = ((bits[s] >> hh) & 1) ? m : 0u;
            }
          }
          for (int X = 0; X < 2; ++X) {
            d.rule[X][0] = (uint8_t)rl[X][0];
            d.rule[X][1] = (uint8_t)rl[X][1];
            d.active[X] = (((bits[0] | bits[1]) >> (2 * X)) & 3) != 0;
          }
          d.bias = 0;  // range tiles: whole 64-key segments per half, masked by the softmax
        }
      }
      if (!more && lane == 0) d.kind = kTileEnd;
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarDFull + slot]);
      if (!more) break;
    }
    if (!ok) { misc[2] = 1; set_error(A.err, kErrTimeout); }
  } else if (warp == kLoaderWarp) {
    // ------------------------------------------------------------ loader
    if (lane == 0) {
      tma_prefetch_desc(&M.q);
      tma_prefetch_desc(&M.k);
      tma_prefetch_desc(&M.v);
      // Q rows of the halves that exist (a tail past n reads zeros)
      int halves = 0;
      for (int hh = 0; hh < 4; ++hh) halves += G.ex[hh];
      mbar_arrive_expect_tx(&bars[kBarQ], (uint32_t)(halves * (D / 64) * 8192));
      for (int hh = 0; hh < 4; ++hh)
        if (G.ex[hh])
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d_hint(sQ + (hh >> 1) * Ly::kTile + c * 16384 + (hh & 1) * 8192, &M.q, &bars[kBarQ], 64 * c,
                        qrow0 + U.sub[hh >> 1].qh[hh & 1] * n + G.row0[hh], 0, policy_evict_first());
    }
    // K and V tiles are re-read by the other items of their KV head: keep them in
    // L2 ahead of Q (read once, evict-first) and O (written with streaming stores)
    const uint64_t kv_policy = policy_evict_last();
    // K(j) into slot 2j, V(j) into 2j+1 (mod kSlots): the MMA releases them in that order
    auto load = [&](int j, bool is_v) -> bool {
      const int idx = 2 * j + (is_v ? 1 : 0);
      const int st = idx % kSlots;
      if (!mbar_wait_idle(&bars[kBarEmpty + st], ((idx / kSlots) & 1) ^ 1, kIdleNs)) return false;
      const TileDesc& d = descs[j % kDescSlots];
      uint8_t* dst = sR + st * Ly::kTile;
      uint64_t* full = &bars[kBarFull + st];
      if (kHasV && !is_v && d.bias) {
        // key-mask slot j mod 2 (free: the K(j - 2) releases came after its last reads):
        // row k, column hh = 0 if half hh attends key k, else -BIG; lane l writes rows 4l..4l+3
        uint8_t* ka = sm + Ly::kAug + (2 + (j & 1)) * 4096;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int k = 4 * lane + q;
          uint32_t w[2];
#pragma unroll
          for (int p2 = 0; p2 < 2; ++p2) {
            const uint32_t lo = ((d.mask[2 * p2][k >> 5] >> (k & 31)) & 1u) ? 0u : (uint32_t)kBf16NegBig;
            const uint32_t hi = ((d.mask[2 * p2 + 1][k >> 5] >> (k & 31)) & 1u) ? 0u : (uint32_t)kBf16NegBig;
            w[p2] = lo | (hi << 16);
          }
          *reinterpret_cast<uint4*>(ka + (k >> 3) * 256 + (k & 7) * 16) = make_uint4(w[0], w[1], 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();  // every lane's rows are written before the full barrier's arrival
      }
      if (!kHasV || d.kind == kTileRange) {
        if (lane == 0) {
          const CUtensorMap* map = is_v ? &M.v : &M.k;
          mbar_arrive_expect_tx(full, Ly::kTile);
          for (int s = 0; s < 2; ++s)
            for (int c = 0; c < D / 64; ++c) tma_load_3d_hint(dst + c * 16384 + s * 8192, map, full, 64 * c, krow0 + d.seg[s], 0, kv_policy);
        }
      } else {
        // eight 16-key segments (lane 8c + x: segment x, columns 64c..): a run
        // of four contiguous segments loads as one 64-row box
        if (lane == 0) mbar_arrive_expect_tx(full, Ly::kTile);
        __syncwarp();
        if (lane < 8 * (D / 64)) {
          const int x = lane & 7, c = lane >> 3, h4 = x & ~3;
          const int s0 = d.seg[h4];
          const bool run = d.seg[h4 + 1] == s0 + 16 && d.seg[h4 + 2] == s0 + 32 && d.seg[h4 + 3] == s0 + 48;
          if (!run)
            tma_load_3d_hint(dst + c * 16384 + x * 2048, is_v ? &M.v16 : &M.k16, full, 64 * c, krow0 + d.seg[x], 0, kv_policy);
          else if (x == h4)
            tma_load_3d_hint(dst + c * 16384 + x * 2048, is_v ? &M.v : &M.k, full, 64 * c, krow0 + s0, 0, kv_policy);
        }
      }
      return true;
    };
    bool ok = true;
    for (int j = 0;; ++j) {
      if (misc[2]) { ok = false; break; }
      if (!mbar_wait_idle(&bars[kBarDFull + j % kDescSlots], (j / kDescSlots) & 1, kIdleNs)) { ok = false; break; }
      if (descs[j % kDescSlots].kind == kTileEnd) { desc_release(j); break; }
      if (!load(j, false) || !load(j, true)) { ok = false; break; }
      desc_release(j);
    }
    if (!ok) { misc[2] = 1; set_error(A.err, kErrTimeout); }
  } else if (warp == kMmaWarp0 || warp == kMmaWarp1) {
    // ------------------------------------------------------------ MMA issuer of sub-item X
    // Each sub-item has its own issuing thread, so one sub-item waiting for its
    // P never holds back the other's MMAs.  Both read the shared K/V ring and
    // each releases every slot once (the empty barriers count two arrivals).
    const int X = warp == kMmaWarp0 ? 0 : 1;
    bool ok = mbar_wait(&bars[kBarQ], 0);
    constexpr uint32_t id_qk = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t id_pv = idesc_bf16_f32(128, D, false, true);
    int pending = -1;  // tile whose PV is owed (always the previous tile of this sub-item)
    int done = 0;      // PVs issued (the first one overwrites O)
    int pphase = 0;
    // Shared-memory descriptors of the operand tiles; a byte offset off within a
    // tile adds off >> 4 to the start-address field (no carry: addresses < 2^18).
    constexpr uint64_t kTileDesc = Ly::kTile >> 4;
    const uint64_t dq = sdesc_sw128(smem_u32(sQ), 16, 1024) + (uint64_t)X * kTileDesc;
    const uint64_t dk = sdesc_sw128(smem_u32(sR), 16, 1024);  // + slot * kTile
    const uint64_t dv = sdesc_sw128(smem_u32(sR), 16384, 1024);
    const uint64_t dqa = sdesc_plain(smem_u32(sm + Ly::kAug + X * 4096), 128, 256);
    const uint64_t dka = sdesc_plain(smem_u32(sm + Ly::kAug + 2 * 4096), 128, 256);  // + (j & 1) * 4096
    const uint32_t tS = tmem + kColS + 128 * X, tO = tmem + kColO + 128 * X;
    auto issue_pv = [&]() -> bool {  // O_X += P_X V of tile `pending`, then release that V slot
      const int vidx = 2 * pending + 1, vst = vidx % kSlots;
      if (!mbar_wait(&bars[kBarPFull + X], pphase & 1)) return false;
      ++pphase;
      if (!mbar_wait(&bars[kBarFull + vst], (vidx / kSlots) & 1)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint64_t v0 = dv + (uint64_t)vst * kTileDesc;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16_ts(tO, tS + 8 * kk, v0 + (uint64_t)(kk * 128), id_pv, (done > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars[kBarEmpty + vst]);
      }
      __syncwarp();
      ++done;
      pending = -1;
      return true;
    };
    if (ok) tc_fence_after();
    for (int j = 0; ok; ++j) {
      if (misc[2] || !desc_full(j)) { ok = false; break; }
      const TileDesc& d = descs[j % kDescSlots];
      const bool end = d.kind == kTileEnd;
      const bool act = d.active[X] != 0;
      const bool bias = kHasV && d.bias != 0;
      desc_release(j);
      if (end) break;
      const int kidx = 2 * j, kst = kidx % kSlots;
      if (!mbar_wait(&bars[kBarFull + kst], (kidx / kSlots) & 1)) { ok = false; break; }
      tc_fence_after();
      if (pending >= 0 && !issue_pv()) { ok = false; break; }  // P_X of the previous tile -> O_X
      if (act) {
        if (lane == 0) {
          const uint64_t k0 = dk + (uint64_t)kst * kTileDesc;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t off = (uint64_t)((kk >> 2) * 1024 + (kk & 3) * 2);  // ((kk/4) * 16384 + (kk%4) * 32) >> 4
            mma_bf16_ss(tS, dq + off, k0 + off, id_qk, kk > 0 ? 1u : 0u);
          }
          if (bias) mma_bf16_ss(tS, dqa, dka + (uint64_t)((j & 1) * (4096 >> 4)), id_qk, 1u);
          mma_commit(&bars[kBarSFull + X]);
        }
        __syncwarp();
        pending = j;
      } else {  // this sub-item never reads V(j): release it once it has landed
        const int vidx = 2 * j + 1;
        if (!mbar_wait(&bars[kBarFull + vidx % kSlots], (vidx / kSlots) & 1)) { ok = false; break; }
        if (lane == 0) mma_commit(&bars[kBarEmpty + vidx % kSlots]);
      }
      if (lane == 0) mma_commit(&bars[kBarEmpty + kst]);  // K(j) consumed by this issuer
      __syncwarp();
    }
    if (ok && pending >= 0 && !issue_pv()) ok = false;
    if (lane == 0) mma_commit(&bars[kBarODone + X]);  // arrives once every MMA issued above has completed
    __syncwarp();
    if (!ok) { misc[2] = 1; set_error(A.err, kErrTimeout); }
  } else if (warp < kSoftWarps) {
    // ------------------------------------------------------------ softmax (sub-item X)
    const int quarter = warp & 3;  // TMEM lanes 32*quarter ..
    const int X = warp >> 2;
    const int r = quarter * 32 + lane;  // tile row = TMEM lane
    const int hh = 2 * X + (r >> 6);
    const int i = G.row0[hh] + (r & 63);
    const bool row_ok = G.ex[hh] && i < n;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const uint32_t colS = kColS + 128 * X, colO = kColO + 128 * X;
    const float c2 = A.scale_log2;
    const int g = U.sub[X].sink, wnd = U.sub[X].window;
    const bool ashape = kHasA && is_ashape;
    float m_used = -INFINITY, l = 0.f;
    unsigned long long count = 0;
    bool ok = true;
    int mine = 0;  // tiles this sub-item has processed

    for (int j = 0;; ++j) {
      if (misc[2]) { ok = false; break; }
      if (!desc_full(j)) { ok = false; break; }
      const TileDesc& d = descs[j % kDescSlots];
      const int kind = d.kind;
      if (kind == kTileEnd) { desc_release(j); break; }
      if (!d.active[X]) { desc_release(j); continue; }
      // ---- validity words of this row's 128 keys (the half's key set only
      // where the tensor core has not masked it)
      const bool bias = kHasV && d.bias != 0;
      uint64_t vw[2] = {0ull, 0ull};
      if (row_ok) {
        // causal keys of each 64-column half are its first c[s] columns: for
        // 64-key segments c = i - start + 1; for 16-key segments keys ascend
        // over the tile, so the count comes from a 3-step search over the
        // eight segment starts and the partial one
        int c0, c1;
        if (!kHasV || kind == kTileRange) {
          c0 = i - d.seg[0] + 1;
          c1 = i - d.seg[1] + 1;
        } else if (d.seg_hi + 15 <= i) {
          c0 = c1 = 64;
        } else {
          int sc = 0;
#pragma unroll
          for (int step = 4; step; step >>= 1)
            if (d.seg[sc + step - 1] + 15 <= i) sc += step;
          c0 = 16 * sc + min(max(i - d.seg[sc] + 1, 0), 16);  // sc <= 7 here
          c1 = c0 - 64;
        }
        const uint64_t hm0 = ((uint64_t)d.mask[hh][1] << 32) | d.mask[hh][0];
        const uint64_t hm1 = ((uint64_t)d.mask[hh][3] << 32) | d.mask[hh][2];
        vw[0] = (bias ? ~0ull : hm0) & low_mask64(c0);
        vw[1] = (bias ? ~0ull : hm1) & low_mask64(c1);
        if (ashape) {
#pragma unroll
          for (int s = 0; s < 2; ++s) {
            const int base = d.seg[s], rule = d.rule[X][s];
            uint64_t keep = 0;
            if (rule & 1) keep |= low_mask64(g - base);             // j < g
            if (rule & 2) keep |= ~low_mask64(i - wnd + 1 - base);  // j > i - w
            vw[s] &= keep;
          }
        }
        if (kCount) count += __popcll(vw[0] & hm0) + __popcll(vw[1] & hm1);
      }
      desc_release(j);

      // ---- S of this tile (its completion also means this sub-item's previous PV is done)
      if (!mbar_wait(&bars[kBarSFull + X], mine & 1)) { ok = false; break; }
      tc_fence_after();
      float sv[128];
      {
        uint32_t* u = reinterpret_cast<uint32_t*>(sv);
#pragma unroll
        for (int c = 0; c < 4; ++c)
          tmem_ld32(tmem + lane_base + colS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(u + 32 * c));
        tmem_ld_wait();
      }
      // The softmax sections of the two sub-items' warps on this SMSP (warp q
      // and warp q + 4) take turns, from the max to the last P store: each runs
      // at full issue rate while the tensor core works for the other, instead
      // of both stretching into each other's MMA window.
      if (kTurnLock) {
        if (lane == 0) {
          const uint64_t t0 = global_timer_ns();
          while (atomicCAS(const_cast<uint32_t*>(&misc[8 + quarter]), 0u, 1u) != 0u)
            if (global_timer_ns() - t0 > MSA_WAIT_LIMIT_NS) { misc[2] = 1; set_error(A.err, kErrTimeout); break; }
        }
        __syncwarp();
      }
      // ---- mask, row max (tree)
      if ((~vw[0]) | (~vw[1])) {
#pragma unroll
        for (int k = 0; k < 64; ++k) sv[k] = ((vw[0] >> k) & 1ull) ? sv[k] : -INFINITY;
#pragma unroll
        for (int k = 0; k < 64; ++k) sv[64 + k] = ((vw[1] >> k) & 1ull) ? sv[64 + k] : -INFINITY;
      }
      float mx[8];
#pragma unroll
      for (int x = 0; x < 8; ++x) mx[x] = max3f(sv[x], sv[8 + x], sv[16 + x]);
#pragma unroll
      for (int k = 24; k < 120; k += 16)
#pragma unroll
        for (int x = 0; x < 8; ++x) mx[x] = max3f(mx[x], sv[k + x], sv[k + 8 + x]);
#pragma unroll
      for (int x = 0; x < 8; ++x) mx[x] = fmaxf(mx[x], sv[120 + x]);
      float mt = max3f(max3f(mx[0], mx[1], mx[2]), max3f(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
      if (kHasV && mt < kMaskedBelow) mt = -INFINITY;  // every key of the tile masked for this row
      const float m_new = fmaxf(m_used, mt * c2);
      const bool need = m_new > m_used + kRescaleThreshold;
      const bool any = __any_sync(0xFFFFFFFFu, need);
      float alpha = 1.f;
      if (any && m_new != -INFINITY) {
        alpha = (m_used == -INFINITY) ? 0.f : ex2(m_used - m_new);
        m_used = m_new;
      }
      const float mref = (m_used == -INFINITY) ? 0.f : m_used;
      const uint64_t c2x2 = pk2(c2, c2), negm = pk2(-mref, -mref);
      uint64_t acc[2] = {pk2(0.f, 0.f), pk2(0.f, 0.f)};
      // ---- P over the first 64 columns of S, kPChunk columns (2 kPChunk keys) at a time
#pragma unroll
      for (int half = 0; half < 64 / kPChunk; ++half) {
        uint32_t pk[kPChunk];
#pragma unroll
        for (int k = 0; k < kPChunk; ++k) {
          const int e = 2 * kPChunk * half + 2 * k;
          const uint64_t x = fma2(pk2(sv[e], sv[e + 1]), c2x2, negm);
          float x0, x1;
          up2(x, x0, x1);
          const uint64_t p = pk2(ex2(x0), ex2(x1));
          acc[k & 1] = add2(acc[k & 1], p);
          float p0, p1;
          up2(p, p0, p1);
          pk[k] = pack_bf16x2(p0, p1);
        }
        tmem_st4(tmem + lane_base + colS + kPChunk * half, pk);
      }
      {
        float a0, a1, a2, a3;
        up2(acc[0], a0, a1);
        up2(acc[1], a2, a3);
        l = l * alpha + ((a0 + a1) + (a2 + a3));
      }
      if (kTurnLock) {
        __syncwarp();
        if (lane == 0) atomicExch(const_cast<uint32_t*>(&misc[8 + quarter]), 0u);
      }
      // ---- rescale O_X (its previous PV completed before S was ready; the next waits for P)
      if (any && mine > 0) {
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tmem + lane_base + colO + 32 * c, o);
          tmem_ld_wait();
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * alpha);
          tmem_st32(tmem + lane_base + colO + 32 * c, o);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarPFull + X]);
      ++mine;
    }
    if (!ok) { misc[2] = 1; set_error(A.err, kErrTimeout); }

    // ---- epilogue: O / l, LSE
    if (!mbar_wait(&bars[kBarODone + X], 0)) { ok = false; misc[2] = 1; set_error(A.err, kErrTimeout); }
    tc_fence_after();
    const int qh = U.sub[X].qh[hh & 1];
    const bool empty = !(m_used > -INFINITY);  // no attended key in any tile: o = 0
    const float inv_l = (!empty && l > 0.f) ? 1.f / l : 0.f;
    const bool have = ok && mine > 0;  // warp-uniform: tcgen05.ld below is warp-collective
    const int64_t orow_idx = (int64_t)qrow0 + (int64_t)qh * n + i;
    __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(A.o) + orow_idx * D;
#pragma unroll 1
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      if (have) {
        tmem_ld32(tmem + lane_base + colO + 32 * c, o);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int x = 0; x < 32; ++x) o[x] = 0u;
      }
      if (row_ok) {
        uint32_t pkd[16];
#pragma unroll
        for (int x = 0; x < 16; ++x)
          pkd[x] = pack_bf16x2(__uint_as_float(o[2 * x]) * inv_l, __uint_as_float(o[2 * x + 1]) * inv_l);
        uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
        for (int x = 0; x < 4; ++x) __stcs(dst + x, make_uint4(pkd[4 * x], pkd[4 * x + 1], pkd[4 * x + 2], pkd[4 * x + 3]));
      }
    }
    if (row_ok && A.lse)
      A.lse[orow_idx] = (!empty && l > 0.f) ? (m_used + __log2f(l)) * 0.69314718055994531f : -INFINITY;
    if (kCount && A.edges) {  // the 32 rows of a warp lie in one half, so in one head
      unsigned long long c = count;
      for (int o = 16; o; o >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
      if (lane == 0 && c) atomicAdd(A.edges + (int64_t)SI.seq * A.Hq + qh, c);
    }
    // every tile of this sub-item is a 64-row x 128-key tile of each of its halves (counted by the half's first warp)
    if (kCount && A.tiles && (quarter & 1) == 0 && lane == 0 && G.ex[hh] && mine > 0)
      atomicAdd(A.tiles + (int64_t)SI.seq * A.Hq + qh, (unsigned long long)mine);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool kCount, int kPat>
msa_status launch_impl(const AttnMaps& maps, const AttnArgs& a, const UnitTable& ut, const SeqTable& st,
                       int64_t items, cudaStream_t stream) {
  auto kern = sparse_attn_kernel<D, kCount, kPat>;
  const int smem = Layout<D>::kAlloc;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return MSA_ERR_CUDA;
  if (items <= 0) return MSA_OK;
  if (items > 0x7FFFFFFF) return MSA_ERR_UNSUPPORTED;
  kern<<<(unsigned)items, kThreads, smem, stream>>>(maps, a, ut, st);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

template <int kPat>
msa_status launch_d(int d, bool count, const AttnMaps& maps, const AttnArgs& a, const UnitTable& ut,
                    const SeqTable& st, int64_t items, cudaStream_t stream) {
  if (d == 128)
    return count ? launch_impl<128, true, kPat>(maps, a, ut, st, items, stream)
                 : launch_impl<128, false, kPat>(maps, a, ut, st, items, stream);
  return count ? launch_impl<64, true, kPat>(maps, a, ut, st, items, stream)
               : launch_impl<64, false, kPat>(maps, a, ut, st, items, stream);
}

msa_status launch_pat(int pat, int d, bool count, const AttnMaps& maps, const AttnArgs& a, const UnitTable& ut,
                      const SeqTable& st, int64_t items, cudaStream_t stream) {
  switch (pat) {
    case kPatA: return launch_d<kPatA>(d, count, maps, a, ut, st, items, stream);
    case kPatV: return launch_d<kPatV>(d, count, maps, a, ut, st, items, stream);
    case kPatB: return launch_d<kPatB>(d, count, maps, a, ut, st, items, stream);
    default: return launch_d<kPatAll>(d, count, maps, a, ut, st, items, stream);
  }
}

}  // namespace

namespace {

// Units of one launch stream (chunks of kMaxUnits, each one kernel launch).
msa_status launch_units(const AttnMaps& maps, const AttnArgs& args, const Unit* units, int n_units, SeqTable& seqs,
                        cudaStream_t stream) {
  for (int base = 0; base < n_units; base += kMaxUnits) {
    UnitTable ut;
    const int cnt = n_units - base < kMaxUnits ? n_units - base : kMaxUnits;
    for (int x = 0; x < cnt; ++x) ut.u[x] = units[base + x];
    std::stable_sort(ut.u, ut.u + cnt, [](const Unit& p, const Unit& q) { return p.kvh < q.kvh; });
    int nb = 0;
    for (int x = 0; x < cnt; ++x)
      if (x == 0 || ut.u[x].kvh != ut.u[x - 1].kvh) ut.band[nb++] = x;
    ut.band[nb] = cnt;
    // items: every unit for every sequence, the sequences in table order
    int64_t items = 0;
    for (int x = 0; x < seqs.count; ++x) {
      seqs.s[x].T = (n_tiles(seqs.s[x].n) + 1) / 2;
      seqs.s[x].item0 = (int32_t)items;
      items += (int64_t)seqs.s[x].T * cnt;
    }
    AttnArgs a = args;
    a.n_units = cnt;
    a.n_bands = nb;
    int pat = 0;
    for (int x = 0; x < cnt; ++x) pat |= 1 << ut.u[x].pattern;
    if (pat != kPatA && pat != kPatV && pat != kPatB) pat = kPatAll;
    const bool count = args.edges != nullptr || args.tiles != nullptr;
    const msa_status st = launch_pat(pat, args.d, count, maps, a, ut, seqs, items, stream);
    if (st != MSA_OK) return st;
  }
  return MSA_OK;
}

}  // namespace

SideStreams* side_streams() {
  static std::mutex mu;
  static SideStreams sets[64];
  static bool made[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!made[dev]) {
    SideStreams& f = sets[dev];
    f.ok = true;
    for (int x = 0; x < 2; ++x) f.ok = f.ok && cudaStreamCreateWithFlags(&f.side[x], cudaStreamNonBlocking) == cudaSuccess;
    for (int x = 0; x < 3; ++x) f.ok = f.ok && cudaEventCreateWithFlags(&f.ev[x], cudaEventDisableTiming) == cudaSuccess;
    made[dev] = true;
  }
  return sets[dev].ok ? &sets[dev] : nullptr;
}

// A launch whose units hold several patterns runs each pattern's units in the
// kernel compiled for that pattern alone, Vertical-Slash on `stream` and the
// others on two side streams forked from it and joined back: the kernels then
// share the SMs, each CTA running only its own pattern's code.
msa_status launch_attention(const AttnMaps& maps, const AttnArgs& args, const Unit* units, int n_units,
                            SeqTable& seqs, cudaStream_t stream) {
  std::vector<Unit> by[3];
  for (int x = 0; x < n_units; ++x) by[units[x].pattern].push_back(units[x]);
  const int kinds = (by[0].empty() ? 0 : 1) + (by[1].empty() ? 0 : 1) + (by[2].empty() ? 0 : 1);
  SideStreams* f = kinds > 1 ? side_streams() : nullptr;
  if (!f) return launch_units(maps, args, units, n_units, seqs, stream);
  std::lock_guard<std::mutex> hold(f->mu);
  if (cudaEventRecord(f->ev[0], stream) != cudaSuccess) return MSA_ERR_CUDA;
  const int order[3] = {kUnitVS, kUnitBlock, kUnitAshape};
  cudaStream_t on[3] = {stream, f->side[0], f->side[1]};
  msa_status st = MSA_OK;
  for (int x = 0; x < 3; ++x) {
    const std::vector<Unit>& u = by[order[x]];
    if (u.empty()) continue;
    if (x > 0 && cudaStreamWaitEvent(on[x], f->ev[0], 0) != cudaSuccess) return MSA_ERR_CUDA;
    const msa_status r = launch_units(maps, args, u.data(), (int)u.size(), seqs, on[x]);
    if (r != MSA_OK && st == MSA_OK) st = r;
  }
  for (int x = 1; x < 3; ++x) {
    if (by[order[x]].empty()) continue;
    if (cudaEventRecord(f->ev[x], on[x]) != cudaSuccess || cudaStreamWaitEvent(stream, f->ev[x], 0) != cudaSuccess)
      return MSA_ERR_CUDA;
  }
  return st;
}

}  // namespace msa
