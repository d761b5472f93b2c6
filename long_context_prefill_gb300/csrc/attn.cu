// Sparse causal attention engine for sm_103a (A-shape, Vertical-Slash and
// Block-Sparse heads in one kernel).
//
// What it computes (MInference page, eq.(1)-(2) restricted to N_h(i), with
// the online-softmax merge of eq.(7)-(8)): for every query row i of a work
// item, o_i = Σ_{j in N(i)} e^{s_ij} v_j / Σ_{j in N(i)} e^{s_ij}.
//
// One CTA processes one item: 128 query rows (two 64-row halves) of one KV
// group against a stream of 128-key tiles that a pattern iterator generates.
//   warp 8     planner: runs the pattern's tile iterator and writes each
//              tile's descriptor (two 64-key segments and per-half validity
//              masks) into a ring, then a terminating descriptor;
//   warp 10    loader: TMA-loads the K and V segments of each tile (any start
//              row), or gathers single key rows (Vertical-Slash columns) with
//              cp.async;
//   warp 9     MMA issuer (one thread): S = Q K^T into TMEM (two buffers),
//              then O += P V into a TMEM accumulator; Q and P are read from
//              TMEM, K and V from shared memory;
//   warps 0-7  softmax: query row r is TMEM lane r; warps w and w+4 share
//              the lanes of quarter w and split the 128 keys (and the O
//              columns) in halves, exchanging the row max through shared
//              memory.  Masks (causal, pattern, sequence end) are applied
//              before the max; O is rescaled in TMEM only when the max grows
//              by more than 2^8; P is written to TMEM as bf16 pairs.
// Every (i, j) pair enters the softmax at most once: tiles partition the keys
// of an item, and masks drop what lies outside N(i) (MInference page §3.2 and
// §5.1 "boundary masks": set to -inf before the max).
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace msa {

namespace {

constexpr int kSoftWarps = 8;
constexpr int kPlannerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kLoaderWarp = 10;
constexpr int kThreads = 32 * (kSoftWarps + 3);
constexpr int kStages = 3;
constexpr int kDescSlots = 8;
constexpr int kDescReaders = kSoftWarps + 2;  // softmax warps, MMA warp, loader warp
constexpr int kMaxStagedBlocks = 512;          // Block-Sparse lists merged in shared memory
constexpr uint32_t kTmemCols = 512;
// TMEM columns: two S buffers, the O accumulator, Q and P (bf16 pairs)
constexpr uint32_t kColS = 0, kColO = 256, kColQ = 384, kColP = 448;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

enum TileKind : int32_t { kTileRange = 0, kTileGather = 1, kTileEnd = 2 };

struct TileDesc {
  int32_t seg[2];   // range tiles: first key of each 64-key segment
  int32_t kind;     // TileKind (kTileEnd: no more tiles in this item)
  int32_t rule;     // A-shape row rule: bit0 keeps j < sink, bit1 keeps j > i - window
  uint32_t mask[2][4];  // per half: bit k = key k of the tile may be attended
  int32_t gidx[128];    // gather tiles: key of column k (-1 = empty)
};

enum {
  kBarQ = 0,
  kBarKFull = 1,
  kBarKEmpty = kBarKFull + kStages,
  kBarVFull = kBarKEmpty + kStages,
  kBarVEmpty = kBarVFull + kStages,
  kBarSFull = kBarVEmpty + kStages,
  kBarSEmpty = kBarSFull + 2,
  kBarPFull = kBarSEmpty + 2,
  kBarPEmpty = kBarPFull + 1,
  kBarDFull = kBarPEmpty + 1,
  kBarDEmpty = kBarDFull + kDescSlots,
  kBarX = kBarDEmpty + kDescSlots,  // row exchange of the two warps of each quarter
  kNumBars = kBarX + 4
};

template <int D>
struct Layout {
  static constexpr int kTile = 128 * D * 2;  // 128 key rows of d_h bf16
  static constexpr int kK = 0;
  static constexpr int kV = kK + kStages * kTile;
  static constexpr int kDesc = kV + kStages * kTile;
  static constexpr int kStage = kDesc + kDescSlots * (int)sizeof(TileDesc);  // gather staging (256 ints)
  static constexpr int kBlk = kStage + 256 * 4;  // Block-Sparse lists and their union
  // row exchange: [2 parities][2 key halves][128] maxima, then [2][128] denominators
  static constexpr int kXchg = kBlk + 4 * kMaxStagedBlocks * 4;
  static constexpr int kBars = kXchg + 6 * 128 * 4;
  static constexpr int kMisc = kBars + kNumBars * 8;
  static constexpr int kTotal = kMisc + 64;
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

__device__ __forceinline__ uint64_t low_mask64(int c) {  // bits [0, c), c clamped to [0, 64]
  c = c < 0 ? 0 : (c > 64 ? 64 : c);
  return c >= 64 ? ~0ull : ((1ull << c) - 1ull);
}

__device__ __forceinline__ uint32_t low_mask32(int c) {
  c = c < 0 ? 0 : (c > 32 ? 32 : c);
  return c >= 32 ? 0xFFFFFFFFu : ((1u << c) - 1u);
}

// Any bit of `bits` (an n-bit map) set in [lo, hi] ∩ [0, n)?
__device__ __forceinline__ bool bits_any(const uint32_t* bits, int n, int lo, int hi) {
  lo = lo < 0 ? 0 : lo;
  hi = hi > n - 1 ? n - 1 : hi;
  if (lo > hi) return false;
  const int w0 = lo >> 5, w1 = hi >> 5;
  for (int w = w0; w <= w1; ++w) {
    uint32_t x = __ldg(bits + w);
    if (w == w0) x &= 0xFFFFFFFFu << (lo & 31);
    if (w == w1) x &= 0xFFFFFFFFu >> (31 - (hi & 31));
    if (x) return true;
  }
  return false;
}

__device__ __forceinline__ bool bit_at(const uint32_t* bits, int j) { return (__ldg(bits + (j >> 5)) >> (j & 31)) & 1u; }

// 32 bits of an nw-word map starting at bit p >= 0 (bits past the end read 0).
__device__ __forceinline__ uint32_t bits_window32(const uint32_t* bits, int nw, int p) {
  const int w = p >> 5, sh = p & 31;
  const uint32_t lo = w < nw ? __ldg(bits + w) : 0u;
  const uint32_t hi = (w + 1) < nw ? __ldg(bits + w + 1) : 0u;
  return __funnelshift_r(lo, hi, sh);
}

__device__ __forceinline__ uint32_t keys_below(int base, int limit) {  // bits k with base + k < limit
  return low_mask32(limit - base);
}

// ------------------------------------------------------------------ item geometry
struct Item {
  int row0[2];   // first query row of each half
  int exists[2]; // half has at least one row < n
  int e[2];      // last row of each half's query block (clipped to n-1)
  int a0;        // 128 * t
};

__device__ __forceinline__ Item make_item(const Unit& U, int t, int n) {
  Item it;
  it.a0 = 128 * t;
  for (int h = 0; h < 2; ++h) {
    it.row0[h] = 128 * t + U.row_off[h];
    it.exists[h] = it.row0[h] < n;
    int e = it.row0[h] + 63;
    it.e[h] = e < n - 1 ? e : n - 1;
  }
  return it;
}

// ------------------------------------------------------------------ A-shape tiles
// MInference page eq.(3): rows i of the item attend j < g or i-w < j <= i.
// The key ranges [0, g) and [a0-w+1, a0+127] (merged when they touch) are cut
// into 128-key tiles; a per-tile row rule applies the exact set.
struct AshapeIter {
  int lo[2], hi[2], rule[2], tiles[2];
  __device__ void init(const Unit& U, const Item& it, int n) {
    const int hi_key = min(it.a0 + 127, n - 1);
    const int g = U.sink, w = U.window;
    const int sw = max(0, it.a0 - w + 1);
    if (sw <= g) {
      lo[0] = 0; hi[0] = hi_key; rule[0] = 3;
      lo[1] = 0; hi[1] = -1; rule[1] = 0;
    } else {
      lo[0] = 0; hi[0] = min(g, n) - 1; rule[0] = 1;
      lo[1] = sw; hi[1] = hi_key; rule[1] = 2;
    }
    for (int r = 0; r < 2; ++r) tiles[r] = hi[r] >= lo[r] ? (hi[r] - lo[r] + 128) / 128 : 0;
  }
  __device__ int count() const { return tiles[0] + tiles[1]; }
  __device__ void emit(int j, int n, TileDesc& d) const {
    const int r = j < tiles[0] ? 0 : 1;
    const int t0 = lo[r] + 128 * (r == 0 ? j : j - tiles[0]);
    d.seg[0] = t0;
    d.seg[1] = t0 + 64;
    d.kind = 0;
    d.rule = rule[r];
    for (int w = 0; w < 4; ++w) {
      const uint32_t m = keys_below(t0 + 32 * w, n);
      d.mask[0][w] = m;
      d.mask[1][w] = m;
    }
  }
};

// ------------------------------------------------------------------ Block-Sparse tiles
// MInference page eq.(6): half h (query block u_h) attends the key blocks J_{u_h}.
// The sorted lists of both halves are merged; every pair of consecutive key
// blocks of the union forms one 128-key tile, and each half keeps only its own
// blocks.  The union is built once per item in shared memory (whole warp
// stages the lists, one lane merges); lists longer than the staging buffer are
// merged straight from global memory.
struct BlockIter {
  const int32_t* J[2];
  int cnt[2], u[2];
  int total;   // blocks in the union
  int pos;     // next union entry to emit
  bool staged; // union lives in shared memory (else merged on the fly)
  int p[2], last;
  int* un;     // union entries: block id | membership bits << 28
  __device__ void init(const Unit& U, const Item& it, const AttnArgs& a, int lane, int* sblk) {
    for (int h = 0; h < 2; ++h) {
      u[h] = it.row0[h] / 64;
      J[h] = nullptr;
      cnt[h] = 0;
      if (it.exists[h]) {
        const int64_t off = (int64_t)U.slot[h] * a.bs_nb + u[h];
        J[h] = a.bs_idx + off * a.bs_topk;
        const int c = __ldg(a.bs_cnt + off);
        cnt[h] = c < 0 ? 0 : (c > a.bs_topk ? a.bs_topk : c);
      }
    }
    pos = 0;
    p[0] = p[1] = 0;
    last = -1;
    un = sblk + 2 * kMaxStagedBlocks;
    staged = cnt[0] <= kMaxStagedBlocks && cnt[1] <= kMaxStagedBlocks;
    if (staged) {
      for (int h = 0; h < 2; ++h)
        for (int x = lane; x < cnt[h]; x += 32) sblk[h * kMaxStagedBlocks + x] = __ldg(J[h] + x);
      __syncwarp();
      if (lane == 0) {
        int x = 0, y = 0, m = 0;
        const int* A0 = sblk;
        const int* A1 = sblk + kMaxStagedBlocks;
        while (x < cnt[0] || y < cnt[1]) {
          const int vx = x < cnt[0] ? A0[x] : 0x7FFFFFFF;
          const int vy = y < cnt[1] ? A1[y] : 0x7FFFFFFF;
          const int v = min(vx, vy);
          int bits = 0;
          if (vx == v) { bits |= 1; ++x; }
          if (vy == v) { bits |= 2; ++y; }
          if (v <= last || v < 0 || v >= (1 << 28)) bits = 3 << 2;  // not ascending / out of range: flagged
          else last = v;
          un[m++] = (v & 0x0FFFFFFF) | (bits << 28);
        }
        total = m;
      }
      total = __shfl_sync(0xFFFFFFFFu, total, 0);
      __syncwarp();
    } else {
      int x = 0, y = 0, m = 0;
      while (x < cnt[0] || y < cnt[1]) {
        const int vx = x < cnt[0] ? __ldg(J[0] + x) : 0x7FFFFFFF;
        const int vy = y < cnt[1] ? __ldg(J[1] + y) : 0x7FFFFFFF;
        if (vx <= vy) ++x;
        if (vy <= vx) ++y;
        ++m;
      }
      total = m;
      last = -1;
    }
  }
  __device__ bool done() const { return pos >= total; }
  __device__ void next_block(int& v, int& bits) {
    if (staged) {
      const int e = un[pos];
      v = e & 0x0FFFFFFF;
      bits = (e >> 28) & 0xF;
      if (bits & 12) bits = -1;
    } else {
      const int vx = p[0] < cnt[0] ? __ldg(J[0] + p[0]) : 0x7FFFFFFF;
      const int vy = p[1] < cnt[1] ? __ldg(J[1] + p[1]) : 0x7FFFFFFF;
      v = min(vx, vy);
      bits = 0;
      if (vx == v) { bits |= 1; ++p[0]; }
      if (vy == v) { bits |= 2; ++p[1]; }
      if (v <= last) bits = -1;
      else last = v;
    }
    ++pos;
  }
  // Lane 0: the next tile (two union entries).
  __device__ void emit(int n, TileDesc& d, int* err) {
    int v0 = 0, b0 = 0, v1 = 0, b1 = 0;
    next_block(v0, b0);
    if (!done()) next_block(v1, b1);
    else { v1 = v0; b1 = 0; }  // odd tail: reload a valid block, fully masked
    int vs[2] = {v0, v1}, bs[2] = {b0, b1};
    for (int s = 0; s < 2; ++s) {
      if (bs[s] < 0) { bs[s] = 0; set_error(err, kErrIndex); }
      for (int h = 0; h < 2; ++h)
        if ((bs[s] >> h & 1) && (vs[s] < 0 || vs[s] > u[h])) { bs[s] &= ~(1 << h); set_error(err, kErrIndex); }
      if (vs[s] < 0 || 64 * vs[s] >= n) { vs[s] = 0; bs[s] = 0; }
    }
    d.kind = kTileRange;
    d.rule = 0;
    for (int s = 0; s < 2; ++s) {
      d.seg[s] = 64 * vs[s];
      for (int w = 0; w < 2; ++w) {
        const uint32_t m = keys_below(64 * vs[s] + 32 * w, n);
        d.mask[0][2 * s + w] = (bs[s] & 1) ? m : 0u;
        d.mask[1][2 * s + w] = (bs[s] & 2) ? m : 0u;
      }
    }
  }
};

// ------------------------------------------------------------------ Vertical-Slash tiles
// Physical set of row i in query block [a, e] (MInference page §2.1 and §4.1):
// keys covered by some slash tile [a-δ, e-δ] (δ in D), plus the vertical
// columns C, restricted to j <= i.  For a full block, key j is covered iff bit
// n-1-a+j of the dilated coverage map is set, so a tile's mask is a 128-bit
// window of that map.  Aligned 128-key windows that some slash tile touches
// become range tiles whose masks include the verticals in them; verticals in
// the other windows are gathered into column tiles.

// Any bit set in [lo, hi] (hi - lo < 160) of an nbits map: every word loaded
// up front, so the loads overlap instead of chaining.
__device__ __forceinline__ bool bits_any5(const uint32_t* bits, int nbits, int lo, int hi) {
  lo = lo < 0 ? 0 : lo;
  hi = hi > nbits - 1 ? nbits - 1 : hi;
  if (lo > hi) return false;
  const int w0 = lo >> 5, w1 = hi >> 5;
  uint32_t x[6];
#pragma unroll
  for (int q = 0; q < 6; ++q) x[q] = (w0 + q <= w1) ? __ldg(bits + w0 + q) : 0u;
  x[0] &= 0xFFFFFFFFu << (lo & 31);
  uint32_t acc = 0u;
#pragma unroll
  for (int q = 0; q < 6; ++q) {
    uint32_t v = x[q];
    if (w0 + q == w1) v &= 0xFFFFFFFFu >> (31 - (hi & 31));
    if (w0 + q <= w1) acc |= v;
  }
  return acc != 0u;
}

struct VSIter {
  const uint32_t* dbits;
  const uint32_t* cbits;
  const uint32_t* cover;
  int cw;  // cover words
  int n, M, hi_key;
  int a[2], e[2], L[2], ex[2];
  int grp;                // first window of the current 32-window group
  uint32_t smask, cmask;  // group windows with slash coverage / with only columns
  int staged;             // columns waiting in the staging list
  __device__ void init(const Unit& U, const Item& it, const AttnArgs& A) {
    n = A.n;
    dbits = A.vs_dbits + (int64_t)U.slot[0] * A.vs_words;
    cbits = A.vs_cbits + (int64_t)U.slot[0] * A.vs_words;
    cover = A.vs_cover + (int64_t)U.slot[0] * A.vs_cover_words;
    cw = A.vs_cover_words;
    hi_key = min(it.a0 + 127, n - 1);
    M = hi_key / 128 + 1;
    for (int h = 0; h < 2; ++h) {
      a[h] = it.row0[h];
      e[h] = it.e[h];
      ex[h] = it.exists[h];
      L[h] = e[h] - a[h] + 1;
    }
    grp = -32;
    smask = cmask = 0u;
    staged = 0;
  }
  // Keys of window w covered by a slash tile of half h?
  __device__ bool half_has_slash(int h, int w) const {
    if (!ex[h]) return false;
    const int j0 = 128 * w;
    const int jhi = min(j0 + 127, e[h]);
    if (j0 > jhi) return false;
    if (L[h] == 64) return bits_any5(cover, 32 * cw, n - 1 - a[h] + j0, n - 1 - a[h] + jhi);
    return bits_any(dbits, n, a[h] - jhi, a[h] - j0 + L[h] - 1);
  }
  __device__ void load_group(int lane) {
    grp += 32;
    const int w = grp + lane;
    bool s = false, c = false;
    if (w < M) {
      s = half_has_slash(0, w) | half_has_slash(1, w);
      c = !s && bits_any5(cbits, n, 128 * w, min(128 * w + 127, hi_key));
    }
    smask = __ballot_sync(0xFFFFFFFFu, s);
    cmask = __ballot_sync(0xFFFFFFFFu, c);
  }
  __device__ void range_masks(int w, int lane, TileDesc& d) const {
    const int j0 = 128 * w;
    for (int h = 0; h < 2; ++h) {
      if (ex[h] && L[h] != 64) {  // partial last block: test each key (whole warp)
        for (int q = 0; q < 4; ++q) {
          const int j = j0 + 32 * q + lane;
          const bool ok = j <= e[h] && (bit_at(cbits, j) || bits_any(dbits, n, a[h] - j, a[h] - j + L[h] - 1));
          const uint32_t b = __ballot_sync(0xFFFFFFFFu, ok);
          if (lane == 0) d.mask[h][q] = b;
        }
      } else if ((lane >> 2) == h) {  // lanes 4h .. 4h+3: one mask word each
        const int q = lane & 3;
        const int base = j0 + 32 * q;
        uint32_t m = 0u;
        if (ex[h] && base <= e[h]) {
          m = bits_window32(cover, cw, n - 1 - a[h] + base) | __ldg(cbits + (base >> 5));
          m &= keys_below(base, e[h] + 1);
        }
        d.mask[h][q] = m;
      }
    }
    if (lane == 0) { d.seg[0] = j0; d.seg[1] = j0 + 64; d.kind = kTileRange; d.rule = 0; }
  }
  __device__ void gather_tile(int lane, int* stage, TileDesc& d) {
    const int take = staged < 128 ? staged : 128;
    for (int k = lane; k < 128; k += 32) d.gidx[k] = k < take ? stage[k] : -1;
    __syncwarp();
    for (int h = 0; h < 2; ++h)
      for (int q = 0; q < 4; ++q) {
        const int g = d.gidx[32 * q + lane];
        const bool ok = ex[h] && g >= 0 && g <= e[h];
        const uint32_t b = __ballot_sync(0xFFFFFFFFu, ok);
        if (lane == 0) d.mask[h][q] = b;
      }
    // shift the rest of the staging list down (rest < take, so the ranges do not overlap)
    const int rest = staged - take;
    for (int k = lane; k < rest; k += 32) stage[k] = stage[take + k];
    __syncwarp();
    staged = rest;
    if (lane == 0) { d.kind = kTileGather; d.rule = 0; d.seg[0] = 0; d.seg[1] = 0; }
  }
  // Produce the next tile into d (whole warp); false when the item has no more tiles.
  __device__ bool emit(int lane, int* stage, TileDesc& d) {
    for (;;) {
      if (staged >= 128) { gather_tile(lane, stage, d); return true; }
      if ((smask | cmask) == 0u) {
        if (grp + 32 >= M) {
          if (staged > 0) { gather_tile(lane, stage, d); return true; }
          return false;
        }
        load_group(lane);
        continue;
      }
      const int b = __ffs(smask | cmask) - 1;
      const bool is_slash = (smask >> b) & 1u;
      smask &= ~(1u << b);
      cmask &= ~(1u << b);
      const int w = grp + b;
      if (is_slash) { range_masks(w, lane, d); return true; }
      // stage this window's columns (ascending)
      const int j0 = 128 * w;
      for (int q = 0; q < 4; ++q) {
        const int j = j0 + 32 * q + lane;
        const bool ok = j <= hi_key && bit_at(cbits, j);
        const uint32_t bb = __ballot_sync(0xFFFFFFFFu, ok);
        if (ok) stage[staged + __popc(bb & ((1u << lane) - 1u))] = j;
        staged += __popc(bb);
      }
      __syncwarp();
    }
  }
};

// ------------------------------------------------------------------ kernel
template <int D, bool kCount>
__global__ void __launch_bounds__(kThreads, 1)
    sparse_attn_kernel(const __grid_constant__ CUtensorMap tk, const __grid_constant__ CUtensorMap tv,
                       const AttnArgs A, const __grid_constant__ UnitTable UT) {
  using Ly = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Ly::kBars);
  TileDesc* descs = reinterpret_cast<TileDesc*>(sm + Ly::kDesc);
  int* stage = reinterpret_cast<int*>(sm + Ly::kStage);
  int* sblk = reinterpret_cast<int*>(sm + Ly::kBlk);
  float* xchg = reinterpret_cast<float*>(sm + Ly::kXchg);
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(sm + Ly::kMisc);  // [0] tmem, [2] abort

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item_id = blockIdx.x;
  const int t = A.T - 1 - item_id / A.n_units;
  const Unit& U = UT.u[item_id % A.n_units];
  const int n = A.n;
  const Item it = make_item(U, t, n);

  if (warp == 0) {
    tmem_alloc(const_cast<uint32_t*>(&misc[0]), kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 32 * kMmaWarp) {
    mbar_init(&bars[kBarQ], kSoftWarps);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars[kBarKFull + s], 1);
      mbar_init(&bars[kBarKEmpty + s], 1);
      mbar_init(&bars[kBarVFull + s], 1);
      mbar_init(&bars[kBarVEmpty + s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&bars[kBarSFull + s], 1);
      mbar_init(&bars[kBarSEmpty + s], kSoftWarps);
    }
    mbar_init(&bars[kBarPFull], kSoftWarps);
    mbar_init(&bars[kBarPEmpty], 1);
    for (int s = 0; s < kDescSlots; ++s) {
      mbar_init(&bars[kBarDFull + s], 1);
      mbar_init(&bars[kBarDEmpty + s], kDescReaders);
    }
    for (int s = 0; s < 4; ++s) mbar_init(&bars[kBarX + s], 64);
    misc[2] = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];

  uint8_t* sK = sm + Ly::kK;
  uint8_t* sV = sm + Ly::kV;
  auto desc_full = [&](int j) { return mbar_wait(&bars[kBarDFull + j % kDescSlots], (j / kDescSlots) & 1); };
  auto desc_release = [&](int j) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[kBarDEmpty + j % kDescSlots]);
  };

  if (warp == kPlannerWarp) {
    // ------------------------------------------------------------ planner
    AshapeIter ai;
    BlockIter bi;
    VSIter vi;
    int T = 0;
    if (U.pattern == kUnitAshape) { ai.init(U, it, n); T = ai.count(); }
    else if (U.pattern == kUnitBlock) bi.init(U, it, A, lane, sblk);
    else vi.init(U, it, A);
    bool ok = true;
    for (int j = 0;; ++j) {
      if (misc[2]) { ok = false; break; }
      const int slot = j % kDescSlots;
      if (!mbar_wait(&bars[kBarDEmpty + slot], ((j / kDescSlots) & 1) ^ 1)) { ok = false; break; }
      TileDesc& d = descs[slot];
      bool more;
      if (U.pattern == kUnitVS) {
        more = vi.emit(lane, stage, d);
      } else if (U.pattern == kUnitAshape) {
        more = j < T;
        if (more && lane == 0) ai.emit(j, n, d);
      } else {
        more = !bi.done();  // the cursor advances in lane 0 only: its answer is the warp's
        more = __shfl_sync(0xFFFFFFFFu, more, 0);
        if (more && lane == 0) bi.emit(n, d, A.err);
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
      tma_prefetch_desc(&tk);
      tma_prefetch_desc(&tv);
    }
    auto load_kv = [&](int j, bool is_v) -> bool {
      const int st = j % kStages;
      const uint32_t ph = ((j / kStages) & 1) ^ 1;
      uint64_t* empty = &bars[(is_v ? kBarVEmpty : kBarKEmpty) + st];
      uint64_t* full = &bars[(is_v ? kBarVFull : kBarKFull) + st];
      if (!mbar_wait(empty, ph)) return false;
      const TileDesc& d = descs[j % kDescSlots];
      uint8_t* dst = (is_v ? sV : sK) + st * Ly::kTile;
      if (d.kind == kTileRange) {
        if (lane == 0) {
          const CUtensorMap* map = is_v ? &tv : &tk;
          mbar_arrive_expect_tx(full, Ly::kTile);
          for (int s = 0; s < 2; ++s)
            for (int c = 0; c < D / 64; ++c) tma_load_3d(dst + c * 16384 + s * 8192, map, full, 64 * c, d.seg[s], U.kvh);
        }
      } else {
        // gather single key rows (16-byte cp.async) into the swizzled layout
        constexpr int kChunks16 = D / 8;
        const uint8_t* gbase = reinterpret_cast<const uint8_t*>(is_v ? A.v : A.k) + (int64_t)U.kvh * n * D * 2;
        for (int idx = lane; idx < 128 * kChunks16; idx += 32) {
          const int r = idx / kChunks16, c16 = idx % kChunks16;
          int key = d.gidx[r];
          key = key < 0 ? 0 : key;  // empty columns reload key 0 (finite data, masked)
          cp_async16(dst + (c16 >> 3) * 16384 + sw128_offset(r, c16 & 7), gbase + ((int64_t)key * D + 8 * c16) * 2);
        }
        cp_async_wait_all();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(full);
      }
      return true;
    };
    // K runs one tile ahead of V; a descriptor is released once its V is issued
    bool ok = true;
    int j = 0;
    for (;; ++j) {
      if (misc[2]) { ok = false; break; }
      if (!desc_full(j)) { ok = false; break; }
      const bool end = descs[j % kDescSlots].kind == kTileEnd;
      if (!end && !load_kv(j, false)) { ok = false; break; }
      if (j > 0) {
        if (!load_kv(j - 1, true)) { ok = false; break; }
        desc_release(j - 1);
      }
      if (end) { desc_release(j); break; }
    }
    if (!ok) { misc[2] = 1; set_error(A.err, kErrTimeout); }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    bool ok = mbar_wait(&bars[kBarQ], 0);
    constexpr uint32_t id_qk = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t id_pv = idesc_bf16_f32(128, D, false, true);
    auto pv = [&](int j) -> bool {
      const int st = j % kStages;
      if (!mbar_wait(&bars[kBarPFull], j & 1)) return false;
      if (!mbar_wait(&bars[kBarVFull + st], (j / kStages) & 1)) return false;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t v0 = smem_u32(sV + st * Ly::kTile);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_bf16_ts(tmem + kColO, tmem + kColP + 8 * kk, sdesc_sw128(v0 + kk * 2048, 16384, 1024), id_pv,
                      (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit(&bars[kBarVEmpty + st]);
        mma_commit(&bars[kBarPEmpty]);
      }
      __syncwarp();
      return true;
    };
    if (ok) tc_fence_after();
    int j = 0;
    for (; ok; ++j) {
      if (misc[2]) { ok = false; break; }
      if (!desc_full(j)) { ok = false; break; }
      const bool end = descs[j % kDescSlots].kind == kTileEnd;
      desc_release(j);
      if (end) break;
      const int st = j % kStages, sb = j & 1;
      ok = mbar_wait(&bars[kBarKFull + st], (j / kStages) & 1) &&
           mbar_wait(&bars[kBarSEmpty + sb], ((j >> 1) & 1) ^ 1);
      if (!ok) break;
      tc_fence_after();
      if (lane == 0) {
        const uint32_t k0 = smem_u32(sK + st * Ly::kTile);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          mma_bf16_ts(tmem + kColS + 128 * sb, tmem + kColQ + 8 * kk, sdesc_sw128(k0 + off, 16, 1024), id_qk,
                      kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars[kBarSFull + sb]);
        mma_commit(&bars[kBarKEmpty + st]);
      }
      __syncwarp();
      if (j > 0) ok = pv(j - 1);
    }
    if (ok && j > 0) ok = pv(j - 1);
    if (!ok) { misc[2] = 1; set_error(A.err, kErrTimeout); }
  } else {
    // ------------------------------------------------------------ softmax warps
    const int quarter = warp & 3;          // TMEM lanes 32*quarter ..
    const int ch = warp >> 2;              // key half of each tile (and O / Q column half)
    const int r = quarter * 32 + lane;     // tile row = TMEM lane
    const int h = r >> 6;
    const int i = it.row0[h] + (r & 63);
    const bool row_ok = i < n;
    const uint32_t lane_base = (uint32_t)(quarter * 32) << 16;
    const float c2 = A.scale_log2;
    const int g = U.sink, wnd = U.window;
    uint64_t* xbar = &bars[kBarX + quarter];  // warps quarter and quarter+4, one phase per exchange
    float m_used = -INFINITY, l = 0.f;
    unsigned long long count = 0;
    bool ok = true;

    // ---- Q row into TMEM (A operand of S = Q K^T): 32 columns of bf16 pairs per writer
    if (D == 128 || ch == 0) {
      const __nv_bfloat16* qrow = reinterpret_cast<const __nv_bfloat16*>(A.q) + ((int64_t)U.qh[h] * n + i) * D;
      const int e0 = D == 128 ? ch * 64 : 0;
      uint32_t qw[32];
#pragma unroll
      for (int x = 0; x < 8; ++x) {
        uint4 v4 = make_uint4(0, 0, 0, 0);
        if (row_ok) v4 = __ldg(reinterpret_cast<const uint4*>(qrow + e0) + x);
        qw[4 * x] = v4.x; qw[4 * x + 1] = v4.y; qw[4 * x + 2] = v4.z; qw[4 * x + 3] = v4.w;
      }
      tmem_st32(tmem + lane_base + kColQ + (D == 128 ? 32 * ch : 0), qw);
    }
    tmem_st_wait();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&bars[kBarQ]);

    int j = 0;
    for (;; ++j) {
      if (misc[2]) { ok = false; break; }
      // ---- tile descriptor -> validity word of this thread's 64 keys
      if (!desc_full(j)) { ok = false; break; }
      const TileDesc& d = descs[j % kDescSlots];
      if (d.kind == kTileEnd) { desc_release(j); break; }
      uint64_t vw = 0ull;
      if (row_ok) {
        const uint64_t m64 = ((uint64_t)d.mask[h][2 * ch + 1] << 32) | d.mask[h][2 * ch];
        if (d.kind == kTileRange) {
          const int base = d.seg[ch];
          vw = m64 & low_mask64(i - base + 1);  // causal: j <= i
          if (d.rule) {
            uint64_t keep = 0;
            if (d.rule & 1) keep |= low_mask64(g - base);             // j < g
            if (d.rule & 2) keep |= ~low_mask64(i - wnd + 1 - base);  // j > i - w
            vw &= keep;
          }
        } else {
          for (int k = 0; k < 64; ++k) {
            const int gj = d.gidx[64 * ch + k];
            if (((m64 >> k) & 1ull) && gj >= 0 && gj <= i) vw |= 1ull << k;
          }
        }
      }
      desc_release(j);
      if (kCount) count += __popcll(vw);

      // ---- S tile (this thread's 64 keys) from TMEM
      const int sb = j & 1;
      if (!mbar_wait(&bars[kBarSFull + sb], (j >> 1) & 1)) { ok = false; break; }
      tc_fence_after();
      float sv[64];
      {
        uint32_t u0[32], u1[32];
        tmem_ld32(tmem + lane_base + kColS + 128 * sb + 64 * ch, u0);
        tmem_ld32(tmem + lane_base + kColS + 128 * sb + 64 * ch + 32, u1);
        tmem_ld_wait();
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          sv[k] = __uint_as_float(u0[k]);
          sv[32 + k] = __uint_as_float(u1[k]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarSEmpty + sb]);

      // ---- mask, row max (tree), exchanged with the partner warp
      if (~vw) {
#pragma unroll
        for (int k = 0; k < 64; ++k) sv[k] = ((vw >> k) & 1ull) ? sv[k] : -INFINITY;
      }
      float mx[8];
#pragma unroll
      for (int x = 0; x < 8; ++x) mx[x] = fmaxf(sv[x], sv[x + 8]);
#pragma unroll
      for (int k = 16; k < 64; k += 8)
#pragma unroll
        for (int x = 0; x < 8; ++x) mx[x] = fmaxf(mx[x], sv[k + x]);
      float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])), fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      float* xc = xchg + (j & 1) * 256;
      xc[ch * 128 + r] = mt;
      mbar_arrive(xbar);
      if (!mbar_wait(xbar, j & 1)) { ok = false; break; }
      mt = fmaxf(mt, xc[(ch ^ 1) * 128 + r]);

      const float m_new = fmaxf(m_used, mt * c2);
      const bool need = m_new > m_used + kRescaleThreshold;
      const bool any = __any_sync(0xFFFFFFFFu, need);  // the partner warp sees the same rows
      float alpha = 1.f;
      if (any && m_new != -INFINITY) {
        alpha = (m_used == -INFINITY) ? 0.f : ex2(m_used - m_new);
        m_used = m_new;
      }
      const float mref = (m_used == -INFINITY) ? 0.f : m_used;
      float rs[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pk[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const float p0 = ex2(fmaf(sv[2 * k], c2, -mref));
        const float p1 = ex2(fmaf(sv[2 * k + 1], c2, -mref));
        rs[k & 3] += p0 + p1;
        pk[k] = pack_bf16x2(p0, p1);
      }
      l = l * alpha + ((rs[0] + rs[1]) + (rs[2] + rs[3]));

      // ---- PV(j-1) must be done before P is overwritten or O is rescaled
      if (j > 0 && !mbar_wait(&bars[kBarPEmpty], (j - 1) & 1)) { ok = false; break; }
      tc_fence_after();
      if (any && j > 0) {
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          uint32_t o[32];
          const uint32_t col = kColO + (D / 2) * ch + 32 * c;
          tmem_ld32(tmem + lane_base + col, o);
          tmem_ld_wait();
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * alpha);
          tmem_st32(tmem + lane_base + col, o);
        }
      }
      tmem_st32(tmem + lane_base + kColP + 32 * ch, pk);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[kBarPFull]);
    }
    if (!ok) { misc[2] = 1; set_error(A.err, kErrTimeout); }
    const int T = j;  // tiles processed

    // ---- epilogue: O / l, LSE (the pair adds its partial denominators)
    const int qh = U.qh[h];
    if (ok && T > 0) {
      if (!mbar_wait(&bars[kBarPEmpty], (T - 1) & 1)) { ok = false; misc[2] = 1; set_error(A.err, kErrTimeout); }
      tc_fence_after();
    }
    xchg[512 + ch * 128 + r] = l;
    mbar_arrive(xbar);
    if (!mbar_wait(xbar, T & 1)) { ok = false; misc[2] = 1; set_error(A.err, kErrTimeout); }
    l += xchg[512 + (ch ^ 1) * 128 + r];
    const float inv_l = l > 0.f ? 1.f / l : 0.f;
    __nv_bfloat16* orow = reinterpret_cast<__nv_bfloat16*>(A.o) + ((int64_t)qh * n + i) * D + (D / 2) * ch;
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
      uint32_t o[32];
      if (ok && T > 0) {
        tmem_ld32(tmem + lane_base + kColO + (D / 2) * ch + 32 * c, o);
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
        for (int x = 0; x < 4; ++x) dst[x] = make_uint4(pkd[4 * x], pkd[4 * x + 1], pkd[4 * x + 2], pkd[4 * x + 3]);
      }
    }
    if (row_ok && A.lse && ch == 0)
      A.lse[(int64_t)qh * n + i] = l > 0.f ? (m_used + __log2f(l)) * 0.69314718055994531f : -INFINITY;
    if (kCount && A.edges) {
      unsigned long long c = count;
      for (int o = 16; o; o >>= 1) c += __shfl_xor_sync(0xFFFFFFFFu, c, o);
      if (lane == 0 && c) atomicAdd(A.edges + qh, c);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool kCount>
msa_status launch_impl(const CUtensorMap& tk, const CUtensorMap& tv, const AttnArgs& a, const UnitTable& ut,
                       cudaStream_t stream) {
  auto kern = sparse_attn_kernel<D, kCount>;
  const int smem = Layout<D>::kAlloc;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return MSA_ERR_CUDA;
  const int64_t items = (int64_t)a.T * a.n_units;
  if (items <= 0) return MSA_OK;
  if (items > 0x7FFFFFFF) return MSA_ERR_UNSUPPORTED;
  kern<<<(unsigned)items, kThreads, smem, stream>>>(tk, tv, a, ut);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

}  // namespace

msa_status launch_attention(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const AttnArgs& args, const Unit* units, int n_units, cudaStream_t stream) {
  (void)tq;  // Q rows are read by the softmax warps straight into TMEM
  for (int base = 0; base < n_units; base += kMaxUnits) {
    UnitTable ut;
    const int cnt = n_units - base < kMaxUnits ? n_units - base : kMaxUnits;
    for (int x = 0; x < cnt; ++x) ut.u[x] = units[base + x];
    AttnArgs a = args;
    a.n_units = cnt;
    msa_status st;
    const bool count = args.edges != nullptr;
    if (args.d == 128)
      st = count ? launch_impl<128, true>(tk, tv, a, ut, stream) : launch_impl<128, false>(tk, tv, a, ut, stream);
    else
      st = count ? launch_impl<64, true>(tk, tv, a, ut, stream) : launch_impl<64, false>(tk, tv, a, ut, stream);
    if (st != MSA_OK) return st;
  }
  return MSA_OK;
}

}  // namespace msa
