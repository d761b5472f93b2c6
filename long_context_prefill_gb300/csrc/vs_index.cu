// Online Vertical-Slash index (MInference page §2.1, §3.1 and §6.2; the
// MInference blog §2.3.2, Vertical-Slash steps 1-3, and §2.3.3 for the sort
// orders and the per-block form).
//
// For each Vertical-Slash head, with R = the last L = min(last_q, n) query
// rows and scores s_ij = scale * q_i.k_j:
//   Ã_ij = exp(s_ij - lse_i) for j <= i, lse_i = log Σ_{j<=i} exp(s_ij)
//   c_j  = Σ_{i in R} Ã_ij                 (vertical score)
//   r_δ  = Σ_{i in R, i >= δ} Ã_{i,i-δ}    (slash score)
//   C = top-v of c, D = top-s of r, ties to the lower index.
//
// Kernels (all on one stream, no host synchronisation):
//   proxy_stats   pass 1, tcgen05 S = Q_R K^T over a key chunk; thread = row;
//                 online (max, sum) per row -> partials
//   proxy_lse     combine the partials into lse per row
//   proxy_scores  pass 2, tcgen05 S^T = K Q_R^T; thread = key; Ã for every
//                 (row, key); c_j summed in registers; slash sums collected
//                 along diagonals with warp shuffles into per-key-block bins
//   slash_finalize  adds each diagonal's bins in a fixed order -> r
//   topk_select   radix select (threshold), then an index-ordered compaction
//                 that writes the sorted lists and the bitmaps
// K is streamed once per pass per group of query heads sharing a KV head (at
// 128K the second pass reads it from DRAM again: K of all groups exceeds L2).
#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <math.h>
#include <string.h>

#include <vector>

#include "internal.h"
#include "ptx.cuh"

namespace msa {

namespace {

constexpr int kPackMaxHeads = 8;
constexpr int kRows = 256;  // query rows per pack (Q tile in shared memory)
// Warps 0..E-1 epilogue, E producer, E+1 MMA.  The scores pass with at most
// 64 rows per head runs 16 epilogue warps (one per 32 keys x 64 columns), the
// other passes 8 (one per 32 keys x 128 columns).
template <int MODE, int LP>
struct ProxyWarps {
  static constexpr int kEpi = (MODE == 2 && LP <= 64) ? 16 : 8;
  static constexpr int kProd = kEpi, kMma = kEpi + 1;
  static constexpr int kThreads = 32 * (kEpi + 2);
  static constexpr int kCols = 256 / (kEpi / 4);  // TMEM columns (proxy rows) per epilogue warp
};
constexpr int kKStages = 3;

// The Vertical-Slash heads of one KV group (at most kPackMaxHeads of them),
// the same for every sequence: a pack is one group pack of one sequence.
struct GroupPack {
  int32_t g;                    // kv head
  int32_t nh;                   // heads in this pack
  int32_t x[kPackMaxHeads];     // slot of each head within its sequence
  int32_t h[kPackMaxHeads];     // query head
};
constexpr int kMaxGroupPacks = 64;
struct PackTable {
  int32_t n_gp, pad;
  GroupPack p[kMaxGroupPacks];
};

struct ProxyArgs {
  const void* q;        // bf16 rows (row = Hq * tok0 + h * n + i)
  int32_t d, Lp;        // proxy rows per head L = min(last_q, n), padded to Lp
  int32_t last_q, Hq, Hkv, n_vs;  // n_vs: Vertical-Slash slots per sequence
  float c2;             // scale * log2(e)
  float2* part;         // [CTAs of the launch, 256] (max, sum) in log2 units (pass 1 out)
  float* lse2;          // [packs of the launch, 256] (pass 2 in)
  float* colsum;        // sequence-major, n per slot: log2 c_j
  float* rpart;         // sequence-major, (4 ntiles + LB) x (LB + 1) x 32 per slot: log2 partial slash sums
  int32_t mode;         // proxy convention bits (MSA_PROXY_*)
  int* err;
};

__device__ __forceinline__ void set_err(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

__device__ __forceinline__ float ex2f(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int D>
struct PLayout {
  static constexpr int kQChunk = kRows * 128;         // 256 rows x 64 columns
  static constexpr int kQ = 0;                        // D/64 chunks
  static constexpr int kKTile = 128 * D * 2;
  static constexpr int kK = kQ + (D / 64) * kQChunk;
  static constexpr int kLse = kK + kKStages * kKTile;  // 256 floats
  static constexpr int kBars = kLse + kRows * 4;
  static constexpr int kNumBars = 2 * kKStages + 4;
  static constexpr int kMisc = kBars + kNumBars * 8;
  static constexpr int kTotal = kMisc + 64;
  static constexpr int kAlloc = kTotal + 1024;
};

// Load the pack's proxy rows into the 128-byte-swizzled Q tile:
// row r = head * Lp + t holds q at position n - L + t (zero if t >= L).
template <int D>
__device__ void load_rows(uint8_t* sQ, const ProxyArgs& A, const GroupPack& P, const SeqInfo& S, int L) {
  constexpr int kC16 = D / 8;
  const int n = S.n;
  for (int idx = threadIdx.x; idx < kRows * kC16; idx += blockDim.x) {
    const int r = idx / kC16, c16 = idx % kC16;
    const int hh = r / A.Lp, t = r % A.Lp;
    uint4 val = make_uint4(0, 0, 0, 0);
    if (hh < P.nh && t < L) {
      const int64_t row = (int64_t)A.Hq * S.tok0 + (int64_t)P.h[hh] * n + (n - L + t);
      val = __ldg(reinterpret_cast<const uint4*>(reinterpret_cast<const uint8_t*>(A.q) + row * D * 2) + c16);
    }
    *reinterpret_cast<uint4*>(sQ + (c16 >> 3) * PLayout<D>::kQChunk + sw128_offset(r, c16 & 7)) = val;
  }
  fence_proxy_async_smem();
}

// MODE 1: statistics pass (S = Q K^T, lane = row).  MODE 2: scores pass
// (S^T = K Q^T, lane = key).  LP: rows per head (32, 64 or 128).
template <int D, int MODE, int LP>
__global__ void __launch_bounds__(ProxyWarps<MODE, LP>::kThreads, 1)
    proxy_kernel(const __grid_constant__ CUtensorMap tk, const ProxyArgs A, const __grid_constant__ PackTable PT,
                 const __grid_constant__ SeqTable ST) {
  using Ly = PLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* sQ = sm + Ly::kQ;
  uint8_t* sK = sm + Ly::kK;
  float* sLse = reinterpret_cast<float*>(sm + Ly::kLse);
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Ly::kBars);
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(sm + Ly::kMisc);
  uint64_t* kfull = bars;
  uint64_t* kempty = bars + kKStages;
  uint64_t* sfull = bars + 2 * kKStages;
  uint64_t* sempty = bars + 2 * kKStages + 2;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // sequence, group pack and key chunk of this CTA
  const int ts = seq_search(ST.count, [&](int x) { return ST.s[x].chunk0; }, (int64_t)blockIdx.x);
  const SeqInfo& SI = ST.s[ts];
  const int local = (int)blockIdx.x - SI.chunk0;
  const int gp = local / SI.chunks, chunk = local % SI.chunks;
  const GroupPack& P = PT.p[gp];
  const int pack_id = ts * PT.n_gp + gp;
  const int n = SI.n;
  const int L = min(A.last_q, n);
  const int ntiles = n_tiles(n);
  const int tiles_per = (ntiles + SI.chunks - 1) / SI.chunks;
  const int tile0 = chunk * tiles_per;
  const int tile1 = min(ntiles, tile0 + tiles_per);
  const int T = max(0, tile1 - tile0);
  const int nrows = P.nh * A.Lp;              // rows holding data (<= 256)
  const int nrt = (nrows + 127) / 128;        // MODE 1: row tiles

  if (warp == 0) {
    tmem_alloc(const_cast<uint32_t*>(&misc[0]), 512);
    tmem_relinquish();
  }
  using PW = ProxyWarps<MODE, LP>;
  if (threadIdx.x == 32 * PW::kMma) {
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&kfull[s], 1);
      mbar_init(&kempty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&sfull[s], 1);
      mbar_init(&sempty[s], PW::kEpi);
    }
    misc[2] = 0;
    fence_mbar_init();
  }
  load_rows<D>(sQ, A, P, SI, L);
  if (MODE == 2)
    for (int r = threadIdx.x; r < kRows; r += blockDim.x) sLse[r] = A.lse2[(int64_t)pack_id * kRows + r];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];

  if (warp == PW::kProd) {
    const int32_t krow0 = A.Hkv * SI.tok0 + P.g * n;  // row of key 0 of this group in the [rows, d] view of k
    if (lane == 0 && T > 0) {
      tma_prefetch_desc(&tk);
      bool ok = true;
      for (int j = 0; j < T && ok; ++j) {
        const int st = j % kKStages;
        if (!mbar_wait(&kempty[st], ((j / kKStages) & 1) ^ 1)) { ok = false; break; }
        const int k0 = (tile0 + j) * 128;
        mbar_arrive_expect_tx(&kfull[st], Ly::kKTile);
        uint8_t* dst = sK + st * Ly::kKTile;
        for (int s = 0; s < 2; ++s)
          for (int c = 0; c < D / 64; ++c)
            tma_load_3d(dst + c * 16384 + s * 8192, &tk, &kfull[st], 64 * c, krow0 + k0 + 64 * s, 0);
      }
      if (!ok) { misc[2] = 1; set_err(A.err, kErrTimeout); }
    }
    __syncwarp();
  } else if (warp == PW::kMma) {
    if (lane == 0 && T > 0) {
      bool ok = true;
      const uint32_t q0 = smem_u32(sQ);
      for (int j = 0; j < T && ok; ++j) {
        const int st = j % kKStages, sb = j & 1;
        if (!mbar_wait(&kfull[st], (j / kKStages) & 1) || !mbar_wait(&sempty[sb], ((j >> 1) & 1) ^ 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t k0 = smem_u32(sK + st * Ly::kKTile);
        if (MODE == 1) {
          constexpr uint32_t id = idesc_bf16_f32(128, 128, false, false);
          for (int rt = 0; rt < nrt; ++rt)
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
              const uint32_t qoff = (kk >> 2) * Ly::kQChunk + rt * 16384 + (kk & 3) * 32;
              mma_bf16_ss(tmem + sb * 256 + rt * 128, sdesc_sw128(q0 + qoff, 16, 1024), sdesc_sw128(k0 + off, 16, 1024),
                          id, kk > 0 ? 1u : 0u);
            }
        } else {
          const uint32_t id = idesc_bf16_f32(128, nrows, false, false);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
            const uint32_t qoff = (kk >> 2) * Ly::kQChunk + (kk & 3) * 32;
            mma_bf16_ss(tmem + sb * 256, sdesc_sw128(k0 + off, 16, 1024), sdesc_sw128(q0 + qoff, 16, 1024), id,
                        kk > 0 ? 1u : 0u);
          }
        }
        mma_commit(&sfull[sb]);
        mma_commit(&kempty[st]);
      }
      if (!ok) { misc[2] = 1; set_err(A.err, kErrTimeout); }
    }
    __syncwarp();
  } else {
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const float c2 = A.c2;
    bool ok = true;
    if (MODE == 1) {
      // ------------------------------------------------ per-row online (max, sum)
      const int rt = warp >> 2;
      const int r = rt * 128 + (warp & 3) * 32 + lane;
      const int t = r % A.Lp;
      const bool row_ok = r < nrows && t < L;
      const int i = n - L + t;  // query position of this row
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < T; ++j) {
        if (misc[2]) { ok = false; break; }
        const int sb = j & 1;
        if (!mbar_wait(&sfull[sb], (j >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        if (rt < nrt) {
          float sv[128];
          uint32_t* u = reinterpret_cast<uint32_t*>(sv);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            tmem_ld32(tmem + lane_base + sb * 256 + rt * 128 + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(u + 32 * c));
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sempty[sb]);
          const int k0 = (tile0 + j) * 128;
          const int lim = row_ok ? min(i, n - 1) - k0 + 1 : 0;  // keys k0 + k valid for k < lim
          if (lim < 128) {
#pragma unroll
            for (int k = 0; k < 128; ++k) sv[k] = k < lim ? sv[k] : -INFINITY;
          }
          float mt = sv[0];
#pragma unroll
          for (int k = 1; k < 128; ++k) mt = fmaxf(mt, sv[k]);
          const float mn = fmaxf(m, mt * c2);
          if (mn != -INFINITY) {
            float acc = 0.f;
#pragma unroll
            for (int k = 0; k < 128; ++k) acc += ex2f(fmaf(sv[k], c2, -mn));
            l = l * ex2f(m - mn) + acc;
            m = mn;
          }
        } else {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sempty[sb]);
        }
      }
      if (rt * 128 < kRows)
        A.part[(int64_t)blockIdx.x * kRows + r] = make_float2(row_ok ? m : -INFINITY, row_ok ? l : 0.f);
    } else {
      // ------------------------------------------------ per-key Ã, column sums, diagonal bins
      // Sums are kept as (max, sum of 2^(x - max)) pairs over log2
      // probabilities x = log2 Ã, so scores far below fp32's range still
      // rank correctly; outputs are log2 of the sums.
      constexpr int HPH = PW::kCols / LP;  // heads per epilogue warp
      constexpr int LB = LP / 32;     // 32-row chunks per head
      const int ch = warp >> 2;            // column group: rows kCols ch .. kCols (ch + 1) - 1
      float col_log[HPH];
      float bin_log[HPH][LB + 1];
      for (int j = 0; j < T; ++j) {
        if (misc[2]) { ok = false; break; }
        const int sb = j & 1;
        if (!mbar_wait(&sfull[sb], (j >> 1) & 1)) { ok = false; break; }
        tc_fence_after();
        const int kb0 = (tile0 + j) * 128 + (warp & 3) * 32;  // first key of this warp's block
        const int key = kb0 + lane;
#pragma unroll
        for (int x = 0; x < HPH; ++x) {
          const int hh = ch * HPH + x;
          if (hh >= P.nh) continue;  // warp-uniform
          float cm = -INFINITY, cs = 0.f;
          float bm[LB + 1], bsum[LB + 1];
#pragma unroll
          for (int m = 0; m <= LB; ++m) { bm[m] = -INFINITY; bsum[m] = 0.f; }
#pragma unroll
          for (int cc = 0; cc < LB; ++cc) {
            const int r0 = hh * LP + cc * 32;  // first row of this 32-row chunk
            uint32_t sraw[32];
            tmem_ld32(tmem + lane_base + sb * 256 + r0, sraw);
            tmem_ld_wait();
            float xv[32];
            float mx = -INFINITY;
            // every (row, key) of this chunk valid (warp-uniform): all 32 rows are
            // proxy rows and every key lies at or before the chunk's first row
            const bool chunk_valid = cc * 32 + 31 < L && kb0 + 31 <= n - L + cc * 32;
            if (chunk_valid) {
#pragma unroll
              for (int tp = 0; tp < 32; ++tp) {
                xv[tp] = fmaf(__uint_as_float(sraw[tp]), c2, -sLse[r0 + tp]);
                mx = fmaxf(mx, xv[tp]);
              }
            } else {
#pragma unroll
              for (int tp = 0; tp < 32; ++tp) {
                const int t = cc * 32 + tp;
                const bool valid = t < L && key <= n - L + t && key < n;
                xv[tp] = valid ? fmaf(__uint_as_float(sraw[tp]), c2, -sLse[r0 + tp]) : -INFINITY;
                mx = fmaxf(mx, xv[tp]);
              }
            }
            // column: running log-sum-exp over the head's rows
            const float nm = fmaxf(cm, mx);
            if (nm != -INFINITY) {
              float acc = 0.f;
#pragma unroll
              for (int tp = 0; tp < 32; ++tp) acc += ex2f(xv[tp] - nm);
              cs = cs * ex2f(cm - nm) + acc;
              cm = nm;
            }
            // diagonal: the slash through (row t, key) has y = key - t; lane
            // receives y = 32*(block - cc) + lane (hi) or one block lower (lo)
            float vsh[32];
            float hm = -INFINITY, lm = -INFINITY;
#pragma unroll
            for (int tp = 0; tp < 32; ++tp) {
              vsh[tp] = __shfl_sync(0xFFFFFFFFu, xv[tp], (lane + tp) & 31);
              if (lane + tp < 32) hm = fmaxf(hm, vsh[tp]);
              else lm = fmaxf(lm, vsh[tp]);
            }
            {
              const float a = fmaxf(bm[cc], hm);
              if (a != -INFINITY) { bsum[cc] *= ex2f(bm[cc] - a); bm[cc] = a; }
              const float b = fmaxf(bm[cc + 1], lm);
              if (b != -INFINITY) { bsum[cc + 1] *= ex2f(bm[cc + 1] - b); bm[cc + 1] = b; }
            }
            float hs = 0.f, ls = 0.f;
            if (chunk_valid) {  // every term finite, so is every bin maximum
#pragma unroll
              for (int tp = 0; tp < 32; ++tp) {
                const bool hi = lane + tp < 32;
                const float e = ex2f(vsh[tp] - (hi ? bm[cc] : bm[cc + 1]));
                if (hi) hs += e;
                else ls += e;
              }
            } else {
#pragma unroll
              for (int tp = 0; tp < 32; ++tp) {
                const bool hi = lane + tp < 32;
                const float e = vsh[tp] != -INFINITY ? ex2f(vsh[tp] - (hi ? bm[cc] : bm[cc + 1])) : 0.f;
                if (hi) hs += e;
                else ls += e;
              }
            }
            bsum[cc] += hs;
            bsum[cc + 1] += ls;
          }
          col_log[x] = (A.mode & MSA_PROXY_COL_MAX) ? cm : (cs > 0.f ? cm + __log2f(cs) : -INFINITY);
#pragma unroll
          for (int m = 0; m <= LB; ++m) bin_log[x][m] = bsum[m] > 0.f ? bm[m] + __log2f(bsum[m]) : -INFINITY;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&sempty[sb]);
        const int kb = kb0 >> 5;  // key block index
        const int nkb = 4 * n_tiles(n);
#pragma unroll
        for (int x = 0; x < HPH; ++x) {
          const int hh = ch * HPH + x;
          if (hh >= P.nh) continue;
          const int64_t slot = P.x[hh];
          if (key < n) A.colsum[(int64_t)A.n_vs * SI.tok0 + slot * n + key] = col_log[x];
          const int64_t rrow = (int64_t)A.n_vs * SI.kb0 + slot * (nkb + LB) + (kb + LB);
#pragma unroll
          for (int m = 0; m <= LB; ++m) A.rpart[((rrow - m) * (LB + 1) + m) * 32 + lane] = bin_log[x][m];
        }
      }
    }
    if (!ok) { misc[2] = 1; set_err(A.err, kErrTimeout); }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// lse2 per row = log2-domain log-sum-exp over the partials of the pack's CTAs.
__global__ void proxy_lse_kernel(const float2* part, int n_gp, const __grid_constant__ SeqTable ST, float* lse2) {
  const int pk = blockIdx.x, r = threadIdx.x;
  const SeqInfo& S = ST.s[pk / n_gp];
  const int64_t c0 = S.chunk0 + (int64_t)(pk % n_gp) * S.chunks;
  const int nchunks = S.chunks;
  float m = -INFINITY;
  for (int c = 0; c < nchunks; ++c) m = fmaxf(m, part[(c0 + c) * kRows + r].x);
  float l = 0.f;
  if (m != -INFINITY)
    for (int c = 0; c < nchunks; ++c) {
      const float2 v = part[(c0 + c) * kRows + r];
      if (v.x != -INFINITY) l += v.y * exp2f(v.x - m);
    }
  lse2[(int64_t)pk * kRows + r] = (l > 0.f) ? m + log2f(l) : INFINITY;  // +inf -> exp2(s - lse) = 0 for empty rows
}

// log2 r_δ = log-sum-exp over the bins (y = n - L - δ) of the key blocks that
// own them, m = 0..LB in order.
// One thread per offset d of a slot (slots of the launch along the grid's y
// dimension, n_vs per sequence).
__global__ void slash_finalize_kernel(const float* rpart, const __grid_constant__ SeqTable ST, int n_vs, int last_q,
                                      int LB, int mode, float* r) {
  const int slots = ST.count * n_vs;
  for (int sl = blockIdx.y; sl < slots; sl += gridDim.y) {
    const SeqInfo& S = ST.s[sl / n_vs];
    const int64_t x = sl % n_vs;
    const int n = S.n, L = min(last_q, n), nkb = 4 * n_tiles(n);
    const int64_t rbase = (int64_t)n_vs * S.kb0 + x * (nkb + LB);
    float* out = r + (int64_t)n_vs * S.tok0 + x * n;
    for (int d = blockIdx.x * blockDim.x + threadIdx.x; d < n; d += gridDim.x * blockDim.x) {
      const int y = n - L - d;
      const int beta = (y >= 0) ? (y >> 5) : -((31 - y) >> 5);  // floor(y / 32)
      const int ln = y - 32 * beta;
      const float* src = rpart + ((rbase + beta + LB) * (LB + 1)) * 32 + ln;
      float v[5];
      float mx = -INFINITY;
#pragma unroll
      for (int m = 0; m < 5; ++m) {
        if (m > LB) break;
        const int kb = beta + m;
        v[m] = (kb < 0 || kb >= nkb) ? -INFINITY : __ldg(src + m * 32);
        mx = fmaxf(mx, v[m]);
      }
      float s = 0.f;
      if (mx != -INFINITY) {
#pragma unroll
        for (int m = 0; m < 5; ++m) {
          if (m > LB) break;
          s += v[m] != -INFINITY ? exp2f(v[m] - mx) : 0.f;
        }
      }
      float lr = s > 0.f ? mx + log2f(s) : -INFINITY;
      if ((mode & MSA_PROXY_SLASH_MEAN) && lr != -INFINITY) lr -= log2f((float)min(L, n - d));  // legal pairs of offset d
      out[d] = lr;
    }
  }
}

// Order-preserving map from float to unsigned (larger float -> larger key).
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t b = __float_as_uint(f == 0.f ? 0.f : f);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// ------------------------------------------------------------------ top-k
constexpr int kTopkThreads = 512;
constexpr int kTopkCluster = 8;  // CTAs per score vector

struct TopkJob {
  const float* vals;
  int32_t* list;   // [cap]
  int32_t* cnt;
  uint32_t* bits;  // [words]
  int32_t k;
  int32_t descending;  // write the list in descending index order
};

// Both score vectors of every slot of the launch: vector 2*sl selects the
// verticals from the column sums, 2*sl+1 the slashes from the slash sums
// (launch slot sl = table entry * n_vs + head rank).
struct TopkArgs {
  const float* colsum;
  const float* slashsum;
  msa_vs_index out;
  int32_t vk, sk, n_vs, pad;
};

// The job of vector `vec`; n: the length of its sequence.
__device__ __forceinline__ TopkJob topk_job(const TopkArgs& a, const SeqTable& st, int vec, int& n) {
  const int sl = vec >> 1;
  const SeqInfo& S = st.s[sl / a.n_vs];
  const int64_t x = sl % a.n_vs;
  n = S.n;
  const int64_t slot = (int64_t)S.seq * a.n_vs + x;                     // slot of the output lists
  const int64_t vbase = (int64_t)a.n_vs * S.tok0 + x * n;              // score vectors
  const int64_t wbase = (int64_t)a.n_vs * S.word0 + x * n_words(n);    // bitmaps
  TopkJob J;
  if ((vec & 1) == 0) {
    J.vals = a.colsum + vbase;
    J.list = a.out.vertical + slot * a.out.v_cap;
    J.cnt = a.out.vertical_cnt + slot;
    J.bits = a.out.vertical_bits + wbase;
    J.k = a.vk;
    J.descending = 0;
  } else {
    J.vals = a.slashsum + vbase;
    J.list = a.out.slash + slot * a.out.s_cap;
    J.cnt = a.out.slash_cnt + slot;
    J.bits = a.out.slash_bits + wbase;
    J.k = a.sk;
    J.descending = 1;
  }
  return J;
}

// One cluster of kTopkCluster CTAs per score vector (cluster c: vector c, as
// in topk_job); CTA r owns words [r cw, (r+1) cw) of the n values, and warp
// w of a CTA a contiguous run of those words, so (CTA, warp, word, lane) is
// index order.  Every pass reads the values with coalesced loads.
//  1. the cluster's min and max order keys fix the bits all keys share;
//  2. radix select, 8 bits per pass from the highest differing bit down: each
//     CTA histograms its keys that match the prefix chosen so far (one
//     histogram per warp, summed), the cluster adds the CTAs' histograms
//     through distributed shared memory, and every CTA picks
//     the same digit.  When the chosen bin holds exactly the keys still needed,
//     every key at or above it is taken and the search stops early; otherwise
//     the k-th largest key T and the number `need` of keys equal to T to keep
//     come out;
//  3. each warp counts its keys above / equal to T with ballots; from the
//     counts of the warps and CTAs before it (index order) it knows where its
//     selected keys go, and writes the bitmap words and the sorted list (ties:
//     lower index first).
constexpr int kDigitBits = 8;
constexpr int kBins = 1 << kDigitBits;
constexpr int kTopkWarps = kTopkThreads / 32;
static_assert(kBins <= kTopkThreads && kBins % 32 == 0, "one bin per thread");

__global__ void __cluster_dims__(kTopkCluster, 1, 1) __launch_bounds__(kTopkThreads, 2)
    topk_kernel(const TopkArgs args, const __grid_constant__ SeqTable ST) {
  namespace cg = cooperative_groups;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  int n = 0;
  const TopkJob J = topk_job(args, ST, (int)(blockIdx.x / kTopkCluster), n);
  __shared__ int whist[kTopkWarps][kBins];  // per-warp histograms of the current pass
  __shared__ int hist[kBins];        // this CTA's histogram of the current pass (read cluster-wide)
  __shared__ int ghist[kBins];       // the cluster's histogram
  __shared__ uint32_t s_mm[2];       // this CTA's min / max key (read cluster-wide)
  __shared__ int s_cnt[2];           // this CTA's keys above / equal to T (read cluster-wide)
  __shared__ int wcnt[kTopkWarps][2];
  __shared__ uint32_t s_u[2];
  __shared__ int s_i[3];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int words = (n + 31) / 32;
  const int cw = (words + kTopkCluster - 1) / kTopkCluster;
  const int w0 = min(words, rank * cw), w1 = min(words, w0 + cw);
  const int x0 = 32 * w0, x1 = min(n, 32 * w1);
  const int k = J.k < n ? J.k : n;
  const bool all = k >= n, none = k <= 0;
  uint32_t T = 0;
  int need = k;
  if (!all && !none) {
    // ---- 1. common leading bits
    uint32_t mn = 0xFFFFFFFFu, mx = 0u;
    for (int x = x0 + tid; x < x1; x += kTopkThreads) {
      const uint32_t key = order_key(J.vals[x]);
      mn = min(mn, key);
      mx = max(mx, key);
    }
    mn = __reduce_min_sync(0xFFFFFFFFu, mn);
    mx = __reduce_max_sync(0xFFFFFFFFu, mx);
    if (lane == 0) { wcnt[warp][0] = (int)mn; wcnt[warp][1] = (int)mx; }
    __syncthreads();
    if (warp == 0) {
      uint32_t a = 0xFFFFFFFFu, b = 0u;
      if (lane < kTopkWarps) { a = (uint32_t)wcnt[lane][0]; b = (uint32_t)wcnt[lane][1]; }
      a = __reduce_min_sync(0xFFFFFFFFu, a);
      b = __reduce_max_sync(0xFFFFFFFFu, b);
      if (lane == 0) { s_mm[0] = a; s_mm[1] = b; }
    }
    cluster.sync();
    if (warp == 0) {
      uint32_t a = 0xFFFFFFFFu, b = 0u;
      if (lane < kTopkCluster) {
        const uint32_t* r = cluster.map_shared_rank(s_mm, lane);
        a = r[0];
        b = r[1];
      }
      a = __reduce_min_sync(0xFFFFFFFFu, a);
      b = __reduce_max_sync(0xFFFFFFFFu, b);
      if (lane == 0) { s_u[0] = a; s_u[1] = b; }
    }
    __syncthreads();
    const uint32_t gmin = s_u[0], gmax = s_u[1];
    if (gmin == gmax) {
      T = gmin;  // every key is equal: the first k by index
    } else {
      // ---- 2. radix select below the shared bits
      int lo = 32 - __clz(gmin ^ gmax);  // bits [0, lo) still open
      uint32_t pmask = lo == 32 ? 0u : ~((1u << lo) - 1u);
      uint32_t prefix = gmin & pmask;
      bool exact = false;
      while (lo > 0) {
        const int width = lo < kDigitBits ? lo : kDigitBits, sft = lo - width;
        const uint32_t dmask = (1u << width) - 1u;
        for (int b = lane; b < kBins; b += 32) whist[warp][b] = 0;
        __syncwarp();
        for (int x = x0 + tid; x < x1; x += kTopkThreads) {
          const uint32_t key = order_key(J.vals[x]);
          if ((key & pmask) == prefix) atomicAdd(&whist[warp][(key >> sft) & dmask], 1);
        }
        __syncthreads();
        if (tid < kBins) {
          int v = 0;
#pragma unroll
          for (int w = 0; w < kTopkWarps; ++w) v += whist[w][tid];
          hist[tid] = v;
        }
        cluster.sync();  // every CTA's histogram is complete
        if (tid < kBins) {
          int v = 0;
#pragma unroll
          for (int r = 0; r < kTopkCluster; ++r) v += cluster.map_shared_rank(hist, r)[tid];
          ghist[tid] = v;
        }
        __syncthreads();
        if (warp == 0) {
          // digit of the need-th largest: suffix sums, kBins / 32 bins per lane (higher lanes hold higher bins)
          constexpr int kPer = kBins / 32;
          int mine = 0;
          for (int b = 0; b < kPer; ++b) mine += ghist[kPer * lane + b];
          int suf = mine;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_down_sync(0xFFFFFFFFu, suf, o);
            if (lane + o < 32) suf += y;
          }
          const int excl = suf - mine;
          const unsigned who = __ballot_sync(0xFFFFFFFFu, excl < need && suf >= need);
          const int src = __ffs(who) - 1;
          if (lane == src) {
            int cum = excl, d = kPer * lane;
            for (int b = kPer - 1; b >= 0; --b) {
              const int c = ghist[kPer * lane + b];
              if (cum + c >= need) { d = kPer * lane + b; break; }
              cum += c;
            }
            s_i[0] = d;
            s_i[1] = cum;
            s_i[2] = ghist[d];
          }
        }
        cluster.sync();  // every CTA has read the histograms of this pass
        need -= s_i[1];
        prefix |= (uint32_t)s_i[0] << sft;
        pmask |= dmask << sft;
        lo = sft;
        if (s_i[2] == need && prefix != 0u) {  // the whole bin is taken: every key >= prefix
          exact = true;
          break;
        }
      }
      if (exact) {
        T = prefix - 1u;
        need = 0;
      } else {
        T = prefix;
      }
    }
  }
  // ---- 3. counts, then placement in index order (warp w: words [ww0, ww1))
  const int pw = (w1 - w0 + kTopkWarps - 1) / kTopkWarps;
  const int ww0 = min(w1, w0 + warp * pw), ww1 = min(w1, ww0 + pw);
  auto word_masks = [&](int wi, unsigned& gt, unsigned& eq) {
    const int x = 32 * wi + lane;
    bool g = false, e = false;
    if (x < n) {
      if (all) {
        g = true;
      } else if (!none) {
        const uint32_t key = order_key(J.vals[x]);
        g = key > T;
        e = key == T;
      }
    }
    gt = __ballot_sync(0xFFFFFFFFu, g);
    eq = __ballot_sync(0xFFFFFFFFu, e);
  };
  int cgt = 0, ceq = 0;
  for (int wi = ww0; wi < ww1; ++wi) {
    unsigned gt, eq;
    word_masks(wi, gt, eq);
    cgt += __popc(gt);
    ceq += __popc(eq);
  }
  if (lane == 0) { wcnt[warp][0] = cgt; wcnt[warp][1] = ceq; }
  __syncthreads();
  if (tid == 0) {
    int tg = 0, te = 0;
    for (int w = 0; w < kTopkWarps; ++w) { tg += wcnt[w][0]; te += wcnt[w][1]; }
    s_cnt[0] = tg;
    s_cnt[1] = te;
  }
  cluster.sync();
  int gt_before = 0, eq_before = 0, total_gt = 0, total_eq = 0;
  for (int r = 0; r < kTopkCluster; ++r) {
    const int* c = cluster.map_shared_rank(s_cnt, r);
    if (r < rank) { gt_before += c[0]; eq_before += c[1]; }
    total_gt += c[0];
    total_eq += c[1];
  }
  cluster.sync();  // the counts have been read: no CTA may exit before that
  for (int w = 0; w < warp; ++w) { gt_before += wcnt[w][0]; eq_before += wcnt[w][1]; }
  const unsigned lt = (1u << lane) - 1u;
  for (int wi = ww0; wi < ww1; ++wi) {
    unsigned gt, eq;
    word_masks(wi, gt, eq);
    // selected: every key above T, and the keys equal to T of rank < need
    const int eq_rank = eq_before + __popc(eq & lt);
    const bool take = ((gt >> lane) & 1u) || (((eq >> lane) & 1u) && eq_rank < need);
    const unsigned sel = __ballot_sync(0xFFFFFFFFu, take);
    if (take) {
      const int pos = gt_before + __popc(gt & lt) + min(eq_rank, need);
      const int outp = J.descending ? (k - 1 - pos) : pos;
      if (outp >= 0 && outp < k) J.list[outp] = 32 * wi + lane;
    }
    if (lane == 0) J.bits[wi] = sel;
    gt_before += __popc(gt);
    eq_before += __popc(eq);
  }
  if (rank == 0 && tid == 0) {
    const int total = total_gt + min(total_eq, need);
    *J.cnt = total < k ? total : k;
  }
}

// Dilated slash coverage: bit z = any offset of D in [n-1-z, n+62-z], z < n+63.
// One thread per output bit, words assembled with a warp ballot.
__global__ void slash_cover_kernel(const uint32_t* dbits, const __grid_constant__ SeqTable ST, int n_vs,
                                   uint32_t* cover) {
  const int slots = ST.count * n_vs;
  for (int sl = blockIdx.y; sl < slots; sl += gridDim.y) {
    const SeqInfo& S = ST.s[sl / n_vs];
    const int64_t x = sl % n_vs;
    const int n = S.n, cover_words = n_cover_words(n);
    const uint32_t* D = dbits + (int64_t)n_vs * S.word0 + x * n_words(n);
    uint32_t* out = cover + (int64_t)n_vs * S.cword0 + x * cover_words;
    const int zt = cover_words * 32;  // a multiple of 32: the ballot below sees whole warps
    for (int z = blockIdx.x * blockDim.x + threadIdx.x; z < zt; z += gridDim.x * blockDim.x) {
      bool any = false;
      if (z < n + 63) {
        int lo = n - 1 - z, hi = n + 62 - z;
        lo = lo < 0 ? 0 : lo;
        hi = hi > n - 1 ? n - 1 : hi;
        for (int w = lo >> 5; w <= (hi >> 5) && lo <= hi; ++w) {
          uint32_t v = __ldg(D + w);
          if (w == (lo >> 5)) v &= 0xFFFFFFFFu << (lo & 31);
          if (w == (hi >> 5)) v &= 0xFFFFFFFFu >> (31 - (hi & 31));
          if (v) { any = true; break; }
        }
      }
      const unsigned b = __ballot_sync(0xFFFFFFFFu, any);
      if ((threadIdx.x & 31) == 0) out[z / 32] = b;
    }
  }
}

// ------------------------------------------------------------------ per-block expansion
// One thread per query block u: merged slash ranges [a-δ, e-δ] ∩ [0, e] in
// ascending order (δ descending), then the verticals c <= e outside them.
__global__ void vs_expand_kernel(const int32_t* vertical, const int32_t* vcnt_p, int vcap, const int32_t* slash,
                                 const int32_t* scnt_p, int scap, int n,
                                 int u_begin, int u_count, int range_cap, int col_cap, int32_t* range_cnt,
                                 int32_t* ranges, int32_t* col_cnt, int32_t* cols) {
  const int x = blockIdx.x * blockDim.x + threadIdx.x;
  if (x >= u_count) return;
  const int u = u_begin + x;
  const int a = 64 * u, e = min(a + 64, n) - 1;
  const int vcnt = min(max(*vcnt_p, 0), vcap), scnt = min(max(*scnt_p, 0), scap);
  int nr = 0, lo = 0, hi = -2;
  bool open = false;
  for (int t = 0; t < scnt; ++t) {  // slash list is δ-descending -> starts ascending
    const int delta = slash[t];
    if (delta < 0 || e - delta < 0) continue;
    const int l0 = max(a - delta, 0), h0 = e - delta;
    if (open && l0 <= hi + 1) {
      hi = max(hi, h0);
    } else {
      if (open) {
        if (nr < range_cap) { ranges[((int64_t)x * range_cap + nr) * 2] = lo; ranges[((int64_t)x * range_cap + nr) * 2 + 1] = hi; }
        ++nr;
      }
      lo = l0; hi = h0; open = true;
    }
  }
  if (open) {
    if (nr < range_cap) { ranges[((int64_t)x * range_cap + nr) * 2] = lo; ranges[((int64_t)x * range_cap + nr) * 2 + 1] = hi; }
    ++nr;
  }
  range_cnt[x] = nr;
  // columns: both lists ascending -> one merge walk
  int nc = 0, rp = 0;
  for (int t = 0; t < vcnt; ++t) {
    const int c = vertical[t];
    if (c < 0 || c > e) continue;
    while (rp < min(nr, range_cap) && ranges[((int64_t)x * range_cap + rp) * 2 + 1] < c) ++rp;
    bool covered = rp < min(nr, range_cap) && ranges[((int64_t)x * range_cap + rp) * 2] <= c;
    if (!covered && nr > range_cap) {  // ranges beyond the cap were dropped: test against the slashes directly
      for (int s = 0; s < scnt && !covered; ++s) {
        const int delta = slash[s];
        covered = delta >= 0 && c >= a - delta && c <= e - delta;
      }
    }
    if (!covered) {
      if (nc < col_cap) cols[(int64_t)x * col_cap + nc] = c;
      ++nc;
    }
  }
  col_cnt[x] = nc;
}

size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }

int padded_rows(int L) { return L <= 32 ? 32 : (L <= 64 ? 64 : 128); }

int sm_count() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1) return 148;
  return sms;
}

// One index pass over a list of sequences: the group packs (the same for
// every sequence), and the launches, each over at most kMaxSeqs sequences
// with their CTA prefixes; K chunks are sized so that all packs of all
// sequences together make about one CTA per SM.
struct VSPlan {
  PackTable pt;
  int n_gp = 0, Lp = 0, LB = 0, v_cap = 0, s_cap = 0;
  std::vector<SeqInfo> seqs;       // token order (kb0 filled)
  std::vector<SeqTable> launches;  // chunk0 / chunks filled
  std::vector<int> ctas;           // CTAs per launch
  int max_ctas = 0, max_packs = 0;
  int64_t tokens = 0, kbs = 0;
  size_t off_part = 0, off_lse = 0, off_col = 0, off_slash = 0, off_rpart = 0, total = 0;
};

// heads null: the worst case for sizing (every head in its own KV group).
bool plan_vs(const msa_shape& s, const int32_t* heads, int32_t n_heads, const msa_head_cfg& cfg, int sms,
             const std::vector<SeqInfo>* seq_list, VSPlan& P) {
  P.seqs = seq_list ? *seq_list : uniform_seqs(s, 0);
  int n_max = 1;
  for (const SeqInfo& x : P.seqs) n_max = x.n > n_max ? x.n : n_max;
  const int L_max = cfg.last_q < n_max ? cfg.last_q : n_max;
  P.Lp = padded_rows(L_max);
  P.LB = P.Lp / 32;
  P.v_cap = cfg.n_vertical < n_max ? cfg.n_vertical : n_max;
  P.s_cap = cfg.n_slash < n_max ? cfg.n_slash : n_max;
  for (SeqInfo& x : P.seqs) {
    x.kb0 = (int32_t)P.kbs;
    P.kbs += 4 * n_tiles(x.n) + P.LB;
    P.tokens += x.n;
  }
  // group packs
  memset(&P.pt, 0, sizeof(P.pt));
  const int per_pack = kRows / P.Lp < kPackMaxHeads ? kRows / P.Lp : kPackMaxHeads;
  if (heads) {
    const int g = s.Hq / s.Hkv;
    for (int kv = 0; kv < s.Hkv; ++kv) {
      GroupPack cur;
      memset(&cur, 0, sizeof(cur));
      cur.g = kv;
      for (int x = 0; x < n_heads; ++x) {
        if (heads[x] / g != kv) continue;
        cur.x[cur.nh] = x;
        cur.h[cur.nh] = heads[x];
        if (++cur.nh == per_pack) {
          if (P.n_gp == kMaxGroupPacks) return false;
          P.pt.p[P.n_gp++] = cur;
          cur.nh = 0;
        }
      }
      if (cur.nh) {
        if (P.n_gp == kMaxGroupPacks) return false;
        P.pt.p[P.n_gp++] = cur;
      }
    }
  } else {
    P.n_gp = n_heads;
  }
  P.pt.n_gp = P.n_gp;
  // K chunks: about one CTA per SM over all packs of all sequences
  int64_t tile_packs = 0;
  for (const SeqInfo& x : P.seqs) tile_packs += (int64_t)P.n_gp * n_tiles(x.n);
  const int64_t tpc = tile_packs > sms ? (tile_packs + sms - 1) / sms : 1;
  std::vector<SeqInfo> live;
  for (const SeqInfo& x : P.seqs)
    if (x.n > 0) live.push_back(x);
  for (size_t b = 0; b < live.size(); b += kMaxSeqs) {
    SeqTable st;
    memset(&st, 0, sizeof(st));
    st.count = (int32_t)(live.size() - b < (size_t)kMaxSeqs ? live.size() - b : (size_t)kMaxSeqs);
    int64_t ctas = 0;
    for (int x = 0; x < st.count; ++x) {
      SeqInfo si = live[b + x];
      const int64_t nt = n_tiles(si.n);
      int64_t ch = (nt + tpc - 1) / tpc;
      ch = ch < 1 ? 1 : (ch > nt ? nt : ch);
      si.chunks = (int32_t)ch;
      si.chunk0 = (int32_t)ctas;
      ctas += (int64_t)P.n_gp * ch;
      st.s[x] = si;
    }
    if (ctas > 0x7FFFFFFF) return false;
    P.launches.push_back(st);
    P.ctas.push_back((int)ctas);
    P.max_ctas = (int)ctas > P.max_ctas ? (int)ctas : P.max_ctas;
    P.max_packs = st.count * P.n_gp > P.max_packs ? st.count * P.n_gp : P.max_packs;
  }
  size_t off = 0;
  P.off_part = off; off = align256(off + sizeof(float2) * (size_t)(P.max_ctas > 0 ? P.max_ctas : 1) * kRows);
  P.off_lse = off;  off = align256(off + sizeof(float) * (size_t)(P.max_packs > 0 ? P.max_packs : 1) * kRows);
  P.off_col = off;  off = align256(off + sizeof(float) * (size_t)n_heads * (size_t)P.tokens);
  P.off_slash = off; off = align256(off + sizeof(float) * (size_t)n_heads * (size_t)P.tokens);
  P.off_rpart = off; off = align256(off + sizeof(float) * (size_t)n_heads * (size_t)P.kbs * (P.LB + 1) * 32);
  P.total = off + 256;
  return true;
}

template <int D, int MODE, int LP>
msa_status launch_proxy(const CUtensorMap& tk, const ProxyArgs& a, const PackTable& pt, const SeqTable& st, int ctas,
                        cudaStream_t stream) {
  auto kern = proxy_kernel<D, MODE, LP>;
  const int smem = PLayout<D>::kAlloc;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return MSA_ERR_CUDA;
  if (ctas <= 0) return MSA_OK;
  kern<<<(unsigned)ctas, ProxyWarps<MODE, LP>::kThreads, smem, stream>>>(tk, a, pt, st);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

template <int D>
msa_status launch_scores(int Lp, const CUtensorMap& tk, const ProxyArgs& a, const PackTable& pt, const SeqTable& st,
                         int ctas, cudaStream_t stream) {
  if (Lp == 32) return launch_proxy<D, 2, 32>(tk, a, pt, st, ctas, stream);
  if (Lp == 64) return launch_proxy<D, 2, 64>(tk, a, pt, st, ctas, stream);
  return launch_proxy<D, 2, 128>(tk, a, pt, st, ctas, stream);
}

}  // namespace

size_t vs_index_ws_bytes(const msa_shape& s, const msa_head_cfg& cfg, const int32_t* heads, int32_t n_heads,
                         const std::vector<SeqInfo>* seqs) {
  VSPlan P;
  if (!plan_vs(s, heads, n_heads, cfg, sm_count(), seqs, P)) return 0;
  // without the heads the pack count is the worst case; so is the CTA count
  // (at most one per SM plus one per pack and sequence)
  if (!heads) {
    const size_t n_seq = P.seqs.size() < (size_t)kMaxSeqs ? P.seqs.size() : (size_t)kMaxSeqs;
    const size_t ctas = (size_t)sm_count() + (size_t)n_heads * n_seq;
    const size_t extra = align256(sizeof(float2) * ctas * kRows) + align256(sizeof(float) * (size_t)n_heads * n_seq * kRows);
    return P.total + extra + 1024;
  }
  return P.total + 1024;
}

msa_status run_vs_index(const msa_shape& s, const void* q, const void* k, const int32_t* heads, int32_t n_heads,
                        const msa_head_cfg& cfg, const msa_vs_index& out, void* ws, size_t ws_bytes,
                        cudaStream_t stream, const std::vector<SeqInfo>* seqs) {
  if (cfg.last_q > 128) return MSA_ERR_UNSUPPORTED;
  if (!out.vertical || !out.vertical_cnt || !out.slash || !out.slash_cnt || !out.vertical_bits || !out.slash_bits ||
      !out.slash_cover)
    return MSA_ERR_INVALID_ARG;
  VSPlan P;
  if (!plan_vs(s, heads, n_heads, cfg, sm_count(), seqs, P)) return MSA_ERR_UNSUPPORTED;
  if (out.v_cap < P.v_cap || out.s_cap < P.s_cap) return MSA_ERR_INVALID_ARG;
  if (!ws || P.total + 256 > ws_bytes) return MSA_ERR_WORKSPACE_TOO_SMALL;
  if (!rows_fit(s.Hq, P.seqs)) return MSA_ERR_UNSUPPORTED;
  uint8_t* w = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ws) + 255) & ~(uintptr_t)255);
  CUtensorMap tk;
  if (!make_bf16_map(&tk, k, 1, (int64_t)s.Hkv * P.tokens, s.d_h, 64)) return MSA_ERR_CUDA;
  ProxyArgs a;
  memset(&a, 0, sizeof(a));
  a.q = q;
  a.d = s.d_h;
  a.Lp = P.Lp;
  a.last_q = cfg.last_q;
  a.Hq = s.Hq;
  a.Hkv = s.Hkv;
  a.n_vs = n_heads;
  a.mode = cfg.proxy;
  const float scale = s.scale > 0.f ? s.scale : 1.0f / sqrtf((float)s.d_h);
  a.c2 = scale * 1.4426950408889634f;
  a.part = reinterpret_cast<float2*>(w + P.off_part);
  a.lse2 = reinterpret_cast<float*>(w + P.off_lse);
  a.colsum = reinterpret_cast<float*>(w + P.off_col);
  a.rpart = reinterpret_cast<float*>(w + P.off_rpart);
  a.err = device_error_word();
  if (!a.err) return MSA_ERR_CUDA;
  float* slashsum = reinterpret_cast<float*>(w + P.off_slash);
  int n_max = 1;
  for (const SeqInfo& x : P.seqs) n_max = x.n > n_max ? x.n : n_max;
  for (size_t L = 0; L < P.launches.size(); ++L) {
    const SeqTable& st = P.launches[L];
    const int ctas = P.ctas[L];
    msa_status r;
    // pass 1: row statistics
    r = s.d_h == 128 ? launch_proxy<128, 1, 64>(tk, a, P.pt, st, ctas, stream)
                     : launch_proxy<64, 1, 64>(tk, a, P.pt, st, ctas, stream);
    if (r != MSA_OK) return r;
    proxy_lse_kernel<<<(unsigned)(st.count * P.n_gp), kRows, 0, stream>>>(a.part, P.n_gp, st, a.lse2);
    note_launch();
    if (cudaGetLastError() != cudaSuccess) return MSA_ERR_CUDA;
    // pass 2: probabilities, column sums and diagonal bins
    r = s.d_h == 128 ? launch_scores<128>(P.Lp, tk, a, P.pt, st, ctas, stream)
                     : launch_scores<64>(P.Lp, tk, a, P.pt, st, ctas, stream);
    if (r != MSA_OK) return r;
    const int slots = st.count * n_heads;
    {
      const int bx = (n_max + 255) / 256 < 1024 ? (n_max + 255) / 256 : 1024;
      const int by = slots < 65535 ? slots : 65535;
      slash_finalize_kernel<<<dim3((unsigned)bx, (unsigned)by), 256, 0, stream>>>(a.rpart, st, n_heads, cfg.last_q,
                                                                                 P.LB, cfg.proxy, slashsum);
      note_launch();
      if (cudaGetLastError() != cudaSuccess) return MSA_ERR_CUDA;
    }
    // top-k for both score vectors of every slot
    TopkArgs ta;
    memset(&ta, 0, sizeof(ta));
    ta.colsum = a.colsum;
    ta.slashsum = slashsum;
    ta.out = out;
    ta.vk = cfg.n_vertical;
    ta.sk = cfg.n_slash;
    ta.n_vs = n_heads;
    topk_kernel<<<(unsigned)(slots * 2 * kTopkCluster), kTopkThreads, 0, stream>>>(ta, st);
    note_launch();
    if (cudaGetLastError() != cudaSuccess) return MSA_ERR_CUDA;
    {
      const int cw = n_cover_words(n_max);
      const int bx = (cw * 32 + 255) / 256 < 1024 ? (cw * 32 + 255) / 256 : 1024;
      const int by = slots < 65535 ? slots : 65535;
      slash_cover_kernel<<<dim3((unsigned)bx, (unsigned)by), 256, 0, stream>>>(out.slash_bits, st, n_heads,
                                                                              out.slash_cover);
      note_launch();
    }
    if (cudaGetLastError() != cudaSuccess) return MSA_ERR_CUDA;
  }
  return MSA_OK;
}

}  // namespace msa

using namespace msa;

extern "C" msa_status msa_vs_expand(const msa_shape* shape, const msa_vs_index* index, int32_t slot, int32_t u_begin,
                                    int32_t u_count, int32_t range_cap, int32_t col_cap, int32_t* range_cnt,
                                    int32_t* ranges, int32_t* col_cnt, int32_t* cols, void* stream) {
  if (!shape || !index || shape->n < 1 || slot < 0 || u_begin < 0 || u_count < 1 || range_cap < 0 || col_cap < 0)
    return MSA_ERR_INVALID_ARG;
  if (!range_cnt || !ranges || !col_cnt || !cols || !index->vertical || !index->slash || !index->vertical_cnt ||
      !index->slash_cnt)
    return MSA_ERR_INVALID_ARG;
  const int nb = ceil_div(shape->n, 64);
  if (u_begin + (int64_t)u_count > nb) return MSA_ERR_INVALID_ARG;
  vs_expand_kernel<<<(u_count + 127) / 128, 128, 0, (cudaStream_t)stream>>>(
      index->vertical + (int64_t)slot * index->v_cap, index->vertical_cnt + slot, index->v_cap,
      index->slash + (int64_t)slot * index->s_cap, index->slash_cnt + slot, index->s_cap,
      shape->n, u_begin, u_count, range_cap, col_cap, range_cnt, ranges, col_cnt, cols);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}
