// Online Block-Sparse index (MInference page eq.(6) and §2.1 last paragraph;
// the MInference blog §2.3.2, Block-Sparse steps 1-3).
//
//   Q̄_u, K̄_v = means of the real tokens of each 64-row block (fp32)
//   r_uv     = Q̄_u . K̄_v                     (fp32, v < u)
//   J_u      = {u} ∪ top_{k_b-1}{v < u} by r_uv, ties to the lower v
//
// Kernels: block_pool (reads Q of the listed heads and K of their KV heads
// once: the byte cost of this index; writes each mean as three bf16 planes),
// block_scores (tcgen05 GEMM over the causal triangle of 128 x 128 tiles of
// block pairs, six plane products accumulated in fp32, written packed), block_topk
// (one warp per query block: rows of up to 2048 candidates in registers with a
// bitwise search for the k-th key, longer rows by radix select; then an
// index-ordered compaction, which leaves J_u ascending).
#include <cuda_bf16.h>
#include <string.h>

#include <vector>

#include "internal.h"
#include "ptx.cuh"

namespace msa {

namespace {

constexpr int kMaxSlots = 512;

__device__ __forceinline__ void set_err(int* err, int code) {
  if (err) atomicCAS(err, 0, code);
}

struct HeadMap {
  int32_t row_head[kMaxSlots];  // pooled head -> b*H + h of the source tensor
};

// Mean of each 64-row block of the `src` heads listed in `map`, for every
// sequence of the launch, written as three bf16 planes whose sum is the fp32
// mean to about 2^-24 (per sequence and head [3, nb, D], sequence-major:
// hi = bf16(m), mid = bf16(m - hi), lo = bf16(m - hi - mid)), so the score
// products can run on the bf16 tensor cores at fp32-like accuracy.
template <int D>
__global__ void __launch_bounds__(128) block_pool_kernel(const __nv_bfloat16* src, int H, int n_pool,
                                                         const __grid_constant__ SeqTable ST,
                                                         const __grid_constant__ HeadMap map, __nv_bfloat16* out) {
  constexpr int kTPR = D / 8;            // threads per row (8 columns each, 16-byte loads)
  constexpr int kGroups = 128 / kTPR;    // rows handled in parallel
  __shared__ float part[kGroups][D];
  // block u of pooled head hx of one sequence of the launch (blocks of all sequences along x)
  const SeqInfo& S = ST.s[seq_search(ST.count, [&](int x) { return ST.s[x].blk0; }, (int64_t)blockIdx.x)];
  const int u = (int)blockIdx.x - S.blk0, hx = blockIdx.y;
  const int n = S.n, nb = n_blocks(n);
  const int tid = threadIdx.x, grp = tid / kTPR, c8 = (tid % kTPR) * 8;
  const int a = 64 * u, e = min(a + 64, n);
  const __nv_bfloat16* base = src + ((int64_t)H * S.tok0 + (int64_t)map.row_head[hx] * n) * D;
  float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  for (int r = a + grp; r < e; r += kGroups) {
    const uint4 raw = __ldg(reinterpret_cast<const uint4*>(base + (int64_t)r * D + c8));
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int x = 0; x < 4; ++x) {
      const float2 f = __bfloat1622float2(p[x]);
      acc[2 * x] += f.x;
      acc[2 * x + 1] += f.y;
    }
  }
#pragma unroll
  for (int x = 0; x < 8; ++x) part[grp][c8 + x] = acc[x];
  __syncthreads();
  for (int c = tid; c < D; c += 128) {
    float s = 0.f;
    for (int g = 0; g < kGroups; ++g) s += part[g][c];
    const float m = s / (float)(e - a);
    const __nv_bfloat16 h = __float2bfloat16_rn(m);
    const float r1 = m - __bfloat162float(h);
    const __nv_bfloat16 md = __float2bfloat16_rn(r1);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(md));
    // planes of head hx of this sequence: rows 3 * (n_pool * nb0 + hx * nb) + plane * nb + u
    __nv_bfloat16* o = out + ((int64_t)3 * ((int64_t)n_pool * S.nb0 + (int64_t)hx * nb) + u) * D + c;
    o[0] = h;
    o[(int64_t)nb * D] = md;
    o[(int64_t)2 * nb * D] = lo;
  }
}

// Packed lower triangle (v <= u) of r_uv = Q̄_u . K̄_v on the tensor cores.
// One CTA per (128-row tile tu of query blocks, slot), heaviest rows first: it
// keeps the three Q̄ planes of its rows in shared memory and streams the key
// tiles tv = 0..tu (three K̄ planes, 64 columns of d per stage, two stages).
// Per stage, six bf16 products accumulate in fp32 in TMEM, smallest first:
// lo.hi + mid.mid + hi.lo + mid.hi + hi.mid + hi.hi (the dropped terms are
// below 2^-24 relative), two accumulators so that the epilogue of one tile
// overlaps the products of the next.  The epilogue stages 32 x 32 pieces in
// shared memory so that each warp writes one packed row segment per store.
//   warp 0: TMA producer, warp 1: MMA issuer (one thread), warps 2-5: epilogue
constexpr int kScThreads = 192;
constexpr int kScStages = 2;

template <int D>
struct ScLayout {
  static constexpr int kChunk = 128 * 64 * 2;              // 128 rows x 64 columns of bf16
  static constexpr int kQ = 0;                             // [plane][D / 64 chunks]
  static constexpr int kK = kQ + 3 * (D / 64) * kChunk;    // [stage][plane]
  static constexpr int kStage = kK + kScStages * 3 * kChunk;
  static constexpr int kBars = kStage + 4 * 32 * 33 * 4;   // epilogue staging, one 32 x 33 per warp
  static constexpr int kMisc = kBars + 16 * 8;
  static constexpr int kTotal = kMisc + 16;
  static constexpr int kAlloc = kTotal + 1024;
  static_assert(kAlloc <= 227 * 1024, "shared memory budget");
};

struct ScArgs {
  int n_bs, n_kv;       // query slots and pooled KV heads per sequence
  float* scores;        // packed triangles of every slot (sequence-major)
  int* err;
};

template <int D>
__global__ void __launch_bounds__(kScThreads, 1)
    block_scores_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                        const __grid_constant__ HeadMap kv_of_slot, const ScArgs A,
                        const __grid_constant__ SeqTable ST) {
  using Ly = ScLayout<D>;
  constexpr int kC = D / 64;  // stages per key tile
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + Ly::kBars);
  uint64_t* qfull = bars;
  uint64_t* kfull = bars + 1;                  // [kScStages]
  uint64_t* kempty = kfull + kScStages;        // [kScStages]
  uint64_t* afull = kempty + kScStages;        // [2]
  uint64_t* aempty = afull + 2;                // [2]
  volatile uint32_t* misc = reinterpret_cast<volatile uint32_t*>(sm + Ly::kMisc);  // [0] TMEM base, [1] abort
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // sequence, then row tile (heaviest first) and slot
  const SeqInfo& S = ST.s[seq_search(ST.count, [&](int x) { return ST.s[x].sc0; }, (int64_t)blockIdx.x)];
  const int local = (int)blockIdx.x - S.sc0;
  const int nb = n_blocks(S.n), T = (nb + 127) / 128;
  const int tu = T - 1 - local / A.n_bs;
  const int sl = local % A.n_bs;
  const int kvp = kv_of_slot.row_head[sl];
  const int ntile = tu + 1;  // key tiles tv = 0 .. tu
  // rows of plane p in the [rows, D] views of the pooled means: 3 (n_heads nb0 + head nb) + p nb
  const int32_t qrow = 3 * (A.n_bs * S.nb0 + sl * nb), krow = 3 * (A.n_kv * S.nb0 + kvp * nb);
  if (warp == 0) {
    tmem_alloc(const_cast<uint32_t*>(&misc[0]), 256);
    tmem_relinquish();
  }
  if (threadIdx.x == 32) {
    mbar_init(qfull, 1);
    for (int x = 0; x < kScStages; ++x) {
      mbar_init(&kfull[x], 1);
      mbar_init(&kempty[x], 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(&afull[x], 1);
      mbar_init(&aempty[x], 4);
    }
    misc[1] = 0;
    fence_mbar_init();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = misc[0];
  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      tma_prefetch_desc(&tq);
      tma_prefetch_desc(&tk);
      mbar_arrive_expect_tx(qfull, 3 * kC * Ly::kChunk);
      for (int p = 0; p < 3; ++p)
        for (int c = 0; c < kC; ++c)
          tma_load_3d(sm + Ly::kQ + (p * kC + c) * Ly::kChunk, &tq, qfull, 64 * c, qrow + p * nb + 128 * tu, 0);
      bool ok = true;
      for (int it = 0; it < ntile * kC && ok; ++it) {
        const int st = it % kScStages;
        if (misc[1] || !mbar_wait(&kempty[st], ((it / kScStages) & 1) ^ 1)) { ok = false; break; }
        const int tv = it / kC, c = it % kC;
        mbar_arrive_expect_tx(&kfull[st], 3 * Ly::kChunk);
        for (int p = 0; p < 3; ++p)
          tma_load_3d(sm + Ly::kK + (st * 3 + p) * Ly::kChunk, &tk, &kfull[st], 64 * c, krow + p * nb + 128 * tv, 0);
      }
      if (!ok) { misc[1] = 1; set_err(A.err, kErrTimeout); }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t id = idesc_bf16_f32(128, 128, false, false);
      const uint64_t dq = sdesc_sw128(smem_u32(sm + Ly::kQ), 16, 1024);
      const uint64_t dk = sdesc_sw128(smem_u32(sm + Ly::kK), 16, 1024);
      constexpr uint64_t kCh = Ly::kChunk >> 4;  // descriptor step of one chunk
      // (Q plane, K plane) of the six products, smallest terms first
      const int pa[6] = {2, 1, 0, 1, 0, 0}, pb[6] = {0, 1, 2, 0, 1, 0};
      bool ok = mbar_wait(qfull, 0);
      if (ok) tc_fence_after();
      int it = 0;
      for (int t = 0; t < ntile && ok; ++t) {
        const int buf = t & 1;
        if (misc[1] || !mbar_wait(&aempty[buf], ((t >> 1) & 1) ^ 1)) { ok = false; break; }
        tc_fence_after();
        for (int c = 0; c < kC; ++c, ++it) {
          const int st = it % kScStages;
          if (!mbar_wait(&kfull[st], (it / kScStages) & 1)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
#pragma unroll
            for (int x = 0; x < 6; ++x) {
              const uint64_t a = dq + (uint64_t)(pa[x] * kC + c) * kCh + 2 * kk;
              const uint64_t b = dk + (uint64_t)(st * 3 + pb[x]) * kCh + 2 * kk;
              mma_bf16_ss(tmem + 128 * buf, a, b, id, (c > 0 || kk > 0 || x > 0) ? 1u : 0u);
            }
          mma_commit(&kempty[st]);
        }
        if (ok) mma_commit(&afull[buf]);
      }
      if (!ok) { misc[1] = 1; set_err(A.err, kErrTimeout); }
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- epilogue
    const int q = warp & 3;  // TMEM lanes 32q ..
    float* st = reinterpret_cast<float*>(sm + Ly::kStage) + (warp - 2) * 32 * 33;
    const int64_t tri_base = (int64_t)A.n_bs * S.tri0 + (int64_t)sl * ((int64_t)nb * (nb + 1) / 2);
    bool ok = true;
    for (int t = 0; t < ntile; ++t) {
      const int buf = t & 1;
      if (misc[1] || !mbar_wait(&afull[buf], (t >> 1) & 1)) { ok = false; break; }
      tc_fence_after();
      const int tv = t;
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t v[32];
        tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + 128 * buf + 32 * cc, v);
        tmem_ld_wait();
#pragma unroll
        for (int x = 0; x < 32; ++x) st[lane * 33 + x] = __uint_as_float(v[x]);
        __syncwarp();
        const int vcol = 128 * tv + 32 * cc + lane;
#pragma unroll 4
        for (int k = 0; k < 32; ++k) {
          const int u = 128 * tu + 32 * q + k;
          if (u < nb && vcol <= u) A.scores[tri_base + (int64_t)u * (u + 1) / 2 + vcol] = st[k * 33 + lane];
        }
        __syncwarp();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&aempty[buf]);
    }
    if (!ok) { misc[1] = 1; set_err(A.err, kErrTimeout); }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

__device__ __forceinline__ uint32_t order_key(float f) {
  uint32_t b = __float_as_uint(f == 0.f ? 0.f : f);  // one zero
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

constexpr int kTopkWarps = 4;

// J_u from a row of u <= 32 R candidates held in registers (key of v = lane +
// 32 i in key[i]; 0, below every real key, for v >= u): the k1-th largest key
// T by a bitwise search on warp counts, then every key above T and the first
// (in index order) equal to it.  The search stops as soon as exactly k1 keys
// reach a candidate (then T = candidate - 1 and no key equal to T is taken).
// Rows are bucketed by length (R = 16, 32, 64) so a short row does not pay for
// the longest one.
template <int R>
__device__ __forceinline__ void topk_row_regs(const float* row, int u, int k1, int topk, int lane, int32_t* out,
                                              int32_t* cnt) {
  uint32_t key[R];
#pragma unroll
  for (int i = 0; i < R; ++i) {
    const int v = lane + 32 * i;
    key[i] = v < u ? order_key(row[v]) : 0u;
  }
  uint32_t T = 0;
  for (int b = 31; b >= 0; --b) {
    const uint32_t cand = T | (1u << b);
    int c = 0;
#pragma unroll
    for (int i = 0; i < R; ++i) c += key[i] >= cand ? 1 : 0;
    c = __reduce_add_sync(0xFFFFFFFFu, c);
    if (c == k1) {  // exactly k1 keys reach cand: they are the set (no tie to break)
      T = cand - 1u;
      break;
    }
    if (c > k1) T = cand;
  }
  int above = 0;
#pragma unroll
  for (int i = 0; i < R; ++i) above += key[i] > T ? 1 : 0;
  above = __reduce_add_sync(0xFFFFFFFFu, above);
  const int need_eq = k1 - above;
  int pos = 0, eq_seen = 0;
#pragma unroll
  for (int i = 0; i < R; ++i) {
    if (32 * i >= u) break;
    const bool gt = key[i] > T, eq = key[i] == T;
    const unsigned eqm = __ballot_sync(0xFFFFFFFFu, eq);
    const int eq_rank = eq_seen + __popc(eqm & ((1u << lane) - 1u));
    const bool sel = gt || (eq && eq_rank < need_eq);
    const unsigned selm = __ballot_sync(0xFFFFFFFFu, sel);
    if (sel) out[pos + __popc(selm & ((1u << lane) - 1u))] = lane + 32 * i;
    pos += __popc(selm);
    eq_seen += __popc(eqm);
  }
  for (int x = k1 + lane; x < topk; x += 32) out[x] = (x == k1) ? u : -1;  // diagonal last (largest id)
  if (lane == 0) *cnt = k1 + 1;
}

// One warp per (slot, query block u): J_u = {u} ∪ top_{k-1} of row u.  Rows
// longer than 2048 candidates use a radix select over a per-warp histogram in
// dynamic shared memory (kTopkWarps x 2048 ints, given only when nb > 2048).
__global__ void __launch_bounds__(32 * kTopkWarps, 4) block_topk_kernel(const float* scores, int n_bs, int topk,
                                                                      const __grid_constant__ SeqTable ST,
                                                                      int64_t jobs, int32_t* J, int32_t* cnt_out) {
  extern __shared__ int hist_all[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t job_l = (int64_t)blockIdx.x * kTopkWarps + warp;
  if (job_l >= jobs) return;
  // sequence (n_bs * blocks jobs each), slot and query block
  const SeqInfo& S = ST.s[seq_search(ST.count, [&](int x) { return (int64_t)n_bs * ST.s[x].blk0; }, job_l)];
  const int nb = n_blocks(S.n);
  const int64_t local = job_l - (int64_t)n_bs * S.blk0;
  const int slot = (int)(local / nb), u = (int)(local % nb);
  const float* row = scores + (int64_t)n_bs * S.tri0 + (int64_t)slot * ((int64_t)nb * (nb + 1) / 2) +
                     (int64_t)u * (u + 1) / 2;
  const int64_t job = (int64_t)n_bs * S.nb0 + (int64_t)slot * nb + u;  // output row (sequence-major)
  int32_t* out = J + job * topk;
  int32_t* cnt = cnt_out;
  const int k1 = min(topk - 1, u);  // picks among v < u
  if (u <= 2048 && k1 < u && k1 > 0) {
    if (u <= 512) topk_row_regs<16>(row, u, k1, topk, lane, out, cnt + job);
    else if (u <= 1024) topk_row_regs<32>(row, u, k1, topk, lane, out, cnt + job);
    else topk_row_regs<64>(row, u, k1, topk, lane, out, cnt + job);
    return;
  }
  int* h = hist_all + warp * 2048;
  uint32_t prefix = 0, pmask = 0;
  int need = k1;
  const bool all = (k1 >= u);
  if (!all && k1 > 0) {
    const int shifts[3] = {21, 10, 0}, widths[3] = {11, 11, 10};
    for (int pass = 0; pass < 3; ++pass) {
      const int sft = shifts[pass], nbins = 1 << widths[pass];
      for (int b = lane; b < nbins; b += 32) h[b] = 0;
      __syncwarp();
      for (int v = lane; v < u; v += 32) {
        const uint32_t key = order_key(row[v]);
        if ((key & pmask) == prefix) atomicAdd(&h[(key >> sft) & (nbins - 1)], 1);
      }
      __syncwarp();
      // digit of the need-th largest: suffix sums over the bins, 64 per lane
      int digit = 0, above = 0;
      {
        const int per = nbins / 32;
        int mine = 0;
        for (int b = 0; b < per; ++b) mine += h[lane * per + b];
        // inclusive suffix over lanes (higher lanes hold higher bins)
        int suf = mine;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_down_sync(0xFFFFFFFFu, suf, o);
          if (lane + o < 32) suf += y;
        }
        const int excl = suf - mine;  // count in lanes above
        const bool here = excl < need && suf >= need;
        const unsigned who = __ballot_sync(0xFFFFFFFFu, here);
        const int src = __ffs(who) - 1;
        int d = 0, ab = 0;
        if (lane == src) {
          int cum = excl;
          for (int b = per - 1; b >= 0; --b) {
            const int c = h[lane * per + b];
            if (cum + c >= need) { d = lane * per + b; break; }
            cum += c;
          }
          ab = cum;
        }
        digit = __shfl_sync(0xFFFFFFFFu, d, src);
        above = __shfl_sync(0xFFFFFFFFu, ab, src);
      }
      need -= above;
      prefix |= (uint32_t)digit << sft;
      pmask |= (uint32_t)(nbins - 1) << sft;
      __syncwarp();
    }
  }
  // index-ordered compaction: every key above the threshold, then the first
  // `need` keys equal to it
  int pos = 0, eq_seen = 0;
  for (int base = 0; base < u; base += 32) {
    const int v = base + lane;
    bool gt = false, eq = false;
    if (v < u) {
      if (all) gt = true;
      else if (k1 > 0) {
        const uint32_t key = order_key(row[v]);
        gt = key > prefix;
        eq = key == prefix;
      }
    }
    const unsigned eqm = __ballot_sync(0xFFFFFFFFu, eq);
    const int eq_rank = eq_seen + __popc(eqm & ((1u << lane) - 1u));
    const bool sel = gt || (eq && eq_rank < need);
    const unsigned selm = __ballot_sync(0xFFFFFFFFu, sel);
    if (sel) {
      const int p = pos + __popc(selm & ((1u << lane) - 1u));
      if (p < k1) out[p] = v;
    }
    pos += __popc(selm);
    eq_seen += __popc(eqm);
  }
  const int got = min(pos, k1);
  for (int x = got + lane; x < topk; x += 32) out[x] = (x == got) ? u : -1;  // diagonal last (largest id)
  if (lane == 0) cnt[job] = got + 1;
}

struct BSPlan {
  std::vector<int32_t> q_rows, kv_rows, kv_of_slot;  // per sequence: query head per slot, KV heads, KV index per slot
  int slots = 0, nkv = 0;                           // per sequence
  std::vector<SeqInfo> seqs;                        // token order
  std::vector<SeqTable> launches;                   // blk0 / sc0 filled
  std::vector<int64_t> blocks, ctas;                // per launch: Σ nb, score CTAs
  int nb_max = 1;
  int64_t nb_total = 0, tri_total = 0;
  size_t off_q = 0, off_k = 0, off_s = 0, total = 0;
};

size_t al256(size_t v) { return (v + 255) & ~(size_t)255; }

// heads null: the upper bound (one KV head per listed head).
BSPlan plan_bs(const msa_shape& s, const int32_t* heads, int32_t n_heads, const std::vector<SeqInfo>* seq_list) {
  BSPlan P;
  P.slots = n_heads;
  const int g = s.Hq / s.Hkv;
  if (heads) {
    std::vector<int> kv_index((size_t)s.Hkv, -1);
    for (int x = 0; x < n_heads; ++x) {
      P.q_rows.push_back(heads[x]);
      const int kv = heads[x] / g;
      if (kv_index[(size_t)kv] < 0) {
        kv_index[(size_t)kv] = (int)P.kv_rows.size();
        P.kv_rows.push_back(kv);
      }
      P.kv_of_slot.push_back(kv_index[(size_t)kv]);
    }
    P.nkv = (int)P.kv_rows.size();
  } else {
    P.nkv = P.slots;  // upper bound
  }
  P.seqs = seq_list ? *seq_list : uniform_seqs(s, 0);
  for (const SeqInfo& x : P.seqs) {
    const int64_t nb = n_blocks(x.n);
    P.nb_total += nb;
    P.tri_total += nb * (nb + 1) / 2;
    P.nb_max = (int)nb > P.nb_max ? (int)nb : P.nb_max;
  }
  std::vector<SeqInfo> live;
  for (const SeqInfo& x : P.seqs)
    if (x.n > 0) live.push_back(x);
  for (size_t b = 0; b < live.size(); b += kMaxSeqs) {
    SeqTable st;
    memset(&st, 0, sizeof(st));
    st.count = (int32_t)(live.size() - b < (size_t)kMaxSeqs ? live.size() - b : (size_t)kMaxSeqs);
    int64_t blk = 0, sc = 0;
    for (int x = 0; x < st.count; ++x) {
      SeqInfo si = live[b + x];
      si.blk0 = (int32_t)blk;
      si.sc0 = (int32_t)sc;
      const int64_t nb = n_blocks(si.n);
      blk += nb;
      sc += (int64_t)P.slots * ((nb + 127) / 128);
      st.s[x] = si;
    }
    P.launches.push_back(st);
    P.blocks.push_back(blk);
    P.ctas.push_back(sc);
  }
  size_t off = 0;
  P.off_q = off; off = al256(off + sizeof(__nv_bfloat16) * 3 * (size_t)P.slots * (size_t)P.nb_total * s.d_h);
  P.off_k = off; off = al256(off + sizeof(__nv_bfloat16) * 3 * (size_t)P.nkv * (size_t)P.nb_total * s.d_h);
  P.off_s = off; off = al256(off + sizeof(float) * (size_t)P.slots * (size_t)P.tri_total);
  P.total = off + 256;
  return P;
}

template <int D>
msa_status run_bs(const msa_shape& s, const void* q, const void* k, const BSPlan& P, int topk, int32_t* J,
                  int32_t* cnt, uint8_t* w, cudaStream_t stream) {
  __nv_bfloat16* qbar = reinterpret_cast<__nv_bfloat16*>(w + P.off_q);  // per sequence [slots, 3, nb, D]
  __nv_bfloat16* kbar = reinterpret_cast<__nv_bfloat16*>(w + P.off_k);  // per sequence [nkv, 3, nb, D]
  float* sc = reinterpret_cast<float*>(w + P.off_s);
  if (P.slots > kMaxSlots || P.nkv > kMaxSlots) return MSA_ERR_UNSUPPORTED;
  HeadMap mq, mk, mslot;
  memset(&mq, 0, sizeof(mq));
  memset(&mk, 0, sizeof(mk));
  memset(&mslot, 0, sizeof(mslot));
  for (int x = 0; x < P.slots; ++x) {
    mq.row_head[x] = P.q_rows[(size_t)x];
    mslot.row_head[x] = P.kv_of_slot[(size_t)x];
  }
  for (int x = 0; x < P.nkv; ++x) mk.row_head[x] = P.kv_rows[(size_t)x];
  // scores on the tensor cores: pooled planes viewed as [rows, D] with 128-row boxes
  CUtensorMap tqm, tkm;
  if (!make_bf16_map(&tqm, qbar, 1, (int64_t)3 * P.slots * P.nb_total, D, 128) ||
      !make_bf16_map(&tkm, kbar, 1, (int64_t)3 * P.nkv * P.nb_total, D, 128))
    return MSA_ERR_CUDA;
  auto kern = block_scores_kernel<D>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, ScLayout<D>::kAlloc) != cudaSuccess)
    return MSA_ERR_CUDA;
  ScArgs sa;
  sa.n_bs = P.slots;
  sa.n_kv = P.nkv;
  sa.scores = sc;
  sa.err = device_error_word();
  if (!sa.err) return MSA_ERR_CUDA;
  const int hist_bytes = P.nb_max > 2048 ? kTopkWarps * 2048 * (int)sizeof(int) : 0;
  for (size_t L = 0; L < P.launches.size(); ++L) {
    const SeqTable& st = P.launches[L];
    if (P.blocks[L] > 0x7FFFFFFF || P.ctas[L] > 0x7FFFFFFF) return MSA_ERR_UNSUPPORTED;
    block_pool_kernel<D><<<dim3((unsigned)P.blocks[L], (unsigned)P.slots), 128, 0, stream>>>(
        reinterpret_cast<const __nv_bfloat16*>(q), s.Hq, P.slots, st, mq, qbar);
    note_launch();
    if (cudaGetLastError() != cudaSuccess) return MSA_ERR_CUDA;
    block_pool_kernel<D><<<dim3((unsigned)P.blocks[L], (unsigned)P.nkv), 128, 0, stream>>>(
        reinterpret_cast<const __nv_bfloat16*>(k), s.Hkv, P.nkv, st, mk, kbar);
    note_launch();
    if (cudaGetLastError() != cudaSuccess) return MSA_ERR_CUDA;
    kern<<<(unsigned)P.ctas[L], kScThreads, ScLayout<D>::kAlloc, stream>>>(tqm, tkm, mslot, sa, st);
    note_launch();
    if (cudaGetLastError() != cudaSuccess) return MSA_ERR_CUDA;
    const int64_t jobs = (int64_t)P.slots * P.blocks[L];
    block_topk_kernel<<<(unsigned)((jobs + kTopkWarps - 1) / kTopkWarps), 32 * kTopkWarps, hist_bytes, stream>>>(
        sc, P.slots, topk, st, jobs, J, cnt);
    note_launch();
    if (cudaGetLastError() != cudaSuccess) return MSA_ERR_CUDA;
  }
  return MSA_OK;
}

}  // namespace

size_t block_index_ws_bytes(const msa_shape& s, int32_t n_heads, const std::vector<SeqInfo>* seqs) {
  return plan_bs(s, nullptr, n_heads, seqs).total + 256;
}
size_t block_index_ws_bytes_exact(const msa_shape& s, const int32_t* heads, int32_t n_heads,
                                  const std::vector<SeqInfo>* seqs) {
  return plan_bs(s, heads, n_heads, seqs).total + 256;
}

msa_status run_block_index(const msa_shape& s, const void* q, const void* k, const int32_t* heads,
                           int32_t n_heads, int32_t topk, int32_t* block_idx, int32_t* block_cnt, void* ws,
                           size_t ws_bytes, cudaStream_t stream, const std::vector<SeqInfo>* seqs) {
  BSPlan P = plan_bs(s, heads, n_heads, seqs);
  for (const SeqInfo& x : P.seqs) {
    const int64_t nb = n_blocks(x.n);
    if (nb * (nb + 1) / 2 > ((int64_t)1 << 40)) return MSA_ERR_UNSUPPORTED;
  }
  if (!rows_fit(s.Hq, P.seqs) || (int64_t)3 * P.slots * P.nb_total >= ((int64_t)1 << 31)) return MSA_ERR_UNSUPPORTED;
  // the workspace query is the worst case (one KV head per listed head); what
  // this call needs counts the KV heads the listed heads actually read
  if (!ws || ws_bytes < P.total + 256) return MSA_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* w = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ws) + 255) & ~(uintptr_t)255);
  if (s.d_h == 128) return run_bs<128>(s, q, k, P, topk, block_idx, block_cnt, w, stream);
  return run_bs<64>(s, q, k, P, topk, block_idx, block_cnt, w, stream);
}

}  // namespace msa
