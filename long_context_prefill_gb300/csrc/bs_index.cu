// Online Block-Sparse index (MInference page eq.(6) and §2.1 last paragraph;
// the MInference blog §2.3.2, Block-Sparse steps 1-3).
//
//   Q̄_u, K̄_v = means of the real tokens of each 64-row block (fp32)
//   r_uv     = Q̄_u . K̄_v                     (fp32, v < u)
//   J_u      = {u} ∪ top_{k_b-1}{v < u} by r_uv, ties to the lower v
//
// Kernels: block_pool (reads Q of the listed heads and K of their KV heads
// once: the byte cost of this index), block_scores (register-blocked fp32
// GEMM over the causal triangle of block pairs, written packed), block_topk
// (one warp per query block: rows of up to 2048 candidates in registers with a
// bitwise search for the k-th key, longer rows by radix select; then an
// index-ordered compaction, which leaves J_u ascending).
#include <cuda_bf16.h>
#include <string.h>

#include <vector>

#include "internal.h"

namespace msa {

namespace {

constexpr int kMaxSlots = 512;

struct HeadMap {
  int32_t row_head[kMaxSlots];  // pooled head -> b*H + h of the source tensor
};

// Mean of each 64-row block of `src` heads listed in `map` (fp32 out [nh, nb, D]).
template <int D>
__global__ void __launch_bounds__(128) block_pool_kernel(const __nv_bfloat16* src, int n, int nb,
                                                         const __grid_constant__ HeadMap map, float* out) {
  constexpr int kTPR = D / 8;            // threads per row (8 columns each, 16-byte loads)
  constexpr int kGroups = 128 / kTPR;    // rows handled in parallel
  __shared__ float part[kGroups][D];
  const int u = blockIdx.x, hx = blockIdx.y;
  const int tid = threadIdx.x, grp = tid / kTPR, c8 = (tid % kTPR) * 8;
  const int a = 64 * u, e = min(a + 64, n);
  const __nv_bfloat16* base = src + ((int64_t)map.row_head[hx] * n) * D;
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
    out[((int64_t)hx * nb + u) * D + c] = s / (float)(e - a);
  }
}

// Packed lower triangle (v <= u) of r_uv = Q̄_u . K̄_v for one slot per
// blockIdx.y; 64 x 64 tiles, 4 x 4 outputs per thread.
template <int D>
__global__ void __launch_bounds__(256) block_scores_kernel(const float* qbar, const float* kbar,
                                                           const __grid_constant__ HeadMap kv_of_slot, int nb,
                                                           float* scores) {
  constexpr int kC = 32;  // reduction columns staged per step
  __shared__ __align__(16) float sq[kC][64 + 4];
  __shared__ __align__(16) float sk[kC][64 + 4];
  // tile (tu, tv) with tv <= tu from the linear tile id
  const int lin = blockIdx.x;
  int tu = (int)((sqrtf(8.f * lin + 1.f) - 1.f) * 0.5f);
  while ((tu + 1) * (tu + 2) / 2 <= lin) ++tu;
  while (tu * (tu + 1) / 2 > lin) --tu;
  const int tv = lin - tu * (tu + 1) / 2;
  const int slot = blockIdx.y;
  const float* qb = qbar + (int64_t)slot * nb * D;
  const float* kb = kbar + (int64_t)kv_of_slot.row_head[slot] * nb * D;
  const int tid = threadIdx.x;
  const int tx = tid % 16, ty = tid / 16;
  float acc[4][4] = {};
  for (int c0 = 0; c0 < D; c0 += kC) {
    for (int idx = tid; idx < 64 * kC; idx += 256) {
      const int r = idx / kC, c = idx % kC;
      const int u = tu * 64 + r, v = tv * 64 + r;
      sq[c][r] = u < nb ? qb[(int64_t)u * D + c0 + c] : 0.f;
      sk[c][r] = v < nb ? kb[(int64_t)v * D + c0 + c] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int c = 0; c < kC; ++c) {
      const float4 a = *reinterpret_cast<const float4*>(&sq[c][ty * 4]);
      const float4 b = *reinterpret_cast<const float4*>(&sk[c][tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
  float* out = scores + (int64_t)slot * ((int64_t)nb * (nb + 1) / 2);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int u = tu * 64 + ty * 4 + i;
    if (u >= nb) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int v = tv * 64 + tx * 4 + j;
      if (v <= u) out[(int64_t)u * (u + 1) / 2 + v] = acc[i][j];
    }
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
__global__ void __launch_bounds__(32 * kTopkWarps) block_topk_kernel(const float* scores, int nb, int topk,
                                                                      int nslots, int32_t* J, int32_t* cnt) {
  extern __shared__ int hist_all[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t job = (int64_t)blockIdx.x * kTopkWarps + warp;
  if (job >= (int64_t)nslots * nb) return;
  const int slot = (int)(job / nb), u = (int)(job % nb);
  const float* row = scores + (int64_t)slot * ((int64_t)nb * (nb + 1) / 2) + (int64_t)u * (u + 1) / 2;
  int32_t* out = J + job * topk;
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
  std::vector<int32_t> q_rows, kv_rows, kv_of_slot;
  int nb, slots, nkv;
  size_t off_q, off_k, off_s, total;
};

size_t al256(size_t v) { return (v + 255) & ~(size_t)255; }

BSPlan plan_bs(const msa_shape& s, const int32_t* heads, int32_t n_heads) {
  BSPlan P;
  P.nb = ceil_div(s.n, 64);
  P.slots = s.B * n_heads;
  const int g = s.Hq / s.Hkv;
  if (heads) {
    std::vector<int> kv_index((size_t)s.B * s.Hkv, -1);
    for (int b = 0; b < s.B; ++b)
      for (int x = 0; x < n_heads; ++x) {
        P.q_rows.push_back(b * s.Hq + heads[x]);
        const int kv = b * s.Hkv + heads[x] / g;
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
  size_t off = 0;
  P.off_q = off; off = al256(off + sizeof(float) * (size_t)P.slots * P.nb * s.d_h);
  P.off_k = off; off = al256(off + sizeof(float) * (size_t)P.nkv * P.nb * s.d_h);
  P.off_s = off; off = al256(off + sizeof(float) * (size_t)P.slots * ((size_t)P.nb * (P.nb + 1) / 2));
  P.total = off + 256;
  return P;
}

template <int D>
msa_status run_bs(const msa_shape& s, const void* q, const void* k, const BSPlan& P, int topk, int32_t* J,
                  int32_t* cnt, uint8_t* w, cudaStream_t stream) {
  float* qbar = reinterpret_cast<float*>(w + P.off_q);
  float* kbar = reinterpret_cast<float*>(w + P.off_k);
  float* sc = reinterpret_cast<float*>(w + P.off_s);
  for (int base = 0; base < P.slots; base += kMaxSlots) {
    const int cntq = P.slots - base < kMaxSlots ? P.slots - base : kMaxSlots;
    HeadMap m;
    memset(&m, 0, sizeof(m));
    for (int x = 0; x < cntq; ++x) m.row_head[x] = P.q_rows[(size_t)(base + x)];
    block_pool_kernel<D><<<dim3(P.nb, cntq), 128, 0, stream>>>(reinterpret_cast<const __nv_bfloat16*>(q), s.n, P.nb,
                                                                m, qbar + (int64_t)base * P.nb * D);
    note_launch();
    if (cudaGetLastError() != cudaSuccess) return MSA_ERR_CUDA;
  }
  for (int base = 0; base < P.nkv; base += kMaxSlots) {
    const int cntk = P.nkv - base < kMaxSlots ? P.nkv - base : kMaxSlots;
    HeadMap m;
    memset(&m, 0, sizeof(m));
    for (int x = 0; x < cntk; ++x) m.row_head[x] = P.kv_rows[(size_t)(base + x)];
    block_pool_kernel<D><<<dim3(P.nb, cntk), 128, 0, stream>>>(reinterpret_cast<const __nv_bfloat16*>(k), s.n, P.nb,
                                                                m, kbar + (int64_t)base * P.nb * D);
    note_launch();
    if (cudaGetLastError() != cudaSuccess) return MSA_ERR_CUDA;
  }
  const int T = (P.nb + 63) / 64;
  const int tiles = T * (T + 1) / 2;
  for (int base = 0; base < P.slots; base += kMaxSlots) {
    const int cs = P.slots - base < kMaxSlots ? P.slots - base : kMaxSlots;
    HeadMap m;
    memset(&m, 0, sizeof(m));
    for (int x = 0; x < cs; ++x) m.row_head[x] = P.kv_of_slot[(size_t)(base + x)];
    block_scores_kernel<D><<<dim3(tiles, cs), 256, 0, stream>>>(
        qbar + (int64_t)base * P.nb * D, kbar, m, P.nb, sc + (int64_t)base * ((int64_t)P.nb * (P.nb + 1) / 2));
    note_launch();
    if (cudaGetLastError() != cudaSuccess) return MSA_ERR_CUDA;
  }
  const int64_t jobs = (int64_t)P.slots * P.nb;
  const int hist_bytes = P.nb > 2048 ? kTopkWarps * 2048 * (int)sizeof(int) : 0;
  block_topk_kernel<<<(unsigned)((jobs + kTopkWarps - 1) / kTopkWarps), 32 * kTopkWarps, hist_bytes, stream>>>(
      sc, P.nb, topk, P.slots, J, cnt);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

}  // namespace

size_t block_index_ws_bytes(const msa_shape& s, int32_t n_heads) { return plan_bs(s, nullptr, n_heads).total + 256; }

msa_status run_block_index(const msa_shape& s, const void* q, const void* k, const int32_t* heads,
                           int32_t n_heads, int32_t topk, int32_t* block_idx, int32_t* block_cnt, void* ws,
                           size_t ws_bytes, cudaStream_t stream) {
  if (!ws || ws_bytes < block_index_ws_bytes(s, n_heads)) return MSA_ERR_WORKSPACE_TOO_SMALL;
  const int nb = ceil_div(s.n, 64);
  if ((int64_t)nb * (nb + 1) / 2 > ((int64_t)1 << 40)) return MSA_ERR_UNSUPPORTED;
  BSPlan P = plan_bs(s, heads, n_heads);
  uint8_t* w = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ws) + 255) & ~(uintptr_t)255);
  if (s.d_h == 128) return run_bs<128>(s, q, k, P, topk, block_idx, block_cnt, w, stream);
  return run_bs<64>(s, q, k, P, topk, block_idx, block_cnt, w, stream);
}

}  // namespace msa
