// Layer-level dispatch (MInference page §5.1 "head dispatch and GQA mapping":
// every head reads its pattern from the layer's config table and is routed to
// its kernel) and the workspace bookkeeping of the exported entry points.
//
// A layer runs over a list of sequences: the B sequences of n tokens of a
// uniform batch, or the sequences of a varlen batch (cost-model page §2.2).
// Either way the online indices of every sequence are built in one pass and
// the attention of every head of every sequence runs in one launch (per 128
// sequences); the workspace holds every sequence's indices, sequence-major.
#include <string.h>

#include <vector>

#include "internal.h"

namespace msa {

msa_status check_shape(const msa_shape* s);
msa_status check_heads(const int32_t* heads, int32_t n_heads, int32_t Hq);

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Carves a workspace into aligned regions.
struct Carver {
  uint8_t* base;
  size_t off;
  template <class T>
  T* take(size_t count) {
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off = align256(off + count * sizeof(T));
    return p;
  }
};

static msa_status check_cfg(const msa_head_cfg& c) {
  switch (c.pattern) {
    case MSA_ASHAPE:
      if (c.sink < 0 || c.window < 1) return MSA_ERR_INVALID_ARG;
      return MSA_OK;
    case MSA_VS:
      if (c.last_q < 1 || c.n_vertical < 0 || c.n_slash < 0) return MSA_ERR_INVALID_ARG;
      if (c.proxy < 0 || c.proxy > 3) return MSA_ERR_INVALID_ARG;
      if (c.block != 64) return MSA_ERR_UNSUPPORTED;
      return MSA_OK;
    case MSA_BLOCK:
      if (c.topk < 1) return MSA_ERR_INVALID_ARG;
      if (c.block != 64) return MSA_ERR_UNSUPPORTED;
      return MSA_OK;
  }
  return MSA_ERR_INVALID_ARG;
}

struct LayerPlan {
  std::vector<int32_t> a_heads, vs_heads, bs_heads;
  msa_head_cfg vs_cfg, bs_cfg;
  std::vector<SeqInfo> seqs;  // token order
  int32_t v_cap = 0, s_cap = 0;
  // workspace regions
  msa_vs_index vs;
  int32_t* bs_idx = nullptr;
  int32_t* bs_cnt = nullptr;
  void* vs_ws = nullptr;
  size_t vs_ws_bytes = 0;
  void* bs_ws = nullptr;
  size_t bs_ws_bytes = 0;
  size_t total = 0;
};

// seqs null: the uniform batch of the shape (B sequences of n tokens).
static msa_status plan_layer(const msa_shape& s, const msa_head_cfg* table, void* ws, LayerPlan& P,
                             const std::vector<SeqInfo>* seqs = nullptr) {
  if (!table) return MSA_ERR_INVALID_ARG;
  memset(&P.vs_cfg, 0, sizeof(P.vs_cfg));
  memset(&P.bs_cfg, 0, sizeof(P.bs_cfg));
  for (int h = 0; h < s.Hq; ++h) {
    msa_status st = check_cfg(table[h]);
    if (st != MSA_OK) return st;
    if (table[h].pattern == MSA_ASHAPE) {
      P.a_heads.push_back(h);
    } else if (table[h].pattern == MSA_VS) {
      if (!P.vs_heads.empty() &&
          (table[h].last_q != P.vs_cfg.last_q || table[h].n_vertical != P.vs_cfg.n_vertical ||
           table[h].n_slash != P.vs_cfg.n_slash || table[h].proxy != P.vs_cfg.proxy))
        return MSA_ERR_UNSUPPORTED;  // one Vertical-Slash budget per layer
      P.vs_cfg = table[h];
      P.vs_heads.push_back(h);
    } else {
      if (!P.bs_heads.empty() && table[h].topk != P.bs_cfg.topk) return MSA_ERR_UNSUPPORTED;
      P.bs_cfg = table[h];
      P.bs_heads.push_back(h);
    }
  }
  P.seqs = seqs ? *seqs : uniform_seqs(s, 0);
  int64_t words = 0, cwords = 0, nbs = 0;
  int32_t n_max = 1;
  for (const SeqInfo& x : P.seqs) {
    words += n_words(x.n);
    cwords += n_cover_words(x.n);
    nbs += n_blocks(x.n);
    n_max = x.n > n_max ? x.n : n_max;
  }
  const int64_t n_seqs = (int64_t)P.seqs.size();
  Carver c{reinterpret_cast<uint8_t*>(ws), 0};
  memset(&P.vs, 0, sizeof(P.vs));
  if (!P.vs_heads.empty()) {
    const int64_t nvs = (int64_t)P.vs_heads.size(), slots = n_seqs * nvs;
    P.v_cap = P.vs_cfg.n_vertical < n_max ? P.vs_cfg.n_vertical : n_max;
    P.s_cap = P.vs_cfg.n_slash < n_max ? P.vs_cfg.n_slash : n_max;
    P.vs.v_cap = P.v_cap;
    P.vs.s_cap = P.s_cap;
    P.vs.vertical = c.take<int32_t>((size_t)(slots * (P.v_cap > 0 ? P.v_cap : 1)));
    P.vs.vertical_cnt = c.take<int32_t>((size_t)slots);
    P.vs.slash = c.take<int32_t>((size_t)(slots * (P.s_cap > 0 ? P.s_cap : 1)));
    P.vs.slash_cnt = c.take<int32_t>((size_t)slots);
    P.vs.vertical_bits = c.take<uint32_t>((size_t)(nvs * words));
    P.vs.slash_bits = c.take<uint32_t>((size_t)(nvs * words));
    P.vs.slash_cover = c.take<uint32_t>((size_t)(nvs * cwords));
    P.vs_ws_bytes = vs_index_ws_bytes(s, P.vs_cfg, P.vs_heads.data(), (int32_t)nvs, &P.seqs);
    if (P.vs_ws_bytes == 0) return MSA_ERR_UNSUPPORTED;
    P.vs_ws = c.take<uint8_t>(P.vs_ws_bytes);
  }
  if (!P.bs_heads.empty()) {
    const int64_t nbsl = (int64_t)P.bs_heads.size();
    P.bs_idx = c.take<int32_t>((size_t)(nbsl * nbs * P.bs_cfg.topk));
    P.bs_cnt = c.take<int32_t>((size_t)(nbsl * nbs));
    P.bs_ws_bytes = block_index_ws_bytes_exact(s, P.bs_heads.data(), (int32_t)nbsl, &P.seqs);
    P.bs_ws = c.take<uint8_t>(P.bs_ws_bytes);
  }
  P.total = c.off + 256;
  return MSA_OK;
}

}  // namespace msa

using namespace msa;

extern "C" {

size_t msa_vs_index_workspace(const msa_shape* shape, const msa_head_cfg* cfg, int32_t n_heads) {
  if (check_shape(shape) != MSA_OK || !cfg || n_heads < 1) return 0;
  return vs_index_ws_bytes(*shape, *cfg, nullptr, n_heads);
}

size_t msa_block_index_workspace(const msa_shape* shape, int32_t block, int32_t n_heads) {
  if (check_shape(shape) != MSA_OK || block != 64 || n_heads < 1) return 0;
  return block_index_ws_bytes(*shape, n_heads);
}

size_t msa_layer_workspace(const msa_shape* shape, const msa_head_cfg* table) {
  if (check_shape(shape) != MSA_OK) return 0;
  LayerPlan P;
  if (plan_layer(*shape, table, nullptr, P) != MSA_OK) return 0;
  return P.total;
}

msa_status msa_build_vs_index(const msa_shape* shape, const void* q, const void* k, const int32_t* heads,
                              int32_t n_heads, const msa_head_cfg* cfg, const msa_vs_index* out, void* ws,
                              size_t ws_bytes, void* stream) {
  msa_status st = check_shape(shape);
  if (st != MSA_OK) return st;
  if ((st = check_heads(heads, n_heads, shape->Hq)) != MSA_OK) return st;
  if (!cfg || !out || !q || !k) return MSA_ERR_INVALID_ARG;
  if (cfg->last_q < 1 || cfg->n_vertical < 0 || cfg->n_slash < 0) return MSA_ERR_INVALID_ARG;
  if (cfg->proxy < 0 || cfg->proxy > 3) return MSA_ERR_INVALID_ARG;
  if (cfg->block != 64) return MSA_ERR_UNSUPPORTED;
  return run_vs_index(*shape, q, k, heads, n_heads, *cfg, *out, ws, ws_bytes, (cudaStream_t)stream);
}

msa_status msa_build_block_index(const msa_shape* shape, const void* q, const void* k, const int32_t* heads,
                                 int32_t n_heads, int32_t block, int32_t topk, int32_t* block_idx,
                                 int32_t* block_cnt, void* ws, size_t ws_bytes, void* stream) {
  msa_status st = check_shape(shape);
  if (st != MSA_OK) return st;
  if ((st = check_heads(heads, n_heads, shape->Hq)) != MSA_OK) return st;
  if (!q || !k || !block_idx || !block_cnt) return MSA_ERR_INVALID_ARG;
  if (topk < 1) return MSA_ERR_INVALID_ARG;
  if (block != 64) return MSA_ERR_UNSUPPORTED;
  return run_block_index(*shape, q, k, heads, n_heads, topk, block_idx, block_cnt, ws, ws_bytes,
                         (cudaStream_t)stream);
}

}  // extern "C"

namespace msa {

static msa_status check_ptrs(const void* q, const void* k, const void* v, const void* o, const float* lse,
                             const int64_t* edges) {
  if (!q || !k) return MSA_ERR_INVALID_ARG;
  for (const void* p : {q, k, v, o})
    if (p && reinterpret_cast<uintptr_t>(p) % 16) return MSA_ERR_INVALID_ARG;
  if (lse && reinterpret_cast<uintptr_t>(lse) % 4) return MSA_ERR_INVALID_ARG;
  if (edges && reinterpret_cast<uintptr_t>(edges) % 8) return MSA_ERR_INVALID_ARG;
  return MSA_OK;
}

// Plan of a workspace for the sequences (null: the shape's uniform batch),
// after checking that it holds the plan.
static msa_status layer_prepare(const msa_shape* shape, const void* q, const void* k, const void* v, const void* o,
                                const float* lse, const int64_t* edges, const msa_head_cfg* table, void* ws,
                                size_t ws_bytes, LayerPlan& W, const std::vector<SeqInfo>* seqs = nullptr) {
  msa_status st = check_shape(shape);
  if (st != MSA_OK) return st;
  if (!table) return MSA_ERR_INVALID_ARG;
  if ((st = check_ptrs(q, k, v, o, lse, edges)) != MSA_OK) return st;
  LayerPlan P;
  if ((st = plan_layer(*shape, table, nullptr, P, seqs)) != MSA_OK) return st;
  if (ws_bytes < P.total || (P.total > 256 && !ws)) return MSA_ERR_WORKSPACE_TOO_SMALL;
  if (!rows_fit(shape->Hq, P.seqs)) return MSA_ERR_UNSUPPORTED;
  void* wsa = ws ? reinterpret_cast<void*>((reinterpret_cast<uintptr_t>(ws) + 255) & ~(uintptr_t)255) : nullptr;
  return plan_layer(*shape, table, wsa, W, seqs);
}

static msa_status layer_index(const msa_shape& s, const void* q, const void* k, const LayerPlan& W,
                              cudaStream_t strm) {
  msa_status st = MSA_OK;
  // both kinds of index: the Block-Sparse one runs on a side stream beside the
  // Vertical-Slash one (separate workspaces; both only read Q and K) and joins back
  SideStreams* f = (!W.vs_heads.empty() && !W.bs_heads.empty()) ? side_streams() : nullptr;
  cudaStream_t bs_strm = strm;
  std::unique_lock<std::mutex> hold;
  if (f) {
    hold = std::unique_lock<std::mutex>(f->mu);
    if (cudaEventRecord(f->ev[0], strm) != cudaSuccess || cudaStreamWaitEvent(f->side[0], f->ev[0], 0) != cudaSuccess)
      return MSA_ERR_CUDA;
    bs_strm = f->side[0];
  }
  if (!W.bs_heads.empty())
    st = run_block_index(s, q, k, W.bs_heads.data(), (int32_t)W.bs_heads.size(), W.bs_cfg.topk, W.bs_idx, W.bs_cnt,
                         W.bs_ws, W.bs_ws_bytes, bs_strm, &W.seqs);
  msa_status vs_st = MSA_OK;
  if (!W.vs_heads.empty())
    vs_st = run_vs_index(s, q, k, W.vs_heads.data(), (int32_t)W.vs_heads.size(), W.vs_cfg, W.vs, W.vs_ws,
                         W.vs_ws_bytes, strm, &W.seqs);
  if (f && (cudaEventRecord(f->ev[1], bs_strm) != cudaSuccess || cudaStreamWaitEvent(strm, f->ev[1], 0) != cudaSuccess))
    return MSA_ERR_CUDA;
  return st != MSA_OK ? st : vs_st;
}

static msa_status layer_attend(const msa_shape& s, const void* q, const void* k, const void* v,
                               const msa_head_cfg* table, void* o, float* lse, int64_t* edges, const LayerPlan& W,
                               cudaStream_t strm, int32_t row_lo = 0, int32_t row_hi = 0x7FFFFFFF,
                               int64_t* tiles = nullptr) {
  std::vector<Unit> units;
  if (!W.a_heads.empty()) {
    std::vector<int32_t> sinks, windows;
    for (int32_t h : W.a_heads) {
      sinks.push_back(table[h].sink);
      windows.push_back(table[h].window);
    }
    ashape_units(s, W.a_heads.data(), (int32_t)W.a_heads.size(), sinks.data(), windows.data(), units);
  }
  if (!W.vs_heads.empty()) vs_units(s, W.vs_heads.data(), (int32_t)W.vs_heads.size(), units);
  if (!W.bs_heads.empty()) block_units(s, W.bs_heads.data(), (int32_t)W.bs_heads.size(), units);
  // heavier patterns first within each KV-head band: the kernel runs a band's items by descending
  // tile pair, then by unit (launch_attention keeps this order when it groups units by KV head)
  std::vector<Unit> ordered;
  for (const Unit& u : units) if (u.pattern == kUnitVS) ordered.push_back(u);
  for (const Unit& u : units) if (u.pattern == kUnitBlock) ordered.push_back(u);
  for (const Unit& u : units) if (u.pattern == kUnitAshape) ordered.push_back(u);
  AttnArgs a;
  memset(&a, 0, sizeof(a));
  a.vs_dbits = W.vs.slash_bits;
  a.vs_cbits = W.vs.vertical_bits;
  a.vs_cover = W.vs.slash_cover;
  a.vs_nslots = (int32_t)W.vs_heads.size();
  a.bs_idx = W.bs_idx;
  a.bs_cnt = W.bs_cnt;
  a.bs_nslots = (int32_t)W.bs_heads.size();
  a.bs_topk = W.bs_heads.empty() ? 1 : W.bs_cfg.topk;
  return attention(s, q, k, v, o, lse, edges, ordered, a, strm, row_lo, row_hi, tiles, &W.seqs);
}

}  // namespace msa

extern "C" {

msa_status msa_layer_index(const msa_shape* shape, const void* q, const void* k, const msa_head_cfg* table,
                           void* ws, size_t ws_bytes, void* stream) {
  LayerPlan W;
  msa_status st = layer_prepare(shape, q, k, nullptr, nullptr, nullptr, nullptr, table, ws, ws_bytes, W);
  if (st != MSA_OK) return st;
  return layer_index(*shape, q, k, W, (cudaStream_t)stream);
}

msa_status msa_layer_attend(const msa_shape* shape, const void* q, const void* k, const void* v,
                            const msa_head_cfg* table, void* o, float* lse, int64_t* edges, void* ws,
                            size_t ws_bytes, void* stream) {
  if (!v || !o) return MSA_ERR_INVALID_ARG;
  LayerPlan W;
  msa_status st = layer_prepare(shape, q, k, v, o, lse, edges, table, ws, ws_bytes, W);
  if (st != MSA_OK) return st;
  return layer_attend(*shape, q, k, v, table, o, lse, edges, W, (cudaStream_t)stream);
}

msa_status msa_layer_attend_stats(const msa_shape* shape, const void* q, const void* k, const void* v,
                                  const msa_head_cfg* table, void* o, float* lse, int64_t* edges, int64_t* tiles,
                                  void* ws, size_t ws_bytes, void* stream) {
  if (!v || !o) return MSA_ERR_INVALID_ARG;
  if (tiles && reinterpret_cast<uintptr_t>(tiles) % 8) return MSA_ERR_INVALID_ARG;
  LayerPlan W;
  msa_status st = layer_prepare(shape, q, k, v, o, lse, edges, table, ws, ws_bytes, W);
  if (st != MSA_OK) return st;
  return layer_attend(*shape, q, k, v, table, o, lse, edges, W, (cudaStream_t)stream, 0, 0x7FFFFFFF, tiles);
}

msa_status msa_prefill_layer(const msa_shape* shape, const void* q, const void* k, const void* v,
                             const msa_head_cfg* table, void* o, float* lse, int64_t* edges, void* ws,
                             size_t ws_bytes, void* stream) {
  if (!v || !o) return MSA_ERR_INVALID_ARG;
  LayerPlan W;
  msa_status st = layer_prepare(shape, q, k, v, o, lse, edges, table, ws, ws_bytes, W);
  if (st != MSA_OK) return st;
  cudaStream_t strm = (cudaStream_t)stream;
  // 1. online indices, 2. every head's sparse attention in one launch; no
  // host synchronisation in between
  if ((st = layer_index(*shape, q, k, W, strm)) != MSA_OK) return st;
  return layer_attend(*shape, q, k, v, table, o, lse, edges, W, strm);
}

// ------------------------------------------------------------------ varlen
// Sequence s of a varlen batch: tokens [cu[s], cu[s+1]); its tensors are the
// s-th [H, n_s, d_h] segment of the packed buffers, i.e. token i of head h is
// row H * cu[s] + h * n_s + i of the [rows, d_h] views the kernels read.
static msa_status varlen_seqs(const msa_shape* shape, const int32_t* cu, int32_t n_seqs, std::vector<SeqInfo>& out) {
  if (!shape || !cu || n_seqs < 1 || cu[0] != 0) return MSA_ERR_INVALID_ARG;
  std::vector<int32_t> lens((size_t)n_seqs);
  for (int32_t x = 0; x < n_seqs; ++x) {
    if (cu[x + 1] < cu[x]) return MSA_ERR_INVALID_ARG;
    if (cu[x + 1] - cu[x] > (1 << 28)) return MSA_ERR_UNSUPPORTED;
    lens[(size_t)x] = cu[x + 1] - cu[x];
  }
  out = build_seqs(lens.data(), n_seqs, 0);
  return MSA_OK;
}

// The shape of a varlen batch: Hq, Hkv, d_h and scale from the caller; B and
// n are placeholders (the lengths come from the sequence list).
static msa_shape varlen_shape(const msa_shape* shape) {
  msa_shape s = *shape;
  s.B = 1;
  s.n = 1;
  return s;
}

size_t msa_layer_varlen_workspace(const msa_shape* shape, const msa_head_cfg* table, const int32_t* cu_seqlens,
                                  int32_t n_seqs) {
  std::vector<SeqInfo> seqs;
  if (!table || varlen_seqs(shape, cu_seqlens, n_seqs, seqs) != MSA_OK) return 0;
  const msa_shape s = varlen_shape(shape);
  if (check_shape(&s) != MSA_OK) return 0;
  LayerPlan P;
  if (plan_layer(s, table, nullptr, P, &seqs) != MSA_OK) return 0;
  return P.total;
}

msa_status msa_prefill_layer_varlen(const msa_shape* shape, const int32_t* cu_seqlens, int32_t n_seqs,
                                    const void* q, const void* k, const void* v, const msa_head_cfg* table, void* o,
                                    float* lse, int64_t* edges, void* ws, size_t ws_bytes, void* stream) {
  if (!shape || !q || !k || !v || !o || !table) return MSA_ERR_INVALID_ARG;
  std::vector<SeqInfo> seqs;
  msa_status st = varlen_seqs(shape, cu_seqlens, n_seqs, seqs);
  if (st != MSA_OK) return st;
  int64_t tokens = 0;
  for (const SeqInfo& x : seqs) tokens += x.n;
  if (tokens == 0) return MSA_OK;  // nothing to attend
  const msa_shape s = varlen_shape(shape);
  LayerPlan W;
  if ((st = layer_prepare(&s, q, k, v, o, lse, edges, table, ws, ws_bytes, W, &seqs)) != MSA_OK) return st;
  cudaStream_t strm = (cudaStream_t)stream;
  // one index pass and one attention launch per pattern over every sequence
  if ((st = layer_index(s, q, k, W, strm)) != MSA_OK) return st;
  return layer_attend(s, q, k, v, table, o, lse, edges, W, strm);
}

msa_status msa_layer_varlen_indices(const msa_shape* shape, const msa_head_cfg* table, const int32_t* cu_seqlens,
                                    int32_t n_seqs, void* ws, int32_t seq, msa_vs_index* vs, int32_t** block_idx,
                                    int32_t** block_cnt) {
  if (!shape || !table || !ws) return MSA_ERR_INVALID_ARG;
  std::vector<SeqInfo> seqs;
  msa_status st = varlen_seqs(shape, cu_seqlens, n_seqs, seqs);
  if (st != MSA_OK) return st;
  if (seq < 0 || seq >= n_seqs || seqs[(size_t)seq].n == 0) return MSA_ERR_INVALID_ARG;
  const msa_shape s = varlen_shape(shape);
  void* wsa = reinterpret_cast<void*>((reinterpret_cast<uintptr_t>(ws) + 255) & ~(uintptr_t)255);
  LayerPlan W;
  if ((st = plan_layer(s, table, wsa, W, &seqs)) != MSA_OK) return st;
  const SeqInfo& S = seqs[(size_t)seq];
  const int64_t nvs = (int64_t)W.vs_heads.size(), nbs = (int64_t)W.bs_heads.size();
  if (vs) {
    *vs = W.vs;
    if (nvs) {
      vs->vertical = W.vs.vertical + (int64_t)seq * nvs * W.vs.v_cap;
      vs->vertical_cnt = W.vs.vertical_cnt + (int64_t)seq * nvs;
      vs->slash = W.vs.slash + (int64_t)seq * nvs * W.vs.s_cap;
      vs->slash_cnt = W.vs.slash_cnt + (int64_t)seq * nvs;
      vs->vertical_bits = W.vs.vertical_bits + nvs * S.word0;
      vs->slash_bits = W.vs.slash_bits + nvs * S.word0;
      vs->slash_cover = W.vs.slash_cover + nvs * S.cword0;
    }
  }
  if (block_idx) *block_idx = nbs ? W.bs_idx + nbs * S.nb0 * W.bs_cfg.topk : nullptr;
  if (block_cnt) *block_cnt = nbs ? W.bs_cnt + nbs * S.nb0 : nullptr;
  return MSA_OK;
}

msa_status msa_layer_attend_rows(const msa_shape* shape, const void* q, const void* k, const void* v,
                                 const msa_head_cfg* table, void* o, float* lse, int64_t* edges, void* ws,
                                 size_t ws_bytes, int32_t row_begin, int32_t row_end, void* stream) {
  if (!shape || !v || !o) return MSA_ERR_INVALID_ARG;
  if (row_begin < 0 || row_end <= row_begin || row_end > shape->n) return MSA_ERR_INVALID_ARG;
  if (row_begin % 256 != 0 || (row_end % 256 != 0 && row_end != shape->n)) return MSA_ERR_INVALID_ARG;
  LayerPlan W;
  msa_status st = layer_prepare(shape, q, k, v, o, lse, edges, table, ws, ws_bytes, W);
  if (st != MSA_OK) return st;
  return layer_attend(*shape, q, k, v, table, o, lse, edges, W, (cudaStream_t)stream, row_begin, row_end);
}

uint64_t msa_kernel_launches(void) { return launch_count(); }

msa_status msa_layer_indices(const msa_shape* shape, const msa_head_cfg* table, void* ws, msa_vs_index* vs,
                             int32_t** block_idx, int32_t** block_cnt) {
  msa_status st = check_shape(shape);
  if (st != MSA_OK) return st;
  if (!ws) return MSA_ERR_INVALID_ARG;
  void* wsa = reinterpret_cast<void*>((reinterpret_cast<uintptr_t>(ws) + 255) & ~(uintptr_t)255);
  LayerPlan W;
  if ((st = plan_layer(*shape, table, wsa, W)) != MSA_OK) return st;
  if (vs) *vs = W.vs;
  if (block_idx) *block_idx = W.bs_idx;
  if (block_cnt) *block_cnt = W.bs_cnt;
  return MSA_OK;
}

}  // extern "C"
