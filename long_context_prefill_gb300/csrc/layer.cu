// Layer-level dispatch (MInference page §5.1 "head dispatch and GQA mapping":
// every head reads its pattern from the layer's config table and is routed to
// its kernel) and the workspace bookkeeping of the exported entry points.
#include <string.h>

#include <vector>

#include "internal.h"

namespace msa {

msa_status check_shape(const msa_shape* s);
msa_status check_heads(const int32_t* heads, int32_t n_heads, int32_t Hq);
void ashape_units(const msa_shape& s, const int32_t* heads, int32_t nh, const int32_t* sink, const int32_t* window,
                  std::vector<Unit>& out);
void vs_units(const msa_shape& s, const int32_t* heads, int32_t nh, int32_t slot_base_per_batch,
              int32_t slots_per_batch, std::vector<Unit>& out);
void block_units(const msa_shape& s, const int32_t* heads, int32_t nh, int32_t slots_per_batch,
                 std::vector<Unit>& out);
msa_status attention(const msa_shape& s, const void* q, const void* k, const void* v, void* o, float* lse,
                     int64_t* edges, const std::vector<Unit>& units, const AttnArgs& idx, cudaStream_t stream,
                     int32_t row_lo = 0, int32_t row_hi = 0x7FFFFFFF, int64_t* tiles = nullptr);

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
  int32_t v_cap = 0, s_cap = 0, words = 0, nb = 0;
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

static msa_status plan_layer(const msa_shape& s, const msa_head_cfg* table, void* ws, LayerPlan& P) {
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
  Carver c{reinterpret_cast<uint8_t*>(ws), 0};
  P.words = ceil_div(s.n, 32);
  P.nb = ceil_div(s.n, 64);
  memset(&P.vs, 0, sizeof(P.vs));
  if (!P.vs_heads.empty()) {
    const int64_t slots = (int64_t)s.B * (int64_t)P.vs_heads.size();
    P.v_cap = P.vs_cfg.n_vertical < s.n ? P.vs_cfg.n_vertical : s.n;
    P.s_cap = P.vs_cfg.n_slash < s.n ? P.vs_cfg.n_slash : s.n;
    P.vs.v_cap = P.v_cap;
    P.vs.s_cap = P.s_cap;
    P.vs.vertical = c.take<int32_t>((size_t)(slots * (P.v_cap > 0 ? P.v_cap : 1)));
    P.vs.vertical_cnt = c.take<int32_t>((size_t)slots);
    P.vs.slash = c.take<int32_t>((size_t)(slots * (P.s_cap > 0 ? P.s_cap : 1)));
    P.vs.slash_cnt = c.take<int32_t>((size_t)slots);
    P.vs.vertical_bits = c.take<uint32_t>((size_t)(slots * P.words));
    P.vs.slash_bits = c.take<uint32_t>((size_t)(slots * P.words));
    P.vs.slash_cover = c.take<uint32_t>((size_t)(slots * ceil_div(s.n + 63, 32)));
    P.vs_ws_bytes = vs_index_ws_bytes(s, P.vs_cfg, (int32_t)P.vs_heads.size());
    P.vs_ws = c.take<uint8_t>(P.vs_ws_bytes);
  }
  if (!P.bs_heads.empty()) {
    const int64_t slots = (int64_t)s.B * (int64_t)P.bs_heads.size();
    P.bs_idx = c.take<int32_t>((size_t)(slots * P.nb * P.bs_cfg.topk));
    P.bs_cnt = c.take<int32_t>((size_t)(slots * P.nb));
    P.bs_ws_bytes = block_index_ws_bytes(s, (int32_t)P.bs_heads.size());
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
  return vs_index_ws_bytes(*shape, *cfg, n_heads);
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

static msa_status layer_prepare(const msa_shape* shape, const void* q, const void* k, const void* v, const void* o,
                                const float* lse, const int64_t* edges, const msa_head_cfg* table, void* ws,
                                size_t ws_bytes, LayerPlan& W) {
  msa_status st = check_shape(shape);
  if (st != MSA_OK) return st;
  if (!q || !k || !table) return MSA_ERR_INVALID_ARG;
  for (const void* p : {q, k, v, o})
    if (p && reinterpret_cast<uintptr_t>(p) % 16) return MSA_ERR_INVALID_ARG;
  if (lse && reinterpret_cast<uintptr_t>(lse) % 4) return MSA_ERR_INVALID_ARG;
  if (edges && reinterpret_cast<uintptr_t>(edges) % 8) return MSA_ERR_INVALID_ARG;
  LayerPlan P;
  if ((st = plan_layer(*shape, table, nullptr, P)) != MSA_OK) return st;
  if (ws_bytes < P.total || (P.total > 256 && !ws)) return MSA_ERR_WORKSPACE_TOO_SMALL;
  void* wsa = ws ? reinterpret_cast<void*>((reinterpret_cast<uintptr_t>(ws) + 255) & ~(uintptr_t)255) : nullptr;
  return plan_layer(*shape, table, wsa, W);
}

static msa_status layer_index(const msa_shape& s, const void* q, const void* k, const LayerPlan& W,
                              cudaStream_t strm) {
  msa_status st = MSA_OK;
  if (!W.vs_heads.empty()) {
    st = run_vs_index(s, q, k, W.vs_heads.data(), (int32_t)W.vs_heads.size(), W.vs_cfg, W.vs, W.vs_ws,
                      W.vs_ws_bytes, strm);
    if (st != MSA_OK) return st;
  }
  if (!W.bs_heads.empty())
    st = run_block_index(s, q, k, W.bs_heads.data(), (int32_t)W.bs_heads.size(), W.bs_cfg.topk, W.bs_idx, W.bs_cnt,
                         W.bs_ws, W.bs_ws_bytes, strm);
  return st;
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
  if (!W.vs_heads.empty()) {
    const int32_t nvs = (int32_t)W.vs_heads.size();
    vs_units(s, W.vs_heads.data(), nvs, 0, nvs, units);
  }
  if (!W.bs_heads.empty())
    block_units(s, W.bs_heads.data(), (int32_t)W.bs_heads.size(), (int32_t)W.bs_heads.size(), units);
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
  a.vs_words = W.words;
  a.vs_cover_words = ceil_div(s.n + 63, 32);
  a.bs_idx = W.bs_idx;
  a.bs_cnt = W.bs_cnt;
  a.bs_topk = W.bs_heads.empty() ? 1 : W.bs_cfg.topk;
  a.bs_nb = W.nb;
  return attention(s, q, k, v, o, lse, edges, ordered, a, strm, row_lo, row_hi, tiles);
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
// s-th [H, n_s, d_h] segment of the packed buffers.  Each sequence is an
// ordinary B = 1 layer on its own segment: its own online indices, its own
// attention, so no index, window or tile reaches another sequence's tokens.
static msa_status check_cu_seqlens(const int32_t* cu, int32_t n_seqs) {
  if (!cu || n_seqs < 1 || cu[0] != 0) return MSA_ERR_INVALID_ARG;
  for (int32_t x = 0; x < n_seqs; ++x) {
    if (cu[x + 1] < cu[x]) return MSA_ERR_INVALID_ARG;
    if (cu[x + 1] - cu[x] > (1 << 28)) return MSA_ERR_UNSUPPORTED;
  }
  return MSA_OK;
}

// Each sequence owns its own region of the workspace (sequence-major), so the
// indices of every sequence are still there after the call.
static size_t varlen_region(const msa_shape* shape, const msa_head_cfg* table, int32_t len) {
  msa_shape ss = *shape;
  ss.B = 1;
  ss.n = len;
  return (msa_layer_workspace(&ss, table) + 255) & ~(size_t)255;
}

size_t msa_layer_varlen_workspace(const msa_shape* shape, const msa_head_cfg* table, const int32_t* cu_seqlens,
                                  int32_t n_seqs) {
  if (!shape || !table || check_cu_seqlens(cu_seqlens, n_seqs) != MSA_OK) return 0;
  size_t need = 256;
  for (int32_t x = 0; x < n_seqs; ++x) {
    const int32_t len = cu_seqlens[x + 1] - cu_seqlens[x];
    if (len == 0) continue;
    const size_t w = varlen_region(shape, table, len);
    if (w == 0) return 0;
    need += w;
  }
  return need;
}

msa_status msa_prefill_layer_varlen(const msa_shape* shape, const int32_t* cu_seqlens, int32_t n_seqs,
                                    const void* q, const void* k, const void* v, const msa_head_cfg* table, void* o,
                                    float* lse, int64_t* edges, void* ws, size_t ws_bytes, void* stream) {
  if (!shape || !q || !k || !v || !o || !table) return MSA_ERR_INVALID_ARG;
  msa_status st = check_cu_seqlens(cu_seqlens, n_seqs);
  if (st != MSA_OK) return st;
  const size_t need = msa_layer_varlen_workspace(shape, table, cu_seqlens, n_seqs);
  if (need == 0) return MSA_ERR_INVALID_ARG;
  if (ws_bytes < need || !ws) return MSA_ERR_WORKSPACE_TOO_SMALL;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ws) + 255) & ~(uintptr_t)255);
  const int64_t hq = shape->Hq, hkv = shape->Hkv, d = shape->d_h;
  size_t off = 0;
  for (int32_t x = 0; x < n_seqs; ++x) {
    const int32_t len = cu_seqlens[x + 1] - cu_seqlens[x];
    if (len == 0) continue;
    msa_shape ss = *shape;
    ss.B = 1;
    ss.n = len;
    const size_t region = varlen_region(shape, table, len);
    const int64_t t0 = cu_seqlens[x];
    const char* qb = static_cast<const char*>(q) + hq * t0 * d * 2;
    const char* kb = static_cast<const char*>(k) + hkv * t0 * d * 2;
    const char* vb = static_cast<const char*>(v) + hkv * t0 * d * 2;
    char* ob = static_cast<char*>(o) + hq * t0 * d * 2;
    if ((st = msa_prefill_layer(&ss, qb, kb, vb, table, ob, lse ? lse + hq * t0 : nullptr,
                                edges ? edges + (int64_t)x * hq : nullptr, base + off, region, stream)) != MSA_OK)
      return st;
    off += region;
  }
  return MSA_OK;
}

msa_status msa_layer_varlen_indices(const msa_shape* shape, const msa_head_cfg* table, const int32_t* cu_seqlens,
                                    int32_t n_seqs, void* ws, int32_t seq, msa_vs_index* vs, int32_t** block_idx,
                                    int32_t** block_cnt) {
  if (!shape || !table || !ws) return MSA_ERR_INVALID_ARG;
  msa_status st = check_cu_seqlens(cu_seqlens, n_seqs);
  if (st != MSA_OK) return st;
  if (seq < 0 || seq >= n_seqs || cu_seqlens[seq + 1] == cu_seqlens[seq]) return MSA_ERR_INVALID_ARG;
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(ws) + 255) & ~(uintptr_t)255);
  size_t off = 0;
  for (int32_t x = 0; x < seq; ++x) {
    const int32_t len = cu_seqlens[x + 1] - cu_seqlens[x];
    if (len) off += varlen_region(shape, table, len);
  }
  msa_shape ss = *shape;
  ss.B = 1;
  ss.n = cu_seqlens[seq + 1] - cu_seqlens[seq];
  return msa_layer_indices(&ss, table, base + off, vs, block_idx, block_cnt);
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
