// Host side of libmsa: argument validation, TMA tensor maps, work-unit
// construction and the exported C entry points declared in include/msa.h.
#include <math.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <vector>

#include "internal.h"
#include "ptx.cuh"

namespace msa {

__device__ int g_device_error = 0;

static std::atomic<uint64_t> g_launches{0};
void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }
uint64_t launch_count() { return g_launches.load(std::memory_order_relaxed); }

int* device_error_word() {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
  return reinterpret_cast<int*>(p);
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

bool make_bf16_map(CUtensorMap* map, const void* base, int64_t BH, int64_t n, int64_t d, int box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)n, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)(d * 2), (cuuint64_t)(n * d * 2)};
  cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ------------------------------------------------------------------ validation
msa_status check_shape(const msa_shape* s) {
  if (!s) return MSA_ERR_INVALID_ARG;
  if (s->B < 1 || s->Hq < 1 || s->Hkv < 1 || s->n < 1 || s->d_h < 1) return MSA_ERR_INVALID_ARG;
  if (s->Hq % s->Hkv != 0) return MSA_ERR_INVALID_ARG;
  if (!(s->scale == s->scale) || isinf(s->scale)) return MSA_ERR_INVALID_ARG;
  if (s->d_h != 64 && s->d_h != 128) return MSA_ERR_UNSUPPORTED;
  if (s->n > (1 << 28)) return MSA_ERR_UNSUPPORTED;
  if ((int64_t)s->B * s->Hq > (1 << 24)) return MSA_ERR_UNSUPPORTED;
  return MSA_OK;
}

static msa_status check_ptr(const void* p, bool required) {
  if (!p) return required ? MSA_ERR_INVALID_ARG : MSA_OK;
  if (reinterpret_cast<uintptr_t>(p) % 16 != 0) return MSA_ERR_INVALID_ARG;
  return MSA_OK;
}

static msa_status check_ptr4(const void* p, bool required) {
  if (!p) return required ? MSA_ERR_INVALID_ARG : MSA_OK;
  if (reinterpret_cast<uintptr_t>(p) % 4 != 0) return MSA_ERR_INVALID_ARG;
  return MSA_OK;
}

msa_status check_heads(const int32_t* heads, int32_t n_heads, int32_t Hq) {
  if (!heads || n_heads < 1 || n_heads > Hq) return MSA_ERR_INVALID_ARG;
  std::vector<char> seen((size_t)Hq, 0);
  for (int32_t x = 0; x < n_heads; ++x) {
    if (heads[x] < 0 || heads[x] >= Hq || seen[(size_t)heads[x]]) return MSA_ERR_INVALID_ARG;
    seen[(size_t)heads[x]] = 1;
  }
  return MSA_OK;
}

float effective_scale(const msa_shape& s) { return s.scale > 0.f ? s.scale : 1.0f / sqrtf((float)s.d_h); }

#define MSA_TRY(x)                       \
  do {                                   \
    msa_status st__ = (x);               \
    if (st__ != MSA_OK) return st__;     \
  } while (0)

static msa_status check_qkv(const msa_shape* s, const void* q, const void* k, const void* v) {
  MSA_TRY(check_shape(s));
  MSA_TRY(check_ptr(q, true));
  MSA_TRY(check_ptr(k, true));
  if (v) MSA_TRY(check_ptr(v, true));
  return MSA_OK;
}

// ------------------------------------------------------------------ units
// Every unit pairs two sub-items that read one KV head; item t of a unit
// covers query tile 2t + offset of each sub-item, so all units of a launch
// have ceil(tiles / 2) items and items of equal t cost about the same.  Heads
// of one KV group are paired (they read the same keys, and their selected
// keys tend to coincide); a head left alone is paired with itself (its even
// and odd query tiles).

static SubUnit sub_unit(int32_t qh0, int32_t qh1, int32_t off0, int32_t off1, int32_t slot0, int32_t slot1,
                        int32_t offset, int32_t sink, int32_t window) {
  SubUnit s;
  memset(&s, 0, sizeof(s));
  s.qh[0] = qh0;
  s.qh[1] = qh1;
  s.row_off[0] = off0;
  s.row_off[1] = off1;
  s.slot[0] = slot0;
  s.slot[1] = slot1;
  s.stride = 2;
  s.offset = offset;
  s.sink = sink;
  s.window = window;
  return s;
}

static void push_unit(std::vector<Unit>& out, int32_t pattern, int32_t kvh, const SubUnit& s0, const SubUnit& s1) {
  Unit u;
  memset(&u, 0, sizeof(u));
  u.pattern = pattern;
  u.kvh = kvh;
  u.has1 = 1;
  u.sub[0] = s0;
  u.sub[1] = s1;
  out.push_back(u);
}

// Positions x (into heads[]) of the heads of each KV group, in heads[] order.
static std::vector<std::vector<int>> kv_groups(const msa_shape& s, const int32_t* heads, int32_t nh) {
  const int g = s.Hq / s.Hkv;
  std::vector<std::vector<int>> G((size_t)s.Hkv);
  for (int x = 0; x < nh; ++x) G[(size_t)(heads[x] / g)].push_back(x);
  return G;
}

// Head-per-sub-item units (A-shape and Vertical-Slash): a pair of heads gives
// two units (even and odd tiles), a single head one unit.  slot[x] is the
// index slot of position x in batch 0; batch b adds b * slots_per_batch.
static void head_units(const msa_shape& s, int32_t pattern, const int32_t* heads, int32_t nh, const int32_t* sink,
                       const int32_t* window, const int32_t* slot, std::vector<Unit>& out) {
  const auto G = kv_groups(s, heads, nh);
  for (int kv = 0; kv < s.Hkv; ++kv) {
    const std::vector<int>& P = G[(size_t)kv];
    auto sub = [&](int x, int offset) {
      const int32_t qh = heads[x];
      const int32_t sl = slot ? slot[x] : 0;
      return sub_unit(qh, qh, 0, 64, sl, sl, offset, sink ? sink[x] : 0, window ? window[x] : 0);
    };
    size_t p = 0;
    for (; p + 1 < P.size(); p += 2)
      for (int o = 0; o < 2; ++o) push_unit(out, pattern, kv, sub(P[p], o), sub(P[p + 1], o));
    if (p < P.size()) push_unit(out, pattern, kv, sub(P[p], 0), sub(P[p], 1));
  }
}

void ashape_units(const msa_shape& s, const int32_t* heads, int32_t nh, const int32_t* sink, const int32_t* window,
                  std::vector<Unit>& out) {
  head_units(s, kUnitAshape, heads, nh, sink, window, nullptr, out);
}

// slot of heads[x] = x (its rank among the sequence's Vertical-Slash slots)
void vs_units(const msa_shape& s, const int32_t* heads, int32_t nh, std::vector<Unit>& out) {
  std::vector<int32_t> slot((size_t)nh);
  for (int x = 0; x < nh; ++x) slot[(size_t)x] = x;
  head_units(s, kUnitVS, heads, nh, nullptr, nullptr, slot.data(), out);
}

// Block-Sparse units: a half is one 64-row query block of one head.  Four
// heads of a KV group at the same query block form one item (their block
// lists tend to coincide); two heads take both blocks of a tile; a single
// head takes both blocks of its even and of its odd tile.
void block_units(const msa_shape& s, const int32_t* heads, int32_t nh, std::vector<Unit>& out) {
  const auto G = kv_groups(s, heads, nh);
  for (int kv = 0; kv < s.Hkv; ++kv) {
    const std::vector<int>& P = G[(size_t)kv];
    const int32_t kvh = kv;
    auto qh = [&](int x) { return heads[P[(size_t)x]]; };
    auto sl = [&](int x) { return P[(size_t)x]; };
    int p = 0;
    const int m = (int)P.size();
    for (; p + 3 < m; p += 4)
      for (int par = 0; par < 2; ++par)
        for (int o = 0; o < 2; ++o)
          push_unit(out, kUnitBlock, kvh,
                    sub_unit(qh(p), qh(p + 1), 64 * par, 64 * par, sl(p), sl(p + 1), o, 0, 0),
                    sub_unit(qh(p + 2), qh(p + 3), 64 * par, 64 * par, sl(p + 2), sl(p + 3), o, 0, 0));
    if (p + 1 < m) {
      for (int o = 0; o < 2; ++o)
        push_unit(out, kUnitBlock, kvh, sub_unit(qh(p), qh(p + 1), 0, 0, sl(p), sl(p + 1), o, 0, 0),
                  sub_unit(qh(p), qh(p + 1), 64, 64, sl(p), sl(p + 1), o, 0, 0));
      p += 2;
    }
    if (p < m)
      push_unit(out, kUnitBlock, kvh, sub_unit(qh(p), qh(p), 0, 64, sl(p), sl(p), 0, 0, 0),
                sub_unit(qh(p), qh(p), 0, 64, sl(p), sl(p), 1, 0, 0));
  }
}

// Failure-detection check: one thread waits on an mbarrier that nothing
// arrives at, with a short limit, and records the timeout in the error word
// exactly as the pipelines' bounded waits do.
__global__ void wait_timeout_check_kernel(uint64_t limit_ns, int* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait(&bar, 0, limit_ns)) atomicCAS(err, 0, kErrTimeout);
  }
}

// Sequences (in token order) with their prefix sums; lens[x] tokens each.
// LB: diagonal-bin rows of the Vertical-Slash scores pass (0 when unused).
std::vector<SeqInfo> build_seqs(const int32_t* lens, int n_seqs, int LB) {
  std::vector<SeqInfo> out;
  int64_t tok = 0, word = 0, cword = 0, nb = 0, kb = 0, tri = 0;
  for (int x = 0; x < n_seqs; ++x) {
    SeqInfo si;
    memset(&si, 0, sizeof(si));
    si.n = lens[x];
    si.tok0 = (int32_t)tok;
    si.word0 = (int32_t)word;
    si.cword0 = (int32_t)cword;
    si.nb0 = (int32_t)nb;
    si.kb0 = (int32_t)kb;
    si.tri0 = tri;
    si.seq = x;
    out.push_back(si);
    tok += lens[x];
    word += n_words(lens[x]);
    cword += n_cover_words(lens[x]);
    const int64_t b = n_blocks(lens[x]);
    nb += b;
    kb += 4 * n_tiles(lens[x]) + LB;
    tri += b * (b + 1) / 2;
  }
  return out;
}

std::vector<SeqInfo> uniform_seqs(const msa_shape& s, int LB) {
  std::vector<int32_t> lens((size_t)s.B, s.n);
  return build_seqs(lens.data(), s.B, LB);
}

// Rows of the [rows, d] views (H * total tokens, plus a tile past the end)
// must fit the int32 coordinates of TMA.
bool rows_fit(int64_t H, const std::vector<SeqInfo>& seqs) {
  int64_t tokens = 0;
  for (const SeqInfo& x : seqs) tokens += x.n;
  return H * tokens + 256 < ((int64_t)1 << 31);
}

msa_status attention(const msa_shape& s, const void* q, const void* k, const void* v, void* o, float* lse,
                     int64_t* edges, const std::vector<Unit>& units, const AttnArgs& idx, cudaStream_t stream,
                     int32_t row_lo, int32_t row_hi, int64_t* tiles, const std::vector<SeqInfo>* seq_list) {
  const std::vector<SeqInfo> own = seq_list ? std::vector<SeqInfo>() : uniform_seqs(s, 0);
  const std::vector<SeqInfo>& seqs = seq_list ? *seq_list : own;
  int64_t tokens = 0;
  for (const SeqInfo& x : seqs) tokens += x.n;
  if (!rows_fit(s.Hq, seqs)) return MSA_ERR_UNSUPPORTED;
  AttnMaps maps;
  if (!make_bf16_map(&maps.q, q, 1, (int64_t)s.Hq * tokens, s.d_h, 64) ||
      !make_bf16_map(&maps.k, k, 1, (int64_t)s.Hkv * tokens, s.d_h, 64) ||
      !make_bf16_map(&maps.v, v, 1, (int64_t)s.Hkv * tokens, s.d_h, 64) ||
      !make_bf16_map(&maps.k16, k, 1, (int64_t)s.Hkv * tokens, s.d_h, 16) ||
      !make_bf16_map(&maps.v16, v, 1, (int64_t)s.Hkv * tokens, s.d_h, 16))
    return MSA_ERR_CUDA;
  AttnArgs a = idx;
  a.d = s.d_h;
  a.Hq = s.Hq;
  a.Hkv = s.Hkv;
  a.scale_log2 = effective_scale(s) * 1.4426950408889634f;
  a.q = q;
  a.k = k;
  a.v = v;
  a.o = o;
  a.lse = lse;
  a.edges = reinterpret_cast<unsigned long long*>(edges);
  a.tiles = reinterpret_cast<unsigned long long*>(tiles);
  a.row_lo = row_lo;
  a.row_hi = row_hi;
  a.err = device_error_word();
  if (!a.err) return MSA_ERR_CUDA;
  // longest sequences first (their items are the heaviest), at most kMaxSeqs per launch
  std::vector<SeqInfo> order;
  for (const SeqInfo& x : seqs)
    if (x.n > 0) order.push_back(x);
  std::stable_sort(order.begin(), order.end(), [](const SeqInfo& p, const SeqInfo& q) { return p.n > q.n; });
  for (size_t b = 0; b < order.size(); b += kMaxSeqs) {
    SeqTable st;
    memset(&st, 0, sizeof(st));
    st.count = (int32_t)(order.size() - b < (size_t)kMaxSeqs ? order.size() - b : (size_t)kMaxSeqs);
    for (int x = 0; x < st.count; ++x) st.s[x] = order[b + x];
    msa_status r = launch_attention(maps, a, units.data(), (int)units.size(), st, stream);
    if (r != MSA_OK) return r;
  }
  return MSA_OK;
}

}  // namespace msa

using namespace msa;

extern "C" {

const char* msa_status_string(msa_status s) {
  switch (s) {
    case MSA_OK: return "ok";
    case MSA_ERR_INVALID_ARG: return "invalid argument";
    case MSA_ERR_UNSUPPORTED: return "unsupported configuration";
    case MSA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MSA_ERR_CUDA: return "CUDA runtime error";
    case MSA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case MSA_ERR_INDEX: return "index entry out of range";
  }
  return "unknown status";
}

msa_status msa_attn_ashape(const msa_shape* shape, const void* q, const void* k, const void* v,
                           const int32_t* heads, int32_t n_heads, int32_t sink, int32_t window, void* o,
                           float* lse, int64_t* edges, void* stream) {
  MSA_TRY(check_qkv(shape, q, k, v));
  MSA_TRY(check_ptr(o, true));
  MSA_TRY(check_ptr4(lse, false));
  MSA_TRY(check_ptr(edges, false));
  MSA_TRY(check_heads(heads, n_heads, shape->Hq));
  if (sink < 0 || window < 1) return MSA_ERR_INVALID_ARG;
  std::vector<Unit> units;
  const std::vector<int32_t> sinks((size_t)n_heads, sink), windows((size_t)n_heads, window);
  ashape_units(*shape, heads, n_heads, sinks.data(), windows.data(), units);
  AttnArgs a;
  memset(&a, 0, sizeof(a));
  return attention(*shape, q, k, v, o, lse, edges, units, a, (cudaStream_t)stream);
}

msa_status msa_attn_dense(const msa_shape* shape, const void* q, const void* k, const void* v, const int32_t* heads,
                          int32_t n_heads, void* o, float* lse, int64_t* edges, void* stream) {
  MSA_TRY(check_qkv(shape, q, k, v));
  // dense causal = A-shape with a window over every key: each row attends j <= i
  return msa_attn_ashape(shape, q, k, v, heads, n_heads, 0, shape->n, o, lse, edges, stream);
}

msa_status msa_attn_vs(const msa_shape* shape, const void* q, const void* k, const void* v, const int32_t* heads,
                       int32_t n_heads, int32_t block, const msa_vs_index* index, void* o, float* lse,
                       int64_t* edges, void* stream) {
  MSA_TRY(check_qkv(shape, q, k, v));
  MSA_TRY(check_ptr(o, true));
  MSA_TRY(check_ptr4(lse, false));
  MSA_TRY(check_ptr(edges, false));
  MSA_TRY(check_heads(heads, n_heads, shape->Hq));
  if (block != 64) return MSA_ERR_UNSUPPORTED;
  if (!index) return MSA_ERR_INVALID_ARG;
  MSA_TRY(check_ptr4(index->vertical_bits, true));
  MSA_TRY(check_ptr4(index->slash_bits, true));
  MSA_TRY(check_ptr4(index->slash_cover, true));
  std::vector<Unit> units;
  vs_units(*shape, heads, n_heads, units);
  AttnArgs a;
  memset(&a, 0, sizeof(a));
  a.vs_dbits = index->slash_bits;
  a.vs_cbits = index->vertical_bits;
  a.vs_cover = index->slash_cover;
  a.vs_nslots = n_heads;
  return attention(*shape, q, k, v, o, lse, edges, units, a, (cudaStream_t)stream);
}

msa_status msa_attn_block(const msa_shape* shape, const void* q, const void* k, const void* v,
                          const int32_t* heads, int32_t n_heads, int32_t block, int32_t topk,
                          const int32_t* block_idx, const int32_t* block_cnt, void* o, float* lse,
                          int64_t* edges, void* stream) {
  MSA_TRY(check_qkv(shape, q, k, v));
  MSA_TRY(check_ptr(o, true));
  MSA_TRY(check_ptr4(lse, false));
  MSA_TRY(check_ptr(edges, false));
  MSA_TRY(check_heads(heads, n_heads, shape->Hq));
  if (block != 64) return MSA_ERR_UNSUPPORTED;
  if (topk < 1) return MSA_ERR_INVALID_ARG;
  MSA_TRY(check_ptr4(block_idx, true));
  MSA_TRY(check_ptr4(block_cnt, true));
  std::vector<Unit> units;
  block_units(*shape, heads, n_heads, units);
  AttnArgs a;
  memset(&a, 0, sizeof(a));
  a.bs_idx = block_idx;
  a.bs_cnt = block_cnt;
  a.bs_topk = topk;
  a.bs_nslots = n_heads;
  return attention(*shape, q, k, v, o, lse, edges, units, a, (cudaStream_t)stream);
}

msa_status msa_check_wait_timeout(int32_t limit_ms, void* stream) {
  if (limit_ms < 1 || limit_ms > 2000) return MSA_ERR_INVALID_ARG;
  int* err = device_error_word();
  if (!err) return MSA_ERR_CUDA;
  wait_timeout_check_kernel<<<1, 32, 0, (cudaStream_t)stream>>>((uint64_t)limit_ms * 1000000ull, err);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

msa_status msa_poll_device_status(void* stream) {
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return MSA_ERR_CUDA;
  int* w = device_error_word();
  if (!w) return MSA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, w, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return MSA_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(w, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return MSA_ERR_CUDA;
  }
  if (v == kErrTimeout) return MSA_ERR_DEVICE_TIMEOUT;
  if (v == kErrIndex) return MSA_ERR_INDEX;
  return MSA_OK;
}

}  // extern "C"
