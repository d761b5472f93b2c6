/*
 * msa.h — C ABI of libmsa: MInference-style dynamic sparse prefill attention
 * on one GB300 (sm_103a).
 *
 * The method (PaperTrace 2.1.2 "MInference: 按 head 模式加速长上下文 Prefill",
 * §1.1, eq.(1)-(2)): each attention head h of one layer restricts the causal
 * softmax of query row i to a candidate set N_h(i) ⊆ {j <= i} and computes
 *   o_hi = Σ_{j in N_h(i)} exp(s_hij) v_hj / Σ_{t in N_h(i)} exp(s_hit),
 *   s_hij = scale * q_hi . k_hj.
 * Which set a head uses comes from a per-head config table (same page, §1.1
 * and §3.1): A-shape (eq.(3)), Vertical-Slash (eq.(5)) or Block-Sparse
 * (eq.(6)).  Vertical-Slash and Block-Sparse sets are built per request from a
 * cheap proxy (§3.1, §6.2; "LLM模型之MInference" blog §2.3.2).
 *
 * Conventions shared by every call:
 *  - Q, O: [B, Hq, n, d_h] bf16; K, V: [B, Hkv, n, d_h] bf16; all contiguous
 *    device memory with 16-byte-aligned base addresses.  LSE: [B, Hq, n] fp32
 *    (natural log of the softmax denominator; -inf for an empty set).
 *  - GQA: query head h reads KV head h / (Hq / Hkv) (same page §5.1, "head
 *    dispatch and GQA mapping"); K/V are never repeated in memory.
 *  - d_h ∈ {64, 128}; Vertical-Slash and Block-Sparse blocks are 64 rows.
 *  - `heads` (host array of n_heads distinct query-head indices in [0, Hq))
 *    selects the heads a call works on; index arrays are laid out by "slot"
 *    = b * n_heads + position in `heads`.
 *  - Every buffer, including the workspace, is allocated and owned by the
 *    caller; the library keeps no allocation between calls.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream).  Arguments are validated on the host before anything
 *    is launched: a bad argument returns an error and launches nothing.
 *    Faults detected on the device (a bounded wait that timed out, an index
 *    out of range) are recorded in a device error word that
 *    msa_poll_device_status() reads; outputs of a failed call are undefined.
 *  - No call synchronises with the host (no device-to-host copy on the path).
 */
#ifndef MSA_H
#define MSA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MSA_API __attribute__((visibility("default")))
#else
#define MSA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MSA_OK = 0,
  MSA_ERR_INVALID_ARG = 1,         /* bad pointer, shape, head list or budget */
  MSA_ERR_UNSUPPORTED = 2,         /* valid request outside the supported set (d_h, block) */
  MSA_ERR_WORKSPACE_TOO_SMALL = 3, /* ws_bytes below the matching *_workspace() size */
  MSA_ERR_CUDA = 4,                /* a CUDA runtime call failed */
  MSA_ERR_DEVICE_TIMEOUT = 5,      /* a kernel's bounded wait gave up (reported by the poll) */
  MSA_ERR_INDEX = 6                /* an index entry out of range (reported by the poll) */
} msa_status;

typedef enum { MSA_ASHAPE = 0, MSA_VS = 1, MSA_BLOCK = 2 } msa_pattern;

/* Problem shape.  scale <= 0 selects 1/sqrt(d_h) (eq.(1)). */
typedef struct {
  int32_t B, Hq, Hkv, n, d_h;
  float scale;
} msa_shape;

/* One head's entry of the layer x head config table (MInference page §1.1:
 * best_pattern per layer and head with its budgets; §6.3: pattern type,
 * vertical / slash counts, block count, window, initial tokens, block size). */
typedef struct {
  int32_t pattern;    /* msa_pattern */
  int32_t sink;       /* A-shape: g initial tokens */
  int32_t window;     /* A-shape: w local window (>= 1) */
  int32_t last_q;     /* Vertical-Slash: proxy rows, the last last_q queries */
  int32_t n_vertical; /* Vertical-Slash: v columns kept */
  int32_t n_slash;    /* Vertical-Slash: s diagonal offsets kept */
  int32_t block;      /* Vertical-Slash / Block-Sparse block size (64) */
  int32_t topk;       /* Block-Sparse: k_b key blocks per query block (>= 1) */
  int32_t proxy;      /* Vertical-Slash proxy convention, MSA_PROXY_* bits (0: sums) */
} msa_head_cfg;

/* Vertical-Slash proxy conventions (msa_head_cfg.proxy bits; MInference page
 * §3.1: a column score may be the maximum over the sampled rows, which keeps a
 * single strong response, or their sum; §6.2: offset d has only the legal
 * pairs (i, i-d) of the sampled rows with i >= d, so a slash sum favours short
 * offsets and a slash mean does not).  0 = column sums and slash sums. */
enum { MSA_PROXY_COL_MAX = 1, MSA_PROXY_SLASH_MEAN = 2 };

/* Vertical-Slash index of a set of heads (device buffers owned by the caller).
 * For slot s (see conventions), with v_cap = min(n_vertical, n) and
 * s_cap = min(n_slash, n), words = ceil(n / 32), cover_words = ceil((n + 63) / 32):
 *   vertical[s * v_cap + t]   column indices C_h, ascending (t < vertical_cnt[s])
 *   slash[s * s_cap + t]      diagonal offsets D_h (δ = i - j), descending
 *   vertical_bits[s * words]  bit j set iff j ∈ C_h
 *   slash_bits[s * words]     bit δ set iff δ ∈ D_h
 *   slash_cover[s * cover_words]  bit z set iff D_h has an offset in
 *       [n-1-z, n+62-z]; for a full 64-row query block [a, a+63], key j is
 *       covered by one of the block's slash tiles iff bit n-1-a+j is set
 *       (the per-tile masks the attention kernel reads with a few word loads)
 * (MInference blog §2.3.3: verticals sorted ascending, slashes descending.) */
typedef struct {
  int32_t* vertical;
  int32_t* vertical_cnt;
  int32_t* slash;
  int32_t* slash_cnt;
  uint32_t* vertical_bits;
  uint32_t* slash_bits;
  uint32_t* slash_cover;
  int32_t v_cap;
  int32_t s_cap;
} msa_vs_index;

/* Status as text (static storage; no counterpart in the pages). */
MSA_API const char* msa_status_string(msa_status s);

/* Workspace sizing (no counterpart in the pages: the caller owns all memory).
 * Workspace bytes msa_build_vs_index needs for n_heads heads with budgets cfg
 * (0 on invalid arguments). */
MSA_API size_t msa_vs_index_workspace(const msa_shape* shape, const msa_head_cfg* cfg, int32_t n_heads);

/* Workspace bytes msa_build_block_index needs (0 on invalid arguments). */
MSA_API size_t msa_block_index_workspace(const msa_shape* shape, int32_t block, int32_t n_heads);

/* Workspace bytes msa_prefill_layer needs for this table (Hq entries); it
 * holds the per-request indices and the index builders' scratch. */
MSA_API size_t msa_layer_workspace(const msa_shape* shape, const msa_head_cfg* table);

/* Online Vertical-Slash index (MInference page §2.1 and §6.2; blog §2.3.2
 * Vertical-Slash steps 1-3).  For each listed head h, with the last
 * L = min(last_q, n) query rows R:
 *   Ã_ij = softmax over j <= i of scale * q_i.k_j       (i in R)
 *   c_j = Σ_{i in R} Ã_ij,  r_δ = Σ_{i in R, i >= δ} Ã_{i,i-δ}
 *   C_h = top-v of c, D_h = top-s of r (ties to the lower index).
 * Scores are fp32 from bf16 tensor-core products.  Writes `out` (layout
 * above).  q: [B,Hq,n,d_h], k: [B,Hkv,n,d_h].  Requires ws_bytes >=
 * msa_vs_index_workspace(shape, cfg, n_heads). */
MSA_API msa_status msa_build_vs_index(const msa_shape* shape, const void* q, const void* k, const int32_t* heads,
                              int32_t n_heads, const msa_head_cfg* cfg, const msa_vs_index* out, void* ws,
                              size_t ws_bytes, void* stream);

/* Online Block-Sparse index (MInference page eq.(6) and §2.1 last paragraph;
 * blog §2.3.2 Block-Sparse steps 1-3): Q̄_u, K̄_v = means of the real tokens
 * of each 64-row block, r_uv = Q̄_u . K̄_v, and
 *   J_u = {u} ∪ top_{k_b - 1} { v < u } by r_uv   (ties to the lower v),
 * i.e. the causal diagonal block is always kept and counts toward k_b.
 * block_idx: [B, n_heads, N_b, topk] int32, ascending, -1 padded;
 * block_cnt: [B, n_heads, N_b] int32 = min(topk, u + 1).  N_b = ceil(n/64).
 * Scores are fp32-accurate: each block mean is split into three bf16 parts and
 * the pair products accumulate in fp32 on the tensor cores. */
MSA_API msa_status msa_build_block_index(const msa_shape* shape, const void* q, const void* k, const int32_t* heads,
                                 int32_t n_heads, int32_t block, int32_t topk, int32_t* block_idx,
                                 int32_t* block_cnt, void* ws, size_t ws_bytes, void* stream);

/* Size of the library's built-in scratch for msa_build_block_index_static
 * (16 MiB of device memory per device, reserved when the library is loaded). */
#define MSA_STATIC_SCRATCH_BYTES (16u << 20)

/* msa_build_block_index without a workspace argument: the same index, built
 * in a scratch array the library holds in device memory, so the call
 * allocates nothing and needs no workspace query.  This entry point has no
 * counterpart in the MInference pages; it exists for callers that hold device
 * tensors from another runtime and have no allocator of their own (or must not
 * call cudaMalloc on their path).
 * Limit: the scratch these heads need must not exceed MSA_STATIC_SCRATCH_BYTES,
 * else MSA_ERR_WORKSPACE_TOO_SMALL is returned and nothing is launched.  The
 * need counts each KV head the listed heads read once, so it is at most
 * msa_block_index_workspace(shape, 64, n_heads) (which assumes one KV head per
 * listed head: for d_h = 128 up to 31 heads at n = 16384, 12 at n = 32768,
 * 4 at n = 65536; with four query heads per KV head, 16 heads at n = 32768 fit).
 * The scratch is shared by all calls on a device: calls that overlap in time
 * (unordered streams, several host threads) race on it and must be ordered.
 * The first call on a device looks up the scratch address (a runtime call),
 * so make one call on each device before the work that must be free of
 * set-up calls.  The looked-up address is cached per device ordinal and is
 * not refreshed: after cudaDeviceReset in the same process, do not call this
 * entry point on that device again.  Arguments and outputs as for
 * msa_build_block_index. */
MSA_API msa_status msa_build_block_index_static(const msa_shape* shape, const void* q, const void* k,
                                                const int32_t* heads, int32_t n_heads, int32_t block, int32_t topk,
                                                int32_t* block_idx, int32_t* block_cnt, void* stream);

/* A-shape attention (MInference page eq.(3)): N_A(i) = {0..min(g-1,i)} ∪
 * {max(0,i-w+1)..i}, exact (each key once).  o: [B,Hq,n,d_h] (only the listed
 * heads are written); lse nullable; edges nullable: if given, [B*Hq] int64
 * device counters to which each head's attended-edge count E_h is ADDED. */
MSA_API msa_status msa_attn_ashape(const msa_shape* shape, const void* q, const void* k, const void* v,
                           const int32_t* heads, int32_t n_heads, int32_t sink, int32_t window, void* o,
                           float* lse, int64_t* edges, void* stream);

/* Dense causal attention (MInference page eq.(1)-(2): N(i) = {0..i}) on the
 * same engine: the baseline the sparse patterns are measured against, and the
 * set every pattern reduces to when its budgets cover all keys.  Arguments as
 * for msa_attn_ashape. */
MSA_API msa_status msa_attn_dense(const msa_shape* shape, const void* q, const void* k, const void* v,
                                  const int32_t* heads, int32_t n_heads, void* o, float* lse, int64_t* edges,
                                  void* stream);

/* Vertical-Slash attention over the physical set of row i in query block
 * u = [a, e] (MInference page §2.1 "1x64 verticals, 64x64 slash tiles" and
 * §4.1 "verticals as points, slashes as intervals"):
 *   N(i) = ( ∪_{δ in D_h} [a-δ, e-δ]  ∪  C_h ) ∩ [0, i].
 * index: as written by msa_build_vs_index for the same `heads`.  Keys that a
 * whole 64-row query block leaves out of a key tile are masked on the tensor
 * core by adding -3.39e38 to their scores, so the raw scores q.k must stay
 * below 1e30 in magnitude (true for any finite bf16 inputs of ordinary
 * range); attended scores are not changed. */
MSA_API msa_status msa_attn_vs(const msa_shape* shape, const void* q, const void* k, const void* v, const int32_t* heads,
                       int32_t n_heads, int32_t block, const msa_vs_index* index, void* o, float* lse,
                       int64_t* edges, void* stream);

/* Block-Sparse attention (MInference page eq.(6)): row i of block u attends
 * the keys of blocks v in J_u with j <= i (the diagonal block is causal).
 * block_idx / block_cnt: as written by msa_build_block_index: for head slot x
 * and query block u, the first block_cnt[x][u] (clamped to [0, topk]) entries
 * of block_idx[x][u] are strictly ascending block ids in [0, u].  Entries that
 * break this are skipped by the kernel and the next msa_poll_device_status
 * returns MSA_ERR_INDEX (the output is then undefined). */
MSA_API msa_status msa_attn_block(const msa_shape* shape, const void* q, const void* k, const void* v,
                          const int32_t* heads, int32_t n_heads, int32_t block, int32_t topk,
                          const int32_t* block_idx, const int32_t* block_cnt, void* o, float* lse,
                          int64_t* edges, void* stream);

/* One layer's sparse prefill attention dispatched per head from the table
 * (MInference page §5.1 "head dispatch": each head reads its pattern, VS and
 * BS heads build their index online, then every head's sparse kernel runs).
 * table: host array of Hq entries.  All indices are built in `ws` (with both
 * kinds present, the Block-Sparse index on a side stream beside the
 * Vertical-Slash one, joined back into `stream`); then each
 * pattern's heads run in one attention launch of a kernel compiled for that
 * pattern, ordered longest-work-first.  When the table holds several
 * patterns, the Vertical-Slash launch runs on `stream` and the others on two
 * library-owned side streams forked from `stream` and joined back into it,
 * so the kernels share the SMs and later work on `stream` sees all of them.
 * No host synchronisation between index and attention. */
MSA_API msa_status msa_prefill_layer(const msa_shape* shape, const void* q, const void* k, const void* v,
                             const msa_head_cfg* table, void* o, float* lse, int64_t* edges, void* ws,
                             size_t ws_bytes, void* stream);

/* Merge of two attention results of the same query rows over disjoint key
 * sets (MInference page §3.2, eq.(7)-(8)): lse = log(e^{lse_a} + e^{lse_b}),
 * o = e^{lse_a - lse} o_a + e^{lse_b - lse} o_b per row, so a pattern computed
 * as separate key sets (verticals apart from slashes, chunks of the keys)
 * recombines into the single-pass result.  rows: number of query rows;
 * o_a, o_b, o: [rows, d_h] bf16 (o may alias o_a or o_b); lse_a, lse_b: [rows]
 * fp32 natural-log LSE as the attention calls return it (-inf: empty part);
 * lse: [rows] fp32 or NULL, must not alias lse_a / lse_b.  Errors:
 * MSA_ERR_INVALID_ARG (null or misaligned pointers, rows < 0, aliased lse),
 * MSA_ERR_UNSUPPORTED (d_h not 64/128). */
MSA_API msa_status msa_merge_attention(int64_t rows, int32_t d_h, const void* o_a, const float* lse_a,
                                       const void* o_b, const float* lse_b, void* o, float* lse, void* stream);

/* Captured dense mass per head (MInference page §5.1: the probability mass
 * outside the sparse set is dropped and the rest renormalised): for each of
 * `heads` rows-blocks of n query rows, mass[h] = (1/n) Σ_i e^{lse_sparse - lse_dense}
 * = the mean over rows of Σ_{j in N(i)} p_ij under the dense causal softmax p.
 * lse_sparse: [heads, n] LSE of the sparse layer; lse_dense: [heads, n] LSE of
 * msa_attn_dense on the same inputs; rows whose sparse set is empty count 0.
 * mass: [heads] fp32.  Deterministic (fixed summation order). */
MSA_API msa_status msa_captured_mass(int64_t heads, int64_t n, const float* lse_sparse, const float* lse_dense,
                                     float* mass, void* stream);

/* Chunked prefill (MInference page §5.2: a scheduler may cut a long prefill
 * into chunks so that it does not block short requests): msa_layer_attend
 * restricted to the query rows [row_begin, row_end) of every head; rows
 * outside are not written.  With the indices built once by msa_layer_index
 * over the whole sequence, the chunks, in any order, reproduce
 * msa_layer_attend's output and LSE bit for bit (each row meets the same
 * tiles in the same order); edges count only the chunk's rows.
 * row_begin: a multiple of 256; row_end: a multiple of 256 or n;
 * 0 <= row_begin < row_end <= n, else MSA_ERR_INVALID_ARG. */
MSA_API msa_status msa_layer_attend_rows(const msa_shape* shape, const void* q, const void* k, const void* v,
                                         const msa_head_cfg* table, void* o, float* lse, int64_t* edges, void* ws,
                                         size_t ws_bytes, int32_t row_begin, int32_t row_end, void* stream);

/* Varlen prefill: a batch of n_seqs sequences of different lengths, packed
 * without padding (cost-model page §2.2: a varlen kernel takes a cumulative
 * length array, processes only real tokens, and keeps every sample's windows
 * and tiles inside its own segment).  cu_seqlens: host array of n_seqs + 1
 * non-decreasing token offsets, cu_seqlens[0] = 0; sequence s has
 * n_s = cu_seqlens[s+1] - cu_seqlens[s] tokens (0 allowed: skipped).  Layout:
 * the sequences' tensors back to back, sequence s as one [H, n_s, d_h] block
 * starting at element H * cu_seqlens[s] * d_h (q, o: H = Hq; k, v: H = Hkv);
 * lse likewise as [Hq, n_s] blocks at Hq * cu_seqlens[s]; edges: [n_seqs, Hq]
 * counters (ADDED to).  shape gives Hq, Hkv, d_h and scale for every sequence
 * (its B and n are ignored).  Every sequence gets its own online indices and
 * its own attention (no index, window or tile reaches another sequence's
 * tokens), computed for the whole batch in one index pass and one attention
 * launch per 128 sequences; the workspace holds every sequence's indices.
 * Inputs must be finite: a key past a sequence's end that a tile covers is
 * weighted by exactly zero.  Requires ws_bytes >= msa_layer_varlen_workspace
 * (...) and Hq * total tokens < 2^31 (else MSA_ERR_UNSUPPORTED).  Errors:
 * invalid cu_seqlens -> MSA_ERR_INVALID_ARG before anything is launched. */
MSA_API size_t msa_layer_varlen_workspace(const msa_shape* shape, const msa_head_cfg* table,
                                          const int32_t* cu_seqlens, int32_t n_seqs);
MSA_API msa_status msa_prefill_layer_varlen(const msa_shape* shape, const int32_t* cu_seqlens, int32_t n_seqs,
                                            const void* q, const void* k, const void* v, const msa_head_cfg* table,
                                            void* o, float* lse, int64_t* edges, void* ws, size_t ws_bytes,
                                            void* stream);

/* Inspection (no counterpart in the pages): msa_layer_indices for sequence
 * `seq` of a msa_prefill_layer_varlen workspace (same shape, table and
 * cu_seqlens): where that call left the sequence's Vertical-Slash index (slot
 * = rank of the head among the table's VS heads) and Block-Sparse index
 * ([n_bs, ceil(n_s/64), topk] and counts).  MSA_ERR_INVALID_ARG for an empty
 * or out-of-range sequence.  Valid until the workspace is reused. */
MSA_API msa_status msa_layer_varlen_indices(const msa_shape* shape, const msa_head_cfg* table,
                                            const int32_t* cu_seqlens, int32_t n_seqs, void* ws, int32_t seq,
                                            msa_vs_index* vs, int32_t** block_idx, int32_t** block_cnt);

/* The two halves of msa_prefill_layer, in order (the time decomposition
 * T = T_index + T_sparse of the MInference page eq.(13)): msa_layer_index
 * builds every Vertical-Slash and Block-Sparse index of the table into `ws`;
 * msa_layer_attend then runs the attention launches that read them.
 * msa_prefill_layer(...) == msa_layer_index(...) followed by
 * msa_layer_attend(...) with the same workspace and stream. */
MSA_API msa_status msa_layer_index(const msa_shape* shape, const void* q, const void* k, const msa_head_cfg* table,
                                   void* ws, size_t ws_bytes, void* stream);
MSA_API msa_status msa_layer_attend(const msa_shape* shape, const void* q, const void* k, const void* v,
                                    const msa_head_cfg* table, void* o, float* lse, int64_t* edges, void* ws,
                                    size_t ws_bytes, void* stream);

/* msa_layer_attend with work counters (measurement; no counterpart in the
 * pages beyond the tile-padding accounting of the cost-model page §3): edges
 * as for msa_layer_attend, and tiles (nullable, [B*Hq] int64 device counters,
 * ADDED to): the number of 64-row x 128-key tiles each query head's rows were
 * processed in, so tiles * 8192 is the (row, key) area the tensor cores
 * covered for that head and E_h / (tiles * 8192) its useful fraction. */
MSA_API msa_status msa_layer_attend_stats(const msa_shape* shape, const void* q, const void* k, const void* v,
                                          const msa_head_cfg* table, void* o, float* lse, int64_t* edges,
                                          int64_t* tiles, void* ws, size_t ws_bytes, void* stream);

/* Failure-detection check (no counterpart in the pages): launches one thread
 * that waits on a barrier nothing arrives at, with the same bounded wait the
 * pipelines use but a limit of limit_ms (1..2000) milliseconds, so that the
 * next msa_poll_device_status returns MSA_ERR_DEVICE_TIMEOUT.  The context
 * stays usable.  Nothing faults, traps or hangs. */
MSA_API msa_status msa_check_wait_timeout(int32_t limit_ms, void* stream);

/* Number of kernels this process has launched through the library so far
 * (all devices; no counterpart in the pages).  Lets a caller count the launches inside a region. */
MSA_API uint64_t msa_kernel_launches(void);

/* Inspection (no counterpart in the pages).  Pointers into a
 * msa_prefill_layer workspace: where that call left the
 * Vertical-Slash index (slot = b * n_vs + rank of the head among the table's
 * VS heads) and the Block-Sparse index (likewise among BS heads).  Any
 * output pointer may be NULL.  Valid until the workspace is reused. */
MSA_API msa_status msa_layer_indices(const msa_shape* shape, const msa_head_cfg* table, void* ws, msa_vs_index* vs,
                             int32_t** block_idx, int32_t** block_cnt);

/* Expand the compact Vertical-Slash index of one slot into the explicit
 * per-query-block form of the MInference blog §2.3.3 (block count / block
 * ranges, column count / column indices) for blocks u_begin .. u_begin +
 * u_count - 1: merged inclusive key ranges ∪_{δ} [a-δ, e-δ] ∩ [0, e] and the
 * verticals c <= e not inside a range, ascending.  Device outputs:
 *   range_cnt[u_count], ranges[u_count][range_cap][2], col_cnt[u_count],
 *   cols[u_count][col_cap].  Entries beyond a cap are dropped and the count
 *   still reports the full number. */
MSA_API msa_status msa_vs_expand(const msa_shape* shape, const msa_vs_index* index, int32_t slot, int32_t u_begin,
                         int32_t u_count, int32_t range_cap, int32_t col_cap, int32_t* range_cnt,
                         int32_t* ranges, int32_t* col_cnt, int32_t* cols, void* stream);

/* Failure detection (no counterpart in the pages).  Synchronise `stream`,
 * read and clear the device error word of the current device.  Returns MSA_OK, MSA_ERR_DEVICE_TIMEOUT, MSA_ERR_INDEX or
 * MSA_ERR_CUDA. */
MSA_API msa_status msa_poll_device_status(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H */
