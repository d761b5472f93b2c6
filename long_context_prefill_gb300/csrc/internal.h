// Declarations shared by the library's translation units (host and device).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <vector>

#include "../../include/msa.h"

namespace msa {

// ------------------------------------------------------------ device error word
// Set (first error wins) by kernels whose bounded wait timed out or that saw an
// out-of-range index; read and cleared by msa_poll_device_status().
enum DeviceError : int { kErrNone = 0, kErrTimeout = 1, kErrIndex = 2 };
int* device_error_word();  // device address of the current device's error word

// Kernel launches made through the library (process-wide counter).
void note_launch();
uint64_t launch_count();

// ------------------------------------------------------------ sequences of a launch
// A launch covers up to kMaxSeqs sequences: a uniform batch is B sequences of
// n tokens, a varlen batch takes its lengths from cu_seqlens.  Token i of head
// h of sequence s is row H * tok0 + h * n + i of the [rows, d_h] view of q, k,
// v and o (H = Hq or Hkv), which for a uniform batch is the [B, H, n, d_h]
// layout.  Every per-(sequence, head) array is sequence-major: the entries of
// sequence s follow those of the sequences before it (the prefix sums below)
// and head x of s sits at x times the sequence's own size, so a uniform batch
// keeps the plain [slots, size] layout.
constexpr int kMaxSeqs = 128;

struct SeqInfo {
  int32_t n, tok0;      // tokens, first token (cu_seqlens[s])
  int32_t word0;        // Σ ceil(n/32) over the sequences before (bitmaps)
  int32_t cword0;       // Σ ceil((n+63)/32) (slash-cover maps)
  int32_t nb0;          // Σ ceil(n/64) (query / key blocks)
  int32_t kb0;          // Σ (4 ceil(n/128) + LB) (Vertical-Slash diagonal bins)
  int32_t item0, T;     // attention items before this sequence; items per unit
  int32_t chunk0, chunks;  // Vertical-Slash proxy CTAs before; CTAs per pack of this sequence
  int32_t sc0;          // Block-Sparse score CTAs before (query-block tiles of 128)
  int32_t seq;          // index of the sequence in its batch (edge and tile counters, index slots)
  int32_t blk0;         // blocks of the sequences before it in this launch's table (flat block grids)
  int32_t pad;
  int64_t tri0;         // Σ nb (nb + 1) / 2 (packed block-score triangles)
};
static_assert(sizeof(SeqInfo) == 64, "SeqInfo layout");

struct SeqTable {
  int32_t count, pad;
  SeqInfo s[kMaxSeqs];
};

__host__ __device__ inline int32_t n_words(int32_t n) { return (n + 31) / 32; }
__host__ __device__ inline int32_t n_cover_words(int32_t n) { return (n + 63 + 31) / 32; }
__host__ __device__ inline int32_t n_blocks(int32_t n) { return (n + 63) / 64; }
__host__ __device__ inline int32_t n_tiles(int32_t n) { return (n + 127) / 128; }

// Index of the sequence holding flat index x, given each sequence's first
// index first(s) (non-decreasing): the last s with first(s) <= x.
template <class F>
__host__ __device__ inline int seq_search(int count, F first, int64_t x) {
  int lo = 0, hi = count - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) / 2;
    if ((int64_t)first(mid) <= x) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// ------------------------------------------------------------ attention work units
// A sub-unit is a stream of 128-row query tiles of one pattern; its tile for
// item t is q-tile t * stride + offset.  Each tile has two 64-row halves: half
// h covers rows 128 * tile + row_off[h] .. +63 of query head qh[h].  Units
// describe one sequence; a launch runs them for every sequence of its
// SeqTable.  A unit pairs two sub-units that read the same
// KV head: one CTA processes both tiles of an item against one shared K/V
// stream (the key tiles either needs).
enum UnitPattern : int32_t { kUnitAshape = 0, kUnitVS = 1, kUnitBlock = 2 };

struct SubUnit {
  int32_t qh[2];      // query head (within its sequence), per half
  int32_t row_off[2]; // 0 or 64
  int32_t slot[2];    // index slot per half within its sequence (VS / BS)
  int32_t stride, offset;
  int32_t sink, window;  // A-shape
};
static_assert(sizeof(SubUnit) == 40, "SubUnit layout");

struct Unit {
  int32_t pattern;
  int32_t kvh;        // kv head (within its sequence)
  int32_t has1;       // sub-unit 1 present
  int32_t pad;
  SubUnit sub[2];
};
static_assert(sizeof(Unit) == 96, "Unit layout");

constexpr int kMaxUnits = 64;
// Units sorted by KV head; band b is units [band[b], band[b+1]).  A launch
// runs the bands one after another (items of a band by descending t), so the
// CTAs resident at any time read few KV heads and their keys stay in L2.
struct UnitTable {
  Unit u[kMaxUnits];
  int32_t band[kMaxUnits + 1];
};

struct AttnArgs {
  int32_t d, n_units;        // items per unit come from each sequence's SeqInfo.T
  int32_t Hq, Hkv;           // heads per sequence (row views: row = H * tok0 + h * n + i)
  int32_t n_bands;           // bands in the unit table
  float scale_log2;  // scale * log2(e)
  const void* q;     // bf16 rows (the kernel reads q, k, v through the TMA maps; the
  const void* k;     // pointers stay in the arguments: dropping them measured 1.5 % slower
  const void* v;     // code for the same work)
  void* o;           // bf16 rows, as q
  float* lse;        // [rows of q] or null
  unsigned long long* edges;  // [sequences * Hq] or null
  unsigned long long* tiles;  // [sequences * Hq] or null: 64-row x 128-key tiles each query head was processed in
  // Vertical-Slash index (sequence-major, vs_nslots slots per sequence)
  const uint32_t* vs_dbits;  // words per slot: bit δ of D
  const uint32_t* vs_cbits;  // words per slot: bit j of C
  const uint32_t* vs_cover;  // cover words per slot: dilated slash coverage (see msa_vs_index)
  int32_t vs_nslots, bs_nslots;
  // Block-Sparse index (sequence-major, bs_nslots slots per sequence)
  const int32_t* bs_idx;  // [blocks of the slot, topk] per slot
  const int32_t* bs_cnt;  // [blocks of the slot] per slot
  int32_t bs_topk, pad;
  int* err;
  int32_t row_lo, row_hi;  // only items whose query rows lie in [row_lo, row_hi) run
};

// TMA views of the attention operands as [rows, d] (one row per token and
// head): Q, K, V with boxes of 64 columns x 64 rows, and K, V again with
// 64 x 16 boxes (16-key segments).
struct AttnMaps {
  CUtensorMap q, k, v, k16, v16;
};

// Launch the attention engine over n_units units per sequence of the table
// (each sequence's T items per unit; fills item0 and T of every entry).
// Two non-blocking side streams and three events per device, made on first
// use (null when they cannot be made): work that may run beside the caller's
// stream forks onto them from an event and joins back with another.  A caller
// holds `mu` while it records, waits and enqueues, so that calls from several
// host threads do not interleave their forks on the shared events.
struct SideStreams {
  cudaStream_t side[2];
  cudaEvent_t ev[3];
  bool ok;
  std::mutex mu;
};
SideStreams* side_streams();

msa_status launch_attention(const AttnMaps& maps, const AttnArgs& args, const Unit* units, int n_units,
                            SeqTable& seqs, cudaStream_t stream);

// ------------------------------------------------------------ host helpers (api.cu)
std::vector<SeqInfo> build_seqs(const int32_t* lens, int n_seqs, int LB);
std::vector<SeqInfo> uniform_seqs(const msa_shape& s, int LB);
bool rows_fit(int64_t H, const std::vector<SeqInfo>& seqs);
void ashape_units(const msa_shape& s, const int32_t* heads, int32_t nh, const int32_t* sink, const int32_t* window,
                  std::vector<Unit>& out);
void vs_units(const msa_shape& s, const int32_t* heads, int32_t nh, std::vector<Unit>& out);
void block_units(const msa_shape& s, const int32_t* heads, int32_t nh, std::vector<Unit>& out);
// Attention over the units for every sequence (a uniform batch when seqs is null).
msa_status attention(const msa_shape& s, const void* q, const void* k, const void* v, void* o, float* lse,
                     int64_t* edges, const std::vector<Unit>& units, const AttnArgs& idx, cudaStream_t stream,
                     int32_t row_lo = 0, int32_t row_hi = 0x7FFFFFFF, int64_t* tiles = nullptr,
                     const std::vector<SeqInfo>* seqs = nullptr);

// ------------------------------------------------------------ TMA tensor maps
// 3-D bf16 map over [BH, n, d] with a box of 64 columns x box_rows rows and
// 128-byte swizzle.  Returns false if the driver rejects it.
bool make_bf16_map(CUtensorMap* map, const void* base, int64_t BH, int64_t n, int64_t d, int box_rows);

// ------------------------------------------------------------ index builders
// Both builders index every sequence of `seqs` (token order; a uniform batch
// when null) in one pass: outputs and workspace regions are sequence-major
// (slot = sequence * n_heads + rank of the head; see SeqInfo).
msa_status run_vs_index(const msa_shape& s, const void* q, const void* k, const int32_t* heads, int32_t n_heads,
                        const msa_head_cfg& cfg, const msa_vs_index& out, void* ws, size_t ws_bytes,
                        cudaStream_t stream, const std::vector<SeqInfo>* seqs = nullptr);
// Workspace of run_vs_index: for the listed heads (heads may be null: the
// worst case, every head in its own KV group).
size_t vs_index_ws_bytes(const msa_shape& s, const msa_head_cfg& cfg, const int32_t* heads, int32_t n_heads,
                         const std::vector<SeqInfo>* seqs = nullptr);

msa_status run_block_index(const msa_shape& s, const void* q, const void* k, const int32_t* heads,
                           int32_t n_heads, int32_t topk, int32_t* block_idx, int32_t* block_cnt, void* ws,
                           size_t ws_bytes, cudaStream_t stream, const std::vector<SeqInfo>* seqs = nullptr);
size_t block_index_ws_bytes(const msa_shape& s, int32_t n_heads, const std::vector<SeqInfo>* seqs = nullptr);
// Bytes the listed heads need (their KV heads counted once; <= block_index_ws_bytes).
size_t block_index_ws_bytes_exact(const msa_shape& s, const int32_t* heads, int32_t n_heads,
                                  const std::vector<SeqInfo>* seqs = nullptr);

inline int32_t ceil_div(int64_t a, int64_t b) { return (int32_t)((a + b - 1) / b); }

}  // namespace msa
