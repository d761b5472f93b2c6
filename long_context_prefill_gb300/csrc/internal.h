// Declarations shared by the library's translation units (host and device).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

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

// ------------------------------------------------------------ attention work units
// A sub-unit is a stream of 128-row query tiles of one pattern; its tile for
// item t is q-tile t * stride + offset.  Each tile has two 64-row halves: half
// h covers rows 128 * tile + row_off[h] .. +63 of query head qh[h] (batch
// folded into the head index).  A unit pairs two sub-units that read the same
// KV head: one CTA processes both tiles of an item against one shared K/V
// stream (the key tiles either needs).
enum UnitPattern : int32_t { kUnitAshape = 0, kUnitVS = 1, kUnitBlock = 2 };

struct SubUnit {
  int32_t qh[2];      // b * Hq + query head, per half
  int32_t row_off[2]; // 0 or 64
  int32_t slot[2];    // index slot per half (VS / BS)
  int32_t stride, offset;
  int32_t sink, window;  // A-shape
};
static_assert(sizeof(SubUnit) == 40, "SubUnit layout");

struct Unit {
  int32_t pattern;
  int32_t kvh;        // b * Hkv + kv head
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
  int32_t n, d, T, n_units;  // T: items per unit in this launch
  int32_t nqt;               // 128-row query tiles over n
  int32_t n_bands;           // bands in the unit table
  float scale_log2;  // scale * log2(e)
  const void* q;     // bf16 [B*Hq, n, d] (the kernel reads q, k, v through the TMA maps; the
  const void* k;     // pointers stay in the arguments: dropping them measured 1.5 % slower
  const void* v;     // code for the same work)
  void* o;           // bf16 [B*Hq, n, d]
  float* lse;        // [B*Hq, n] or null
  unsigned long long* edges;  // [B*Hq] or null
  unsigned long long* tiles;  // [B*Hq] or null: 64-row x 128-key tiles each query head was processed in
  // Vertical-Slash index (slot-indexed)
  const uint32_t* vs_dbits;  // [slots, words] bit δ of D
  const uint32_t* vs_cbits;  // [slots, words] bit j of C
  const uint32_t* vs_cover;  // [slots, cover_words] dilated slash coverage (see msa_vs_index)
  int32_t vs_words, vs_cover_words;
  // Block-Sparse index
  const int32_t* bs_idx;  // [slots, N_b, topk]
  const int32_t* bs_cnt;  // [slots, N_b]
  int32_t bs_topk, bs_nb;
  int* err;
  int32_t row_lo, row_hi;  // only items whose query rows lie in [row_lo, row_hi) run
};

// TMA views of the attention operands as [BH, n, d]: Q, K, V with boxes of
// 64 columns x 64 rows, and K, V again with 64 x 16 boxes (16-key segments).
struct AttnMaps {
  CUtensorMap q, k, v, k16, v16;
};

// Launch the attention engine over n_units units of T items each.
msa_status launch_attention(const AttnMaps& maps, const AttnArgs& args, const Unit* units, int n_units,
                            cudaStream_t stream);

// ------------------------------------------------------------ TMA tensor maps
// 3-D bf16 map over [BH, n, d] with a box of 64 columns x box_rows rows and
// 128-byte swizzle.  Returns false if the driver rejects it.
bool make_bf16_map(CUtensorMap* map, const void* base, int64_t BH, int64_t n, int64_t d, int box_rows);

// ------------------------------------------------------------ index builders
msa_status run_vs_index(const msa_shape& s, const void* q, const void* k, const int32_t* heads, int32_t n_heads,
                        const msa_head_cfg& cfg, const msa_vs_index& out, void* ws, size_t ws_bytes,
                        cudaStream_t stream);
size_t vs_index_ws_bytes(const msa_shape& s, const msa_head_cfg& cfg, int32_t n_heads);

msa_status run_block_index(const msa_shape& s, const void* q, const void* k, const int32_t* heads,
                           int32_t n_heads, int32_t topk, int32_t* block_idx, int32_t* block_cnt, void* ws,
                           size_t ws_bytes, cudaStream_t stream);
size_t block_index_ws_bytes(const msa_shape& s, int32_t n_heads);
// Bytes the listed heads need (their KV heads counted once; <= block_index_ws_bytes).
size_t block_index_ws_bytes_exact(const msa_shape& s, const int32_t* heads, int32_t n_heads);

inline int32_t ceil_div(int64_t a, int64_t b) { return (int32_t)((a + b - 1) / b); }

}  // namespace msa
