// Vertical-Slash online index (placeholder until the proxy kernels land).
#include "internal.h"

namespace msa {
size_t vs_index_ws_bytes(const msa_shape& s, const msa_head_cfg& cfg, int32_t n_heads) { return 256; }
msa_status run_vs_index(const msa_shape& s, const void* q, const void* k, const int32_t* heads, int32_t n_heads,
                        const msa_head_cfg& cfg, const msa_vs_index& out, void* ws, size_t ws_bytes,
                        cudaStream_t stream) {
  return MSA_ERR_UNSUPPORTED;
}
}  // namespace msa

extern "C" msa_status msa_vs_expand(const msa_shape* shape, const msa_vs_index* index, int32_t slot, int32_t u_begin,
                                    int32_t u_count, int32_t range_cap, int32_t col_cap, int32_t* range_cnt,
                                    int32_t* ranges, int32_t* col_cnt, int32_t* cols, void* stream) {
  return MSA_ERR_UNSUPPORTED;
}
