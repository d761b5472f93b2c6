// Block-Sparse online index (placeholder until the pooling kernels land).
#include "internal.h"

namespace msa {
size_t block_index_ws_bytes(const msa_shape& s, int32_t n_heads) { return 256; }
msa_status run_block_index(const msa_shape& s, const void* q, const void* k, const int32_t* heads,
                           int32_t n_heads, int32_t topk, int32_t* block_idx, int32_t* block_cnt, void* ws,
                           size_t ws_bytes, cudaStream_t stream) {
  return MSA_ERR_UNSUPPORTED;
}
}  // namespace msa
