// Block-Sparse index builder that allocates nothing: its scratch is a
// file-scope device array instead of a caller-provided workspace.
//
// Callers this serves: code that holds device tensors some other runtime
// allocated and has no device allocator of its own to size and create a
// workspace (a C host program driving the library from another framework's
// buffers), or that must not call cudaMalloc/cudaFree on its path because
// those calls synchronise the device and stall the other runtime's streams.
//
// The array is shared by every call on a device: calls that overlap in time
// (different streams without ordering between them, or different host
// threads) race on it.  Issue them on one stream or order them with events.
#include <atomic>

#include "internal.h"

namespace msa {

// Holds the pooled block means and the packed block-score triangle of one call
// (the same regions the workspace of msa_build_block_index holds).  Every
// region is fully written before it is read, so nothing is cleared.
static __device__ __align__(256) uint8_t g_block_index_scratch[MSA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
static std::atomic<void*> g_scratch_addr[kMaxDevices];

// Device address of the scratch on the current device, looked up once per
// device (with that device current).  The first call on a device performs the
// lookup, so it should come before any work a caller wants free of runtime
// set-up calls.  The cache is keyed by device ordinal only: after a
// cudaDeviceReset (or any teardown of the device's primary context) in the
// same process the cached address is stale, and this entry point must not be
// called again on that device.
static void* scratch_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    if (cudaGetSymbolAddress(&p, g_block_index_scratch) != cudaSuccess) return nullptr;
    g_scratch_addr[dev].store(p, std::memory_order_release);
  }
  return p;
}

msa_status check_shape(const msa_shape* s);
msa_status check_heads(const int32_t* heads, int32_t n_heads, int32_t Hq);

}  // namespace msa

using namespace msa;

extern "C" {

msa_status msa_build_block_index_static(const msa_shape* shape, const void* q, const void* k, const int32_t* heads,
                                        int32_t n_heads, int32_t block, int32_t topk, int32_t* block_idx,
                                        int32_t* block_cnt, void* stream) {
  msa_status st = check_shape(shape);
  if (st != MSA_OK) return st;
  if ((st = check_heads(heads, n_heads, shape->Hq)) != MSA_OK) return st;
  if (!q || !k || !block_idx || !block_cnt) return MSA_ERR_INVALID_ARG;
  if (topk < 1) return MSA_ERR_INVALID_ARG;
  if (block != 64) return MSA_ERR_UNSUPPORTED;
  // what these heads need: each KV head they read is pooled once
  const size_t need = block_index_ws_bytes_exact(*shape, heads, n_heads);
  if (need > (size_t)MSA_STATIC_SCRATCH_BYTES) return MSA_ERR_WORKSPACE_TOO_SMALL;
  void* ws = scratch_address();
  if (!ws) return MSA_ERR_CUDA;
  return run_block_index(*shape, q, k, heads, n_heads, topk, block_idx, block_cnt, ws, MSA_STATIC_SCRATCH_BYTES,
                         (cudaStream_t)stream);
}

}  // extern "C"
