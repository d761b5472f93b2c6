// Merge of two attention results over disjoint key sets of the same query
// rows (MInference page §3.2, eq.(7)-(8): partial softmax states combine
// through their maxima and sums).  With lse = log Σ e^{s} of each part,
//   lse = log(e^{lse_a} + e^{lse_b}),  o = e^{lse_a - lse} o_a + e^{lse_b - lse} o_b,
// so a pattern split into separately computed key sets (verticals apart
// from slashes, or the chunks of a key range) recombines exactly.  An empty
// part (lse = -inf) contributes nothing; two empty parts give o = 0, -inf.
#include <cuda_bf16.h>
#include <math.h>

#include "internal.h"

namespace msa {

namespace {

// 8 columns (16 bytes) per thread, D / 8 threads per row.
template <int D>
__global__ void __launch_bounds__(256) merge_kernel(const __nv_bfloat16* oa, const float* la, const __nv_bfloat16* ob,
                                                    const float* lb, __nv_bfloat16* o, float* lo, int64_t rows) {
  constexpr int kTPR = D / 8;
  const int64_t idx = blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
  const int64_t r = idx / kTPR;
  const int c = (int)(idx % kTPR) * 8;
  if (r >= rows) return;
  const float a = la[r], b = lb[r];
  const float m = fmaxf(a, b);
  float wa = 0.f, wb = 0.f, l = -INFINITY;
  if (m != -INFINITY) {
    wa = expf(a - m);
    wb = expf(b - m);
    const float s = wa + wb;
    l = m + logf(s);
    wa /= s;
    wb /= s;
  }
  const uint4 xa = *reinterpret_cast<const uint4*>(oa + r * D + c);
  const uint4 xb = *reinterpret_cast<const uint4*>(ob + r * D + c);
  const __nv_bfloat162* pa = reinterpret_cast<const __nv_bfloat162*>(&xa);
  const __nv_bfloat162* pb = reinterpret_cast<const __nv_bfloat162*>(&xb);
  uint4 y;
  __nv_bfloat162* py = reinterpret_cast<__nv_bfloat162*>(&y);
#pragma unroll
  for (int x = 0; x < 4; ++x) {
    const float2 fa = __bfloat1622float2(pa[x]), fb = __bfloat1622float2(pb[x]);
    py[x] = __floats2bfloat162_rn(wa * fa.x + wb * fb.x, wa * fa.y + wb * fb.y);
  }
  *reinterpret_cast<uint4*>(o + r * D + c) = y;
  if (c == 0 && lo) lo[r] = l;
}

}  // namespace

}  // namespace msa

using namespace msa;

extern "C" msa_status msa_merge_attention(int64_t rows, int32_t d_h, const void* o_a, const float* lse_a,
                                          const void* o_b, const float* lse_b, void* o, float* lse, void* stream) {
  if (rows < 0 || (d_h != 64 && d_h != 128)) return rows < 0 ? MSA_ERR_INVALID_ARG : MSA_ERR_UNSUPPORTED;
  if (!o_a || !lse_a || !o_b || !lse_b || !o) return MSA_ERR_INVALID_ARG;
  for (const void* p : {o_a, o_b, static_cast<const void*>(o)})
    if (reinterpret_cast<uintptr_t>(p) % 16) return MSA_ERR_INVALID_ARG;
  for (const float* p : {lse_a, lse_b, static_cast<const float*>(lse)})
    if (p && reinterpret_cast<uintptr_t>(p) % 4) return MSA_ERR_INVALID_ARG;
  if (lse && (lse == lse_a || lse == lse_b)) return MSA_ERR_INVALID_ARG;  // every thread of a row reads the inputs
  if (rows == 0) return MSA_OK;
  const int64_t threads = rows * (d_h / 8);
  const int64_t blocks = (threads + 255) / 256;
  if (blocks > 0x7FFFFFFF) return MSA_ERR_UNSUPPORTED;
  cudaStream_t s = (cudaStream_t)stream;
  if (d_h == 128)
    merge_kernel<128><<<(unsigned)blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(o_a), lse_a,
                                                        static_cast<const __nv_bfloat16*>(o_b), lse_b,
                                                        static_cast<__nv_bfloat16*>(o), lse, rows);
  else
    merge_kernel<64><<<(unsigned)blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(o_a), lse_a,
                                                       static_cast<const __nv_bfloat16*>(o_b), lse_b,
                                                       static_cast<__nv_bfloat16*>(o), lse, rows);
  note_launch();
  return cudaGetLastError() == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}

// ------------------------------------------------------------------ captured mass
// Share of each row's dense softmax mass that the sparse set keeps (MInference
// page §5.1: the probability outside the candidates is dropped and the rest
// renormalised): Σ_{j in N(i)} e^{s_ij} / Σ_{j <= i} e^{s_ij} = e^{lse_sparse(i)
// - lse_dense(i)}.  One CTA per head averages it over the head's rows in a
// fixed order (deterministic).
namespace msa {
namespace {
__global__ void __launch_bounds__(256) captured_mass_kernel(const float* ls, const float* ld, int64_t n, float* mass) {
  __shared__ double part[256];
  const int64_t h = blockIdx.x;
  double acc = 0.0;
  for (int64_t i = threadIdx.x; i < n; i += 256) {
    const float a = ls[h * n + i], b = ld[h * n + i];
    if (a != -INFINITY && b != -INFINITY) acc += (double)expf(a - b);
  }
  part[threadIdx.x] = acc;
  __syncthreads();
  for (int s = 128; s > 0; s >>= 1) {
    if ((int)threadIdx.x < s) part[threadIdx.x] += part[threadIdx.x + s];
    __syncthreads();
  }
  if (threadIdx.x == 0) mass[h] = (float)(part[0] / (double)n);
}
}  // namespace
}  // namespace msa

extern "C" msa_status msa_captured_mass(int64_t heads, int64_t n, const float* lse_sparse, const float* lse_dense,
                                        float* mass, void* stream) {
  if (heads < 0 || n < 1 || !lse_sparse || !lse_dense || !mass) return MSA_ERR_INVALID_ARG;
  for (const float* p : {lse_sparse, lse_dense, static_cast<const float*>(mass)})
    if (reinterpret_cast<uintptr_t>(p) % 4) return MSA_ERR_INVALID_ARG;
  if (heads == 0) return MSA_OK;
  if (heads > 0x7FFFFFFF) return MSA_ERR_UNSUPPORTED;
  msa::captured_mass_kernel<<<(unsigned)heads, 256, 0, (cudaStream_t)stream>>>(lse_sparse, lse_dense, n, mass);
  msa::note_launch();
  return cudaGetLastError() == cudaSuccess ? MSA_OK : MSA_ERR_CUDA;
}
