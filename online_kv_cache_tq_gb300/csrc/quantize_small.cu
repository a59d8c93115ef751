// Quantize-append for small batches (a decode step appends one token per
// sequence): one CTA of 512 threads per head vector.
//
// Same arithmetic as the other quantizers (甲子光年 article §2 第一階段 /
// 第二階段): n = ||x||, y = R x / n, nearest Lloyd-Max level, and for keys the
// rotated residual r' = R x - n c[code], its norm and the signs of S' r'.
// R^T and S'^T are read from global memory (L2-resident after first use), so
// a launch costs a few microseconds instead of staging 128 KB of constants
// per CTA.
#include <cuda_bf16.h>

#include "gemv512.cuh"
#include "kernels.h"

namespace tq {
namespace {

// Blocks [0, first.n_vec) quantize `first`, the rest `second` (K and V of one
// append in a single launch).  Thread (o, q) of the 512 works on rotated
// coordinate o; the four copies of o split the matrix-vector products and
// threads q == 0 (warps 0-3) write the results.
__global__ void __launch_bounds__(kGemvThreads) quantize_small_kernel(QuantizeArgs first, QuantizeArgs second,
                                                                      bool bf16) {
  __shared__ float x_s[kDim];
  __shared__ float r_s[kDim];
  __shared__ float red_s[4 * kDim];
  __shared__ float part_s[4];
  const bool in_first = static_cast<int>(blockIdx.x) < first.n_vec;
  const QuantizeArgs& a = in_first ? first : second;
  const int v = in_first ? blockIdx.x : blockIdx.x - first.n_vec;
  const int o = threadIdx.x & 127;
  const bool lead = threadIdx.x < 128;
  const int lane = o & 31;
  const int warp = o >> 5;
  const int token = v / a.n_kv;
  const int head = v - token * a.n_kv;

  const long long idx = static_cast<long long>(v) * kDim + o;
  const float x = bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(a.x)[idx])
                       : reinterpret_cast<const float*>(a.x)[idx];
  if (lead) x_s[o] = x;
  const float n = sqrtf(sum128(x * x, part_s));          // its barriers also publish x_s
  const float yv = gemv512(a.Rt, x_s, red_s);           // (R x)_o
  const float y = n > 0.f ? yv / n : 0.f;
  int code = 0;
  for (int t = 0; t + 1 < (1 << a.bits); ++t) code += (y > a.bounds[t]) ? 1 : 0;

  const long long cache_rows = static_cast<long long>(a.num_blocks) * a.block_size;
  const long long slot = a.slots[token];
  const bool ok = slot >= 0 && slot < cache_rows;
  if (slot >= cache_rows && threadIdx.x == 0) atomicCAS(a.error, 0, kErrSlot);
  const long long blk = ok ? slot / a.block_size : 0;
  const int off = ok ? static_cast<int>(slot - blk * a.block_size) : 0;
  const long long row = (blk * a.n_kv + head) * a.block_size + off;

  if (a.transposed) {
    if (ok && lead) {
      unsigned* words = reinterpret_cast<unsigned*>(a.codes);
      const unsigned mask = 1u << (off & 31);
      for (int p = 0; p < a.bits; ++p) {
        unsigned* w = words + transposed_word(blk, head, a.n_kv, a.bits, p, o, a.block_size, off);
        if ((code >> p) & 1) atomicOr(w, mask); else atomicAnd(w, ~mask);
      }
    }
  } else {
    for (int p = 0; p < a.bits; ++p) {
      const unsigned word = __ballot_sync(0xffffffffu, (code >> p) & 1);
      if (ok && lead && lane == 0) reinterpret_cast<unsigned*>(a.codes + row * (a.bits * 16))[p * 4 + warp] = word;
    }
  }
  if (ok && threadIdx.x == 0) a.norm[row] = n;

  if (a.qjl != nullptr) {
    const float r = fmaf(-n, a.levels[code], yv);
    if (lead) r_s[o] = r;
    const float gamma = sqrtf(sum128(r * r, part_s));    // its barriers also publish r_s
    const float z = gemv512(a.Spt, r_s, red_s);
    const unsigned word = __ballot_sync(0xffffffffu, z > 0.f);
    if (ok && lead && lane == 0) reinterpret_cast<unsigned*>(a.qjl + row * 16)[warp] = word;
    if (ok && threadIdx.x == 0) a.rnorm[row] = gamma;
  }
}

}  // namespace

cudaError_t launch_quantize_small(const QuantizeArgs* first, const QuantizeArgs* second, bool bf16,
                                  cudaStream_t stream) {
  const int n = (first ? first->n_vec : 0) + (second ? second->n_vec : 0);
  if (n <= 0) return cudaSuccess;
  QuantizeArgs none{};
  quantize_small_kernel<<<n, kGemvThreads, 0, stream>>>(first ? *first : none, second ? *second : none, bf16);
  return cudaGetLastError();
}

}  // namespace tq
