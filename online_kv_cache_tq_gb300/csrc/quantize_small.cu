// Quantize-append for small batches (a decode step appends one token per
// sequence): one CTA per head vector, thread o owns rotated coordinate o.
//
// Same arithmetic as the other quantizers (甲子光年 article §2 第一階段 /
// 第二階段): n = ||x||, y = R x / n, nearest Lloyd-Max level, and for keys the
// rotated residual r' = R x - n c[code], its norm and the signs of S' r'.
// R^T and S'^T are read from global memory (L2-resident after first use), so
// a launch costs a few microseconds instead of staging 128 KB of constants
// per CTA.
#include <cuda_bf16.h>

#include "kernels.h"

namespace tq {
namespace {

constexpr int kThreads = 128;

__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  const float s = (red[0] + red[1]) + (red[2] + red[3]);
  __syncthreads();
  return s;
}

// out[o] = sum_i w[i][o] * in[i] (w row-major [128][128]).
__device__ __forceinline__ float gemv_col(const float* __restrict__ w, const float* in) {
  const int o = threadIdx.x;
  float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
#pragma unroll 8
  for (int i = 0; i < kDim; i += 4) {
    acc0 = fmaf(__ldg(w + (i + 0) * kDim + o), in[i + 0], acc0);
    acc1 = fmaf(__ldg(w + (i + 1) * kDim + o), in[i + 1], acc1);
    acc2 = fmaf(__ldg(w + (i + 2) * kDim + o), in[i + 2], acc2);
    acc3 = fmaf(__ldg(w + (i + 3) * kDim + o), in[i + 3], acc3);
  }
  return (acc0 + acc1) + (acc2 + acc3);
}

// Blocks [0, first.n_vec) quantize `first`, the rest `second` (K and V of one
// append in a single launch).
__global__ void __launch_bounds__(kThreads) quantize_small_kernel(QuantizeArgs first, QuantizeArgs second,
                                                                  bool bf16) {
  __shared__ float x_s[kDim];
  __shared__ float r_s[kDim];
  __shared__ float red_s[4];
  const bool in_first = static_cast<int>(blockIdx.x) < first.n_vec;
  const QuantizeArgs& a = in_first ? first : second;
  const int v = in_first ? blockIdx.x : blockIdx.x - first.n_vec;
  const int o = threadIdx.x;
  const int lane = o & 31;
  const int warp = o >> 5;
  const int token = v / a.n_kv;
  const int head = v - token * a.n_kv;

  const long long idx = static_cast<long long>(v) * kDim + o;
  const float x = bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(a.x)[idx])
                       : reinterpret_cast<const float*>(a.x)[idx];
  x_s[o] = x;
  const float n = sqrtf(block_sum(x * x, red_s));
  const float yv = gemv_col(a.Rt, x_s);                 // (R x)_o, synchronised by block_sum above
  const float y = n > 0.f ? yv / n : 0.f;
  int code = 0;
  for (int t = 0; t + 1 < (1 << a.bits); ++t) code += (y > a.bounds[t]) ? 1 : 0;

  const long long cache_rows = static_cast<long long>(a.num_blocks) * a.block_size;
  const long long slot = a.slots[token];
  const bool ok = slot >= 0 && slot < cache_rows;
  if (slot >= cache_rows && o == 0) atomicCAS(a.error, 0, kErrSlot);
  const long long blk = ok ? slot / a.block_size : 0;
  const int off = ok ? static_cast<int>(slot - blk * a.block_size) : 0;
  const long long row = (blk * a.n_kv + head) * a.block_size + off;

  if (a.transposed) {
    if (ok) {
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
      if (ok && lane == 0) reinterpret_cast<unsigned*>(a.codes + row * (a.bits * 16))[p * 4 + warp] = word;
    }
  }
  if (ok && o == 0) a.norm[row] = n;

  if (a.qjl != nullptr) {
    const float r = fmaf(-n, a.levels[code], yv);
    r_s[o] = r;
    const float gamma = sqrtf(block_sum(r * r, red_s));
    const float z = gemv_col(a.Spt, r_s);
    const unsigned word = __ballot_sync(0xffffffffu, z > 0.f);
    if (ok && lane == 0) reinterpret_cast<unsigned*>(a.qjl + row * 16)[warp] = word;
    if (ok && o == 0) a.rnorm[row] = gamma;
  }
}

}  // namespace

cudaError_t launch_quantize_small(const QuantizeArgs* first, const QuantizeArgs* second, bool bf16,
                                  cudaStream_t stream) {
  const int n = (first ? first->n_vec : 0) + (second ? second->n_vec : 0);
  if (n <= 0) return cudaSuccess;
  QuantizeArgs none{};
  quantize_small_kernel<<<n, kThreads, 0, stream>>>(first ? *first : none, second ? *second : none, bf16);
  return cudaGetLastError();
}

}  // namespace tq
