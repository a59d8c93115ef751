// 128 x 128 matrix-vector product and reductions for the per-vector kernels
// of one decode step: THREADS = 128 * copies threads, thread (o, q =
// threadIdx.x / 128) working on output o.
#pragma once

namespace tq {

constexpr int kGemvThreads = 512;   // merge: four threads per coordinate
constexpr int kVecThreads = 256;    // append and query preparation: two threads per coordinate

// out[o] = sum_i w[i * 128 + o] * in_s[i] for o = threadIdx.x % 128.  Thread
// (o, q) sums the 128 / copies terms i in [q * 128 / copies, ...) in batches of
// 32 loads in flight at once, and the partial sums meet in red_s ([copies][128]
// floats).  Every thread returns out[o]; in_s must be visible to all threads
// before the call, and red_s is free again on return.
template <int THREADS>
__device__ __forceinline__ float gemv(const float* __restrict__ w, const float* in_s, float* red_s) {
  constexpr int kCopies = THREADS / 128, kTerms = 128 / kCopies;
  const int o = threadIdx.x & 127, q = threadIdx.x >> 7;
  float acc0 = 0.f, acc1 = 0.f, acc2 = 0.f, acc3 = 0.f;
#pragma unroll
  for (int k0 = 0; k0 < kTerms; k0 += 32) {
    const float* wp = w + (kTerms * q + k0) * 128 + o;
    float v[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) v[k] = __ldg(wp + k * 128);
    const float* x = in_s + kTerms * q + k0;
#pragma unroll
    for (int k = 0; k < 32; k += 4) {
      acc0 = fmaf(v[k + 0], x[k + 0], acc0);
      acc1 = fmaf(v[k + 1], x[k + 1], acc1);
      acc2 = fmaf(v[k + 2], x[k + 2], acc2);
      acc3 = fmaf(v[k + 3], x[k + 3], acc3);
    }
  }
  red_s[q * 128 + o] = (acc0 + acc1) + (acc2 + acc3);
  __syncthreads();
  float r = red_s[o];
#pragma unroll
  for (int c = 1; c < kCopies; ++c) r += red_s[c * 128 + o];
  __syncthreads();
  return r;
}

// Sum of v over the 128 values o (each held by threads o, o + 128, ...): the
// first four warps reduce into part_s ([4] floats); every thread gets the sum.
__device__ __forceinline__ float sum128(float v, float* part_s) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  if (threadIdx.x < 128 && (threadIdx.x & 31) == 0) part_s[threadIdx.x >> 5] = v;
  __syncthreads();
  const float s = (part_s[0] + part_s[1]) + (part_s[2] + part_s[3]);
  __syncthreads();
  return s;
}

}  // namespace tq
