// Reconstruction-error monitor: how far the stage-1 reconstructions held in
// the cache are from the vectors they encode (intelliparadigm.com §3.3 keeps
// a running mean of ||original - quantized||_2 to watch a deployment; 甲子光年
// article §2 第一階段 defines the reconstruction n R^T c[code]).
//
// One warp per head vector, eight per 256-thread CTA: lane l holds rotated
// coordinates l + 32 k.  ||x - n R^T c|| = ||R x - n c|| (R is orthogonal),
// so the warp computes y = R x (R^T read from global memory, L1/L2-resident),
// reads the vector's codes and stored norm from the cache, and accumulates
// ||y - n c||, its square, ||x||^2 and the count into four doubles.
#include <cuda_bf16.h>

#include "kernels.h"

namespace tq {
namespace {

constexpr int kMonWarps = 8;

__global__ void __launch_bounds__(32 * kMonWarps) monitor_kernel(QuantizeArgs a, bool bf16, double* stats) {
  __shared__ float x_s[kMonWarps][kDim];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int v = blockIdx.x * kMonWarps + warp;
  if (v >= a.n_vec) return;                     // (no block-wide barrier below)
  const int token = v / a.n_kv, head = v - token * a.n_kv;
  const long long slot = a.slots[token];
  const long long cache_rows = static_cast<long long>(a.num_blocks) * a.block_size;
  if (slot < 0 || slot >= cache_rows) return;   // skipped tokens have no cache row
  const long long blk = slot / a.block_size;
  const int off = static_cast<int>(slot - blk * a.block_size);
  const long long row = (blk * a.n_kv + head) * a.block_size + off;

  float xx = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const long long idx = static_cast<long long>(v) * kDim + lane + 32 * k;
    const float x = bf16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(a.x)[idx])
                         : reinterpret_cast<const float*>(a.x)[idx];
    x_s[warp][lane + 32 * k] = x;
    xx = fmaf(x, x, xx);
  }
  __syncwarp();
  float y[4] = {0.f, 0.f, 0.f, 0.f};
  for (int i = 0; i < kDim; ++i) {
    const float xi = x_s[warp][i];
#pragma unroll
    for (int k = 0; k < 4; ++k) y[k] = fmaf(__ldg(a.Rt + i * kDim + lane + 32 * k), xi, y[k]);
  }
  const float n = load_norm(a.norm, row, a.norm16);
  float rr = 0.f;
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const int o = lane + 32 * k;
    int code = 0;
    for (int p = 0; p < a.bits; ++p) {
      unsigned w;
      if (a.transposed) {
        w = reinterpret_cast<const unsigned*>(a.codes)[transposed_word(blk, head, a.n_kv, a.bits, p, o, a.block_size,
                                                                       off)] >> (off & 31);
      } else {
        w = reinterpret_cast<const unsigned*>(a.codes + row * (a.bits * 16))[p * 4 + (o >> 5)] >> (o & 31);
      }
      code |= static_cast<int>(w & 1u) << p;
    }
    const float r = fmaf(-n, a.levels[code], y[k]);
    rr = fmaf(r, r, rr);
  }
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) {
    rr += __shfl_xor_sync(0xffffffffu, rr, s);
    xx += __shfl_xor_sync(0xffffffffu, xx, s);
  }
  if (lane == 0) {
    atomicAdd(stats + 0, sqrt(static_cast<double>(rr)));
    atomicAdd(stats + 1, static_cast<double>(rr));
    atomicAdd(stats + 2, static_cast<double>(xx));
    atomicAdd(stats + 3, 1.0);
  }
}

}  // namespace

cudaError_t launch_monitor(const QuantizeArgs& a, bool bf16, double* stats, cudaStream_t stream) {
  if (a.n_vec <= 0) return cudaSuccess;
  monitor_kernel<<<(a.n_vec + kMonWarps - 1) / kMonWarps, 32 * kMonWarps, 0, stream>>>(a, bf16, stats);
  return cudaGetLastError();
}

}  // namespace tq
