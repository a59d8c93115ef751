// SIMT quantize-append: the fp32 CUDA-core reference path of the write side.
//
// Per head vector x (甲子光年 article §2 第一階段 / 第二階段):
//   n = ||x||, y = R x / n, code_j = #{i : t_i < y_j} (nearest Lloyd-Max level),
//   codes stored as bit-planes; for keys additionally the rotated residual
//   r' = R x - n c[code] (= R (x - x_hat)), its norm, and the signs of S' r'
//   (S' = S R^T, so S' r' = S (x - x_hat): intelliparadigm.com §2.1.2).
//
// One CTA of 128 threads holds R^T (and S'^T) in shared memory and walks
// 32-vector tiles: a register-tiled fp32 GEMM (thread o owns output row o of
// all 32 vectors), then one warp per vector for norm, codes, ballot-packed
// planes and the residual.  Lane l of that warp owns coordinates l, l+32,
// l+64, l+96, so ballot i of plane p is exactly word i of the stored plane.
#include <cuda_bf16.h>

#include "kernels.h"

namespace tq {
namespace {

constexpr int kTile = 32;
constexpr int kThreads = 128;

__device__ __forceinline__ float load_elem(const void* base, long long idx, bool bf16) {
  if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
  return reinterpret_cast<const float*>(base)[idx];
}

// out[v][o] = sum_i in[v][i] * w[i][o] for the 32 vectors of a tile.
__device__ __forceinline__ void tile_gemm(const float* in, const float* w, float* out) {
  const int o = threadIdx.x;
  float acc[kTile];
#pragma unroll
  for (int v = 0; v < kTile; ++v) acc[v] = 0.f;
  for (int i = 0; i < kDim; i += 4) {
    const float w0 = w[(i + 0) * kDim + o];
    const float w1 = w[(i + 1) * kDim + o];
    const float w2 = w[(i + 2) * kDim + o];
    const float w3 = w[(i + 3) * kDim + o];
#pragma unroll
    for (int v = 0; v < kTile; ++v) {
      const float4 xv = *reinterpret_cast<const float4*>(in + v * kDim + i);
      float a = acc[v];
      a = fmaf(xv.x, w0, a);
      a = fmaf(xv.y, w1, a);
      a = fmaf(xv.z, w2, a);
      a = fmaf(xv.w, w3, a);
      acc[v] = a;
    }
  }
#pragma unroll
  for (int v = 0; v < kTile; ++v) out[v * kDim + o] = acc[v];
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

__global__ void __launch_bounds__(kThreads) quantize_simt_kernel(QuantizeArgs a, bool bf16) {
  extern __shared__ __align__(16) float smem[];
  const bool qjl = a.qjl != nullptr;
  float* rt_s = smem;
  float* spt_s = rt_s + kDim * kDim;
  float* x_s = qjl ? spt_s + kDim * kDim : spt_s;
  float* y_s = x_s + kTile * kDim;
  __shared__ float lev_s[kMaxLevels];
  __shared__ float bnd_s[kMaxLevels];

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int n_levels = 1 << a.bits;

  for (int idx = tid; idx < kDim * kDim / 4; idx += kThreads) {
    reinterpret_cast<float4*>(rt_s)[idx] = reinterpret_cast<const float4*>(a.Rt)[idx];
    if (qjl) reinterpret_cast<float4*>(spt_s)[idx] = reinterpret_cast<const float4*>(a.Spt)[idx];
  }
  if (tid < kMaxLevels) {
    lev_s[tid] = tid < n_levels ? a.levels[tid] : 0.f;
    bnd_s[tid] = a.bounds[tid];
  }
  __syncthreads();

  const int row_bytes = a.bits * 16;
  const long long cache_rows = static_cast<long long>(a.num_blocks) * a.block_size;
  const int n_tiles = (a.n_vec + kTile - 1) / kTile;

  for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x) {
    const int base = tile * kTile;
    for (int idx = tid; idx < kTile * kDim; idx += kThreads) {
      const int v = idx / kDim;
      const int gv = base + v;
      x_s[idx] = gv < a.n_vec ? load_elem(a.x, static_cast<long long>(gv) * kDim + (idx % kDim), bf16) : 0.f;
    }
    __syncthreads();
    tile_gemm(x_s, rt_s, y_s);
    __syncthreads();

    for (int v = warp; v < kTile; v += kThreads / 32) {
      const int gv = base + v;
      if (gv >= a.n_vec) break;
      const int token = gv / a.n_kv;
      const int head = gv - token * a.n_kv;
      const long long slot = slot_of(a, token);
      long long row = -1;
      if (slot >= 0 && slot < cache_rows) {
        const long long blk = slot / a.block_size;
        row = (blk * a.n_kv + head) * a.block_size + (slot - blk * a.block_size);
      } else if (slot >= cache_rows && lane == 0) {
        atomicCAS(a.error, 0, kErrSlot);
      }

      float xv[4], yv[4];
      float ss = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        xv[i] = x_s[v * kDim + lane + 32 * i];
        yv[i] = y_s[v * kDim + lane + 32 * i];
        ss = fmaf(xv[i], xv[i], ss);
      }
      const float n = sqrtf(warp_sum(ss));
      int code[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float y = n > 0.f ? yv[i] / n : 0.f;
        int c = 0;
        for (int t = 0; t + 1 < n_levels; ++t) c += (y > bnd_s[t]) ? 1 : 0;
        code[i] = c;
      }
      if (a.transposed) {
        // token-transposed field: one bit per (plane, coordinate) in the word
        // of this token's 32-token group; other tokens' bits are left alone
        if (row >= 0) {
          const long long blk = slot / a.block_size;
          const int off = static_cast<int>(slot - blk * a.block_size);
          unsigned* words = reinterpret_cast<unsigned*>(a.codes);
          const unsigned mask = 1u << (off & 31);
          for (int p = 0; p < a.bits; ++p) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              unsigned* w = words + transposed_word(blk, head, a.n_kv, a.bits, p, lane + 32 * i, a.block_size, off);
              if ((code[i] >> p) & 1) atomicOr(w, mask); else atomicAnd(w, ~mask);
            }
          }
        }
      } else {
        // Bit-planes: ballot over lanes gives word i of plane p directly.
        for (int p = 0; p < a.bits; ++p) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const unsigned word = __ballot_sync(0xffffffffu, (code[i] >> p) & 1);
            if (row >= 0 && lane == p * 4 + i) {
              reinterpret_cast<unsigned*>(a.codes + row * row_bytes)[p * 4 + i] = word;
            }
          }
        }
      }
      if (row >= 0 && lane == 0) store_norm(a.norm, row, n, a.norm16);
      if (qjl) {
        // the residual against the norm as stored (what the decoder reconstructs with)
        const float ns = stored_norm(n, a.norm16);
        float rs = 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float r = yv[i] - ns * lev_s[code[i]];
          x_s[v * kDim + lane + 32 * i] = r;
          rs = fmaf(r, r, rs);
        }
        const float gamma = sqrtf(warp_sum(rs));
        if (row >= 0 && lane == 0) store_norm(a.rnorm, row, gamma, a.norm16);
      }
    }
    if (qjl) {
      __syncthreads();
      tile_gemm(x_s, spt_s, y_s);
      __syncthreads();
      for (int v = warp; v < kTile; v += kThreads / 32) {
        const int gv = base + v;
        if (gv >= a.n_vec) break;
        const int token = gv / a.n_kv;
        const int head = gv - token * a.n_kv;
        const long long slot = slot_of(a, token);
        if (slot < 0 || slot >= cache_rows) continue;
        const long long blk = slot / a.block_size;
        const long long row = (blk * a.n_kv + head) * a.block_size + (slot - blk * a.block_size);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const unsigned word = __ballot_sync(0xffffffffu, y_s[v * kDim + lane + 32 * i] > 0.f);
          if (lane == i) reinterpret_cast<unsigned*>(a.qjl + row * 16)[i] = word;
        }
      }
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_quantize_simt(const QuantizeArgs& args, bool bf16, int num_sms, cudaStream_t stream) {
  if (args.n_vec <= 0) return cudaSuccess;
  const bool qjl = args.qjl != nullptr;
  const size_t smem = sizeof(float) * ((qjl ? 2 : 1) * kDim * kDim + 2 * kTile * kDim);
  cudaError_t err = cudaFuncSetAttribute(quantize_simt_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
  if (err != cudaSuccess) return err;
  const int n_tiles = (args.n_vec + kTile - 1) / kTile;
  const int grid = n_tiles < num_sms ? n_tiles : num_sms;
  quantize_simt_kernel<<<grid, kThreads, smem, stream>>>(args, bf16);
  return cudaGetLastError();
}

}  // namespace tq
