// Decode attention over the packed cache: the SIMT split-K partials kernel,
// in the rotated space (the query preparation and the combine/back-rotation
// are in vector_kernels.cu).
//
// Estimator (甲子光年 article §2 第二階段; intelliparadigm.com §2.1.2, §2.2):
//   <q, k> ~= n_k <R q, c_K[code]> + gamma sqrt(pi/2)/m <S' R q, 2 bits - 1>
// Attention (seo-farm page §2 and §4): softmax over the whole context with the
// query uncompressed; values accumulate as n_v c_V[code] in the rotated space
// and one back-rotation out = R^T acc / l ends the step (R^T R = I).
//
// Work decomposition: one CTA per (context chunk of kChunk tokens, KV head,
// sequence) computes all G = n_q / n_kv query heads of that KV head, so every
// packed byte is read once per step.  Phase 1 (one thread per token) scores
// the chunk, phase 2 takes per-head max/sum, phase 3 (lane l owns coordinates
// l + 32 i) accumulates values, phase 4 reduces warps and writes the partial
// (m, l, acc[128]) that the combine kernel merges.
#include <cuda_bf16.h>

#include "kernels.h"

namespace tq {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kTokPerThread = kChunk / kThreads;

__device__ __forceinline__ void record(int* error, int code) { atomicCAS(error, 0, code); }

__device__ __forceinline__ int context_of(const DecodeArgs& a, int b) {
  int ctx = a.context_lens[b];
  const int cap = min(a.max_context, a.max_blocks * a.block_size);
  if (ctx < 0 || ctx > cap) {
    record(a.error, kErrContext);
    ctx = ctx < 0 ? 0 : cap;
  }
  return ctx;
}

template <int G>
__global__ void __launch_bounds__(kThreads) attention_kernel(DecodeArgs a) {
  const int chunk = blockIdx.x;
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;
  const int ctx = context_of(a, b);
  const int start = chunk * kChunk;
  if (start >= ctx) return;
  const int n_local = min(kChunk, ctx - start);

  __shared__ __align__(16) float qr_s[G][kDim];
  __shared__ __align__(16) float qs_s[G][kDim];
  __shared__ float p_s[G][kChunk];
  __shared__ long long row_s[kChunk];
  __shared__ float lk_s[kMaxLevels];
  __shared__ float lv_s[kMaxLevels];
  __shared__ float red_s[kWarps][G];
  __shared__ float stat_s[2][G];

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const bool qjl = a.k_qjl != nullptr;
  const int qbase = b * a.n_q + kvh * G;
  // one partial entry per chunk: entry (query head, chunk) of a [.][max_chunks] array
  if (chunk == 0 && tid < G)
    a.ws_seg[qbase + tid] = SegInfo{(qbase + tid) * a.max_chunks, (ctx + kChunk - 1) / kChunk, 1, 0};

  for (int idx = tid; idx < G * kDim; idx += kThreads) {
    const int g = idx / kDim, j = idx % kDim;
    const float* src = a.ws_q + static_cast<long long>(qbase + g) * 2 * kDim;
    qr_s[g][j] = src[j];
    qs_s[g][j] = qjl ? src[kDim + j] : 0.f;
  }
  if (tid < kMaxLevels) {
    lk_s[tid] = a.tables->k_levels[tid];
    lv_s[tid] = a.tables->v_levels[tid];
  }
  __syncthreads();

  // Phase 1: one thread per token computes the G scores.
  const int kbytes = a.k_bits * 16;
  for (int r = 0; r < kTokPerThread; ++r) {
    const int tl = tid + r * kThreads;
    if (tl >= n_local) break;
    const int tok = start + tl;
    const int lblk = tok / a.block_size;
    const int phys = a.block_table ? a.block_table[static_cast<long long>(b) * a.max_blocks + lblk]
                                   : b * a.max_blocks + lblk;
    long long row = -1;
    if (phys >= 0 && phys < a.num_blocks) {
      row = (static_cast<long long>(phys) * a.n_kv + kvh) * a.block_size + (tok - lblk * a.block_size);
    } else {
      record(a.error, kErrBlock);
    }
    row_s[tl] = row;
    if (row < 0) {
#pragma unroll
      for (int g = 0; g < G; ++g) p_s[g][tl] = -INFINITY;
      continue;
    }
    uint4 kw[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      kw[p] = p < a.k_bits ? reinterpret_cast<const uint4*>(a.k_codes + row * kbytes)[p] : make_uint4(0, 0, 0, 0);
    }
    const uint4 sw = qjl ? reinterpret_cast<const uint4*>(a.k_qjl + row * 16)[0] : make_uint4(0, 0, 0, 0);
    const float nk = load_norm(a.k_norm, row, a.norm16);
    const float gk = qjl ? load_norm(a.k_rnorm, row, a.norm16) : 0.f;
    float mse[G], qj[G];
#pragma unroll
    for (int g = 0; g < G; ++g) { mse[g] = 0.f; qj[g] = 0.f; }
#pragma unroll
    for (int wi = 0; wi < 4; ++wi) {
      const unsigned w0 = wi == 0 ? kw[0].x : wi == 1 ? kw[0].y : wi == 2 ? kw[0].z : kw[0].w;
      const unsigned w1 = wi == 0 ? kw[1].x : wi == 1 ? kw[1].y : wi == 2 ? kw[1].z : kw[1].w;
      const unsigned w2 = wi == 0 ? kw[2].x : wi == 1 ? kw[2].y : wi == 2 ? kw[2].z : kw[2].w;
      const unsigned w3 = wi == 0 ? kw[3].x : wi == 1 ? kw[3].y : wi == 2 ? kw[3].z : kw[3].w;
      const unsigned ws = wi == 0 ? sw.x : wi == 1 ? sw.y : wi == 2 ? sw.z : sw.w;
#pragma unroll
      for (int jq = 0; jq < 32; jq += 4) {
        float lev[4], sg[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int jj = jq + u;
          const int code = ((w0 >> jj) & 1) | (((w1 >> jj) & 1) << 1) | (((w2 >> jj) & 1) << 2) |
                           (((w3 >> jj) & 1) << 3);
          lev[u] = lk_s[code];
          sg[u] = ((ws >> jj) & 1) ? 1.f : -1.f;
        }
        const int j = wi * 32 + jq;
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float4 qr = *reinterpret_cast<const float4*>(&qr_s[g][j]);
          const float4 qs = *reinterpret_cast<const float4*>(&qs_s[g][j]);
          mse[g] = fmaf(qr.x, lev[0], fmaf(qr.y, lev[1], fmaf(qr.z, lev[2], fmaf(qr.w, lev[3], mse[g]))));
          qj[g] = fmaf(qs.x, sg[0], fmaf(qs.y, sg[1], fmaf(qs.z, sg[2], fmaf(qs.w, sg[3], qj[g]))));
        }
      }
    }
    const float ck = gk * a.qjl_coef;
#pragma unroll
    for (int g = 0; g < G; ++g) p_s[g][tl] = a.scale * fmaf(nk, mse[g], ck * qj[g]);
  }
  __syncthreads();

  // Phase 2: per-head max and sum over the chunk; scores become weights.
  for (int g = 0; g < G; ++g) {
    float mx = -INFINITY;
    for (int tl = tid; tl < n_local; tl += kThreads) mx = fmaxf(mx, p_s[g][tl]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    if (lane == 0) red_s[warp][g] = mx;
  }
  __syncthreads();
  if (tid < G) {
    float mx = -INFINITY;
    for (int w = 0; w < kWarps; ++w) mx = fmaxf(mx, red_s[w][tid]);
    stat_s[0][tid] = mx;
  }
  __syncthreads();
  for (int g = 0; g < G; ++g) {
    const float mx = stat_s[0][g];
    float sum = 0.f;
    for (int tl = tid; tl < n_local; tl += kThreads) {
      const float e = mx == -INFINITY ? 0.f : __expf(p_s[g][tl] - mx);
      p_s[g][tl] = e;
      sum += e;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (lane == 0) red_s[warp][g] = sum;
  }
  __syncthreads();
  if (tid < G) {
    float sum = 0.f;
    for (int w = 0; w < kWarps; ++w) sum += red_s[w][tid];
    stat_s[1][tid] = sum;
  }
  __syncthreads();

  // Phase 3: values, lane l owns coordinates l + 32 i.
  float acc[G][4];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[g][i] = 0.f;
  for (int tl = warp; tl < n_local; tl += kWarps) {
    const long long row = row_s[tl];
    if (row < 0) continue;
    // token-transposed value codes: bit (off % 32) of the word of this
    // token's 32-token group, per plane and coordinate
    const long long bh = row / a.block_size;          // (block * n_kv + head)
    const int off = static_cast<int>(row - bh * a.block_size);
    const unsigned* words = reinterpret_cast<const unsigned*>(a.v_codes);
    const long long base = (bh * a.v_bits * 128) * (a.block_size / 32) + off / 32;
    const float nv = load_norm(a.v_norm, row, a.norm16);
    float val[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      int code = 0;
      for (int p = 0; p < a.v_bits; ++p) {
        const unsigned w = words[base + static_cast<long long>(p * 128 + lane + 32 * i) * (a.block_size / 32)];
        code |= ((w >> (off & 31)) & 1) << p;
      }
      val[i] = nv * lv_s[code];
    }
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float pg = p_s[g][tl];
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[g][i] = fmaf(pg, val[i], acc[g][i]);
    }
  }
  __syncthreads();

  // Phase 4: reduce the warps' accumulators through shared memory (reusing
  // the score buffer, G * kChunk >= kWarps * G * kDim floats) and store.
  float* red = &p_s[0][0];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int i = 0; i < 4; ++i) red[(warp * G + g) * kDim + lane + 32 * i] = acc[g][i];
  __syncthreads();
  for (int idx = tid; idx < G * kDim; idx += kThreads) {
    const int g = idx / kDim, j = idx % kDim;
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) s += red[(w * G + g) * kDim + j];
    float* part = a.ws_part + (static_cast<long long>(qbase + g) * a.max_chunks + chunk) * kPartStride;
    part[4 + j] = s;
    if (j == 0) {
      part[0] = stat_s[0][g];
      part[1] = stat_s[1][g];
    }
  }
}

}  // namespace

cudaError_t launch_decode_partials(const DecodeArgs& args, cudaStream_t stream) {
  if (args.polar) return launch_polar_partials(args, stream);
  if (args.batch <= 0 || args.max_chunks <= 0) return cudaSuccess;
  dim3 grid(args.max_chunks, args.n_kv, args.batch);
  switch (args.group) {
    case 1: attention_kernel<1><<<grid, kThreads, 0, stream>>>(args); break;
    case 2: attention_kernel<2><<<grid, kThreads, 0, stream>>>(args); break;
    case 4: attention_kernel<4><<<grid, kThreads, 0, stream>>>(args); break;
    case 8: attention_kernel<8><<<grid, kThreads, 0, stream>>>(args); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}


}  // namespace tq
