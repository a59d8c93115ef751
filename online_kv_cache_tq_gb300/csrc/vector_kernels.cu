// Per-vector kernels of a decode step: quantize-append of the step's new keys
// and values (one vector per 256-thread CTA), the query preparation of decode
// attention (two query heads per 256-thread CTA; a fused launch runs both for
// a step), and the merge of the split-K partials with the back-rotation (two
// query heads per 512-thread CTA).
//
// Same arithmetic as the tile quantizers (甲子光年 article §2 第一階段 /
// 第二階段) and the decode estimator (§2 第二階段: <q, k> ~= n <R q, c[code]>
// + gamma sqrt(pi/2)/m <S' R q, 2 bits - 1>; out = R^T acc / l, seo-farm page
// §4).  R^T, S'^T and R are read from global memory (L2-resident after first
// use), so a launch costs a few microseconds instead of staging 128 KB of
// constants per CTA.
#include <cuda_bf16.h>

#include "e4m3_pieces.cuh"
#include "gemv512.cuh"
#include "kernels.h"

namespace tq {
namespace {

constexpr int kQueriesPerCta = 2;   // query heads prepared by one block

__device__ __forceinline__ float load_elem(const void* base, long long idx, bool bf16) {
  if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
  return reinterpret_cast<const float*>(base)[idx];
}


// Quantize head vector v of `a` (n = ||x||, y = R x / n, nearest level, and
// for keys the rotated residual r' = R x - n c[code], its norm and the signs
// of S' r').  Thread (o, q) of the 256 works on rotated coordinate o; the
// two copies of o split the matrix-vector products and threads q == 0
// (warps 0-3) write the results.
__device__ __forceinline__ void quantize_vector(const QuantizeArgs& a, int v, bool bf16) {
  __shared__ float x_s[kDim];
  __shared__ float r_s[kDim];
  __shared__ float red_s[4 * kDim];
  __shared__ float part_s[4];
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
  const float yv = gemv<kVecThreads>(a.Rt, x_s, red_s);           // (R x)_o
  const float y = n > 0.f ? yv / n : 0.f;
  int code = 0;
  for (int t = 0; t + 1 < (1 << a.bits); ++t) code += (y > a.bounds[t]) ? 1 : 0;

  const long long cache_rows = static_cast<long long>(a.num_blocks) * a.block_size;
  const long long slot = slot_of(a, token);
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
    const float z = gemv<kVecThreads>(a.Spt, r_s, red_s);
    const unsigned word = __ballot_sync(0xffffffffu, z > 0.f);
    if (ok && lead && lane == 0) reinterpret_cast<unsigned*>(a.qjl + row * 16)[warp] = word;
    if (ok && threadIdx.x == 0) a.rnorm[row] = gamma;
  }
}


// Query heads v0 .. v0 + nv - 1 (nv <= kQueriesPerCta; consecutive heads
// share every matrix load): ws_q[v] = (R q, S' R q), the projection taken as
// S q since S' = S R^T; with ws_bk, also each head's tensor-core score
// operand: e4m3 pieces of 2 sigma_0 a_S (R q)_j / beta_j per key sign plane S
// and of 2 sigma_1 (S q)_j / beta_j (sigma_0, sigma_1 powers of two that bound
// the pieces; beta_j the bit scale of coordinate j), and the sums that turn
// the 0/1 bit products into +-1 sign products.  256 threads: thread (o, m)
// computes coordinate o of R q (m = 0) or of S q (m = 1) for every head, so
// the two products run side by side.
__device__ __forceinline__ void prepare_queries(const DecodeArgs& a, int v0, int nv, bool bf16) {
  constexpr int QN = kQueriesPerCta;
  __shared__ __align__(16) float q_s[QN][kDim];
  __shared__ float stat_s[2][4][2 * QN];        // [m][warp]: max, then sum, per head
  const int o = threadIdx.x & 127, m = threadIdx.x >> 7;
  const int lane = threadIdx.x & 31, warp = (threadIdx.x >> 5) & 3;
  for (int i = threadIdx.x; i < QN * kDim; i += kVecThreads) {
    const int j = i >> 7;
    q_s[j][i & 127] = j < nv ? load_elem(a.q, static_cast<long long>(v0) * kDim + i, bf16) : 0.f;
  }
  __syncthreads();
  const bool proj = m == 1;
  const bool active = !proj || a.qjl_m > 0;
  float acc[QN];
#pragma unroll
  for (int j = 0; j < QN; ++j) acc[j] = 0.f;
  if (active) {
    const float* w = (proj ? a.St : a.Rt) + o;
#pragma unroll
    for (int k0 = 0; k0 < kDim; k0 += 32) {
      float v[32];
#pragma unroll
      for (int k = 0; k < 32; ++k) v[k] = __ldg(w + (k0 + k) * kDim);
#pragma unroll
      for (int k = 0; k < 32; k += 4)
#pragma unroll
        for (int j = 0; j < QN; ++j) {
          const float4 x = *reinterpret_cast<const float4*>(&q_s[j][k0 + k]);
          acc[j] = fmaf(v[k], x.x, acc[j]);
          acc[j] = fmaf(v[k + 1], x.y, acc[j]);
          acc[j] = fmaf(v[k + 2], x.z, acc[j]);
          acc[j] = fmaf(v[k + 3], x.w, acc[j]);
        }
    }
#pragma unroll
    for (int j = 0; j < QN; ++j)
      if (j < nv) a.ws_q[static_cast<long long>(v0 + j) * 2 * kDim + m * kDim + o] = acc[j];
  }
  if (a.ws_bk == nullptr) return;
  const int planes = 1 << (a.k_bits - 1);
  float amax = 0.f, asum = 0.f;
  for (int s = 0; s < planes; ++s) {
    amax = fmaxf(amax, fabsf(a.tables->k_walsh[s]));
    asum += a.tables->k_walsh[s];
  }
  const float ib = 2.f * bit_inv_scale(o);
  // per head: max of the scaled magnitudes (sigma) and sum of the coordinates
  float red[2 * QN];
#pragma unroll
  for (int j = 0; j < QN; ++j) {
    red[j] = fabsf(acc[j]) * (proj ? ib : amax * ib);
    red[QN + j] = acc[j];
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
#pragma unroll
    for (int j = 0; j < 2 * QN; ++j) {
      const float u = __shfl_xor_sync(0xffffffffu, red[j], off);
      red[j] = j < QN ? fmaxf(red[j], u) : red[j] + u;
    }
  if (lane == 0)
#pragma unroll
    for (int j = 0; j < 2 * QN; ++j) stat_s[m][warp][j] = red[j];
  __syncthreads();
  const int kpos = k_position(o);
  const int items = planes + (a.qjl_m > 0 ? 1 : 0);
#pragma unroll
  for (int j = 0; j < QN; ++j) {
    if (j >= nv) break;
    const float sig0 = piece_scale(fmaxf(fmaxf(stat_s[0][0][j], stat_s[0][1][j]), fmaxf(stat_s[0][2][j], stat_s[0][3][j])));
    const float sig1 = piece_scale(fmaxf(fmaxf(stat_s[1][0][j], stat_s[1][1][j]), fmaxf(stat_s[1][2][j], stat_s[1][3][j])));
    uint8_t* dst = a.ws_bk + static_cast<long long>(v0 + j) * a.bk_stride;
    if (!proj) {
      for (int s = 0; s < planes; ++s)
        write_pieces_rows<kQPieces>(dst + s * kQPieces * 128, kpos, a.tables->k_walsh[s] * acc[j] * ib * sig0);
    } else if (a.qjl_m > 0) {
      write_pieces_rows<kQPieces>(dst + planes * kQPieces * 128, kpos, acc[j] * ib * sig1);
    }
    if (threadIdx.x == 0) {
      const float sum_qr = (stat_s[0][0][QN + j] + stat_s[0][1][QN + j]) + (stat_s[0][2][QN + j] + stat_s[0][3][QN + j]);
      const float sum_qs = (stat_s[1][0][QN + j] + stat_s[1][1][QN + j]) + (stat_s[1][2][QN + j] + stat_s[1][3][QN + j]);
      float* hdr = reinterpret_cast<float*>(dst + items * kQPieces * 128);
      hdr[0] = sig0;
      hdr[1] = sig1;
      hdr[2] = 1.f / sig0;      // exact: powers of two
      hdr[3] = 1.f / sig1;
      hdr[4] = asum * sum_qr;   // sum_S a_S <q_rot, 1>: the -1 half of every sign
      hdr[5] = sum_qs;
      hdr[6] = 0.f;
      hdr[7] = 0.f;
    }
  }
}

__device__ __forceinline__ int context_of(const DecodeArgs& a, int b) {
  int ctx = a.context_lens[b];
  const int cap = min(a.max_context, a.max_blocks * a.block_size);
  if (ctx < 0 || ctx > cap) {
    atomicCAS(a.error, 0, kErrContext);
    ctx = ctx < 0 ? 0 : cap;
  }
  return ctx;
}

// out[v] = R^T (merged acc / merged l) for the query heads v = 2 blockIdx.x
// and 2 blockIdx.x + 1 (one head when the count is odd).  kGemvThreads = 512:
// thread (o, q) merges coordinate o of head q / 2 over the chunks c with
// c % 2 == q % 2 as a running (m, l, acc); the two copies of a head merge
// theirs; then thread (o, q) sums the terms [32 q, 32 q + 32) of both heads'
// back-rotations from one set of loads of R.  Every thread's chunk loads are
// independent, so a launch is a few memory round trips long.
__global__ void __launch_bounds__(kGemvThreads) combine_kernel(DecodeArgs a) {
  constexpr int kHeads = 2;
  __shared__ float o_s[kHeads][kDim];
  __shared__ float red_s[4][kHeads][kDim];
  __shared__ float ml_s[2][4];
  const int t = threadIdx.x;
  const int o = t & 127, q = t >> 7;
  static_assert(kGemvThreads == 512, "threads (o, q) with q = 0..3");
  const int n_vec = a.batch * a.n_q;
  const int vec = kHeads * blockIdx.x + (q >> 1);           // this thread's head in the merge
  const bool live = vec < n_vec;
  asm volatile("griddepcontrol.wait;" ::: "memory");   // the partials (no-op unless launched early)
  float m = -INFINITY, l = 0.f, acc = 0.f;
  if (live) {
    const int ctx = context_of(a, vec / a.n_q);
    const int n_chunks = (ctx + kChunk - 1) / kChunk;
    const float* part = a.ws_part + static_cast<long long>(vec) * a.max_chunks * kPartStride;
    for (int c0 = q & 1; c0 < n_chunks; c0 += 2 * 4) {
      float mc[4], lc[4], ac[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = c0 + 2 * j;
        mc[j] = c < n_chunks ? part[c * kPartStride] : -INFINITY;
        lc[j] = c < n_chunks ? part[c * kPartStride + 1] : 0.f;
        ac[j] = c < n_chunks ? part[c * kPartStride + 4 + o] : 0.f;
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (mc[j] == -INFINITY) continue;
        const float mn = fmaxf(m, mc[j]);
        const float so = m == -INFINITY ? 0.f : __expf(m - mn), sn = __expf(mc[j] - mn);
        l = fmaf(l, so, lc[j] * sn);
        acc = fmaf(acc, so, ac[j] * sn);
        m = mn;
      }
    }
  }
  red_s[q][0][o] = acc;
  if (o == 0) {
    ml_s[0][q] = m;
    ml_s[1][q] = l;
  }
  __syncthreads();
  if ((q & 1) == 0) {                             // copies q and q + 1 of head q / 2
    const float mt = fmaxf(ml_s[0][q], ml_s[0][q + 1]);
    float lt = 0.f, at = 0.f;
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const float w = ml_s[0][q + c] == -INFINITY ? 0.f : __expf(ml_s[0][q + c] - mt);
      lt = fmaf(w, ml_s[1][q + c], lt);
      at = fmaf(w, red_s[q + c][0][o], at);
    }
    o_s[q >> 1][o] = lt > 0.f ? at / lt : 0.f;
  }
  __syncthreads();
  // out[h][o] = sum_i R[o][i] o_s[h][i]: R stored as w[i * 128 + o]; thread q takes i in [32 q, 32 q + 32)
  float s0 = 0.f, s1 = 0.f;
  {
    const float* wp = a.R + (32 * q) * kDim + o;
    float v[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) v[k] = __ldg(wp + k * kDim);
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      s0 = fmaf(v[k], o_s[0][32 * q + k], s0);
      s1 = fmaf(v[k], o_s[1][32 * q + k], s1);
    }
  }
  red_s[q][0][o] = s0;
  red_s[q][1][o] = s1;
  __syncthreads();
  if (q < kHeads) {
    const int v = kHeads * blockIdx.x + q;
    if (v < n_vec)
      a.out[static_cast<long long>(v) * kDim + o] =
          (red_s[0][q][o] + red_s[1][q][o]) + (red_s[2][q][o] + red_s[3][q][o]);
  }
}

// Blocks [0, first.n_vec) quantize `first`, the rest `second` (K and V of one
// append in a single launch).
__global__ void __launch_bounds__(kVecThreads) quantize_small_kernel(QuantizeArgs first, QuantizeArgs second,
                                                                      bool bf16) {
  const bool in_first = static_cast<int>(blockIdx.x) < first.n_vec;
  quantize_vector(in_first ? first : second, in_first ? blockIdx.x : blockIdx.x - first.n_vec, bf16);
}

__global__ void __launch_bounds__(kVecThreads) qprep_kernel(DecodeArgs a, bool bf16) {
  const int v0 = blockIdx.x * kQueriesPerCta;
  prepare_queries(a, v0, min(kQueriesPerCta, a.batch * a.n_q - v0), bf16);
}

// One decode step's per-vector work: blocks [0, n_k) quantize the new keys,
// [n_k, 2 n_k) the new values, the rest prepare the queries, kQueriesPerCta
// heads per block.  The decode
// partials kernel that follows may start as soon as these blocks run (it
// waits for their results where it reads them).
__global__ void __launch_bounds__(kVecThreads) step_prep_kernel(QuantizeArgs ka, QuantizeArgs va, bool kv_bf16,
                                                                 DecodeArgs da, bool q_bf16) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int blk = blockIdx.x;
  if (blk < ka.n_vec) quantize_vector(ka, blk, kv_bf16);
  else if (blk < 2 * ka.n_vec) quantize_vector(va, blk - ka.n_vec, kv_bf16);
  else {
    const int v0 = (blk - 2 * ka.n_vec) * kQueriesPerCta;
    prepare_queries(da, v0, min(kQueriesPerCta, da.batch * da.n_q - v0), q_bf16);
  }
}

}  // namespace

cudaError_t launch_quantize_small(const QuantizeArgs* first, const QuantizeArgs* second, bool bf16,
                                  cudaStream_t stream) {
  const int n = (first ? first->n_vec : 0) + (second ? second->n_vec : 0);
  if (n <= 0) return cudaSuccess;
  QuantizeArgs none{};
  quantize_small_kernel<<<n, kVecThreads, 0, stream>>>(first ? *first : none, second ? *second : none, bf16);
  return cudaGetLastError();
}

cudaError_t launch_decode_prepare(const DecodeArgs& args, bool bf16, cudaStream_t stream) {
  const int n_vec = args.batch * args.n_q;
  if (n_vec <= 0) return cudaSuccess;
  qprep_kernel<<<(n_vec + kQueriesPerCta - 1) / kQueriesPerCta, kVecThreads, 0, stream>>>(args, bf16);
  return cudaGetLastError();
}

cudaError_t launch_decode_finish(const DecodeArgs& args, cudaStream_t stream, bool early) {
  const int n_vec = args.batch * args.n_q;
  if (n_vec <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((n_vec + 1) / 2);             // two query heads per block
  cfg.blockDim = dim3(kGemvThreads);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = early ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, combine_kernel, args);
}

cudaError_t launch_step_prep(const QuantizeArgs& ka, const QuantizeArgs& va, bool kv_bf16, const DecodeArgs& da,
                             bool q_bf16, cudaStream_t stream) {
  const int n = 2 * ka.n_vec + (da.batch * da.n_q + kQueriesPerCta - 1) / kQueriesPerCta;
  if (n <= 0) return cudaSuccess;
  step_prep_kernel<<<n, kVecThreads, 0, stream>>>(ka, va, kv_bf16, da, q_bf16);
  return cudaGetLastError();
}

}  // namespace tq
