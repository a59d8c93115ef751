// Per-vector kernels of a decode step: quantize-append of the step's new keys
// and values (one or four vectors per 256-thread CTA), the query preparation of decode
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

// Query heads prepared by one block: two for a decode step's few hundred
// (more blocks in flight, the launch is latency-bound), eight beyond
// kManyQueries, where the matrix loads (128 KB of R^T and S^T from L2 per
// block) dominate.
constexpr int kQueriesPerCta = 2;
constexpr int kQueriesPerCtaMany = 8;
constexpr int kManyQueries = 1024;

__device__ __forceinline__ float load_elem(const void* base, long long idx, bool bf16) {
  if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
  return reinterpret_cast<const float*>(base)[idx];
}


// out[j] = sum_i w[i * 128 + o] * x_s[j][i] for the NV vectors x_s[j] and
// o = threadIdx.x % 128: thread (o, hf) sums the 64 terms i in [64 hf, 64 hf
// + 64) with 32 loads of w in flight, every load serving all NV vectors; the
// halves meet in red_s.  Every thread returns out[j] for its o; x_s must be
// visible to all threads before the call, and red_s is free again on return.
template <int NV>
__device__ __forceinline__ void matvec_batch(const float* __restrict__ w, const float (*x_s)[kDim],
                                             float (*red_s)[NV][kDim], float (&out)[NV]) {
  const int o = threadIdx.x & 127, hf = threadIdx.x >> 7;
  float acc[NV];
#pragma unroll
  for (int j = 0; j < NV; ++j) acc[j] = 0.f;
#pragma unroll
  for (int i0 = 0; i0 < 64; i0 += 32) {
    const float* wp = w + (64 * hf + i0) * kDim + o;
    float v[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) v[k] = __ldg(wp + k * kDim);
#pragma unroll
    for (int k = 0; k < 32; ++k)
#pragma unroll
      for (int j = 0; j < NV; ++j) acc[j] = fmaf(v[k], x_s[j][64 * hf + i0 + k], acc[j]);
  }
#pragma unroll
  for (int j = 0; j < NV; ++j) red_s[hf][j][o] = acc[j];
  __syncthreads();
#pragma unroll
  for (int j = 0; j < NV; ++j) out[j] = red_s[0][j][o] + red_s[1][j][o];
  __syncthreads();
}

// Quantize head vectors v0 .. v0 + nv - 1 of `a` (nv <= NV): n = ||x||,
// y = R x / n, nearest level, and for keys the rotated residual
// r' = R x - n c[code], its norm and the signs of S' r'.  Thread (o, hf) of
// the 256 works on rotated coordinate o of every vector; the two halves split
// each matrix-vector product (every matrix load serves the NV vectors), and
// the threads of half 0 write the results.
template <int NV>
__device__ __forceinline__ void quantize_vectors(const QuantizeArgs& a, int v0, int nv, bool bf16) {
  __shared__ __align__(16) float x_s[NV][kDim];   // inputs, then residuals
  __shared__ float red_s[2][NV][kDim];
  __shared__ float nrm_s[NV][4], rnrm_s[NV][4];   // per-warp partial sums of squares
  const int o = threadIdx.x & 127;
  const bool lead = threadIdx.x < 128;
  const int lane = o & 31;
  const int warp = o >> 5;
  for (int i = threadIdx.x; i < NV * kDim; i += kVecThreads) {
    const int j = i >> 7;
    x_s[j][i & 127] = j < nv ? load_elem(a.x, static_cast<long long>(v0) * kDim + i, bf16) : 0.f;
  }
  __syncthreads();
  if (lead) {
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      float sq = x_s[j][o] * x_s[j][o];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
      if (lane == 0) nrm_s[j][warp] = sq;
    }
  }
  float yv[NV];
  matvec_batch<NV>(a.Rt, x_s, red_s, yv);          // (R x_j)_o; its barriers also publish nrm_s
  const long long cache_rows = static_cast<long long>(a.num_blocks) * a.block_size;
  float n[NV];
  int code[NV];
  long long row[NV], blk[NV];
  int off[NV];
  bool ok[NV];
#pragma unroll
  for (int j = 0; j < NV; ++j) {
    n[j] = sqrtf((nrm_s[j][0] + nrm_s[j][1]) + (nrm_s[j][2] + nrm_s[j][3]));
    const float y = n[j] > 0.f ? yv[j] / n[j] : 0.f;
    code[j] = 0;
    for (int t = 0; t + 1 < (1 << a.bits); ++t) code[j] += (y > a.bounds[t]) ? 1 : 0;
    const int v = v0 + j;
    const int token = v / a.n_kv;
    const int head = v - token * a.n_kv;
    const long long slot = j < nv ? slot_of(a, token) : -1;
    ok[j] = slot >= 0 && slot < cache_rows;
    if (j < nv && slot >= cache_rows && threadIdx.x == 0) atomicCAS(a.error, 0, kErrSlot);
    blk[j] = ok[j] ? slot / a.block_size : 0;
    off[j] = ok[j] ? static_cast<int>(slot - blk[j] * a.block_size) : 0;
    row[j] = (blk[j] * a.n_kv + head) * a.block_size + off[j];
    if (a.transposed) {
      if (ok[j] && lead) {
        unsigned* words = reinterpret_cast<unsigned*>(a.codes);
        const unsigned mask = 1u << (off[j] & 31);
        for (int p = 0; p < a.bits; ++p) {
          unsigned* w = words + transposed_word(blk[j], head, a.n_kv, a.bits, p, o, a.block_size, off[j]);
          if ((code[j] >> p) & 1) atomicOr(w, mask); else atomicAnd(w, ~mask);
        }
      }
    } else {
      for (int p = 0; p < a.bits; ++p) {
        const unsigned word = __ballot_sync(0xffffffffu, (code[j] >> p) & 1);
        if (ok[j] && lead && lane == 0) reinterpret_cast<unsigned*>(a.codes + row[j] * (a.bits * 16))[p * 4 + warp] = word;
      }
    }
    if (ok[j] && threadIdx.x == 0) store_norm(a.norm, row[j], n[j], a.norm16);
  }

  if (a.qjl != nullptr) {
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      // the residual against the norm as stored (what the decoder reconstructs with)
      const float r = fmaf(-stored_norm(n[j], a.norm16), a.levels[code[j]], yv[j]);
      if (lead) {
        x_s[j][o] = r;                            // (x_s is no longer read: the last barrier passed)
        float sq = r * r;
#pragma unroll
        for (int off2 = 16; off2 > 0; off2 >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off2);
        if (lane == 0) rnrm_s[j][warp] = sq;
      }
    }
    __syncthreads();
    float z[NV];
    matvec_batch<NV>(a.Spt, x_s, red_s, z);
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const float gamma = sqrtf((rnrm_s[j][0] + rnrm_s[j][1]) + (rnrm_s[j][2] + rnrm_s[j][3]));
      const unsigned word = __ballot_sync(0xffffffffu, z[j] > 0.f);
      if (ok[j] && lead && lane == 0) reinterpret_cast<unsigned*>(a.qjl + row[j] * 16)[warp] = word;
      if (ok[j] && threadIdx.x == 0) store_norm(a.rnorm, row[j], gamma, a.norm16);
    }
  }
}

// Appended vectors per block of a decode step: one for a few hundred (more
// blocks in flight: the launch is latency-bound), four beyond
// kManyAppends per tensor, where the matrix loads dominate.
constexpr int kManyAppends = 256;

// Totals of N values (a power of two, at most 32) over the 32 lanes of a warp:
// at every shuffle step the value set halves (lanes with bit `off` set keep
// the upper half and send the lower), N - 1 + log2(32 / N) shuffles in all.
// Returns the total of value *idx, which every lane of its 32 / N lanes holds.
template <int N, typename Op>
__device__ __forceinline__ float halving_reduce(const float (&v)[N], int lane, int* idx, Op op) {
  static_assert(N >= 1 && N <= 32 && (N & (N - 1)) == 0, "a power of two up to 32");
  float cur[N];
#pragma unroll
  for (int j = 0; j < N; ++j) cur[j] = v[j];
  int base = 0;
#pragma unroll
  for (int n = N, off = 16; n > 1; n >>= 1, off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? cur[i] : cur[i + n / 2];
      const float keep = upper ? cur[i + n / 2] : cur[i];
      cur[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, off));
    }
    if (upper) base += n / 2;
  }
#pragma unroll
  for (int off = 16 / N; off > 0; off >>= 1) cur[0] = op(cur[0], __shfl_xor_sync(0xffffffffu, cur[0], off));
  *idx = base;
  return cur[0];
}

// Query heads v0 .. v0 + nv - 1 (nv <= QN; consecutive heads
// share every matrix load): ws_q[v] = (R q, S' R q), the projection taken as
// S q since S' = S R^T; with ws_bk, also each head's tensor-core score
// operand: e4m3 pieces of 2 sigma_0 a_S (R q)_j / beta_j per key sign plane S
// and of 2 sigma_1 (S q)_j / beta_j (sigma_0, sigma_1 powers of two that bound
// the pieces; beta_j the bit scale of coordinate j), and the sums that turn
// the 0/1 bit products into +-1 sign products.  256 threads: thread (o, m)
// computes coordinate o of R q (m = 0) or of S q (m = 1) for every head, so
// the two products run side by side.
template <int QN>
__device__ __forceinline__ void prepare_queries(const DecodeArgs& a, int v0, int nv, bool bf16) {
  __shared__ __align__(16) float q_s[QN][kDim];
  __shared__ float stat_s[2][4][2 * QN];        // [m][warp]: max, then sum, per head
  const int o = threadIdx.x & 127, m = threadIdx.x >> 7;
  const int lane = threadIdx.x & 31, warp = (threadIdx.x >> 5) & 3;
  // the partials kernel that follows counts finished segments per (sequence,
  // KV head) from zero (at most batch * n_q groups)
  if (a.ws_ticket != nullptr && threadIdx.x < nv) a.ws_ticket[v0 + threadIdx.x] = 0;
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
    // even and odd terms in the two halves of a paired FMA, added at the end
    float2 acc2[QN];
#pragma unroll
    for (int j = 0; j < QN; ++j) acc2[j] = make_float2(0.f, 0.f);
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
          acc2[j] = __ffma2_rn(make_float2(v[k], v[k + 1]), make_float2(x.x, x.y), acc2[j]);
          acc2[j] = __ffma2_rn(make_float2(v[k + 2], v[k + 3]), make_float2(x.z, x.w), acc2[j]);
        }
    }
#pragma unroll
    for (int j = 0; j < QN; ++j) acc[j] = acc2[j].x + acc2[j].y;
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
  // per head: max of the scaled magnitudes (sigma) and sum of the coordinates,
  // each a halving reduction over the warp
  float mx[QN], sm[QN];
#pragma unroll
  for (int j = 0; j < QN; ++j) {
    mx[j] = fabsf(acc[j]) * (proj ? ib : amax * ib);
    sm[j] = acc[j];
  }
  int jm, js;
  const float wmax = halving_reduce<QN>(mx, lane, &jm, [](float x, float y) { return fmaxf(x, y); });
  const float wsum = halving_reduce<QN>(sm, lane, &js, [](float x, float y) { return x + y; });
  constexpr int kLanesPer = 32 / QN;              // lanes that hold the same head's total
  if ((lane & (kLanesPer - 1)) == 0) {
    stat_s[m][warp][jm] = wmax;
    stat_s[m][warp][QN + js] = wsum;
  }
  __syncthreads();
  // once per (product, head): the piece scale sigma, a power of two
  __shared__ float sig_s[2][QN];
  if (threadIdx.x < 2 * QN) {
    const int mm = threadIdx.x / QN, j = threadIdx.x % QN;
    sig_s[mm][j] = piece_scale(fmaxf(fmaxf(stat_s[mm][0][j], stat_s[mm][1][j]), fmaxf(stat_s[mm][2][j], stat_s[mm][3][j])));
  }
  __syncthreads();
  const int kpos = k_position(o);
  const int items = planes + (a.qjl_m > 0 ? 1 : 0);
#pragma unroll
  for (int j = 0; j < QN; ++j) {
    if (j >= nv) break;
    uint8_t* dst = a.ws_bk + static_cast<long long>(v0 + j) * a.bk_stride;
    if (!proj) {
      const float y = acc[j] * ib * sig_s[0][j];
      for (int s = 0; s < planes; s += 2)           // (planes: 1, or an even count)
        if (s + 1 < planes)
          write_pieces_rows2<kQPieces>(dst + s * kQPieces * 128, dst + (s + 1) * kQPieces * 128, kpos,
                                       a.tables->k_walsh[s] * y, a.tables->k_walsh[s + 1] * y);
        else
          write_pieces_rows<kQPieces>(dst + s * kQPieces * 128, kpos, a.tables->k_walsh[s] * y);
    } else if (a.qjl_m > 0) {
      write_pieces_rows<kQPieces>(dst + planes * kQPieces * 128, kpos, acc[j] * ib * sig_s[1][j]);
    }
  }
  if (threadIdx.x < nv) {
    const int j = threadIdx.x;
    const float sig0 = sig_s[0][j], sig1 = sig_s[1][j];
    const float sum_qr = (stat_s[0][0][QN + j] + stat_s[0][1][QN + j]) + (stat_s[0][2][QN + j] + stat_s[0][3][QN + j]);
    const float sum_qs = (stat_s[1][0][QN + j] + stat_s[1][1][QN + j]) + (stat_s[1][2][QN + j] + stat_s[1][3][QN + j]);
    float* hdr = reinterpret_cast<float*>(a.ws_bk + static_cast<long long>(v0 + j) * a.bk_stride + items * kQPieces * 128);
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
// thread (o, q) merges coordinate o of head q / 2 over the partial entries c
// (listed by the head's SegInfo) with c % 2 == q % 2 as a running (m, l, acc);
// the two copies of a head merge theirs; then thread (o, q) sums the terms
// [32 q, 32 q + 32) of both heads' back-rotations from one set of loads of R.
// Every thread's entry loads are independent, so a launch is a few memory
// round trips long.
__global__ void __launch_bounds__(kGemvThreads) combine_kernel(DecodeArgs a, DecodeArgs second, int n_src) {
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
  // the entries of every source (one cache, or the two parts of a split
  // context), merged as one running (m, l, acc)
  for (int src = 0; src < n_src && live; ++src) {
    const DecodeArgs& s = src == 0 ? a : second;
    const int ctx = context_of(s, vec / s.n_q);
    // (a sequence without context has no entries, and its segment record is stale)
    SegInfo seg = ctx > 0 ? s.ws_seg[vec] : SegInfo{0, 0, 0, 0};
    // (a partials CTA that stopped early leaves a stale record: check it)
    if (ctx > 0 && (seg.count < 0 || seg.base < 0 || seg.stride < 1 ||
                    static_cast<long long>(seg.base) +
                            static_cast<long long>(seg.count > 0 ? seg.count - 1 : 0) * seg.stride >= s.part_cap)) {
      if (o == 0) atomicCAS(s.error, 0, kErrPartials);
      seg = SegInfo{0, 0, 0, 0};
    }
    const int n_entries = seg.count;
    for (int c0 = q & 1; c0 < n_entries; c0 += 2 * 4) {
      float mc[4], lc[4], ac[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int c = c0 + 2 * j;
        const float* part = s.ws_part + (static_cast<long long>(seg.base) + static_cast<long long>(c) * seg.stride) * kPartStride;
        mc[j] = c < n_entries ? part[0] : -INFINITY;
        lc[j] = c < n_entries ? part[1] : 0.f;
        ac[j] = c < n_entries ? part[4 + o] : 0.f;
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
  quantize_vectors<1>(in_first ? first : second, in_first ? blockIdx.x : blockIdx.x - first.n_vec, 1, bf16);
}

template <int QN>
__global__ void __launch_bounds__(kVecThreads) qprep_kernel(DecodeArgs a, bool bf16) {
  const int v0 = blockIdx.x * QN;
  prepare_queries<QN>(a, v0, min(QN, a.batch * a.n_q - v0), bf16);
}

// One decode step's per-vector work: blocks [0, n_k) quantize the new keys,
// [n_k, 2 n_k) the new values, the rest prepare the queries, QN
// heads per block.  The decode
// partials kernel that follows may start as soon as these blocks run (it
// waits for their results where it reads them).
template <int NV, int QN>
__global__ void __launch_bounds__(kVecThreads) step_prep_kernel(QuantizeArgs ka, QuantizeArgs va, bool kv_bf16,
                                                                 DecodeArgs da, bool q_bf16) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int blk = blockIdx.x;
  const int nb = (ka.n_vec + NV - 1) / NV;        // blocks per tensor
  if (blk < 2 * nb) {
    const QuantizeArgs& x = blk < nb ? ka : va;
    const int v0 = (blk < nb ? blk : blk - nb) * NV;
    quantize_vectors<NV>(x, v0, min(NV, x.n_vec - v0), kv_bf16);
  } else {
    const int v0 = (blk - 2 * nb) * QN;
    prepare_queries<QN>(da, v0, min(QN, da.batch * da.n_q - v0), q_bf16);
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
  if (n_vec > kManyQueries) {
    constexpr int QN = kQueriesPerCtaMany;
    qprep_kernel<QN><<<(n_vec + QN - 1) / QN, kVecThreads, 0, stream>>>(args, bf16);
  } else {
    constexpr int QN = kQueriesPerCta;
    qprep_kernel<QN><<<(n_vec + QN - 1) / QN, kVecThreads, 0, stream>>>(args, bf16);
  }
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
  return cudaLaunchKernelEx(&cfg, combine_kernel, args, args, 1);
}

cudaError_t launch_decode_finish_parts(const DecodeArgs& first, const DecodeArgs& second, cudaStream_t stream) {
  const int n_vec = first.batch * first.n_q;
  if (n_vec <= 0) return cudaSuccess;
  combine_kernel<<<(n_vec + 1) / 2, kGemvThreads, 0, stream>>>(first, second, 2);
  return cudaGetLastError();
}

cudaError_t launch_step_prep(const QuantizeArgs& ka, const QuantizeArgs& va, bool kv_bf16, const DecodeArgs& da,
                             bool q_bf16, cudaStream_t stream) {
  const int n_vec = da.batch * da.n_q;
  const bool many_q = n_vec > kManyQueries, many_kv = ka.n_vec > kManyAppends;
  auto launch = [&](auto kernel, int nv, int qn) {
    const int n = 2 * ((ka.n_vec + nv - 1) / nv) + (n_vec + qn - 1) / qn;
    if (n <= 0) return cudaSuccess;
    kernel<<<n, kVecThreads, 0, stream>>>(ka, va, kv_bf16, da, q_bf16);
    return cudaGetLastError();
  };
  if (many_kv && many_q) return launch(step_prep_kernel<4, kQueriesPerCtaMany>, 4, kQueriesPerCtaMany);
  if (many_kv) return launch(step_prep_kernel<4, kQueriesPerCta>, 4, kQueriesPerCta);
  if (many_q) return launch(step_prep_kernel<1, kQueriesPerCtaMany>, 1, kQueriesPerCtaMany);
  return launch(step_prep_kernel<1, kQueriesPerCta>, 1, kQueriesPerCta);
}

}  // namespace tq
