// PolarQuant (the intelliparadigm.com page, §2.1.1 step 2) as an alternative
// stage-1 codec.  After the rotation y = R x, adjacent coordinates are paired,
// each pair becomes a radius and an angle, the angle is rounded to the nearest
// multiple of pi/12 (24 sectors), and the radii are paired again, level after
// level, until the vector's norm is left.
//
// Record of a head vector (64 bytes, one little-endian bit stream): the 64
// level-1 codes (0..23) x 5 bits, then the 63 codes of levels 2..7 (0..6,
// both members of a pair are radii) x 3 bits; the final radius is the norm
// field (float32).  Keys and values are coded alike and carry no QJL bits.
//
// Quantize: 256 threads take 32 vectors; thread (o, h) forms y_o of vectors
// 16 h .. 16 h + 15 from column o of R^T (every load of R serves sixteen
// vectors, so R is read from L2 once per 32 vectors); the levels then run
// through two shared buffers, one pair of every vector per thread and pass,
// and 16 threads per vector pack the record.
// Decode: one CTA per (512-token chunk, KV head, sequence), like the CUDA-core
// decode; per 32-token tile, eight threads per token expand its record
// top-down into the 128 rotated coordinates (16 each, a padded token-major
// row in shared memory), the G scores <q_rot, y_hat> follow from float4
// reads, then the values the same way with the softmax weights; the partial
// (m, l, acc) goes to the merge that back-rotates (seo-farm page §2:
// out = R^T o_rot).
#include <cuda_bf16.h>

#include "kernels.h"
#include "polar_codes.cuh"

namespace tq {
namespace {

constexpr int kPThreads = 256;
constexpr int kPVecs = 32;              // vectors per quantize block (16 per 128-thread half)
constexpr int kPHalf = kPVecs / 2;
constexpr int kRecordWords = kPolarRecordWords;
constexpr int kUpperBit = kPolarUpperBit;
constexpr int kPTile = 32;              // tokens per decode tile
constexpr int kYRow = kDim + 4;         // padded row of a decoded vector (float4 reads by 8 lanes hit distinct banks)

__device__ __forceinline__ int upper_offset(int level) { return polar_upper_offset(level); }
__device__ __forceinline__ int angle_code(float second, float first, bool level1) {
  return polar_angle_code(second, first, level1);
}

__device__ __forceinline__ float load_x(const void* base, long long idx, bool bf16) {
  if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[idx]);
  return reinterpret_cast<const float*>(base)[idx];
}

__global__ void __launch_bounds__(kPThreads) polar_quantize_kernel(QuantizeArgs a, bool bf16) {
  __shared__ __align__(16) float x_s[kPVecs][kDim];
  __shared__ __align__(16) float h_s[kPVecs][kDim];   // radii of odd levels (rows of kDim, the first half used)
  __shared__ float rad_s[kPVecs];
  __shared__ uint8_t c1_s[kPVecs][64];          // level-1 codes
  __shared__ uint8_t cu_s[kPVecs][64];          // levels 2..7 (63 codes)
  const int t = threadIdx.x, o = t & (kDim - 1), hv = t >> 7;
  const int v0 = blockIdx.x * kPVecs;
  for (int i = t; i < kPVecs * kDim; i += kPThreads) {
    const int j = i >> 7;
    x_s[j][i & 127] = v0 + j < a.n_vec ? load_x(a.x, static_cast<long long>(v0) * kDim + i, bf16) : 0.f;
  }
  __syncthreads();
  // y_o = sum_i R[o][i] x_i of vectors 16 hv .. 16 hv + 15, 16 loads of R^T in flight
  float y[kPHalf];
#pragma unroll
  for (int e = 0; e < kPHalf; ++e) y[e] = 0.f;
  const float* w = a.Rt + o;
#pragma unroll 1
  for (int i0 = 0; i0 < kDim; i0 += 16) {
    float r[16];
#pragma unroll
    for (int k = 0; k < 16; ++k) r[k] = __ldg(w + (i0 + k) * kDim);
#pragma unroll
    for (int k = 0; k < 16; k += 4)
#pragma unroll
      for (int e = 0; e < kPHalf; ++e) {
        const float4 xv = *reinterpret_cast<const float4*>(&x_s[kPHalf * hv + e][i0 + k]);
        y[e] = fmaf(r[k], xv.x, fmaf(r[k + 1], xv.y, fmaf(r[k + 2], xv.z, fmaf(r[k + 3], xv.w, y[e]))));
      }
  }
  // y into x_s (every thread has read x_s), then the levels: level L pairs
  // the 2^(8-L) values of every vector in one buffer into radii in the other
  // (x_s and h_s alternate), one pair per thread and pass, all lanes busy
  __syncthreads();
#pragma unroll
  for (int e = 0; e < kPHalf; ++e) x_s[kPHalf * hv + e][o] = y[e];
  __syncthreads();
#pragma unroll
  for (int lvl = 1; lvl <= 7; ++lvl) {
    const int pairs = kDim >> lvl;                       // pairs per vector at this level
    const float* src = (lvl & 1) ? &x_s[0][0] : &h_s[0][0];
    float* dst = (lvl & 1) ? &h_s[0][0] : &x_s[0][0];
    for (int idx = t; idx < kPVecs * pairs; idx += kPThreads) {
      const int vi = idx / pairs, p = idx - vi * pairs;
      const float2 fs = *reinterpret_cast<const float2*>(src + vi * kDim + 2 * p);   // (first, second)
      const int code = angle_code(fs.y, fs.x, lvl == 1);
      if (lvl == 1) c1_s[vi][p] = static_cast<uint8_t>(code);
      else cu_s[vi][upper_offset(lvl) + p] = static_cast<uint8_t>(code);
      const float rho = sqrtf(fmaf(fs.x, fs.x, fs.y * fs.y));
      if (lvl == 7) rad_s[vi] = rho;
      else dst[vi * kDim + p] = rho;
    }
    __syncthreads();
  }
  // pack: thread (vector vi, word wd) builds bits 32 wd .. 32 wd + 31 of the record
  for (int idx = t; idx < kPVecs * kRecordWords; idx += kPThreads) {
    const int vi = idx >> 4, wd = idx & 15;
    const int v = v0 + vi;
    if (v < a.n_vec) {
      const uint32_t word = polar_record_word(c1_s[vi], cu_s[vi], wd);
      const int token = v / a.n_kv, head = v - token * a.n_kv;
      const long long slot = slot_of(a, token);
      const long long cache_rows = static_cast<long long>(a.num_blocks) * a.block_size;
      if (slot >= cache_rows) {
        if (wd == 0) atomicCAS(a.error, 0, kErrSlot);
      } else if (slot >= 0) {
        const long long blk = slot / a.block_size;
        const long long row = (blk * a.n_kv + head) * a.block_size + (slot - blk * a.block_size);
        reinterpret_cast<uint32_t*>(a.codes + row * (4 * kRecordWords))[wd] = word;
        if (wd == 0) reinterpret_cast<float*>(a.norm)[row] = rad_s[vi];
      }
    }
  }
}

__device__ __forceinline__ int chunk_context(const DecodeArgs& a, int b) {
  int ctx = a.context_lens[b];
  const int cap = min(a.max_context, a.max_blocks * a.block_size);
  if (ctx < 0 || ctx > cap) {
    atomicCAS(a.error, 0, kErrContext);
    ctx = ctx < 0 ? 0 : cap;
  }
  return ctx;
}

// 64 bits of a record row (kRecordWords + 1 words, the last 0) from bit
// `pos` on, the bits past the row's end zero.
__device__ __forceinline__ uint64_t record_window(const uint32_t* rec, int pos) {
  const int w = pos >> 5;
  return ((static_cast<uint64_t>(rec[w + 1]) << 32) | rec[w]) >> (pos & 31);
}

// Rotated coordinates 16 part .. 16 part + 15 of one record, from the top:
// the three ancestors above the part's subtree (levels 7, 6, 5), then its
// subtree level by level (4 .. 1), a node's radius r becoming r cos(theta)
// and r sin(theta) for its pair (cs_s: cos and sin of the 24 sector angles).
// The part's codes come from four 64-bit windows of the record held in
// registers: its level-1 codes (40 bits from bit 40 part), its level-2 codes
// (12 bits), the level-3 codes (48 bits from bit 416) and the level 4-7 codes
// (45 bits from bit 464).
__device__ __forceinline__ void expand_part(const uint32_t* rec, float radius, int part, const float2* cs_s,
                                            float (&v)[16]) {
  const uint64_t w1 = record_window(rec, 40 * part);
  const uint64_t w2 = record_window(rec, kUpperBit + 3 * (polar_upper_offset(2) + 4 * part));
  const uint64_t w3 = record_window(rec, kUpperBit + 3 * polar_upper_offset(3));
  const uint64_t w4 = record_window(rec, kUpperBit + 3 * polar_upper_offset(4));
  // code of node `node` at upper level L (3 .. 7)
  auto upper = [&](int level, int node) {
    const int bit = 3 * (polar_upper_offset(level) + node);
    return level >= 4 ? static_cast<int>((w4 >> (bit - 3 * polar_upper_offset(4))) & 7u)
                      : static_cast<int>((w3 >> (bit - 3 * polar_upper_offset(3))) & 7u);
  };
  float r = radius;
#pragma unroll
  for (int lvl = 7; lvl >= 5; --lvl) {
    const float2 cs = cs_s[upper(lvl, part >> (lvl - 4))];
    r *= ((part >> (lvl - 5)) & 1) ? cs.y : cs.x;
  }
  v[0] = r;
  {
    const float2 cs = cs_s[upper(4, part)];                          // level 4: one node
    v[1] = v[0] * cs.y;
    v[0] = v[0] * cs.x;
  }
#pragma unroll
  for (int k = 1; k >= 0; --k) {                                    // level 3: two nodes
    const float2 cs = cs_s[upper(3, 2 * part + k)];
    const float parent = v[k];
    v[2 * k] = parent * cs.x;
    v[2 * k + 1] = parent * cs.y;
  }
#pragma unroll
  for (int k = 3; k >= 0; --k) {                                    // level 2: four nodes
    const float2 cs = cs_s[static_cast<int>((w2 >> (3 * k)) & 7u)];
    const float parent = v[k];
    v[2 * k] = parent * cs.x;
    v[2 * k + 1] = parent * cs.y;
  }
#pragma unroll
  for (int k = 7; k >= 0; --k) {                                    // level 1: eight nodes, codes 0 .. 23
    const float2 cs = cs_s[static_cast<int>((w1 >> (5 * k)) & 31u)];
    const float parent = v[k];
    v[2 * k] = parent * cs.x;
    v[2 * k + 1] = parent * cs.y;
  }
}

template <int G>
__global__ void __launch_bounds__(kPThreads) polar_attention_kernel(DecodeArgs a) {
  const int chunk = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int t = threadIdx.x;
  const int ctx = chunk_context(a, b);
  const int qbase = b * a.n_q + kvh * G;
  // one partial entry per chunk: entry (query head, chunk) of a [.][max_chunks] array
  if (chunk == 0 && t < G) a.ws_seg[qbase + t] = SegInfo{(qbase + t) * a.max_chunks, (ctx + kChunk - 1) / kChunk, 1, 0};
  const int start = chunk * kChunk;
  if (start >= ctx) return;
  const int n_local = min(kChunk, ctx - start);

  __shared__ __align__(16) float q_s[G][8][20];   // q_rot in 16-coordinate parts, rows padded to 20 (no bank conflicts)
  __shared__ __align__(16) float y_s[kPTile][kYRow];   // one tile's decoded vectors, token-major
  __shared__ __align__(16) float p_s[kChunk][G];   // scores, then softmax weights (a token's heads side by side)
  __shared__ uint32_t rec_s[kPTile][kRecordWords + 1];
  __shared__ float rad_s[kPTile];
  __shared__ long long row_s[kChunk];
  __shared__ float2 cs_s[24];                  // cos, sin of the sector angles k pi / 12
  __shared__ float red_s[kPThreads / 32][G];
  __shared__ float stat_s[2][G];

  for (int i = t; i < G * kDim; i += kPThreads)
    q_s[i / kDim][(i % kDim) >> 4][i & 15] = a.ws_q[static_cast<long long>(qbase + i / kDim) * 2 * kDim + i % kDim];
  if (t < 24) {
    cs_s[t] = make_float2(cospif(t / 12.f), sinpif(t / 12.f));
  }
  for (int tl = t; tl < kChunk; tl += kPThreads) {
    long long row = -1;
    if (tl < n_local) {
      const int tok = start + tl;
      const int lblk = tok / a.block_size;
      const long long phys = a.block_table ? a.block_table[static_cast<long long>(b) * a.max_blocks + lblk]
                                           : static_cast<long long>(b) * a.max_blocks + lblk;
      if (phys >= 0 && phys < a.num_blocks) {
        row = (phys * a.n_kv + kvh) * a.block_size + (tok - lblk * a.block_size);
      } else {
        atomicCAS(a.error, 0, kErrBlock);
      }
    }
    row_s[tl] = row;
  }
  __syncthreads();

  const int tok_i = t >> 3, part = t & 7;      // expansion: token of the tile, 16-coordinate part
  const int n_tiles = (n_local + kPTile - 1) / kPTile;
  // one tile's records into rec_s and radii into rad_s (invalid tokens: radius 0)
  // one tile's records and radii: fetched into registers one tile ahead
  // (the loads fly while the current tile is expanded and used), then
  // stashed into rec_s / rad_s (invalid tokens: zero record, radius 0)
  uint2 wv = make_uint2(0u, 0u);
  float rd = 0.f;
  auto fetch_tile = [&](const uint8_t* codes, const void* norms, int tile) {
    const long long row = row_s[tile * kPTile + tok_i];
    wv = row >= 0 ? reinterpret_cast<const uint2*>(codes + row * (4 * kRecordWords))[part] : make_uint2(0u, 0u);
    rd = part == 0 && row >= 0 ? reinterpret_cast<const float*>(norms)[row] : 0.f;
  };
  auto stash_tile = [&]() {
    rec_s[tok_i][2 * part] = wv.x;
    rec_s[tok_i][2 * part + 1] = wv.y;
    if (part == 0) {
      rec_s[tok_i][kRecordWords] = 0u;
      rad_s[tok_i] = rd;
    }
  };
  auto expand_tile = [&]() {
    float v[16];
    expand_part(rec_s[tok_i], rad_s[tok_i], part, cs_s, v);
#pragma unroll
    for (int k = 0; k < 16; k += 4)
      *reinterpret_cast<float4*>(&y_s[tok_i][16 * part + k]) = make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
  };

  // ---- scores: s = scale <q_rot, y_hat_k> per (token, head): each thread takes
  // the share of its expanded 16 coordinates in every head's score, and the
  // eight lanes of a token add their shares ----
  fetch_tile(a.k_codes, a.k_norm, 0);
  for (int tile = 0; tile < n_tiles; ++tile) {
    stash_tile();
    __syncthreads();
    if (tile + 1 < n_tiles) fetch_tile(a.k_codes, a.k_norm, tile + 1);
    else fetch_tile(a.v_codes, a.v_norm, 0);     // (the first value tile, while the softmax runs)
    float v[16];
    expand_part(rec_s[tok_i], rad_s[tok_i], part, cs_s, v);
    float sc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float2 acc = make_float2(0.f, 0.f);
#pragma unroll
      for (int k = 0; k < 16; k += 4) {
        const float4 qv = *reinterpret_cast<const float4*>(&q_s[h][part][k]);
        acc = __ffma2_rn(make_float2(v[k], v[k + 1]), make_float2(qv.x, qv.y), acc);
        acc = __ffma2_rn(make_float2(v[k + 2], v[k + 3]), make_float2(qv.z, qv.w), acc);
      }
      sc[h] = acc.x + acc.y;
    }
#pragma unroll
    for (int off = 4; off > 0; off >>= 1)          // (the token's eight lanes are consecutive)
#pragma unroll
      for (int h = 0; h < G; ++h) sc[h] += __shfl_xor_sync(0xffffffffu, sc[h], off);
    // lane `part` of the token writes head `part`'s score (G <= 8)
    float mine = sc[0];
#pragma unroll
    for (int h = 1; h < G; ++h) mine = part == h ? sc[h] : mine;
    const int tl = tile * kPTile + tok_i;
    if (part < G && tl < kChunk) p_s[tl][part] = tl < n_local && row_s[tl] >= 0 ? a.scale * mine : -INFINITY;
    __syncthreads();                              // (rec_s is rewritten by the next stash)
  }

  // ---- softmax over the chunk: per-head max, weights e^(s - m), their sum ----
  const int lane = t & 31, warp = t >> 5;
  float part_v[G];
#pragma unroll
  for (int h = 0; h < G; ++h) part_v[h] = -INFINITY;
  for (int tl = t; tl < n_local; tl += kPThreads)
#pragma unroll
    for (int h = 0; h < G; ++h) part_v[h] = fmaxf(part_v[h], p_s[tl][h]);
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part_v[h] = fmaxf(part_v[h], __shfl_xor_sync(0xffffffffu, part_v[h], off));
  if (lane == 0)
#pragma unroll
    for (int h = 0; h < G; ++h) red_s[warp][h] = part_v[h];
  __syncthreads();
  if (t < G) {
    float m = -INFINITY;
    for (int w = 0; w < kPThreads / 32; ++w) m = fmaxf(m, red_s[w][t]);
    stat_s[0][t] = m;
  }
  __syncthreads();
  float mh[G];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    mh[h] = stat_s[0][h];
    part_v[h] = 0.f;
  }
  for (int tl = t; tl < kChunk; tl += kPThreads)   // (weight 0 past the context, for the value loop)
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float s = p_s[tl][h];
      const float e = tl >= n_local || s == -INFINITY || mh[h] == -INFINITY ? 0.f : __expf(s - mh[h]);
      p_s[tl][h] = e;
      part_v[h] += e;
    }
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part_v[h] += __shfl_xor_sync(0xffffffffu, part_v[h], off);
  __syncthreads();                              // red_s was read above
  if (lane == 0)
#pragma unroll
    for (int h = 0; h < G; ++h) red_s[warp][h] = part_v[h];
  __syncthreads();
  if (t < G) {
    float l = 0.f;
    for (int w = 0; w < kPThreads / 32; ++w) l += red_s[w][t];
    stat_s[1][t] = l;
  }

  // ---- values: acc[h][j] = sum_t w[h][t] y_hat_v[t][j]; thread (j, th) takes every head over the
  // tile's tokens 16 th .. 16 th + 15 (past the context: weight 0 and a zero record) ----
  const int j = t & (kDim - 1), th = t >> 7;
  float acc[G];
#pragma unroll
  for (int h = 0; h < G; ++h) acc[h] = 0.f;
  for (int tile = 0; tile < n_tiles; ++tile) {
    stash_tile();
    __syncthreads();
    if (tile + 1 < n_tiles) fetch_tile(a.v_codes, a.v_norm, tile + 1);
    expand_tile();
    __syncthreads();
#pragma unroll 4
    for (int i = 0; i < kPTile / 2; ++i) {
      const int tok = (kPTile / 2) * th + i;
      const float yv = y_s[tok][j];
      const float* w = p_s[tile * kPTile + tok];
      if constexpr (G % 4 == 0) {
#pragma unroll
        for (int h = 0; h < G; h += 4) {
          const float4 w4 = *reinterpret_cast<const float4*>(w + h);
          acc[h] = fmaf(w4.x, yv, acc[h]);
          acc[h + 1] = fmaf(w4.y, yv, acc[h + 1]);
          acc[h + 2] = fmaf(w4.z, yv, acc[h + 2]);
          acc[h + 3] = fmaf(w4.w, yv, acc[h + 3]);
        }
      } else {
#pragma unroll
        for (int h = 0; h < G; ++h) acc[h] = fmaf(w[h], yv, acc[h]);
      }
    }
    __syncthreads();
  }
  // the two token halves meet in the decoded tile's buffer (free after the last barrier)
  float* const half_s = &y_s[0][0];             // [G][kDim]
  if (th == 1)
#pragma unroll
    for (int h = 0; h < G; ++h) half_s[h * kDim + j] = acc[h];
  __syncthreads();
  if (th == 0)
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float* part_p = a.ws_part + (static_cast<long long>(qbase + h) * a.max_chunks + chunk) * kPartStride;
      part_p[4 + j] = acc[h] + half_s[h * kDim + j];
      if (j == 0) {
        part_p[0] = stat_s[0][h];
        part_p[1] = stat_s[1][h];
      }
    }
}

}  // namespace

cudaError_t launch_polar_quantize(const QuantizeArgs& a, bool bf16, cudaStream_t stream) {
  if (a.n_vec <= 0) return cudaSuccess;
  polar_quantize_kernel<<<(a.n_vec + kPVecs - 1) / kPVecs, kPThreads, 0, stream>>>(a, bf16);
  return cudaGetLastError();
}

cudaError_t launch_polar_partials(const DecodeArgs& a, cudaStream_t stream) {
  if (a.batch <= 0 || a.max_chunks <= 0) return cudaSuccess;
  dim3 grid(a.max_chunks, a.n_kv, a.batch);
  switch (a.group) {
    case 1: polar_attention_kernel<1><<<grid, kPThreads, 0, stream>>>(a); break;
    case 2: polar_attention_kernel<2><<<grid, kPThreads, 0, stream>>>(a); break;
    case 4: polar_attention_kernel<4><<<grid, kPThreads, 0, stream>>>(a); break;
    case 8: polar_attention_kernel<8><<<grid, kPThreads, 0, stream>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace tq
