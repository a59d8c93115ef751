// Decode partials on the tensor cores (sm_103a tcgen05, fp8 operands).
//
// Same quantity as the SIMT partials kernel (甲子光年 article §2 第二階段: the
// stage-1 inner product plus the unbiased QJL correction; seo-farm §2/§4:
// softmax in the rotated space, values accumulated there), computed as two
// small GEMMs per 128-token tile with every cached bit used as an exact
// fp8 operand:
//
// * A symmetric Lloyd-Max codebook is a sum of sign planes: with
//   s_p = 2 bit_p - 1, level(code) = sum_S a_S prod_{p in S} s_p over the odd
//   subsets S of code bits (one plane per subset; the triple products are the
//   XOR of three bit-planes).  So <q, c[code]> = sum_S a_S <q, s_S>.  Each
//   +-1 is exact in e4m3.
// * The other operand (a_S q_rot, the projected query q_s, and the softmax
//   weights) is split into e4m3 pieces x = sum_i p_i 16^-i / sigma (sigma a
//   power of two), one piece per GEMM column; each piece holds about four more
//   bits: 6 pieces for query coefficients (fp32-level scores), 3 for softmax
//   weights (relative 2^-13).  Products are exact and accumulate in fp32 in
//   tensor memory.
//
// Scores:  D_S[token][head, piece] = sum_k A_K[token][k] B_K[head, piece][k]
//          (A_K: the token's key sign planes, written into tensor memory by the
//          thread that owns the token; B_K: pieces of a_S q_rot and of q_s).
// Values:  D_O[dim][plane, head, piece] += sum_t A_V[dim][t] B_V[head, piece][t]
//          (A_V: the sign planes of one coordinate across 128 tokens, read
//          directly from the token-transposed value field by the thread that
//          owns the coordinate; B_V: pieces of exp(s - m) n_v).
// The output of a CTA is the same split-K partial (m, l, acc[128]) the SIMT
// kernel writes, merged by the same finish kernel.
//
// One CTA of 256 threads per (512-token chunk, KV head, sequence); threads t
// and t + 128 share tensor-memory lane t and split its work (sign planes,
// accumulator columns, softmax-weight pieces) between them.  At the start, thread 0 copies the chunk's packed
// fields (whole cache blocks, contiguous per block and head) into shared
// memory with bulk asynchronous copies while all threads build B_K.  Thread 0
// issues the MMAs between barriers and alone waits on their completion (time-
// bounded mbarrier waits, error code 4); the others wait at the barrier.
#include <cuda_fp8.h>

#include "kernels.h"
#include "tc_ptx.cuh"

namespace tq {
namespace {

constexpr int kTile = 128;                  // tokens per tile = tensor-memory lanes
constexpr int kTiles = kChunk / kTile;      // tiles per chunk
constexpr int kThreads = 256;               // two threads per tensor-memory lane
constexpr int kQPieces = 6;                 // e4m3 pieces of a query coefficient
constexpr int kVPieces = 3;                 // e4m3 pieces of a softmax weight

__host__ __device__ constexpr int round16(int x) { return (x + 15) / 16 * 16; }
__host__ __device__ constexpr int score_cols(int g) { return round16(kQPieces * g); }   // per group
__host__ __device__ constexpr int value_cols(int g) { return round16(kVPieces * g); }   // per value plane

// Position along K of coordinate (or token) i inside a 128-element block: the
// e4m3 operand byte built from bit i sits at 32 (i/32) + 4 (i%8) + (i%32)/8,
// because one 32-bit register is built from bits i, i+8, i+16, i+24 of a word.
__device__ __forceinline__ int k_position(int i) { return 32 * (i >> 5) + 4 * (i & 7) + ((i & 31) >> 3); }

// Byte offset of (row n, K position k) in a K-major operand stored with the
// 128-byte swizzle (rows of 128 bytes, 16-byte chunk c of row n at c ^ (n % 8)).
__device__ __forceinline__ int sw128(int n, int k) { return n * 128 + ((((k >> 4) ^ (n & 7))) << 4) + (k & 15); }

// Store the e4m3 +-1 image of one 32-bit word of bits (bit 1 -> +1.0 = 0x38,
// bit 0 -> -1.0 = 0xB8) as eight columns: column j holds bits j, j+8, j+16,
// j+24 of the word.
__device__ __forceinline__ void store_signs(uint32_t taddr, uint32_t w) {
  const uint32_t inv = ~w;
  auto col = [inv](int j) { return ((inv << (7 - j)) & 0x80808080u) | 0x38383838u; };
  ptx::tmem_st8(taddr, col(0), col(1), col(2), col(3), col(4), col(5), col(6), col(7));
}

// Code-bit subset of sign plane s (same order as kWalshSets): the single bits
// first, then the triples ({0,1,2} at 3 bits; {0,1,2},{0,1,3},{0,2,3},{1,2,3}
// at 4 bits, i.e. all four bits but one).
__device__ __forceinline__ int walsh_set(int bits, int s) {
  if (s < bits) return 1 << s;
  return bits == 3 ? 7 : 15 ^ (1 << (7 - s));
}

// Word of sign plane `set` (XOR of the chosen bit-planes) without indexing
// registers dynamically.
__device__ __forceinline__ uint32_t plane_word(uint32_t b0, uint32_t b1, uint32_t b2, uint32_t b3, int set) {
  const uint32_t m0 = (set & 1) ? ~0u : 0u, m1 = (set & 2) ? ~0u : 0u;
  const uint32_t m2 = (set & 4) ? ~0u : 0u, m3 = (set & 8) ? ~0u : 0u;
  return (b0 & m0) ^ (b1 & m1) ^ (b2 & m2) ^ (b3 & m3);
}

__device__ __forceinline__ uint8_t to_e4m3(float x) {
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3));
}
__device__ __forceinline__ float from_e4m3(uint8_t b) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(b), __NV_E4M3);
  return __half2float(__half(h));
}

// Power of two sigma with sigma * maxabs <= 200 (so every e4m3 piece stays
// below the format's 448 limit), 1 when maxabs is 0.
__device__ __forceinline__ float piece_scale(float maxabs) {
  if (!(maxabs > 0.f)) return 1.f;
  return exp2f(floorf(log2f(200.f / maxabs)));
}

// Write the e4m3 pieces of y (row `row0 + i` for piece i): each piece is the
// e4m3 rounding of what the previous pieces left, times 16.
template <int N>
__device__ __forceinline__ void write_pieces(uint8_t* b, int row0, int kpos, float y) {
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const uint8_t p = to_e4m3(y);
    b[sw128(row0 + i, kpos)] = p;
    y = (y - from_e4m3(p)) * 16.f;
  }
}

// 16^-i for the piece index i (an exact power of two built from its exponent
// field, so no call is left for the compiler to make).
__device__ __forceinline__ float inv16_pow(int i) { return __int_as_float((127 - 4 * i) << 23); }

// Reduce N values per thread over warps [w0, w0 + nw) of the block at once
// (one pair of barriers for all N); every thread gets the results of its range.
template <int N, typename Op>
__device__ __forceinline__ void block_reduce(float (&v)[N], float* red, int w0, int nw, Op op) {
#pragma unroll
  for (int j = 0; j < N; ++j)
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v[j] = op(v[j], __shfl_xor_sync(0xffffffffu, v[j], off));
  __syncthreads();
  if ((threadIdx.x & 31) == 0)
#pragma unroll
    for (int j = 0; j < N; ++j) red[(threadIdx.x >> 5) * N + j] = v[j];
  __syncthreads();
#pragma unroll
  for (int j = 0; j < N; ++j) {
    float r = red[w0 * N + j];
    for (int w = 1; w < nw; ++w) r = op(r, red[(w0 + w) * N + j]);
    v[j] = r;
  }
}
struct MaxOp { __device__ float operator()(float a, float b) const { return fmaxf(a, b); } };
struct SumOp { __device__ float operator()(float a, float b) const { return a + b; } };

__device__ __forceinline__ int context_of(const DecodeArgs& a, int b) {
  int ctx = a.context_lens[b];
  const int cap = min(a.max_context, a.max_blocks * a.block_size);
  if (ctx < 0 || ctx > cap) {
    atomicCAS(a.error, 0, kErrContext);
    ctx = ctx < 0 ? 0 : cap;
  }
  return ctx;
}

// Build sign planes [s0, s1) of one tensor-memory row from bit-plane words
// bw[p][c] and store plane s at column 32 s; with `last_is_sign` the last
// plane is the QJL sign word sgn[c] instead.
__device__ __forceinline__ void store_planes(uint32_t row_addr, const uint32_t (&bw)[4][4], int bits, int s0, int s1,
                                             bool last_is_sign, const uint32_t (&sgn)[4]) {
  for (int s = s0; s < s1; ++s) {
    const bool sign = last_is_sign && s == s1 - 1;
    const int set = walsh_set(bits, s);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const uint32_t w = sign ? sgn[c] : plane_word(bw[0][c], bw[1][c], bw[2][c], bw[3][c], set);
      store_signs(row_addr + 32 * s + 8 * c, w);
    }
  }
}

}  // namespace

// Tensor-memory columns and dynamic shared memory the kernel needs.
struct TcLayout {
  int pk, pq, pv;           // key sign planes, QJL plane (0/1), value sign planes
  int n1, n2, no;           // score columns (mse, qjl), value columns per plane
  int col_s, col_o, cols, tmem;
  int kbytes, vblock;       // key code bytes per token; value code bytes per (block, head)
  int off_bmse, off_bqjl, off_bv, off_scores, off_qjl, off_kc, off_kq, off_kn, off_kr, off_vn, off_vc, smem_bytes;
};

TcLayout tc_layout(int group, int k_bits, bool qjl, int v_bits, int block_size) {
  TcLayout l{};
  l.pk = 1 << (k_bits - 1);
  l.pq = qjl ? 1 : 0;
  l.pv = 1 << (v_bits - 1);
  l.n1 = score_cols(group);
  l.n2 = qjl ? l.n1 : 0;
  l.no = value_cols(group);
  // The value phase starts after every score column has been read, so its
  // sign planes and accumulators reuse the key phase's columns.
  l.col_s = 32 * (l.pk + l.pq);
  l.col_o = 32 * l.pv;
  const int key_cols = l.col_s + l.n1 + l.n2, value_cols_total = l.col_o + l.pv * l.no;
  l.cols = key_cols > value_cols_total ? key_cols : value_cols_total;
  l.tmem = 32;
  while (l.tmem < l.cols) l.tmem *= 2;
  l.kbytes = k_bits * 16;
  l.vblock = v_bits * 128 * block_size / 8;
  int o = 0;
  l.off_bmse = o; o += l.n1 * l.pk * 128;
  l.off_bqjl = o; o += l.n2 * 128;
  l.off_bv = o; o += kTiles * l.no * 128;
  l.off_scores = o; o += group * kChunk * 4;
  l.off_qjl = o; o += group * kTile * 4;
  l.off_kc = o; o += kChunk * l.kbytes;
  l.off_kq = o; o += kChunk * 16;
  l.off_kn = o; o += kChunk * 4;
  l.off_kr = o; o += kChunk * 4;
  l.off_vn = o; o += kChunk * 4;
  l.off_vc = o; o += (kChunk / block_size) * l.vblock;
  l.smem_bytes = o + 1024;
  return l;
}

template <int G>
__global__ void __launch_bounds__(kThreads, 2) attention_tc_kernel(DecodeArgs a, TcLayout L) {
  constexpr int N1 = score_cols(G), NO = value_cols(G);
  const int chunk = blockIdx.x;
  const int kvh = blockIdx.y;
  const int b = blockIdx.z;
  const int ctx = context_of(a, b);
  const int start = chunk * kChunk;
  if (start >= ctx) return;
  const int n_local = min(kChunk, ctx - start);
  const int n_tiles = (n_local + kTile - 1) / kTile;
  const int bs = a.block_size;
  const int n_blk = (n_local + bs - 1) / bs;          // blocks of this chunk (block_size divides kChunk)

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* b_mse = smem + L.off_bmse;
  uint8_t* b_qjl = smem + L.off_bqjl;
  uint8_t* b_v = smem + L.off_bv;
  float* scores = reinterpret_cast<float*>(smem + L.off_scores);   // [G][kChunk]
  float* qjl_part = reinterpret_cast<float*>(smem + L.off_qjl);    // [G][kTile]
  uint8_t* kc_s = smem + L.off_kc;                                  // [kChunk][kbytes]
  uint8_t* kq_s = smem + L.off_kq;                                  // [kChunk][16]
  float* kn_s = reinterpret_cast<float*>(smem + L.off_kn);
  float* kr_s = reinterpret_cast<float*>(smem + L.off_kr);
  float* vn_s = reinterpret_cast<float*>(smem + L.off_vn);
  uint32_t* vc_s = reinterpret_cast<uint32_t*>(smem + L.off_vc);   // [blk][plane][dim][bs/32]
  __shared__ __align__(8) uint64_t bar_in, bar_s, bar_o;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s, ok_s;
  __shared__ float red_s[(kThreads / 32) * (G + 1)];
  __shared__ float sig_s[2][G];                 // piece scales of the mse / qjl columns
  __shared__ float stat_s[2][G];                // chunk max, chunk sum per head
  __shared__ int blk_ok_s[kChunk / 32];         // physical block of each block slot is valid
  __shared__ float sv_s;                        // piece scale of the softmax weights

  const int t = threadIdx.x;
  const int lane = t & (kTile - 1);             // tensor-memory lane (token or coordinate)
  const int half = t >> 7;                      // which of the two threads of the lane
  const uint32_t row_addr = static_cast<uint32_t>(((t >> 5) & 3) * 32) << 16;
  const bool qjl = a.k_qjl != nullptr;
  const int qbase = b * a.n_q + kvh * G;
  volatile int* abort = &abort_s;

  // zero the B operands (padding rows must be 0)
  for (int i = t; i < L.off_scores / 16; i += kThreads) reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  if (t == 0) {
    abort_s = 0;
    ptx::mbar_init(&bar_in, 1);
    ptx::mbar_init(&bar_s, 1);
    ptx::mbar_init(&bar_o, 1);
    ptx::fence_mbar_init();
  }
  if (t < 32) {
    ptx::tmem_alloc(&tmem_base_s, L.tmem);
    ptx::tmem_relinquish();
  }
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_base_s;

  // ---- prefetch the chunk's packed fields into shared memory ----
  if (t == 0) {
    uint32_t total = 0;
    for (int k = 0; k < n_blk; ++k) {
      const int lblk = (start / bs) + k;
      const int phys = a.block_table ? a.block_table[static_cast<long long>(b) * a.max_blocks + lblk]
                                     : b * a.max_blocks + lblk;
      const bool valid = phys >= 0 && phys < a.num_blocks;
      blk_ok_s[k] = valid;
      if (!valid) {
        atomicCAS(a.error, 0, kErrBlock);
        continue;
      }
      const int rows = min(bs, (n_local - k * bs + 31) / 32 * 32);
      // key codes, key norm, value norm (+ QJL signs and residual norm) per row, value block
      total += rows * (L.kbytes + 4 + 4 + (qjl ? 16 + 4 : 0)) + L.vblock;
    }
    ptx::mbar_arrive_expect_tx(&bar_in, total);
    for (int k = 0; k < n_blk; ++k) {
      if (!blk_ok_s[k]) continue;
      const int lblk = (start / bs) + k;
      const int phys = a.block_table ? a.block_table[static_cast<long long>(b) * a.max_blocks + lblk]
                                     : b * a.max_blocks + lblk;
      const int rows = min(bs, (n_local - k * bs + 31) / 32 * 32);
      const long long r0 = (static_cast<long long>(phys) * a.n_kv + kvh) * bs;    // first row of this block
      const int tl0 = k * bs;
      ptx::bulk_load(kc_s + tl0 * L.kbytes, a.k_codes + r0 * L.kbytes, rows * L.kbytes, &bar_in);
      if (qjl) {
        ptx::bulk_load(kq_s + tl0 * 16, a.k_qjl + r0 * 16, rows * 16, &bar_in);
        ptx::bulk_load(kr_s + tl0, a.k_rnorm + r0, rows * 4, &bar_in);
      }
      ptx::bulk_load(kn_s + tl0, a.k_norm + r0, rows * 4, &bar_in);
      ptx::bulk_load(vn_s + tl0, a.v_norm + r0, rows * 4, &bar_in);
      ptx::bulk_load(vc_s + k * (L.vblock / 4), a.v_codes + (static_cast<long long>(phys) * a.n_kv + kvh) * L.vblock,
                     L.vblock, &bar_in);
    }
  }

  // ---- B_K: e4m3 pieces of a_S q_rot per key sign plane, and of q_s ----
  // (overlaps the copies; half 0 writes the mse operand, half 1 the qjl one)
  {
    const int d = lane;
    const int kpos = k_position(d);
    float amax = 0.f;
    for (int s = 0; s < L.pk; ++s) amax = fmaxf(amax, fabsf(a.tables->k_walsh[s]));
    float m[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float* src = a.ws_q + static_cast<long long>(qbase + h) * 2 * kDim;
      m[h] = fabsf(half == 0 ? src[d] * amax : (qjl ? src[kDim + d] : 0.f));
    }
    // max over this half's 128 values (warps 4 half .. 4 half + 3)
    block_reduce(m, red_s, 4 * half, 4, MaxOp());
    if (lane == 0)
#pragma unroll
      for (int h = 0; h < G; ++h) sig_s[half][h] = piece_scale(m[h]);
    __syncthreads();
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float* src = a.ws_q + static_cast<long long>(qbase + h) * 2 * kDim;
      if (half == 0) {
        const float q = src[d] * sig_s[0][h];
        for (int s = 0; s < L.pk; ++s)
          write_pieces<kQPieces>(b_mse + s * L.n1 * 128, h * kQPieces, kpos, a.tables->k_walsh[s] * q);
      } else if (qjl) {
        write_pieces<kQPieces>(b_qjl, h * kQPieces, kpos, src[kDim + d] * sig_s[1][h]);
      }
    }
  }
  ptx::fence_async_shared();
  if (t == 0) ok_s = ptx::wait_bar(&bar_in, 0, abort, a.error, kErrTimeout);
  __syncthreads();
  bool ok = ok_s;

  const uint32_t idesc_s = ptx::idesc_e4m3_f32(128, N1);
  const uint32_t idesc_o = ptx::idesc_e4m3_f32(128, NO);
  uint32_t ph_s = 0, ph_o = 0;
  const int nk_planes = L.pk + L.pq;
  const int k_split = (nk_planes + 1) / 2;        // half 0 builds planes [0, k_split), half 1 the rest

  // ---- scores, one 128-token tile at a time ----
  for (int tile = 0; tile < n_tiles && ok; ++tile) {
    const int tl = tile * kTile + lane;
    const bool valid = tl < n_local && blk_ok_s[tl / bs];
    {
      uint32_t bw[4][4] = {};
      uint32_t sgn[4] = {};
      if (valid) {
        const uint4* kc = reinterpret_cast<const uint4*>(kc_s + tl * L.kbytes);
#pragma unroll
        for (int p = 0; p < 4; ++p) {
          if (p < a.k_bits) {
            const uint4 w = kc[p];
            bw[p][0] = w.x; bw[p][1] = w.y; bw[p][2] = w.z; bw[p][3] = w.w;
          }
        }
        if (qjl) {
          const uint4 w = reinterpret_cast<const uint4*>(kq_s + tl * 16)[0];
          sgn[0] = w.x; sgn[1] = w.y; sgn[2] = w.z; sgn[3] = w.w;
        }
      }
      const int s0 = half == 0 ? 0 : k_split, s1 = half == 0 ? k_split : nk_planes;
      store_planes(tmem + row_addr, bw, a.k_bits, s0, s1, qjl && s1 == nk_planes, sgn);
    }
    ptx::tmem_wait_st();
    ptx::tc_fence_before();
    __syncthreads();
    if (t == 0) {
      ptx::tc_fence_after();
      for (int s = 0; s < L.pk; ++s)
        for (int kk = 0; kk < 4; ++kk)
          ptx::mma_e4m3_tmem_a(tmem + L.col_s, tmem + 32 * s + 8 * kk,
                               ptx::desc_k_sw128(ptx::smem_u32(b_mse + s * L.n1 * 128) + 32 * kk), idesc_s,
                               (s | kk) != 0);
      if (qjl)
        for (int kk = 0; kk < 4; ++kk)
          ptx::mma_e4m3_tmem_a(tmem + L.col_s + L.n1, tmem + 32 * L.pk + 8 * kk,
                               ptx::desc_k_sw128(ptx::smem_u32(b_qjl) + 32 * kk), idesc_s, kk != 0);
      ptx::mma_commit(&bar_s);
      ok_s = ptx::wait_bar(&bar_s, ph_s, abort, a.error, kErrTimeout);
    }
    ph_s ^= 1;
    __syncthreads();
    ok = ok_s;
    if (!ok) break;
    ptx::tc_fence_after();
    // half 0 combines the mse columns, half 1 the qjl columns of the lane's token
    float acc[G];
#pragma unroll
    for (int h = 0; h < G; ++h) acc[h] = 0.f;
    if (half == 0 || qjl) {
#pragma unroll
      for (int c0 = 0; c0 < N1; c0 += 16) {
        uint32_t v[16];
        ptx::tmem_ld16(tmem + row_addr + L.col_s + half * N1 + c0, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int h = (c0 + i) / kQPieces, piece = (c0 + i) % kQPieces;
          if (h < G) acc[h] = fmaf(__uint_as_float(v[i]), inv16_pow(piece), acc[h]);
        }
      }
    }
    ptx::tc_fence_before();
    if (half == 1) {
      const float gk = valid && qjl ? kr_s[tl] : 0.f;
#pragma unroll
      for (int h = 0; h < G; ++h) qjl_part[h * kTile + lane] = gk * a.qjl_coef * (acc[h] / sig_s[1][h]);
    }
    __syncthreads();
    if (half == 0) {
      const float nk = valid ? kn_s[tl] : 0.f;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float s = a.scale * fmaf(nk, acc[h] / sig_s[0][h], qjl_part[h * kTile + lane]);
        scores[h * kChunk + tl] = valid ? s : -INFINITY;
      }
    }
  }
  __syncthreads();

  // ---- softmax statistics over the chunk; B_V pieces of exp(s - m) n_v ----
  if (ok) {
    float mx[G + 1];                      // per-head score max, then the value-norm max
#pragma unroll
    for (int h = 0; h <= G; ++h) mx[h] = h < G ? -INFINITY : 0.f;
    for (int i = t; i < n_local; i += kThreads) {
#pragma unroll
      for (int h = 0; h < G; ++h) mx[h] = fmaxf(mx[h], scores[h * kChunk + i]);
      if (blk_ok_s[i / bs]) mx[G] = fmaxf(mx[G], vn_s[i]);
    }
    block_reduce(mx, red_s, 0, kThreads / 32, MaxOp());
    float l[G];
#pragma unroll
    for (int h = 0; h < G; ++h) l[h] = 0.f;
    for (int i = t; i < n_tiles * kTile; i += kThreads) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float e = (i < n_local && mx[h] != -INFINITY) ? __expf(scores[h * kChunk + i] - mx[h]) : 0.f;
        scores[h * kChunk + i] = e;
        l[h] += e;
      }
    }
    block_reduce(l, red_s, 0, kThreads / 32, SumOp());
    if (t == 0)
#pragma unroll
      for (int h = 0; h < G; ++h) {
        stat_s[0][h] = mx[h];
        stat_s[1][h] = l[h];
      }
    const float vmax = mx[G];
    const float sv = piece_scale(vmax);
    // thread (lane, half) writes tile tiles [half, half + 2, ...] of its token slot
    const int kpos = k_position(lane);
    for (int tile = half; tile < n_tiles; tile += 2) {
      const int tl = tile * kTile + lane;
      const float nv = (tl < n_local && blk_ok_s[tl / bs]) ? vn_s[tl] * sv : 0.f;
#pragma unroll
      for (int h = 0; h < G; ++h)
        write_pieces<kVPieces>(b_v + tile * L.no * 128, h * kVPieces, kpos, scores[h * kChunk + tl] * nv);
    }
    if (t == 0) sv_s = sv;
    ptx::fence_async_shared();
    __syncthreads();
  }
  const float sv = sv_s;

  // ---- values: the two threads of lane d own coordinate d, splitting its sign planes ----
  const int words_per_dim = bs / 32;
  const int v_split = (L.pv + 1) / 2;
  for (int tile = 0; tile < n_tiles && ok; ++tile) {
    {
      uint32_t bw[4][4] = {};                          // [bit-plane][32-token group]
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const int tl = tile * kTile + 32 * g;
        if (tl < n_local && blk_ok_s[tl / bs]) {
          const int k = tl / bs, grp = (tl % bs) / 32;
          const uint32_t* base = vc_s + k * (L.vblock / 4) + grp;
#pragma unroll
          for (int p = 0; p < 4; ++p)
            if (p < a.v_bits) bw[p][g] = base[(p * 128 + lane) * words_per_dim];
        }
      }
      store_planes(tmem + row_addr, bw, a.v_bits, half == 0 ? 0 : v_split, half == 0 ? v_split : L.pv, false, bw[0]);
    }
    ptx::tmem_wait_st();
    ptx::tc_fence_before();
    __syncthreads();
    if (t == 0) {
      ptx::tc_fence_after();
      for (int s = 0; s < L.pv; ++s)
        for (int kk = 0; kk < 4; ++kk)
          ptx::mma_e4m3_tmem_a(tmem + L.col_o + s * L.no, tmem + 32 * s + 8 * kk,
                               ptx::desc_k_sw128(ptx::smem_u32(b_v + tile * L.no * 128) + 32 * kk), idesc_o,
                               (tile | kk) != 0);
      ptx::mma_commit(&bar_o);
      ok_s = ptx::wait_bar(&bar_o, ph_o, abort, a.error, kErrTimeout);
    }
    ph_o ^= 1;
    __syncthreads();
    ok = ok_s;
  }

  // ---- partial output of this chunk: half h reads planes [h * v_split, ...) ----
  if (ok) {
    ptx::tc_fence_after();
    float o[G];
#pragma unroll
    for (int h = 0; h < G; ++h) o[h] = 0.f;
    for (int s = half == 0 ? 0 : v_split; s < (half == 0 ? v_split : L.pv); ++s) {
      const float ws = a.tables->v_walsh[s];
#pragma unroll
      for (int c0 = 0; c0 < NO; c0 += 16) {
        uint32_t v[16];
        ptx::tmem_ld16(tmem + row_addr + L.col_o + s * L.no + c0, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int h = (c0 + i) / kVPieces, piece = (c0 + i) % kVPieces;
          if (h < G) o[h] = fmaf(ws * inv16_pow(piece), __uint_as_float(v[i]), o[h]);
        }
      }
    }
    ptx::tc_fence_before();
    if (half == 1) {
#pragma unroll
      for (int h = 0; h < G; ++h) qjl_part[h * kTile + lane] = o[h];
    }
    __syncthreads();
    if (half == 0) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float* part = a.ws_part + (static_cast<long long>(qbase + h) * a.max_chunks + chunk) * kPartStride;
        part[4 + lane] = (o[h] + qjl_part[h * kTile + lane]) / sv;
        if (lane == 0) {
          part[0] = stat_s[0][h];
          part[1] = stat_s[1][h];
        }
      }
    }
  } else if (t == 0) {
    // a wait gave up: let every issued copy and MMA finish before the memory goes
    ptx::drain_bar(&bar_in, 0);
    ptx::mma_commit(&bar_s);
    ptx::drain_bar(&bar_s, ph_s);
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (t < 32) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, L.tmem);
  }
}

bool tc_decode_supported(const DecodeArgs& a, bool walsh_ok) {
  if (!walsh_ok || a.block_size % 32 != 0 || kChunk % a.block_size != 0) return false;
  if (a.group != 1 && a.group != 2 && a.group != 4 && a.group != 8) return false;
  const TcLayout l = tc_layout(a.group, a.k_bits, a.k_qjl != nullptr, a.v_bits, a.block_size);
  return l.cols <= 512 && l.smem_bytes <= 200 * 1024;
}

template <int G>
cudaError_t launch_g(const DecodeArgs& a, cudaStream_t stream) {
  const TcLayout l = tc_layout(G, a.k_bits, a.k_qjl != nullptr, a.v_bits, a.block_size);
  cudaError_t err = cudaFuncSetAttribute(attention_tc_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         l.smem_bytes);
  if (err != cudaSuccess) return err;
  dim3 grid(a.max_chunks, a.n_kv, a.batch);
  attention_tc_kernel<G><<<grid, kThreads, l.smem_bytes, stream>>>(a, l);
  return cudaGetLastError();
}

cudaError_t launch_decode_partials_tc(const DecodeArgs& a, cudaStream_t stream) {
  if (a.batch <= 0 || a.max_chunks <= 0) return cudaSuccess;
  switch (a.group) {
    case 1: return launch_g<1>(a, stream);
    case 2: return launch_g<2>(a, stream);
    case 4: return launch_g<4>(a, stream);
    case 8: return launch_g<8>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tq
