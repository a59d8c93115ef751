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
//   bits: 5 pieces for query coefficients (4 with eight query heads per KV
//   head, relative 2^-17), 3 for softmax weights (relative 2^-13).  Products
//   are exact and accumulate in fp32 in tensor memory.
//
// Scores:  D_S[token][head, piece] = sum_k A_K[token][k] B_K[head, piece][k]
//          (A_K: the token's key sign planes, written into tensor memory by the
//          thread that owns the token; B_K: pieces of a_S q_rot and of q_s).
// Values:  D_O[dim][plane, head, piece] += sum_t A_V[dim][t] B_V[head, piece][t]
//          (A_V: the sign planes of one coordinate across 128 tokens, read
//          directly from the token-transposed value field by the thread that
//          owns the coordinate; B_V: pieces of exp(s - m) n_v).
// A persistent grid of 288-thread CTAs (two per SM) takes the real chunks of
// the batch -- items (sequence, KV head, 512- or 256-token chunk) numbered in
// that order -- in equal contiguous runs; a CTA merges the consecutive items
// of one (sequence, KV head) as it goes and writes one split-K partial
// (m, l, acc[128]) per such segment, which the CTA that completes a group
// merges (atomic ticket) or a merge launch does.  Warps 0-7
// build operands: threads t and t + 128 share tensor-memory lane t and split
// its work (two of the four 32-bit words of every sign plane, half of the
// accumulator columns, half of the operand pieces).  Warp 8 is the control
// warp: lane k copies block k of an item's packed fields (contiguous per
// block and head) into shared memory with bulk asynchronous copies, one item
// ahead, and an elected lane issues every MMA.  The two sides meet only on mbarriers: the
// builders store a tile's sign planes into one of two tensor-memory slots (or,
// with four MSE planes, the tile's two units into the two slots) and arrive;
// the control warp issues that tile's MMAs and commits; the builders build the
// next tile meanwhile and wait on the commit only to read the accumulators or
// to reuse the slot.  Every wait is time-bounded (error code 4) and a failed
// wait makes every other wait give up.
#include <cuda_fp8.h>

#include <type_traits>

#include "e4m3_pieces.cuh"
#include "kernels.h"
#include "tc_ptx.cuh"

namespace tq {
namespace {

constexpr int kTile = 128;                  // tokens per tile = tensor-memory lanes
constexpr int kBuilders = 256;              // warps 0-7: two threads per tensor-memory lane
constexpr int kThreads = kBuilders + 32;     // warp 8: copies and MMA issue
constexpr int kVPieces = 3;                 // e4m3 pieces of a softmax weight
constexpr int kMaxPending = 8;              // group merges a CTA may defer

__host__ __device__ constexpr int round16(int x) { return (x + 15) / 16 * 16; }
// Score accumulator columns: the query heads of a group are split into two
// halves (threads t < 128 read the first, t >= 128 the second); head h's
// pieces sit at column score_half(g) * (h / half_heads(g)) + q_pieces(g) * (h %
// half_heads(g)), so each thread reads 16-column groups of its own heads only.
// Eight heads use the first four of the prepared pieces (relative precision
// 2^-17 per query coefficient), which keeps a CTA within 256 tensor-memory
// columns and lets two CTAs share an SM; fewer heads use all kQPieces.
__host__ __device__ constexpr int q_pieces(int g) { return g >= 8 ? 4 : kQPieces; }
__host__ __device__ constexpr int half_heads(int g) { return g >= 2 ? g / 2 : 1; }
__host__ __device__ constexpr int score_half(int g) { return round16(q_pieces(g) * half_heads(g)); }
__host__ __device__ constexpr int score_cols(int g) { return g >= 2 ? 2 * score_half(g) : score_half(g); }
__host__ __device__ constexpr int score_row(int g, int h, int piece) {
  return score_half(g) * (h / half_heads(g)) + q_pieces(g) * (h % half_heads(g)) + piece;
}
__host__ __device__ constexpr int value_cols(int g) { return round16(kVPieces * g); }   // per value plane

// Byte offset of (row n, K position k) in a K-major operand stored with the
// 128-byte swizzle (rows of 128 bytes, 16-byte chunk c of row n at c ^ (n % 8)).
__device__ __forceinline__ int sw128(int n, int k) { return n * 128 + ((((k >> 4) ^ (n & 7))) << 4) + (k & 15); }

// Store the 0/beta_j e4m3 image of one 32-bit word of bits as eight columns:
// column j holds bits j, j+8, j+16, j+24 of the word, each as 0 or the power
// of two beta_j of bit_inv_scale: bits 0-2 stay in place, bits 3-7 move down
// by three (one shift and eight masks per word), so every byte has one bit
// among its three mantissa bits and lowest two exponent bits (2^-9 .. 2^-5).
// The arithmetic sits inside the asm block so that the compiler keeps only
// the word, not eight operand registers per plane, live across planes.
__device__ __forceinline__ void store_bits(uint32_t taddr, uint32_t w) {
  asm volatile(
      "{\n\t.reg .b32 h, c0, c1, c2, c3, c4, c5, c6, c7;\n\t"
      "shr.b32 h, %1, 3;\n\t"
      "and.b32 c0, %1, 0x01010101;\n\t"
      "and.b32 c1, %1, 0x02020202;\n\t"
      "and.b32 c2, %1, 0x04040404;\n\t"
      "and.b32 c3, h, 0x01010101;\n\t"
      "and.b32 c4, h, 0x02020202;\n\t"
      "and.b32 c5, h, 0x04040404;\n\t"
      "and.b32 c6, h, 0x08080808;\n\t"
      "and.b32 c7, h, 0x10101010;\n\t"
      "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {c0, c1, c2, c3, c4, c5, c6, c7};\n\t}\n"
      ::"r"(taddr), "r"(w)
      : "memory");
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

// Sign planes of one key tile for BITS-bit codes (the Walsh sets fold to
// constants), words w0 and w0 + 1 of each plane; the QJL plane follows.
template <int BITS>
__device__ __forceinline__ void key_planes(uint32_t base, const uint32_t (&bw)[4][2], const uint32_t (&sg)[2],
                                           bool qjl, int w0) {
  constexpr int P = 1 << (BITS - 1);
#pragma unroll
  for (int s = 0; s < P; ++s) {
    const int set = walsh_set(BITS, s);
#pragma unroll
    for (int c = 0; c < 2; ++c)
      store_bits(base + 32 * s + 8 * (w0 + c), plane_word(bw[0][c], bw[1][c], bw[2][c], bw[3][c], set));
  }
  if (qjl)
#pragma unroll
    for (int c = 0; c < 2; ++c) store_bits(base + 32 * P + 8 * (w0 + c), sg[c]);
}

// Unit u of a key tile built in two units (3-bit MSE codes: four sign
// planes): unit 0 holds sign planes 0-2, unit 1 sign plane 3 and then the QJL
// plane; words w0 and w0 + 1 of each.
__device__ __forceinline__ void key_unit3(uint32_t base, const uint32_t (&bw)[4][2], const uint32_t (&sg)[2], bool qjl,
                                          int w0, int unit) {
  if (unit == 0) {
#pragma unroll
    for (int s = 0; s < 3; ++s)
#pragma unroll
      for (int c = 0; c < 2; ++c)
        store_bits(base + 32 * s + 8 * (w0 + c), plane_word(bw[0][c], bw[1][c], bw[2][c], bw[3][c], walsh_set(3, s)));
  } else {
#pragma unroll
    for (int c = 0; c < 2; ++c) store_bits(base + 8 * (w0 + c), plane_word(bw[0][c], bw[1][c], bw[2][c], bw[3][c], walsh_set(3, 3)));
    if (qjl)
#pragma unroll
      for (int c = 0; c < 2; ++c) store_bits(base + 32 + 8 * (w0 + c), sg[c]);
  }
}

// Value sign plane S of BITS-bit codes (compile-time Walsh set) at `col`.
template <int BITS, int S>
__device__ __forceinline__ void value_plane(uint32_t col, const uint32_t (&bw)[4][2], int w0) {
  if constexpr (S < (1 << (BITS - 1))) {
    constexpr int set = S < BITS ? 1 << S : (BITS == 3 ? 7 : 15 ^ (1 << (7 - S)));
#pragma unroll
    for (int c = 0; c < 2; ++c)
      store_bits(col + 8 * (w0 + c), plane_word(bw[0][c], bw[1][c], bw[2][c], bw[3][c], set));
  }
}

// Value sign planes 2 pair and 2 pair + 1 (those that exist) into a slot;
// one straight-line case per pair keeps only two planes' words live.
template <int BITS>
__device__ __forceinline__ void value_pair(uint32_t base, const uint32_t (&bw)[4][2], int pair, int w0) {
  switch (pair) {
    case 0: value_plane<BITS, 0>(base, bw, w0); value_plane<BITS, 1>(base + 32, bw, w0); break;
    case 1: value_plane<BITS, 2>(base, bw, w0); value_plane<BITS, 3>(base + 32, bw, w0); break;
    case 2: value_plane<BITS, 4>(base, bw, w0); value_plane<BITS, 5>(base + 32, bw, w0); break;
    default: value_plane<BITS, 6>(base, bw, w0); value_plane<BITS, 7>(base + 32, bw, w0); break;
  }
}

// Barrier of the 256 builder threads only (named barrier 1).
__device__ __forceinline__ void builder_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Builder barrier that also ANDs a flag over the 256 builders, so that every
// builder takes the same decision after it (a per-thread read of the abort
// word could differ between warps when the control warp sets it meanwhile).
__device__ __forceinline__ bool builder_all(bool flag) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, 1, 256, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(flag))
      : "memory");
  return r != 0;
}

// Inclusive-exclusive scan of v over the threads of the CTA in thread order
// (every thread takes part): returns the CTA total, *excl the sum over the
// threads before this one.  warp_s holds one int per warp.
template <int THREADS>
__device__ __forceinline__ int cta_scan(int v, int* excl, int* warp_s) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_s[warp] = x;
  __syncthreads();
  int before = 0, total = 0;
#pragma unroll
  for (int w = 0; w < THREADS / 32; ++w) {
    const int sw = warp_s[w];
    before += w < warp ? sw : 0;
    total += sw;
  }
  __syncthreads();
  *excl = before + x - v;
  return total;
}

struct MaxOp {
  __device__ float operator()(float a, float b) const { return fmaxf(a, b); }
};
struct SumOp {
  __device__ float operator()(float a, float b) const { return a + b; }
  __device__ float identity() const { return 0.f; }
};

// Per-warp totals of N values per thread over the eight builder warps (one
// pair of barriers for all N): afterwards red[w * N + j] holds warp w's total
// of value j.  Within a warp the value set halves at every shuffle step (lanes
// with bit `off` set keep the upper half and send the lower): P = N rounded
// up to a power of two takes P - 1 + log2(32 / P) shuffles instead of 5 N.
// Warps 0-3 and 4-7 are the two builder halves, which own different query
// heads, so callers combine the four totals of one half in warp order.
// With `all`, the first barrier also ANDs *all over the builders (as
// builder_all).
template <int N, typename Op>
__device__ __forceinline__ void warp_totals(const float (&v)[N], float* red, Op op, bool* all = nullptr) {
  constexpr int P = N <= 1 ? 1 : N <= 2 ? 2 : N <= 4 ? 4 : N <= 8 ? 8 : N <= 16 ? 16 : 32;
  static_assert(N <= 32, "at most 32 values");
  const int lane = threadIdx.x & 31;
  float cur[P];
#pragma unroll
  for (int j = 0; j < P; ++j) cur[j] = j < N ? v[j] : op.identity();
  int idx = 0;
#pragma unroll
  for (int n = P, off = 16; n > 1; n >>= 1, off >>= 1) {
    const bool upper = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? cur[i] : cur[i + n / 2];
      const float keep = upper ? cur[i + n / 2] : cur[i];
      cur[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, off));
    }
    if (upper) idx += n / 2;
  }
#pragma unroll
  for (int off = 16 / P; off > 0; off >>= 1) cur[0] = op(cur[0], __shfl_xor_sync(0xffffffffu, cur[0], off));
  if (all != nullptr) *all = builder_all(*all);  // the previous reduction's totals were read
  else builder_sync();
  if ((lane & (32 / P - 1)) == 0 && idx < N) red[(threadIdx.x >> 5) * N + idx] = cur[0];
  builder_sync();
}

// The same for maxima: one warp-wide float max reduction per value
// (redux.sync.max.f32), lane j then stores value j's total.
template <int N>
__device__ __forceinline__ void warp_totals(const float (&v)[N], float* red, MaxOp, bool* all = nullptr) {
  static_assert(N <= 32, "at most 32 values");
  const int lane = threadIdx.x & 31;
  float r[N];
#pragma unroll
  for (int j = 0; j < N; ++j) asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r[j]) : "f"(v[j]));
  if (all != nullptr) *all = builder_all(*all);  // the previous reduction's totals were read
  else builder_sync();
  float mine = r[0];
#pragma unroll
  for (int j = 1; j < N; ++j) mine = lane == j ? r[j] : mine;
  if (lane < N) red[(threadIdx.x >> 5) * N + lane] = mine;
  builder_sync();
}

// Total of value j over the four warps of builder half `hf`, in warp order.
template <int N, typename Op>
__device__ __forceinline__ float half_total(const float* red, int hf, int j, Op op) {
  float r = red[(4 * hf) * N + j];
#pragma unroll
  for (int w = 1; w < 4; ++w) r = op(r, red[(4 * hf + w) * N + j]);
  return r;
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

}  // namespace

// Tensor-memory columns and dynamic shared memory the kernel needs.
//
// Key phase: k_slots slots of kp = 32 (pk + pq) columns (the sign planes of
// one tile), then the score accumulators (n1 mse + n2 qjl columns); with four
// MSE planes (3-bit MSE keys) two slots of a whole tile do not fit, and a tile
// is built as two units instead -- MSE planes 0-2 in slot 0, plane 3 and the
// QJL plane in slot 1 (k_units = 2, kp = 96) -- so that one unit is built while
// the other's MMAs run.  Value phase (after every score has been read, so it
// reuses the same columns): two slots of 64 columns (two value sign planes
// each), then pv accumulator blocks of no columns.  Two key slots are used when
// they fit beside the rest; the allocation is a power of two of at least 32
// columns.
struct TcLayout {
  int pk, pq, pv;           // key sign planes, QJL plane (0/1), value sign planes
  int n1, n2, no;           // score columns (mse, qjl), value columns per plane
  int kp, k_slots;          // columns per key slot, key slots (1 or 2)
  int k_units;              // units a key tile is built in (1, or 2 with four MSE planes)
  int v_slots;              // value slots of kValueSlot columns (2 to kMaxValueSlots)
  int col_s, col_o, cols, tmem;
  int kbytes, vblock;       // key code bytes per token; value code bytes per (block, head)
  int chunk;                // tokens per work item (512, or 256 when 512 would not fit two CTAs per SM)
  int off_bmse, off_bqjl, off_bv, off_s0, off_s1, off_sacc, off_kc, off_kq, off_kn, off_kr, off_vn, off_vc, smem_bytes;
};

constexpr int kHeadMergeThreads = 512;      // per-query-head merge: four quarters of 128 lanes
constexpr int kValueSlot = 64;              // columns of one value slot (two sign planes)
constexpr int kMaxValueSlots = 4;

__host__ __device__ constexpr TcLayout tc_layout(int group, int k_bits, bool qjl, int v_bits, int block_size,
                                                 int chunk) {
  TcLayout l{};
  l.chunk = chunk;
  l.pk = 1 << (k_bits - 1);
  l.pq = qjl ? 1 : 0;
  l.pv = 1 << (v_bits - 1);
  l.n1 = score_cols(group);
  l.n2 = qjl ? l.n1 : 0;
  l.no = value_cols(group);
  l.kp = 32 * (l.pk + l.pq);
  // value slots: as many as fit beside the accumulators in the allocation the
  // key phase needs (at least two), so the builders run further ahead of the MMAs
  const int vacc = l.pv * l.no;
  const int vcols = 2 * kValueSlot + vacc;
  auto kcols = [&](int slots) { return slots * l.kp + l.n1 + l.n2; };
  auto mx = [](int x, int y) { return x > y ? x : y; };
  l.k_units = 1;
  if (mx(kcols(2), vcols) <= 256) {
    l.k_slots = 2;
  } else if (l.pk == 4 && mx(2 * 96 + l.n1 + l.n2, vcols) <= 256) {
    l.k_units = 2;                          // a tile as two units of at most three planes
    l.kp = 96;
    l.k_slots = 2;
  } else if (mx(kcols(1), vcols) <= 256) {
    l.k_slots = 1;
  } else if (mx(kcols(2), vcols) <= 512) {
    l.k_slots = 2;
  } else {
    l.k_slots = 1;
  }
  l.col_s = l.k_slots * l.kp;
  l.cols = mx(kcols(l.k_slots), vcols);
  l.tmem = 32;
  while (l.tmem < l.cols) l.tmem *= 2;
  l.v_slots = 2;
  while (l.v_slots < kMaxValueSlots && (l.v_slots + 1) * kValueSlot + vacc <= l.tmem) ++l.v_slots;
  l.col_o = l.v_slots * kValueSlot;
  l.kbytes = k_bits * 16;
  l.vblock = v_bits * 128 * block_size / 8;
  int o = 0;
  l.off_bmse = o; o += l.n1 * l.pk * 128;
  l.off_bqjl = o; o += l.n2 * 128;
  l.off_bv = o; o += (chunk / kTile) * l.no * 128;
  // s1 (the other half's output sums, and scratch of the final merges) lies
  // inside s0 past its first G x kTile floats: the scores are dead by the time
  // s1 is written, and the merges use s0's first part and s1 together
  l.off_s0 = o; o += group * chunk * 4;
  l.off_s1 = l.off_s0 + group * kTile * 4;
  l.off_sacc = o; o += group * kTile * 4;
  l.off_kc = o; o += chunk * l.kbytes;
  l.off_kq = o; o += chunk * 16;
  l.off_kn = o; o += chunk * 4;
  l.off_kr = o; o += chunk * 4;
  l.off_vn = o; o += chunk * 4;
  l.off_vc = o; o += (chunk / block_size) * l.vblock;
  l.smem_bytes = o + 1024;
  // more than half of tensor memory: keep a second CTA off the SM instead of
  // letting it wait in the allocator
  if (l.tmem > 256 && l.smem_bytes < 120 * 1024) l.smem_bytes = 120 * 1024;
  return l;
}

namespace {

// 2^x on the special-function unit (ex2.approx.ftz); the softmax takes
// exp(y) as 2^(y log2 e).
__device__ __forceinline__ float ex2_approx(float x) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// Time-bounded wait on an mbarrier phase by the calling thread (suspending
// between polls); false after a timeout anywhere in the CTA.
// The result is made warp-uniform, since tensor-memory loads and stores that
// follow are warp-collective.
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int* abort, int* error) {
  return __all_sync(0xffffffffu, ptx::wait_bar(bar, parity, abort, error, kErrTimeout));
}

}  // namespace

// R[64 half + i][lane], i < 64: the rows of R that thread (lane, half) needs for
// the back-rotation (a handle constant: no launch writes it).
__device__ __forceinline__ void load_r_half(const float* R, int half, int lane, float (&w)[64]) {
  const float* rp = R + (64 * half) * kDim + lane;
#pragma unroll
  for (int i = 0; i < 64; ++i) w[i] = __ldg(rp + i * kDim);
}

// merge_segments (below) with the rows of R already in registers (load_r_half).
template <int G>
__device__ __forceinline__ void merge_segments_r(const float (&w)[64], const float* ws_part, float* out, int ent0,
                                                 int n_seg, int qbase, float* orot, float* s1, int half, int lane) {
  constexpr int HG = half_heads(G);
  constexpr int kBatch = 8;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    if (h / HG != half) continue;
    float m = -INFINITY, l = 0.f, acc = 0.f;
    for (int sg0 = 0; sg0 < n_seg; sg0 += kBatch) {
      float pm[kBatch], pl[kBatch], pa[kBatch];
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const float* part = ws_part + (static_cast<long long>(ent0) + static_cast<long long>(sg0 + k) * G + h) *
                                          kPartStride;
        const bool in = sg0 + k < n_seg;
        pm[k] = in ? __ldcg(part) : -INFINITY;
        pl[k] = in ? __ldcg(part + 1) : 0.f;
        pa[k] = in ? __ldcg(part + 4 + lane) : 0.f;
      }
      float mn = m;
#pragma unroll
      for (int k = 0; k < kBatch; ++k) mn = fmaxf(mn, pm[k]);
      if (mn == -INFINITY) continue;
      const float so = m == -INFINITY ? 0.f : __expf(m - mn);
      l *= so;
      acc *= so;
#pragma unroll
      for (int k = 0; k < kBatch; ++k) {
        const float sn = pm[k] == -INFINITY ? 0.f : __expf(pm[k] - mn);
        l = fmaf(pl[k], sn, l);
        acc = fmaf(pa[k], sn, acc);
      }
      m = mn;
    }
    orot[h * kTile + lane] = l > 0.f ? acc / l : 0.f;
  }
  builder_sync();
  // out[h][o] = sum_i R[i][o] o_rot[h][i]: thread (o = lane, half) sums i in [64 half, 64 half + 64)
  float r[G];
#pragma unroll
  for (int h = 0; h < G; ++h) r[h] = 0.f;
#pragma unroll
  for (int k = 0; k < 64; k += 4)
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float4 v = *reinterpret_cast<const float4*>(orot + h * kTile + 64 * half + k);
      r[h] = fmaf(w[k], v.x, fmaf(w[k + 1], v.y, fmaf(w[k + 2], v.z, fmaf(w[k + 3], v.w, r[h]))));
    }
  if (half == 1)
#pragma unroll
    for (int h = 0; h < G; ++h) s1[h * kTile + lane] = r[h];
  builder_sync();
  if (half == 0)
#pragma unroll
    for (int h = 0; h < G; ++h) out[static_cast<long long>(qbase + h) * kDim + lane] = r[h] + s1[h * kTile + lane];
  builder_sync();
}

// Merge the n_seg segments of one group (its G heads' entries at ent0 + s G +
// h), divide by the softmax sum and back-rotate into out (seo-farm page §2:
// out = R^T o_rot).  Called by every builder thread (lane, half); half h
// merges the heads it owns, then each half sums 64 of the 128 terms of every
// head's back-rotation.  Latency-bound: the loads of up to eight segments, and
// all 64 loads of R a thread needs, are in flight at once.  Not inlined: it
// runs about twice per CTA, and those loads must not take registers from the
// per-tile loop.
template <int G>
__device__ __noinline__ void merge_segments(const float* ws_part, const float* R, float* out, int ent0,
                                            int n_seg, int qbase, float* orot, float* s1, int half, int lane) {
  float w[64];                                  // loaded while the segments merge
  load_r_half(R, half, lane, w);
  merge_segments_r<G>(w, ws_part, out, ent0, n_seg, qbase, orot, s1, half, lane);
}

// One work item: (sequence b, KV head kvh, chunk) of a non-empty chunk.  The
// items of a launch are the real chunks in the order (b, kvh, chunk), numbered
// 0 .. T - 1; CTA c takes the run [c per_cta, (c + 1) per_cta), so every CTA
// gets the same number of chunks whatever the spread of context lengths.  A
// (sequence, KV head) group's consecutive items in one CTA form a segment whose
// partials are merged in the CTA; group g has one segment per CTA in
// [first_cta, last_cta], stored as entry slot g + c (unique: a CTA's groups
// increase with c, and a group's CTAs with g).
struct Item {
  int b, kvh, chunk, ctx, start, n_local, n_tiles, n_blk, group;
  int g0, nch;                                  // the group's first item index and item count
  // CTAs whose runs hold the group's first and last item
  __device__ __forceinline__ int first_cta(int per_cta) const { return g0 / per_cta; }
  __device__ __forceinline__ int last_cta(int per_cta) const { return (g0 + nch - 1) / per_cta; }
};

// Walks the items [first, last) of a CTA from the (b, kvh, chunk) of `first`;
// a sequence's context length is read when the walk enters the sequence, and
// sequences without tokens are stepped over.
struct ItemCursor {
  int it, last, b, kvh, chunk, ctx, nch, csz;
  __device__ ItemCursor(const DecodeArgs& a, int csz_, int first, int last_, int b0, int kvh0, int chunk0)
      : it(first), last(last_), b(b0), kvh(kvh0), chunk(chunk0), csz(csz_) {
    ctx = first < last ? context_of(a, b) : 0;
    nch = (ctx + csz - 1) / csz;
  }
  __device__ __forceinline__ void advance(const DecodeArgs& a) {
    ++it;
    if (++chunk < nch) return;
    chunk = 0;
    if (++kvh < a.n_kv) return;
    kvh = 0;
    if (it >= last) return;
    do {
      if (b + 1 >= a.batch) {             // (only if the lengths changed under the launch)
        it = last;
        return;
      }
      ++b;
      ctx = context_of(a, b);
      nch = (ctx + csz - 1) / csz;
    } while (nch == 0);
  }
  // the next item, if any
  __device__ __forceinline__ bool next(const DecodeArgs& a, int bs_shift, Item& x) {
    if (it >= last) return false;
    x.b = b;
    x.kvh = kvh;
    x.chunk = chunk;
    x.ctx = ctx;
    x.start = chunk * csz;
    x.n_local = min(csz, ctx - x.start);
    x.n_tiles = (x.n_local + kTile - 1) / kTile;
    x.n_blk = (x.n_local + (1 << bs_shift) - 1) >> bs_shift;
    x.group = b * a.n_kv + kvh;
    x.g0 = it - chunk;
    x.nch = nch;
    advance(a);
    return true;
  }
};

// KB, VB, QJ: key MSE bits, value bits and QJL plane (0/1) fixed at compile
// time, or 0, 0, -1 to take them from the arguments; NB: the stored norms'
// width (16 or 32 bits), or 0 to take it from the arguments; BS: the block
// size, or 0 to take it from the arguments.  Two CTAs per SM cap a
// thread at 96 registers (the register file is split over four sub-partitions
// of 16384, and one of them holds five of the two CTAs' eighteen warps).
template <int G, int KB, int VB, int QJ, int CH, int NB, int BS>
__global__ void __launch_bounds__(kThreads, 2) attention_tc_kernel(DecodeArgs a, TcLayout layout) {
  // (with the widths and the block size fixed, the layout -- the one the host
  // computed for the launch -- folds to constants)
  constexpr bool kFixedLayout = KB > 0 && VB > 0 && QJ >= 0 && BS > 0;
  constexpr TcLayout kLayout = kFixedLayout ? tc_layout(G, KB, QJ == 1, VB, BS, CH) : TcLayout{};
  const TcLayout L = kFixedLayout ? kLayout : layout;
  constexpr int N1 = score_cols(G), NO = value_cols(G);
  const int t = threadIdx.x;

  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned, as an offset from smem_raw so that accesses stay shared-space
  uint8_t* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);

  // ---- work split: the real chunks of every sequence, an equal run per CTA ----
  __shared__ int scan_s[kThreads / 32];
  __shared__ int split_s[3];                    // (b, kvh, chunk) of this CTA's first item
  // sequences without context (CTA 0 of a merging launch), in the B operand
  // region, which is zeroed after this prologue (at least 2 KB at any shape)
  int* const empty_s = reinterpret_cast<int*>(smem);
  __shared__ int n_empty_s;
  int n_chunks_total = 0;
  int ch0 = 0, excl0 = 0;                       // pass 0: this thread's sequence (b = t)
  for (int b0 = 0; b0 < a.batch; b0 += kThreads) {
    const int b = b0 + t;
    const int ctx = b < a.batch ? context_of(a, b) : -1;
    const int ch = ctx > 0 ? (ctx + CH - 1) / CH : 0;
    if (a.merge_in_partials && blockIdx.x == 0) {
      // a sequence without context has a zero output, which no item writes
      if (t == 0) n_empty_s = 0;
      __syncthreads();
      if (ctx == 0) empty_s[atomicAdd(&n_empty_s, 1)] = b;
      __syncthreads();
      const int n_empty = n_empty_s;
      for (int e = 0; e < n_empty; ++e) {
        float4* row = reinterpret_cast<float4*>(a.out + static_cast<long long>(empty_s[e]) * a.n_q * kDim);
        for (int i = t; i < a.n_q * (kDim / 4); i += kThreads) row[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
      __syncthreads();
    }
    int excl;
    n_chunks_total += cta_scan<kThreads>(ch, &excl, scan_s);
    if (b0 == 0) {
      ch0 = ch;
      excl0 = excl;
    }
  }
  const int n_items = n_chunks_total * a.n_kv;
  const int per_cta = max(1, (n_items + static_cast<int>(gridDim.x) - 1) / static_cast<int>(gridDim.x));
  const int first = static_cast<int>(blockIdx.x) * per_cta;
  const int last = min(n_items, first + per_cta);
  if (first >= last) return;                    // (uniform: no tensor memory or barrier is set up yet)
  // the sequence holding item `first`: items of sequence b are [lo, lo + ch n_kv)
  auto locate = [&](int b, int ch, int before) {
    const int lo = before * a.n_kv;
    if (ch > 0 && first >= lo && first < lo + ch * a.n_kv) {
      split_s[0] = b;
      split_s[1] = (first - lo) / ch;
      split_s[2] = (first - lo) % ch;
    }
  };
  if (a.batch <= kThreads) {
    locate(t, ch0, excl0);                      // (one pass held the whole batch)
  } else {
    int base = 0;                               // chunks of the sequences before this pass
    for (int b0 = 0; b0 < a.batch; b0 += kThreads) {
      const int b = b0 + t;
      const int ctx = b < a.batch ? context_of(a, b) : 0;
      const int ch = (ctx + CH - 1) / CH;
      int excl;
      const int tot = cta_scan<kThreads>(ch, &excl, scan_s);
      locate(b, ch, base + excl);
      base += tot;
    }
  }
  __syncthreads();

  const int bs = BS > 0 ? BS : a.block_size;          // a power of two that divides CH
  const int bs_shift = BS > 0 ? 31 - __clz(BS) : 31 - __clz(bs);

  const int k_bits = KB > 0 ? KB : a.k_bits;
  const int v_bits = VB > 0 ? VB : a.v_bits;
  const int pk = KB > 0 ? 1 << (KB - 1) : L.pk;     // key sign planes
  const int pq = QJ >= 0 ? QJ : L.pq;                // QJL plane
  const int pv = VB > 0 ? 1 << (VB - 1) : L.pv;     // value sign planes
  const int kp = L.kp;                               // columns per key slot
  const int kbytes = 16 * k_bits;                    // key code bytes per token
  const int vblock = v_bits * 16 * bs;               // value code bytes per (block, head)
  const int k_slots = L.k_slots;
  const bool k_two = L.k_units == 2;                 // a key tile in two units (slot 0: planes 0-2; slot 1: 3 + QJL)

  uint8_t* b_mse = smem + L.off_bmse;
  uint8_t* b_qjl = smem + L.off_bqjl;
  uint8_t* b_v = smem + L.off_bv;
  float* s0 = reinterpret_cast<float*>(smem + L.off_s0);           // [G][CH] scores
  float* s1 = reinterpret_cast<float*>(smem + L.off_s1);           // [G][kTile]: output halves (inside s0)
  float* seg_acc = reinterpret_cast<float*>(smem + L.off_sacc);    // [G][kTile]: the segment's running acc
  uint8_t* kc_s = smem + L.off_kc;                                  // [CH][kbytes]
  uint8_t* kq_s = smem + L.off_kq;                                  // [CH][16]
  uint8_t* kn_s = smem + L.off_kn;                                  // [CH] norms, float32 or float16
  uint8_t* kr_s = smem + L.off_kr;
  uint8_t* vn_s = smem + L.off_vn;
  const bool n16 = NB == 0 ? a.norm16 : NB == 16;                   // norms stored as float16
  const int nb = n16 ? 2 : 4;                                       // bytes of a stored norm
  auto norm_at = [&](const uint8_t* f, int i) {
    return n16 ? __half2float(reinterpret_cast<const __half*>(f)[i]) : reinterpret_cast<const float*>(f)[i];
  };
  uint32_t* vc_s = reinterpret_cast<uint32_t*>(smem + L.off_vc);   // [blk][plane][dim][bs/32]
  // kin / vin: an item's key / value fields landed (one phase per item);
  // kfree / vfree: the builders are done with the key / value fields of an
  // item (256 arrivals); kfull / vfull: the builders stored a slot's planes
  // (256 arrivals); kdone / vdone: the slot's MMAs completed (commit; kdone
  // once per key tile); kudone: the first unit's MMAs of a key tile built in
  // two units completed; sfree: the builders read the score accumulators
  // (256 arrivals); bar_d: drain
  __shared__ __align__(8) uint64_t kin, vin, kfree, vfree, kfull[2], kdone, kudone, sfree, vfull[kMaxValueSlots],
      vdone[kMaxValueSlots], bar_d;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;
  __shared__ float red_s[(kBuilders / 32) * (2 * half_heads(G) + 1)];   // warp totals of up to 2 HG + 1 values
  __shared__ float stat_s[G];                   // chunk max per head
  __shared__ float4 mrg_s[G];                   // per head: the factors of the segment merge (so, si / sv, -a_sum wsum si)
  __shared__ int blk_ok_s[2][CH / 32];          // per item parity: physical block of each block slot is valid
  __shared__ float sv_s;                        // piece scale of the softmax weights
  __shared__ float4 cst_s[G];                   // per head: 1/sigma_mse, 1/sigma_qjl, -ones_mse, -ones_qjl
  __shared__ float vw_s[8];                     // odd Walsh coefficients of the value codebook
  __shared__ int4 pend_s[kMaxPending];          // groups whose merge this CTA owes: (entry base, n_seg, qbase)
  __shared__ int n_pend_s;

  const bool builder = t < kBuilders;
  const int lane = t & (kTile - 1);             // tensor-memory lane (token or coordinate)
  const int half = (t >> 7) & 1;                // which of the two threads of the lane
  const int w0 = 2 * half;                      // this thread's words of every sign plane: w0, w0 + 1
  const uint32_t row_addr = static_cast<uint32_t>(((t >> 5) & 3) * 32) << 16;
  const bool qjl = QJ >= 0 ? QJ == 1 : a.k_qjl != nullptr;
  volatile int* abort = &abort_s;
  const int n_pairs = (pv + 1) / 2;

  // zero the B operands once (their padding rows stay 0)
  for (int i = t; i < L.off_s0 / 16; i += kThreads) reinterpret_cast<uint4*>(smem)[i] = make_uint4(0, 0, 0, 0);
  ptx::fence_async_shared();                    // the MMAs read these bytes through the async proxy
  if (t < 8) vw_s[t] = a.tables->v_walsh[t];
  if (t == kBuilders) {
    abort_s = 0;
    ptx::mbar_init(&kin, 1);
    ptx::mbar_init(&vin, 1);
    ptx::mbar_init(&kfree, kBuilders);
    ptx::mbar_init(&vfree, kBuilders);
    ptx::mbar_init(&kfull[0], kBuilders);
    ptx::mbar_init(&kfull[1], kBuilders);
    ptx::mbar_init(&kdone, 1);
    ptx::mbar_init(&kudone, 1);
    ptx::mbar_init(&sfree, kBuilders);
    for (int i = 0; i < kMaxValueSlots; ++i) {
      ptx::mbar_init(&vfull[i], kBuilders);
      ptx::mbar_init(&vdone[i], 1);
    }
    ptx::mbar_init(&bar_d, 32);
    ptx::fence_mbar_init();
  }
  if (!builder) {
    ptx::tmem_alloc(&tmem_base_s, L.tmem);
    ptx::tmem_relinquish();
  }
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  bool ok = true;
  int drain_k = 0, drain_v = 0;                 // control warp: copy rounds to drain after a failure

  if (!builder) {
    // =================== control warp: copies one item ahead, every MMA ===================
    const int ln = t - kBuilders;
    // lane k copies block k of an item: the key fields (keys = true) or the value fields
    int kin_issued = 0, vin_issued = 0;         // copy rounds issued on kin / vin (one phase each)
    auto copy_fields = [&](const Item& x, int seq, bool keys) {
      ++(keys ? kin_issued : vin_issued);
      bool valid = false;
      long long phys = 0;
      int rows = 0;
      uint32_t bytes = 0;
      if (ln < x.n_blk) {
        const int lblk = (x.start >> bs_shift) + ln;
        phys = a.block_table ? a.block_table[static_cast<long long>(x.b) * a.max_blocks + lblk]
                             : static_cast<long long>(x.b) * a.max_blocks + lblk;
        valid = phys >= 0 && phys < a.num_blocks;
        if (keys) {
          blk_ok_s[seq & 1][ln] = valid;
          if (!valid) atomicCAS(a.error, 0, kErrBlock);
        }
        rows = min(bs, (x.n_local - ln * bs + 31) / 32 * 32);
        if (valid) bytes = keys ? rows * (kbytes + nb + (qjl ? 16 + nb : 0)) : rows * nb + vblock;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) bytes += __shfl_xor_sync(0xffffffffu, bytes, off);
      __syncwarp();                             // blk_ok_s before the arrival the builders acquire
      if (ln == 0) ptx::mbar_arrive_expect_tx(keys ? &kin : &vin, bytes);
      __syncwarp();
      // the chunk holding position ctx - 1 may hold the token a decode step's
      // append (the grid this one may overlap) is writing: wait for that grid
      if (x.start + x.n_local == x.ctx) asm volatile("griddepcontrol.wait;" ::: "memory");
      if (valid) {
        const long long r0 = (phys * a.n_kv + x.kvh) * bs;    // first row of this block
        const int tl0 = ln * bs;
        if (keys) {
          ptx::bulk_load(kc_s + tl0 * kbytes, a.k_codes + r0 * kbytes, rows * kbytes, &kin);
          if (qjl) {
            ptx::bulk_load(kq_s + tl0 * 16, a.k_qjl + r0 * 16, rows * 16, &kin);
            ptx::bulk_load(kr_s + tl0 * nb, static_cast<const uint8_t*>(a.k_rnorm) + r0 * nb, rows * nb, &kin);
          }
          ptx::bulk_load(kn_s + tl0 * nb, static_cast<const uint8_t*>(a.k_norm) + r0 * nb, rows * nb, &kin);
        } else {
          ptx::bulk_load(vn_s + tl0 * nb, static_cast<const uint8_t*>(a.v_norm) + r0 * nb, rows * nb, &vin);
          ptx::bulk_load(vc_s + ln * (vblock / 4), a.v_codes + (phys * a.n_kv + x.kvh) * vblock, vblock,
                         &vin);
        }
      }
    };
    const uint32_t idesc_s = ptx::idesc_e4m3_f32(128, N1);
    const uint32_t idesc_o = ptx::idesc_e4m3_f32(128, NO);
    // the start-address field of a descriptor counts 16-byte units: +2 per 32-byte K step
    const uint64_t desc_mse = ptx::desc_k_sw128(ptx::smem_u32(b_mse));
    const uint64_t desc_qjl = ptx::desc_k_sw128(ptx::smem_u32(b_qjl));
    const uint64_t desc_v = ptx::desc_k_sw128(ptx::smem_u32(b_v));
    const uint32_t mse_plane_step = (L.n1 * 128) >> 4, v_tile_step = (L.no * 128) >> 4;
    const uint32_t d_mse = tmem + L.col_s;
    ItemCursor cursor(a, CH, first, last, split_s[0], split_s[1], split_s[2]);
    int seq = 0, ktile = 0;
    int vslot = 0, vwrap = 0;                   // value unit counter as (slot, times round the slots)
    Item cur, nxt;
    bool have = cursor.next(a, bs_shift, cur);
    if (have) {
      copy_fields(cur, 0, true);
      copy_fields(cur, 0, false);
    }
    while (have && ok) {
      const bool more = cursor.next(a, bs_shift, nxt);
      // scores: tile i once its planes are stored and the previous tile's accumulators were read
      for (int i = 0; i < cur.n_tiles && ok; ++i, ++ktile) {
        if (k_two) {
          // unit 0 (MSE planes 0-2, slot 0) once stored and the previous tile's scores were read
          ok = wait_phase(&kfull[0], ktile & 1, abort, a.error);
          if (ok && ktile > 0) ok = wait_phase(&sfree, (ktile - 1) & 1, abort, a.error);
          if (ok && ptx::elect_one()) {
            ptx::tc_fence_after();
#pragma unroll
            for (int s = 0; s < 3; ++s)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                ptx::mma_e4m3_tmem_a(d_mse, tmem + 32 * s + 8 * kk, desc_mse + s * mse_plane_step + 2 * kk, idesc_s,
                                     (s | kk) != 0);
            ptx::mma_commit(&kudone);
          }
          __syncwarp();
          // unit 1 (MSE plane 3 and the QJL plane, slot 1)
          if (ok) ok = wait_phase(&kfull[1], ktile & 1, abort, a.error);
          if (ok && ptx::elect_one()) {
            ptx::tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              ptx::mma_e4m3_tmem_a(d_mse, tmem + kp + 8 * kk, desc_mse + 3 * mse_plane_step + 2 * kk, idesc_s, true);
            if (qjl)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                ptx::mma_e4m3_tmem_a(d_mse + N1, tmem + kp + 32 + 8 * kk, desc_qjl + 2 * kk, idesc_s, kk != 0);
            if (!(a.debug_withhold && blockIdx.x == 0 && ktile == 0)) ptx::mma_commit(&kdone);
          }
          __syncwarp();
          continue;
        }
        const int slot = k_slots == 2 ? (ktile & 1) : 0;
        ok = wait_phase(&kfull[slot], (k_slots == 2 ? ktile >> 1 : ktile) & 1, abort, a.error);
        if (ok && ktile > 0) ok = wait_phase(&sfree, (ktile - 1) & 1, abort, a.error);
        if (ok && ptx::elect_one()) {
          ptx::tc_fence_after();
          uint32_t a_col = tmem + slot * kp;
          uint64_t dsc = desc_mse;
          for (int s = 0; s < pk; ++s) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              ptx::mma_e4m3_tmem_a(d_mse, a_col + 8 * kk, dsc + 2 * kk, idesc_s, (s | kk) != 0);
            a_col += 32;
            dsc += mse_plane_step;
          }
          if (qjl)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              ptx::mma_e4m3_tmem_a(d_mse + N1, a_col + 8 * kk, desc_qjl + 2 * kk, idesc_s, kk != 0);
          // (a test of the bounded waits withholds the first commit of CTA 0)
          if (!(a.debug_withhold && blockIdx.x == 0 && ktile == 0)) ptx::mma_commit(&kdone);
        }
        __syncwarp();
      }
      // the next item's key fields, once the builders are done with this item's
      if (ok && more) {
        ok = wait_phase(&kfree, seq & 1, abort, a.error);
        if (ok) copy_fields(nxt, seq + 1, true);
      }
      // values: unit u (tile u / n_pairs, plane pair u % n_pairs) from slot u % v_slots
      const int n_units = cur.n_tiles * n_pairs;
      for (int u = 0, tile = 0, pair = 0; u < n_units && ok; ++u) {
        const int slot = vslot;
        ok = wait_phase(&vfull[slot], vwrap & 1, abort, a.error);
        if (ok && ptx::elect_one()) {
          ptx::tc_fence_after();
          const uint64_t dsc = desc_v + tile * v_tile_step;
          const uint32_t a_col = tmem + slot * kValueSlot;
          const uint32_t d_col = tmem + L.col_o + 2 * pair * L.no;
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            ptx::mma_e4m3_tmem_a(d_col, a_col + 8 * kk, dsc + 2 * kk, idesc_o, (tile | kk) != 0);
          if (2 * pair + 1 < pv)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              ptx::mma_e4m3_tmem_a(d_col + L.no, a_col + 32 + 8 * kk, dsc + 2 * kk, idesc_o, (tile | kk) != 0);
          ptx::mma_commit(&vdone[slot]);
        }
        __syncwarp();
        if (++pair == n_pairs) {
          pair = 0;
          ++tile;
        }
        if (++vslot == L.v_slots) {
          vslot = 0;
          ++vwrap;
        }
      }
      // the next item's value fields, once the builders loaded this item's value words
      if (ok && more) {
        ok = wait_phase(&vfree, seq & 1, abort, a.error);
        if (ok) copy_fields(nxt, seq + 1, false);
      }
      cur = nxt;
      have = more;
      ++seq;
    }
    drain_k = kin_issued;
    drain_v = vin_issued;
  } else {
    // =================== builders ===================
    constexpr int HG = half_heads(G), HC = score_half(G);
    ItemCursor cursor(a, CH, first, last, split_s[0], split_s[1], split_s[2]);
    int seq = 0, ktile = 0, cur_group = -1;
    int vslot = 0, vwrap = 0;                     // value unit counter as (slot, times round the slots)
    const int wpd_shift = bs_shift - 5;         // log2 of the words per coordinate in a block
    const int kpos_lane = k_position(lane);     // K position of this lane's token in a tile
    // The CTA's segment of the current group is merged chunk by chunk: thread
    // t < G keeps head t's running max and sum in registers (seg_m, seg_l),
    // acc[coordinate lane] of head h is in seg_acc, read and written only by
    // the thread that owns (h, lane).
    float seg_m = -INFINITY, seg_l = 0.f;
#pragma unroll
    for (int h = 0; h < G; ++h)
      if (h / HG == half) seg_acc[h * kTile + lane] = 0.f;

    if (t == 0) n_pend_s = 0;

    Item x;
    bool have = cursor.next(a, bs_shift, x);
    while (ok && have) {
      const int group = x.group;
      const int qbase = x.b * a.n_q + x.kvh * G;
      const int* blk_ok = blk_ok_s[seq & 1];
      // B_K: the group's prepared score operand pieces into the swizzled layout
      // (the previous item's score MMAs have completed: its last kdone was
      // waited for); row n = score_row(G, h, i) of plane s, 16-byte chunk c of
      // a row at c ^ (n % 8)
      if (group != cur_group) {
        asm volatile("griddepcontrol.wait;" ::: "memory");   // the query operands come from the previous grid
        const int nk = pk + pq;
        constexpr int QP = q_pieces(G);
        const int per_head = nk * QP * 8;           // 16-byte chunks per head taken
        for (int idx = t; idx < G * per_head; idx += kBuilders) {
          const int h = idx / per_head, r = idx - h * per_head;
          const int s = r / (QP * 8), i = (r / 8) % QP, c = r % 8;
          const uint4 v = reinterpret_cast<const uint4*>(a.ws_bk + static_cast<long long>(qbase + h) * a.bk_stride)
              [(s * kQPieces + i) * 8 + c];
          const int n = score_row(G, h, i);
          uint8_t* dst = s < pk ? b_mse + s * L.n1 * 128 : b_qjl;
          *reinterpret_cast<uint4*>(dst + n * 128 + ((c ^ (n & 7)) << 4)) = v;
        }
        // per head: 1 / sigma_mse, 1 / sigma_qjl, and the -1 halves of the +-1 sums
        if (t < 4 * G) {
          const int h = t >> 2, k = t & 3;
          const float* hdr = reinterpret_cast<const float*>(a.ws_bk + static_cast<long long>(qbase + h) * a.bk_stride +
                                                            nk * kQPieces * 128);
          reinterpret_cast<float*>(cst_s + h)[k] = k < 2 ? hdr[2 + k] : -hdr[4 + (k - 2)];
        }
        ptx::fence_async_shared();
        builder_sync();
        cur_group = group;
      }
      ok = wait_phase(&kin, seq & 1, abort, a.error);

      // thread (lane, half) owns the query heads h with h / HG == half: it turns
      // their accumulators of a key tile into the scaled scores of token lane,
      // s = scale (n_k <q_rot, k_mse> + gamma coef <q_s, signs>), into s0, and
      // keeps their running max (an accumulator holds sigma times the 0/1-bit
      // sum, so the +-1 sum is acc / sigma - ones)
      float mx[HG + 1];                           // owned heads' score max, then the value-norm max
#pragma unroll
      for (int j = 0; j <= HG; ++j) mx[j] = j < HG ? -INFINITY : 0.f;
      // (templated on the half, so that the owned heads are compile-time indices;
      // `release` runs once the last accumulator column is in registers, so the
      // next tile's MMAs may start while the scores are being formed)
      auto read_scores_half = [&](int i, auto half_c, auto release) {
        constexpr int H0 = decltype(half_c)::value * HG;
        if constexpr (H0 < G) {
          const int tl = i * kTile + lane;
          const bool valid = tl < x.n_local && blk_ok[tl >> bs_shift];
          // a head's pieces p_0 .. p_{Q-1} sum as p_0 + (p_1 + (p_2 + ...) / 16) / 16 (Horner: Q - 1 FMAs);
          // four pieces as (p_0 + p_2 / 256) + (p_1 + p_3 / 256) / 16, the first step on both pairs at once
          constexpr int QP = q_pieces(G);
          auto piece_sum = [](const uint32_t* v) {
            if constexpr (QP == 4) {
              const float2 h = __ffma2_rn(make_float2(__uint_as_float(v[2]), __uint_as_float(v[3])),
                                          make_float2(0.00390625f, 0.00390625f),
                                          make_float2(__uint_as_float(v[0]), __uint_as_float(v[1])));
              return fmaf(h.y, 0.0625f, h.x);
            } else {
              float r = __uint_as_float(v[QP - 1]);
#pragma unroll
              for (int i = QP - 2; i >= 0; --i) r = fmaf(r, 0.0625f, __uint_as_float(v[i]));
              return r;
            }
          };
          float am[HG], aq[HG];
#pragma unroll
          for (int j = 0; j < HG; ++j) am[j] = aq[j] = 0.f;
          static_assert(HC == 16, "one 16-column load per half and kind");
          {
            uint32_t v[16];
            ptx::tmem_ld16(tmem + row_addr + L.col_s + (H0 / HG) * HC, v);
#pragma unroll
            for (int j = 0; j < HG; ++j) am[j] = piece_sum(v + j * QP);
            if (qjl) {
              ptx::tmem_ld16(tmem + row_addr + L.col_s + N1 + (H0 / HG) * HC, v);
              release();
#pragma unroll
              for (int j = 0; j < HG; ++j) aq[j] = piece_sum(v + j * QP);
            } else {
              release();
            }
          }
          const float kn = norm_at(kn_s, tl), kr = norm_at(kr_s, tl);   // (tl < CH: in bounds; selected below)
          const float nk = valid ? a.scale * kn : 0.f;
          const float gk = valid && qjl ? a.scale * kr * a.qjl_coef : 0.f;
#pragma unroll
          for (int j = 0; j < HG; ++j) {
            const int h = H0 + j;
            if (h >= G) break;
            // (mse, qv) = (am / sigma_mse - ones_mse, aq / sigma_qjl - ones_qjl) in one paired FMA, the
            // head's constants in one 16-byte shared-memory load (kept in registers across the key phase
            // they would take sixteen); without QJL aq = 0 and gk = 0, so the second half drops out
            const float4 c = cst_s[h];
            const float2 mq2 = __ffma2_rn(make_float2(am[j], aq[j]), make_float2(c.x, c.y), make_float2(c.z, c.w));
            const float mse = mq2.x, qv = mq2.y;
            const float sc = valid ? fmaf(nk, mse, gk * qv) : -INFINITY;
            s0[h * CH + i * kTile + kpos_lane] = sc;   // (in K order: the weights read four at once)
            mx[j] = fmaxf(mx[j], sc);
          }
        } else {
          release();                              // (G = 1: the second half owns no head)
        }
      };
      // wait for the MMAs of key tile i (global index g), read its accumulators, release them
      auto take_scores = [&](int i, int g) {
        ok = ok && wait_phase(&kdone, g & 1, abort, a.error);
        ptx::tc_fence_after();
        auto release = [&]() {
          ptx::tc_fence_before();
          ptx::mbar_arrive(&sfree);
        };
        if (!ok) release();
        else if (half == 0) read_scores_half(i, std::integral_constant<int, 0>{}, release);
        else read_scores_half(i, std::integral_constant<int, 1>{}, release);
      };

      // ---- scores: the planes of tile i are built while the MMAs of tile i - 1 run ----
      const int k0 = ktile;
      for (int i = 0; i < x.n_tiles && ok; ++i, ++ktile) {
        const int slot = k_slots == 2 ? (ktile & 1) : 0;
        if (k_two) {
          // slot 0 once the previous tile's unit-0 MMAs completed
          if (ktile > 0) {
            ok = wait_phase(&kudone, (ktile - 1) & 1, abort, a.error);
            ptx::tc_fence_after();
          }
        } else if (k_slots == 1 && i > 0) {
          take_scores(i - 1, ktile - 1);
        }
        if (!ok) break;
        const int tl = i * kTile + lane;
        // loaded for every token slot of the tile (tl < CH, inside the
        // copied fields): a slot past the context or in a skipped block holds
        // stale but finite operand bytes, and its score is set to -inf
        uint32_t bw[4][2] = {};
        uint32_t sg[2] = {};
        {
          const uint2* kc = reinterpret_cast<const uint2*>(kc_s + tl * kbytes);
#pragma unroll
          for (int p = 0; p < 4; ++p)
            if (p < k_bits) {
              const uint2 w = kc[2 * p + half];
              bw[p][0] = w.x;
              bw[p][1] = w.y;
            }
          if (qjl) {
            const uint2 w = reinterpret_cast<const uint2*>(kq_s + tl * 16)[half];
            sg[0] = w.x;
            sg[1] = w.y;
          }
        }
        if (k_two) {
          // unit 0 into slot 0; the previous tile's scores (which frees slot 1); unit 1 into slot 1
          key_unit3(tmem + row_addr, bw, sg, qjl, w0, 0);
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          ptx::mbar_arrive(&kfull[0]);
          if (i > 0) take_scores(i - 1, ktile - 1);
          if (!ok) break;
          key_unit3(tmem + row_addr + kp, bw, sg, qjl, w0, 1);
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          ptx::mbar_arrive(&kfull[1]);
          continue;
        }
        const uint32_t base = tmem + row_addr + slot * kp;
        switch (k_bits) {
          case 1: key_planes<1>(base, bw, sg, qjl, w0); break;
          case 2: key_planes<2>(base, bw, sg, qjl, w0); break;
          case 3: key_planes<3>(base, bw, sg, qjl, w0); break;
          default: key_planes<4>(base, bw, sg, qjl, w0); break;
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(&kfull[slot]);
        if (k_slots == 2 && i > 0) take_scores(i - 1, ktile - 1);
      }
      if (ok) take_scores(x.n_tiles - 1, k0 + x.n_tiles - 1);
      ptx::mbar_arrive(&kfree);                   // this item's key fields are no longer read
      ok = ok && wait_phase(&vin, seq & 1, abort, a.error);

      // ---- softmax max over the chunk; B_V pieces of exp(s - m) n_v ----
      // (after a failed wait the loop reads stale but in-bounds norms, and every
      // builder leaves at the barrier that ANDs the flags)
      // The norm of a slot past the context or in a skipped block -- stale or
      // uncopied bytes -- is set to 0 in place, so the weight loop below needs
      // no validity test: such a slot's score is -inf, its exponential 0, and
      // its weight 0 * 0.
      for (int i = t; i < x.n_tiles * kTile; i += kBuilders) {
        if (i < x.n_local && blk_ok[i >> bs_shift]) {
          mx[HG] = fmaxf(mx[HG], norm_at(vn_s, i));
        } else if (n16) {
          reinterpret_cast<uint16_t*>(vn_s)[i] = 0;
        } else {
          reinterpret_cast<float*>(vn_s)[i] = 0.f;
        }
      }
      {
        // chunk max of the owned heads over this half's warps; value-norm max over all
        ok = ok && *abort == 0;
        warp_totals(mx, red_s, MaxOp(), &ok);
        if (!ok) break;
        float vmax = 0.f;
#pragma unroll
        for (int w = 0; w < kBuilders / 32; ++w) vmax = fmaxf(vmax, red_s[w * (HG + 1) + HG]);
#pragma unroll
        for (int j = 0; j < HG; ++j) {
          mx[j] = half_total<HG + 1>(red_s, half, j, MaxOp());
          if ((t & 127) == 0 && half * HG + j < G) stat_s[half * HG + j] = mx[j];
        }
        mx[HG] = vmax;
      }
      // the pieces carry 2 e n_v sv / beta_t, below 2 * 64 * max n_v * sv
      const float sv = piece_scale(2.f * kMaxBitInvScale * mx[HG]);
      // Thread t takes head hq = warp % G and, per pass, one quad of a tile:
      // tokens 32 g + i + 8 k (k = 0..3) sit at the consecutive K positions
      // 32 g + 4 i + k, so their scores (stored in K order) are one float4 and
      // every piece of their four weights is one 32-bit word of its B_V row.
      // (kBuilders is a multiple of 32 G, so every pass of a thread has the same head.)
      const int hq = (t >> 5) % G;
      const float mq = half_total<HG + 1>(red_s, hq / HG, hq % HG, MaxOp());   // head hq's chunk max
      float lw0 = 0.f, lw1 = 0.f;                 // head hq: sum of e, sum of e n_v
      {
        const int q = t & 31, gq = q >> 3, i = q & 7;
        const int kp0 = 32 * gq + 4 * i;
        // ib: a power of two, so lw1 is summed ib-scaled and rescaled exactly after the loop
        const float ib = 2.f * bit_inv_scale(i) * sv;
        constexpr float kLog2e = 1.4426950408889634f;
        const float2 l2e = make_float2(kLog2e, kLog2e);
        // (the same rounding for every token; a head without a valid token in
        // the chunk has m = -inf and every score -inf: 2^(-inf) = 0, not nan)
        const float nm = mq == -INFINITY ? 0.f : -mq * kLog2e;
        const float2 nml = make_float2(nm, nm);
        const float2 ib2 = make_float2(ib, ib);
        float2 se2 = make_float2(0.f, 0.f), sw2 = make_float2(0.f, 0.f);   // sums of e and of e n_v ib
        const int units = x.n_tiles * 32 * G;
        for (int u = t; u < units; u += kBuilders) {
          const int tile = u / (32 * G);
          const int tl0 = tile * kTile + 32 * gq + i;           // tokens tl0 + 8 k
          const float4 sc = *reinterpret_cast<const float4*>(s0 + hq * CH + tile * kTile + kp0);
          // exp(s - m) = 2^(s log2 e - m log2 e), two tokens per fused multiply-add
          const float2 a01 = __ffma2_rn(make_float2(sc.x, sc.y), l2e, nml);
          const float2 a23 = __ffma2_rn(make_float2(sc.z, sc.w), l2e, nml);
          const float2 e01 = make_float2(ex2_approx(a01.x), ex2_approx(a01.y));
          const float2 e23 = make_float2(ex2_approx(a23.x), ex2_approx(a23.y));
          const float2 n01 = __fmul2_rn(make_float2(norm_at(vn_s, tl0), norm_at(vn_s, tl0 + 8)), ib2);
          const float2 n23 = __fmul2_rn(make_float2(norm_at(vn_s, tl0 + 16), norm_at(vn_s, tl0 + 24)), ib2);
          const float2 w01 = __fmul2_rn(e01, n01), w23 = __fmul2_rn(e23, n23);
          se2 = __fadd2_rn(se2, __fadd2_rn(e01, e23));
          sw2 = __fadd2_rn(sw2, __fadd2_rn(w01, w23));
          float w[4] = {w01.x, w01.y, w23.x, w23.y};
          uint8_t* rows = b_v + tile * L.no * 128;
#pragma unroll
          for (int p = 0; p < kVPieces; ++p) {
            const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(w[0], w[1]), __NV_SATFINITE, __NV_E4M3);
            const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(w[2], w[3]), __NV_SATFINITE, __NV_E4M3);
            *reinterpret_cast<uint32_t*>(rows + sw128(hq * kVPieces + p, kp0)) =
                static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
            if (p + 1 < kVPieces) {               // each piece is the e4m3 rounding of what is left, times 16
              const float2 bl = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(lo, __NV_E4M3)));
              const float2 bh = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(hi, __NV_E4M3)));
              // (w - b) exactly (b is w's nearest e4m3 value), then times 16; two tokens per instruction
              const float2 m1 = make_float2(-1.f, -1.f), x16 = make_float2(16.f, 16.f);
              const float2 d01 = __fmul2_rn(__ffma2_rn(bl, m1, make_float2(w[0], w[1])), x16);
              const float2 d23 = __fmul2_rn(__ffma2_rn(bh, m1, make_float2(w[2], w[3])), x16);
              w[0] = d01.x;
              w[1] = d01.y;
              w[2] = d23.x;
              w[3] = d23.y;
            }
          }
        }
        lw0 = se2.x + se2.y;
        lw1 = (sw2.x + sw2.y) * (1.f / ib);       // exact scaling: ib is a power of two
      }
      if (t == 0) sv_s = sv;
      // (no barrier: every builder's B_V pieces precede its first vfull arrival,
      // and the control warp issues a value MMA only after all 256 arrived)
      ptx::fence_async_shared();

      // ---- values: lane d owns coordinate d; units of two sign planes rotate through the slots ----
      int last_slot = 0, last_wrap = 0;
      for (int tile = 0; tile < x.n_tiles && ok; ++tile) {
        uint32_t bw[4][2] = {};                   // [bit-plane][this thread's 32-token groups]
        // (every 32-token group of the tile, inside the copied fields: a group
        // past the context or in a skipped block gets weight 0)
        if constexpr (BS > 0 && BS % 64 == 0) {
          // the thread's two groups are consecutive words of one block's rows, at an even word: one 8-byte load
          const int tl = tile * kTile + 32 * w0;
          const uint32_t* src = vc_s + (tl >> bs_shift) * (vblock / 4) + ((tl & (bs - 1)) >> 5) + (lane << wpd_shift);
#pragma unroll
          for (int p = 0; p < 4; ++p)
            if (p < v_bits) {
              const uint2 pw = *reinterpret_cast<const uint2*>(src + ((p * 128) << wpd_shift));
              bw[p][0] = pw.x;
              bw[p][1] = pw.y;
            }
        } else {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int tl = tile * kTile + 32 * (w0 + c);
            const uint32_t* src =
                vc_s + (tl >> bs_shift) * (vblock / 4) + ((tl & (bs - 1)) >> 5) + (lane << wpd_shift);
#pragma unroll
            for (int p = 0; p < 4; ++p)
              if (p < v_bits) bw[p][c] = src[(p * 128) << wpd_shift];
          }
        }
        if (tile == x.n_tiles - 1) ptx::mbar_arrive(&vfree);   // the value fields are no longer read
        // (a compile-time trip count when the value width is fixed, so the
        // plane pair of every unit folds)
        constexpr int kMaxPairs = VB > 0 ? ((1 << (VB - 1)) + 1) / 2 : 4;
#pragma unroll
        for (int pair = 0; pair < kMaxPairs; ++pair) {
          if (pair >= n_pairs || !ok) break;
          const int slot = vslot;
          last_slot = vslot;
          last_wrap = vwrap;
          if (++vslot == L.v_slots) {
            vslot = 0;
            ++vwrap;
          }
          if (last_wrap > 0) {                    // the slot's previous unit has completed
            ok = wait_phase(&vdone[slot], (last_wrap - 1) & 1, abort, a.error);
            ptx::tc_fence_after();
            if (!ok) break;
          }
          const uint32_t base = tmem + row_addr + slot * kValueSlot;
          switch (v_bits) {
            case 1: value_pair<1>(base, bw, pair, w0); break;
            case 2: value_pair<2>(base, bw, pair, w0); break;
            case 3: value_pair<3>(base, bw, pair, w0); break;
            default: value_pair<4>(base, bw, pair, w0); break;
          }
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          ptx::mbar_arrive(&vfull[slot]);
        }
      }
      {
        // sums of e and of e n_v per head (while the last value MMAs run): warp w holds head w % G's,
        // added in warp order
        const float lw[2] = {lw0, lw1};
        warp_totals(lw, red_s, SumOp());
        if (t < G) {
          float se = 0.f, sw = 0.f;
          for (int w = t; w < kBuilders / 32; w += G) {
            se += red_s[2 * w];
            sw += red_s[2 * w + 1];
          }
          // head t: this chunk's (max, sum) into the segment's, and the factors every lane applies to its
          // acc: acc so + (o / sv - a_sum wsum) si
          const float mi = stat_s[t];
          const float mn = fmaxf(seg_m, mi);
          const float so = seg_m == -INFINITY ? 0.f : __expf(seg_m - mn);
          const float si = mi == -INFINITY ? 0.f : __expf(mi - mn);
          float a_sum = 0.f;                      // sum_S a_S: the -1 half of every sign product
          for (int s = 0; s < pv; ++s) a_sum += vw_s[s];
          const float sis = si / sv_s;            // exact: sv is a power of two
          mrg_s[t] = make_float4(so, sis, -a_sum * sw * si, 0.f);
          seg_m = mn;
          seg_l = fmaf(seg_l, so, se * si);
        }
      }

      // the item's last commit (a commit covers every earlier MMA)
      if (ok) ok = wait_phase(&vdone[last_slot], last_wrap & 1, abort, a.error);
      ptx::tc_fence_after();

      // ---- partial output of this chunk: half h reads the planes s with s % 2 == h ----
      float o[G];
#pragma unroll
      for (int h = 0; h < G; ++h) o[h] = 0.f;
      if (ok) {
        for (int s = half; s < pv; s += 2) {
          const float ws = vw_s[s];
#pragma unroll
          for (int c0 = 0; c0 < NO; c0 += 16) {
            uint32_t v[16];
            ptx::tmem_ld16(tmem + row_addr + L.col_o + s * L.no + c0, v);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int h = (c0 + j) / kVPieces, piece = (c0 + j) % kVPieces;
              if (h < G) o[h] = fmaf(ws * inv16_pow(piece), __uint_as_float(v[j]), o[h]);
            }
          }
        }
      }
      ptx::tc_fence_before();
      // each half keeps the heads it owns; the other half's sums for them come through s1
#pragma unroll
      for (int h = 0; h < G; ++h)
        if (h / HG != half) s1[h * kTile + lane] = o[h];
      ok = builder_all(ok && *abort == 0);
      if (ok) {
        // this chunk's acc into the segment's running acc
#pragma unroll
        for (int h = 0; h < G; ++h) {
          if (h / HG != half) continue;
          const float4 c = mrg_s[h];
          seg_acc[h * kTile + lane] = fmaf(seg_acc[h * kTile + lane], c.x, fmaf(o[h] + s1[h * kTile + lane], c.y, c.z));
        }
      }
      // (no barrier before the next item: the ones in its key and softmax phases
      // come before anything there writes s1, stat_s or mrg_s)
      Item y;
      const bool more = cursor.next(a, bs_shift, y);
      if (ok && (!more || y.group != x.group)) {
        // ---- the segment ends: its partials go to entry slot group + CTA ----
        const long long ent0 = (static_cast<long long>(x.group) + blockIdx.x) * G;
#pragma unroll
        for (int h = 0; h < G; ++h) {
          if (h / HG != half) continue;
          a.ws_part[(ent0 + h) * kPartStride + 4 + lane] = seg_acc[h * kTile + lane];
          seg_acc[h * kTile + lane] = 0.f;
        }
        if (t < G) {
          float* part = a.ws_part + (ent0 + t) * kPartStride;
          part[0] = seg_m;
          part[1] = seg_l;
          seg_m = -INFINITY;
          seg_l = 0.f;
        }
        const int f_cta = x.first_cta(per_cta);
        const int n_seg = x.last_cta(per_cta) - f_cta + 1;
        if (f_cta == static_cast<int>(blockIdx.x) && t < G)
          a.ws_seg[qbase + t] = SegInfo{(x.group + f_cta) * G + t, n_seg, G, 0};
        if (a.merge_in_partials) {
          // The CTA that ends a group's last segment owes its merge.  It runs
          // the merges it owes after its last item (a merge here would stall
          // the copy and MMA pipeline): listed in shared memory, or, when the
          // list is full, marked in the group's ticket word (-1 - CTA) and
          // found again by walking the run once more.
          builder_sync();                         // every builder's partial stores precede the ticket
          if (t == 0) {
            bool owe = true;                      // (a group inside this run has no other contributor)
            if (n_seg > 1) {
              // one acquire-release add at GPU scope: it publishes this CTA's partials (every builder's
              // stores precede it through the barrier above), and the CTA that completes the count sees
              // every other contributor's
              int prev;
              asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;" : "=r"(prev) : "l"(a.ws_ticket + x.group) : "memory");
              owe = prev == n_seg - 1;
            }
            if (owe) {
              if (n_pend_s < kMaxPending) {
                pend_s[n_pend_s++] = make_int4((x.group + f_cta) * G, n_seg, qbase, 0);
              } else {
                a.ws_ticket[x.group] = -1 - static_cast<int>(blockIdx.x);
                n_pend_s = kMaxPending + 1;       // (overflow)
              }
            }
          }
        }
      }
      x = y;
      have = more;
      ++seq;
    }
    if (ok && a.merge_in_partials) {
      // the merges this CTA owes, by every builder (uniform: read after a barrier)
      builder_sync();
      const int np = n_pend_s;
      for (int p = 0; p < min(np, kMaxPending); ++p) {
        const int4 e = pend_s[p];
        merge_segments<G>(a.ws_part, a.R, a.out, e.x, e.y, e.z, s0, s1, half, lane);
      }
      if (np > kMaxPending) {
        // the overflow: the run's groups once more, those whose ticket word names this CTA
        ItemCursor again(a, CH, first, last, split_s[0], split_s[1], split_s[2]);
        Item y;
        int prev = -1;
        while (again.next(a, bs_shift, y)) {
          if (y.group == prev) continue;
          prev = y.group;
          if (__ldcg(a.ws_ticket + y.group) != -1 - static_cast<int>(blockIdx.x)) continue;
          const int f_cta = y.first_cta(per_cta);
          merge_segments<G>(a.ws_part, a.R, a.out, (y.group + f_cta) * G, y.last_cta(per_cta) - f_cta + 1,
                            y.b * a.n_q + y.kvh * G, s0, s1, half, lane);
        }
      }
    }
  }

  // a grid launched as a programmatic dependent of this one may start once
  // every CTA got here (and waits for this grid before it reads anything)
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  ptx::tc_fence_before();
  __syncthreads();
  if (!builder) {
    if (*abort != 0) {
      // a wait gave up: let every issued copy and MMA finish before the memory
      // goes (each lane commits, covering whichever lane issued)
      ptx::mma_commit(&bar_d);
      if (t == kBuilders) {
        if (drain_k > 0) ptx::drain_bar(&kin, (drain_k - 1) & 1);
        if (drain_v > 0) ptx::drain_bar(&vin, (drain_v - 1) & 1);
        ptx::drain_bar(&bar_d, 0);
      }
      __syncwarp();
    }
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, L.tmem);
  }
}

// Whether two CTAs of this layout fit an SM: half of tensor memory each, and
// dynamic plus static shared memory (under kStaticSmemBound for every build)
// plus the driver's per-CTA reservation within half of the SM's shared memory
// (queried once from the current device; 228 KB and 1 KB if the query fails).
constexpr int kStaticSmemBound = 1536;
bool two_ctas_fit(const TcLayout& l) {
  static const int per_sm_half = [] {
    int dev = 0, per_sm = 0, reserved = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess) {
      per_sm = 228 * 1024;
      reserved = 1024;
    }
    return per_sm / 2 - reserved;
  }();
  return l.tmem <= 256 && l.smem_bytes + kStaticSmemBound <= per_sm_half;
}

// Chunk length of the tensor-core kernel for this shape: 512 tokens, or 256
// when a 512-token layout would not leave room for two CTAs per SM and the
// blocks divide 256 (the partials are per segment, so the chunk length is the
// kernel's own choice).
int tc_chunk(const DecodeArgs& a) {
  const TcLayout l = tc_layout(a.group, a.k_bits, a.k_qjl != nullptr, a.v_bits, a.block_size, 512);
  const bool two = two_ctas_fit(l);
  return !two && 256 % a.block_size == 0 ? 256 : 512;
}

bool tc_decode_supported(const DecodeArgs& a, bool walsh_ok) {
  if (!walsh_ok || a.ws_bk == nullptr || a.block_size % 32 != 0 || 512 % a.block_size != 0) return false;
  if (a.k_bits < 1 || a.k_bits > 4 || a.v_bits < 1 || a.v_bits > 4) return false;
  if (a.group != 1 && a.group != 2 && a.group != 4 && a.group != 8) return false;
  const TcLayout l = tc_layout(a.group, a.k_bits, a.k_qjl != nullptr, a.v_bits, a.block_size, tc_chunk(a));
  return l.cols <= 512 && l.smem_bytes <= 200 * 1024;
}

// CTAs of the persistent tensor-core grid: two per SM when a CTA's tensor
// memory and shared memory leave room for a second, else one; no more than
// the batch could have chunks, and at least one (with no chunk at all it still
// writes the zero outputs).
int tc_grid(const DecodeArgs& a) {
  const int chunk = tc_chunk(a);
  const TcLayout l = tc_layout(a.group, a.k_bits, a.k_qjl != nullptr, a.v_bits, a.block_size, chunk);
  const int per_sm = two_ctas_fit(l) ? 2 : 1;
  const int max_items = (a.max_context + chunk - 1) / chunk;
  const long long bound = static_cast<long long>(a.batch) * a.n_kv * max_items;
  const long long slots = static_cast<long long>(per_sm) * (a.num_sms > 0 ? a.num_sms : 148);
  return static_cast<int>(bound < 1 ? 1 : bound < slots ? bound : slots);
}

template <int G>
cudaError_t launch_g(const DecodeArgs& a, cudaStream_t stream, bool early) {
  const int chunk = tc_chunk(a);
  const TcLayout l = tc_layout(G, a.k_bits, a.k_qjl != nullptr, a.v_bits, a.block_size, chunk);
  // 3-bit keys (2 MSE bits + the QJL bit) with 3-bit values, and (eight
  // query heads per KV head) 4-bit keys with 2-bit values, in 64-token blocks
  // and 512-token items, have their own builds with the widths, the norm
  // width, the block size and so the layout folded in; other shapes are read
  // at run time
  const bool common = a.k_qjl != nullptr && chunk == 512 && a.block_size == 64;
  const bool k3v3 = common && a.k_bits == 2 && a.v_bits == 3;
  const bool k4v2 = common && G == 8 && a.k_bits == 3 && a.v_bits == 2;
  auto kernel = chunk == 512 ? attention_tc_kernel<G, 0, 0, -1, 512, 0, 0> : attention_tc_kernel<G, 0, 0, -1, 256, 0, 0>;
  if (k3v3)
    kernel = a.norm16 ? attention_tc_kernel<G, 2, 3, 1, 512, 16, 64> : attention_tc_kernel<G, 2, 3, 1, 512, 32, 64>;
  if constexpr (G == 8)
    if (k4v2)
      kernel = a.norm16 ? attention_tc_kernel<G, 3, 2, 1, 512, 16, 64> : attention_tc_kernel<G, 3, 2, 1, 512, 32, 64>;
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, l.smem_bytes);
  if (err != cudaSuccess) return err;
  // a persistent grid (tc_grid); the kernel splits the real chunks of the
  // batch into equal runs, one per CTA, so that consecutive items share the
  // query operands and the next item's fields load while the current one
  // computes
  const int n_ctas = tc_grid(a);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = l.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = early ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, a, l);
}

// The merge as its own launch, one 256-thread CTA per (sequence, KV head)
// group: merge_segments over the entries the partials kernel listed for the
// group (slot group + CTA, G heads side by side), so that R is loaded once
// per G heads.  A programmatic dependent of the partials kernel: it waits for
// that grid before it reads any entry.
template <int G>
__global__ void __launch_bounds__(kBuilders) merge_groups_kernel(DecodeArgs a) {
  __shared__ __align__(16) float orot_s[G * kTile];
  __shared__ __align__(16) float half_s[G * kTile];
  const int g = blockIdx.x;
  const int b = g / a.n_kv, kvh = g - b * a.n_kv;
  const int qbase = b * a.n_q + kvh * G;
  const int half = (threadIdx.x >> 7) & 1, lane = threadIdx.x & 127;
  const int ctx = context_of(a, b);
  float w[64];                                    // (R is no output of the partials launch: loaded before the wait)
  load_r_half(a.R, half, lane, w);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (ctx == 0) {
    for (int i = threadIdx.x; i < G * kDim; i += kBuilders) a.out[static_cast<long long>(qbase) * kDim + i] = 0.f;
    return;
  }
  const SegInfo seg = a.ws_seg[qbase];            // head 0: entries base + s G, the others follow it
  // (a partials CTA that stopped early leaves a stale record: check it)
  if (seg.count < 1 || seg.base < 0 || seg.stride != G ||
      static_cast<long long>(seg.base) + static_cast<long long>(seg.count) * G > a.part_cap) {
    if (threadIdx.x == 0) atomicCAS(a.error, 0, kErrPartials);
    for (int i = threadIdx.x; i < G * kDim; i += kBuilders) a.out[static_cast<long long>(qbase) * kDim + i] = 0.f;
    return;
  }
  merge_segments_r<G>(w, a.ws_part, a.out, seg.base, seg.count, qbase, orot_s, half_s, half, lane);
}

// The merge as its own launch for a few (sequence, KV head) groups with many
// segments each (long contexts over a small batch): one 512-thread CTA per
// query head, whose four quarters merge every fourth segment side by side with
// sixteen segments' loads in flight each, so that a head's merge is about one
// memory round trip long and the heads run on different SMs.  Thread
// (lane, quarter) holds coordinate lane; then thread (o = lane, quarter) sums
// 32 of the 128 terms of the back-rotation.
template <int G>
__global__ void __launch_bounds__(kHeadMergeThreads) merge_heads_kernel(DecodeArgs a) {
  constexpr int kQ = kHeadMergeThreads / kTile;   // quarters of 128 lanes
  constexpr int kBatch = 16;                      // a quarter's segment loads in flight at once
  __shared__ float ml_s[kQ][2];
  __shared__ float acc_s[kQ][kTile];
  __shared__ __align__(16) float orot_s[kTile];
  const int v = blockIdx.x;                       // query head b n_q + hq
  const int b = v / a.n_q;
  const int h = (v - b * a.n_q) % G;              // head within its group
  const int qbase = v - h;
  const int t = threadIdx.x, qt = t / kTile, lane = t & (kTile - 1);
  constexpr int kRows = kDim / kQ;                // rows of R per quarter
  float w[kRows];                                 // R[kRows qt + i][lane] (no output of the partials launch:
  const float* rp = a.R + (kRows * qt) * kDim + lane;   // loaded before the wait)
#pragma unroll
  for (int i = 0; i < kRows; ++i) w[i] = __ldg(rp + i * kDim);
  const int ctx = context_of(a, b);
  asm volatile("griddepcontrol.wait;" ::: "memory");
  float* const out = a.out + static_cast<long long>(v) * kDim;
  if (ctx == 0) {
    if (t < kDim) out[t] = 0.f;
    return;
  }
  const SegInfo seg = a.ws_seg[qbase];            // head 0: entries base + s G, head h at + h
  // (a partials CTA that stopped early leaves a stale record: check it)
  if (seg.count < 1 || seg.base < 0 || seg.stride != G ||
      static_cast<long long>(seg.base) + static_cast<long long>(seg.count) * G > a.part_cap) {
    if (t == 0) atomicCAS(a.error, 0, kErrPartials);
    if (t < kDim) out[t] = 0.f;
    return;
  }
  // this quarter's segments s = qt, qt + kQ, ... as a running (m, l, acc)
  float m = -INFINITY, l = 0.f, acc = 0.f;
  for (int s0 = qt; s0 < seg.count; s0 += kQ * kBatch) {
    float pm[kBatch], pl[kBatch], pa[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int sg = s0 + kQ * k;
      const float* part = a.ws_part + (static_cast<long long>(seg.base) + static_cast<long long>(sg) * G + h) *
                                          kPartStride;
      const bool in = sg < seg.count;
      pm[k] = in ? __ldcg(part) : -INFINITY;
      pl[k] = in ? __ldcg(part + 1) : 0.f;
      pa[k] = in ? __ldcg(part + 4 + lane) : 0.f;
    }
    float mn = m;
#pragma unroll
    for (int k = 0; k < kBatch; ++k) mn = fmaxf(mn, pm[k]);
    if (mn == -INFINITY) continue;
    const float so = m == -INFINITY ? 0.f : __expf(m - mn);
    l *= so;
    acc *= so;
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const float sn = pm[k] == -INFINITY ? 0.f : __expf(pm[k] - mn);
      l = fmaf(pl[k], sn, l);
      acc = fmaf(pa[k], sn, acc);
    }
    m = mn;
  }
  // the quarters' sums, then o_rot = acc / l
  if (lane == 0) {
    ml_s[qt][0] = m;
    ml_s[qt][1] = l;
  }
  acc_s[qt][lane] = acc;
  __syncthreads();
  if (qt == 0) {
    float mn = -INFINITY;
#pragma unroll
    for (int q = 0; q < kQ; ++q) mn = fmaxf(mn, ml_s[q][0]);
    float lt = 0.f, at = 0.f;
#pragma unroll
    for (int q = 0; q < kQ; ++q) {
      const float mq = ml_s[q][0];
      const float sq = mq == -INFINITY ? 0.f : __expf(mq - mn);
      lt = fmaf(ml_s[q][1], sq, lt);
      at = fmaf(acc_s[q][lane], sq, at);
    }
    orot_s[lane] = lt > 0.f ? at / lt : 0.f;
  }
  __syncthreads();
  // out[o] = sum_i R[i][o] o_rot[i] (seo-farm page §2: out = R^T o_rot): quarter qt sums kRows of the terms
  float r = 0.f;
#pragma unroll
  for (int k = 0; k < kRows; k += 4) {
    const float4 o4 = *reinterpret_cast<const float4*>(orot_s + kRows * qt + k);
    r = fmaf(w[k], o4.x, fmaf(w[k + 1], o4.y, fmaf(w[k + 2], o4.z, fmaf(w[k + 3], o4.w, r))));
  }
  acc_s[qt][lane] = r;                            // (quarter 0 read acc_s before the last barrier)
  __syncthreads();
  if (qt == 0) out[lane] = (acc_s[0][lane] + acc_s[1][lane]) + (acc_s[2][lane] + acc_s[3][lane]);
}

template <int G>
cudaError_t launch_merge_g(const DecodeArgs& a, cudaStream_t stream) {
  const bool per_head = tc_merge_per_head(a);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(per_head ? a.batch * a.n_q : a.batch * a.n_kv);
  cfg.blockDim = dim3(per_head ? kHeadMergeThreads : kBuilders);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return per_head ? cudaLaunchKernelEx(&cfg, merge_heads_kernel<G>, a)
                  : cudaLaunchKernelEx(&cfg, merge_groups_kernel<G>, a);
}

cudaError_t launch_merge_groups_tc(const DecodeArgs& a, cudaStream_t stream) {
  if (a.batch <= 0) return cudaSuccess;
  switch (a.group) {
    case 1: return launch_merge_g<1>(a, stream);
    case 2: return launch_merge_g<2>(a, stream);
    case 4: return launch_merge_g<4>(a, stream);
    case 8: return launch_merge_g<8>(a, stream);
    default: return cudaErrorInvalidValue;
  }
}

// Segments of a (sequence, KV head) group at full context: the group's chunks
// over the run length a CTA takes when every sequence is max_context long,
// plus one for a run boundary inside the group.
long long tc_segments_estimate(const DecodeArgs& a) {
  const int chunk = tc_chunk(a);
  const long long chunks = (a.max_context + chunk - 1) / chunk;
  const long long items = static_cast<long long>(a.batch) * a.n_kv * chunks;
  const long long ctas = tc_grid(a);
  const long long per_cta = items / ctas > 0 ? items / ctas : 1;
  return (chunks + per_cta - 1) / per_cta + 1;
}

bool tc_merge_in_partials(const DecodeArgs& a) {
  // a CTA owes the merges of the groups that end in its run: with more groups
  // than CTAs (short, ragged contexts) some runs hold many, and the CTAs that
  // owe most set the launch's end; with many segments per group (long
  // contexts over a small batch) one CTA would merge them all at the end.  A
  // merge launch spreads either over the GPU.
  return static_cast<long long>(a.batch) * a.n_kv <= tc_grid(a) && tc_segments_estimate(a) <= 8;
}

bool tc_merge_per_head(const DecodeArgs& a) {
  // fewer groups than SMs: a CTA per query head keeps more SMs merging
  return static_cast<long long>(a.batch) * a.n_kv < (a.num_sms > 0 ? a.num_sms : 148);
}

cudaError_t launch_decode_partials_tc(const DecodeArgs& a, cudaStream_t stream, bool early) {
  if (a.batch <= 0) return cudaSuccess;
  switch (a.group) {
    case 1: return launch_g<1>(a, stream, early);
    case 2: return launch_g<2>(a, stream, early);
    case 4: return launch_g<4>(a, stream, early);
    case 8: return launch_g<8>(a, stream, early);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tq
