// Tensor-core quantize-append for bf16 head vectors (sm_103a: TMA + tcgen05).
//
// Same arithmetic as the SIMT path (甲子光年 article §2 第一階段 / 第二階段):
// n = ||x||, Y = R x, code_j = #{i : t_i < Y_j / n}, bit-plane packing; keys
// also get r' = Y - n c[code], gamma = ||r'|| and sign(S' r') (S' = S R^T).
//
// The two products are dense 128 x 128 contractions over a tile of 128
// vectors, so they run on the tensor cores with fp32 accumulation in tensor
// memory.  To keep codes bit-exact against an fp64 reference outside a 1e-5
// band around the decision boundaries, every fp32 constant W is split into
// bf16 W_hi + W_lo (x is bf16 already, exact): Y = X R_hi^T + X R_lo^T (two
// passes), and the fp32 residual is split too: Z = r_hi S'_hi^T + r_hi S'_lo^T
// + r_lo S'_hi^T (three passes).  The split leaves a relative error near 2^-17.
//
// A tile is 128 consecutive tokens of one KV head (a 3-D TMA box), so each
// epilogue warp holds 32 consecutive tokens of one head: value codes, which
// the cache stores token-transposed, are transposed 32 x 32 bits at a time
// with warp shuffles and stored as whole words when the 32 slots are
// contiguous and aligned (prefill), or set bit by bit with atomics otherwise.
//
// BITS = 0 is the PolarQuant epilogue (the intelliparadigm.com page, §2.1.1
// step 2) on the same rotation: each thread pairs its 32 coordinates through
// levels 1..5 in registers, the four threads of a vector meet in shared
// memory for levels 6 and 7, and the 64-byte records are packed from the
// codes staged there; the radius stored is the exact norm.
//
// One persistent CTA per SM, 18 warps:
//   warp 0      TMA producer: R/S' hi/lo once, then 128-token tiles of X;
//   warp 1      tcgen05.mma issuer (and owner of the tensor-memory columns);
//   warps 2..17 epilogue: warp w reads tensor-memory lanes 32 (w % 4) .. +31
//               (one vector per lane) and the 32 columns 32 g .. 32 g + 31,
//               g = (w - 2) / 4, so four threads share a vector and each
//               takes 32 of its coordinates: the norm and the residual norm
//               are summed over the four in shared memory; codes, bit-plane
//               words, residual hi/lo for the second product and QJL sign
//               words are per 32 coordinates.
// The accumulators are double-buffered in tensor memory, so the products of
// the next tile run while the epilogue works on the current one.
// Operands sit in shared memory in the 128-byte swizzled K-major layout that
// TMA writes and tcgen05 descriptors read (two 64-column K blocks per matrix).
// Every mbarrier wait is bounded in time; on a timeout the CTA records an
// error, drains what it has in flight, frees its tensor memory and returns.
#include <cuda.h>
#include <cuda_bf16.h>

#include <utility>

#include "kernels.h"
#include "polar_codes.cuh"
#include "tc_ptx.cuh"

namespace tq {
namespace {

constexpr int kTileRows = 128;
constexpr int kKBlock = 64;                       // bf16 columns per 128-byte swizzle row
constexpr int kHalfBytes = kTileRows * 128;       // one K block of a 128-row operand: 16 KB
constexpr int kMatBytes = 2 * kHalfBytes;         // one 128 x 128 bf16 operand: 32 KB
constexpr int kEpiWarps = 16;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kThreads = 64 + kEpiThreads;
constexpr int kCvtWarps = 4;                      // fp32 inputs: warps that split X into bf16 hi/lo
constexpr int kThreadsF32 = kThreads + 32 * kCvtWarps;
constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(128, 128);

// Shared memory: the bf16 hi/lo images of R (and S'), X stages and, with the
// QJL bit, the partial residual norms of two tiles.  Tensor memory: Y buffers
// of 128 columns (with the QJL bit each turns into the residual, hi and lo
// bf16, once its Y is read, and serves as the A operand of the second
// product) and, with the QJL bit, one Z buffer.
// fp32 inputs (F32) hold each X stage as two bf16 operands, X_hi and X_lo
// (X_hi = bf16(X), X_lo = bf16(X - X_hi)), and the exact fp32 squared norms
// of the stage's 128 rows.
template <bool QJL, bool F32 = false>
struct Layout {
  static constexpr int kW = QJL ? 4 : 2;          // R_hi, R_lo (, S'_hi, S'_lo)
  static constexpr int kStageBytes = F32 ? 2 * kMatBytes : kMatBytes;
  static constexpr int kStages = F32 ? (QJL ? 1 : 2) : (QJL ? 2 : 3);   // X tiles in flight
  static constexpr int kW0 = 0;
  static constexpr int kX0 = kW * kMatBytes;
  static constexpr int kRs0 = kX0 + kStages * kStageBytes;   // [2][4][128] floats
  static constexpr int kNrm0 = kRs0 + (QJL ? 2 * 4 * kTileRows * 4 : 0);   // F32: [kStages][128] floats
  static constexpr int kBytes = kNrm0 + (F32 ? kStages * kTileRows * 4 : 0);
  // PolarQuant epilogue (BITS = 0): one tile's codes, [128 rows][64 level-1 |
  // 63 upper + 1] bytes, then the level-5 radii [128 rows][4] floats
  static constexpr int kPolar0 = kBytes;
  static constexpr int kPolarBytes = kBytes + kTileRows * 128 + kTileRows * 4 * 4;
  static_assert(kPolarBytes > kPolar0, "the PolarQuant region follows the rest");
  static constexpr int kYBufs = QJL ? 3 : 2;
  static constexpr uint32_t kZCol = 3 * 128;
  static constexpr uint32_t kTmemCols = QJL ? 512 : 256;
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Lane i holds row i of a 32 x 32 bit matrix (bit j = column j); afterwards
// lane j holds column j (bit i = row i).  Five butterfly stages; in stage k
// (distance sh = 16 >> k) a lane keeps the bits of its half of every 2 sh
// block and takes the other half from its partner lane, rotated into place
// (left by sh for the lower lane of a pair, right by sh for the upper: the
// bits a rotation wraps around fall in the half the lane keeps), so a stage
// is a shuffle, a funnel shift and one select-by-mask.  The per-lane masks
// and rotations are set once.
struct LaneTranspose {
  uint32_t keep[5];
  uint32_t rot[5];
  __device__ __forceinline__ explicit LaneTranspose(int lane) {
    const uint32_t masks[5] = {0x0000FFFFu, 0x00FF00FFu, 0x0F0F0F0Fu, 0x33333333u, 0x55555555u};
#pragma unroll
    for (int k = 0; k < 5; ++k) {
      const int sh = 16 >> k;
      const bool upper = (lane & sh) != 0;
      keep[k] = upper ? ~masks[k] : masks[k];
      rot[k] = upper ? 32 - sh : sh;
    }
  }
  __device__ __forceinline__ uint32_t operator()(uint32_t x) const {
#pragma unroll
    for (int k = 0; k < 5; ++k) {
      const uint32_t o = __shfl_xor_sync(0xffffffffu, x, 16 >> k);
      const uint32_t z = __funnelshift_l(o, o, rot[k]);
      x = (x & keep[k]) | (z & ~keep[k]);
    }
    return x;
  }
};

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Barrier of the epilogue warps only (named barrier 1) that also ORs a flag
// over them, so that every epilogue thread takes the same exit decision.
__device__ __forceinline__ bool epi_sync_any(bool flag) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(flag)), "n"(kEpiThreads)
      : "memory");
  return r != 0;
}

// The bits of code = #{i : t_i < y} for non-decreasing boundaries t (the
// Lloyd-Max midpoints are), found by binary search from the top bit: with the
// bits above p forming the prefix k, code >= c holds exactly when y > t[c - 1],
// so bit p is y > t[k 2^(p+1) + 2^p - 1]. The candidates of each level are
// narrowed by the bits already found, lowest first, with selects only.
template <int BITS>
__device__ __forceinline__ void code_bits(float y, const float (&t)[(1 << BITS) - 1], bool (&b)[BITS]) {
#pragma unroll
  for (int p = BITS - 1; p >= 0; --p) {
    float cand[1 << (BITS - 1)];
#pragma unroll
    for (int k = 0; k < (1 << (BITS - 1 - p)); ++k) cand[k] = t[(2 * k + 1) * (1 << p) - 1];
#pragma unroll
    for (int q = p + 1; q < BITS; ++q)
#pragma unroll
      for (int k = 0; k < (1 << (BITS - 1 - q)); ++k) cand[k] = b[q] ? cand[2 * k + 1] : cand[2 * k];
    b[p] = y > cand[0];
  }
}

// levels[code] for the code whose bits are b, by selects (lowest bit first).
template <int BITS>
__device__ __forceinline__ float level_of(const float (&levels)[1 << BITS], const bool (&b)[BITS]) {
  float cand[1 << BITS];
#pragma unroll
  for (int k = 0; k < (1 << BITS); ++k) cand[k] = levels[k];
#pragma unroll
  for (int q = 0; q < BITS; ++q)
#pragma unroll
    for (int k = 0; k < (1 << (BITS - 1 - q)); ++k) cand[k] = b[q] ? cand[2 * k + 1] : cand[2 * k];
  return cand[0];
}

// The same search for 2-, 3- and 4-bit codes in one block of predicated PTX:
// each compare feeds the next level's boundary select and a predicated OR of
// bit j into its plane word (one logic instruction per plane bit where a
// select and an OR would be two).  With LEV it also returns levels[code]
// (2 and 3 bits).
template <int BITS, bool LEV, int J>
__device__ __forceinline__ float decide(float y, const float (&t)[(1 << BITS) - 1], const float (&l)[1 << BITS],
                                        uint32_t (&pl)[BITS]) {
  static_assert(BITS >= 2 && BITS <= 4 && !(BITS == 4 && LEV), "2- to 4-bit codes, levels up to 3 bits");
  float lev = 0.f;
  if constexpr (BITS == 4) {
    // boundaries by (q3 q2 q1): level 2 from t3 / t11, level 1 from t1 t5 t9
    // t13, level 0 from the even ones
    asm("{\n\t.reg .pred q3, q2, q1, q0;\n\t.reg .f32 ta, tb, tc, td, e0, e1, e2, e3, f0, f1, g;\n\t"
        "setp.gt.f32 q3, %4, %5;\n\t@q3 or.b32 %0, %0, %20;\n\t"
        "selp.f32 ta, %7, %6, q3;\n\t"
        "setp.gt.f32 q2, %4, ta;\n\t@q2 or.b32 %1, %1, %20;\n\t"
        "selp.f32 tb, %9, %8, q2;\n\tselp.f32 tc, %11, %10, q2;\n\tselp.f32 td, tc, tb, q3;\n\t"
        "setp.gt.f32 q1, %4, td;\n\t@q1 or.b32 %2, %2, %20;\n\t"
        "selp.f32 e0, %13, %12, q1;\n\tselp.f32 e1, %15, %14, q1;\n\t"
        "selp.f32 e2, %17, %16, q1;\n\tselp.f32 e3, %19, %18, q1;\n\t"
        "selp.f32 f0, e1, e0, q2;\n\tselp.f32 f1, e3, e2, q2;\n\tselp.f32 g, f1, f0, q3;\n\t"
        "setp.gt.f32 q0, %4, g;\n\t@q0 or.b32 %3, %3, %20;\n\t}"
        : "+r"(pl[3]), "+r"(pl[2]), "+r"(pl[1]), "+r"(pl[0])
        : "f"(y), "f"(t[7]), "f"(t[3]), "f"(t[11]), "f"(t[1]), "f"(t[5]), "f"(t[9]), "f"(t[13]), "f"(t[0]),
          "f"(t[2]), "f"(t[4]), "f"(t[6]), "f"(t[8]), "f"(t[10]), "f"(t[12]), "f"(t[14]), "n"(1u << J));
  } else if constexpr (BITS == 3 && !LEV) {
    asm("{\n\t.reg .pred q2, q1, q0;\n\t.reg .f32 ta, tb, tc, td;\n\t"
        "setp.gt.f32 q2, %3, %4;\n\t@q2 or.b32 %0, %0, %11;\n\t"
        "selp.f32 ta, %6, %5, q2;\n\t"
        "setp.gt.f32 q1, %3, ta;\n\t@q1 or.b32 %1, %1, %11;\n\t"
        "selp.f32 tb, %10, %9, q1;\n\tselp.f32 tc, %8, %7, q1;\n\tselp.f32 td, tb, tc, q2;\n\t"
        "setp.gt.f32 q0, %3, td;\n\t@q0 or.b32 %2, %2, %11;\n\t}"
        : "+r"(pl[2]), "+r"(pl[1]), "+r"(pl[0])
        : "f"(y), "f"(t[3]), "f"(t[1]), "f"(t[5]), "f"(t[0]), "f"(t[2]), "f"(t[4]), "f"(t[6]), "n"(1u << J));
  } else if constexpr (BITS == 3) {
    // with the level: levels[code] selected by q0, then q1, then q2
    asm("{\n\t.reg .pred q2, q1, q0;\n\t.reg .f32 ta, tb, tc, td, la, lb, lc, ld, lf, lg;\n\t"
        "setp.gt.f32 q2, %4, %5;\n\t@q2 or.b32 %0, %0, %20;\n\t"
        "selp.f32 ta, %7, %6, q2;\n\t"
        "setp.gt.f32 q1, %4, ta;\n\t@q1 or.b32 %1, %1, %20;\n\t"
        "selp.f32 tb, %11, %10, q1;\n\tselp.f32 tc, %9, %8, q1;\n\tselp.f32 td, tb, tc, q2;\n\t"
        "setp.gt.f32 q0, %4, td;\n\t@q0 or.b32 %2, %2, %20;\n\t"
        "selp.f32 la, %13, %12, q0;\n\tselp.f32 lb, %15, %14, q0;\n\t"
        "selp.f32 lc, %17, %16, q0;\n\tselp.f32 ld, %19, %18, q0;\n\t"
        "selp.f32 lf, lb, la, q1;\n\tselp.f32 lg, ld, lc, q1;\n\tselp.f32 %3, lg, lf, q2;\n\t}"
        : "+r"(pl[2]), "+r"(pl[1]), "+r"(pl[0]), "=f"(lev)
        : "f"(y), "f"(t[3]), "f"(t[1]), "f"(t[5]), "f"(t[0]), "f"(t[2]), "f"(t[4]), "f"(t[6]), "f"(l[0]),
          "f"(l[1]), "f"(l[2]), "f"(l[3]), "f"(l[4]), "f"(l[5]), "f"(l[6]), "f"(l[7]), "n"(1u << J));
  } else if constexpr (LEV) {
    asm("{\n\t.reg .pred q1, q0;\n\t.reg .f32 ta, la, lb;\n\t"
        "setp.gt.f32 q1, %3, %4;\n\t@q1 or.b32 %0, %0, %11;\n\t"
        "selp.f32 ta, %6, %5, q1;\n\t"
        "setp.gt.f32 q0, %3, ta;\n\t@q0 or.b32 %1, %1, %11;\n\t"
        "selp.f32 la, %10, %9, q0;\n\tselp.f32 lb, %8, %7, q0;\n\tselp.f32 %2, la, lb, q1;\n\t}"
        : "+r"(pl[1]), "+r"(pl[0]), "=f"(lev)
        : "f"(y), "f"(t[1]), "f"(t[0]), "f"(t[2]), "f"(l[0]), "f"(l[1]), "f"(l[2]), "f"(l[3]), "n"(1u << J));
  } else {
    asm("{\n\t.reg .pred q1, q0;\n\t.reg .f32 ta;\n\t"
        "setp.gt.f32 q1, %2, %3;\n\t@q1 or.b32 %0, %0, %6;\n\t"
        "selp.f32 ta, %5, %4, q1;\n\t"
        "setp.gt.f32 q0, %2, ta;\n\t@q0 or.b32 %1, %1, %6;\n\t}"
        : "+r"(pl[1]), "+r"(pl[0])
        : "f"(y), "f"(t[1]), "f"(t[0]), "f"(t[2]), "n"(1u << J));
  }
  return lev;
}

// f(integral_constant<int, J>) for J = 0 .. N-1 (compile-time bit positions).
template <typename F, int... Js>
__device__ __forceinline__ void for_each_index(F&& f, std::integer_sequence<int, Js...>) {
  (f(std::integral_constant<int, Js>{}), ...);
}

// Byte offset, within an X tile, of the first 16-byte chunk that the thread of
// coordinate group g reads from row `row` (K block g / 2, chunk (g % 2) * 4,
// 128-byte swizzle).
__device__ __forceinline__ int x_partial_offset(int g, int row) {
  return (g >> 1) * kHalfBytes + row * 128 + ((((g & 1) * 4) ^ (row & 7)) << 4);
}

template <int BITS, bool QJL, bool TRANS, bool F32>
__global__ void __launch_bounds__(F32 ? kThreadsF32 : kThreads, 1)
    quantize_tc_kernel(const __grid_constant__ CUtensorMap x_map, const __grid_constant__ CUtensorMap w_map,
                       QuantizeArgs a) {
  using L = Layout<QJL, F32>;
  constexpr bool POLAR = BITS == 0;
  constexpr int kLevels = 1 << BITS;
  constexpr int kBounds = POLAR ? 1 : kLevels - 1;   // (array sizes: no codebook with PolarQuant)
  constexpr int kPlanes = POLAR ? 1 : BITS;
  extern __shared__ uint8_t smem_raw[];
  // y_full[b]: the first products of Y buffer b are in tensor memory;
  // y_empty[b]: the epilogue is done with buffer b (Y read, and with the QJL
  // bit its residual consumed by the second products); res_full[b]: the
  // residual of buffer b is stored; z_full / z_empty: the second products are
  // in the Z buffer / were read.
  __shared__ __align__(8) uint64_t w_full, x_full[L::kStages], x_empty[L::kStages], y_full[3], y_empty[3],
      res_full[3], z_full, z_empty, drain;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;

  // 1024-byte aligned, as an offset from smem_raw so that accesses stay shared-space
  uint8_t* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int n_tt = (a.n_tokens + kTileRows - 1) / kTileRows;   // token tiles per head
  const int n_tiles = n_tt * a.n_kv;
  volatile int* abort = &abort_s;

  if (tid == 0) {
    abort_s = 0;
    ptx::mbar_init(&w_full, 1);
    for (int s = 0; s < L::kStages; ++s) {
      ptx::mbar_init(&x_full[s], F32 ? 32 * kCvtWarps : 1);   // the TMA copy, or every converter thread
      ptx::mbar_init(&x_empty[s], kEpiThreads);
    }
    for (int b = 0; b < 3; ++b) {
      ptx::mbar_init(&y_full[b], 1);
      ptx::mbar_init(&y_empty[b], kEpiThreads);
      ptx::mbar_init(&res_full[b], kEpiThreads);
    }
    ptx::mbar_init(&z_full, 1);
    ptx::mbar_init(&z_empty, kEpiThreads);
    ptx::mbar_init(&drain, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 1) {
    ptx::tmem_alloc(&tmem_base_s, L::kTmemCols);
    ptx::tmem_relinquish();
  }
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = tmem_base_s;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      ptx::prefetch_tensor_map(&x_map);
      ptx::prefetch_tensor_map(&w_map);
      ptx::mbar_arrive_expect_tx(&w_full, L::kW * kMatBytes);
      for (int m = 0; m < L::kW; ++m)
        for (int kb = 0; kb < 2; ++kb)
          ptx::tma_load_2d(smem + L::kW0 + m * kMatBytes + kb * kHalfBytes, &w_map, &w_full, kb * kKBlock,
                           m * kTileRows);
      int it = 0, last_stage = -1;
      uint32_t last_phase = 0;
      for (int tile = blockIdx.x; !F32 && tile < n_tiles; tile += gridDim.x, ++it) {
        const int s = it % L::kStages;
        const uint32_t ph = (it / L::kStages) & 1;
        if (!ptx::wait_bar(&x_empty[s], ph ^ 1, abort, a.error, kErrTimeout)) break;
        ptx::mbar_arrive_expect_tx(&x_full[s], kMatBytes);
        for (int kb = 0; kb < 2; ++kb)
          ptx::tma_load_3d(smem + L::kX0 + s * kMatBytes + kb * kHalfBytes, &x_map, &x_full[s], kb * kKBlock,
                           tile / n_tt, (tile % n_tt) * kTileRows);
        last_stage = s;
        last_phase = ph;
      }
      if (*abort) {
        ptx::drain_bar(&w_full, 0);
        if (last_stage >= 0) ptx::drain_bar(&x_full[last_stage], last_phase);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    // Y of tile i goes to buffer i % kYBufs; with the QJL bit the second
    // products of tile i - 1 follow those of tile i, so that they run while
    // the epilogue works on the first half of tile i.
    if (lane == 0) {
      bool ok = ptx::wait_bar(&w_full, 0, abort, a.error, kErrTimeout);
      const uint32_t w_base = ptx::smem_u32(smem + L::kW0);
      // second products of tile j: Z = r_hi S'_hi + r_hi S'_lo + r_lo S'_hi,
      // the residual read from tensor memory (thread group g stored
      // coordinates 32 g .. 32 g + 31 as 16 hi columns, then 16 lo columns)
      auto issue_z = [&](int j) -> bool {
        const int b = j % 3;
        if (!ptx::wait_bar(&res_full[b], (j / 3) & 1, abort, a.error, kErrTimeout)) return false;
        if (j > 0 && !ptx::wait_bar(&z_empty, (j - 1) & 1, abort, a.error, kErrTimeout)) return false;
        ptx::tc_fence_after();
        const uint32_t r_base = tmem + b * 128;
        uint32_t acc = 0;
#pragma unroll
        for (int pass = 0; pass < 3; ++pass) {
          const uint32_t lo = pass == 2 ? 16 : 0;
          const int b_sel = pass == 1 ? 3 : 2;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {          // 16 coordinates per step
            const uint32_t a_col = r_base + 32 * (ks >> 1) + 8 * (ks & 1) + lo;
            const uint32_t off = (ks >> 2) * kHalfBytes + (ks & 3) * 32;
            ptx::mma_bf16_tmem_a(tmem + L::kZCol, a_col, ptx::desc_k_sw128(w_base + b_sel * kMatBytes + off), kIdesc,
                                 acc);
            acc = 1;
          }
        }
        ptx::mma_commit(&z_full);
        return true;
      };
      int it = 0;
      for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x, ++it) {
        const int s = it % L::kStages;
        const uint32_t ph = (it / L::kStages) & 1;
        const int b = it % L::kYBufs;
        const uint32_t yb = tmem + b * 128;
        ok = ptx::wait_bar(&x_full[s], ph, abort, a.error, kErrTimeout);
        // the buffer's previous tile (it - kYBufs) is done with
        ok = ok && ptx::wait_bar(&y_empty[b], ((it / L::kYBufs) & 1) ^ 1, abort, a.error, kErrTimeout);
        if (!ok) break;
        ptx::tc_fence_after();
        const uint32_t x_base = ptx::smem_u32(smem + L::kX0 + s * L::kStageBytes);
        uint32_t acc = 0;
        // X R_hi, X R_lo (bf16 X exact); fp32 X: X_hi R_hi, X_hi R_lo, X_lo R_hi
#pragma unroll
        for (int pass = 0; pass < (F32 ? 3 : 2); ++pass) {
          const uint32_t a_off = pass == 2 ? kMatBytes : 0;
          const int b_sel = pass == 1 ? 1 : 0;
#pragma unroll
          for (int kb = 0; kb < 2; ++kb) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              const uint32_t off = kb * kHalfBytes + ks * 32;
              ptx::mma_bf16(yb, ptx::desc_k_sw128(x_base + a_off + off),
                            ptx::desc_k_sw128(w_base + b_sel * kMatBytes + off), kIdesc, acc);
              acc = 1;
            }
          }
        }
        ptx::mma_commit(&y_full[b]);
        if (QJL && it > 0) ok = issue_z(it - 1);
      }
      if (QJL && ok && it > 0) ok = issue_z(it - 1);
      if (*abort) {
        ptx::mma_commit(&drain);
        ptx::drain_bar(&drain, 0);
      }
    }
  } else if (F32 && warp >= 2 + kEpiWarps) {
    // ---------------- converters (fp32 X): bf16 hi/lo operands and exact norms ----------------
    // warp cw takes rows 32 cw .. 32 cw + 31 of a tile, one row at a time: lane
    // l reads coordinates 4 l .. 4 l + 3 (the row's 512 bytes in one coalesced
    // load) and stores them as bf16 hi and lo into the 128-byte swizzled
    // K-major stage the MMA reads (K block l / 16, 16-byte chunk (l % 16) / 2)
    const int cw = warp - (2 + kEpiWarps);
    float* const nrm_s = reinterpret_cast<float*>(smem + L::kNrm0);
    const float* x = static_cast<const float*>(a.x);
    const int kb = lane >> 4, chunk = (lane & 15) >> 1;
    int it = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
      const int s = it % L::kStages;
      const uint32_t ph = (it / L::kStages) & 1;
      if (!__all_sync(0xffffffffu, ptx::wait_bar(&x_empty[s], ph ^ 1, abort, a.error, kErrTimeout))) break;
      uint8_t* const st = smem + L::kX0 + s * L::kStageBytes;
      const int head = tile / n_tt, tok0 = (tile % n_tt) * kTileRows;
#pragma unroll 4
      for (int r = 0; r < 32; ++r) {
        const int row = 32 * cw + r, token = tok0 + row;
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (token < a.n_tokens)
          v = *reinterpret_cast<const float4*>(x + (static_cast<long long>(token) * a.n_kv + head) * kDim + 4 * lane);
        const __nv_bfloat162 h01 = __floats2bfloat162_rn(v.x, v.y), h23 = __floats2bfloat162_rn(v.z, v.w);
        const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
        const __nv_bfloat162 l01 = __floats2bfloat162_rn(v.x - f01.x, v.y - f01.y);
        const __nv_bfloat162 l23 = __floats2bfloat162_rn(v.z - f23.x, v.w - f23.y);
        const int off = kb * kHalfBytes + row * 128 + ((chunk ^ (row & 7)) << 4) + (lane & 1) * 8;
        *reinterpret_cast<uint2*>(st + off) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&h01), *reinterpret_cast<const uint32_t*>(&h23));
        *reinterpret_cast<uint2*>(st + kMatBytes + off) =
            make_uint2(*reinterpret_cast<const uint32_t*>(&l01), *reinterpret_cast<const uint32_t*>(&l23));
        float ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, v.w * v.w)));
#pragma unroll
        for (int off2 = 16; off2 > 0; off2 >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off2);
        if (lane == 0) nrm_s[s * kTileRows + row] = ss;
      }
      ptx::fence_async_shared();                  // the generic stores, before the MMA reads the stage
      ptx::mbar_arrive(&x_full[s]);
    }
  } else {
    // ---------------- epilogue: four threads per vector, 32 coordinates each ----------------
    const int quarter = warp & 3;                 // tensor-memory lanes this warp may access
    const int g = (warp - 2) >> 2;                // its coordinate group: 32 g .. 32 g + 31
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const LaneTranspose transpose(lane);          // (used by the token-transposed value codes)
    float bnd[kBounds];
#pragma unroll
    for (int i = 0; i < kLevels - 1; ++i) bnd[i] = a.bounds[i];
    float lev[kLevels];                           // read only by the QJL residual
#pragma unroll
    for (int i = 0; i < kLevels; ++i) lev[i] = QJL ? a.levels[i] : 0.f;
    const long long cache_rows = static_cast<long long>(a.num_blocks) * a.block_size;
    const bool bs_pow2 = (a.block_size & (a.block_size - 1)) == 0;
    const int bs_shift = __ffs(a.block_size) - 1;
    float* const rs_s = reinterpret_cast<float*>(smem + L::kRs0);   // [tile parity][g][row]

    // the QJL signs and the residual norm of tile j (second half of its epilogue)
    auto finish_qjl = [&](int j, long long dstp) {
      const bool zok = __all_sync(0xffffffffu, ptx::wait_bar(&z_full, j & 1, abort, a.error, kErrTimeout));
      if (!zok) return;                           // the next barrier ends every epilogue warp
      ptx::tc_fence_after();
      uint32_t zr[32];
      ptx::tmem_ld32(lane_addr + L::kZCol + 32 * g, zr);
      ptx::tc_fence_before();
      ptx::mbar_arrive(&z_empty);
      ptx::mbar_arrive(&y_empty[j % 3]);          // its residual has been consumed too
      uint32_t word = 0;
      for_each_index(
          [&](auto kc) {
            constexpr int k = decltype(kc)::value;
            // bit k = (z_k > 0), as a predicated OR
            asm("{\n\t.reg .pred q;\n\tsetp.gt.f32 q, %1, 0f00000000;\n\t@q or.b32 %0, %0, %2;\n\t}"
                : "+r"(word)
                : "f"(__uint_as_float(zr[k])), "n"(1u << k));
          },
          std::make_integer_sequence<int, 32>{});
      if (dstp >= 0) {
        reinterpret_cast<uint32_t*>(a.qjl + dstp * 16)[g] = word;
        const float* r4 = rs_s + (j & 1) * 4 * kTileRows + row;
        if (g == 0)
          store_norm(a.rnorm, dstp, sqrtf((r4[0] + r4[kTileRows]) + (r4[2 * kTileRows] + r4[3 * kTileRows])),
                     a.norm16);
      }
    };

    int it = 0;
    bool alive = true;
    long long dst_prev = -1;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
      const int s = it % L::kStages;
      const uint32_t ph = (it / L::kStages) & 1;
      const int b = it % L::kYBufs;
      const uint32_t yb = lane_addr + b * 128;

      // destination row first: its global loads overlap the waits below
      const int head = tile / n_tt;
      const int token = (tile % n_tt) * kTileRows + row;
      long long dst = -1;
      long long slot = -1;
      long long blk = 0;
      if (token < a.n_tokens) {
        slot = slot_of(a, token);
        if (slot >= 0 && slot < cache_rows) {
          blk = bs_pow2 ? (slot >> bs_shift) : slot / a.block_size;
          dst = (blk * a.n_kv + head) * a.block_size + (slot - blk * a.block_size);
        } else if (slot >= cache_rows) {
          if (g == 0) atomicCAS(a.error, 0, kErrSlot);
          slot = -1;
        }
      }

      bool ok = ptx::wait_bar(&x_full[s], ph, abort, a.error, kErrTimeout);
      // the partial norm from this group's 32 bf16 coordinates of the X row
      // (K block g / 2, 16-byte chunks (g % 2) * 4 .. + 3, chunk c of a row at c ^ (row % 8))
      uint8_t* const x_tile = smem + L::kX0 + s * L::kStageBytes;
      const uint8_t* xrow = x_tile + (g >> 1) * kHalfBytes + row * 128;
      float ss = 0.f;
      if (ok && !F32) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int c = (g & 1) * 4 + q;
          const uint4 v = *reinterpret_cast<const uint4*>(xrow + ((c ^ (row & 7)) << 4));
          const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float lo = bf16_lo(w[e]), hi = bf16_hi(w[e]);
            ss = fmaf(lo, lo, ss);
            ss = fmaf(hi, hi, ss);
          }
        }
      }
      ok = ok && ptx::wait_bar(&y_full[b], (it / L::kYBufs) & 1, abort, a.error, kErrTimeout);
      // Once the products have read X, the first 4 bytes this thread read carry
      // its partial sum to the other three threads of the row (no other thread
      // reads those bytes, and the stage is refilled only after all have read).
      if (ok && !F32) *reinterpret_cast<float*>(x_tile + x_partial_offset(g, row)) = ss;
      // a failed wait anywhere ends every epilogue warp (the tcgen05.ld below
      // needs whole warps, the barriers below all 16); this barrier also
      // publishes the previous tile's partial residual norms
      if (epi_sync_any(!ok || *abort)) {
        alive = false;
        break;
      }
      // (fp32 X: the exact norm the converters left with the stage)
      const float n =
          F32 ? sqrtf(reinterpret_cast<const float*>(smem + L::kNrm0)[s * kTileRows + row])
              : sqrtf((*reinterpret_cast<const float*>(x_tile + x_partial_offset(0, row)) +
                       *reinterpret_cast<const float*>(x_tile + x_partial_offset(1, row))) +
                      (*reinterpret_cast<const float*>(x_tile + x_partial_offset(2, row)) +
                       *reinterpret_cast<const float*>(x_tile + x_partial_offset(3, row))));
      ptx::fence_async_shared();                  // the generic write above, before TMA refills the stage
      ptx::mbar_arrive(&x_empty[s]);
      // y = Y / n against t is taken as Y against n t (a zero vector compares
      // y = 0 against t): one product per boundary instead of one per coordinate
      const float n_eff = n > 0.f ? n : 1.f;
      const float ns = stored_norm(n, a.norm16);  // the residual is against the norm as stored
      float tn[kBounds];
#pragma unroll
      for (int i = 0; i < kLevels - 1; ++i) tn[i] = bnd[i] * n_eff;

      ptx::tc_fence_after();
      if constexpr (POLAR) {
        uint32_t yr[32];
        ptx::tmem_ld32(yb + 32 * g, yr);
        ptx::tc_fence_before();
        ptx::mbar_arrive(&y_empty[b]);            // this buffer may take the tile after next
        uint8_t* const pc = smem + L::kPolar0 + row * 128;   // [0, 64) level 1, [64, 127) levels 2..7
        float* const r5 = reinterpret_cast<float*>(smem + L::kPolar0 + kTileRows * 128) + row * 4;
        // levels 1..5 over coordinates 32 g .. 32 g + 31: at level L this
        // thread's pairs are g 2^(5-L) + i; radii overwrite the front of v
        float v[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(yr[j]);
#pragma unroll
        for (int lvl = 1; lvl <= 5; ++lvl) {
#pragma unroll
          for (int i = 0; i < (32 >> lvl); ++i) {
            const float first = v[2 * i], second = v[2 * i + 1];
            const int p = (g << (5 - lvl)) + i;
            const int code = polar_angle_code(second, first, lvl == 1);
            if (lvl == 1) pc[p] = static_cast<uint8_t>(code);
            else pc[64 + polar_upper_offset(lvl) + p] = static_cast<uint8_t>(code);
            v[i] = sqrtf(fmaf(first, first, second * second));
          }
        }
        r5[g] = v[0];
        epi_sync_any(false);                      // every thread's codes and level-5 radius are staged
        if (g == 0) {
          pc[64 + 60] = static_cast<uint8_t>(polar_angle_code(r5[1], r5[0], false));
          pc[64 + 61] = static_cast<uint8_t>(polar_angle_code(r5[3], r5[2], false));
          const float r60 = sqrtf(fmaf(r5[0], r5[0], r5[1] * r5[1]));
          const float r61 = sqrtf(fmaf(r5[2], r5[2], r5[3] * r5[3]));
          pc[64 + 62] = static_cast<uint8_t>(polar_angle_code(r61, r60, false));
        }
        epi_sync_any(false);
        if (dst >= 0) {
          uint4 wv;
          wv.x = polar_record_word(pc, pc + 64, 4 * g);
          wv.y = polar_record_word(pc, pc + 64, 4 * g + 1);
          wv.z = polar_record_word(pc, pc + 64, 4 * g + 2);
          wv.w = polar_record_word(pc, pc + 64, 4 * g + 3);
          reinterpret_cast<uint4*>(a.codes + dst * (4 * kPolarRecordWords))[g] = wv;
          if (g == 0) reinterpret_cast<float*>(a.norm)[dst] = n;
        }
        continue;                                 // (the next tile's first barrier frees the staged codes)
      }
      uint32_t planes[kPlanes];
      float rs = 0.f;
      {
        uint32_t yr[32];
        ptx::tmem_ld32(yb + 32 * g, yr);
#pragma unroll
        for (int p = 0; p < BITS; ++p) planes[p] = 0;
        float r[32];
        if constexpr (POLAR) {
          // (handled above)
        } else if constexpr (BITS == 2 || BITS == 3 || (BITS == 4 && !QJL)) {
          for_each_index(
              [&](auto jc) {
                constexpr int j = decltype(jc)::value;
                const float yv = __uint_as_float(yr[j]);
                const float lv = decide<BITS, QJL, j>(yv, tn, lev, planes);
                if (QJL) {
                  r[j] = fmaf(-ns, lv, yv);
                  rs = fmaf(r[j], r[j], rs);
                }
              },
              std::make_integer_sequence<int, 32>{});
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const float yv = __uint_as_float(yr[j]);
            bool bits[BITS];
            code_bits<BITS>(yv, tn, bits);
#pragma unroll
            for (int p = 0; p < BITS; ++p) planes[p] |= bits[p] ? (1u << j) : 0u;
            if (QJL) {
              r[j] = fmaf(-ns, level_of<BITS>(lev, bits), yv);
              rs = fmaf(r[j], r[j], rs);
            }
          }
        }
        if (QJL) {
          // the residual over this thread's (already read) Y columns: hi
          // bf16 pairs in the first 16, lo pairs in the last 16
          uint32_t rw[32];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const float r0 = r[2 * e], r1 = r[2 * e + 1];
            rw[e] = pack_bf16x2(r0, r1);
            rw[16 + e] = pack_bf16x2(r0 - bf16_lo(rw[e]), r1 - bf16_hi(rw[e]));
          }
          ptx::tmem_st32(yb + 32 * g, rw);
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          ptx::mbar_arrive(&res_full[b]);
        } else {
          ptx::tc_fence_before();
          ptx::mbar_arrive(&y_empty[b]);          // this buffer may take the tile after next
        }
      }
      if (TRANS) {
        // token-transposed codes: whole words when the warp's 32 slots are
        // contiguous and start a 32-token group, single bits otherwise
        const long long slot0 = __shfl_sync(0xffffffffu, slot, 0);
        const bool aligned = __all_sync(0xffffffffu, dst >= 0 && slot == slot0 + lane && (slot0 & 31) == 0);
        unsigned* words = reinterpret_cast<unsigned*>(a.codes);
        if (aligned) {
          const long long blk0 = __shfl_sync(0xffffffffu, blk, 0);
          const int off0 = static_cast<int>(slot0 - blk0 * a.block_size);
#pragma unroll
          for (int p = 0; p < BITS; ++p)
            words[transposed_word(blk0, head, a.n_kv, BITS, p, 32 * g + lane, a.block_size, off0)] =
                transpose(planes[p]);
        } else if (dst >= 0) {
          const int off = static_cast<int>(slot - blk * a.block_size);
          const unsigned mask = 1u << (off & 31);
          for (int p = 0; p < BITS; ++p)
            for (int j = 0; j < 32; ++j) {
              unsigned* w = words + transposed_word(blk, head, a.n_kv, BITS, p, 32 * g + j, a.block_size, off);
              if ((planes[p] >> j) & 1) atomicOr(w, mask); else atomicAnd(w, ~mask);
            }
        }
      } else if (dst >= 0) {
        uint32_t* out = reinterpret_cast<uint32_t*>(a.codes + dst * (BITS * 16));
#pragma unroll
        for (int p = 0; p < BITS; ++p) out[p * 4 + g] = planes[p];
      }
      if (dst >= 0 && g == 0) store_norm(a.norm, dst, n, a.norm16);
      if (QJL) {
        // rs_s[it & 1] is read after the next tile's first barrier and written
        // again two tiles later, after every thread has passed that barrier
        rs_s[(it & 1) * 4 * kTileRows + g * kTileRows + row] = rs;
        if (it > 0) finish_qjl(it - 1, dst_prev);
        dst_prev = dst;
      }
    }
    if (QJL && alive && it > 0 && !epi_sync_any(*abort)) finish_qjl(it - 1, dst_prev);
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, L::kTmemCols);
  }
}

template <int BITS, bool QJL, bool TRANS, bool F32>
cudaError_t launch_bits(const CUtensorMap& x_map, const CUtensorMap& w_map, const QuantizeArgs& a, int grid,
                        cudaStream_t stream) {
  const int smem = (BITS == 0 ? Layout<QJL, F32>::kPolarBytes : Layout<QJL, F32>::kBytes) + 1024;
  cudaError_t err = cudaFuncSetAttribute(quantize_tc_kernel<BITS, QJL, TRANS, F32>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  quantize_tc_kernel<BITS, QJL, TRANS, F32><<<grid, F32 ? kThreadsF32 : kThreads, smem, stream>>>(x_map, w_map, a);
  return cudaGetLastError();
}

template <int BITS, bool F32>
cudaError_t launch_kind(const CUtensorMap& x_map, const CUtensorMap& w_map, const QuantizeArgs& a, int grid,
                        cudaStream_t stream) {
  if (a.qjl != nullptr) return launch_bits<BITS, true, false, F32>(x_map, w_map, a, grid, stream);
  if (a.transposed) return launch_bits<BITS, false, true, F32>(x_map, w_map, a, grid, stream);
  return launch_bits<BITS, false, false, F32>(x_map, w_map, a, grid, stream);
}

template <int BITS>
cudaError_t launch_dtype(const CUtensorMap& x_map, const CUtensorMap& w_map, const QuantizeArgs& a, int grid,
                         bool f32, cudaStream_t stream) {
  return f32 ? launch_kind<BITS, true>(x_map, w_map, a, grid, stream)
             : launch_kind<BITS, false>(x_map, w_map, a, grid, stream);
}

}  // namespace

cudaError_t launch_quantize_tc(const QuantizeArgs& a, const CUtensorMap& x_map, const CUtensorMap& w_map,
                               int num_sms, bool f32, cudaStream_t stream) {
  if (a.n_vec <= 0) return cudaSuccess;
  if (a.qjl != nullptr && a.transposed) return cudaErrorInvalidValue;
  const int n_tiles = ((a.n_tokens + kTileRows - 1) / kTileRows) * a.n_kv;
  const int grid = n_tiles < num_sms ? n_tiles : num_sms;
  switch (a.bits) {
    case 0:   // PolarQuant records
      return f32 ? launch_bits<0, false, false, true>(x_map, w_map, a, grid, stream)
                 : launch_bits<0, false, false, false>(x_map, w_map, a, grid, stream);
    case 1: return launch_dtype<1>(x_map, w_map, a, grid, f32, stream);
    case 2: return launch_dtype<2>(x_map, w_map, a, grid, f32, stream);
    case 3: return launch_dtype<3>(x_map, w_map, a, grid, f32, stream);
    case 4: return launch_dtype<4>(x_map, w_map, a, grid, f32, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tq
