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

#include "kernels.h"
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
constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(128, 128);

template <bool QJL>
struct Layout {
  static constexpr int kW = QJL ? 4 : 2;          // R_hi, R_lo (, S'_hi, S'_lo)
  static constexpr int kStages = QJL ? 1 : 3;     // X tiles in flight
  static constexpr int kW0 = 0;
  static constexpr int kX0 = kW * kMatBytes;
  static constexpr int kRes0 = kX0 + kStages * kMatBytes;
  static constexpr int kBytes = kRes0 + (QJL ? 2 * kMatBytes : 0);
  static constexpr uint32_t kBufCols = QJL ? 256 : 128;     // Y (+ Z) of one tile
  static constexpr uint32_t kTmemCols = 2 * kBufCols;        // two tiles in flight
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Lane i holds row i of a 32 x 32 bit matrix (bit j = column j); afterwards
// lane j holds column j (bit i = row i).  Five butterfly stages.
__device__ __forceinline__ uint32_t transpose32(uint32_t x, int lane) {
  const uint32_t masks[5] = {0x0000FFFFu, 0x00FF00FFu, 0x0F0F0F0Fu, 0x33333333u, 0x55555555u};
#pragma unroll
  for (int k = 0; k < 5; ++k) {
    const int sh = 16 >> k;
    const uint32_t m = masks[k];
    const uint32_t o = __shfl_xor_sync(0xffffffffu, x, sh);
    x = (lane & sh) ? ((x & ~m) | ((o & ~m) >> sh)) : ((x & m) | ((o & m) << sh));
  }
  return x;
}

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

// Byte offset, within an X tile, of the first 16-byte chunk that the thread of
// coordinate group g reads from row `row` (K block g / 2, chunk (g % 2) * 4,
// 128-byte swizzle).
__device__ __forceinline__ int x_partial_offset(int g, int row) {
  return (g >> 1) * kHalfBytes + row * 128 + ((((g & 1) * 4) ^ (row & 7)) << 4);
}

template <int BITS, bool QJL, bool TRANS>
__global__ void __launch_bounds__(kThreads, 1)
    quantize_tc_kernel(const __grid_constant__ CUtensorMap x_map, const __grid_constant__ CUtensorMap w_map,
                       QuantizeArgs a) {
  using L = Layout<QJL>;
  constexpr int kLevels = 1 << BITS;
  extern __shared__ uint8_t smem_raw[];
  // y_full / z_full: the products of a tile's buffer are in tensor memory;
  // y_empty: the epilogue read that buffer (its second product, if any, too)
  __shared__ __align__(8) uint64_t w_full, x_full[L::kStages], x_empty[L::kStages], y_full[2], y_empty[2],
      res_full, z_full[2], drain;
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
      ptx::mbar_init(&x_full[s], 1);
      ptx::mbar_init(&x_empty[s], kEpiThreads);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&y_full[b], 1);
      ptx::mbar_init(&y_empty[b], kEpiThreads);
      ptx::mbar_init(&z_full[b], 1);
    }
    ptx::mbar_init(&res_full, kEpiThreads);
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
      for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
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
    if (lane == 0) {
      bool ok = ptx::wait_bar(&w_full, 0, abort, a.error, kErrTimeout);
      const uint32_t w_base = ptx::smem_u32(smem + L::kW0);
      int it = 0;
      for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x, ++it) {
        const int s = it % L::kStages;
        const uint32_t ph = (it / L::kStages) & 1;
        const int buf = it & 1;
        const uint32_t yb = tmem + buf * L::kBufCols;
        if (!ptx::wait_bar(&x_full[s], ph, abort, a.error, kErrTimeout)) break;
        // the buffer's previous tile (it - 2) has been read by the epilogue
        if (!ptx::wait_bar(&y_empty[buf], ((it >> 1) & 1) ^ 1, abort, a.error, kErrTimeout)) break;
        ptx::tc_fence_after();
        const uint32_t x_base = ptx::smem_u32(smem + L::kX0 + s * kMatBytes);
        uint32_t acc = 0;
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {          // R_hi, then R_lo
#pragma unroll
          for (int kb = 0; kb < 2; ++kb) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              const uint32_t off = kb * kHalfBytes + ks * 32;
              ptx::mma_bf16(yb, ptx::desc_k_sw128(x_base + off),
                            ptx::desc_k_sw128(w_base + pass * kMatBytes + off), kIdesc, acc);
              acc = 1;
            }
          }
        }
        ptx::mma_commit(&y_full[buf]);
        if (QJL) {
          if (!ptx::wait_bar(&res_full, it & 1, abort, a.error, kErrTimeout)) break;
          ptx::tc_fence_after();
          const uint32_t res_base = ptx::smem_u32(smem + L::kRes0);
          // (r_hi, S'_hi), (r_hi, S'_lo), (r_lo, S'_hi)
          acc = 0;
#pragma unroll
          for (int pass = 0; pass < 3; ++pass) {
            const int a_sel = pass == 2 ? 1 : 0;
            const int b_sel = pass == 1 ? 3 : 2;
#pragma unroll
            for (int kb = 0; kb < 2; ++kb) {
#pragma unroll
              for (int ks = 0; ks < 4; ++ks) {
                const uint32_t off = kb * kHalfBytes + ks * 32;
                ptx::mma_bf16(yb + 128, ptx::desc_k_sw128(res_base + a_sel * kMatBytes + off),
                              ptx::desc_k_sw128(w_base + b_sel * kMatBytes + off), kIdesc, acc);
                acc = 1;
              }
            }
          }
          ptx::mma_commit(&z_full[buf]);
        }
      }
      if (*abort) {
        ptx::mma_commit(&drain);
        ptx::drain_bar(&drain, 0);
      }
    }
  } else {
    // ---------------- epilogue: four threads per vector, 32 coordinates each ----------------
    const int quarter = warp & 3;                 // tensor-memory lanes this warp may access
    const int g = (warp - 2) >> 2;                // its coordinate group: 32 g .. 32 g + 31
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    float bnd[kLevels - 1];
#pragma unroll
    for (int i = 0; i < kLevels - 1; ++i) bnd[i] = a.bounds[i];
    float lev[kLevels];                           // read only by the QJL residual
#pragma unroll
    for (int i = 0; i < kLevels; ++i) lev[i] = QJL ? a.levels[i] : 0.f;
    const long long cache_rows = static_cast<long long>(a.num_blocks) * a.block_size;
    const bool bs_pow2 = (a.block_size & (a.block_size - 1)) == 0;
    const int bs_shift = __ffs(a.block_size) - 1;
    int it = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
      const int s = it % L::kStages;
      const uint32_t ph = (it / L::kStages) & 1;
      const int buf = it & 1;
      const uint32_t yb = lane_addr + buf * L::kBufCols;

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
      uint8_t* const x_tile = smem + L::kX0 + s * kMatBytes;
      const uint8_t* xrow = x_tile + (g >> 1) * kHalfBytes + row * 128;
      float ss = 0.f;
      if (ok) {
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
      ok = ok && ptx::wait_bar(&y_full[buf], (it >> 1) & 1, abort, a.error, kErrTimeout);
      // Once the products have read X, the first 4 bytes this thread read carry
      // its partial sum to the other three threads of the row (no other thread
      // reads those bytes, and the stage is refilled only after all have read).
      if (ok) *reinterpret_cast<float*>(x_tile + x_partial_offset(g, row)) = ss;
      // a failed wait anywhere ends every epilogue warp (the tcgen05.ld below
      // needs whole warps, the barriers below all 16)
      if (epi_sync_any(!ok || *abort)) break;
      const float n = sqrtf((*reinterpret_cast<const float*>(x_tile + x_partial_offset(0, row)) +
                             *reinterpret_cast<const float*>(x_tile + x_partial_offset(1, row))) +
                            (*reinterpret_cast<const float*>(x_tile + x_partial_offset(2, row)) +
                             *reinterpret_cast<const float*>(x_tile + x_partial_offset(3, row))));
      ptx::fence_async_shared();                  // the generic write above, before TMA refills the stage
      ptx::mbar_arrive(&x_empty[s]);
      const float inv = n > 0.f ? 1.f / n : 0.f;

      ptx::tc_fence_after();
      uint32_t planes[BITS];
      float rs = 0.f;
      {
        uint32_t yr[32];
        ptx::tmem_ld32(yb + 32 * g, yr);
#pragma unroll
        for (int p = 0; p < BITS; ++p) planes[p] = 0;
        float r[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float yv = __uint_as_float(yr[j]);
          const float y = yv * inv;
          bool b[BITS];
          code_bits<BITS>(y, bnd, b);
#pragma unroll
          for (int p = 0; p < BITS; ++p) planes[p] |= b[p] ? (1u << j) : 0u;
          if (QJL) {
            r[j] = fmaf(-n, level_of<BITS>(lev, b), yv);
            rs = fmaf(r[j], r[j], rs);
          }
        }
        if (QJL) {
          // 32 coordinates = 4 chunks of 8 in K block g / 2, chunks (g % 2) * 4 .. + 3
          uint8_t* res_hi = smem + L::kRes0 + (g >> 1) * kHalfBytes + row * 128;
          uint8_t* res_lo = res_hi + kMatBytes;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int chunk = (g & 1) * 4 + q;
            const int off = (chunk ^ (row & 7)) << 4;
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float r0 = r[q * 8 + 2 * e], r1 = r[q * 8 + 2 * e + 1];
              hw[e] = pack_bf16x2(r0, r1);
              lw[e] = pack_bf16x2(r0 - bf16_lo(hw[e]), r1 - bf16_hi(hw[e]));
            }
            *reinterpret_cast<uint4*>(res_hi + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(res_lo + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
        }
      }
      if (!QJL) {
        ptx::tc_fence_before();
        ptx::mbar_arrive(&y_empty[buf]);          // this buffer may take the tile after next
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
                transpose32(planes[p], lane);
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
      if (dst >= 0 && g == 0) a.norm[dst] = n;
      if (QJL) {
        ptx::fence_async_shared();
        ptx::mbar_arrive(&res_full);
        const bool zok = ptx::wait_bar(&z_full[buf], (it >> 1) & 1, abort, a.error, kErrTimeout);
        // the second products are done with the residual tile: its first 2 KB
        // carry the partial residual norms until the next tile's first barrier
        float* const rs_x = reinterpret_cast<float*>(smem + L::kRes0);
        if (zok) rs_x[g * kTileRows + row] = rs;
        if (epi_sync_any(!zok)) break;
        ptx::tc_fence_after();
        uint32_t zr[32];
        ptx::tmem_ld32(yb + 128 + 32 * g, zr);
        ptx::tc_fence_before();
        ptx::mbar_arrive(&y_empty[buf]);          // this buffer (Y and Z) may take the tile after next
        uint32_t word = 0;
#pragma unroll
        for (int j = 0; j < 32; ++j) word |= (__uint_as_float(zr[j]) > 0.f ? 1u : 0u) << j;
        if (dst >= 0) {
          reinterpret_cast<uint32_t*>(a.qjl + dst * 16)[g] = word;
          if (g == 0)
            a.rnorm[dst] = sqrtf((rs_x[row] + rs_x[kTileRows + row]) + (rs_x[2 * kTileRows + row] + rs_x[3 * kTileRows + row]));
        }
      }
      // No barrier closes the tile: the residual tile is rewritten only after
      // the next tile's first barrier, which a thread passes once every thread
      // has read this tile's partial residual norms.
    }
  }

  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, L::kTmemCols);
  }
}

template <int BITS, bool QJL, bool TRANS>
cudaError_t launch_bits(const CUtensorMap& x_map, const CUtensorMap& w_map, const QuantizeArgs& a, int grid,
                        cudaStream_t stream) {
  const int smem = Layout<QJL>::kBytes + 1024;
  cudaError_t err = cudaFuncSetAttribute(quantize_tc_kernel<BITS, QJL, TRANS>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  quantize_tc_kernel<BITS, QJL, TRANS><<<grid, kThreads, smem, stream>>>(x_map, w_map, a);
  return cudaGetLastError();
}

template <int BITS>
cudaError_t launch_kind(const CUtensorMap& x_map, const CUtensorMap& w_map, const QuantizeArgs& a, int grid,
                        cudaStream_t stream) {
  if (a.qjl != nullptr) return launch_bits<BITS, true, false>(x_map, w_map, a, grid, stream);
  if (a.transposed) return launch_bits<BITS, false, true>(x_map, w_map, a, grid, stream);
  return launch_bits<BITS, false, false>(x_map, w_map, a, grid, stream);
}

}  // namespace

cudaError_t launch_quantize_tc(const QuantizeArgs& a, const CUtensorMap& x_map, const CUtensorMap& w_map,
                               int num_sms, cudaStream_t stream) {
  if (a.n_vec <= 0) return cudaSuccess;
  if (a.qjl != nullptr && a.transposed) return cudaErrorInvalidValue;
  const int n_tiles = ((a.n_tokens + kTileRows - 1) / kTileRows) * a.n_kv;
  const int grid = n_tiles < num_sms ? n_tiles : num_sms;
  switch (a.bits) {
    case 1: return launch_kind<1>(x_map, w_map, a, grid, stream);
    case 2: return launch_kind<2>(x_map, w_map, a, grid, stream);
    case 3: return launch_kind<3>(x_map, w_map, a, grid, stream);
    case 4: return launch_kind<4>(x_map, w_map, a, grid, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tq
