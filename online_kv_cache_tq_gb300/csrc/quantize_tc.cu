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
// One persistent CTA per SM, 6 warps:
//   warp 0      TMA producer: R/S' hi/lo once, then 128-token tiles of X;
//   warp 1      tcgen05.mma issuer (and owner of the tensor-memory columns);
//   warps 2..5  epilogue, one thread per vector (tensor-memory lane): norm from
//               the X tile, codes and bit-planes from Y, residual hi/lo written
//               back to shared memory as the A operand of the second product,
//               then the QJL signs from Z.
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
constexpr int kThreads = 192;
constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(128, 128);

template <bool QJL>
struct Layout {
  static constexpr int kW = QJL ? 4 : 2;          // R_hi, R_lo (, S'_hi, S'_lo)
  static constexpr int kStages = QJL ? 1 : 3;     // X tiles in flight
  static constexpr int kW0 = 0;
  static constexpr int kX0 = kW * kMatBytes;
  static constexpr int kRes0 = kX0 + kStages * kMatBytes;
  static constexpr int kBytes = kRes0 + (QJL ? 2 * kMatBytes : 0);
  static constexpr uint32_t kTmemCols = QJL ? 256 : 128;
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

template <int BITS, bool QJL, bool TRANS>
__global__ void __launch_bounds__(kThreads, 1)
    quantize_tc_kernel(const __grid_constant__ CUtensorMap x_map, const __grid_constant__ CUtensorMap w_map,
                       QuantizeArgs a) {
  using L = Layout<QJL>;
  constexpr int kLevels = 1 << BITS;
  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t w_full, x_full[L::kStages], x_empty[L::kStages], y_full, y_empty, res_full,
      z_full, drain;
  __shared__ uint32_t tmem_base_s;
  __shared__ int abort_s;
  __shared__ float lev_s[kMaxLevels];

  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
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
      ptx::mbar_init(&x_empty[s], 128);
    }
    ptx::mbar_init(&y_full, 1);
    ptx::mbar_init(&y_empty, 128);
    ptx::mbar_init(&res_full, 128);
    ptx::mbar_init(&z_full, 1);
    ptx::mbar_init(&drain, 1);
    ptx::fence_mbar_init();
  }
  if (tid < kMaxLevels) lev_s[tid] = tid < kLevels ? a.levels[tid] : 0.f;
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
        if (!ptx::wait_bar(&x_full[s], ph, abort, a.error, kErrTimeout)) break;
        if (!ptx::wait_bar(&y_empty, (it & 1) ^ 1, abort, a.error, kErrTimeout)) break;
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
              ptx::mma_bf16(tmem, ptx::desc_k_sw128(x_base + off),
                            ptx::desc_k_sw128(w_base + pass * kMatBytes + off), kIdesc, acc);
              acc = 1;
            }
          }
        }
        ptx::mma_commit(&y_full);
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
                ptx::mma_bf16(tmem + 128, ptx::desc_k_sw128(res_base + a_sel * kMatBytes + off),
                              ptx::desc_k_sw128(w_base + b_sel * kMatBytes + off), kIdesc, acc);
                acc = 1;
              }
            }
          }
          ptx::mma_commit(&z_full);
        }
      }
      if (*abort) {
        ptx::mma_commit(&drain);
        ptx::drain_bar(&drain, 0);
      }
    }
  } else {
    // ---------------- epilogue: one thread per vector ----------------
    const int quarter = warp & 3;                 // tensor-memory lanes this warp may access
    const int row = quarter * 32 + lane;
    const uint32_t lane_addr = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    float bnd[kLevels - 1];
#pragma unroll
    for (int i = 0; i < kLevels - 1; ++i) bnd[i] = a.bounds[i];
    const long long cache_rows = static_cast<long long>(a.num_blocks) * a.block_size;
    int it = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++it) {
      const int s = it % L::kStages;
      const uint32_t ph = (it / L::kStages) & 1;
      bool ok = ptx::wait_bar(&x_full[s], ph, abort, a.error, kErrTimeout);
      ok = ok && ptx::wait_bar(&y_full, it & 1, abort, a.error, kErrTimeout);
      if (!__all_sync(0xffffffffu, ok)) break;    // tcgen05.ld below needs the whole warp
      // norm from the bf16 X row (swizzled: 16-byte chunk c of a row sits at c ^ (row % 8))
      const uint8_t* xrow = smem + L::kX0 + s * kMatBytes + row * 128;
      float ss = 0.f;
#pragma unroll
      for (int kb = 0; kb < 2; ++kb) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const uint4 q = *reinterpret_cast<const uint4*>(xrow + kb * kHalfBytes + ((c ^ (row & 7)) << 4));
          const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float lo = bf16_lo(w[e]), hi = bf16_hi(w[e]);
            ss = fmaf(lo, lo, ss);
            ss = fmaf(hi, hi, ss);
          }
        }
      }
      ptx::mbar_arrive(&x_empty[s]);
      const float n = sqrtf(ss);
      const float inv = n > 0.f ? 1.f / n : 0.f;

      const int head = tile / n_tt;
      const int token = (tile % n_tt) * kTileRows + row;
      long long dst = -1;
      long long slot = -1;
      if (token < a.n_tokens) {
        slot = slot_of(a, token);
        if (slot >= 0 && slot < cache_rows) {
          const long long blk = slot / a.block_size;
          dst = (blk * a.n_kv + head) * a.block_size + (slot - blk * a.block_size);
        } else if (slot >= cache_rows) {
          atomicCAS(a.error, 0, kErrSlot);
          slot = -1;
        }
      }

      ptx::tc_fence_after();
      uint32_t planes[BITS][4];
      float rs = 0.f;
      uint8_t* res_hi = smem + L::kRes0 + row * 128;
      uint8_t* res_lo = res_hi + kMatBytes;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t yr[32];
        ptx::tmem_ld32(lane_addr + c * 32, yr);
#pragma unroll
        for (int p = 0; p < BITS; ++p) planes[p][c] = 0;
        float r[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float yv = __uint_as_float(yr[j]);
          const float y = yv * inv;
          int code = 0;
#pragma unroll
          for (int i = 0; i < kLevels - 1; ++i) code += (y > bnd[i]) ? 1 : 0;
#pragma unroll
          for (int p = 0; p < BITS; ++p) planes[p][c] |= static_cast<uint32_t>((code >> p) & 1) << j;
          if (QJL) {
            r[j] = fmaf(-n, lev_s[code], yv);
            rs = fmaf(r[j], r[j], rs);
          }
        }
        if (QJL) {
          // 32 coordinates = 4 chunks of 8 in K block c/2, chunks (c%2)*4 .. +3
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int chunk = (c & 1) * 4 + q;
            const int off = (c >> 1) * kHalfBytes + ((chunk ^ (row & 7)) << 4);
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
      ptx::tc_fence_before();
      ptx::mbar_arrive(&y_empty);
      if (TRANS) {
        // token-transposed codes: whole words when the warp's 32 slots are
        // contiguous and start a 32-token group, single bits otherwise
        const long long slot0 = __shfl_sync(0xffffffffu, slot, 0);
        const bool aligned = __all_sync(0xffffffffu, dst >= 0 && slot == slot0 + lane && (slot0 & 31) == 0);
        unsigned* words = reinterpret_cast<unsigned*>(a.codes);
        if (aligned) {
          const long long blk = slot0 / a.block_size;
          const int off0 = static_cast<int>(slot0 - blk * a.block_size);
#pragma unroll
          for (int p = 0; p < BITS; ++p)
#pragma unroll
            for (int c = 0; c < 4; ++c)
              words[transposed_word(blk, head, a.n_kv, BITS, p, 32 * c + lane, a.block_size, off0)] =
                  transpose32(planes[p][c], lane);
        } else if (dst >= 0) {
          const long long blk = slot / a.block_size;
          const int off = static_cast<int>(slot - blk * a.block_size);
          const unsigned mask = 1u << (off & 31);
          for (int p = 0; p < BITS; ++p)
            for (int c = 0; c < 4; ++c)
              for (int j = 0; j < 32; ++j) {
                unsigned* w = words + transposed_word(blk, head, a.n_kv, BITS, p, 32 * c + j, a.block_size, off);
                if ((planes[p][c] >> j) & 1) atomicOr(w, mask); else atomicAnd(w, ~mask);
              }
        }
      } else if (dst >= 0) {
        uint4* out = reinterpret_cast<uint4*>(a.codes + dst * (BITS * 16));
#pragma unroll
        for (int p = 0; p < BITS; ++p) out[p] = make_uint4(planes[p][0], planes[p][1], planes[p][2], planes[p][3]);
      }
      if (dst >= 0) a.norm[dst] = n;
      if (QJL) {
        ptx::fence_async_shared();
        ptx::mbar_arrive(&res_full);
        const bool zok = ptx::wait_bar(&z_full, it & 1, abort, a.error, kErrTimeout);
        if (!__all_sync(0xffffffffu, zok)) break;
        ptx::tc_fence_after();
        uint32_t sw[4];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t zr[32];
          ptx::tmem_ld32(lane_addr + 128 + c * 32, zr);
          uint32_t word = 0;
#pragma unroll
          for (int j = 0; j < 32; ++j) word |= (__uint_as_float(zr[j]) > 0.f ? 1u : 0u) << j;
          sw[c] = word;
        }
        ptx::tc_fence_before();
        if (dst >= 0) {
          *reinterpret_cast<uint4*>(a.qjl + dst * 16) = make_uint4(sw[0], sw[1], sw[2], sw[3]);
          a.rnorm[dst] = sqrtf(rs);
        }
      }
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
