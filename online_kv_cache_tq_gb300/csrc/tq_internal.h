// Internal declarations shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>

#include "tq.h"

#include <cuda.h>

namespace tq {

constexpr int kDim = 128;       // head dimension supported by the kernels
constexpr int kMaxLevels = 16;  // 4-bit codebooks at most

// Codebook tables as the kernels read them (float32, one struct in device
// memory).  Boundaries are padded with +inf so a kernel may compare against
// all 15 entries whatever the bit width.
struct DeviceTables {
  float k_levels[kMaxLevels];
  float k_bounds[kMaxLevels];
  float v_levels[kMaxLevels];
  float v_bounds[kMaxLevels];
  // Coefficients of a codebook written in sign planes: with s_p = 2 bit_p - 1
  // for the bits of a code, level(code) = sum_S walsh[S] * prod_{p in S} s_p
  // over the odd subsets S (1 plane at 1 bit, 2 at 2 bits, 4 at 3 bits:
  // {0},{1},{2},{0,1,2}; 8 at 4 bits: {0},{1},{2},{3},{0,1,2},{0,1,3},{0,2,3},
  // {1,2,3}).  Exact for the symmetric Lloyd-Max codebooks.
  float k_walsh[8];
  float v_walsh[8];
};

// Odd sign-plane subsets, as bit masks over the code bits, in walsh[] order.
constexpr int kWalshSets[4][8] = {{1}, {1, 2}, {1, 2, 4, 7}, {1, 2, 4, 8, 7, 11, 13, 14}};

// Host-side construction products (fp64), independent of any device.
struct HostTables {
  std::vector<double> R;         // d x d, y = R x
  std::vector<double> S;         // m x d
  std::vector<double> Sp;        // m x d, S' = S R^T (acts on rotated residuals)
  std::vector<double> k_levels;  // 2^k_mse_bits
  std::vector<double> k_bounds;
  std::vector<double> v_levels;  // 2^v_bits
  std::vector<double> v_bounds;
};

// Build R, S, S' and the codebooks on the host (host_builder.cpp).
void build_host_tables(int d, int qjl_m, uint64_t seed, int k_mse_bits, int v_bits, HostTables* out);

// Every host-side check of tq_decode_attention for a workspace of
// workspace_bytes (api.cu); launches nothing.
tq_status check_decode_call(const tq_codebook* book, const void* q, tq_dtype dtype, int batch, int n_q_heads,
                            int n_kv_heads, const tq_cache_view* cache, const int32_t* block_table, int max_blocks,
                            const int32_t* context_lens, int max_context, float scale, float* out,
                            size_t workspace_bytes);

}  // namespace tq

struct tq_codebook {
  tq_config cfg;
  int device;         // -1: host-only handle
  int k_mse_bits;
  int v_bits;
  tq::HostTables host;
  // Device copies (float32 unless noted), owned by the handle.
  float* d_R;         // [d][d] row-major R
  float* d_Rt;        // [d][d] R transposed
  float* d_Spt;       // [d][m] S' transposed (column k of S' is row k)
  float* d_St;        // [d][m] S transposed: S q = S' R q for a query q
  uint16_t* d_rot_tc; // bf16 hi/lo operand images for the tensor-core quantizer
  tq::DeviceTables* d_tables;
  int* d_error;       // first device-side error code, 0 when none
  int num_sms;
  CUtensorMap w_map;  // TMA map of d_rot_tc as [512][128] bf16
  bool walsh_ok;      // both codebooks are exactly odd-symmetric (sign-plane decode usable)
  bool norm16;        // norms stored as float16 (norm_bits 16)
  bool polar;         // PolarQuant records instead of Lloyd-Max codes (codec TQ_CODEC_POLAR)
  int debug_withhold; // tq_debug_withhold_commit (tests of the bounded waits only)
};
