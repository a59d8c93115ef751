// Kernel launchers (CUDA translation units) called by the C ABI layer.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "tq_internal.h"

namespace tq {

// Error codes a kernel records in the handle's error word.
enum DeviceError : int { kErrSlot = 1, kErrBlock = 2, kErrContext = 3, kErrTimeout = 4, kErrPartials = 5 };

struct QuantizeArgs {
  const void* x;          // [n_tokens][n_kv][128], bf16 or fp32
  int n_vec;              // n_tokens * n_kv_heads
  int n_tokens;
  int n_kv;
  bool transposed;        // codes field stored token-transposed (values)
  const int64_t* slots;   // [n_tokens]; null: a decode step, slot derived below
  const int32_t* step_block_table;   // decode step: [n_tokens][step_max_blocks] (null: identity)
  const int32_t* step_context_lens;  // decode step: token b is position context_lens[b] - 1 of sequence b
  int step_max_blocks;
  uint8_t* codes;         // field base, bits * 16 bytes per item
  uint8_t* qjl;           // field base, 16 bytes per item (null: no QJL)
  void* norm;             // float32, or float16 with norm16
  void* rnorm;            // null when no QJL
  bool norm16;
  int num_blocks;
  int block_size;
  int bits;               // MSE bits of this tensor
  const float* levels;    // 2^bits device floats
  const float* bounds;    // 15 device floats, +inf padded
  const float* Rt;        // [128][128], Rt[i][o] = R[o][i]
  const float* Spt;       // [128][128], Spt[j][k] = S'[k][j]
  int* error;
};

// Norm fields hold float32, or float16 (rounded to nearest) with norm16.
__device__ __forceinline__ float load_norm(const void* p, long long i, bool n16) {
  return n16 ? __half2float(reinterpret_cast<const __half*>(p)[i]) : reinterpret_cast<const float*>(p)[i];
}
__device__ __forceinline__ void store_norm(void* p, long long i, float v, bool n16) {
  if (n16) reinterpret_cast<__half*>(p)[i] = __float2half_rn(v);
  else reinterpret_cast<float*>(p)[i] = v;
}
// The value a norm field will hold for v (what the decoder reconstructs with).
__device__ __forceinline__ float stored_norm(float v, bool n16) { return n16 ? __half2float(__float2half_rn(v)) : v; }

// Cache slot of token `token` of an append: slot_mapping[token], or for a
// decode step (one token per sequence, slots == null) the slot of position
// context_lens[token] - 1 of that sequence under its block table (-1, i.e.
// skipped, for an empty context).
__device__ __forceinline__ long long slot_of(const QuantizeArgs& a, int token) {
  if (a.slots != nullptr) return a.slots[token];
  const int pos = a.step_context_lens[token] - 1;
  if (pos < 0) return -1;
  const int lblk = pos / a.block_size;
  if (lblk >= a.step_max_blocks) return static_cast<long long>(a.num_blocks) * a.block_size;   // out of range
  const long long phys = a.step_block_table ? a.step_block_table[static_cast<long long>(token) * a.step_max_blocks + lblk]
                                            : static_cast<long long>(token) * a.step_max_blocks + lblk;
  if (phys < 0) return static_cast<long long>(a.num_blocks) * a.block_size;
  return phys * a.block_size + pos % a.block_size;
}


// Small batches (up to kSmallQuantize vectors per tensor): one CTA per
// vector; K and V (either may be null) share one launch.
constexpr int kSmallQuantize = 1024;
cudaError_t launch_quantize_small(const QuantizeArgs* first, const QuantizeArgs* second, bool bf16,
                                  cudaStream_t stream);

// Tile quantizer on the tensor cores; x_map tiles bf16 x as [n_tokens][n_kv][128]
// in boxes of 64 columns x 1 head x 128 tokens (128-byte swizzle), w_map tiles
// the handle's bf16 hi/lo images of R and S' as [512][128].  f32: x is fp32,
// read by converter warps into bf16 hi/lo operands (x_map unused).
cudaError_t launch_quantize_tc(const QuantizeArgs& args, const CUtensorMap& x_map, const CUtensorMap& w_map,
                               int num_sms, bool f32, cudaStream_t stream);

// Where the split-K partials of one query head are: entries base,
// base + stride, ..., base + (count - 1) stride of the partials array, each
// (m, l, 2 pad, acc[128]).  The SIMT kernel writes one entry per 512-token
// chunk (stride 1); the tensor-core kernel one per run of consecutive chunks
// that a CTA processed (stride G, the entries of a group's G query heads
// side by side).
struct SegInfo {
  int base, count, stride, pad;
};

struct DecodeArgs {
  const void* q;            // [batch][n_q][128]
  int batch, n_q, n_kv, group;
  const uint8_t* k_codes;
  const uint8_t* k_qjl;     // null: no QJL
  const void* k_norm;       // float32, or float16 with norm16
  const void* k_rnorm;
  const uint8_t* v_codes;
  const void* v_norm;
  bool norm16;
  int num_blocks, block_size;
  int k_bits, v_bits, qjl_m;
  const int32_t* block_table;  // null: identity
  int max_blocks;
  const int32_t* context_lens;
  int max_context;
  float scale;
  float qjl_coef;           // sqrt(pi/2) / m
  float* out;               // [batch][n_q][128]
  float* ws_q;              // [batch*n_q][256]: rotated query, projected query
  float* ws_part;           // partial entries of kPartStride floats (see SegInfo)
  uint8_t* ws_bk;           // [batch*n_q][bk_stride]: tensor-core score operand pieces (null: not built)
  int* ws_ticket;           // [batch*n_q]: per (sequence, KV head) count of finished segments
  SegInfo* ws_seg;          // [batch*n_q]: where each query head's partials are
  int bk_stride;
  int max_chunks;
  int merge_in_partials;    // the tensor-core kernel merges and writes `out` itself
  long long part_cap;       // partial entries the workspace holds (merges check records against it)
  int debug_withhold;       // tests of the bounded waits: CTA 0 withholds its first score commit
  const float* R;           // [128][128] row-major
  const float* Rt;
  const float* Spt;
  const float* St;          // [128][128], St[i][k] = S[k][i]: the projected query S' R q = S q
  const DeviceTables* tables;
  int* error;
  int num_sms;              // of the handle's device
  bool polar;               // PolarQuant records (polar.cu) instead of Lloyd-Max codes
};

// Word (uint32 units) of a token-transposed codes field holding plane p,
// coordinate `dim` of the 32-token group of slot offset `off` in block `blk`.
__host__ __device__ inline long long transposed_word(long long blk, int head, int n_kv, int bits, int p, int dim,
                                                     int block_size, int off) {
  return (((blk * n_kv + head) * bits + p) * 128 + dim) * (block_size / 32) + off / 32;
}

constexpr int kChunk = 512;       // context tokens per split-K work item
constexpr int kQPieces = 5;       // e4m3 pieces of a query coefficient (tensor-core decode)

// Bytes of one query head's tensor-core score operand in the decode
// workspace: for each key sign plane and the QJL plane, kQPieces rows of 128
// e4m3 bytes (row i: piece i of 2 a_S q_rot / beta or of 2 q_s / beta, in the
// K order of k_position), then 8 floats: sigma_mse, sigma_qjl, their
// inverses, (sum_S a_S) (sum_j q_rot_j), sum_k q_s_k, and two unused.
constexpr int kBkHeader = 32;
__host__ __device__ constexpr int bk_head_bytes(int k_mse_bits, bool qjl) {
  return ((k_mse_bits >= 1 ? (1 << (k_mse_bits - 1)) : 0) + (qjl ? 1 : 0)) * kQPieces * 128 + kBkHeader;
}
constexpr int kPartStride = 132;  // m, l, 2 pad, acc[128]

// Partial entries a decode workspace holds: one per (query head, chunk) for
// the SIMT kernel, and for the tensor-core kernel one per (query head,
// segment), where a (sequence, KV head) group has one segment per CTA whose
// run of chunks touches it, i.e. at most n_groups + n_ctas segments of G
// entries, n_ctas <= 2 num_sms.
__host__ __device__ constexpr long long partial_entries(long long n_vec, int max_chunks, int num_sms) {
  return n_vec * max_chunks > n_vec + 16ll * num_sms ? n_vec * max_chunks : n_vec + 16ll * num_sms;
}

cudaError_t launch_decode_prepare(const DecodeArgs& args, bool bf16, cudaStream_t stream);

// Reconstruction-error statistics of appended vectors (monitor.cu): adds
// sum ||x - x_hat||, sum ||x - x_hat||^2, sum ||x||^2 and the vector count
// into stats[0..3] (x_hat: the stage-1 reconstruction the cache holds).
cudaError_t launch_monitor(const QuantizeArgs& args, bool bf16, double* stats, cudaStream_t stream);

// Quantize-append of one new key and value per sequence (ka and va share the
// shape, at most kSmallQuantize vectors each) and the query preparation of
// the same decode step, in one launch.
cudaError_t launch_step_prep(const QuantizeArgs& ka, const QuantizeArgs& va, bool kv_bf16, const DecodeArgs& da,
                             bool q_bf16, cudaStream_t stream);
cudaError_t launch_decode_partials(const DecodeArgs& args, cudaStream_t stream);

// PolarQuant codec (polar.cu): records of keys or values (args.codes: 64 bytes
// per item, args.norm: the float32 final radius), and the split-K partials of
// a PolarQuant cache in the CUDA-core kernel's entry layout.
cudaError_t launch_polar_quantize(const QuantizeArgs& args, bool bf16, cudaStream_t stream);
cudaError_t launch_polar_partials(const DecodeArgs& args, cudaStream_t stream);

// Tensor-core partials (fp8 sign planes, decode_tc.cu) for the shapes it
// supports: G in {1, 2, 4, 8}, tensor-memory columns within 512, and
// odd-symmetric codebooks; the SIMT kernel serves every other shape.
bool tc_decode_supported(const DecodeArgs& args, bool walsh_ok);
// early: launched as a programmatic dependent of the decode step's fused
// append + query preparation; the kernel waits for that grid only before it
// reads the query operands and the chunk that holds the appended token.
cudaError_t launch_decode_partials_tc(const DecodeArgs& args, cudaStream_t stream, bool early);
// Whether the tensor-core kernel should merge in place (few groups per CTA)
// rather than leave the merge to launch_merge_groups_tc, a programmatic
// dependent launch.
bool tc_merge_in_partials(const DecodeArgs& args);
// Whether that merge launch takes one CTA per query head (few groups: long
// contexts over a small batch) rather than one per group.
bool tc_merge_per_head(const DecodeArgs& args);
int tc_grid(const DecodeArgs& args);   // CTAs of the persistent tensor-core grid
int tc_chunk(const DecodeArgs& args);  // tokens per work item of the tensor-core kernel
cudaError_t launch_merge_groups_tc(const DecodeArgs& args, cudaStream_t stream);
// early: launched as a programmatic dependent of the tensor-core partials
// kernel (the merge waits for it before reading the partials).
cudaError_t launch_decode_finish(const DecodeArgs& args, cudaStream_t stream, bool early = false);
// The merge over the partials of two parts of every sequence's context (two
// caches, each with its own handle and workspace; the same R), into first.out.
cudaError_t launch_decode_finish_parts(const DecodeArgs& first, const DecodeArgs& second, cudaStream_t stream);

}  // namespace tq
