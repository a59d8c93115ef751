/*
 * tq.h -- C ABI of the TurboQuant KV-cache engine (sm_103a).
 *
 * The method (TurboQuant, "Online Vector Quantization with Near-optimal
 * Distortion Rate", as described by the 甲子光年 article on admirer.cn, §2):
 *   stage 1 (§2 第一階段): keep the vector norm, rotate the unit vector with a
 *     random orthogonal R, replace every rotated coordinate by the nearest level
 *     of a Lloyd-Max codebook built once for the rotated-coordinate Beta law;
 *   stage 2 (§2 第二階段): for keys, spend b-1 bits on stage 1 and one bit per
 *     projected coordinate on QJL, sign(S * residual), plus the residual norm,
 *     which makes the inner-product estimate unbiased.
 * Decode attention runs directly on the packed cache (seo-farm page §4: the
 * query is not compressed; attention reads the de-quantized cache), in the
 * rotated space, with one back-rotation by R^T at the end (seo-farm page §2:
 * R^T R = I leaves attention unchanged).
 *
 * Conventions shared by every entry point
 * - All functions return tq_status; TQ_OK is 0.  Argument checks run on the
 *   host before anything is launched; a rejected call launches nothing and
 *   leaves every buffer untouched.
 * - Device pointers are plain CUDA device addresses on the handle's device and
 *   are owned by the caller (the library never frees them).  The only memory
 *   the library owns is the handle's (R, S' = S R^T, codebooks, an error word).
 * - Launches are asynchronous on the caller's stream (cudaStream_t passed as
 *   void*; NULL is the legacy default stream).  No entry point synchronises
 *   except tq_codebook_build, tq_codebook_destroy and tq_get_last_device_error.
 * - Launch failures map to TQ_ERR_CUDA.  Bad indices met on the device (a slot
 *   or block id outside the cache) never trap: the kernel skips that item and
 *   records an error code readable with tq_get_last_device_error.
 * - A handle is immutable after build and may be used from several streams.
 */
#ifndef TQ_H_
#define TQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  TQ_OK = 0,
  TQ_ERR_INVALID_ARG = 1, /* null pointer, bad size, inconsistent shapes      */
  TQ_ERR_UNSUPPORTED = 2, /* valid but not built: d != 128, bits outside 1..4 */
  TQ_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed             */
  TQ_ERR_OOM = 4,         /* host or device allocation failed (build only)    */
  TQ_ERR_WORKSPACE = 5,   /* decode workspace null or smaller than required   */
  TQ_ERR_DEVICE = 6       /* a kernel met an invalid slot/block id (see below) */
} tq_status;

typedef enum { TQ_BF16 = 0, TQ_FP32 = 1 } tq_dtype;

/* Configuration.  d: head dimension (128 only).  k_bits: total key bits per
 * coordinate; with QJL on (qjl_m > 0) keys use k_bits-1 MSE bits + the 1-bit
 * sketch, so k_bits is 2..5; with QJL off keys use k_bits MSE bits (1..4).
 * v_bits: value MSE bits (1..4).  qjl_m: QJL projection rows (0 = off, or
 * 128).  seed: seeds the SplitMix64 stream that draws R (Haar, via QR of a
 * Gaussian matrix) and S.  block_size: tokens per cache block, a multiple of
 * 32 for device handles.  norm_bits: width of the stored norms (the vector
 * norm and, for keys, the residual norm): 32 (or 0) for float32, 16 for
 * float16, which saves 6 of the 108 bytes of a (token, head) at 3/3 bits;
 * the key residual is then taken against the float16 norm, the value the
 * decoder reconstructs.  codec: TQ_CODEC_TURBOQUANT (0) for the stage above,
 * or TQ_CODEC_POLAR (1) for PolarQuant, the alternative stage 1 of the
 * intelliparadigm.com page (§2.1.1 step 2): after the same rotation,
 * coordinates are paired into (radius, angle) level after level, every angle
 * rounded to a multiple of pi/12, the final radius kept; keys and values are
 * both coded so (k_bits and v_bits are ignored), qjl_m must be 0 and norms
 * are float32.  A PolarQuant record is 64 bytes (64 level-1 codes 0..23 x 5
 * bits, then the 63 codes of levels 2..7, 0..6, x 3 bits, one little-endian
 * bit stream), token-major for values too. */
typedef enum { TQ_CODEC_TURBOQUANT = 0, TQ_CODEC_POLAR = 1 } tq_codec;

typedef struct {
  int d;
  int k_bits;
  int v_bits;
  int qjl_m;
  uint64_t seed;
  int block_size;
  int norm_bits;
  int codec;
} tq_config;

typedef struct tq_codebook tq_codebook; /* opaque, library-owned */

/* The compressed cache: caller-owned device arrays, each laid out as
 * [num_blocks][n_kv_heads][block_size][item], item sizes from
 * tq_cache_field_bytes.  Key codes are bit-planes per token: plane p holds
 * bit p of every code, coordinate j at bit j%8 of byte j/8 of the plane.
 * Value codes are stored token-transposed inside each block so that decode
 * can contract over tokens: the value field of one (block, head) is
 * [v_bits][d][block_size/8] bytes, and for plane p and coordinate j, bit t%8
 * of byte t/8 holds bit p of the code of the token at offset t (the same
 * bytes per token as the key layout).  QJL bit k is bit k%8 of byte k/8, set
 * when the k-th projected residual is > 0.  Norms are float32, or float16
 * when the handle was built with norm_bits 16.  Every pointer must be 16-byte
 * aligned; k_qjl/k_rnorm may be NULL when qjl_m == 0. */
typedef struct {
  void* k_codes;
  void* k_qjl;
  void* k_norm;
  void* k_rnorm;
  void* v_codes;
  void* v_norm;
  int num_blocks;
  int n_kv_heads;
  int block_size;
} tq_cache_view;

/* Build a handle: draws R and S, computes S' = S R^T and the Lloyd-Max
 * codebooks in fp64 on the host, then uploads float32 copies (and bf16 hi/lo
 * splits for the tensor-core rotation) to `device`.  device < 0 builds a
 * host-only handle whose tables can be inspected but which the kernels
 * reject.  Synchronous.  Ownership of *out passes to the caller, who frees it
 * with tq_codebook_destroy. */
tq_status tq_codebook_build(const tq_config* cfg, int device, tq_codebook** out);
tq_status tq_codebook_destroy(tq_codebook* book);

/* fp64 copies of the codebook: which = 0 keys, 1 values.  levels gets
 * 2^bits ascending values, bounds the 2^bits - 1 midpoints (either may be
 * NULL).  *bits (may be NULL) receives the MSE bit width of that codebook. */
tq_status tq_codebook_levels(const tq_codebook* book, int which, double* levels, double* bounds,
                             int* bits);

/* fp64 copies of R (d x d, row-major, y = R x) and S (qjl_m x d, row-major);
 * either may be NULL. */
tq_status tq_codebook_matrices(const tq_codebook* book, double* R, double* S);

/* Bytes per (token, head) item of the six cache fields, in the order
 * k_codes, k_qjl, k_norm, k_rnorm, v_codes, v_norm (0 for absent fields). */
tq_status tq_cache_field_bytes(const tq_codebook* book, size_t bytes_per_item[6]);

/* Quantize-append (the write path; 甲子光年 article §2 第一階段 for the
 * norm, rotation, Lloyd-Max code and bit packing of every vector, §2 第二階段
 * for the keys' QJL sign bits and residual norm).  k, v: device [n_tokens][n_kv_heads][d]
 * in `dtype`, contiguous, 16-byte aligned; either may be NULL to skip that
 * tensor.  slot_mapping: device int64 [n_tokens]; token t goes to slot
 * slot_mapping[t] (block = slot / block_size, offset = slot % block_size);
 * a negative slot skips the token; a slot >= num_blocks*block_size is skipped
 * and recorded as a device error.  Writes every field of every (token, head).
 * Asynchronous on `stream`. */
tq_status tq_quantize_append(const tq_codebook* book, const void* k, const void* v, tq_dtype dtype,
                             int n_tokens, int n_kv_heads, const int64_t* slot_mapping,
                             const tq_cache_view* cache, void* stream);

/* Reconstruction-error monitor (intelliparadigm.com §3.3 tracks the running
 * mean of ||original - quantized||_2 in a deployment; the reconstruction is
 * the stage-1 one of 甲子光年 article §2 第一階段, x_hat = n R^T c[code]).
 * For the vectors x: device [n_tokens][n_kv_heads][d] in `dtype` that an
 * earlier tq_quantize_append wrote at slot_mapping (same slots, same cache),
 * which = 0 for keys, 1 for values, the call ADDS into stats (device, four
 * doubles, 8-byte aligned): sum over vectors of ||x - x_hat||, of
 * ||x - x_hat||^2, of ||x||^2, and the number of vectors (negative or
 * out-of-range slots are skipped).  A caller keeps a running mean by zeroing
 * stats once and calling this after each append; stats[0] / stats[3] is the
 * mean error, stats[1] / stats[2] the relative squared error.  For keys with
 * QJL, ||x - x_hat|| is also the stored residual norm.  Reads the cache only;
 * asynchronous on `stream`; calls that overlap on the GPU may add into the
 * same stats. */
tq_status tq_reconstruction_error(const tq_codebook* book, const void* x, tq_dtype dtype, int which, int n_tokens,
                                  int n_kv_heads, const int64_t* slot_mapping, const tq_cache_view* cache,
                                  double* stats, void* stream);

/* Workspace bytes tq_decode_attention needs for this batch shape (the
 * split-K partials and the rotated/projected queries).  max_context bounds
 * every context_lens[b]. */
size_t tq_decode_workspace_bytes(const tq_codebook* book, int batch, int n_q_heads, int max_context);

/* Decode attention (the read path; 甲子光年 article §2 第二階段 for the score
 * estimate n <R q, c[code]> + gamma sqrt(pi/2)/m <S q, 2 bits - 1>, seo-farm
 * page §4 for attention over the de-quantized cache with the query left
 * uncompressed, §2 for working in the rotated space and back-rotating once)
 * for one new query token per sequence.
 * q: device [batch][n_q_heads][d] in `dtype`.  Query head h reads KV head
 * h / (n_q_heads / n_kv_heads).  block_table: device int32 [batch][max_blocks]
 * of physical block ids, or NULL for the identity layout (sequence b owns
 * blocks b*max_blocks .. b*max_blocks + max_blocks - 1).  context_lens: device
 * int32 [batch], each in [0, max_context] and <= max_blocks*block_size; a
 * zero-length sequence yields a zero output row.  scale: softmax scale, 0
 * selects 1/sqrt(d).  out: device float32 [batch][n_q_heads][d].  workspace:
 * device scratch of at least tq_decode_workspace_bytes(book, batch,
 * n_q_heads, max_context) bytes, 256-byte aligned, not used by any concurrent
 * call.  Asynchronous on `stream`. */
tq_status tq_decode_attention(const tq_codebook* book, const void* q, tq_dtype dtype, int batch,
                              int n_q_heads, int n_kv_heads, const tq_cache_view* cache,
                              const int32_t* block_table, int max_blocks,
                              const int32_t* context_lens, int max_context, float scale, float* out,
                              void* workspace, size_t workspace_bytes, void* stream);

/* One decode step in one call: append one new key and value per sequence at
 * position context_lens[b] - 1 of sequence b (the slot follows from
 * block_table exactly as decode reads it), then decode attention for one
 * query per sequence over the cache that now holds them.  k_new, v_new:
 * device [batch][n_kv_heads][d] in kv_dtype (both required when batch > 0);
 * every other argument as in tq_decode_attention, and context_lens already
 * counts the appended token (a sequence with context 0 appends nothing).
 * Equivalent to tq_quantize_append with those slots followed by
 * tq_decode_attention.  When batch * n_kv_heads <= 1024 the append and the
 * query preparation share one launch, and the partials kernel starts while
 * it runs (a programmatic dependent launch that waits for it only where it
 * reads the query operands and the chunk holding the appended token).
 * Asynchronous on `stream`. */
tq_status tq_decode_step(const tq_codebook* book, const void* k_new, const void* v_new, tq_dtype kv_dtype,
                         const void* q, tq_dtype q_dtype, int batch, int n_q_heads, int n_kv_heads,
                         const tq_cache_view* cache, const int32_t* block_table, int max_blocks,
                         const int32_t* context_lens, int max_context, float scale, float* out,
                         void* workspace, size_t workspace_bytes, void* stream);

/* Device workspace bytes tq_decode_step_host needs: the decode workspace of
 * (batch, n_q_heads, max_context) after a staging area for one step's inputs
 * (k_new, v_new, q, context_lens) and output. 0 for invalid arguments. */
size_t tq_decode_step_host_workspace_bytes(const tq_codebook* book, int batch, int n_q_heads, int n_kv_heads,
                                           int max_context, tq_dtype kv_dtype, tq_dtype q_dtype);

/* tq_decode_step with the step's inputs and output in HOST memory, for a
 * caller whose tokens arrive from and leave to the host: k_new_h, v_new_h
 * [batch][n_kv_heads][128] (kv_dtype), q_h [batch][n_q_heads][128] (q_dtype),
 * context_lens_h [batch] int32 (each sequence's length including the new
 * token) and out_h [batch][n_q_heads][128] fp32 are host addresses; they
 * should be page-locked (cudaHostAlloc / pinned) so that the copies overlap
 * the host, pageable memory works but its copies block the calling thread.
 * The call copies the inputs into the staging area at the start of
 * `workspace` (one cudaMemcpyAsync each), runs tq_decode_step on those device
 * copies with the rest of the workspace, and copies the output back, all in
 * order on `stream`: out_h holds the result once the caller synchronises the
 * stream, and the host inputs may be reused only then. block_table stays a
 * device array (it belongs to the cache, not to the step). Argument meaning,
 * checks and errors are those of tq_decode_step, plus TQ_ERR_WORKSPACE when
 * workspace_bytes is below tq_decode_step_host_workspace_bytes, and
 * TQ_ERR_CUDA when a copy cannot be queued. */
tq_status tq_decode_step_host(const tq_codebook* book, const void* k_new_h, const void* v_new_h,
                              tq_dtype kv_dtype, const void* q_h, tq_dtype q_dtype, int batch, int n_q_heads,
                              int n_kv_heads, const tq_cache_view* cache, const int32_t* block_table,
                              int max_blocks, const int32_t* context_lens_h, int max_context, float scale,
                              float* out_h, void* workspace, size_t workspace_bytes, void* stream);

/* The first stage of tq_decode_step, for callers that run the stages one at a
 * time (then tq_decode_partials and tq_decode_finish with the step's
 * arguments): the append of k_new / v_new and the query preparation, in one
 * launch when batch * n_kv_heads <= 1024.  Arguments as tq_decode_step. */
tq_status tq_decode_step_prepare(const tq_codebook* book, const void* k_new, const void* v_new,
                                 tq_dtype kv_dtype, const void* q, tq_dtype q_dtype, int batch,
                                 int n_q_heads, int n_kv_heads, const tq_cache_view* cache,
                                 const int32_t* block_table, int max_blocks, const int32_t* context_lens,
                                 int max_context, void* workspace, size_t workspace_bytes, void* stream);

/* The three stages tq_decode_attention runs, callable one at a time on the
 * same stream with the same arguments and workspace (e.g. to overlap query
 * preparation with other work, or to time the stages):
 *   tq_decode_prepare  -- rotated query R q and projected query S' R q into
 *                         the workspace (seo-farm page §4: the query is rotated,
 *                         not quantized);
 *   tq_decode_partials -- per context chunk and KV head: scores from the packed
 *                         codes plus the QJL correction (甲子光年 §2 第二階段),
 *                         chunk max/sum and the value sum in the rotated space.
 *                         With out == NULL it leaves split-K partials in the
 *                         workspace for tq_decode_finish.  With an `out`
 *                         (device float32 [batch][n_q_heads][d]) it leaves the
 *                         final output there instead, as tq_decode_attention's
 *                         last two stages do (the tensor-core kernel merges
 *                         each (sequence, KV head) in place or is followed by
 *                         a merge launch, as tq_decode_plan reports; after the
 *                         CUDA-core kernel the merge runs as a second launch);
 *                         calling tq_decode_finish afterwards is allowed and
 *                         redundant;
 *   tq_decode_finish   -- merge the partials, divide by the softmax sum and
 *                         back-rotate by R^T into `out`.
 * Argument meaning, checks and errors are those of tq_decode_attention. */
tq_status tq_decode_prepare(const tq_codebook* book, const void* q, tq_dtype dtype, int batch,
                            int n_q_heads, int max_context, void* workspace, size_t workspace_bytes,
                            void* stream);
tq_status tq_decode_partials(const tq_codebook* book, int batch, int n_q_heads, int n_kv_heads,
                             const tq_cache_view* cache, const int32_t* block_table, int max_blocks,
                             const int32_t* context_lens, int max_context, float scale, float* out,
                             void* workspace, size_t workspace_bytes, void* stream);
tq_status tq_decode_finish(const tq_codebook* book, int batch, int n_q_heads,
                           const int32_t* context_lens, int max_context, int max_blocks, float* out,
                           void* workspace, size_t workspace_bytes, void* stream);

/* Size of the scratch array compiled into the library for
 * tq_decode_attention_static: 16 MiB per GPU that loads the library, held
 * until the process exits. */
#define TQ_STATIC_WORKSPACE_BYTES (16u << 20)

/* tq_decode_attention for callers that cannot allocate device memory (for
 * example a serving runtime whose memory pool owns the whole GPU, or a loop
 * where a device allocation and the synchronisation it may cause are not
 * allowed).  Same arguments, checks and results as tq_decode_attention, but
 * the split-K scratch is a fixed array inside the library instead of a
 * caller-supplied workspace; the call allocates nothing.  The paper has no
 * counterpart: this is an interface convenience, not part of the method.
 * - Returns TQ_ERR_WORKSPACE when tq_decode_workspace_bytes(book, batch,
 *   n_q_heads, max_context) exceeds TQ_STATIC_WORKSPACE_BYTES (e.g. 512
 *   query vectors at context 8192 need about 5 MiB).
 * - The first call on a device looks up the array's device address (with the
 *   handle's device made current briefly, a host-side query that allocates
 *   nothing); make that first call before any stream capture.  The address is
 *   kept per device and looked up again when the device's current context is
 *   a new one (after cudaDeviceReset, which also invalidates every handle:
 *   rebuild the handles, then make the first call again before any capture).
 * - Arguments are checked (TQ_ERR_INVALID_ARG, TQ_ERR_UNSUPPORTED,
 *   TQ_ERR_WORKSPACE) before the look-up, and nothing is launched on an error.
 * - Every call on a device shares the one array, and a call leaves its
 *   contents behind; nothing in it has to start at zero, because each call
 *   writes every scratch value it reads.  Calls that overlap on the GPU
 *   (different streams, or different threads without ordering) race on the
 *   array and give wrong results: serialise them. */
tq_status tq_decode_attention_static(const tq_codebook* book, const void* q, tq_dtype dtype, int batch,
                                     int n_q_heads, int n_kv_heads, const tq_cache_view* cache,
                                     const int32_t* block_table, int max_blocks,
                                     const int32_t* context_lens, int max_context, float scale, float* out,
                                     void* stream);

/* Which decode-partials kernel tq_decode_attention / tq_decode_partials run
 * for this shape: *tensor_cores = 1 for the tensor-core kernel (fp8 sign-plane
 * GEMMs; shapes with n_q_heads / n_kv_heads in {1, 2, 4, 8} whose operands fit
 * in tensor memory), 0 for the CUDA-core kernel.  Host only; launches nothing. */
tq_status tq_decode_kernel_kind(const tq_codebook* book, int n_q_heads, int n_kv_heads, int* tensor_cores);

/* Decode attention over a context held in two caches of different bit
 * widths (the yfxerp.com page, §2.3 "dynamic bit-width scheduling": the
 * prompt's keys and values kept at 4 bits from prefill, the generated ones at
 * 3 bits): for every sequence b, the first context_lens[b] tokens of the
 * first part and the second part's context_lens[b] tokens form one context
 * under one softmax (the order within a context does not matter to decode
 * attention).  Each part has its own handle, cache, block table and lengths
 * (fields as in tq_decode_attention); the two handles must share d, qjl_m
 * and the seed, i.e. R and S (else TQ_ERR_INVALID_ARG), so that one query
 * rotation and one back-rotation serve both; their bit widths and norm
 * widths may differ.  Either part of a sequence may be empty; a sequence with
 * both empty yields a zero output row.  workspace: device scratch of
 * tq_decode_parts_workspace_bytes bytes, 256-byte aligned.  Asynchronous on
 * `stream`. */
typedef struct {
  const tq_codebook* book;
  const tq_cache_view* cache;
  const int32_t* block_table;
  int max_blocks;
  const int32_t* context_lens;
  int max_context;
} tq_context_part;
size_t tq_decode_parts_workspace_bytes(const tq_context_part* first, const tq_context_part* second, int batch,
                                       int n_q_heads);
tq_status tq_decode_attention_parts(const tq_context_part* first, const tq_context_part* second, const void* q,
                                    tq_dtype dtype, int batch, int n_q_heads, int n_kv_heads, float scale, float* out,
                                    void* workspace, size_t workspace_bytes, void* stream);

/* How tq_decode_attention / tq_decode_step run this shape (host only; launches
 * nothing): tensor_cores 1 for the tensor-core partials kernel (else the
 * CUDA-core one); merge_in_partials 1 when that kernel merges each (sequence,
 * KV head) group and writes the output itself (at most as many groups as
 * CTAs, and few segments per group at max_context), 0 when a merge launch
 * follows it; partials_ctas the CTAs of its persistent grid (0 for the
 * CUDA-core kernel); chunk_tokens the context tokens of one work item;
 * merge_ctas the CTAs of the merge launch (0 when there is none): one per
 * group, or one per query head when there are fewer groups than SMs. */
typedef struct {
  int tensor_cores;
  int merge_in_partials;
  int partials_ctas;
  int chunk_tokens;
  int merge_ctas;
} tq_decode_plan_info;
tq_status tq_decode_plan(const tq_codebook* book, int batch, int n_q_heads, int n_kv_heads, int max_context,
                         tq_decode_plan_info* info);

/* Synchronise `stream`, then return (and clear) the first device-side error
 * code recorded since the last call: 0 none, 1 slot out of range in
 * quantize-append, 2 block id out of range in decode, 3 context length out of
 * range in decode, 4 a kernel's internal wait timed out (the kernel stopped
 * early; its outputs are incomplete), 5 a merge found the partials of a
 * (sequence, KV head) missing or out of range (after a code 4 in the same
 * call, or tq_decode_finish without tq_decode_partials; those outputs are
 * zero).  Returns TQ_ERR_DEVICE when *code != 0. */
tq_status tq_get_last_device_error(const tq_codebook* book, void* stream, int* code);

/* A test aid for the bounded waits, off by default: while enabled on a
 * handle, the first CTA of the tensor-core decode kernel withholds the commit
 * of its first score MMAs, so its builders' wait for them runs out after the
 * kernels' one-second limit.  The call then ends normally with that CTA
 * stopped early (its in-flight copies and MMAs drained, its tensor memory
 * freed): tq_get_last_device_error reports code 4 and the outputs are
 * incomplete; later calls with it disabled are unaffected.  Not for use in
 * production. */
tq_status tq_debug_withhold_commit(tq_codebook* book, int enable);

/* Static description of a status code. */
const char* tq_status_string(tq_status status);

#ifdef __cplusplus
}
#endif

#endif /* TQ_H_ */
