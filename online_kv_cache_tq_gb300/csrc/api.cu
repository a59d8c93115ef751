// C ABI of the engine: handle lifetime, host-side argument checks, launches.
#include <algorithm>
#include <cmath>
#include <cstddef>
#include <cstring>
#include <new>
#include <vector>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "kernels.h"
#include "tq.h"
#include "tq_internal.h"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult res;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &res) !=
            cudaSuccess ||
        res != cudaDriverEntryPointSuccess) {
      ptr = nullptr;
    }
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }();
  return fn;
}

// 3-D map over head vectors x [n_tokens][n_kv][128] bf16: boxes of 64
// columns x 1 head x 128 tokens (128-byte swizzle), so one tile holds 128
// consecutive tokens of one head.
bool encode_tokens_bf16(CUtensorMap* map, const void* base, uint64_t n_tokens, uint64_t n_kv) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (fn == nullptr || n_tokens == 0 || n_kv == 0) return false;
  cuuint64_t dims[3] = {128, n_kv, n_tokens};
  cuuint64_t strides[2] = {128 * 2, n_kv * 128 * 2};
  cuuint32_t box[3] = {64, 1, 128};
  cuuint32_t elem[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, elem,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 2-D map over a row-major [rows][128] bf16 array, 64 x 128 boxes, 128-byte
// swizzle (the K-major operand layout of the tensor-core quantizer).
bool encode_rows_bf16(CUtensorMap* map, const void* base, uint64_t rows) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (fn == nullptr || rows == 0) return false;
  cuuint64_t dims[2] = {128, rows};
  cuuint64_t strides[1] = {128 * 2};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t elem[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, elem,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct DeviceGuard {
  int prev = -1;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (dev >= 0 && dev != prev) cudaSetDevice(dev);
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

void free_device(tq_codebook* b) {
  cudaFree(b->d_R);
  cudaFree(b->d_Rt);
  cudaFree(b->d_Spt);
  cudaFree(b->d_St);
  cudaFree(b->d_rot_tc);
  cudaFree(b->d_tables);
  cudaFree(b->d_error);
  b->d_R = b->d_Rt = b->d_Spt = b->d_St = nullptr;
  b->d_rot_tc = nullptr;
  b->d_tables = nullptr;
  b->d_error = nullptr;
}

template <typename T>
cudaError_t upload(T** dst, const std::vector<T>& src) {
  cudaError_t err = cudaMalloc(reinterpret_cast<void**>(dst), src.size() * sizeof(T));
  if (err != cudaSuccess) return err;
  return cudaMemcpy(*dst, src.data(), src.size() * sizeof(T), cudaMemcpyHostToDevice);
}

uint16_t bf16_bits(float x) {
  __nv_bfloat16 h = __float2bfloat16_rn(x);
  uint16_t out;
  std::memcpy(&out, &h, sizeof(out));
  return out;
}

float bf16_value(uint16_t bits) {
  uint32_t w = static_cast<uint32_t>(bits) << 16;
  float out;
  std::memcpy(&out, &w, sizeof(out));
  return out;
}

// Sign-plane coefficients of a codebook (see DeviceTables); returns whether
// they reproduce every level to 1e-12 relative (an odd-symmetric codebook).
bool walsh_coefficients(const std::vector<double>& levels, int bits, float* out) {
  const int count = 1 << bits;
  const int planes = 1 << (bits - 1);
  std::vector<double> coef(planes, 0.0);
  double scale = 0.0;
  for (double c : levels) scale = std::max(scale, std::fabs(c));
  for (int s = 0; s < planes; ++s) {
    const int set = tq::kWalshSets[bits - 1][s];
    for (int code = 0; code < count; ++code) {
      double sign = 1.0;
      for (int p = 0; p < bits; ++p)
        if (set & (1 << p)) sign *= ((code >> p) & 1) ? 1.0 : -1.0;
      coef[s] += levels[code] * sign;
    }
    coef[s] /= count;
  }
  bool ok = true;
  for (int code = 0; code < count; ++code) {
    double v = 0.0;
    for (int s = 0; s < planes; ++s) {
      const int set = tq::kWalshSets[bits - 1][s];
      double sign = 1.0;
      for (int p = 0; p < bits; ++p)
        if (set & (1 << p)) sign *= ((code >> p) & 1) ? 1.0 : -1.0;
      v += coef[s] * sign;
    }
    if (std::fabs(v - levels[code]) > 1e-12 * scale) ok = false;
  }
  for (int s = 0; s < 8; ++s) out[s] = s < planes ? static_cast<float>(coef[s]) : 0.f;
  return ok;
}

tq_status upload_tables(tq_codebook* b) {
  const int d = b->cfg.d;
  const int m = b->cfg.qjl_m;
  const tq::HostTables& h = b->host;
  std::vector<float> R(d * d), Rt(d * d), Spt(d * d, 0.f), St(d * d, 0.f);
  for (int i = 0; i < d; ++i) {
    for (int j = 0; j < d; ++j) {
      R[i * d + j] = static_cast<float>(h.R[i * d + j]);
      Rt[j * d + i] = static_cast<float>(h.R[i * d + j]);
    }
  }
  for (int k = 0; k < m; ++k)
    for (int j = 0; j < d; ++j) {
      Spt[j * d + k] = static_cast<float>(h.Sp[k * d + j]);
      St[j * d + k] = static_cast<float>(h.S[k * d + j]);
    }
  // bf16 hi/lo images of R and S' (row-major, [out][in]) for the tensor-core
  // quantizer: W = hi + lo with hi = bf16(W), lo = bf16(W - hi).
  std::vector<uint16_t> tc(4 * d * d, 0);
  for (int i = 0; i < d * d; ++i) {
    const float r = static_cast<float>(h.R[i]);
    tc[i] = bf16_bits(r);
    tc[d * d + i] = bf16_bits(r - bf16_value(tc[i]));
    const float s = i < m * d ? static_cast<float>(h.Sp[i]) : 0.f;
    tc[2 * d * d + i] = bf16_bits(s);
    tc[3 * d * d + i] = bf16_bits(s - bf16_value(tc[2 * d * d + i]));
  }
  tq::DeviceTables t;
  for (int i = 0; i < tq::kMaxLevels; ++i) {
    t.k_levels[i] = i < static_cast<int>(h.k_levels.size()) ? static_cast<float>(h.k_levels[i]) : 0.f;
    t.v_levels[i] = i < static_cast<int>(h.v_levels.size()) ? static_cast<float>(h.v_levels[i]) : 0.f;
    t.k_bounds[i] = i < static_cast<int>(h.k_bounds.size()) ? static_cast<float>(h.k_bounds[i]) : INFINITY;
    t.v_bounds[i] = i < static_cast<int>(h.v_bounds.size()) ? static_cast<float>(h.v_bounds[i]) : INFINITY;
  }
  b->walsh_ok = walsh_coefficients(h.k_levels, b->k_mse_bits, t.k_walsh) &&
                walsh_coefficients(h.v_levels, b->v_bits, t.v_walsh) && !b->polar;
  std::vector<tq::DeviceTables> tv(1, t);
  std::vector<int> zero(1, 0);
  cudaError_t err = upload(&b->d_R, R);
  if (err == cudaSuccess) err = upload(&b->d_Rt, Rt);
  if (err == cudaSuccess) err = upload(&b->d_Spt, Spt);
  if (err == cudaSuccess) err = upload(&b->d_St, St);
  if (err == cudaSuccess) err = upload(&b->d_rot_tc, tc);
  if (err == cudaSuccess) err = upload(&b->d_tables, tv);
  if (err == cudaSuccess) err = upload(&b->d_error, zero);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(&b->num_sms, cudaDevAttrMultiProcessorCount, b->device);
  if (err == cudaSuccess && !encode_rows_bf16(&b->w_map, b->d_rot_tc, 4 * static_cast<uint64_t>(d))) {
    err = cudaErrorInvalidValue;
  }
  if (err != cudaSuccess) {
    free_device(b);
    return err == cudaErrorMemoryAllocation ? TQ_ERR_OOM : TQ_ERR_CUDA;
  }
  return TQ_OK;
}

bool valid_device_handle(const tq_codebook* b) { return b != nullptr && b->device >= 0 && b->d_tables != nullptr; }

bool valid_cache(const tq_codebook* b, const tq_cache_view* c) {
  if (c == nullptr || c->num_blocks <= 0 || c->n_kv_heads <= 0 || c->block_size != b->cfg.block_size) return false;
  if (!c->k_codes || !c->k_norm || !c->v_codes || !c->v_norm) return false;
  if (!aligned16(c->k_codes) || !aligned16(c->k_norm) || !aligned16(c->v_codes) || !aligned16(c->v_norm)) return false;
  if (b->cfg.qjl_m > 0) {
    if (!c->k_qjl || !c->k_rnorm || !aligned16(c->k_qjl) || !aligned16(c->k_rnorm)) return false;
  }
  return true;
}

// Device address of one array inside the handle's DeviceTables.
const float* table_field(const tq_codebook* b, size_t offset) {
  return reinterpret_cast<const float*>(reinterpret_cast<const char*>(b->d_tables) + offset);
}

// Larger batches go to the tensor-core tile quantizer (bf16 x through TMA;
// fp32 x split into bf16 hi/lo by converter warps); small batches are handled
// by tq_quantize_append directly.
cudaError_t launch_quantize(const tq_codebook* b, const tq::QuantizeArgs& a, bool bf16, cudaStream_t s) {
  if (!bf16) return tq::launch_quantize_tc(a, b->w_map, b->w_map, b->num_sms, true, s);   // (x_map unused)
  CUtensorMap x_map;
  if (!encode_tokens_bf16(&x_map, a.x, static_cast<uint64_t>(a.n_tokens), static_cast<uint64_t>(a.n_kv))) {
    return cudaErrorInvalidValue;
  }
  return tq::launch_quantize_tc(a, x_map, b->w_map, b->num_sms, false, s);
}

constexpr size_t kWsAlign = 256;
size_t round_up(size_t x) { return (x + kWsAlign - 1) / kWsAlign * kWsAlign; }

int max_chunks_for(int max_context) { return (max_context + tq::kChunk - 1) / tq::kChunk; }

}  // namespace

extern "C" {

tq_status tq_codebook_build(const tq_config* cfg, int device, tq_codebook** out) {
  if (cfg == nullptr || out == nullptr) return TQ_ERR_INVALID_ARG;
  *out = nullptr;
  const bool host_only = device < 0;
  if (cfg->d <= 0 || cfg->d % 8 != 0 || cfg->d > 1024 || cfg->block_size <= 0) return TQ_ERR_INVALID_ARG;
  if (cfg->qjl_m < 0 || cfg->qjl_m % 8 != 0 || cfg->qjl_m > 1024) return TQ_ERR_INVALID_ARG;
  if (cfg->norm_bits != 0 && cfg->norm_bits != 16 && cfg->norm_bits != 32) return TQ_ERR_INVALID_ARG;
  if (cfg->codec != TQ_CODEC_TURBOQUANT && cfg->codec != TQ_CODEC_POLAR) return TQ_ERR_INVALID_ARG;
  const bool polar = cfg->codec == TQ_CODEC_POLAR;
  // PolarQuant: no codebooks and no QJL bits, float32 radii, a power-of-two
  // head dimension (the pairing levels); the handle still draws R
  if (polar && (cfg->qjl_m != 0 || cfg->norm_bits == 16 || (cfg->d & (cfg->d - 1)) != 0)) return TQ_ERR_UNSUPPORTED;
  const int k_mse = polar ? 1 : cfg->qjl_m > 0 ? cfg->k_bits - 1 : cfg->k_bits;
  const int v_mse = polar ? 1 : cfg->v_bits;
  if (k_mse < 1 || k_mse > 4 || v_mse < 1 || v_mse > 4) return TQ_ERR_UNSUPPORTED;
  if (!host_only && (cfg->d != tq::kDim || (cfg->qjl_m != 0 && cfg->qjl_m != tq::kDim))) return TQ_ERR_UNSUPPORTED;
  if (!host_only && cfg->block_size % 32 != 0) return TQ_ERR_UNSUPPORTED;
  tq_codebook* b = new (std::nothrow) tq_codebook();
  if (b == nullptr) return TQ_ERR_OOM;
  b->cfg = *cfg;
  b->device = host_only ? -1 : device;
  b->k_mse_bits = k_mse;
  b->v_bits = v_mse;
  b->norm16 = cfg->norm_bits == 16;
  b->polar = polar;
  try {
    tq::build_host_tables(cfg->d, cfg->qjl_m, cfg->seed, k_mse, v_mse, &b->host);
  } catch (const std::bad_alloc&) {
    delete b;
    return TQ_ERR_OOM;
  }
  if (!host_only) {
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess || device >= count) {
      delete b;
      return TQ_ERR_CUDA;
    }
    DeviceGuard guard(device);
    tq_status st = upload_tables(b);
    if (st != TQ_OK) {
      delete b;
      return st;
    }
  }
  *out = b;
  return TQ_OK;
}

tq_status tq_codebook_destroy(tq_codebook* book) {
  if (book == nullptr) return TQ_ERR_INVALID_ARG;
  if (book->device >= 0) {
    DeviceGuard guard(book->device);
    cudaDeviceSynchronize();
    free_device(book);
  }
  delete book;
  return TQ_OK;
}

tq_status tq_codebook_levels(const tq_codebook* book, int which, double* levels, double* bounds, int* bits) {
  if (book == nullptr || (which != 0 && which != 1)) return TQ_ERR_INVALID_ARG;
  if (book->polar) return TQ_ERR_UNSUPPORTED;     // (PolarQuant has no codebook)
  const std::vector<double>& lv = which == 0 ? book->host.k_levels : book->host.v_levels;
  const std::vector<double>& bd = which == 0 ? book->host.k_bounds : book->host.v_bounds;
  if (levels) std::memcpy(levels, lv.data(), lv.size() * sizeof(double));
  if (bounds) std::memcpy(bounds, bd.data(), bd.size() * sizeof(double));
  if (bits) *bits = which == 0 ? book->k_mse_bits : book->v_bits;
  return TQ_OK;
}

tq_status tq_codebook_matrices(const tq_codebook* book, double* R, double* S) {
  if (book == nullptr) return TQ_ERR_INVALID_ARG;
  if (R) std::memcpy(R, book->host.R.data(), book->host.R.size() * sizeof(double));
  if (S) std::memcpy(S, book->host.S.data(), book->host.S.size() * sizeof(double));
  return TQ_OK;
}

tq_status tq_cache_field_bytes(const tq_codebook* book, size_t bytes_per_item[6]) {
  if (book == nullptr || bytes_per_item == nullptr) return TQ_ERR_INVALID_ARG;
  const size_t d = static_cast<size_t>(book->cfg.d);
  const bool qjl = book->cfg.qjl_m > 0;
  if (book->polar) {
    // a 64-byte record at d = 128 (d/2 angles x 5 bits + d/2 - 1 angles x 3 bits, rounded up to 16 bytes)
    const size_t rec = ((d / 2 * 5 + (d / 2 - 1) * 3 + 127) / 128) * 16;
    const size_t items[6] = {rec, 0, 4, 0, rec, 4};
    std::memcpy(bytes_per_item, items, sizeof(items));
    return TQ_OK;
  }
  bytes_per_item[0] = book->k_mse_bits * d / 8;
  bytes_per_item[1] = qjl ? static_cast<size_t>(book->cfg.qjl_m) / 8 : 0;
  const size_t nb = book->norm16 ? 2 : 4;
  bytes_per_item[2] = nb;
  bytes_per_item[3] = qjl ? nb : 0;
  bytes_per_item[4] = book->v_bits * d / 8;
  bytes_per_item[5] = nb;
  return TQ_OK;
}

}  // extern "C"

namespace {

// Validate an append and fill the launch arguments of its keys and values.
tq_status append_args(const tq_codebook* book, const void* k, const void* v, tq_dtype dtype, int n_tokens,
                      int n_kv_heads, const int64_t* slot_mapping, const tq_cache_view* cache, tq::QuantizeArgs* ka,
                      tq::QuantizeArgs* va) {
  if (!valid_device_handle(book)) return TQ_ERR_INVALID_ARG;
  if (dtype != TQ_BF16 && dtype != TQ_FP32) return TQ_ERR_INVALID_ARG;
  if (n_tokens < 0 || n_kv_heads <= 0 || !valid_cache(book, cache) || cache->n_kv_heads != n_kv_heads) {
    return TQ_ERR_INVALID_ARG;
  }
  if (n_tokens == 0) return TQ_OK;
  if (k == nullptr && v == nullptr) return TQ_ERR_INVALID_ARG;
  if ((k && !aligned16(k)) || (v && !aligned16(v))) return TQ_ERR_INVALID_ARG;
  if (static_cast<long long>(n_tokens) * n_kv_heads > (1ll << 31) - 1) return TQ_ERR_INVALID_ARG;
  tq::QuantizeArgs base{};
  base.n_vec = n_tokens * n_kv_heads;
  base.n_tokens = n_tokens;
  base.n_kv = n_kv_heads;
  base.slots = slot_mapping;
  base.num_blocks = cache->num_blocks;
  base.block_size = cache->block_size;
  base.Rt = book->d_Rt;
  base.Spt = book->d_Spt;
  base.error = book->d_error;
  base.norm16 = book->norm16;
  *ka = base;
  *va = base;
  ka->x = k;
  ka->codes = static_cast<uint8_t*>(cache->k_codes);
  ka->qjl = book->cfg.qjl_m > 0 ? static_cast<uint8_t*>(cache->k_qjl) : nullptr;
  ka->norm = cache->k_norm;
  ka->rnorm = book->cfg.qjl_m > 0 ? cache->k_rnorm : nullptr;
  ka->bits = book->polar ? 0 : book->k_mse_bits;   // (0: PolarQuant records)
  ka->transposed = false;
  ka->levels = table_field(book, offsetof(tq::DeviceTables, k_levels));
  ka->bounds = table_field(book, offsetof(tq::DeviceTables, k_bounds));
  va->x = v;
  va->codes = static_cast<uint8_t*>(cache->v_codes);
  va->qjl = nullptr;
  va->norm = cache->v_norm;
  va->rnorm = nullptr;
  va->bits = book->polar ? 0 : book->v_bits;
  va->transposed = !book->polar;                  // (PolarQuant value records are token-major)
  va->levels = table_field(book, offsetof(tq::DeviceTables, v_levels));
  va->bounds = table_field(book, offsetof(tq::DeviceTables, v_bounds));
  return TQ_OK;
}

// Launch a validated append (either tensor may be absent).
tq_status run_append(const tq_codebook* book, const void* k, const void* v, const tq::QuantizeArgs& ka,
                     const tq::QuantizeArgs& va, bool bf16, cudaStream_t s) {
  if (book->polar && ka.n_vec <= tq::kSmallQuantize) {
    // a decode step's few vectors: the CUDA-core PolarQuant kernel (the tile
    // quantizer's PolarQuant epilogue takes larger appends)
    if (k && tq::launch_polar_quantize(ka, bf16, s) != cudaSuccess) return TQ_ERR_CUDA;
    if (v && tq::launch_polar_quantize(va, bf16, s) != cudaSuccess) return TQ_ERR_CUDA;
    return TQ_OK;
  }
  if (ka.n_vec <= tq::kSmallQuantize) {
    // a decode step: keys and values in one launch, one CTA per vector
    return tq::launch_quantize_small(k ? &ka : nullptr, v ? &va : nullptr, bf16, s) == cudaSuccess ? TQ_OK
                                                                                                    : TQ_ERR_CUDA;
  }
  if (k && launch_quantize(book, ka, bf16, s) != cudaSuccess) return TQ_ERR_CUDA;
  if (v && launch_quantize(book, va, bf16, s) != cudaSuccess) return TQ_ERR_CUDA;
  return TQ_OK;
}

}  // namespace

extern "C" {

tq_status tq_quantize_append(const tq_codebook* book, const void* k, const void* v, tq_dtype dtype,
                             int n_tokens, int n_kv_heads, const int64_t* slot_mapping,
                             const tq_cache_view* cache, void* stream) {
  if (n_tokens > 0 && slot_mapping == nullptr) return TQ_ERR_INVALID_ARG;
  tq::QuantizeArgs ka{}, va{};
  const tq_status st = append_args(book, k, v, dtype, n_tokens, n_kv_heads, slot_mapping, cache, &ka, &va);
  if (st != TQ_OK || n_tokens == 0) return st;
  return run_append(book, k, v, ka, va, dtype == TQ_BF16, static_cast<cudaStream_t>(stream));
}

tq_status tq_reconstruction_error(const tq_codebook* book, const void* x, tq_dtype dtype, int which, int n_tokens,
                                  int n_kv_heads, const int64_t* slot_mapping, const tq_cache_view* cache,
                                  double* stats, void* stream) {
  if (which != 0 && which != 1) return TQ_ERR_INVALID_ARG;
  if (book != nullptr && book->polar) return TQ_ERR_UNSUPPORTED;   // (stage-1 reconstructions of Lloyd-Max codes)
  if (n_tokens > 0 && (slot_mapping == nullptr || x == nullptr || stats == nullptr)) return TQ_ERR_INVALID_ARG;
  if (stats != nullptr && (reinterpret_cast<uintptr_t>(stats) & 7u) != 0) return TQ_ERR_INVALID_ARG;
  tq::QuantizeArgs ka{}, va{};
  const tq_status st = append_args(book, which == 0 ? x : nullptr, which == 1 ? x : nullptr, dtype, n_tokens,
                                   n_kv_heads, slot_mapping, cache, &ka, &va);
  if (st != TQ_OK || n_tokens == 0) return st;
  return tq::launch_monitor(which == 0 ? ka : va, dtype == TQ_BF16, stats, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? TQ_OK
             : TQ_ERR_CUDA;
}

}  // extern "C"

namespace {

// Per query head: the tensor-core score operand pieces (only for codebooks
// the tensor-core decode can take).
size_t bk_bytes(const tq_codebook* book) {
  if (!book->walsh_ok || book->k_mse_bits < 1 || book->k_mse_bits > 4) return 0;
  return static_cast<size_t>(tq::bk_head_bytes(book->k_mse_bits, book->cfg.qjl_m > 0));
}

// Decode workspace regions (byte offsets, each 256-byte aligned): rotated and
// projected queries, split-K partial entries, tensor-core score operands,
// per-group segment tickets and per-query-head segment records.
struct DecodeLayout {
  size_t q, part, bk, ticket, seg, total;
};

DecodeLayout decode_layout(const tq_codebook* book, int batch, int n_q_heads, int max_context) {
  const size_t vecs = static_cast<size_t>(batch) * n_q_heads;
  DecodeLayout l;
  l.q = 0;
  l.part = l.q + round_up(vecs * 2 * tq::kDim * sizeof(float));
  const long long entries = tq::partial_entries(static_cast<long long>(vecs), max_chunks_for(max_context),
                                                book->num_sms > 0 ? book->num_sms : 160);
  l.bk = l.part + round_up(static_cast<size_t>(entries) * tq::kPartStride * sizeof(float));
  l.ticket = l.bk + round_up(vecs * bk_bytes(book));
  l.seg = l.ticket + round_up(vecs * sizeof(int));
  l.total = l.seg + round_up(vecs * sizeof(tq::SegInfo));
  return l;
}

}  // namespace

extern "C" {

size_t tq_decode_workspace_bytes(const tq_codebook* book, int batch, int n_q_heads, int max_context) {
  if (book == nullptr || batch <= 0 || n_q_heads <= 0 || max_context < 0) return 0;
  const DecodeLayout l = decode_layout(book, batch, n_q_heads, max_context);
  return l.total;
}

}  // extern "C"

namespace {

enum Stage { kPrepare = 1, kPartials = 2, kFinish = 4 };

// Validate the arguments a decode stage uses and fill the launch arguments.
tq_status decode_args(const tq_codebook* book, int stages, const void* q, tq_dtype dtype, int batch,
                      int n_q_heads, int n_kv_heads, const tq_cache_view* cache, const int32_t* block_table,
                      int max_blocks, const int32_t* context_lens, int max_context, float scale, float* out,
                      void* workspace, size_t workspace_bytes, tq::DecodeArgs* a) {
  if (!valid_device_handle(book)) return TQ_ERR_INVALID_ARG;
  if (batch < 0 || n_q_heads <= 0 || max_context < 0) return TQ_ERR_INVALID_ARG;
  *a = tq::DecodeArgs{};
  if (stages & kPrepare) {
    if (dtype != TQ_BF16 && dtype != TQ_FP32) return TQ_ERR_INVALID_ARG;
    if (batch > 0 && (q == nullptr || !aligned16(q))) return TQ_ERR_INVALID_ARG;
  }
  if (stages & kPartials) {
    if (n_kv_heads <= 0 || n_q_heads % n_kv_heads != 0) return TQ_ERR_INVALID_ARG;
    if (!valid_cache(book, cache) || cache->n_kv_heads != n_kv_heads) return TQ_ERR_INVALID_ARG;
    if (!(scale >= 0.f) || !std::isfinite(scale)) return TQ_ERR_INVALID_ARG;
    const int group = n_q_heads / n_kv_heads;
    if (group != 1 && group != 2 && group != 4 && group != 8) return TQ_ERR_UNSUPPORTED;
    if (block_table == nullptr && static_cast<long long>(batch) * max_blocks > cache->num_blocks) {
      return TQ_ERR_INVALID_ARG;
    }
    // work items (sequence, KV head, chunk) are numbered in int
    if (static_cast<long long>(batch) * n_kv_heads * max_chunks_for(max_context) >= (1ll << 31)) {
      return TQ_ERR_INVALID_ARG;
    }
  }
  if (stages & (kPartials | kFinish)) {
    if (max_blocks <= 0) return TQ_ERR_INVALID_ARG;
    if (batch > 0 && context_lens == nullptr) return TQ_ERR_INVALID_ARG;
  }
  if ((stages & kFinish) && batch > 0 && (out == nullptr || !aligned16(out))) return TQ_ERR_INVALID_ARG;
  if (batch == 0) return TQ_OK;
  const size_t need = tq_decode_workspace_bytes(book, batch, n_q_heads, max_context);
  if (workspace == nullptr || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) {
    return TQ_ERR_WORKSPACE;
  }
  a->q = q;
  a->batch = batch;
  a->n_q = n_q_heads;
  if (stages & kPartials) {
    a->n_kv = n_kv_heads;
    a->group = n_q_heads / n_kv_heads;
    a->k_codes = static_cast<const uint8_t*>(cache->k_codes);
    a->k_qjl = book->cfg.qjl_m > 0 ? static_cast<const uint8_t*>(cache->k_qjl) : nullptr;
    a->k_norm = cache->k_norm;
    a->k_rnorm = book->cfg.qjl_m > 0 ? cache->k_rnorm : nullptr;
    a->v_codes = static_cast<const uint8_t*>(cache->v_codes);
    a->v_norm = cache->v_norm;
    a->norm16 = book->norm16;
    a->num_blocks = cache->num_blocks;
  }
  a->block_size = book->cfg.block_size;
  a->k_bits = book->k_mse_bits;
  a->v_bits = book->v_bits;
  a->qjl_m = book->cfg.qjl_m;
  a->block_table = block_table;
  a->max_blocks = max_blocks;
  a->context_lens = context_lens;
  a->max_context = max_context;
  a->scale = scale > 0.f ? scale : 1.0f / std::sqrt(static_cast<float>(book->cfg.d));
  a->qjl_coef = book->cfg.qjl_m > 0 ? static_cast<float>(std::sqrt(M_PI / 2.0) / book->cfg.qjl_m) : 0.f;
  a->out = out;
  const DecodeLayout l = decode_layout(book, batch, n_q_heads, max_context);
  char* ws = static_cast<char*>(workspace);
  a->ws_q = reinterpret_cast<float*>(ws + l.q);
  a->ws_part = reinterpret_cast<float*>(ws + l.part);
  a->max_chunks = max_chunks_for(max_context);
  const size_t bk = bk_bytes(book);
  a->ws_bk = bk == 0 ? nullptr : reinterpret_cast<uint8_t*>(ws + l.bk);
  a->ws_ticket = reinterpret_cast<int*>(ws + l.ticket);
  a->ws_seg = reinterpret_cast<tq::SegInfo*>(ws + l.seg);
  a->part_cap = static_cast<long long>((l.bk - l.part) / (tq::kPartStride * sizeof(float)));
  a->debug_withhold = book->debug_withhold;
  a->bk_stride = static_cast<int>(bk);
  a->R = book->d_R;
  a->Rt = book->d_Rt;
  a->Spt = book->d_Spt;
  a->St = book->d_St;
  a->tables = book->d_tables;
  a->error = book->d_error;
  a->num_sms = book->num_sms;
  a->polar = book->polar;
  // with an output, the tensor-core path either merges in the partials kernel
  // (few groups per CTA) or in a dependent merge launch (see launch_partials_and_merge)
  a->merge_in_partials = (stages & kPartials) && out != nullptr && tq::tc_decode_supported(*a, book->walsh_ok) &&
                         tq::tc_merge_in_partials(*a);
  return TQ_OK;
}

tq_status launched(cudaError_t err) { return err == cudaSuccess ? TQ_OK : TQ_ERR_CUDA; }

}  // namespace

namespace tq {

tq_status check_decode_call(const tq_codebook* book, const void* q, tq_dtype dtype, int batch, int n_q_heads,
                            int n_kv_heads, const tq_cache_view* cache, const int32_t* block_table, int max_blocks,
                            const int32_t* context_lens, int max_context, float scale, float* out,
                            size_t workspace_bytes) {
  DecodeArgs a;
  // any non-null 256-byte aligned address stands for the workspace: only its
  // size and alignment are checked
  return decode_args(book, kPrepare | kPartials | kFinish, q, dtype, batch, n_q_heads, n_kv_heads, cache,
                     block_table, max_blocks, context_lens, max_context, scale, out, reinterpret_cast<void*>(256),
                     workspace_bytes, &a);
}

}  // namespace tq

namespace {

// Partials and the merge into `out`: the tensor-core kernel merges in place
// (the CTA that finishes a (sequence, KV head) group's last segment merges
// it); after the SIMT kernel the merge kernel runs.  early: the previous
// launch on the stream is a decode step's fused append + query preparation
// and the tensor-core kernel may overlap it (programmatic dependent launch).
cudaError_t launch_partials_and_merge(const tq_codebook* book, const tq::DecodeArgs& a, cudaStream_t s,
                                      bool early = false) {
  if (a.merge_in_partials) return tq::launch_decode_partials_tc(a, s, early);
  if (tq::tc_decode_supported(a, book->walsh_ok)) {
    const cudaError_t err = tq::launch_decode_partials_tc(a, s, early);
    return err == cudaSuccess ? tq::launch_merge_groups_tc(a, s) : err;
  }
  const cudaError_t err = tq::launch_decode_partials(a, s);
  return err == cudaSuccess ? tq::launch_decode_finish(a, s) : err;
}

// Partials only (the staged call without an output): tensor-core kernel where
// supported, SIMT otherwise.
cudaError_t launch_partials(const tq_codebook* book, const tq::DecodeArgs& a, cudaStream_t s) {
  if (tq::tc_decode_supported(a, book->walsh_ok)) return tq::launch_decode_partials_tc(a, s, false);
  return tq::launch_decode_partials(a, s);
}

}  // namespace

extern "C" {

tq_status tq_decode_attention(const tq_codebook* book, const void* q, tq_dtype dtype, int batch,
                              int n_q_heads, int n_kv_heads, const tq_cache_view* cache,
                              const int32_t* block_table, int max_blocks, const int32_t* context_lens,
                              int max_context, float scale, float* out, void* workspace,
                              size_t workspace_bytes, void* stream) {
  tq::DecodeArgs a;
  tq_status st = decode_args(book, kPrepare | kPartials | kFinish, q, dtype, batch, n_q_heads, n_kv_heads, cache,
                             block_table, max_blocks, context_lens, max_context, scale, out, workspace,
                             workspace_bytes, &a);
  if (st != TQ_OK || batch == 0) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st = launched(tq::launch_decode_prepare(a, dtype == TQ_BF16, s));
  if (st == TQ_OK) st = launched(launch_partials_and_merge(book, a, s));
  return st;
}

}  // extern "C"

namespace {

// Arguments of a decode step: the append of one key and value per sequence
// at position context_lens[b] - 1 (slots derived on the device from the
// block table) and the decode stages.
tq_status step_args(const tq_codebook* book, const void* k_new, const void* v_new, tq_dtype kv_dtype, const void* q,
                    tq_dtype q_dtype, int batch, int n_q_heads, int n_kv_heads, const tq_cache_view* cache,
                    const int32_t* block_table, int max_blocks, const int32_t* context_lens, int max_context,
                    float scale, float* out, void* workspace, size_t workspace_bytes, int stages,
                    tq::QuantizeArgs* ka, tq::QuantizeArgs* va, tq::DecodeArgs* a) {
  if (batch > 0 && (k_new == nullptr || v_new == nullptr)) return TQ_ERR_INVALID_ARG;
  tq_status st = append_args(book, k_new, v_new, kv_dtype, batch, n_kv_heads, nullptr, cache, ka, va);
  if (st != TQ_OK) return st;
  st = decode_args(book, stages, q, q_dtype, batch, n_q_heads, n_kv_heads, cache, block_table, max_blocks,
                   context_lens, max_context, scale, out, workspace, workspace_bytes, a);
  if (st != TQ_OK) return st;
  if (batch > 0 && (max_blocks <= 0 || context_lens == nullptr)) return TQ_ERR_INVALID_ARG;
  for (tq::QuantizeArgs* x : {ka, va}) {
    x->step_block_table = block_table;
    x->step_context_lens = context_lens;
    x->step_max_blocks = max_blocks;
  }
  return TQ_OK;
}

// Launch the append and query preparation of a validated step.
tq_status run_step_prepare(const tq_codebook* book, const void* k_new, const void* v_new, bool kv_bf16,
                           const tq::QuantizeArgs& ka, const tq::QuantizeArgs& va, const tq::DecodeArgs& a,
                           bool q_bf16, cudaStream_t s, bool* fused) {
  *fused = ka.n_vec <= tq::kSmallQuantize && !book->polar;
  if (*fused) return launched(tq::launch_step_prep(ka, va, kv_bf16, a, q_bf16, s));
  tq_status st = run_append(book, k_new, v_new, ka, va, kv_bf16, s);
  if (st == TQ_OK) st = launched(tq::launch_decode_prepare(a, q_bf16, s));
  return st;
}

}  // namespace

extern "C" {

tq_status tq_decode_step_prepare(const tq_codebook* book, const void* k_new, const void* v_new,
                                 tq_dtype kv_dtype, const void* q, tq_dtype q_dtype, int batch, int n_q_heads,
                                 int n_kv_heads, const tq_cache_view* cache, const int32_t* block_table,
                                 int max_blocks, const int32_t* context_lens, int max_context, void* workspace,
                                 size_t workspace_bytes, void* stream) {
  tq::QuantizeArgs ka{}, va{};
  tq::DecodeArgs a;
  tq_status st = step_args(book, k_new, v_new, kv_dtype, q, q_dtype, batch, n_q_heads, n_kv_heads, cache,
                           block_table, max_blocks, context_lens, max_context, 0.f, nullptr, workspace,
                           workspace_bytes, kPrepare | kPartials, &ka, &va, &a);
  if (st != TQ_OK || batch == 0) return st;
  bool fused;
  return run_step_prepare(book, k_new, v_new, kv_dtype == TQ_BF16, ka, va, a, q_dtype == TQ_BF16,
                          static_cast<cudaStream_t>(stream), &fused);
}

tq_status tq_decode_step(const tq_codebook* book, const void* k_new, const void* v_new, tq_dtype kv_dtype,
                         const void* q, tq_dtype q_dtype, int batch, int n_q_heads, int n_kv_heads,
                         const tq_cache_view* cache, const int32_t* block_table, int max_blocks,
                         const int32_t* context_lens, int max_context, float scale, float* out, void* workspace,
                         size_t workspace_bytes, void* stream) {
  tq::QuantizeArgs ka{}, va{};
  tq::DecodeArgs a;
  tq_status st = step_args(book, k_new, v_new, kv_dtype, q, q_dtype, batch, n_q_heads, n_kv_heads, cache,
                           block_table, max_blocks, context_lens, max_context, scale, out, workspace,
                           workspace_bytes, kPrepare | kPartials | kFinish, &ka, &va, &a);
  if (st != TQ_OK || batch == 0) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  bool fused;
  st = run_step_prepare(book, k_new, v_new, kv_dtype == TQ_BF16, ka, va, a, q_dtype == TQ_BF16, s, &fused);
  // after the fused launch, the partials kernel starts early: only the chunk
  // holding the appended token, and the query operands, wait for it
  if (st == TQ_OK) st = launched(launch_partials_and_merge(book, a, s, fused));
  return st;
}

}  // extern "C"

namespace {

// Staging layout of tq_decode_step_host: k_new, v_new, q, context_lens, out.
struct HostStaging {
  size_t k, v, q, ctx, out, total;
};

bool host_staging(int batch, int n_q_heads, int n_kv_heads, tq_dtype kv_dtype, tq_dtype q_dtype, HostStaging* h) {
  if (batch < 0 || n_q_heads <= 0 || n_kv_heads <= 0) return false;
  if ((kv_dtype != TQ_BF16 && kv_dtype != TQ_FP32) || (q_dtype != TQ_BF16 && q_dtype != TQ_FP32)) return false;
  const size_t kv_elem = kv_dtype == TQ_BF16 ? 2 : 4, q_elem = q_dtype == TQ_BF16 ? 2 : 4;
  h->k = h->v = static_cast<size_t>(batch) * n_kv_heads * tq::kDim * kv_elem;
  h->q = static_cast<size_t>(batch) * n_q_heads * tq::kDim * q_elem;
  h->ctx = static_cast<size_t>(batch) * sizeof(int32_t);
  h->out = static_cast<size_t>(batch) * n_q_heads * tq::kDim * sizeof(float);
  h->total = round_up(h->k) + round_up(h->v) + round_up(h->q) + round_up(h->ctx) + round_up(h->out);
  return true;
}

}  // namespace

extern "C" {

size_t tq_decode_step_host_workspace_bytes(const tq_codebook* book, int batch, int n_q_heads, int n_kv_heads,
                                           int max_context, tq_dtype kv_dtype, tq_dtype q_dtype) {
  HostStaging h;
  if (!host_staging(batch, n_q_heads, n_kv_heads, kv_dtype, q_dtype, &h)) return 0;
  const size_t ws = tq_decode_workspace_bytes(book, batch, n_q_heads, max_context);
  return ws == 0 ? 0 : h.total + ws;
}

tq_status tq_decode_step_host(const tq_codebook* book, const void* k_new_h, const void* v_new_h,
                              tq_dtype kv_dtype, const void* q_h, tq_dtype q_dtype, int batch, int n_q_heads,
                              int n_kv_heads, const tq_cache_view* cache, const int32_t* block_table,
                              int max_blocks, const int32_t* context_lens_h, int max_context, float scale,
                              float* out_h, void* workspace, size_t workspace_bytes, void* stream) {
  HostStaging h;
  if (book == nullptr || !host_staging(batch, n_q_heads, n_kv_heads, kv_dtype, q_dtype, &h)) {
    return TQ_ERR_INVALID_ARG;
  }
  if (batch == 0) return TQ_OK;
  if (k_new_h == nullptr || v_new_h == nullptr || q_h == nullptr || context_lens_h == nullptr || out_h == nullptr) {
    return TQ_ERR_INVALID_ARG;
  }
  if (workspace == nullptr || workspace_bytes < h.total) return TQ_ERR_WORKSPACE;
  char* base = static_cast<char*>(workspace);
  void* k_d = base;
  void* v_d = base + round_up(h.k);
  void* q_d = base + round_up(h.k) + round_up(h.v);
  int32_t* ctx_d = reinterpret_cast<int32_t*>(base + round_up(h.k) + round_up(h.v) + round_up(h.q));
  float* out_d = reinterpret_cast<float*>(base + round_up(h.k) + round_up(h.v) + round_up(h.q) + round_up(h.ctx));
  // every check of the step (handle, shapes, cache, workspace) before a copy is queued
  {
    tq::QuantizeArgs ka{}, va{};
    tq::DecodeArgs a;
    const tq_status chk = step_args(book, k_d, v_d, kv_dtype, q_d, q_dtype, batch, n_q_heads, n_kv_heads, cache,
                                    block_table, max_blocks, ctx_d, max_context, scale, out_d, base + h.total,
                                    workspace_bytes - h.total, kPrepare | kPartials | kFinish, &ka, &va, &a);
    if (chk != TQ_OK) return chk;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t err = cudaMemcpyAsync(k_d, k_new_h, h.k, cudaMemcpyHostToDevice, s);
  if (err == cudaSuccess) err = cudaMemcpyAsync(v_d, v_new_h, h.v, cudaMemcpyHostToDevice, s);
  if (err == cudaSuccess) err = cudaMemcpyAsync(q_d, q_h, h.q, cudaMemcpyHostToDevice, s);
  if (err == cudaSuccess) err = cudaMemcpyAsync(ctx_d, context_lens_h, h.ctx, cudaMemcpyHostToDevice, s);
  if (err != cudaSuccess) return TQ_ERR_CUDA;
  const tq_status st = tq_decode_step(book, k_d, v_d, kv_dtype, q_d, q_dtype, batch, n_q_heads, n_kv_heads, cache,
                                      block_table, max_blocks, ctx_d, max_context, scale, out_d, base + h.total,
                                      workspace_bytes - h.total, stream);
  if (st != TQ_OK) return st;
  return cudaMemcpyAsync(out_h, out_d, h.out, cudaMemcpyDeviceToHost, s) == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

tq_status tq_decode_prepare(const tq_codebook* book, const void* q, tq_dtype dtype, int batch, int n_q_heads,
                            int max_context, void* workspace, size_t workspace_bytes, void* stream) {
  tq::DecodeArgs a;
  tq_status st = decode_args(book, kPrepare, q, dtype, batch, n_q_heads, 0, nullptr, nullptr, 1, nullptr,
                             max_context, 0.f, nullptr, workspace, workspace_bytes, &a);
  if (st != TQ_OK || batch == 0) return st;
  return launched(tq::launch_decode_prepare(a, dtype == TQ_BF16, static_cast<cudaStream_t>(stream)));
}

tq_status tq_decode_partials(const tq_codebook* book, int batch, int n_q_heads, int n_kv_heads,
                             const tq_cache_view* cache, const int32_t* block_table, int max_blocks,
                             const int32_t* context_lens, int max_context, float scale, float* out,
                             void* workspace, size_t workspace_bytes, void* stream) {
  tq::DecodeArgs a;
  const int stages = out != nullptr ? kPartials | kFinish : kPartials;
  tq_status st = decode_args(book, stages, nullptr, TQ_FP32, batch, n_q_heads, n_kv_heads, cache, block_table,
                             max_blocks, context_lens, max_context, scale, out, workspace, workspace_bytes, &a);
  if (st != TQ_OK || batch == 0) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (out != nullptr) return launched(launch_partials_and_merge(book, a, s));
  return launched(launch_partials(book, a, s));
}

tq_status tq_decode_finish(const tq_codebook* book, int batch, int n_q_heads, const int32_t* context_lens,
                           int max_context, int max_blocks, float* out, void* workspace, size_t workspace_bytes,
                           void* stream) {
  tq::DecodeArgs a;
  tq_status st = decode_args(book, kFinish, nullptr, TQ_FP32, batch, n_q_heads, 0, nullptr, nullptr, max_blocks,
                             context_lens, max_context, 0.f, out, workspace, workspace_bytes, &a);
  if (st != TQ_OK || batch == 0) return st;
  return launched(tq::launch_decode_finish(a, static_cast<cudaStream_t>(stream)));
}

tq_status tq_decode_kernel_kind(const tq_codebook* book, int n_q_heads, int n_kv_heads, int* tensor_cores) {
  if (!valid_device_handle(book) || tensor_cores == nullptr || n_q_heads <= 0 || n_kv_heads <= 0 ||
      n_q_heads % n_kv_heads != 0) {
    return TQ_ERR_INVALID_ARG;
  }
  tq::DecodeArgs a{};
  a.group = n_q_heads / n_kv_heads;
  a.block_size = book->cfg.block_size;
  a.k_bits = book->k_mse_bits;
  a.v_bits = book->v_bits;
  a.k_qjl = book->cfg.qjl_m > 0 ? reinterpret_cast<const uint8_t*>(1) : nullptr;
  a.ws_bk = bk_bytes(book) > 0 ? reinterpret_cast<uint8_t*>(1) : nullptr;   // null checks only
  *tensor_cores = tq::tc_decode_supported(a, book->walsh_ok) ? 1 : 0;
  return TQ_OK;
}

size_t tq_decode_parts_workspace_bytes(const tq_context_part* first, const tq_context_part* second, int batch,
                                       int n_q_heads) {
  if (first == nullptr || second == nullptr || first->book == nullptr || second->book == nullptr) return 0;
  const size_t w1 = tq_decode_workspace_bytes(first->book, batch, n_q_heads, first->max_context);
  const size_t w2 = tq_decode_workspace_bytes(second->book, batch, n_q_heads, second->max_context);
  return w1 == 0 || w2 == 0 ? 0 : round_up(w1) + w2;
}

tq_status tq_decode_attention_parts(const tq_context_part* first, const tq_context_part* second, const void* q,
                                    tq_dtype dtype, int batch, int n_q_heads, int n_kv_heads, float scale, float* out,
                                    void* workspace, size_t workspace_bytes, void* stream) {
  if (first == nullptr || second == nullptr || !valid_device_handle(first->book) ||
      !valid_device_handle(second->book)) {
    return TQ_ERR_INVALID_ARG;
  }
  const tq_codebook* b1 = first->book;
  const tq_codebook* b2 = second->book;
  // one rotation and one projection for both parts: the parts' rotated-space
  // partials merge, and one back-rotation serves both
  if (b1->device != b2->device || b1->cfg.d != b2->cfg.d || b1->cfg.qjl_m != b2->cfg.qjl_m ||
      b1->host.R != b2->host.R || b1->host.S != b2->host.S) {
    return TQ_ERR_INVALID_ARG;
  }
  if (batch > 0 && (out == nullptr || !aligned16(out))) return TQ_ERR_INVALID_ARG;
  const size_t w1 = tq_decode_workspace_bytes(b1, batch, n_q_heads, first->max_context);
  const size_t w2 = tq_decode_workspace_bytes(b2, batch, n_q_heads, second->max_context);
  if (batch > 0 && (workspace == nullptr || workspace_bytes < round_up(w1) + w2)) return TQ_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  tq::DecodeArgs a1, a2;
  tq_status st = decode_args(b1, kPrepare | kPartials, q, dtype, batch, n_q_heads, n_kv_heads, first->cache,
                             first->block_table, first->max_blocks, first->context_lens, first->max_context, scale,
                             out, ws, w1, &a1);
  if (st == TQ_OK)
    st = decode_args(b2, kPrepare | kPartials, q, dtype, batch, n_q_heads, n_kv_heads, second->cache,
                     second->block_table, second->max_blocks, second->context_lens, second->max_context, scale, out,
                     batch > 0 ? ws + round_up(w1) : nullptr, w2, &a2);
  if (st != TQ_OK || batch == 0) return st;
  a1.merge_in_partials = a2.merge_in_partials = 0;   // the parts merge together below
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool bf16 = dtype == TQ_BF16;
  st = launched(tq::launch_decode_prepare(a1, bf16, s));
  if (st == TQ_OK) st = launched(launch_partials(b1, a1, s));
  if (st == TQ_OK) st = launched(tq::launch_decode_prepare(a2, bf16, s));
  if (st == TQ_OK) st = launched(launch_partials(b2, a2, s));
  if (st == TQ_OK) st = launched(tq::launch_decode_finish_parts(a1, a2, s));
  return st;
}

tq_status tq_decode_plan(const tq_codebook* book, int batch, int n_q_heads, int n_kv_heads, int max_context,
                         tq_decode_plan_info* info) {
  if (!valid_device_handle(book) || info == nullptr || batch <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 ||
      n_q_heads % n_kv_heads != 0 || max_context < 0) {
    return TQ_ERR_INVALID_ARG;
  }
  tq::DecodeArgs a{};
  a.batch = batch;
  a.n_q = n_q_heads;
  a.n_kv = n_kv_heads;
  a.group = n_q_heads / n_kv_heads;
  a.block_size = book->cfg.block_size;
  a.k_bits = book->k_mse_bits;
  a.v_bits = book->v_bits;
  a.max_context = max_context;
  a.num_sms = book->num_sms;
  a.k_qjl = book->cfg.qjl_m > 0 ? reinterpret_cast<const uint8_t*>(1) : nullptr;
  a.ws_bk = bk_bytes(book) > 0 ? reinterpret_cast<uint8_t*>(1) : nullptr;   // null checks only
  const bool tc = tq::tc_decode_supported(a, book->walsh_ok);
  info->tensor_cores = tc ? 1 : 0;
  info->merge_in_partials = tc && tq::tc_merge_in_partials(a) ? 1 : 0;
  info->partials_ctas = tc ? tq::tc_grid(a) : 0;
  info->chunk_tokens = tc ? tq::tc_chunk(a) : tq::kChunk;
  const int n_vec = batch * n_q_heads;
  info->merge_ctas = !tc ? (n_vec + 1) / 2
                         : info->merge_in_partials ? 0 : tq::tc_merge_per_head(a) ? n_vec : batch * n_kv_heads;
  return TQ_OK;
}

tq_status tq_debug_withhold_commit(tq_codebook* book, int enable) {
  if (!valid_device_handle(book)) return TQ_ERR_INVALID_ARG;
  book->debug_withhold = enable ? 1 : 0;
  return TQ_OK;
}

tq_status tq_get_last_device_error(const tq_codebook* book, void* stream, int* code) {
  if (!valid_device_handle(book) || code == nullptr) return TQ_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return TQ_ERR_CUDA;
  int value = 0;
  if (cudaMemcpy(&value, book->d_error, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return TQ_ERR_CUDA;
  if (cudaMemset(book->d_error, 0, sizeof(int)) != cudaSuccess) return TQ_ERR_CUDA;
  *code = value;
  return value == 0 ? TQ_OK : TQ_ERR_DEVICE;
}

const char* tq_status_string(tq_status status) {
  switch (status) {
    case TQ_OK: return "ok";
    case TQ_ERR_INVALID_ARG: return "invalid argument";
    case TQ_ERR_UNSUPPORTED: return "unsupported configuration";
    case TQ_ERR_CUDA: return "CUDA error";
    case TQ_ERR_OOM: return "out of memory";
    case TQ_ERR_WORKSPACE: return "workspace missing or too small";
    case TQ_ERR_DEVICE: return "device-side error recorded";
  }
  return "unknown status";
}

}  // extern "C"
