// Decode attention without any device allocation: the split-K scratch lives in
// a fixed-size array compiled into the library instead of a caller-supplied
// workspace.
//
// Some callers cannot allocate device memory when they decode: serving
// runtimes that reserve the whole GPU through their own memory pool at start
// and refuse any other allocation, and latency-critical loops where a
// cudaMalloc (which may synchronise the device) must never happen.  They call
// tq_decode_attention_static instead of tq_decode_attention and pass only
// their inputs and outputs.
#include <cuda_runtime.h>

#include <mutex>

#include "tq.h"
#include "tq_internal.h"

namespace {

constexpr int kMaxDevices = 64;

// Scratch shared by every call on a device; each GPU that loads the library
// holds it until the process exits.
static __device__ __align__(256) unsigned char decode_scratch[TQ_STATIC_WORKSPACE_BYTES];

void* scratch_ptr[kMaxDevices] = {};
std::mutex scratch_mutex;

// Device address of decode_scratch on `device`, looked up once per device
// with that device current (the host-side name is only a stand-in).
void* scratch_address(int device) {
  if (device < 0 || device >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(scratch_mutex);
  if (scratch_ptr[device] == nullptr) {
    int prev = -1;
    if (cudaGetDevice(&prev) != cudaSuccess) return nullptr;
    if (prev != device && cudaSetDevice(device) != cudaSuccess) return nullptr;
    void* ptr = nullptr;
    const cudaError_t err = cudaGetSymbolAddress(&ptr, decode_scratch);
    if (prev != device) cudaSetDevice(prev);
    if (err != cudaSuccess) return nullptr;
    scratch_ptr[device] = ptr;
  }
  return scratch_ptr[device];
}

}  // namespace

extern "C" tq_status tq_decode_attention_static(const tq_codebook* book, const void* q, tq_dtype dtype, int batch,
                                                int n_q_heads, int n_kv_heads, const tq_cache_view* cache,
                                                const int32_t* block_table, int max_blocks,
                                                const int32_t* context_lens, int max_context, float scale,
                                                float* out, void* stream) {
  if (book == nullptr || book->device < 0) return TQ_ERR_INVALID_ARG;
  if (tq_decode_workspace_bytes(book, batch, n_q_heads, max_context) > TQ_STATIC_WORKSPACE_BYTES) {
    return TQ_ERR_WORKSPACE;
  }
  void* scratch = scratch_address(book->device);
  if (scratch == nullptr) return TQ_ERR_CUDA;
  return tq_decode_attention(book, q, dtype, batch, n_q_heads, n_kv_heads, cache, block_table, max_blocks,
                             context_lens, max_context, scale, out, scratch, TQ_STATIC_WORKSPACE_BYTES, stream);
}
