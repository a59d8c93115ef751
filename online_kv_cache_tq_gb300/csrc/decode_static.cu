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
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "tq.h"
#include "tq_internal.h"

namespace {

constexpr int kMaxDevices = 64;

// Scratch shared by every call on a device; each GPU that loads the library
// holds it until the process exits.
static __device__ __align__(256) unsigned char decode_scratch[TQ_STATIC_WORKSPACE_BYTES];

using CtxGetCurrentFn = CUresult (*)(CUcontext*);

// cuCtxGetCurrent from the driver, looked up once through the runtime.
CtxGetCurrentFn ctx_get_current() {
  static CtxGetCurrentFn fn = [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult res;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &res) != cudaSuccess ||
        res != cudaDriverEntryPointSuccess) {
      ptr = nullptr;
    }
    return reinterpret_cast<CtxGetCurrentFn>(ptr);
  }();
  return fn;
}

struct ScratchSlot {
  CUcontext ctx = nullptr;   // context the address belongs to
  void* ptr = nullptr;
};
ScratchSlot scratch_slots[kMaxDevices];
std::mutex scratch_mutex;

// Device address of decode_scratch on `device` (the host-side name is only a
// stand-in).  Looked up with that device current the first time, and again
// whenever the device's current context is not the one the address was taken
// in (after a device reset the module, and with it the array, is loaded anew).
void* scratch_address(int device) {
  std::lock_guard<std::mutex> lock(scratch_mutex);
  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) return nullptr;
  if (prev != device && cudaSetDevice(device) != cudaSuccess) return nullptr;
  // (without the driver's context query every call looks the address up)
  CtxGetCurrentFn get = ctx_get_current();
  CUcontext ctx = nullptr;
  if (get == nullptr || get(&ctx) != CUDA_SUCCESS) ctx = nullptr;
  ScratchSlot& slot = scratch_slots[device];
  if (slot.ptr == nullptr || ctx == nullptr || slot.ctx != ctx) {
    void* ptr = nullptr;
    slot = ScratchSlot{};
    if (cudaGetSymbolAddress(&ptr, decode_scratch) == cudaSuccess) {
      CUcontext now = nullptr;              // (the look-up binds the context if none was current)
      if (get == nullptr || get(&now) != CUDA_SUCCESS) now = nullptr;
      slot.ctx = now;
      slot.ptr = ptr;
    }
  }
  void* out = slot.ptr;
  if (prev != device) cudaSetDevice(prev);
  return out;
}

}  // namespace

extern "C" tq_status tq_decode_attention_static(const tq_codebook* book, const void* q, tq_dtype dtype, int batch,
                                                int n_q_heads, int n_kv_heads, const tq_cache_view* cache,
                                                const int32_t* block_table, int max_blocks,
                                                const int32_t* context_lens, int max_context, float scale,
                                                float* out, void* stream) {
  // the handle and the device range first, then every argument and the scratch
  // size, and only then the (host-side) look-up of the array's address
  if (book == nullptr || book->device < 0 || book->device >= kMaxDevices || book->d_tables == nullptr) {
    return TQ_ERR_INVALID_ARG;
  }
  if (batch > 0 && tq_decode_workspace_bytes(book, batch, n_q_heads, max_context) > TQ_STATIC_WORKSPACE_BYTES) {
    return TQ_ERR_WORKSPACE;
  }
  const tq_status chk = tq::check_decode_call(book, q, dtype, batch, n_q_heads, n_kv_heads, cache, block_table,
                                              max_blocks, context_lens, max_context, scale, out,
                                              TQ_STATIC_WORKSPACE_BYTES);
  if (chk != TQ_OK || batch == 0) return chk;
  void* scratch = scratch_address(book->device);
  if (scratch == nullptr) return TQ_ERR_CUDA;
  return tq_decode_attention(book, q, dtype, batch, n_q_heads, n_kv_heads, cache, block_table, max_blocks,
                             context_lens, max_context, scale, out, scratch, TQ_STATIC_WORKSPACE_BYTES, stream);
}
