// fixed_scratch.cu -- paged decode attention for callers that cannot allocate device memory.
//
// pkv_paged_decode_attention needs a caller-provided workspace for its split-K partial
// results.  Some callers have no way to provide one: for example a plain C host program
// or plugin that links only this library and has no device allocator of its own, or a host
// runtime that owns the whole device heap and does not let libraries call cudaMalloc (which
// may also synchronise the device at a moment the caller cannot afford).  This entry point
// serves them: its scratch is a file-scope __device__ array of a fixed size
// (PKV_FIXED_SCRATCH_BYTES), which every GPU that loads the library keeps until the process
// exits.  The caller still passes every input and output.
//
// The array's name is only a host-side stand-in in host code, never a device address, so
// the address handed to the kernels is obtained with cudaGetSymbolAddress, once per device,
// with that device current, on the first call made on that device.
#include <mutex>

#include "kernels.h"
#include "pkv.h"

namespace pkv {
namespace {

constexpr int kMaxScratchDevices = 64;

static __device__ __align__(256) unsigned char g_fixed_scratch[PKV_FIXED_SCRATCH_BYTES];

std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxScratchDevices] = {};

// Device address of g_fixed_scratch on the current device (looked up once per device).
int fixed_scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxScratchDevices) {
    cudaGetLastError();
    return PKV_ERR_NO_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_fixed_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return e != cudaSuccess ? PKV_ERR_CUDA_BASE + (int)e : PKV_ERR_NO_DEVICE;
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

extern "C" int pkv_paged_decode_attention_fixed_scratch(
    void* out, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, const int32_t* context_lens, float scale, int32_t window,
    const pkv_dims* dims, int32_t* error_word, void* stream) {
  // Invalid dims, and shapes whose partial results do not fit the fixed scratch, are
  // refused by the shared validation before anything is enqueued (clear status).  The
  // scratch's ticket counters start at zero (static storage) and every call leaves them so.
  void* scratch = nullptr;
  if (pkv_decode_workspace_bytes(dims) != 0) {
    const int st = pkv::fixed_scratch_address(&scratch);
    if (st != PKV_OK) return st;
  }
  return pkv::decode_common(out, q, k_cache, v_cache, block_tables, context_lens, nullptr, nullptr,
                            0, scale, window, scratch, (size_t)PKV_FIXED_SCRATCH_BYTES, dims,
                            error_word, stream, false);
}
