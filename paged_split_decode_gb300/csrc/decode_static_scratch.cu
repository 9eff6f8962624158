// decode_static_scratch.cu -- decode_paged for callers that cannot allocate
// device memory.
//
// decode_paged needs a workspace for its split-K partials, which the caller
// normally allocates. Some callers cannot: code that runs where
// cudaMalloc is not allowed (inside a custom allocator's own callbacks, a
// plugin host that hands out no device buffers, or a process that must not
// grow its device footprint after start-up). This file gives them one entry
// point that uses a fixed scratch array compiled into the library instead.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "launch.h"
#include "pdecode.h"

namespace {

// Size of the built-in scratch. Every GPU on which this entry point has been
// called holds this array until the process exits (under CUDA's lazy module
// loading the driver takes the memory at the first call, not when the
// library is loaded).
constexpr size_t kStaticScratchBytes = PD_STATIC_SCRATCH_BYTES;

// File-scope device array. In host code its name is only a host-side stand-in
// for the symbol; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};
unsigned long long g_ctx[kMaxDevices] = {};  // context the address belongs to (0: none yet)

// Device address of g_scratch on the current device: looked up with that
// device current, once per device and context (a cudaDeviceReset makes a new
// context, whose module may place the array elsewhere, so it is looked up
// again there).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  const unsigned long long ctx = pd::current_context_id();
  std::lock_guard<std::mutex> lock(g_mu);
  if (ctx == 0 || g_ctx[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
    g_ctx[dev] = ctx;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" pd_status decode_paged_static_scratch(const void* q, const void* k_cache,
                                                 const void* v_cache, const int32_t* block_table,
                                                 const int32_t* seq_lens, float scale, int window,
                                                 int qlen, int num_splits, void* out,
                                                 const pd_dims* dims, uint32_t* error_flag,
                                                 void* stream) {
  if (!dims) return PD_ERR_NULL;
  const size_t need = pd_workspace_bytes(dims, qlen, num_splits, 0);
  if (need > kStaticScratchBytes) return PD_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (need > 0 && scratch_address(&scratch) != cudaSuccess) return PD_ERR_CUDA;
  return decode_paged(q, k_cache, v_cache, block_table, seq_lens, scale, window, qlen, num_splits,
                      out, dims, scratch, scratch ? kStaticScratchBytes : 0, error_flag, stream);
}
