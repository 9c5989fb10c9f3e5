// noalloc.cu -- relattn_decode_noalloc: split-KV decode whose split partials
// live in a fixed device array owned by this library, so the caller supplies
// no workspace and nothing is allocated.
//
// Who needs this: callers that cannot call cudaMalloc (or any allocating
// routine) at the point where they run attention -- a serving engine that
// hands all free device memory to its own pool up front (KV cache, activation
// arena) and has nothing left to lend; a plugin or custom-op host that offers
// no workspace hook; a latency-critical path where cudaMalloc's implicit
// device-wide synchronisation is not acceptable.  They still pass their own
// inputs and outputs; only the scratch moves into the library.
//
// The scratch is one file-scope __device__ array of kScratchBytes.  Every GPU
// that loads the library holds it until the process exits.  All calls on a
// device share it and it keeps the previous call's contents; nothing has to
// start at zero, because every partial the combine reads is written by the
// split kernel of the same call.  Two calls whose kernels overlap on the GPU
// (different streams without ordering) race on the array.
#include <mutex>

#include "../../include/relattn.h"
#include "launch.h"

namespace {

constexpr size_t kScratchBytes = RELATTN_NOALLOC_SCRATCH_BYTES;
__device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_ptr[kMaxDevices];
void *g_scratch_ctx[kMaxDevices];   // the context g_scratch_ptr[dev] was looked up in

// Device address of the scratch array on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// with that device current: on the first call on the device, and again
// whenever the current context differs from the one of the last lookup (a
// cudaDeviceReset makes a new primary context, into which the module, and the
// array with it, is loaded again, possibly at another address).
relattn_status scratch_for_current_device(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RELATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  void *ctx = relattn::current_cu_context();
  if (!g_scratch_ptr[dev] || !ctx || ctx != g_scratch_ctx[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return RELATTN_ERR_CUDA;
    g_scratch_ptr[dev] = p;
    g_scratch_ctx[dev] = relattn::current_cu_context();
  }
  *out = g_scratch_ptr[dev];
  return RELATTN_OK;
}

}  // namespace

extern "C" relattn_status relattn_decode_noalloc(const relattn_params *params, void *stream) {
  if (!params) return RELATTN_ERR_INVALID_ARG;
  size_t need = 0;
  relattn_status st = relattn_decode_workspace_size(params, &need);
  if (st != RELATTN_OK) return st;
  if (need > kScratchBytes) return RELATTN_ERR_WORKSPACE;
  relattn_params p = *params;
  p.workspace = nullptr;
  p.workspace_bytes = 0;
  if (need > 0) {
    if ((st = scratch_for_current_device(&p.workspace)) != RELATTN_OK) return st;
    p.workspace_bytes = kScratchBytes;
  }
  return relattn_decode(&p, stream);
}
