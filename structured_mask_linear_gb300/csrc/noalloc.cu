// Forward without any device allocation: the workspace is a fixed array in the library
// itself instead of memory the caller provides.
//
// Who needs this: code that may not call cudaMalloc (or any allocator) while it runs,
// for example a caller inside a region where the CUDA context is shared with a caching
// allocator it must not disturb, a plugin whose host owns all device memory, or a caller
// that cannot size or keep a workspace between calls.  Such a caller still passes its
// own inputs and outputs; only the scratch space moves into the library.
//
// The array costs every GPU that loads this library LOGLINEAR_STATIC_WORKSPACE_BYTES of
// device memory until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "ll_internal.cuh"

namespace {

// Scratch for loglinear_fwd_static_workspace(); one copy per device.
static __device__ __align__(256) unsigned char g_static_workspace[LOGLINEAR_STATIC_WORKSPACE_BYTES];

std::mutex g_ws_mu;
void* g_ws_addr[128];  // device address of g_static_workspace, per device ordinal

// Looks up (once per device, with that device current) the device address of the array.
// Host code must never pass the symbol itself to a kernel: on the host it only names a
// shadow copy, not device memory.
ll_status static_workspace(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return LL_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_ws_mu);
  if (!g_ws_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_workspace) != cudaSuccess || !p) return LL_ERR_CUDA;
    g_ws_addr[dev] = p;
  }
  *out = g_ws_addr[dev];
  return LL_OK;
}

}  // namespace

extern "C" ll_status loglinear_fwd_static_workspace(const ll_shape* shape, const void* q,
                                                    const void* k, const void* v, const float* a,
                                                    const float* lambda, void* o, float* states_out,
                                                    float* state_logscale_out, int state_levels,
                                                    void* stream) {
  if (!shape) return LL_ERR_NULL;
  const size_t need = loglinear_fwd_workspace_bytes(shape);
  if (need == 0) return loglinear_fwd(shape, q, k, v, a, lambda, o, nullptr, 0, states_out,
                                      state_logscale_out, state_levels, stream);  // reports the shape error
  if (need > (size_t)LOGLINEAR_STATIC_WORKSPACE_BYTES) return LL_ERR_WORKSPACE;
  void* ws = nullptr;
  ll_status st = static_workspace(&ws);
  if (st != LL_OK) return st;
  // Nothing in the workspace needs to start at zero: every word is written before it is
  // read within one call.
  return loglinear_fwd(shape, q, k, v, a, lambda, o, ws, (size_t)LOGLINEAR_STATIC_WORKSPACE_BYTES,
                       states_out, state_logscale_out, state_levels, stream);
}
