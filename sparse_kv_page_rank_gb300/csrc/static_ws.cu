// locks_decode_step_static: the fused decode step run in a workspace the
// library owns, for callers that cannot allocate device memory themselves.
//
// The workspace is a file-scope device array, created with the module in each
// context that loads the library and kept until the context ends.  Host code
// may not pass the array's name to a kernel (on the host it only stands for
// the symbol), so its device address comes from cudaGetSymbolAddress.  The
// address is looked up again at every call made outside stream capture, so a
// call after cudaDeviceReset (a new context, a new copy of the array) uses the
// new array; a call being captured takes the address of the device's last
// uncaptured call, because the lookup may load the module.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/locks.h"

namespace {

constexpr size_t kStaticWsBytes = LOCKS_STATIC_WS_BYTES;
static __device__ __align__(256) unsigned char g_static_ws[kStaticWsBytes];

constexpr int kMaxDevices = 128;
std::mutex g_mutex;
void* g_ws_addr[kMaxDevices] = {};  // last looked-up address of g_static_ws, per device ordinal

// Device address of the array on the current device: a fresh lookup unless
// `stream` is capturing, then the last one made on this device.
locks_status_t static_ws_address(cudaStream_t stream, void** addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LOCKS_ERR_CUDA;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) return LOCKS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) return LOCKS_ERR_CUDA;
    g_ws_addr[dev] = p;
  } else if (!g_ws_addr[dev]) {
    return LOCKS_ERR_CUDA;  // no uncaptured call on this device yet
  }
  *addr = g_ws_addr[dev];
  return LOCKS_OK;
}

}  // namespace

extern "C" LOCKS_API locks_status_t locks_decode_step_static(const locks_cache_t* cache,
                                                             const locks_summary_t* summary,
                                                             const locks_params_t* params, const void* q,
                                                             void* out, float* lse, int32_t* sel_pages,
                                                             int32_t* sel_count, int32_t* device_error,
                                                             void* stream) {
  size_t need = 0;
  locks_status_t st = locks_workspace_size(cache, summary, params, &need);
  if (st != LOCKS_OK) return st;
  if (need > kStaticWsBytes) return LOCKS_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  void* ws = nullptr;
  if ((st = static_ws_address(s, &ws)) != LOCKS_OK) return st;
  // the error word and the counters must start at zero; clear every byte used
  if (cudaMemsetAsync(ws, 0, need, s) != cudaSuccess) return LOCKS_ERR_CUDA;
  st = locks_decode_step(cache, summary, params, q, out, lse, sel_pages, sel_count, ws, need, stream);
  if (st != LOCKS_OK) return st;
  if (device_error &&
      cudaMemcpyAsync(device_error, ws, sizeof(int32_t), cudaMemcpyDeviceToDevice, s) != cudaSuccess)
    return LOCKS_ERR_CUDA;
  return LOCKS_OK;
}
