// k3moe_layer_static: the MoE layer without a caller-provided workspace.
//
// Some callers cannot call cudaMalloc at all: code embedded in a host program that owns every
// device allocation through its own pool or arena and forbids stray allocations, and
// latency-critical callers that cannot pay for cudaMalloc's implicit device synchronisation.
// For them this entry point takes its scratch from a fixed array in device memory that the
// library itself declares, so a call allocates nothing. The caller still provides the inputs and
// the output buffer.
//
// Properties a caller must know:
//  * The array is K3MOE_STATIC_SCRATCH_BYTES (4 MiB) per device and stays resident on every GPU
//    that loads the library, until the process exits.
//  * Calls whose workspace (k3moe_workspace_bytes(cfg, T)) exceeds it return
//    K3MOE_ERR_WORKSPACE; at the d_model 7168 / d_ff 1536 / 896-expert top-16 shape with 2 shared
//    experts, calls of up to 6 tokens are served and 7 or more are refused.
//  * All calls on a device share the one array and it keeps the previous call's contents; the
//    part a call needs is cleared (cudaMemsetAsync, which allocates nothing) at the start of each
//    call. Two calls whose work overlaps on the GPU (different streams, or different host threads
//    without ordering) race on the array and give wrong results.
//  * The first call on each device looks up the array's device address (cudaGetSymbolAddress,
//    with that device current) and caches it; make that first call before any stream capture.
//  * Bad data found on the device is not reported by this entry point (there is no workspace the
//    caller could pass to k3moe_check_device_status); use k3moe_layer to check data.
//  * Argument checks and status codes are k3moe_layer's; nothing is launched when they fail.
//  * The cached address belongs to the device's context at the first call: resetting the device
//    (cudaDeviceReset) after that and calling again is not supported.
#include <cstdint>
#include <mutex>

#include "../../include/k3moe.h"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[K3MOE_STATIC_SCRATCH_BYTES];

void* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mutex;

// Device address of the static scratch on the current device (looked up once per device).
cudaError_t static_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" k3moe_status k3moe_layer_static(const k3moe_config* cfg, const void* x, int64_t T, const float* w_router,
                                           const float* bias, const uint8_t* routed_records,
                                           const uint8_t* shared_records, float* y, void* stream) {
  // the argument checks of k3moe_layer, and its status codes: with zero tokens it validates the
  // config and the pointers and launches nothing
  k3moe_status s = k3moe_layer(cfg, x, 0, w_router, nullptr, bias, routed_records, shared_records, y, nullptr,
                               nullptr, nullptr, 0, stream);
  if (s != K3MOE_OK) return s;
  if (T < 0) return K3MOE_ERR_INVALID_ARGUMENT;
  if (T == 0) return K3MOE_OK;
  const size_t need = k3moe_workspace_bytes(cfg, T);
  if (need == 0) return K3MOE_ERR_INVALID_ARGUMENT;  // token count beyond the library's limits
  if (need > (size_t)K3MOE_STATIC_SCRATCH_BYTES) return K3MOE_ERR_WORKSPACE;
  void* ws = nullptr;
  if (static_scratch(&ws) != cudaSuccess) return K3MOE_ERR_CUDA;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, need, st) != cudaSuccess) return K3MOE_ERR_CUDA;
  return k3moe_layer(cfg, x, T, w_router, nullptr, bias, routed_records, shared_records, y, nullptr, nullptr, ws, need,
                     stream);
}
