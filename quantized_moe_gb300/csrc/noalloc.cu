// Routing for callers that cannot allocate device memory.
//
// Some callers of this library cannot call cudaMalloc: an inference engine that carves all of
// its device memory up front with its own allocator and forbids later allocations, a plugin
// host that owns the memory budget, or a latency-critical path where cudaMalloc may
// synchronise the device. ds4moe_route_noalloc gives them the router step (fp32 logits,
// sigmoid top-k, renormalised weights) without a handle and without any allocation: the
// logits live in a fixed, file-scope device array instead of a per-handle workspace.
//
// The array (DS4MOE_NOALLOC_MAX_LOGITS floats plus an error word, ~1 MiB) is part of the
// library image, so every GPU that loads the library holds it until the process exits. Host
// code cannot use the array's name as a device address; the first call on each device, with
// that device current, looks the address up with cudaGetSymbolAddress and caches it, and raises
// the router kernel's shared-memory limit in that device's context. Make that first call before
// any stream capture. Every call on a device shares the one array and leaves the last call's
// logits in it: calls whose kernels may overlap on the GPU (different streams, no ordering
// between them) race on it.
#include <mutex>

#include "../../include/ds4moe.h"
#include "common.cuh"

namespace ds4 {
int set_error(int code, const char* msg);  // records the message returned by ds4moe_last_error
}

namespace {

constexpr int kScratchFloats = DS4MOE_NOALLOC_MAX_LOGITS + 64;  // logits, then the error word
static __device__ __align__(256) float g_route_scratch[kScratchFloats];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
float* g_scratch_ptr[kMaxDevices] = {};  // device address of g_route_scratch, per device; set once the
                                         // device's set-up (address and kernel attribute) succeeded

int scratch_for_current_device(float** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return ds4::set_error(DS4MOE_ERR_CUDA, "ds4moe_route_noalloc: no current CUDA device");
  }
  if (dev < 0 || dev >= kMaxDevices) return ds4::set_error(DS4MOE_ERR_INVALID_ARG, "ds4moe_route_noalloc: device ordinal above 63");
  std::lock_guard<std::mutex> lock(g_setup_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess || !p) {
      cudaGetLastError();
      return ds4::set_error(DS4MOE_ERR_CUDA, "ds4moe_route_noalloc: cudaGetSymbolAddress of the static scratch failed");
    }
    e = ds4::router_logits_prepare();  // kernel attributes live in each device's context
    if (e != cudaSuccess) {
      cudaGetLastError();
      return ds4::set_error(DS4MOE_ERR_CUDA, "ds4moe_route_noalloc: setting the router kernel's shared-memory limit failed");
    }
    g_scratch_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_scratch_ptr[dev];
  return DS4MOE_OK;
}

}  // namespace

extern "C" int ds4moe_route_noalloc(const float* router_w, const float* router_b, const void* x, int32_t n_tokens,
                                    int32_t d, int32_t n_experts, int32_t top_k, int32_t* idx, float* w,
                                    void* stream) {
  if (n_tokens < 0) return ds4::set_error(DS4MOE_ERR_INVALID_ARG, "ds4moe_route_noalloc: n_tokens is negative");
  if (d <= 0 || d % 128 || d > 12288)
    return ds4::set_error(DS4MOE_ERR_INVALID_ARG, "ds4moe_route_noalloc: d must be a positive multiple of 128 up to 12288");
  if (n_experts < 1 || n_experts > 256 || top_k < 1 || top_k > 16 || top_k > n_experts)
    return ds4::set_error(DS4MOE_ERR_INVALID_ARG, "ds4moe_route_noalloc: need 1 <= top_k <= min(n_experts, 16), n_experts <= 256");
  if ((int64_t)n_tokens * n_experts > DS4MOE_NOALLOC_MAX_LOGITS)
    return ds4::set_error(DS4MOE_ERR_CAPACITY,
                          "ds4moe_route_noalloc: n_tokens * n_experts exceeds the static scratch of "
                          "DS4MOE_NOALLOC_MAX_LOGITS (262144) logits");
  if (n_tokens == 0) return DS4MOE_OK;
  if (!router_w || !x || !idx || !w) return ds4::set_error(DS4MOE_ERR_INVALID_ARG, "ds4moe_route_noalloc: NULL pointer");
  if ((uintptr_t)x & 15 || (uintptr_t)router_w & 15)
    return ds4::set_error(DS4MOE_ERR_INVALID_ARG, "ds4moe_route_noalloc: x and router_w must be 16-byte aligned");
  float* scratch = nullptr;
  const int rc = scratch_for_current_device(&scratch);
  if (rc != DS4MOE_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* logits = scratch;
  int* err = reinterpret_cast<int*>(scratch + DS4MOE_NOALLOC_MAX_LOGITS);
  // the top-k kernel's error word starts at zero (only table-routed tokens, which this call does
  // not route, would set it); the logits are fully written before they are read
  cudaError_t e = cudaMemsetAsync(err, 0, sizeof(int), st);
  if (e == cudaSuccess) {
    ds4::launch_router_logits(static_cast<const __nv_bfloat16*>(x), n_tokens, d, router_w, router_b, n_experts,
                              logits, st);
    ds4::launch_topk(logits, n_tokens, n_experts, top_k, nullptr, 0, nullptr, 0, idx, w, err, st);
    e = cudaGetLastError();
  }
  if (e != cudaSuccess) return ds4::set_error(DS4MOE_ERR_CUDA, cudaGetErrorString(e));
  return DS4MOE_OK;
}
