// qi21_step_noalloc: the denoiser step for callers that cannot allocate
// device memory. The step's workspace (modulated-LN rows, the qkv panel,
// the attention output, the SwiGLU hidden rows and the tanh-ed modulation)
// lives in a file-scope static device array instead of a caller buffer.
//
// Who needs this: a caller whose device memory is owned by another
// allocator and who has no workspace to hand over, or one that runs under a
// no-allocation-after-start-up rule (cudaMalloc can synchronise the whole
// device and stall every other stream, which a latency-bound serving loop
// cannot afford). Such callers still own their inputs and outputs; only the
// scratch moves into the library.
#include <cuda_runtime.h>

#include <cstdio>
#include <mutex>

#include "../../include/qi21.h"
#include "internal.h"

namespace {

// Held by every GPU that loads this library until the process exits.
static __device__ __align__(256) unsigned char g_step_scratch[QI21_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the static scratch on the current device, looked up on
// the first call per device (in host code the array's name is only a
// host-side stand-in, never a device address).
int scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
    return qi21::report_error(QI21_ERR_CUDA, "qi21_step_noalloc: no usable current device");
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_step_scratch);
    if (e != cudaSuccess || p == nullptr) {
      char msg[160];
      snprintf(msg, sizeof msg, "qi21_step_noalloc: cudaGetSymbolAddress of the static scratch failed: %s",
               cudaGetErrorString(e));
      return qi21::report_error(QI21_ERR_CUDA, msg);
    }
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return QI21_OK;
}

}  // namespace

extern "C" int qi21_step_noalloc(const qi21_geom* g, const qi21_layer* layers,
                                 const qi21_kvcache* cache, const float* x_in, float* x_out,
                                 const float* mods, void* stream) {
  int rc = qi21_geom_check(g);
  if (rc != QI21_OK) return rc;
  int32_t n = 0;
  rc = qi21_kvcache_info(cache, nullptr, &n, nullptr);
  if (rc != QI21_OK) return rc;
  const size_t need = qi21_workspace_bytes(g, n);
  if (need > static_cast<size_t>(QI21_NOALLOC_SCRATCH_BYTES)) {
    char msg[200];
    snprintf(msg, sizeof msg,
             "qi21_step_noalloc: %d target rows need %zu bytes of scratch; the static scratch holds %zu "
             "(use qi21_step with a caller workspace)",
             n, need, static_cast<size_t>(QI21_NOALLOC_SCRATCH_BYTES));
    return qi21::report_error(QI21_ERR_WORKSPACE, msg);
  }
  if (qi21::profiling_on())
    return qi21::report_error(QI21_ERR_STATE,
                              "qi21_step_noalloc: event profiling is on (it creates CUDA events)");
  void* ws = nullptr;
  rc = scratch_address(&ws);
  if (rc != QI21_OK) return rc;
  return qi21_step(g, layers, cache, x_in, x_out, mods, nullptr, ws,
                   static_cast<size_t>(QI21_NOALLOC_SCRATCH_BYTES), stream);
}
