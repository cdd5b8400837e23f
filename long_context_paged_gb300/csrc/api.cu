// Host-side glue of the C ABI: error text, device status word, SM count cache, version.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "pa_common.cuh"

namespace pa {
namespace {
thread_local char g_last_error[256] = "";
std::mutex g_sm_mutex;
int g_sm_count[64] = {0};
}  // namespace

pa_status record_cuda_error(cudaError_t err, const char* where) {
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%d)", where, cudaGetErrorString(err),
           static_cast<int>(err));
  return PA_ERR_CUDA;
}

void snprintf_error(const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
}

int sm_count_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return -1;
  std::lock_guard<std::mutex> lock(g_sm_mutex);
  if (g_sm_count[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    g_sm_count[dev] = n;
  }
  return g_sm_count[dev];
}

}  // namespace pa

extern "C" pa_status pa_read_device_status(int32_t* status, uint32_t* flags_out,
                                           pa_stream_t stream) {
  if (!status || !flags_out) return PA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  int32_t host = 0;
  cudaError_t e = cudaMemcpyAsync(&host, status, sizeof(int32_t), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess) e = cudaMemsetAsync(status, 0, sizeof(int32_t), st);
  if (e != cudaSuccess) return pa::record_cuda_error(e, "pa_read_device_status");
  *flags_out = static_cast<uint32_t>(host);
  return PA_OK;
}

extern "C" const char* pa_status_string(pa_status s) {
  switch (s) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported shape or type";
    case PA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case PA_ERR_CUDA: return "CUDA error";
  }
  return "unknown status";
}

extern "C" const char* pa_last_error(void) { return pa::g_last_error; }

extern "C" int32_t pa_version(void) { return 200; }
