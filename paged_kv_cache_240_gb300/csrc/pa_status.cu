// pa_status.cu -- status helpers of the C ABI.
#include <cuda_runtime.h>

#include "pa.h"
#include "pa_internal.h"

namespace {
thread_local cudaError_t g_last_cuda_error = cudaSuccess;
}

void pa_internal::record_cuda_error(cudaError_t e) { g_last_cuda_error = e; }

extern "C" const char* pa_last_cuda_error(void) {
  return g_last_cuda_error == cudaSuccess ? "no CUDA error" : cudaGetErrorString(g_last_cuda_error);
}

extern "C" const char* pa_status_str(pa_status status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_DEVICE_DATA: return "PA_ERR_DEVICE_DATA";
    case PA_ERR_OUT_OF_BLOCKS: return "PA_ERR_OUT_OF_BLOCKS";
  }
  return "PA_ERR_UNKNOWN";
}

extern "C" pa_status pa_check_flags(int32_t flags) {
  return flags == 0 ? PA_OK : PA_ERR_DEVICE_DATA;
}
