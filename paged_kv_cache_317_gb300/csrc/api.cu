// Library information and device error-record helpers of the C ABI.
#include <cuda_runtime.h>

#include "common.cuh"

extern "C" int pa_version(void) { return PAGEDKV_VERSION; }

extern "C" const char* pa_status_string(int status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported configuration";
    case PA_ERR_CUDA: return "CUDA error";
    case PA_ERR_BAD_BLOCK: return "block number out of range";
    case PA_ERR_BAD_SLOT: return "slot out of range";
    case PA_ERR_BAD_SEQ_LEN: return "sequence length out of range";
    case PA_ERR_TIMEOUT: return "device wait timed out";
    case PA_ERR_OOM: return "out of free blocks";
    case PA_ERR_NO_SEQ: return "unknown sequence";
    case PA_ERR_SEQ_EXISTS: return "sequence already exists";
    case PA_ERR_REFCOUNT: return "allocator state inconsistent";
    default: return "unknown status";
  }
}

extern "C" int pa_error_clear(int32_t* error_record, void* stream) {
  if (!error_record) return PA_ERR_INVALID_ARG;
  return cudaMemsetAsync(error_record, 0, PA_ERROR_RECORD_WORDS * sizeof(int32_t),
                         static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

extern "C" int pa_error_read(const int32_t* error_record, int32_t* host_out, void* stream) {
  if (!error_record || !host_out) return PA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(host_out, error_record, PA_ERROR_RECORD_WORDS * sizeof(int32_t),
                      cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return PA_ERR_CUDA;
  return cudaStreamSynchronize(st) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
