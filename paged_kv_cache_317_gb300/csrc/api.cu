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

// Self-test of the bounded wait every kernel uses: one warp waits on an
// mbarrier phase that completes only if `arrive` is set.  Without the arrival
// the wait gives up after `limit_ns` and records PA_ERR_TIMEOUT, exactly as a
// stalled pipeline inside a real kernel would; the kernel then returns normally.
namespace {
__global__ void bounded_wait_selftest_kernel(int32_t* err, unsigned long long limit_ns,
                                             int arrive) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    pagedkv::mbar_init(&bar, 1);
    pagedkv::fence_mbar_init();
  }
  __syncthreads();
  if (arrive && threadIdx.x == 0) pagedkv::mbar_arrive(&bar);
  const bool ok = pagedkv::mbar_wait_bounded(&bar, 0, limit_ns);
  if (!__all_sync(pagedkv::kFullMask, ok) && threadIdx.x == 0)
    pagedkv::report_error(err, PA_ERR_TIMEOUT, 0, 0);
}
}  // namespace

extern "C" int pa_selftest_bounded_wait(int32_t* error_record, int arrive,
                                        unsigned long long limit_ns, void* stream) {
  if (!error_record || limit_ns == 0 || limit_ns > pagedkv::kWaitLimitNs)
    return PA_ERR_INVALID_ARG;
  bounded_wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      error_record, limit_ns, arrive);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
