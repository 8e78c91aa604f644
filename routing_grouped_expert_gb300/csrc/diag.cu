// Diagnostics: exercise the bounded waits of the grouped GEMM -- the mbarrier
// wait of every pipeline stage, and the counter wait with which FC2 waits for
// a token block's FC1 tiles -- on a barrier or counter that nothing ever
// advances, so the timeout path can be tested without a fault or a hang.
#include "moe_common.cuh"
#include "ptx.cuh"

namespace {

__global__ void wait_timeout_kernel(int* status, unsigned long long limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  moe::ptx::mbar_init(&bar, 1);
  moe::ptx::fence_mbar_init();
  // Phase 0 never completes: no thread arrives on `bar`.
  if (!moe::ptx::mbar_wait(&bar, 0, nullptr, limit_ns))
    moe::set_status(status, MOE_ERR_TIMEOUT, moe::kWaitDetailDrain + 1);
}

// The wait of FC2's producer for a token block's FC1 tiles, on a counter
// that nothing increments.
__global__ void count_wait_timeout_kernel(int* status, const int* cnt,
                                          unsigned long long limit_ns) {
  if (threadIdx.x != 0) return;
  if (!moe::ptx::wait_count(cnt, 1, nullptr, limit_ns))
    moe::set_status(status, MOE_ERR_TIMEOUT, moe::kWaitDetailDrain + 2);
}

}  // namespace

extern "C" moe_status moe_diag_count_wait_timeout(void* ws, size_t ws_bytes, long long limit_ns,
                                                  void* stream) {
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < 256)
    return MOE_ERR_WORKSPACE;
  if (limit_ns < 1000000LL || limit_ns > 2000000000LL) return MOE_ERR_INVALID_ARG;
  if (!moe::device_is_sm103()) return MOE_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* status = static_cast<int*>(ws);
  // status word, detail, and the counter at word 32 start at zero
  if (cudaMemsetAsync(status, 0, 33 * sizeof(int), s) != cudaSuccess) return MOE_ERR_CUDA;
  count_wait_timeout_kernel<<<1, 32, 0, s>>>(status, status + 32, (unsigned long long)limit_ns);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

extern "C" moe_status moe_diag_wait_timeout(void* ws, size_t ws_bytes, long long limit_ns,
                                            void* stream) {
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < 256)
    return MOE_ERR_WORKSPACE;
  if (limit_ns < 1000000LL || limit_ns > 2000000000LL) return MOE_ERR_INVALID_ARG;
  if (!moe::device_is_sm103()) return MOE_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* status = static_cast<int*>(ws);
  if (cudaMemsetAsync(status, 0, 2 * sizeof(int), s) != cudaSuccess) return MOE_ERR_CUDA;
  wait_timeout_kernel<<<1, 32, 0, s>>>(status, (unsigned long long)limit_ns);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
