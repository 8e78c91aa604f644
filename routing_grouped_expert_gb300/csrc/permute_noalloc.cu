// moe_permute_noalloc: the permute step for callers that cannot allocate
// device memory.  Its scratch -- per-chunk histograms and bases, the token
// block plan and a status word -- lives in one fixed array in device memory
// instead of a caller-supplied workspace.  The kernels are the same ones
// moe_permute launches; only where their scratch lives differs.
#include <atomic>

#include "moe_common.cuh"

// The scratch: MOE_PERMUTE_NOALLOC_SCRATCH_BYTES on every GPU on which the
// library's device code is loaded, held until the process exits.  All calls
// share it and it keeps the last call's contents.
static __device__ __align__(256) int32_t g_permute_scratch[MOE_PERMUTE_NOALLOC_SCRATCH_BYTES /
                                                           sizeof(int32_t)];

namespace {

constexpr size_t kScratchInts = MOE_PERMUTE_NOALLOC_SCRATCH_BYTES / sizeof(int32_t);
constexpr int kMaxDevices = 64;
// Device address of g_permute_scratch, looked up once per device.  In host
// code the array's name is only a host-side stand-in, never a device pointer.
std::atomic<int32_t*> g_scratch_addr[kMaxDevices];

size_t round64(size_t v) { return (v + 63) / 64 * 64; }

// Ints of scratch one call needs: status, chunk histograms, block plan.
size_t scratch_ints(int T, int E, int k) {
  const size_t C = (size_t)moe::num_chunks(T, k);
  const size_t NB = (size_t)moe::max_blocks((long long)T * k, E);
  return 64 + round64(C * E) + round64((size_t)E + 1) + 64 + round64(NB);
}

cudaError_t scratch_address(int32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  int32_t* a = g_scratch_addr[dev].load(std::memory_order_relaxed);
  if (a == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_permute_scratch);
    if (e != cudaSuccess) return e;
    a = static_cast<int32_t*>(p);
    g_scratch_addr[dev].store(a, std::memory_order_relaxed);
  }
  *out = a;
  return cudaSuccess;
}

bool aligned_ptr(const void* p) {
  return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0;
}

}  // namespace

extern "C" moe_status moe_permute_noalloc(const int32_t* topk_idx, int T, int E, int k,
                                          int32_t* counts, int32_t* offsets,
                                          int32_t* sorted_src, int32_t* dest_of,
                                          void* stream) {
  if (T < 0 || E < 1 || E > MOE_MAX_EXPERTS || k < 1 || k > E || k > MOE_MAX_TOPK ||
      (long long)T * k >= (1LL << 31))
    return MOE_ERR_INVALID_ARG;
  if (!aligned_ptr(counts) || !aligned_ptr(offsets)) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!aligned_ptr(topk_idx) || !aligned_ptr(sorted_src) || !aligned_ptr(dest_of)))
    return MOE_ERR_INVALID_ARG;
  if (scratch_ints(T, E, k) > kScratchInts) return MOE_ERR_WORKSPACE;
  if (!moe::device_is_sm103()) return MOE_ERR_UNSUPPORTED;
  int32_t* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return MOE_ERR_CUDA;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int C = moe::num_chunks(T, k);
  int32_t* status = scratch;
  int32_t* chunk = scratch + 64;
  int32_t* block_off = chunk + round64((size_t)C * E);
  int32_t* num_blocks = block_off + round64((size_t)E + 1);
  int32_t* block_expert = num_blocks + 64;

  // The status word must start at zero; every other region is fully
  // written by the kernels before it is read.
  if (cudaMemsetAsync(status, 0, 2 * sizeof(int32_t), s) != cudaSuccess) return MOE_ERR_CUDA;
  if (T == 0) {
    if (cudaMemsetAsync(counts, 0, (size_t)E * sizeof(int32_t), s) != cudaSuccess ||
        cudaMemsetAsync(offsets, 0, (size_t)(E + 1) * sizeof(int32_t), s) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  }
  if (moe::launch_count(topk_idx, T, E, k, chunk, status, s) != cudaSuccess ||
      moe::launch_scan(chunk, C, E, counts, offsets, block_off, num_blocks, block_expert,
                       moe::kBlockRows, s) !=
          cudaSuccess ||
      moe::launch_scatter(topk_idx, T, E, k, chunk, sorted_src, dest_of, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
