// moe_permute_noalloc: the permute step for callers that cannot allocate
// device memory.  Its scratch -- per-chunk histograms and bases, the token
// block plan and a status word -- lives in one fixed array in device memory
// instead of a caller-supplied workspace.  The kernels are the same ones
// moe_permute launches; only where their scratch lives differs.
#include <cuda.h>

#include <mutex>

#include "moe_common.cuh"

// The scratch: MOE_PERMUTE_NOALLOC_SCRATCH_BYTES on every GPU on which the
// library's device code is loaded, held until the process exits.  All calls
// share it and it keeps the last call's contents.
static __device__ __align__(256) int32_t g_permute_scratch[MOE_PERMUTE_NOALLOC_SCRATCH_BYTES /
                                                           sizeof(int32_t)];

namespace {

constexpr size_t kScratchInts = MOE_PERMUTE_NOALLOC_SCRATCH_BYTES / sizeof(int32_t);

size_t round64(size_t v) { return (v + 63) / 64 * 64; }

// Ints of scratch one call needs: status, chunk histograms, block plan.
size_t scratch_ints(int T, int E, int k) {
  const size_t C = (size_t)moe::num_chunks(T, k);
  const size_t NB = (size_t)moe::max_blocks((long long)T * k, E);
  return 64 + round64(C * E) + round64((size_t)E + 1) + 64 + round64(NB);
}

// The device address of g_permute_scratch differs per CUDA context (each
// context loads the library's device code on its own, and a device reset
// replaces the context), so it is looked up once per context, keyed by the
// context's process-unique ID.  In host code the array's name is only a
// host-side stand-in, never a device pointer.
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<Fn>(p);
}

struct AddrCache {
  std::mutex mu;
  static constexpr int kSlots = 64;
  unsigned long long ctx_id[kSlots] = {};
  int32_t* addr[kSlots] = {};
  int next = 0;
};
AddrCache g_cache;

cudaError_t scratch_address(int32_t** out) {
  static const CtxGetCurrentFn get_ctx = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  if (get_ctx == nullptr || get_id == nullptr) return cudaErrorNotSupported;
  CUcontext ctx = nullptr;
  if (get_ctx(&ctx) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  if (ctx == nullptr) {
    // no context yet on this thread: cudaSetDevice makes the current device's
    // primary context current (creating it if needed)
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaSetDevice(dev);
    if (e != cudaSuccess) return e;
    if (get_ctx(&ctx) != CUDA_SUCCESS || ctx == nullptr) return cudaErrorDeviceUninitialized;
  }
  unsigned long long id = 0;
  if (get_id(ctx, &id) != CUDA_SUCCESS) return cudaErrorDeviceUninitialized;
  std::lock_guard<std::mutex> lock(g_cache.mu);
  for (int i = 0; i < AddrCache::kSlots; ++i)
    if (g_cache.addr[i] != nullptr && g_cache.ctx_id[i] == id) {
      *out = g_cache.addr[i];
      return cudaSuccess;
    }
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_permute_scratch);
  if (e != cudaSuccess) return e;
  const int slot = g_cache.next;
  g_cache.next = (slot + 1) % AddrCache::kSlots;
  g_cache.ctx_id[slot] = id;
  g_cache.addr[slot] = static_cast<int32_t*>(p);
  *out = g_cache.addr[slot];
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
      moe::launch_scatter(topk_idx, T, E, k, chunk, offsets, sorted_src, dest_of, s) !=
          cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}
