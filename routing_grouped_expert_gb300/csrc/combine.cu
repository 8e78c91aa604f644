// Step 4: weighted return to token order, the final top-k sum
// ("MegaFlux", §2.1; "MegaScale-Infer", §3.2 step (4)):
//   out[t] = sum_{j<k} topk_w[t,j] * y_sorted[dest_of[t*k+j]]
// One CTA per (token, 1024-column slice); each thread owns 8 consecutive
// columns (one 16-byte vector) and sums the k expert rows in slot order in
// fp32, so the result is bit-identical run to run.
#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kCombineThreads = 128;

__device__ __forceinline__ void bf16x8_to_f32(const int4& v, float (&f)[8]) {
  const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 q = __bfloat1622float2(p[i]);
    f[2 * i] = q.x;
    f[2 * i + 1] = q.y;
  }
}

__global__ void __launch_bounds__(kCombineThreads)
combine_kernel(const __nv_bfloat16* __restrict__ y_sorted, const int32_t* __restrict__ dest_of,
               const float* __restrict__ topk_w, int H, int k,
               __nv_bfloat16* __restrict__ out, const __nv_bfloat16* __restrict__ y_shared) {
  __shared__ int s_row[MOE_MAX_TOPK];
  __shared__ float s_w[MOE_MAX_TOPK];
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  if (threadIdx.x < k) {
    s_row[threadIdx.x] = dest_of[(size_t)t * k + threadIdx.x];
    s_w[threadIdx.x] = topk_w ? topk_w[(size_t)t * k + threadIdx.x] : 1.0f;   // null: unweighted
  }
  __syncthreads();
  const int nv = H / 8;
  for (int v = blockIdx.y * kCombineThreads + threadIdx.x; v < nv;
       v += gridDim.y * kCombineThreads) {
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    for (int j = 0; j < k; ++j) {
      const int4 raw =
          __ldg(reinterpret_cast<const int4*>(y_sorted + (size_t)s_row[j] * H) + v);
      float f[8];
      bf16x8_to_f32(raw, f);
      const float w = s_w[j];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = fmaf(w, f[i], acc[i]);
    }
    if (y_shared != nullptr) {   // always-active expert, weight one, after the slots
      const int4 raw = __ldg(reinterpret_cast<const int4*>(y_shared + (size_t)t * H) + v);
      float f[8];
      bf16x8_to_f32(raw, f);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += f[i];
    }
    int4 o;
    __nv_bfloat162* po = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
    for (int i = 0; i < 4; ++i) po[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
    reinterpret_cast<int4*>(out + (size_t)t * H)[v] = o;
  }
}

}  // namespace

cudaError_t launch_combine(const __nv_bfloat16* y_sorted, const int32_t* dest_of,
                           const float* topk_w, int T, int H, int k, __nv_bfloat16* out,
                           cudaStream_t s, const __nv_bfloat16* y_shared, bool pdl) {
  if (T == 0) return cudaSuccess;
  const int slices = (H / 8 + kCombineThreads - 1) / kCombineThreads;
  // tokens on the x dimension (up to 2^31 - 1), column slices on y
  return launch_k(combine_kernel, dim3(T, slices), dim3(kCombineThreads), 0, s, pdl, y_sorted,
                  dest_of, topk_w, H, k, out, y_shared);
}

}  // namespace moe
