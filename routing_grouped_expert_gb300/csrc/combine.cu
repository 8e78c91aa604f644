// Step 4: weighted return to token order, the final top-k sum
// ("MegaFlux", §2.1; "MegaScale-Infer", §3.2 step (4)):
//   out[t] = sum_{j<k} topk_w[t,j] * y_sorted[dest_of[t*k+j]]
// One CTA per (token, 1024-column slice); each thread owns 8 consecutive
// columns (one 16-byte vector) and sums the k expert rows in slot order in
// fp32, so the result is bit-identical run to run.  A slot whose dest_of is
// -1 (an out-of-range expert index in the permute) adds nothing.
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

// OutT: __nv_bfloat16 (the layer's output, rounded once) or float (the
// unrounded fp32 sum, for layers whose partial outputs are summed elsewhere).
template <typename OutT>
__global__ void __launch_bounds__(kCombineThreads)
combine_kernel(const __nv_bfloat16* __restrict__ y_sorted, const int32_t* __restrict__ dest_of,
               const float* __restrict__ topk_w, int H, int k, int P,
               OutT* __restrict__ out, const __nv_bfloat16* __restrict__ y_shared) {
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
      const int row = s_row[j];
      if (row < 0 || row >= P) continue;   // an assignment that took no position
      const int4 raw = __ldg(reinterpret_cast<const int4*>(y_sorted + (size_t)row * H) + v);
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
    if constexpr (sizeof(OutT) == 4) {
      float4* o = reinterpret_cast<float4*>(out + (size_t)t * H) + 2 * v;
      o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    } else {
      int4 o;
      __nv_bfloat162* po = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
      for (int i = 0; i < 4; ++i) po[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
      reinterpret_cast<int4*>(out + (size_t)t * H)[v] = o;
    }
  }
}

// out[i] = bf16(in[i]), round to nearest even; 8 values per thread.
__global__ void __launch_bounds__(256)
cast_bf16_kernel(const float* __restrict__ in, __nv_bfloat16* __restrict__ out, size_t n) {
  const size_t i0 = ((size_t)blockIdx.x * blockDim.x + threadIdx.x) * 8;
  if (i0 + 8 <= n) {
    const float4 a = reinterpret_cast<const float4*>(in + i0)[0];
    const float4 b = reinterpret_cast<const float4*>(in + i0)[1];
    int4 o;
    __nv_bfloat162* po = reinterpret_cast<__nv_bfloat162*>(&o);
    po[0] = __floats2bfloat162_rn(a.x, a.y);
    po[1] = __floats2bfloat162_rn(a.z, a.w);
    po[2] = __floats2bfloat162_rn(b.x, b.y);
    po[3] = __floats2bfloat162_rn(b.z, b.w);
    *reinterpret_cast<int4*>(out + i0) = o;
  } else {
    for (size_t i = i0; i < n; ++i) out[i] = __float2bfloat16_rn(in[i]);
  }
}

}  // namespace

cudaError_t launch_cast_bf16(const float* in, __nv_bfloat16* out, size_t n, cudaStream_t s) {
  if (n == 0) return cudaSuccess;
  const size_t threads = (n + 7) / 8;
  cast_bf16_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(in, out, n);
  return cudaGetLastError();
}

cudaError_t launch_combine(const __nv_bfloat16* y_sorted, const int32_t* dest_of,
                           const float* topk_w, int T, int H, int k, __nv_bfloat16* out,
                           cudaStream_t s, const __nv_bfloat16* y_shared, bool pdl) {
  if (T == 0) return cudaSuccess;
  const int slices = (H / 8 + kCombineThreads - 1) / kCombineThreads;
  // tokens on the x dimension (up to 2^31 - 1), column slices on y
  return launch_k(combine_kernel<__nv_bfloat16>, dim3(T, slices), dim3(kCombineThreads), 0, s,
                  pdl, y_sorted, dest_of, topk_w, H, k, T * k, out, y_shared);
}

cudaError_t launch_combine_f32(const __nv_bfloat16* y_sorted, const int32_t* dest_of,
                               const float* topk_w, int T, int H, int k, float* out,
                               cudaStream_t s, bool pdl) {
  if (T == 0) return cudaSuccess;
  const int slices = (H / 8 + kCombineThreads - 1) / kCombineThreads;
  return launch_k(combine_kernel<float>, dim3(T, slices), dim3(kCombineThreads), 0, s, pdl,
                  y_sorted, dest_of, topk_w, H, k, T * k, out,
                  static_cast<const __nv_bfloat16*>(nullptr));
}

}  // namespace moe
