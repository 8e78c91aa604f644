// The backward's memory-bound steps around the DGrad/WGrad GEMMs:
//   dY[p]  = w[t,j] * dout[t]                 (combine backward, p = dest_of[t*k+j])
//   dw_tj  = <dout[t], y_p>                    (routing-weight gradient)
//   dlogits[t, e_j] = p_j (dw_j - sum_i p_i dw_i), zero elsewhere
// with p the softmax of the k selected logits (the router's weights before
// their fp32 rounding).  Every sum runs in a fixed order.
#include <math.h>

#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kDwThreads = 128;

// dY[dest_of[t * k + j]] = bf16(w[t, j] * dout[t]) for every slot j < k:
// each row of dout is read once (one warp per segment of 4 x 32 16-byte
// vectors, all four loads of a lane in flight) and stored, scaled, at its k
// places in expert order.
constexpr int kScaleUnroll = 4;
__global__ void __launch_bounds__(256)
scale_gather_kernel(const __nv_bfloat16* __restrict__ dout, const int32_t* __restrict__ dest_of,
                    const float* __restrict__ topk_w, int T, int H, int k,
                    __nv_bfloat16* __restrict__ dY) {
  const int nv = H / 8;
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const int upr = (nv + 32 * kScaleUnroll - 1) / (32 * kScaleUnroll);   // segments per row
  const long long units = (long long)T * upr;
  for (long long wu = blockIdx.x * wpb + (threadIdx.x >> 5); wu < units;
       wu += (long long)gridDim.x * wpb) {
    const int t = (int)(wu / upr);
    const int v0 = (int)(wu - (long long)t * upr) * 32 * kScaleUnroll + lane;
    const int4* src = reinterpret_cast<const int4*>(dout + (size_t)t * H);
    float2 f[kScaleUnroll][4];
#pragma unroll
    for (int u = 0; u < kScaleUnroll; ++u) {
      if (v0 + 32 * u >= nv) continue;
      const int4 r = __ldg(src + v0 + 32 * u);
      const __nv_bfloat162* in = reinterpret_cast<const __nv_bfloat162*>(&r);
#pragma unroll
      for (int c = 0; c < 4; ++c) f[u][c] = __bfloat1622float2(in[c]);
    }
    for (int j = 0; j < k; ++j) {
      const size_t a = (size_t)t * k + j;
      const float w = __ldg(topk_w + a);
      int4* dst = reinterpret_cast<int4*>(dY + (size_t)__ldg(dest_of + a) * H);
#pragma unroll
      for (int u = 0; u < kScaleUnroll; ++u) {
        if (v0 + 32 * u >= nv) continue;
        int4 o;
        __nv_bfloat162* po = reinterpret_cast<__nv_bfloat162*>(&o);
#pragma unroll
        for (int c = 0; c < 4; ++c) po[c] = __floats2bfloat162_rn(w * f[u][c].x, w * f[u][c].y);
        dst[v0 + 32 * u] = o;
      }
    }
  }
}

// One CTA per token: dw over the k slots, then the token's dlogits row.
__global__ void __launch_bounds__(kDwThreads)
dw_dlogits_kernel(const __nv_bfloat16* __restrict__ dout, const __nv_bfloat16* __restrict__ y,
                  const int32_t* __restrict__ dest_of, const int32_t* __restrict__ topk_idx,
                  const float* __restrict__ logits, int H, int E, int k,
                  float* __restrict__ dlogits) {
  __shared__ int s_row[MOE_MAX_TOPK];
  __shared__ float s_part[kDwThreads / 32][MOE_MAX_TOPK];
  __shared__ float s_dw[MOE_MAX_TOPK];
  const int t = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x < k) s_row[threadIdx.x] = dest_of[(size_t)t * k + threadIdx.x];
  for (int e = threadIdx.x; e < E; e += kDwThreads) dlogits[(size_t)t * E + e] = 0.f;
  __syncthreads();
  float acc[MOE_MAX_TOPK];
#pragma unroll
  for (int j = 0; j < MOE_MAX_TOPK; ++j) acc[j] = 0.f;
  const int nv = H / 8;
  for (int v = threadIdx.x; v < nv; v += kDwThreads) {
    const int4 dr = __ldg(reinterpret_cast<const int4*>(dout + (size_t)t * H) + v);
    const __nv_bfloat162* d2 = reinterpret_cast<const __nv_bfloat162*>(&dr);
    float d[8];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float2 f = __bfloat1622float2(d2[c]);
      d[2 * c] = f.x;
      d[2 * c + 1] = f.y;
    }
#pragma unroll
    for (int j = 0; j < MOE_MAX_TOPK; ++j) {
      if (j >= k) break;
      const int4 yr = __ldg(reinterpret_cast<const int4*>(y + (size_t)s_row[j] * H) + v);
      const __nv_bfloat162* y2 = reinterpret_cast<const __nv_bfloat162*>(&yr);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const float2 f = __bfloat1622float2(y2[c]);
        acc[j] = fmaf(d[2 * c], f.x, acc[j]);
        acc[j] = fmaf(d[2 * c + 1], f.y, acc[j]);
      }
    }
  }
#pragma unroll
  for (int j = 0; j < MOE_MAX_TOPK; ++j) {
    if (j >= k) break;
    float v = acc[j];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0) s_part[warp][j] = v;
  }
  __syncthreads();
  if (threadIdx.x < k) {
    float v = 0.f;
#pragma unroll
    for (int w = 0; w < kDwThreads / 32; ++w) v += s_part[w][threadIdx.x];
    s_dw[threadIdx.x] = v;
  }
  __syncthreads();
  if (warp == 0) {
    // softmax of the selected logits (slot 0 holds the largest) and its Jacobian
    const int e = lane < k ? topk_idx[(size_t)t * k + lane] : 0;
    const float l = lane < k ? logits[(size_t)t * E + e] : 0.f;
    const float m = __shfl_sync(0xffffffffu, l, 0);
    const float ex = lane < k ? expf(l - m) : 0.f;
    float sum = ex;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    const float p = ex / sum;
    const float dw = lane < k ? s_dw[lane] : 0.f;
    float pd = p * dw;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) pd += __shfl_xor_sync(0xffffffffu, pd, off);
    if (lane < k) dlogits[(size_t)t * E + e] = p * (dw - pd);
  }
}

}  // namespace

cudaError_t launch_scale_gather(const __nv_bfloat16* dout, const int32_t* dest_of,
                                const float* topk_w, int T, int H, int k, __nv_bfloat16* dY,
                                cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const long long segs = (long long)T * ((H / 8 + 127) / 128);
  const long long want = (segs + 7) / 8;                  // 8 warps (segments) per CTA
  const int grid = (int)(want < 8LL * device_sm_count() ? want : 8LL * device_sm_count());
  scale_gather_kernel<<<grid, 256, 0, s>>>(dout, dest_of, topk_w, T, H, k, dY);
  return cudaGetLastError();
}

cudaError_t launch_dw_dlogits(const __nv_bfloat16* dout, const __nv_bfloat16* y,
                              const int32_t* dest_of, const int32_t* topk_idx,
                              const float* logits, int T, int H, int E, int k, float* dlogits,
                              cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  dw_dlogits_kernel<<<T, kDwThreads, 0, s>>>(dout, y, dest_of, topk_idx, logits, H, E, k,
                                             dlogits);
  return cudaGetLastError();
}

}  // namespace moe
