// Step 1: top-k gating and weight normalisation, one warp per token
// ("MegaScale-Infer", §3.4 Fused Kernels, steps (1) and (3)), fused with
// the per-chunk expert histogram that step (2) needs (integer atomic adds
// into a zeroed table, so the counts do not depend on their order).
//
// Selection is k rounds of a warp arg-max on the raw fp32 logits: a larger
// value wins, equal values (IEEE ==, so -0.0 ties +0.0) go to the lower
// expert index.  The weights are the softmax over the k selected logits,
// in fp32 with the largest selected logit subtracted first.
#include "route_token.cuh"

namespace moe {
namespace {

constexpr int kRouteThreads = 256;   // 8 warps, one token each

template <int kPerLane>
__global__ void __launch_bounds__(kRouteThreads)
route_topk_kernel(const float* __restrict__ logits, int T, int E, int k, int tpc,
                  int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                  int32_t* __restrict__ chunk_hist, int* __restrict__ status) {
  // first kernel of the fused chain (launched in stream order): the next one
  // may start as soon as every CTA has begun; it waits for this one to finish
  pdl_trigger();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t = blockIdx.x * (kRouteThreads / 32) + warp;   // one token per warp
  if (t >= T) return;
  int my_idx;
  float my_w;
  const bool nonfinite = route_token<kPerLane>(logits + (size_t)t * E, E, k, lane, &my_idx, &my_w);
  if (lane < k) {
    topk_idx[(size_t)t * k + lane] = my_idx;
    topk_w[(size_t)t * k + lane] = my_w;
    // integer counts: the order of the atomic adds does not change them
    if (chunk_hist && my_idx >= 0 && my_idx < E)
      atomicAdd(&chunk_hist[(size_t)(t / tpc) * E + my_idx], 1);
  }
  if (nonfinite && lane == 0) set_status(status, MOE_ERR_NONFINITE);
}

// Per-chunk histogram of a caller-supplied topk_idx (moe_permute on its own).
__global__ void __launch_bounds__(kChunkAssign)
count_kernel(const int32_t* __restrict__ topk_idx, int P, int E, int chunk_assign,
             int32_t* __restrict__ chunk_hist, int* __restrict__ status) {
  extern __shared__ int hist_s[];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist_s[e] = 0;
  __syncthreads();
  const int a = blockIdx.x * chunk_assign + threadIdx.x;
  if (threadIdx.x < chunk_assign && a < P) {
    const int e = topk_idx[a];
    if (e >= 0 && e < E)
      atomicAdd(&hist_s[e], 1);
    else
      set_status(status, MOE_ERR_INVALID_ARG);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    chunk_hist[(size_t)blockIdx.x * E + e] = hist_s[e];
}

// chunk_hist, when given, must hold zeros: the kernel adds each chunk's
// per-expert counts into it.
template <int kPerLane>
cudaError_t launch_route_t(const float* logits, int T, int E, int k, int32_t* topk_idx,
                           float* topk_w, int32_t* chunk_hist, int* status, cudaStream_t s) {
  const int tpc = tokens_per_chunk(k);
  const int warps = kRouteThreads / 32;
  route_topk_kernel<kPerLane><<<(T + warps - 1) / warps, kRouteThreads, 0, s>>>(
      logits, T, E, k, tpc, topk_idx, topk_w, chunk_hist, status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* topk_idx,
                         float* topk_w, int32_t* chunk_hist, int* status, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  if (E <= 32) return launch_route_t<1>(logits, T, E, k, topk_idx, topk_w, chunk_hist, status, s);
  if (E <= 64) return launch_route_t<2>(logits, T, E, k, topk_idx, topk_w, chunk_hist, status, s);
  if (E <= 128) return launch_route_t<4>(logits, T, E, k, topk_idx, topk_w, chunk_hist, status, s);
  if (E <= 256) return launch_route_t<8>(logits, T, E, k, topk_idx, topk_w, chunk_hist, status, s);
  if (E <= 512)
    return launch_route_t<16>(logits, T, E, k, topk_idx, topk_w, chunk_hist, status, s);
  return launch_route_t<32>(logits, T, E, k, topk_idx, topk_w, chunk_hist, status, s);
}

cudaError_t launch_count(const int32_t* topk_idx, int T, int E, int k, int32_t* chunk_hist,
                         int* status, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const int C = num_chunks(T, k);
  const int chunk_assign = tokens_per_chunk(k) * k;
  count_kernel<<<C, kChunkAssign, (size_t)E * sizeof(int), s>>>(topk_idx, T * k, E, chunk_assign,
                                                                chunk_hist, status);
  return cudaGetLastError();
}

}  // namespace moe
