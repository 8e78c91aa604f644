// The steps either side of the routed path: the router projection
// logits = x W_g (the gating network that decides each token's experts,
// "MegaScale-Infer" §3.2 item 2; "Piper" §II-A) and the plan of a shared,
// always-active expert that sees every token ("Piper", Table I, "R + S").
//
// With E >= 64 the router is a tensor-core GEMM on the grouped-GEMM engine
// (one "expert" whose weight matrix is W_g).  With fewer experts it is a
// skinny product bound by reading x once, done here on the CUDA cores:
// each CTA owns a few tokens, its threads stride over H, and the per-expert
// partial sums are reduced across warps in a fixed order.
#include "moe_common.cuh"

namespace moe {
namespace {

template <int kE, int kTok>
__global__ void __launch_bounds__(256)
router_simt_kernel(const __nv_bfloat16* __restrict__ x, const __nv_bfloat16* __restrict__ Wg,
                   int T, int H, int E, float* __restrict__ logits) {
  // CTA = kTok tokens; its 8 warps split H (warp w takes h = 32 w + lane,
  // stepping by 256); partial sums meet in shared memory and are added in
  // warp order, so the result does not depend on scheduling.
  __shared__ float part[8][kTok][kE];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t0 = blockIdx.x * kTok;
  float acc[kTok][kE];
#pragma unroll
  for (int i = 0; i < kTok; ++i)
#pragma unroll
    for (int e = 0; e < kE; ++e) acc[i][e] = 0.f;
  for (int h = threadIdx.x; h < H; h += 256) {
    float xv[kTok];
#pragma unroll
    for (int i = 0; i < kTok; ++i)
      xv[i] = (t0 + i < T) ? __bfloat162float(x[(size_t)(t0 + i) * H + h]) : 0.f;
    const __nv_bfloat16* w = Wg + (size_t)h * E;
#pragma unroll
    for (int e = 0; e < kE; ++e) {
      const float wv = (e < E) ? __bfloat162float(w[e]) : 0.f;
#pragma unroll
      for (int i = 0; i < kTok; ++i) acc[i][e] = fmaf(xv[i], wv, acc[i][e]);
    }
  }
#pragma unroll
  for (int i = 0; i < kTok; ++i)
#pragma unroll
    for (int e = 0; e < kE; ++e) {
      float v = acc[i][e];
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      if (lane == 0) part[warp][i][e] = v;
    }
  __syncthreads();
  for (int j = threadIdx.x; j < kTok * kE; j += 256) {
    const int i = j / kE, e = j % kE;
    if (e < E && t0 + i < T) {
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) v += part[w][i][e];
      logits[(size_t)(t0 + i) * E + e] = v;
    }
  }
}

template <int kE, int kTok>
cudaError_t launch_simt(const __nv_bfloat16* x, const __nv_bfloat16* Wg, int T, int H, int E,
                        float* logits, cudaStream_t s) {
  router_simt_kernel<kE, kTok><<<(T + kTok - 1) / kTok, 256, 0, s>>>(x, Wg, T, H, E, logits);
  return cudaGetLastError();
}

__global__ void single_expert_offsets_kernel(int32_t* offsets, int T) {
  offsets[0] = 0;
  offsets[1] = T;
}

}  // namespace

cudaError_t launch_router(const __nv_bfloat16* x, const __nv_bfloat16* Wg, int T, int H, int E,
                          const SingleExpertPlan& plan, float* logits, int* status,
                          cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  if (E >= 64)
    return launch_router_gemm(x, Wg, T, H, E, plan.offsets, plan.block_off, plan.num_blocks,
                              plan.block_expert, logits, status, s);
  if (E <= 8) return launch_simt<8, 8>(x, Wg, T, H, E, logits, s);
  if (E <= 16) return launch_simt<16, 8>(x, Wg, T, H, E, logits, s);
  if (E <= 32) return launch_simt<32, 4>(x, Wg, T, H, E, logits, s);
  return launch_simt<64, 2>(x, Wg, T, H, E, logits, s);
}

cudaError_t launch_single_expert_plan(int T, int beta, const SingleExpertPlan& plan,
                                      cudaStream_t s) {
  single_expert_offsets_kernel<<<1, 1, 0, s>>>(plan.offsets, T);
  cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  return launch_plan(plan.offsets, 1, T, plan.block_off, plan.num_blocks, plan.block_expert,
                     beta, nullptr, s);
}

}  // namespace moe
