// The per-token top-k routing of one warp, shared by the route kernel and
// the fused small-batch route + permute kernel: k rounds of a warp arg-max on
// the raw fp32 logits (a larger value wins; equal values -- IEEE ==, so -0.0
// ties +0.0 -- go to the lower expert index), then the softmax over the k
// selected logits in fp32 with the largest one subtracted first
// ("MegaScale-Infer", §3.4 Fused Kernels, steps (1) and (3)).
#pragma once

#include <math.h>

#include "moe_common.cuh"

namespace moe {

struct RouteCand {
  float v;
  int i;   // expert index, -1 = no candidate
};

// True when candidate b should replace a.
__device__ __forceinline__ bool route_better(const RouteCand& b, const RouteCand& a) {
  if (b.i < 0) return false;
  if (a.i < 0) return true;
  return b.v > a.v || (b.v == a.v && b.i < a.i);
}

// Called by all 32 lanes of a warp for token row `row` of E logits.  Lane
// j < k returns slot j's expert in *idx and its weight in *w; the return
// value is true (on every lane) if the row holds a NaN or infinite logit,
// which is ranked as -inf so the picks stay distinct and in range.
// route_token_vals does the same from logits the lanes have already loaded
// (raw[i] = logit of expert lane + 32 i, any value for experts >= E), so a
// caller can have several tokens' loads in flight at once.
template <int kPerLane>
__device__ __forceinline__ bool route_token_vals(const float (&raw)[kPerLane], int E, int k,
                                                 int lane, int* idx, float* w) {
  bool nonfinite = false;
  float v[kPerLane];
#pragma unroll
  for (int i = 0; i < kPerLane; ++i) {
    const int e = lane + 32 * i;
    float x = (e < E) ? raw[i] : -INFINITY;
    if (e < E && !isfinite(x)) {
      nonfinite = true;
      if (isnan(x)) x = -INFINITY;   // keep the order total; the status reports it
    }
    v[i] = x;
  }
  uint32_t taken = 0;
  float my_sel = 0.f;
  int my_idx = 0;
  for (int j = 0; j < k; ++j) {
    RouteCand c{-INFINITY, -1};
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
      const int e = lane + 32 * i;
      if (e < E && !((taken >> i) & 1u)) {
        RouteCand d{v[i], e};
        if (route_better(d, c)) c = d;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      RouteCand o{__shfl_xor_sync(0xffffffffu, c.v, off), __shfl_xor_sync(0xffffffffu, c.i, off)};
      if (route_better(o, c)) c = o;
    }
    if (c.i >= 0 && (c.i & 31) == lane) taken |= 1u << (c.i >> 5);
    if (lane == j) {
      my_sel = c.v;
      my_idx = c.i;
    }
  }
  // softmax over the k selected logits (slot 0 holds the largest)
  const float m = __shfl_sync(0xffffffffu, my_sel, 0);
  const float ex = (lane < k) ? expf(my_sel - m) : 0.f;
  float sum = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  *idx = my_idx;
  *w = ex / sum;
  return __any_sync(0xffffffffu, nonfinite);
}

template <int kPerLane>
__device__ __forceinline__ bool route_token(const float* __restrict__ row, int E, int k, int lane,
                                            int* idx, float* w) {
  float raw[kPerLane];
#pragma unroll
  for (int i = 0; i < kPerLane; ++i) {
    const int e = lane + 32 * i;
    raw[i] = (e < E) ? __ldg(row + e) : 0.f;
  }
  return route_token_vals<kPerLane>(raw, E, k, lane, idx, w);
}

}  // namespace moe
