// The per-token top-k routing of one warp, shared by the route kernel and
// the fused small-batch route + permute kernel: k rounds of a warp arg-max on
// the raw fp32 logits (a larger value wins; equal values -- IEEE ==, so -0.0
// ties +0.0 -- go to the lower expert index), then the softmax over the k
// selected logits in fp32 with the largest one subtracted first
// ("MegaScale-Infer", §3.4 Fused Kernels, steps (1) and (3)).  Each lane
// sorts its own logits once; a round is then two warp reductions (redux) over
// the lanes' current heads.
#pragma once

#include <math.h>

#include "moe_common.cuh"

namespace moe {

// Called by all 32 lanes of a warp for token row `row` of E logits.  Lane
// j < k returns slot j's expert in *idx and its weight in *w; the return
// value is true (on every lane) if the row holds a NaN or infinite logit,
// which is ranked as -inf so the picks stay distinct and in range.
// route_token_vals does the same from logits the lanes have already loaded
// (raw[i] = logit of expert lane + 32 i, any value for experts >= E), so a
// caller can have several tokens' loads in flight at once.
// Order-preserving key of a candidate's logit: a larger value gives a larger
// key, -0.0 and +0.0 the same key (they tie, as IEEE == has it); key 0 is "no
// candidate", below every value (-inf included).
__device__ __forceinline__ uint32_t route_key(float x) {
  const uint32_t b = x == 0.f ? 0u : __float_as_uint(x);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float route_key_value(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

template <int kPerLane>
__device__ __forceinline__ bool route_token_vals(const float (&raw)[kPerLane], int E, int k,
                                                 int lane, int* idx, float* w) {
  bool nonfinite = false;
  // this lane's candidates: keys, and their slots i (expert lane + 32 i)
  uint32_t key[kPerLane];
  int slot[kPerLane];
#pragma unroll
  for (int i = 0; i < kPerLane; ++i) {
    const int e = lane + 32 * i;
    float x = (e < E) ? raw[i] : -INFINITY;
    if (e < E && !isfinite(x)) {
      nonfinite = true;
      if (isnan(x)) x = -INFINITY;   // keep the order total; the status reports it
    }
    key[i] = e < E ? route_key(x) : 0u;
    slot[i] = i;
  }
  // Sort them once, larger key first (odd-even transposition, swapping only on
  // a strictly smaller key, so equal keys keep ascending expert order); then
  // round j's pick is the best head over the warp, and only the winning lane
  // moves on to its next candidate.
#pragma unroll
  for (int pass = 0; pass < kPerLane; ++pass) {
#pragma unroll
    for (int i = pass & 1; i + 1 < kPerLane; i += 2) {
      if (key[i] < key[i + 1]) {
        const uint32_t tk = key[i];
        key[i] = key[i + 1];
        key[i + 1] = tk;
        const int ts = slot[i];
        slot[i] = slot[i + 1];
        slot[i + 1] = ts;
      }
    }
  }
  uint32_t my_key = 0;
  int my_idx = 0;
  for (int j = 0; j < k; ++j) {
    // the largest head key, then the lowest expert index holding it
    const uint32_t m = __reduce_max_sync(0xffffffffu, key[0]);
    const uint32_t cand = (key[0] == m && m != 0u) ? (uint32_t)(lane + 32 * slot[0]) : ~0u;
    const uint32_t win = __reduce_min_sync(0xffffffffu, cand);
    if (lane == j) {
      my_key = m;
      my_idx = (int)win;
    }
    if (m != 0u && (int)(win & 31u) == lane) {
#pragma unroll
      for (int i = 0; i + 1 < kPerLane; ++i) {
        key[i] = key[i + 1];
        slot[i] = slot[i + 1];
      }
      key[kPerLane - 1] = 0u;
    }
  }
  const float my_sel = route_key_value(my_key);
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
