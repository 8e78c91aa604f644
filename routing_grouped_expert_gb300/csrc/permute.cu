// Step 2: per-expert counts, exclusive scan, and the stable counting-sort
// scatter into per-expert groups ("MegaScale-Infer", §3.4 Fused Kernels,
// steps (2) and (4)).  Inside an expert, assignments a = t*k + j keep
// ascending a, i.e. order by token then top-k position ("MegaFlux", §A.2).
//
// Three kernels, all deterministic (no order-dependent atomics):
//   count/route : histogram of each chunk of assignments (order-free atomics
//                 on integers only);
//   scan        : per-expert prefix over chunks -> each chunk's base position,
//                 exclusive scan over experts -> offsets, plus the token-block
//                 plan (blocks of <= 128 rows per expert, "MegaFlux", §3.1);
//   scatter     : rank of each assignment among equal experts inside its
//                 chunk (warp match + per-warp counts), base + rank.
#include "moe_common.cuh"
#include "route_token.cuh"

namespace moe {
namespace {

constexpr int kScanThreads = 1024;

// Exclusive scan of one int per thread over a block of kScanThreads threads.
__device__ __forceinline__ int block_exclusive_scan(int v, int* total, int* warp_sums) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += u;
  }
  __syncthreads();   // warp_sums may be in use by a previous call
  if (lane == 31) warp_sums[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
    int wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += u;
    }
    warp_sums[lane] = wi - w;   // exclusive prefix of warp totals
    if (lane == 31) warp_sums[32] = wi;
  }
  __syncthreads();
  *total = warp_sums[32];
  return warp_sums[warp] + incl - v;
}

// counts -> block_off (exclusive prefix of ceil(count / beta)),
// num_blocks, and block_expert[b] = expert of block b.
__device__ __forceinline__ void write_block_plan(int e, int E, int cnt, int beta,
                                                 int32_t* block_off, int32_t* num_blocks,
                                                 int32_t* block_expert, int* warp_sums) {
  const int nb = (e < E) ? (cnt + beta - 1) / beta : 0;
  int total_nb;
  const int boff = block_exclusive_scan(nb, &total_nb, warp_sums);
  if (e < E) {
    block_off[e] = boff;
    for (int b = 0; b < nb; ++b) block_expert[boff + b] = e;
  }
  if (threadIdx.x == 0) {
    block_off[E] = total_nb;
    *num_blocks = total_nb;
  }
}

// The chunk table [C][E] is staged in shared memory when it fits (every
// thread's loads in flight at once, instead of C / 8 dependent rounds of loads
// per expert); larger tables are read in place.
constexpr int kScanSmemMax = 160 * 1024;
__host__ __device__ inline bool scan_in_smem(int C, int E) {
  return (size_t)C * E * 4 <= kScanSmemMax;
}

__global__ void __launch_bounds__(kScanThreads)
scan_kernel(int32_t* __restrict__ chunk_hist, int C, int E, int32_t* __restrict__ counts,
            int32_t* __restrict__ offsets, int32_t* __restrict__ block_off,
            int32_t* __restrict__ num_blocks, int32_t* __restrict__ block_expert, int beta) {
  __shared__ int warp_sums[33];
  extern __shared__ int hist_s[];   // [C][E] when staged
  pdl_wait();
  pdl_trigger();
  const int e = threadIdx.x;
  constexpr int kBatch = 8;   // loads in flight per thread
  if (scan_in_smem(C, E)) {
    const int n = C * E;
    for (int i0 = threadIdx.x; i0 < n; i0 += kBatch * kScanThreads) {
      int v[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int i = i0 + b * kScanThreads;
        v[b] = i < n ? chunk_hist[i] : 0;
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        const int i = i0 + b * kScanThreads;
        if (i < n) hist_s[i] = v[b];
      }
    }
    __syncthreads();
    int cnt = 0;
    if (e < E)
      for (int c = 0; c < C; ++c) cnt += hist_s[c * E + e];
    int total;
    const int off = block_exclusive_scan(e < E ? cnt : 0, &total, warp_sums);
    if (e < E) {
      counts[e] = cnt;
      offsets[e] = off;
      // chunk c's rows of expert e start at off + (its rows in chunks < c)
      int run = off;
      for (int c = 0; c < C; ++c) {
        const int v = hist_s[c * E + e];
        chunk_hist[(size_t)c * E + e] = run;
        run += v;
      }
    }
    if (e == 0) offsets[E] = total;
    write_block_plan(e, E, cnt, beta, block_off, num_blocks, block_expert, warp_sums);
    return;
  }
  int cnt = 0;
  if (e < E) {
    // the expert's count over all chunks (loads only, batched)
    for (int c0 = 0; c0 < C; c0 += kBatch) {
      int v[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) v[i] = c0 + i < C ? chunk_hist[(size_t)(c0 + i) * E + e] : 0;
#pragma unroll
      for (int i = 0; i < kBatch; ++i) cnt += v[i];
    }
  }
  int total;
  const int off = block_exclusive_scan(e < E ? cnt : 0, &total, warp_sums);
  if (e < E) {
    counts[e] = cnt;
    offsets[e] = off;
    // chunk c's rows of expert e start at off + (its rows in chunks < c)
    int run = off;
    for (int c0 = 0; c0 < C; c0 += kBatch) {
      int v[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) v[i] = c0 + i < C ? chunk_hist[(size_t)(c0 + i) * E + e] : 0;
#pragma unroll
      for (int i = 0; i < kBatch; ++i) {
        if (c0 + i < C) chunk_hist[(size_t)(c0 + i) * E + e] = run;
        run += v[i];
      }
    }
  }
  if (e == 0) offsets[E] = total;
  write_block_plan(e, E, cnt, beta, block_off, num_blocks, block_expert, warp_sums);
}

// The block plan of caller-supplied offsets (moe_grouped_ffn).  Offsets that
// are not a valid grouping of P rows (offsets[0] != 0, a decrease, or
// offsets[E] > P) would size the plan past its table: they set
// MOE_ERR_INVALID_ARG and leave an empty plan, so the GEMMs do nothing.
__global__ void __launch_bounds__(kScanThreads)
plan_kernel(const int32_t* __restrict__ offsets, int E, int P, int32_t* __restrict__ block_off,
            int32_t* __restrict__ num_blocks, int32_t* __restrict__ block_expert, int beta,
            int* __restrict__ status) {
  __shared__ int warp_sums[33];
  __shared__ int bad;
  const int e = threadIdx.x;
  if (e == 0) bad = offsets[0] != 0 || offsets[E] > P;
  __syncthreads();
  const int cnt = (e < E) ? offsets[e + 1] - offsets[e] : 0;
  if (cnt < 0) bad = 1;
  __syncthreads();
  if (bad) {
    if (e == 0) {
      if (status != nullptr) set_status(status, MOE_ERR_INVALID_ARG);
      block_off[E] = 0;
      *num_blocks = 0;
    }
    return;
  }
  write_block_plan(e, E, cnt, beta, block_off, num_blocks, block_expert, warp_sums);
}

// An assignment whose expert index is out of range takes no position:
// dest_of[a] = -1, and the positions past the valid ones, [offsets[E], P),
// hold -1 in sorted_src (the gather and the combine skip both).
__global__ void __launch_bounds__(kChunkAssign)
scatter_kernel(const int32_t* __restrict__ topk_idx, int P, int E, int chunk_assign,
               const int32_t* __restrict__ chunk_base, const int32_t* __restrict__ offsets,
               int32_t* __restrict__ sorted_src, int32_t* __restrict__ dest_of) {
  extern __shared__ int cnt[];   // [warps][E]
  pdl_wait();
  pdl_trigger();
  const int nw = blockDim.x >> 5;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int i = threadIdx.x; i < nw * E; i += blockDim.x) cnt[i] = 0;
  __syncthreads();
  const int a = blockIdx.x * chunk_assign + threadIdx.x;
  int e = (threadIdx.x < chunk_assign && a < P) ? topk_idx[a] : -1;
  if (e >= E) e = -1;
  const unsigned peers = __match_any_sync(0xffffffffu, e);
  const int rank_w = __popc(peers & ((1u << lane) - 1u));
  if (e >= 0 && rank_w == 0) cnt[warp * E + e] = __popc(peers);
  __syncthreads();
  for (int x = threadIdx.x; x < E; x += blockDim.x) {
    int s = 0;
    for (int w = 0; w < nw; ++w) {
      const int v = cnt[w * E + x];
      cnt[w * E + x] = s;
      s += v;
    }
  }
  __syncthreads();
  if (e >= 0) {
    const int pos = chunk_base[(size_t)blockIdx.x * E + e] + cnt[warp * E + e] + rank_w;
    sorted_src[pos] = a;
    dest_of[a] = pos;
  } else if (threadIdx.x < chunk_assign && a < P) {
    dest_of[a] = -1;
  }
  // the valid assignments fill [0, offsets[E]); mark the rest of sorted_src
  if (threadIdx.x < chunk_assign && a < P && a >= offsets[E]) sorted_src[a] = -1;
}

// Small batches (T*k <= kSmallRouteAssign, E <= kSmallRouteExperts): routing,
// counts, scan, block plan and the stable scatter in one launch, with the
// same results as the route, scan and scatter kernels.  Every CTA routes 32
// tokens (one per warp, as the route kernel); the CTA that finishes last --
// each takes a ticket from a counter after a fence, and the last ticket
// holder goes on, so no CTA waits for another -- counts, scans and
// scatters all T*k assignments: thread a ranks assignment a among the equal
// experts of its warp (warp match), and the per-warp counts give each warp's
// base inside the expert, i.e. ascending a within every expert, as in the
// chunked kernels.  It then zeroes the counter for the next launch.
constexpr int kSmallRouteThreads = 1024;

template <int kPerLane>
__global__ void __launch_bounds__(kSmallRouteThreads)
route_permute_small_kernel(const float* __restrict__ logits, int T, int E, int k, int beta,
                           int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                           int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
                           int32_t* __restrict__ block_off, int32_t* __restrict__ num_blocks,
                           int32_t* __restrict__ block_expert, int32_t* __restrict__ sorted_src,
                           int32_t* __restrict__ dest_of, int* __restrict__ ticket,
                           int* __restrict__ status) {
  __shared__ int cnt[32 * kSmallRouteExperts];   // [warp][expert]: count, then base
  __shared__ int off_s[kSmallRouteExperts];
  __shared__ int warp_sums[33];
  __shared__ int last;
  // first kernel of the fused chain (launched in stream order)
  pdl_trigger();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int t = blockIdx.x * (kSmallRouteThreads / 32) + warp;
  if (t < T) {
    int my_idx;
    float my_w;
    const bool nonfinite =
        route_token<kPerLane>(logits + (size_t)t * E, E, k, lane, &my_idx, &my_w);
    if (lane < k) {
      topk_idx[(size_t)t * k + lane] = my_idx;
      topk_w[(size_t)t * k + lane] = my_w;
    }
    if (nonfinite && lane == 0) set_status(status, MOE_ERR_NONFINITE);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();   // this CTA's picks are visible before its ticket
    last = atomicAdd(ticket, 1) == (int)gridDim.x - 1;
  }
  __syncthreads();
  if (!last) return;
  __threadfence();   // every other CTA's picks, published before their tickets
  for (int i = threadIdx.x; i < 32 * E; i += kSmallRouteThreads) cnt[i] = 0;
  __syncthreads();
  // counts per warp of assignments, rank inside the warp
  const int P = T * k;
  const int a = threadIdx.x;
  int e = a < P ? __ldcg(topk_idx + a) : -1;
  if (e >= E) e = -1;
  const unsigned peers = __match_any_sync(0xffffffffu, e);
  const int rank_w = __popc(peers & ((1u << lane) - 1u));
  if (e >= 0 && rank_w == 0) cnt[warp * E + e] = __popc(peers);
  __syncthreads();
  // per expert: the warps' bases (prefix over warps) and the total
  int total_e = 0;
  if (threadIdx.x < E) {
    int run = 0;
    for (int w = 0; w < 32; ++w) {
      const int v = cnt[w * E + threadIdx.x];
      cnt[w * E + threadIdx.x] = run;
      run += v;
    }
    total_e = run;
  }
  int total;
  const int off = block_exclusive_scan(threadIdx.x < E ? total_e : 0, &total, warp_sums);
  if (threadIdx.x < E) {
    counts[threadIdx.x] = total_e;
    offsets[threadIdx.x] = off;
    off_s[threadIdx.x] = off;
  }
  if (threadIdx.x == 0) offsets[E] = total;
  write_block_plan(threadIdx.x, E, total_e, beta, block_off, num_blocks, block_expert,
                   warp_sums);
  __syncthreads();
  // the stable scatter, with the -1 markers of the chunked kernels
  if (e >= 0) {
    const int pos = off_s[e] + cnt[warp * E + e] + rank_w;
    sorted_src[pos] = a;
    dest_of[a] = pos;
  } else if (a < P) {
    dest_of[a] = -1;
  }
  if (a < P && a >= total) sorted_src[a] = -1;
  if (threadIdx.x == 0) *ticket = 0;   // for the next launch
}

// x_perm[p] = x[sorted_src[p] / k]: one warp per segment of 4 x 32 16-byte
// vectors of a row (segments grid-strided), all four loads of a lane in
// flight before its stores.  Positions holding -1 (no assignment) are skipped.
constexpr int kGatherUnroll = 4;
__global__ void __launch_bounds__(256)
gather_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ sorted_src, int P,
              int H, int k, __nv_bfloat16* __restrict__ x_perm) {
  pdl_wait();
  pdl_trigger();
  const int nv = H / 8;
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const int upr = (nv + 32 * kGatherUnroll - 1) / (32 * kGatherUnroll);   // segments per row
  const long long units = (long long)P * upr;
  for (long long w = blockIdx.x * wpb + (threadIdx.x >> 5); w < units;
       w += (long long)gridDim.x * wpb) {
    const int row = (int)(w / upr);
    const int v0 = (int)(w - (long long)row * upr) * 32 * kGatherUnroll + lane;
    const int a = __ldg(sorted_src + row);
    if (a < 0 || a >= P) continue;   // no assignment at this position
    const int4* src = reinterpret_cast<const int4*>(x) + (size_t)(a / k) * nv;
    int4* dst = reinterpret_cast<int4*>(x_perm) + (size_t)row * nv;
    int4 r[kGatherUnroll];
#pragma unroll
    for (int u = 0; u < kGatherUnroll; ++u)
      if (v0 + 32 * u < nv) r[u] = __ldg(src + v0 + 32 * u);
#pragma unroll
    for (int u = 0; u < kGatherUnroll; ++u)
      if (v0 + 32 * u < nv) dst[v0 + 32 * u] = r[u];
  }
}

// x_perm[dest_of[t * k + j]] = x[t] for every slot j < k: each row of x is
// read once (one warp per segment of 4 x 32 16-byte vectors, segments
// grid-strided, all four loads of a lane in flight) and stored at its k
// places in expert order.
__global__ void __launch_bounds__(256)
gather_tokens_kernel(const __nv_bfloat16* __restrict__ x, const int32_t* __restrict__ dest_of,
                     int T, int H, int k, __nv_bfloat16* __restrict__ x_perm) {
  pdl_wait();
  pdl_trigger();
  const int nv = H / 8;
  const int lane = threadIdx.x & 31;
  const int wpb = blockDim.x >> 5;
  const int upr = (nv + 32 * kGatherUnroll - 1) / (32 * kGatherUnroll);   // segments per row
  const long long units = (long long)T * upr;
  for (long long w = blockIdx.x * wpb + (threadIdx.x >> 5); w < units;
       w += (long long)gridDim.x * wpb) {
    const int t = (int)(w / upr);
    const int v0 = (int)(w - (long long)t * upr) * 32 * kGatherUnroll + lane;
    const int4* src = reinterpret_cast<const int4*>(x) + (size_t)t * nv;
    int4 r[kGatherUnroll];
#pragma unroll
    for (int u = 0; u < kGatherUnroll; ++u)
      if (v0 + 32 * u < nv) r[u] = __ldg(src + v0 + 32 * u);
    for (int j = 0; j < k; ++j) {
      const int p = __ldg(dest_of + (size_t)t * k + j);
      if (p < 0) continue;   // an assignment that took no position
      int4* dst = reinterpret_cast<int4*>(x_perm) + (size_t)p * nv;
#pragma unroll
      for (int u = 0; u < kGatherUnroll; ++u)
        if (v0 + 32 * u < nv) dst[v0 + 32 * u] = r[u];
    }
  }
}

}  // namespace

cudaError_t launch_scan(int32_t* chunk_hist, int C, int E, int32_t* counts, int32_t* offsets,
                        int32_t* block_off, int32_t* num_blocks, int32_t* block_expert,
                        int beta, cudaStream_t s, bool pdl) {
  const size_t smem = scan_in_smem(C, E) ? (size_t)C * E * 4 : 0;
  if (smem > 48 * 1024) {
    static const cudaError_t attr = cudaFuncSetAttribute(
        scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kScanSmemMax);
    if (attr != cudaSuccess) return attr;
  }
  return launch_k(scan_kernel, dim3(1), dim3(kScanThreads), smem, s, pdl, chunk_hist, C, E, counts,
                  offsets, block_off, num_blocks, block_expert, beta);
}

cudaError_t launch_route_permute_small(const float* logits, int T, int E, int k, int beta,
                                      int32_t* topk_idx, float* topk_w, int32_t* counts,
                                      int32_t* offsets, int32_t* block_off, int32_t* num_blocks,
                                      int32_t* block_expert, int32_t* sorted_src,
                                      int32_t* dest_of, int* ticket, int* status,
                                      cudaStream_t s) {
  if (!route_permute_small_ok(T, E, k)) return cudaErrorInvalidValue;
  if (T == 0) return cudaSuccess;
  const int grid = (T + kSmallRouteThreads / 32 - 1) / (kSmallRouteThreads / 32);
#define MOE_SMALL_ROUTE(N)                                                                   \
  route_permute_small_kernel<N><<<grid, kSmallRouteThreads, 0, s>>>(                           \
      logits, T, E, k, beta, topk_idx, topk_w, counts, offsets, block_off, num_blocks,         \
      block_expert, sorted_src, dest_of, ticket, status)
  if (E <= 32) MOE_SMALL_ROUTE(1);
  else if (E <= 64) MOE_SMALL_ROUTE(2);
  else if (E <= 128) MOE_SMALL_ROUTE(4);
  else MOE_SMALL_ROUTE(8);
#undef MOE_SMALL_ROUTE
  return cudaGetLastError();
}

cudaError_t launch_plan(const int32_t* offsets, int E, int P, int32_t* block_off,
                        int32_t* num_blocks, int32_t* block_expert, int beta, int* status,
                        cudaStream_t s) {
  plan_kernel<<<1, kScanThreads, 0, s>>>(offsets, E, P, block_off, num_blocks, block_expert, beta,
                                         status);
  return cudaGetLastError();
}

cudaError_t launch_scatter(const int32_t* topk_idx, int T, int E, int k,
                           const int32_t* chunk_base, const int32_t* offsets,
                           int32_t* sorted_src, int32_t* dest_of, cudaStream_t s, bool pdl) {
  if (T == 0) return cudaSuccess;
  const int C = num_chunks(T, k);
  const int chunk_assign = tokens_per_chunk(k) * k;
  const size_t smem = (size_t)(kChunkAssign / 32) * E * sizeof(int);
  // 16 warps x E counters; above the default 48 KB when E > 768.
  cudaError_t err = cudaFuncSetAttribute(
      scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
      (int)((kChunkAssign / 32) * MOE_MAX_EXPERTS * sizeof(int)));
  if (err != cudaSuccess) return err;
  return launch_k(scatter_kernel, dim3(C), dim3(kChunkAssign), smem, s, pdl, topk_idx, T * k, E,
                  chunk_assign, chunk_base, offsets, sorted_src, dest_of);
}

cudaError_t launch_gather(const __nv_bfloat16* x, const int32_t* sorted_src, int P, int H, int k,
                          __nv_bfloat16* x_perm, cudaStream_t s, bool pdl) {
  if (P == 0) return cudaSuccess;
  const long long segs = (long long)P * ((H / 8 + 127) / 128);
  const long long want = (segs + 7) / 8;                  // 8 warps (segments) per CTA
  const int grid = (int)(want < 8LL * device_sm_count() ? want : 8LL * device_sm_count());
  return launch_k(gather_kernel, dim3(grid), dim3(256), 0, s, pdl, x, sorted_src, P, H, k,
                  x_perm);
}

cudaError_t launch_gather_tokens(const __nv_bfloat16* x, const int32_t* dest_of, int T, int H,
                                 int k, __nv_bfloat16* x_perm, cudaStream_t s, bool pdl) {
  if (T == 0) return cudaSuccess;
  const long long segs = (long long)T * ((H / 8 + 127) / 128);
  const long long want = (segs + 7) / 8;                  // 8 warps (segments) per CTA
  const int grid = (int)(want < 8LL * device_sm_count() ? want : 8LL * device_sm_count());
  return launch_k(gather_tokens_kernel, dim3(grid), dim3(256), 0, s, pdl, x, dest_of, T, H, k,
                  x_perm);
}

}  // namespace moe
