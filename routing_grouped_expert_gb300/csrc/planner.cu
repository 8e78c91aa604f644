// The expert-replica planner on the device ("MegaFlux: Skew-Resilient MoE
// Megakernels via Pipelined Expert Replication", §3.1 Planner: replica
// placement and token-block assignment; §A.1 Greedy placement and
// refinement; §A.2 Reduction-aware planning and routed-assignment ordering).
//
// From the per-expert row counts of a routing, for G expert-parallel GPUs
// that each own a contiguous range of experts:
//   1. blocks b_e = ceil(c_e / beta), the load proxy; tau = ceil(sum b / G);
//   2. q0: every block on its expert's owner;
//   3. four bounded greedy searches from q0 -- donor priority (overloaded GPUs
//      by load, or (GPU, expert) pairs by block count) x fan-out (one new
//      replica per expert per round, or several) -- each moving blocks of
//      overloaded GPUs to GPUs that hold the expert, else to a new replica on
//      the least-loaded GPU below tau with a free slot, for at most s + 2
//      rounds (s = the replica budget per GPU) or until a round moves nothing;
//   4. the candidate with the smallest maximum load wins, then the one with
//      fewer replicas, then the earlier search;
//   5. refinement: drop replicas the other holders can absorb without
//      exceeding the maximum load, then move single blocks between holders of
//      an expert whose loads differ by two or more;
//   6. with a reduction penalty lambda (backward plans): remove, from the GPU
//      with the largest load + lambda * (remote replicas of its experts), its
//      remote replica with the smallest allocation below lambda, while it has
//      one; keep the result only if its penalised maximum is below that of q0,
//      else the plan is q0;
//   7. each expert's rows (routed order) are cut into its blocks and handed to
//      its holders in ascending GPU order.
// Ties always go to the lower GPU index, then the lower expert.  The plan is a
// deterministic function of the counts.
//
// One CTA of four warps: warp w runs search w (its lane 0 walks the plan;
// the lanes sort each round's donor list together), then warp 0 refines.
// Plans live in the caller's workspace: per search n[E][G] block counts, a
// holder mask per expert, loads and replica counts per GPU.
#include "moe_common.cuh"

namespace moe {
namespace {

constexpr int kSearches = 4;
constexpr int kPlanThreads = 32 * kSearches;

struct PlanBuf {
  int* n;          // [E][G] blocks of expert e on GPU g
  uint64_t* hold;  // [E] GPUs holding e (bit g)
  int* L;          // [G] load
  int* used;       // [G] replica slots in use
  int* newr;       // [E] new replicas of e this round
  long long* key;  // [E * G] sort keys of this round's (donor, expert) pairs
  int* cand;       // [E * G] those pairs, e * G + d, in the order found
  int* order;      // [E * G] the pairs in processing order: d * E + e
};

__device__ __forceinline__ int owner_of(int e, int E, int G) {
  return (int)((long long)e * G / E);
}

// The plan's buffers inside the workspace, slot i (0..3 searches, 4 final,
// 5 q0 scratch).
__device__ PlanBuf plan_buf(char* ws, int i, int E, int G) {
  const size_t eg = (size_t)E * G;
  const size_t per = align_up(eg * 4, 256) + align_up((size_t)E * 8, 256) +
                     2 * align_up((size_t)G * 4, 256) + align_up((size_t)E * 4, 256) +
                     align_up(eg * 8, 256) + 2 * align_up(eg * 4, 256);
  char* p = ws + per * i;
  PlanBuf b;
  b.n = reinterpret_cast<int*>(p);
  p += align_up(eg * 4, 256);
  b.hold = reinterpret_cast<uint64_t*>(p);
  p += align_up((size_t)E * 8, 256);
  b.L = reinterpret_cast<int*>(p);
  p += align_up((size_t)G * 4, 256);
  b.used = reinterpret_cast<int*>(p);
  p += align_up((size_t)G * 4, 256);
  b.newr = reinterpret_cast<int*>(p);
  p += align_up((size_t)E * 4, 256);
  b.key = reinterpret_cast<long long*>(p);
  p += align_up(eg * 8, 256);
  b.cand = reinterpret_cast<int*>(p);
  p += align_up(eg * 4, 256);
  b.order = reinterpret_cast<int*>(p);
  return b;
}

// q0 into plan buffer `b` (warp-cooperative).
__device__ void init_q0(PlanBuf b, const int* blocks, int E, int G, int lane) {
  for (int i = lane; i < E * G; i += 32) {
    const int e = i / G, g = i - e * G;
    b.n[i] = g == owner_of(e, E, G) ? blocks[e] : 0;
  }
  for (int e = lane; e < E; e += 32) b.hold[e] = 1ull << owner_of(e, E, G);
  __syncwarp();
  for (int g = lane; g < G; g += 32) {
    int s = 0;
    for (int e = 0; e < E; ++e) s += b.n[e * G + g];
    b.L[g] = s;
    b.used[g] = 0;
  }
  __syncwarp();
}

__device__ void copy_plan(PlanBuf dst, PlanBuf src, int E, int G, int lane) {
  for (int i = lane; i < E * G; i += 32) dst.n[i] = src.n[i];
  for (int e = lane; e < E; e += 32) dst.hold[e] = src.hold[e];
  for (int g = lane; g < G; g += 32) {
    dst.L[g] = src.L[g];
    dst.used[g] = src.used[g];
  }
  __syncwarp();
}

__device__ __forceinline__ bool holds(const PlanBuf& b, int e, int g) {
  return (b.hold[e] >> g) & 1ull;
}

// Step 3: one bounded greedy search (the whole warp calls it; lane 0 moves
// blocks, all lanes sort).  donor 0 = by GPU load, 1 = by (GPU, expert)
// block count; fanout 0 = one new replica per expert per round, 1 = several.
__device__ void greedy_search(PlanBuf b, int E, int G, int tau, int budget, int rounds, int donor,
                              int fanout, int lane) {
  for (int round = 0; round < rounds; ++round) {
    for (int e = lane; e < E; e += 32) b.newr[e] = 0;
    // the round's (donor, expert) pairs, keyed so that ascending key order is
    // the processing order; keys use the loads and counts at the round start
    int np = 0;
    if (lane == 0) {
      for (int i = 0; i < E * G; ++i) {
        const int e = i / G, d = i - e * G;
        if (b.L[d] <= tau || b.n[i] <= 0) continue;
        const long long nn = b.n[i], Ld = b.L[d];
        long long k;
        if (donor == 0) {
          // rank of d among the overloaded GPUs by (-L, d); then (-n, e)
          int rank = 0;
          for (int h = 0; h < G; ++h)
            if (b.L[h] > tau && (b.L[h] > Ld || (b.L[h] == Ld && h < d))) ++rank;
          k = ((long long)rank << 52) | ((0xFFFFFll - nn) << 20) | e;
        } else {
          k = ((0xFFFFFll - nn) << 40) | ((0xFFFFFll - Ld) << 16) | ((long long)d << 10) | e;
        }
        b.key[np] = k;
        b.cand[np] = i;
        ++np;
      }
    }
    np = __shfl_sync(0xffffffffu, np, 0);
    __syncwarp();
    for (int q = lane; q < np; q += 32) {   // keys are distinct: rank = sorted position
      const long long k = b.key[q];
      int rank = 0;
      for (int j = 0; j < np; ++j) rank += b.key[j] < k;
      const int i = b.cand[q], e = i / G, d = i - e * G;
      b.order[rank] = d * E + e;
    }
    __syncwarp();
    int moved = 0;
    if (lane == 0) {
      for (int q = 0; q < np; ++q) {
        const int d = b.order[q] / E, e = b.order[q] - d * E;
        while (b.L[d] > tau && b.n[e * G + d] > 0) {
          int r = -1;
          for (int g = 0; g < G; ++g)   // a GPU that already holds e, least loaded
            if (g != d && holds(b, e, g) && b.L[g] < tau && (r < 0 || b.L[g] < b.L[r])) r = g;
          if (r < 0) {
            if (fanout == 0 && b.newr[e] >= 1) break;
            for (int g = 0; g < G; ++g)   // a new replica
              if (!holds(b, e, g) && b.L[g] < tau && b.used[g] < budget &&
                  (r < 0 || b.L[g] < b.L[r]))
                r = g;
            if (r < 0) break;
            b.hold[e] |= 1ull << r;
            b.used[r] += 1;
            b.newr[e] += 1;
          }
          int m = b.L[d] - tau;
          m = min(m, tau - b.L[r]);
          m = min(m, b.n[e * G + d]);
          b.n[e * G + d] -= m;
          b.n[e * G + r] += m;
          b.L[d] -= m;
          b.L[r] += m;
          moved = 1;
        }
      }
    }
    moved = __shfl_sync(0xffffffffu, moved, 0);
    __syncwarp();
    if (!moved) break;
  }
}

// A replica (a non-owner holder) with no block is dropped (lane 0).
__device__ void drop_empty(PlanBuf b, int E, int G) {
  for (int e = 0; e < E; ++e)
    for (int g = 0; g < G; ++g)
      if (g != owner_of(e, E, G) && holds(b, e, g) && b.n[e * G + g] == 0) {
        b.hold[e] &= ~(1ull << g);
        b.used[g] -= 1;
      }
}

__device__ int max_load(const PlanBuf& b, int G) {
  int m = 0;
  for (int g = 0; g < G; ++g) m = max(m, b.L[g]);
  return m;
}

__device__ int replica_count(const PlanBuf& b, int E, int G) {
  int r = 0;
  for (int e = 0; e < E; ++e) r += __popcll(b.hold[e]) - 1;
  return r;
}

// Step 5 (lane 0): prune redundant replicas, then single-block moves.
__device__ void refine(PlanBuf b, int E, int G) {
  drop_empty(b, E, G);
  for (bool changed = true; changed;) {
    changed = false;
    const int M = max_load(b, G);
    // replicas in (GPU, expert) order
    for (int g = 0; g < G && !changed; ++g)
      for (int e = 0; e < E && !changed; ++e) {
        if (g == owner_of(e, E, G) || !holds(b, e, g)) continue;
        int v = b.n[e * G + g];
        long long room = 0;
        for (int h = 0; h < G; ++h)
          if (h != g && holds(b, e, h)) room += M - b.L[h];
        if (v > room) continue;
        // fill the other holders, least loaded first (ties: lower index);
        // filling one never changes the order of the ones after it
        uint64_t left = b.hold[e] & ~(1ull << g);
        while (left != 0 && v > 0) {
          int h = -1;
          for (int x = 0; x < G; ++x)
            if ((left >> x) & 1ull && (h < 0 || b.L[x] < b.L[h])) h = x;
          left &= ~(1ull << h);
          const int m = min(v, M - b.L[h]);
          b.n[e * G + h] += m;
          b.L[h] += m;
          v -= m;
        }
        b.L[g] -= b.n[e * G + g];
        b.n[e * G + g] = 0;
        b.hold[e] &= ~(1ull << g);
        b.used[g] -= 1;
        changed = true;
      }
  }
  // single blocks from a holder to another holder at least two lighter
  for (;;) {
    int g1 = -1, ee = -1, g2 = -1;
    uint64_t done = 0;   // GPUs already tried, in (-load, index) order
    for (int t = 0; t < G && g1 < 0; ++t) {
      int d = -1;
      for (int x = 0; x < G; ++x)
        if (!((done >> x) & 1ull) && (d < 0 || b.L[x] > b.L[d])) d = x;
      done |= 1ull << d;
      for (int e = 0; e < E; ++e) {
        if (b.n[e * G + d] == 0) continue;
        int r = -1;
        for (int x = 0; x < G; ++x)
          if (x != d && holds(b, e, x) && b.L[d] - b.L[x] >= 2 && (r < 0 || b.L[x] < b.L[r]))
            r = x;
        if (r >= 0) {
          g1 = d;
          ee = e;
          g2 = r;
          break;
        }
      }
    }
    if (g1 < 0) break;
    b.n[ee * G + g1] -= 1;
    b.n[ee * G + g2] += 1;
    b.L[g1] -= 1;
    b.L[g2] += 1;
  }
  drop_empty(b, E, G);
}

// max over GPUs of load + lambda * (remote replicas of experts it owns)
__device__ long long penalised_max(const PlanBuf& b, int E, int G, long long lam) {
  long long best = 0;
  for (int g = 0; g < G; ++g) {
    long long own = 0;
    for (int e = 0; e < E; ++e)
      if (owner_of(e, E, G) == g) own += __popcll(b.hold[e]) - 1;
    best = max(best, (long long)b.L[g] + lam * own);
  }
  return best;
}

// Step 6a (lane 0): reduction-aware pruning in place.
__device__ void reduction_prune(PlanBuf b, int E, int G, long long lam) {
  for (;;) {
    int sel = -1;
    long long selv = 0;
    for (int g = 0; g < G; ++g) {
      long long own = 0;
      for (int e = 0; e < E; ++e)
        if (owner_of(e, E, G) == g) own += __popcll(b.hold[e]) - 1;
      const long long v = (long long)b.L[g] + lam * own;
      if (sel < 0 || v > selv) {
        sel = g;
        selv = v;
      }
    }
    // its remote replica with the smallest allocation below lambda: (v, e, g)
    int be = -1, bg = -1, bv = 0;
    for (int e = 0; e < E; ++e) {
      if (owner_of(e, E, G) != sel) continue;
      for (int g = 0; g < G; ++g) {
        if (g == sel || !holds(b, e, g)) continue;
        const int v = b.n[e * G + g];
        if ((long long)v < lam && (be < 0 || v < bv)) {
          be = e;
          bg = g;
          bv = v;
        }
      }
    }
    if (be < 0) return;
    b.n[be * G + sel] += bv;
    b.L[sel] += bv;
    b.n[be * G + bg] = 0;
    b.L[bg] -= bv;
    b.hold[be] &= ~(1ull << bg);
    b.used[bg] -= 1;
  }
}

__global__ void __launch_bounds__(kPlanThreads)
plan_replicas_kernel(const int32_t* __restrict__ counts, int E, int G, int beta, int budget,
                     int rounds, long long lam, char* ws, int32_t* __restrict__ n_out,
                     int32_t* __restrict__ rows_out, int32_t* __restrict__ load_out,
                     int32_t* __restrict__ info) {
  __shared__ int s_tau;
  __shared__ int s_pick;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int* blocks = reinterpret_cast<int*>(ws);
  char* pws = ws + align_up((size_t)E * 4, 256);
  for (int e = threadIdx.x; e < E; e += blockDim.x) blocks[e] = (counts[e] + beta - 1) / beta;
  __syncthreads();
  if (threadIdx.x == 0) {
    long long tot = 0;
    for (int e = 0; e < E; ++e) tot += blocks[e];
    s_tau = (int)((tot + G - 1) / G);
  }
  __syncthreads();
  const int tau = s_tau;
  // steps 2-3: the four searches, one per warp
  PlanBuf mine = plan_buf(pws, warp, E, G);
  init_q0(mine, blocks, E, G, lane);
  greedy_search(mine, E, G, tau, budget, rounds, warp >> 1, warp & 1, lane);
  if (lane == 0) drop_empty(mine, E, G);
  __syncthreads();
  // step 4: the winner
  if (threadIdx.x == 0) {
    int best = 0, bm = 0, br = 0;
    for (int i = 0; i < kSearches; ++i) {
      PlanBuf c = plan_buf(pws, i, E, G);
      const int m = max_load(c, G), r = replica_count(c, E, G);
      if (i == 0 || m < bm || (m == bm && r < br)) {
        best = i;
        bm = m;
        br = r;
      }
    }
    s_pick = best;
  }
  __syncthreads();
  if (warp != 0) return;
  PlanBuf fin = plan_buf(pws, kSearches, E, G);
  copy_plan(fin, plan_buf(pws, s_pick, E, G), E, G, lane);
  int which = s_pick;
  if (lane == 0) refine(fin, E, G);
  __syncwarp();
  if (lam >= 0) {
    // step 6: reduction-aware pruning, kept only if it beats q0
    PlanBuf q0 = plan_buf(pws, kSearches + 1, E, G);
    init_q0(q0, blocks, E, G, lane);
    if (lane == 0) {
      reduction_prune(fin, E, G, lam);
      if (!(penalised_max(fin, E, G, lam) < penalised_max(q0, E, G, lam))) which = kSearches;
    }
    which = __shfl_sync(0xffffffffu, which, 0);
    if (which == kSearches) copy_plan(fin, q0, E, G, lane);
  }
  __syncwarp();
  // step 7 and the outputs
  for (int e = lane; e < E; e += 32) {
    int pos = 0;
    for (int g = 0; g < G; ++g) {
      const int v = fin.n[e * G + g];
      n_out[e * G + g] = v;
      rows_out[2 * (e * G + g)] = min(pos * beta, counts[e]);
      pos += v;
      rows_out[2 * (e * G + g) + 1] = min(pos * beta, counts[e]);
    }
  }
  for (int g = lane; g < G; g += 32) load_out[g] = fin.L[g];
  if (lane == 0) {
    info[0] = which;
    info[1] = tau;
    info[2] = replica_count(fin, E, G);
    info[3] = max_load(fin, G);
  }
}

}  // namespace

size_t plan_ws_bytes(int E, int G) {
  const size_t eg = (size_t)E * G;
  const size_t per = align_up(eg * 4, 256) + align_up((size_t)E * 8, 256) +
                     2 * align_up((size_t)G * 4, 256) + align_up((size_t)E * 4, 256) +
                     align_up(eg * 8, 256) + 2 * align_up(eg * 4, 256);
  return align_up((size_t)E * 4, 256) + per * (kSearches + 2);
}

cudaError_t launch_plan_replicas(const int32_t* counts, int E, int G, int beta, int budget,
                                 int rounds, long long lam, void* ws, int32_t* n_out,
                                 int32_t* rows_out, int32_t* load_out, int32_t* info,
                                 cudaStream_t s) {
  plan_replicas_kernel<<<1, kPlanThreads, 0, s>>>(counts, E, G, beta, budget, rounds, lam,
                                                  static_cast<char*>(ws), n_out, rows_out,
                                                  load_out, info);
  return cudaGetLastError();
}

}  // namespace moe
