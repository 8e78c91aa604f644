// Backward WGrad of the expert GEMMs ("MegaFlux", §2.1: the backward streams
// token blocks through DGrad and WGrad), per expert e over its routed rows:
//   dW2[e] = h_e^T dY_e              (kNumB = 1: A = h, B = dY)
//   dW1[e] = x_e^T dg_e, dW3[e] = x_e^T du_e   (kNumB = 2: A = x, B = dg, du)
// i.e. D[m, n] = sum over the expert's rows p of A[p, m] * B[p, n].
//
// Tile = (expert, rows m of dW, columns n of dW); K = the expert's rows in
// stages of 64.  Tile shapes: with few rows per expert, 128 rows x 256
// columns per B operand with two accumulator buffers (the epilogue of one tile
// overlaps the MMAs of the next; dW1 and dW3 in two launches); otherwise,
// with kPairM (whenever the sizes are multiples of 256), 256 x 256 (two
// 128-row A sub-tiles sharing the B columns) in one TMEM buffer, which halves
// the operand bytes staged per MMA; else 128 x 128 per B operand with two
// buffers.  Both operands are row-major [P, *] buffers read as MN-major
// tensor-core operands, one TMA box per operand and stage (a 3-D view: 64
// columns, rows, 64-column atoms).  The last stage of an expert usually runs
// past its rows into the next expert's: its MMAs stop at the last 16-row K
// group holding rows of the expert, and a warp of its own zeroes the rest of
// that group in shared memory (whole 128-byte rows, so the swizzle does not
// matter) and fences it for the tensor core before handing the stage on.
// Experts without rows get zero gradients.
//
// Warp roles: warp 0 TMA producer, warp 1 MMA (lane 0 issues), warps 2-9
// epilogue, warp 10 tail rows.  The epilogue converts 32 rows x 64 columns
// at a time to bf16 in a 128-byte-swizzled staging buffer of its own (4 KB
// per warp) and writes it with a TMA store, so the gradient leaves in whole
// lines without holding the warp; each 128-column group of the accumulator is
// handed back as soon as it is read, the next chunk read before the current
// one is stored.  Every wait is bounded and reports MOE_ERR_TIMEOUT.
#include <cuda.h>

#include "moe_common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

using namespace ptx;

constexpr int BM = kTileM;            // dW rows per MMA
constexpr int BK = 64;                // routed rows per stage
constexpr int kBox = 64 * BK * 2;     // one 64-column x 64-row box: 8 KB
constexpr int kEpiWarps = 8;
constexpr int kZeroWarp = 2 + kEpiWarps;   // clears the rows of a stage past its expert
constexpr int kThreads = 32 * (kZeroWarp + 1);
// Epilogue staging buffers per warp (each 32 rows x 64 columns); with more
// than one, a warp converts its next chunk while earlier stores still read.
#ifndef MOE_WGRAD_STG_BUFS
#define MOE_WGRAD_STG_BUFS 1
#endif
constexpr int kStgBufs = MOE_WGRAD_STG_BUFS;
constexpr int kStgBytes = 32 * 64 * 2;
constexpr int kSmemBudget = kStgBufs == 1 ? 196608 : 163840;   // operand ring
constexpr uint64_t kWaitLimitNs = 1000000000ull;

template <int kNumB, bool kPairM, int kBN_>
struct WCfg {
  static constexpr int kMS = kPairM ? 2 : 1;   // 128-row A sub-tiles
  static constexpr int kBN = kBN_;             // columns per B operand
  static constexpr int kTileRows = kMS * BM;
  static constexpr int kABytes = kMS * 2 * kBox;
  static constexpr int kBBytes = (kBN / 64) * kBox;
  static constexpr int kStageBytes = kABytes + kNumB * kBBytes;
  static constexpr int kStages = kSmemBudget / kStageBytes;
  static constexpr int kAccCols = kMS * kNumB * kBN;
  static constexpr int kAccBufs = kPairM ? 1 : 2;
  static constexpr int kRegions = kAccCols / 128;   // 128-column groups released one by one
  static constexpr int kTmemCols = kAccBufs * kAccCols;
  static constexpr int kBarOffset = kStages * kStageBytes;
  static constexpr int kStgOffset = kBarOffset + 1024;              // 1 KB-aligned for the swizzle
  static constexpr int kSmemBytes = kStgOffset + kEpiWarps * kStgBufs * kStgBytes + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  static_assert(kStages >= 2 && kStages <= 8, "stages");
  static_assert(kTmemCols == 256 || kTmemCols == 512, "TMEM allocation");
  static_assert(kBN == 128 || kBN == 256, "B tile width");
};

struct WBars {
  uint64_t full[8];
  uint64_t ready[8];   // a stage's data landed and its rows past the expert are cleared
  uint64_t empty[8];
  uint64_t acc_full[2];
  uint64_t acc_empty[2][4];   // per buffer, per 128-column group
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

struct WItem {
  int e, m0, n0, row0, rows;
};

template <int kTileRows, int kBN>
__device__ __forceinline__ WItem decode_witem(int w, int n_m, int n_n, const int32_t* offsets) {
  WItem it;
  const int per = n_m * n_n;
  it.e = w / per;
  const int r = w - it.e * per;
  // row tile outer, column tile inner: CTAs running side by side write
  // neighbouring column ranges of the same gradient rows (measured slightly
  // faster than the transposed order when experts have few rows, and within
  // noise of it when they have many)
  it.m0 = (r / n_n) * kTileRows;
  it.n0 = (r % n_n) * kBN;
  it.row0 = offsets[it.e];
  it.rows = offsets[it.e + 1] - it.row0;
  return it;
}

// Store a 2-D box from shared memory to global with an L2 cache hint (bulk
// async-group of the issuing thread); the shared source must be fenced for
// the async proxy first.
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x,
                                             int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint"
      " [%0, {%2, %3}], [%1], %4;" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(src)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void bulk_commit() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
// Until at most kPending committed stores of this thread still read shared memory.
template <int kPending>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(kPending) : "memory");
}
// Until every committed store of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <int kNumB, bool kPairM, int kBN_>
__global__ void __launch_bounds__(kThreads, 1)
wgrad_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB0,
             const __grid_constant__ CUtensorMap tmB1, const __grid_constant__ CUtensorMap tmO0,
             const __grid_constant__ CUtensorMap tmO1, const int32_t* __restrict__ offsets,
             int E, int M_total, int N_total, int* __restrict__ status) {
  using C = WCfg<kNumB, kPairM, kBN_>;
  constexpr int kBN = C::kBN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  WBars* bars = reinterpret_cast<WBars*>(smem + C::kBarOffset);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_m = M_total / C::kTileRows, n_n = N_total / kBN;
  const int total = E * n_m * n_n;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->ready[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int b = 0; b < C::kAccBufs; ++b) {
      mbar_init(&bars->acc_full[b], 1);
      for (int g = 0; g < C::kRegions; ++g) mbar_init(&bars->acc_empty[b][g], kEpiWarps);
    }
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA);
    prefetch_tmap(&tmB0);
    if (kNumB == 2) prefetch_tmap(&tmB1);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = bars->tmem_base;
  volatile int* abort_flag = &bars->abort;

  if (warp == 0) {
    // ------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_last();   // an expert's rows are re-read per tile
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
        const WItem it = decode_witem<C::kTileRows, kBN>(w, n_m, n_n, offsets);
        const int nkb = (it.rows + BK - 1) / BK;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&bars->empty[stage], phase ^ 1u, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          uint8_t* sA = smem + stage * C::kStageBytes;
          uint64_t* fb = &bars->full[stage];
          const int r = it.row0 + kb * BK;
          mbar_arrive_expect_tx(fb, C::kStageBytes);
          // one box per operand: all its 64-column atoms, 64 rows each
          tma_load_3d(sA, &tmA, fb, 0, r, it.m0 / 64, pol);
#pragma unroll
          for (int b = 0; b < kNumB; ++b)
            tma_load_3d(sA + C::kABytes + b * C::kBBytes, b == 0 ? &tmB0 : &tmB1, fb, 0, r,
                        it.n0 / 64, pol);
          ++issued;
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        set_status(status, MOE_ERR_TIMEOUT, kWaitDetailProducer);
        *abort_flag = 1;
      }
      for (int i = issued > C::kStages ? issued - C::kStages : 0; i < issued; ++i)
        mbar_wait(&bars->full[i % C::kStages], (uint32_t)((i / C::kStages) & 1), nullptr,
                  kWaitLimitNs);
    }
  } else if (warp == 1) {
    // ---------------------------------- MMA issuer (lane 0) and tail zeroing
    const uint32_t sbase = smem_u32(smem);
    const uint32_t idesc = idesc_bf16(BM, kBN, /*a_mn=*/true, /*b_mn=*/true);
    int stage = 0, acc = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
      const WItem it = decode_witem<C::kTileRows, kBN>(w, n_m, n_n, offsets);
      const int nkb = (it.rows + BK - 1) / BK;
      // The accumulator's 128-column groups are handed back by the epilogue one
      // at a time; the first stage of a tile waits for each group just before
      // its first MMA, so the next tile starts while the last one is drained.
      auto group_free = [&](int g) {
        return __all_sync(0xffffffffu, mbar_wait(&bars->acc_empty[acc][g], acc_phase ^ 1u,
                                                 abort_flag, kWaitLimitNs));
      };
      if (nkb == 0) {   // an expert with no rows: nothing to accumulate
        for (int g = 0; g < C::kRegions && ok; ++g) ok = group_free(g);
        if (!ok) break;
      }
      const uint32_t d0 = tmem_base + (uint32_t)(acc * C::kAccCols);
      for (int kb = 0; kb < nkb; ++kb) {
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&bars->ready[stage], phase, abort_flag, kWaitLimitNs))) {
          ok = false;
          break;
        }
        // the MMAs cover only the 16-row K groups holding rows of the expert
        const int valid = it.rows - kb * BK;     // rows of this expert in the stage
        const int nkk = valid >= BK ? BK / 16 : (valid + 15) >> 4;
        tc_fence_after();
        const uint32_t a0 = sbase + (uint32_t)(stage * C::kStageBytes);
        if (kb == 0) {
          // first stage: accumulator by accumulator, each once its columns are free
          // (per accumulator the K order is the same as in the later stages)
#pragma unroll
          for (int t = 0; t < C::kMS * kNumB; ++t) {
            const int ms = t / kNumB, b = t % kNumB;
            for (int g = t * (kBN / 128); g < (t + 1) * (kBN / 128) && ok; ++g) ok = group_free(g);
            if (!ok) break;
            tc_fence_after();
            if (lane == 0) {
#pragma unroll
              for (int kk = 0; kk < BK / 16; ++kk) {
                if (kk >= nkk) break;
                const uint64_t da = sdesc_sw128(a0 + ms * 2 * kBox + kk * 2048, kBox, 1024);
                const uint64_t db =
                    sdesc_sw128(a0 + C::kABytes + b * C::kBBytes + kk * 2048, kBox, 1024);
                mma_bf16_ss(d0 + (uint32_t)(t * kBN), da, db, idesc, kk ? 1u : 0u);
              }
            }
            __syncwarp();
          }
          if (!ok) break;
          if (lane == 0) mma_commit(&bars->empty[stage]);
        } else if (lane == 0) {
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            if (kk >= nkk) break;
            // both operands MN-major: 64-wide atoms 8 KB apart, 8-row groups 1 KB
            // apart, K step of 16 rows = 2 KB
#pragma unroll
            for (int ms = 0; ms < C::kMS; ++ms) {
              const uint64_t da = sdesc_sw128(a0 + ms * 2 * kBox + kk * 2048, kBox, 1024);
#pragma unroll
              for (int b = 0; b < kNumB; ++b) {
                const uint64_t db =
                    sdesc_sw128(a0 + C::kABytes + b * C::kBBytes + kk * 2048, kBox, 1024);
                mma_bf16_ss(d0 + (uint32_t)((ms * kNumB + b) * kBN), da, db, idesc, 1u);
              }
            }
          }
          mma_commit(&bars->empty[stage]);
        }
        __syncwarp();
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!ok) break;
      if (lane == 0) mma_commit(&bars->acc_full[acc]);   // also for an expert with no rows
      __syncwarp();
      if (++acc == C::kAccBufs) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (lane == 0) {
      if (!ok) {
        set_status(status, MOE_ERR_TIMEOUT, kWaitDetailMma);
        *abort_flag = 1;
      }
      mma_commit(&bars->drain);
      if (!mbar_wait(&bars->drain, 0, nullptr, kWaitLimitNs))
        set_status(status, MOE_ERR_TIMEOUT, kWaitDetailDrain);
    }
  } else if (warp == kZeroWarp) {
    // ------------------------------------------------- tail rows of a stage
    // The last stage of an expert's tile ends inside a 16-row K group or
    // runs past it: rows past the expert in the last group the MMAs read (the
    // next expert's, or the zero fill past the end) are cleared in every box
    // of the stage (whole 128-byte rows, so the swizzle does not matter) and
    // fenced for the tensor core before the stage is handed to the MMA warp.
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
      const WItem it = decode_witem<C::kTileRows, kBN>(w, n_m, n_n, offsets);
      const int nkb = (it.rows + BK - 1) / BK;
      for (int kb = 0; kb < nkb; ++kb) {
        if (!__all_sync(0xffffffffu,
                        mbar_wait(&bars->full[stage], phase, abort_flag, kWaitLimitNs))) {
          ok = false;
          break;
        }
        const int valid = it.rows - kb * BK;
        const int pad = (((valid + 15) >> 4) << 4) - valid;   // 0..15 when valid < BK
        if (valid < BK && pad > 0) {
          uint4* base = reinterpret_cast<uint4*>(smem + stage * C::kStageBytes) + valid * 8;
#pragma unroll
          for (int bx = 0; bx < C::kStageBytes / kBox; ++bx)
            for (int i = lane; i < pad * 8; i += 32)
              base[bx * (kBox / 16) + i] = make_uint4(0, 0, 0, 0);
          fence_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->ready[stage]);
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (!ok && lane == 0) {
      set_status(status, MOE_ERR_TIMEOUT, kWaitDetailMma);
      *abort_flag = 1;
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;            // TMEM lane quadrant this warp may read
    const int half = (warp - 2) >> 2;  // which alternate 64-column chunks it takes
    uint8_t* stg0 = smem + C::kStgOffset + (warp - 2) * kStgBufs * kStgBytes;
    int nstg = 0;   // chunks staged by this warp so far
    const uint64_t pol_out = policy_evict_first();   // written once, not read here
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < total; w += gridDim.x) {
      const WItem it = decode_witem<C::kTileRows, kBN>(w, n_m, n_n, offsets);
      if (!__all_sync(0xffffffffu, mbar_wait(&bars->acc_full[acc], acc_phase, abort_flag,
                                             kWaitLimitNs))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * C::kAccCols);
      // The warp's chunks of the tile: chunk i is accumulator t = i / kCPT,
      // columns 64 * half + 128 * (i % kCPT), i.e. the warp's part of
      // 128-column group i.  Chunk i + 1 is read from TMEM and its group
      // handed back before chunk i is converted and stored, so the next tile's
      // MMAs wait for the drain one chunk less.
      constexpr int kCPT = kBN / 128;
      constexpr int kNC = C::kMS * kNumB * kCPT;
      uint32_t v[2][64];
      auto read_chunk = [&](int i, uint32_t* dst) {
        if (it.rows > 0) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tmem_ld_32x32b_x16(tb + (i / kCPT) * kBN + 64 * half + 128 * (i % kCPT) + 16 * j,
                               *reinterpret_cast<uint32_t(*)[16]>(dst + 16 * j));
          tmem_ld_wait();
        } else {
#pragma unroll
          for (int c = 0; c < 64; ++c) dst[c] = 0u;
        }
        // this warp's part of the 128-column group is read: hand it back
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->acc_empty[acc][i]);
      };
      read_chunk(0, v[0]);
#pragma unroll
      for (int i = 0; i < kNC; ++i) {
        if (i + 1 < kNC) read_chunk(i + 1, v[(i + 1) & 1]);
        const uint32_t* src = v[i & 1];
        const int t = i / kCPT, ms = t / kNumB, b = t % kNumB;
        const int orow = it.e * M_total + it.m0 + ms * BM + q * 32;   // the warp's first row
        // the store that last used this buffer has read it
        if (lane == 0) bulk_wait_read<kStgBufs - 1>();
        __syncwarp();
        uint8_t* stg = stg0 + (nstg++ % kStgBufs) * kStgBytes;
        // row `lane` of the box: 16-byte chunk j sits at j ^ (row & 7) (128B swizzle)
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          uint4 pk;
          __nv_bfloat162* p2 = reinterpret_cast<__nv_bfloat162*>(&pk);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            p2[c] = __floats2bfloat162_rn(__uint_as_float(src[8 * j + 2 * c]),
                                          __uint_as_float(src[8 * j + 2 * c + 1]));
          *reinterpret_cast<uint4*>(stg + lane * 128 + ((j ^ (lane & 7)) << 4)) = pk;
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d(b == 0 ? &tmO0 : &tmO1, stg, it.n0 + 64 * half + 128 * (i % kCPT), orow,
                       pol_out);
          bulk_commit();
        }
      }
      if (++acc == C::kAccBufs) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (lane == 0) {
      bulk_wait_all();   // every gradient tile written before the CTA leaves
      if (!ok) {
        set_status(status, MOE_ERR_TIMEOUT, kWaitDetailEpilogue);
        *abort_flag = 1;
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// Row-major [P, cols] buffer as MN-major operand boxes of `atoms` 64-column
// atoms x 64 rows: a 3-D view (64 columns, rows, atoms) whose box lands in
// shared memory atom by atom, each atom 64 rows of 128 bytes, as the
// tensor-core descriptors expect; one TMA instruction moves the whole box.
bool map_rows64(CUtensorMap* m, const void* X, int cols, int P, int atoms) {
  const cuuint64_t d[3] = {64, (cuuint64_t)P, (cuuint64_t)cols / 64};
  const cuuint64_t st[2] = {(cuuint64_t)cols * 2, 128};
  const cuuint32_t box[3] = {64, (cuuint32_t)BK, (cuuint32_t)atoms};
  return make_tensor_map_bf16(m, X, 3, reinterpret_cast<const unsigned long long*>(d),
                              reinterpret_cast<const unsigned long long*>(st),
                              reinterpret_cast<const unsigned int*>(box));
}

// Gradient [E, M, N] (N contiguous) as 2-D [E * M, N] store boxes of 32 rows
// x 64 columns.
bool map_grad_out(CUtensorMap* m, const void* W, int E, int M, int N) {
  const cuuint64_t d[2] = {(cuuint64_t)N, (cuuint64_t)E * M};
  const cuuint64_t st[1] = {(cuuint64_t)N * 2};
  const cuuint32_t box[2] = {64, 32};
  return make_tensor_map_bf16(m, W, 2, reinterpret_cast<const unsigned long long*>(d),
                              reinterpret_cast<const unsigned long long*>(st),
                              reinterpret_cast<const unsigned int*>(box));
}

template <int kNumB, bool kPairM, int kBN>
cudaError_t launch_w(const __nv_bfloat16* A, int a_cols, const __nv_bfloat16* B0,
                     const __nv_bfloat16* B1, int b_cols, int P, const int32_t* offsets, int E,
                     __nv_bfloat16* o0, __nv_bfloat16* o1, int* status, cudaStream_t s) {
  using C = WCfg<kNumB, kPairM, kBN>;
  const int M_total = a_cols, N_total = b_cols;
  CUtensorMap ma, mb0, mb1, mo0, mo1;
  if (!map_rows64(&ma, A, a_cols, P, 2 * C::kMS) || !map_rows64(&mb0, B0, b_cols, P, kBN / 64) ||
      !map_rows64(&mb1, B1, b_cols, P, kBN / 64) ||
      !map_grad_out(&mo0, o0, E, M_total, N_total) || !map_grad_out(&mo1, o1, E, M_total, N_total))
    return cudaErrorInvalidValue;
  auto kern = wgrad_kernel<kNumB, kPairM, kBN>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (err != cudaSuccess) return err;
  const long long items = (long long)E * (M_total / C::kTileRows) * (N_total / C::kBN);
  const int grid = (int)(items < device_sm_count() ? items : device_sm_count());
  kern<<<grid, kThreads, C::kSmemBytes, s>>>(ma, mb0, mb1, mo0, mo1, offsets, E, M_total,
                                             N_total, status);
  return cudaGetLastError();
}


// Wide tiles up to this many routed rows per expert on average.
#ifndef MOE_WGRAD_WIDE_MAX_ROWS
#define MOE_WGRAD_WIDE_MAX_ROWS 64
#endif
bool wgrad_wide(int P, int E) { return (long long)P <= (long long)MOE_WGRAD_WIDE_MAX_ROWS * E; }

}  // namespace

cudaError_t launch_wgrad(const __nv_bfloat16* x_perm, const __nv_bfloat16* h,
                         const __nv_bfloat16* dY, const __nv_bfloat16* dg,
                         const __nv_bfloat16* du, const int32_t* offsets, int P, int H, int F,
                         int E, __nv_bfloat16* dW1, __nv_bfloat16* dW3, __nv_bfloat16* dW2,
                         int* status, cudaStream_t s) {
  if (P == 0) return cudaSuccess;
  // Tile shapes.  Wide: 128 rows x 256 columns per launch and B operand (dW1
  // and dW3 in two launches), two accumulator buffers, so the epilogue of a
  // tile runs under the MMAs of the next.  Paired: 256 x 256 (dW2) or
  // 256 x 128 x 2 (dW1, dW3) in one buffer, fewer operand bytes per MMA but the
  // epilogue only partly hidden.
  const bool wide = wgrad_wide(P, E);
  cudaError_t err;
  if (wide && H % 256 == 0)
    err = launch_w<1, false, 256>(h, F, dY, dY, H, P, offsets, E, dW2, dW2, status, s);
  else if (H % 256 == 0 && F % 256 == 0)
    err = launch_w<1, true, 256>(h, F, dY, dY, H, P, offsets, E, dW2, dW2, status, s);
  else
    err = launch_w<1, false, 128>(h, F, dY, dY, H, P, offsets, E, dW2, dW2, status, s);
  if (err != cudaSuccess) return err;
  if (wide && F % 256 == 0) {
    err = launch_w<1, false, 256>(x_perm, H, dg, dg, F, P, offsets, E, dW1, dW1, status, s);
    if (err != cudaSuccess) return err;
    return launch_w<1, false, 256>(x_perm, H, du, du, F, P, offsets, E, dW3, dW3, status, s);
  }
  return H % 256 == 0
             ? launch_w<2, true, 128>(x_perm, H, dg, du, F, P, offsets, E, dW1, dW3, status, s)
             : launch_w<2, false, 128>(x_perm, H, dg, du, F, P, offsets, E, dW1, dW3, status, s);
}

}  // namespace moe
