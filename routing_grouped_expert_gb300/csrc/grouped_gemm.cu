// Step 3: the per-expert SwiGLU FFN as a persistent grouped GEMM on the
// 5th-generation tensor cores (tcgen05, accumulators in TMEM, operands
// staged by TMA).
//
//   FC1 ("FFN Input", MegaScale-Infer §3.4 Performance Simulation Model):
//       g = x W1[e], u = x W3[e], h = silu(g) * u        (SwiGLU in the epilogue)
//   FC2 ("FFN Output"):  y = h W2[e]
// with W_gate = W1, W_up = W3 in R^{H x F} and W_down = W2 in R^{F x H}
// ("Piper", §III-A, Table III).
//
// Tile = (expert e, token block b, feature tile m): the expert's rows are cut
// into ceil(rows / beta) blocks, as in "MegaFlux" §3.1 (blocks of at most
// beta rows), here of equal size rather than full blocks plus one partial
// one, so no block is a near-empty tail.  The GEMM is computed transposed
// (D^T = W^T X^T): the weight tile is the 128-row M operand, read MN-major
// straight from the caller's [E, K, N] layout; the token block is the N
// operand (N = rows rounded up to 16), so a skinny decode block costs no
// padded MMA work.
//
// Scheduling: every CTA is persistent (one per SM) and walks the flat tile
// list round-robin.  Tiles are ordered expert-major, then in groups of up to
// 16 blocks of that expert, then feature tile, then block: the blocks of a
// hot expert are spread over all SMs and run side by side on the same weight
// tile, the single-GPU counterpart of replicating a hot expert
// ("MegaScale-Infer", §3.4 Load Balancing; "MegaFlux", §3.1-3.2).
//
// Warp roles (320 threads): warp 0 = TMA producer, warp 1 = MMA issuer and
// TMEM owner, warps 2-9 = epilogue (TMEM -> registers -> global): two warps
// per TMEM lane quadrant, taking alternate 16-column chunks.  Shared
// memory holds a ring of operand stages; where TMEM has room for two
// accumulator buffers the epilogue of one tile overlaps the MMAs of the
// next.  Every wait is bounded; a wait that runs out sets MOE_ERR_TIMEOUT
// and all roles leave.
#include <cuda.h>

#include "moe_common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

using namespace ptx;

constexpr int BM = kTileM;          // weight rows (output features) per MMA (M)
constexpr int BK = kTileK;          // K per pipeline stage
constexpr int kAHalfBytes = 64 * BK * 2;          // one 64-feature TMA box: 8 KB
constexpr int kABytes = BM * BK * 2;              // 16 KB per weight tile per stage
constexpr int kBBoxBytes = kRowBox * BK * 2;      // 32 token rows: 4 KB
constexpr int kEpiWarps = 8;                      // two per TMEM lane quadrant
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kSmemBudget = 204800;               // operand ring: 200 KB
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s per wait

// kNumA weight tiles of 128 rows share each token block:
//   FC1 (kGLU): gate and up tiles of the same 128 features;
//   FC2 with kNumA = 2: two adjacent 128-feature tiles of W2.
// kBN = token rows per block (beta), kAccBufs = TMEM accumulator buffers,
// kOutF32 = fp32 output (router logits) instead of bf16.
template <int kNumA, bool kGLU, int kBN, int kAccBufs, bool kOutF32 = false>
struct Cfg {
  static constexpr int kBBytes = kBN * BK * 2;
  static constexpr int kStageBytes = kNumA * kABytes + kBBytes;
  static constexpr int kStages = kSmemBudget / kStageBytes;
  static constexpr int kAccCols = kNumA * kBN;            // fp32 columns per buffer
  static constexpr int kTmemCols = kAccBufs * kAccCols;
  static constexpr int kFeatPerItem = kGLU ? BM : kNumA * BM;
  static constexpr int kBarOffset = kStages * kStageBytes;
  static constexpr int kSmemBytes = kBarOffset + 256 + 1024;
  static_assert(kTmemCols == 128 || kTmemCols == 256 || kTmemCols == 512, "TMEM allocation");
  static_assert(kStages >= 2 && kStages <= 8, "stages");
  static_assert(!kGLU || kNumA == 2, "SwiGLU needs the gate and up tiles");
  static_assert(!kOutF32 || (kNumA == 1 && !kGLU), "fp32 output: single plain tile");
};

struct Bars {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Bars) <= 256, "barrier block too large");

struct Item {
  int e, row0, nrows, mt, nb;   // nb: token blocks of this expert
};

// Flat tile index -> (expert, first row, rows, feature tile).
template <int kBN>
__device__ __forceinline__ Item decode_item(int w, int n_mt, const int32_t* block_expert,
                                            const int32_t* block_off, const int32_t* offsets) {
  const int q = w / n_mt;                 // some block of the tile's expert
  const int e = block_expert[q];
  const int b0 = block_off[e];
  const int nb = block_off[e + 1] - b0;
  const int local = w - b0 * n_mt;
  const int gspan = kGroupBlocks * n_mt;
  const int g = local / gspan;
  const int gsize = min(kGroupBlocks, nb - g * kGroupBlocks);
  const int r = local - g * gspan;
  const int mt = r / gsize;
  const int b = g * kGroupBlocks + (r - mt * gsize);
  // The expert's rows are cut into nb blocks of equal size (a multiple of
  // 16 rows, at most kBN): a block count above one then never leaves a
  // near-empty tail block that would stream the whole weight tile for a
  // handful of rows.  Since size <= kBN and nb = ceil(rows / kBN), the last
  // block is never empty.
  const int beg = offsets[e];
  const int cnt = offsets[e + 1] - beg;
  const int bsz = min(kBN, ((cnt + nb - 1) / nb + 15) & ~15);
  Item it;
  it.e = e;
  it.mt = mt;
  it.row0 = beg + b * bsz;
  it.nrows = min(bsz, cnt - b * bsz);
  it.nb = nb;
  return it;
}

template <int kNumA, bool kGLU, int kBN, int kAccBufs, bool kOutF32>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA0,
                    const __grid_constant__ CUtensorMap tmA1,
                    const __grid_constant__ CUtensorMap tmB,
                    const int32_t* __restrict__ offsets, const int32_t* __restrict__ block_off,
                    const int32_t* __restrict__ num_blocks_ptr,
                    const int32_t* __restrict__ block_expert, int n_mt, int K,
                    void* __restrict__ out_ptr, int ld_out, int m_valid,
                    int* __restrict__ status) {
  using C = Cfg<kNumA, kGLU, kBN, kAccBufs, kOutF32>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kBarOffset);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total = *num_blocks_ptr * n_mt;
  const int nkb = K / BK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int b = 0; b < kAccBufs; ++b) {
      mbar_init(&bars->acc_full[b], 1);
      mbar_init(&bars->acc_empty[b], kEpiWarps);   // one arrival per epilogue warp
    }
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA0);
    if (kGLU) prefetch_tmap(&tmA1);
    prefetch_tmap(&tmB);
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
      // Weights: a tile read by a single token block is streamed past L2
      // (evict-first); when an expert has several blocks, its sibling blocks
      // read the same tile moments later, so it is kept (evict-normal).
      const uint64_t pol_once = policy_evict_first();
      const uint64_t pol_shared = policy_evict_normal();
      const uint64_t pol_x = policy_evict_last();    // token rows: reused
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
        const Item it = decode_item<kBN>(w, n_mt, block_expert, block_off, offsets);
        const int nbox = (it.nrows + kRowBox - 1) / kRowBox;
        const uint32_t bytes = kNumA * kABytes + nbox * kBBoxBytes;
        const int f0 = it.mt * C::kFeatPerItem;
        const uint64_t pol_w = it.nb > 1 ? pol_shared : pol_once;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&bars->empty[stage], phase ^ 1u, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          uint8_t* sA = smem + stage * C::kStageBytes;
          uint8_t* sB = sA + kNumA * kABytes;
          uint64_t* fb = &bars->full[stage];
          const int k0 = kb * BK;
          mbar_arrive_expect_tx(fb, bytes);
#pragma unroll
          for (int a = 0; a < kNumA; ++a) {
            const CUtensorMap* map = (kGLU && a == 1) ? &tmA1 : &tmA0;
            const int fa = f0 + (kGLU ? 0 : a * BM);
            tma_load_3d(sA + a * kABytes, map, fb, fa, k0, it.e, pol_w);
            tma_load_3d(sA + a * kABytes + kAHalfBytes, map, fb, fa + 64, k0, it.e, pol_w);
          }
          for (int bx = 0; bx < nbox; ++bx)
            tma_load_2d(sB + bx * kBBoxBytes, &tmB, fb, k0, it.row0 + bx * kRowBox, pol_x);
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
      // No TMA write may land after the CTA exits: wait for the last loads.
      for (int i = issued > C::kStages ? issued - C::kStages : 0; i < issued; ++i)
        mbar_wait(&bars->full[i % C::kStages], (uint32_t)((i / C::kStages) & 1), nullptr,
                  kWaitLimitNs);
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t sbase = smem_u32(smem);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int w = blockIdx.x; w < total && ok; w += gridDim.x) {
        const Item it = decode_item<kBN>(w, n_mt, block_expert, block_off, offsets);
        const int n = (it.nrows + 15) & ~15;
        const uint32_t idesc = idesc_bf16(BM, n, /*a_mn=*/true, /*b_mn=*/false);
        if (!mbar_wait(&bars->acc_empty[acc], acc_phase ^ 1u, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d0 = tmem_base + (uint32_t)(acc * C::kAccCols);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&bars->full[stage], phase, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = sbase + (uint32_t)(stage * C::kStageBytes);
          const uint32_t b0 = a0 + (uint32_t)(kNumA * kABytes);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint32_t accum = (kb | kk) ? 1u : 0u;
            // N operand: K-major rows of 128 B; K step of 16 = 32 B inside the atom.
            const uint64_t db = sdesc_sw128(b0 + kk * 32, 16, 1024);
            // M operand: MN-major; 64-feature atoms 8 KB apart (LBO), 8 K-rows
            // per 1 KB group (SBO); K step of 16 = 16 rows = 2 KB.
#pragma unroll
            for (int a = 0; a < kNumA; ++a)
              mma_bf16_ss(d0 + (uint32_t)(a * kBN),
                          sdesc_sw128(a0 + a * kABytes + kk * 2048, kAHalfBytes, 1024), db,
                          idesc, accum);
          }
          mma_commit(&bars->empty[stage]);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&bars->acc_full[acc]);
        if (++acc == kAccBufs) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        set_status(status, MOE_ERR_TIMEOUT, kWaitDetailMma);
        *abort_flag = 1;
      }
      // Every MMA issued so far completes before TMEM is released.
      mma_commit(&bars->drain);
      if (!mbar_wait(&bars->drain, 0, nullptr, kWaitLimitNs))
        set_status(status, MOE_ERR_TIMEOUT, kWaitDetailDrain);
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;            // TMEM lane quadrant this warp may read
    const int half = (warp - 2) >> 2;  // which alternate 16-column chunks it takes
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int w = blockIdx.x; w < total; w += gridDim.x) {
      const Item it = decode_item<kBN>(w, n_mt, block_expert, block_off, offsets);
      const bool got = mbar_wait(&bars->acc_full[acc], acc_phase, abort_flag, kWaitLimitNs);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const int feat = it.mt * C::kFeatPerItem + q * 32 + lane;
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * C::kAccCols);
      if constexpr (kOutF32) {
        // fp32 output; rows of a partial weight tile (feature >= m_valid) are
        // zero padding and are not stored.
        float* col = static_cast<float*>(out_ptr) + (size_t)it.row0 * ld_out + feat;
        const bool store = feat < m_valid;
        for (int c0 = 16 * half; c0 < it.nrows; c0 += 32) {
          uint32_t g[16];
          tmem_ld_32x32b_x16(tb + c0, g);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 16; ++c)
            if (store && c0 + c < it.nrows) col[(size_t)(c0 + c) * ld_out] = __uint_as_float(g[c]);
        }
      } else {
      __nv_bfloat16* col =
          static_cast<__nv_bfloat16*>(out_ptr) + (size_t)it.row0 * ld_out + feat;
      for (int c0 = 16 * half; c0 < it.nrows; c0 += 32) {
        uint32_t g[16];
        tmem_ld_32x32b_x16(tb + c0, g);
        if constexpr (kGLU) {
          uint32_t u[16];
          tmem_ld_32x32b_x16(tb + kBN + c0, u);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            if (c0 + c < it.nrows) {
              const float gv = __uint_as_float(g[c]);
              const float hv = __fdividef(gv * __uint_as_float(u[c]), 1.0f + __expf(-gv));
              col[(size_t)(c0 + c) * ld_out] = __float2bfloat16_rn(hv);
            }
          }
        } else if constexpr (kNumA == 2) {
          uint32_t g2[16];
          tmem_ld_32x32b_x16(tb + kBN + c0, g2);
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            if (c0 + c < it.nrows) {
              col[(size_t)(c0 + c) * ld_out] = __float2bfloat16_rn(__uint_as_float(g[c]));
              col[(size_t)(c0 + c) * ld_out + BM] = __float2bfloat16_rn(__uint_as_float(g2[c]));
            }
          }
        } else {
          tmem_ld_wait();
#pragma unroll
          for (int c = 0; c < 16; ++c)
            if (c0 + c < it.nrows)
              col[(size_t)(c0 + c) * ld_out] = __float2bfloat16_rn(__uint_as_float(g[c]));
        }
      }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->acc_empty[acc]);
      if (++acc == kAccBufs) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (!ok && lane == 0) {
      set_status(status, MOE_ERR_TIMEOUT, kWaitDetailEpilogue);
      *abort_flag = 1;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// bf16 tensor map with a 128-byte swizzle; dims/strides innermost first.
bool make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
              const cuuint64_t* strides, const cuuint32_t* box) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base), dims,
             strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int kNumA, bool kGLU, int kBN, int kAccBufs, bool kOutF32 = false>
cudaError_t launch_gemm(const CUtensorMap& a0, const CUtensorMap& a1, const CUtensorMap& b,
                        const int32_t* offsets, const int32_t* block_off,
                        const int32_t* num_blocks, const int32_t* block_expert, int M_total,
                        int K, long long nb_max, void* out, int ld_out, int* status,
                        cudaStream_t s) {
  using C = Cfg<kNumA, kGLU, kBN, kAccBufs, kOutF32>;
  auto kern = grouped_gemm_kernel<kNumA, kGLU, kBN, kAccBufs, kOutF32>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (err != cudaSuccess) return err;
  // a partial last feature tile (router with E not a multiple of 128) is
  // zero-filled by the TMA and not stored
  const int n_mt = (M_total + C::kFeatPerItem - 1) / C::kFeatPerItem;
  const long long items = nb_max * n_mt;
  const int grid = (int)(items < device_sm_count() ? items : device_sm_count());
  kern<<<grid, kThreads, C::kSmemBytes, s>>>(a0, a1, b, offsets, block_off, num_blocks,
                                             block_expert, n_mt, K, out, ld_out, M_total,
                                             status);
  return cudaGetLastError();
}

// FC2 pairs two W2 tiles when H allows it and K is long enough that the
// single-buffered epilogue is a small share of a tile.
#ifndef MOE_FC2_PAIR_MIN_F
#define MOE_FC2_PAIR_MIN_F 0
#endif
bool fc2_paired(int H, int F) { return H % (2 * BM) == 0 && F >= MOE_FC2_PAIR_MIN_F; }

}  // namespace

int ffn_block_rows(int P, int E, int H, int F) {
  (void)H;
  (void)F;
  switch (ffn_mode(P, E)) {
    case FfnMode::kTiny: return kBlockRowsTiny;
    case FfnMode::kSmall: return kBlockRows;
    default: return kBlockRowsLarge;
  }
}

cudaError_t launch_grouped_ffn(const __nv_bfloat16* x_perm, const int32_t* offsets,
                               const int32_t* block_off, const int32_t* num_blocks,
                               const int32_t* block_expert, const __nv_bfloat16* W1,
                               const __nv_bfloat16* W3, const __nv_bfloat16* W2, int P, int H,
                               int F, int E, __nv_bfloat16* h, __nv_bfloat16* y, int* status,
                               cudaStream_t s, cudaEvent_t after_fc1) {
  if (P == 0) return cudaSuccess;
  CUtensorMap mW1, mW3, mW2, mX, mH;
  const cuuint64_t dW13[3] = {(cuuint64_t)F, (cuuint64_t)H, (cuuint64_t)E};
  const cuuint64_t sW13[2] = {(cuuint64_t)F * 2, (cuuint64_t)H * F * 2};
  const cuuint64_t dW2[3] = {(cuuint64_t)H, (cuuint64_t)F, (cuuint64_t)E};
  const cuuint64_t sW2[2] = {(cuuint64_t)H * 2, (cuuint64_t)F * H * 2};
  const cuuint32_t boxW[3] = {64, (cuuint32_t)BK, 1};
  const cuuint64_t dX[2] = {(cuuint64_t)H, (cuuint64_t)P};
  const cuuint64_t sX[1] = {(cuuint64_t)H * 2};
  const cuuint64_t dH[2] = {(cuuint64_t)F, (cuuint64_t)P};
  const cuuint64_t sH[1] = {(cuuint64_t)F * 2};
  const cuuint32_t boxRows[2] = {(cuuint32_t)BK, (cuuint32_t)kRowBox};
  if (!make_map(&mW1, W1, 3, dW13, sW13, boxW) || !make_map(&mW3, W3, 3, dW13, sW13, boxW) ||
      !make_map(&mW2, W2, 3, dW2, sW2, boxW) || !make_map(&mX, x_perm, 2, dX, sX, boxRows) ||
      !make_map(&mH, h, 2, dH, sH, boxRows))
    return cudaErrorInvalidValue;
  cudaError_t err;
  const FfnMode mode = ffn_mode(P, E);
  if (mode == FfnMode::kTiny) {
    const long long nb_max = max_blocks(P, E, kBlockRowsTiny);
    err = launch_gemm<2, true, kBlockRowsTiny, 2>(mW1, mW3, mX, offsets, block_off, num_blocks,
                                                  block_expert, F, H, nb_max, h, F, status, s);
    if (err != cudaSuccess) return err;
    if (after_fc1 != nullptr && (err = cudaEventRecord(after_fc1, s)) != cudaSuccess) return err;
    return launch_gemm<1, false, kBlockRowsTiny, 2>(mW2, mW2, mH, offsets, block_off,
                                                    num_blocks, block_expert, H, F, nb_max, y, H,
                                                    status, s);
  }
  if (mode == FfnMode::kSmall) {
    const long long nb_max = max_blocks(P, E, kBlockRows);
    err = launch_gemm<2, true, kBlockRows, 2>(mW1, mW3, mX, offsets, block_off, num_blocks,
                                              block_expert, F, H, nb_max, h, F, status, s);
    if (err != cudaSuccess) return err;
    if (after_fc1 != nullptr && (err = cudaEventRecord(after_fc1, s)) != cudaSuccess) return err;
    return launch_gemm<1, false, kBlockRows, 2>(mW2, mW2, mH, offsets, block_off, num_blocks,
                                                block_expert, H, F, nb_max, y, H, status, s);
  }
  const long long nb_max = max_blocks(P, E, kBlockRowsLarge);
  err = launch_gemm<2, true, kBlockRowsLarge, 1>(mW1, mW3, mX, offsets, block_off, num_blocks,
                                                 block_expert, F, H, nb_max, h, F, status, s);
  if (err != cudaSuccess) return err;
  if (after_fc1 != nullptr && (err = cudaEventRecord(after_fc1, s)) != cudaSuccess) return err;
  if (fc2_paired(H, F))
    return launch_gemm<2, false, kBlockRowsLarge, 1>(mW2, mW2, mH, offsets, block_off,
                                                     num_blocks, block_expert, H, F, nb_max, y,
                                                     H, status, s);
  return launch_gemm<1, false, kBlockRowsLarge, 2>(mW2, mW2, mH, offsets, block_off, num_blocks,
                                                   block_expert, H, F, nb_max, y, H, status, s);
}

cudaError_t launch_router_gemm(const __nv_bfloat16* x, const __nv_bfloat16* Wg, int T, int H,
                               int E, const int32_t* offsets, const int32_t* block_off,
                               const int32_t* num_blocks, const int32_t* block_expert,
                               float* logits, int* status, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  // logits^T = Wg^T x^T: one "expert" whose weight matrix is Wg [H, E]
  CUtensorMap mG, mX;
  const cuuint64_t dG[3] = {(cuuint64_t)E, (cuuint64_t)H, 1};
  const cuuint64_t sG[2] = {(cuuint64_t)E * 2, (cuuint64_t)H * E * 2};
  const cuuint32_t boxW[3] = {64, (cuuint32_t)BK, 1};
  const cuuint64_t dX[2] = {(cuuint64_t)H, (cuuint64_t)T};
  const cuuint64_t sX[1] = {(cuuint64_t)H * 2};
  const cuuint32_t boxRows[2] = {(cuuint32_t)BK, (cuuint32_t)kRowBox};
  if (!make_map(&mG, Wg, 3, dG, sG, boxW) || !make_map(&mX, x, 2, dX, sX, boxRows))
    return cudaErrorInvalidValue;
  const FfnMode mode = ffn_mode(T, 1);
  if (mode == FfnMode::kTiny)
    return launch_gemm<1, false, kBlockRowsTiny, 2, true>(
        mG, mG, mX, offsets, block_off, num_blocks, block_expert, E, H,
        max_blocks(T, 1, kBlockRowsTiny), logits, E, status, s);
  if (mode == FfnMode::kSmall)
    return launch_gemm<1, false, kBlockRows, 2, true>(mG, mG, mX, offsets, block_off, num_blocks,
                                                      block_expert, E, H,
                                                      max_blocks(T, 1, kBlockRows), logits, E,
                                                      status, s);
  return launch_gemm<1, false, kBlockRowsLarge, 2, true>(
      mG, mG, mX, offsets, block_off, num_blocks, block_expert, E, H,
      max_blocks(T, 1, kBlockRowsLarge), logits, E, status, s);
}

}  // namespace moe
