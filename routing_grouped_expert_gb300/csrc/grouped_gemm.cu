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
// Scheduling: every CTA is persistent (one per SM) and takes tiles of the
// flat tile list from an on-device queue (a counter advanced once per tile)
// or, where that measured slower, round-robin.  Tiles are ordered
// expert-major, then in groups of up to 16 blocks of that expert, then
// feature tile, then block: the blocks of a hot expert are spread over all
// SMs and run side by side on the same weight tile, the single-GPU
// counterpart of replicating a hot expert ("MegaScale-Infer", §3.4 Load
// Balancing; "MegaFlux", §3.1-3.2).
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
constexpr int BK = kTileK;          // K per pipeline stage (the default; see Cfg::kBK)
constexpr int kEpiWarps = 8;                      // two per TMEM lane quadrant
constexpr int kThreads = 64 + 32 * kEpiWarps;
constexpr int kSmemBudget = 204800;               // operand ring: at most 200 KB
constexpr int kSmemMax = 232448;                  // dynamic shared memory per CTA (227 KB)
constexpr int kStgBox = 16 * 32 * 2;              // epilogue store box: 16 rows x 32 features
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // 1 s per wait

// What the epilogue does with the fp32 accumulators.
enum : int {
  kEpiBf16 = 0,        // out = acc (bf16); kNumA = 2: two adjacent 128-feature tiles
  kEpiSwiglu = 1,      // out = silu(acc0) * acc1 (bf16): FC1
  kEpiSwigluSave = 2,  // as kEpiSwiglu, and g = acc0, u = acc1 kept (bf16) for the backward
  kEpiF32 = 3,         // out = acc (fp32); features >= m_valid not stored: router logits
  kEpiSwigluBwd = 4,   // acc = dh: dg = dh*u*s*(1 + g(1 - s)), du = dh*g*s, s = sigmoid(g)
};

// kNumA weight tiles of 128 rows share each token block (FC1: gate and up of
// the same features; otherwise, with kNumA = 2: two adjacent feature tiles,
// which halves the token-block bytes staged per MMA).
// kBN = token rows per block, kAccBufs = TMEM accumulator buffers.
// kAKMajor: the weight tile is read K-major (the backward's W^T products)
// instead of MN-major.  kDualK: the K loop runs twice, first over
// (A0, B0) then over (A1, B1), into one accumulator (dx = dg W1^T + du W3^T).
// kPair: two CTAs of a cluster compute one tile of twice the features (M =
// 256 per MMA, .cta_group::2); each stages its own weight tiles and half of
// the token block (kBN / 2 rows), so the stages are smaller and the ring
// deeper (FC1: four stages of 48 KB instead of three of 64 KB).
template <int kNumA, int kEpi, int kBN, int kAccBufs, bool kAKMajor = false,
          bool kDualK = false, bool kPair = false>
struct Cfg {
  static constexpr bool kGLU = kEpi == kEpiSwiglu || kEpi == kEpiSwigluSave;
  static constexpr int kBK = BK;
  static constexpr int kAHalfBytes = 64 * kBK * 2;      // one 64-feature atom of a weight tile
  static constexpr int kABytes = BM * kBK * 2;          // one 128-feature weight tile
  static constexpr int kRowBytes = kBK * 2;             // one token row of the N operand
  static constexpr int kBBoxBytes = kRowBox * kRowBytes;   // 32 token rows
  static constexpr int kBRows = kPair ? kBN / 2 : kBN;      // token rows staged by this CTA
  static constexpr int kBBytes = kBRows * kRowBytes;
  static constexpr int kStageBytes = kNumA * kABytes + kBBytes;
  // bf16 outputs per accumulator column: each leaves through a 16-row x
  // 32-feature staging box (1 KB per warp) and a TMA store
  static constexpr int kOuts = kEpi == kEpiSwiglu ? 1 : kEpi == kEpiSwigluSave ? 3
                             : kEpi == kEpiBf16 ? kNumA : kEpi == kEpiSwigluBwd ? 2 * kNumA : 0;
  static constexpr int kStgSet = kOuts * kStgBox;   // one chunk's boxes
  static constexpr int ring_stages(int slots) {
    return kSmemBudget / kStageBytes < (kSmemMax - 2048 - kEpiWarps * slots * kStgSet) / kStageBytes
               ? kSmemBudget / kStageBytes
               : (kSmemMax - 2048 - kEpiWarps * slots * kStgSet) / kStageBytes;
  }
  // two staging sets per warp (a chunk is staged while the previous one is
  // still being stored) when that costs no operand stage, else one
  static constexpr int kStgSlots = ring_stages(2) == ring_stages(1) ? 2 : 1;
  static constexpr int kStgPerWarp = kStgSlots * kStgSet;
  static constexpr int kStages = ring_stages(kStgSlots);
  static constexpr int kAccCols = kNumA * kBN;            // fp32 columns per buffer
  static constexpr int kTmemCols = kAccBufs * kAccCols;
  // With a single accumulator buffer, the epilogue hands its token columns back
  // in groups of 64 and the next tile's first-stage MMAs wait only for the
  // group they write, so the epilogue overlaps the next tile's main loop.
  static constexpr int kRegions = kAccBufs == 1 ? kBN / 64 : 0;
  static_assert(kRegions <= 4, "region barriers");
  static constexpr int kFeatPerItem = kGLU ? BM : kNumA * BM;
  static constexpr int kBarOffset = kStages * kStageBytes;
  static constexpr int kStgOffset = kBarOffset + 1024;
  static constexpr int kSmemBytes = kStgOffset + kEpiWarps * kStgPerWarp + 1024;
  static_assert(kSmemBytes <= kSmemMax, "shared memory per CTA");
  static_assert(kTmemCols == 128 || kTmemCols == 256 || kTmemCols == 512, "TMEM allocation");
  static_assert(kStages >= 2 && kStages <= 8, "stages");
  static_assert(!kGLU || kNumA == 2, "SwiGLU needs the gate and up tiles");
  static_assert(kEpi != kEpiF32 || kNumA == 1, "single tile");
  static_assert(!kDualK || kAKMajor, "two-phase K: K-major weight tiles");
  // pairs: FC1 of the forward (SwiGLU, one accumulator buffer), 256-row blocks
  static_assert(!kPair || (kEpi == kEpiSwiglu && kBN == 256 && kAccBufs == 1 && !kAKMajor &&
                           !kDualK),
                "CTA pairs: forward FC1 with 256-row blocks");
};

constexpr int kSegRing = 4;   // segments the producer may run ahead of the other roles


struct Bars {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t seg_full[kSegRing];    // a segment published by the producer
  uint64_t seg_empty[kSegRing];   // ... and read by the MMA warp and every epilogue warp
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t acc_region[4];   // one accumulator buffer: its 64-token-column groups
  uint64_t sk_written;      // split tiles: every epilogue warp stored its partial
  uint64_t sk_decided;      // split tiles: whether this CTA finishes the tile
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int sk_last;
  int4 seg[kSegRing];   // (tile, first K stage, end K stage, 0); tile < 0: no more
};
static_assert(sizeof(Bars) <= 1024, "barrier block too large");

struct Item {
  int e, row0, nrows, mt, nb;   // nb: token blocks of this expert
  int blk;                      // the token block's index in the whole plan
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
  it.blk = b0 + b;
  return it;
}

// Balanced K split ("stream-K") of a persistent grouped GEMM whose tile count
// is not a multiple of the CTA count: the tiles' K stages are laid end to
// end and each CTA takes an equal contiguous range, so a tile may be cut
// between two neighbouring CTAs.  Each part stores its fp32 partial tile in
// a slot of its own CTA and counts itself in at the boundary; the second to
// arrive adds the other's partial (two-term fp32 sums commute, so the result
// does not depend on which CTA finishes) and stores the tile.  Nothing waits
// on another CTA.
struct StreamK {
  float* part;   // [CTAs][2] slots of [kNumA][kTileM][kBN]: 0 the CTA's first part, 1 its last
  int* cnt;      // [CTAs] arrivals at each CTA boundary, zero between launches
  size_t slot_bytes;   // capacity of one slot
  int* queue;    // head of the tile queue, zero between launches (nullptr: fixed order)
};

// The (tile, K-stage range) segments a CTA processes, in order.  Whole tiles
// come from the tile queue: a counter in global memory that each CTA's
// producer advances by one per tile it takes (without a queue, CTA c takes
// tiles c, c + G, ...).  Tiles leave the queue in list order, so the CTAs
// running side by side work on neighbouring tiles, which share weight rows and
// token blocks in L2 and DRAM pages, and a CTA that drew short tiles takes more
// of them.  Every CTA draws exactly one index past the whole tiles; the one
// that draws the last of those resets the counter for the next launch.  With a
// balanced split, the last one to two rounds' worth of tiles (between G and 2G
// of them) are instead cut into equal contiguous K ranges, one per CTA; each
// range is at least one tile long, so a tile is cut between at most two
// neighbouring CTAs.  The split balances the CTAs by itself and needs each to
// take the same whole tiles before it, so it runs with the fixed order.
struct Segments {
  long long u, end;   // the CTA's range of (tile, stage) units in the split tail
  int w, step, nkb, round_robin_end;
  bool sk, drawn_past = false;
  int* queue;
  // `cta` of `ctas`: this CTA's place among the tile takers (a CTA pair
  // takes its tiles together, as one)
  __device__ Segments(bool split_ok, int total, int nkb_, int* queue_, int cta, int ctas)
      : step(ctas), nkb(nkb_), queue(queue_) {
    const int G = ctas;
    sk = split_ok && total > G && total % G != 0;
    round_robin_end = sk ? (total / G - 1) * G : total;
    // the split assumes every CTA takes the same number of whole tiles: fixed order
    if (sk) queue = nullptr;
    const long long base = (long long)round_robin_end * nkb;
    const long long U = (long long)(total - round_robin_end) * nkb;
    u = base + U * cta / G;
    end = base + U * (cta + 1) / G;
    w = queue ? atomicAdd(queue, 1) : cta;
  }
  __device__ bool next(int& wo, int& kb0, int& kb1) {
    if (w < round_robin_end) {
      wo = w;
      kb0 = 0;
      kb1 = nkb;
      w = queue ? atomicAdd(queue, 1) : w + step;   // the draw is awaited only by the next call
      return true;
    }
    if (queue && !drawn_past) {   // this CTA's one draw past the whole tiles
      drawn_past = true;
      if (w == round_robin_end + step - 1) atomicExch(queue, 0);
    }
    if (!sk || u >= end) return false;
    wo = (int)(u / nkb);
    kb0 = (int)(u - (long long)wo * nkb);
    kb1 = (int)min((long long)nkb, kb0 + (end - u));
    u += kb1 - kb0;
    return true;
  }
};

// Tensor maps of the bf16 outputs ([rows, ld], boxes of 16 rows x 32 features):
// h / y / dx, or h, g, u (forward with saves), or dg, du (SwiGLU backward).
struct OutMaps {
  CUtensorMap m[3];
};

// Token-row tensor maps of the N operand ([P, K], K contiguous), per K phase:
// boxes of 32, 64, 128 and 256 rows x 64 K, so a block's rows (rounded up to
// 32) arrive in at most three TMA instructions per stage.
struct RowMaps {
  CUtensorMap m[2][4];
};

// Four rows (y0..y3) of 64 K each from a 2-D tensor map whose box is one row
// high, stored as consecutive 128-byte rows at dst (the map's swizzle applied).
__device__ __forceinline__ void tma_gather4(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int x, int y0, int y1, int y2, int y3,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y0), "r"(y1),
      "r"(y2), "r"(y3), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, const void* src, int x,
                                             int y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::
                   "l"(reinterpret_cast<uint64_t>(map)),
               "r"(smem_u32(src)), "r"(x), "r"(y)
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
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Orders this thread's generic-proxy global accesses with its async-proxy
// (TMA) ones.
__device__ __forceinline__ void fence_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Token-block dependencies between FC1 and FC2 of one forward, which then run
// as two overlapping launches: FC1 (kDepSignal) lets FC2 launch as soon as it
// starts, and after the h rows of a tile are stored each of its epilogue warps
// counts itself in at the tile's token block; FC2 (kDepWait, launched with
// programmatic stream serialization) waits, before loading a tile's h rows,
// until its block's count reaches every FC1 tile of the block.  FC1 never
// waits on FC2, and every FC1 CTA is resident before any FC2 CTA launches
// (one CTA per SM), so the waits end; each is bounded like the pipeline's.
enum : int { kDepNone = 0, kDepSignal = 1, kDepWait = 2 };

// kGather: the token rows of the N operand are gathered straight from x
// ([T, K], token-major) by TMA tile::gather4 loads -- row p of an expert
// group is token sorted_src[p] / k -- so no expert-ordered copy of x is made
// (FC1 of the forward).  rows.m[0][0] is then a tensor map of x with boxes of
// one row x 64 K; the producer warp's lanes each gather four rows at a time.
//
// kPair: the CTAs run as clusters of two (see Cfg).  A pair takes the tiles
// of the list as one: tile (expert, block, m) covers features [2m, 2m + 2) x
// kFeatPerItem, rank r of the pair the r-th half.  Rank r stages the block's
// rows [r hb, r hb + hb), hb = rows rounded up to 32, halved (N = 2 hb, a
// multiple of 32).  Rank 0 waits for
// both halves of a stage (its full barrier counts both ranks' bytes), issues
// the MMAs and signals stage release, accumulator ready and drain on the
// barriers of both ranks; each rank reads its own accumulator, stores its own
// features and hands the accumulator back to rank 0.  Each MMA spans the whole
// block (N = 2 hb): its first hb columns come from rank 0's rows and the rest
// from rank 1's, so accumulator column c holds block row c on both ranks.
// (Measured: splitting the block into MMAs of N = 128 or 64, which would let
// the next tile start on the columns already read, makes every pair MMA cost
// about as much as a full one -- the fine-grained FC1 1.4x and 2.2x slower.)
template <int kNumA, int kEpi, int kBN, int kAccBufs, bool kAKMajor, bool kDualK, bool kGather,
          bool kPair>
__global__ void __launch_bounds__(kThreads, 1)
grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA0,
                    const __grid_constant__ CUtensorMap tmA1,
                    const __grid_constant__ RowMaps rows, int a_atoms,
                    const int32_t* __restrict__ offsets, const int32_t* __restrict__ block_off,
                    const int32_t* __restrict__ num_blocks_ptr,
                    const int32_t* __restrict__ block_expert, int n_mt, int K,
                    void* __restrict__ out_ptr, int ld_out, int m_valid, EpiAux aux,
                    const __grid_constant__ OutMaps outs, StreamK sk,
                    const int32_t* __restrict__ gather_src, int gather_k,
                    int* __restrict__ blk_done, int blk_target, int dep,
                    int* __restrict__ status) {
  using C = Cfg<kNumA, kEpi, kBN, kAccBufs, kAKMajor, kDualK, kPair>;
  constexpr int kBK = C::kBK;
  static_assert(!kGather || (!kDualK && !kAKMajor), "gathered rows: forward products only");
  static_assert(!kPair || !kGather, "CTA pairs: rows staged by plain tile loads");
  constexpr bool kGLU = C::kGLU;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + C::kBarOffset);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int total = *num_blocks_ptr * n_mt;
  // The balanced split for one weight tile with two accumulator buffers and a
  // bf16 output (FC2 and DGrad dx of small token blocks).  Measured elsewhere
  // it loses: with one accumulator buffer the cut tiles' partial stores stall
  // the next tile's MMAs, and FC1 prefers every CTA on neighbouring tiles.
  constexpr bool kSKCapable = kEpi == kEpiBf16 && kNumA == 1 && kAccBufs == 2;
  constexpr size_t kSlot = (size_t)kNumA * BM * kBN;   // floats of one partial tile
  const bool sk_ok = kSKCapable && !kPair && sk.part != nullptr;
  const uint32_t rank = kPair ? cluster_ctarank() : 0u;   // within the pair
  const int nkb = K / kBK;                        // K stages per phase
  const int nkb_all = kDualK ? 2 * nkb : nkb;

  // FC2 may launch on SMs this grid leaves (it waits per token block)
  if (dep == kDepSignal) pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
    }
    for (int i = 0; i < kSegRing; ++i) {
      mbar_init(&bars->seg_full[i], 1);
      mbar_init(&bars->seg_empty[i], 1 + kEpiWarps);
    }
    for (int b = 0; b < kAccBufs; ++b) {
      mbar_init(&bars->acc_full[b], 1);
      mbar_init(&bars->acc_empty[b], kEpiWarps);   // one arrival per epilogue warp
    }
    // pairs: rank 0's group barriers count both ranks' epilogue warps
    for (int r = 0; r < C::kRegions; ++r)
      mbar_init(&bars->acc_region[r], (kPair ? 2 : 1) * kEpiWarps);
    mbar_init(&bars->sk_written, kEpiWarps);
    mbar_init(&bars->sk_decided, 1);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmA0);
    if (kGLU || kDualK) prefetch_tmap(&tmA1);
    for (int ph = 0; ph < (kDualK ? 2 : 1); ++ph)
      for (int j = 0; j < 4; ++j) prefetch_tmap(&rows.m[ph][j]);
  }
  if (warp == 1) {
    if constexpr (kPair) {
      tmem_alloc_pair(&bars->tmem_base, C::kTmemCols);
      tmem_relinquish_pair();
    } else {
      tmem_alloc(&bars->tmem_base, C::kTmemCols);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  // pairs: both ranks' barriers are initialised before either signals the other's
  if constexpr (kPair) cluster_sync(); else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = bars->tmem_base;
  volatile int* abort_flag = &bars->abort;
  // A role that gives up stops the other roles of its CTA and of its pair.
  auto raise_abort = [=]() {
    *abort_flag = 1;
    if constexpr (kPair)
      st_cluster_u32(mapa_shared(smem_u32(const_cast<int*>(&bars->abort)), rank ^ 1u), 1u);
  };

  if (warp == 0 && kGather) {
    // ----------------------------------- TMA producer, gathered token rows
    // Lane 0 draws the segments, waits for free stages and loads the weight
    // tiles; every lane then gathers its share of the block's token rows
    // (kRowsPerLane rows, four per instruction) into the same stage.
    constexpr int kRowsPerLane = kBN / 32 < 4 ? 4 : kBN / 32;
    const uint64_t pol_once = policy_evict_first();
    const uint64_t pol_shared = policy_evict_normal();
    const uint64_t pol_x = policy_evict_last();      // x rows: reused by every feature tile
    const CUtensorMap* xmap = &rows.m[0][0];
    int stage = 0, issued = 0;
    uint32_t phase = 0;
    bool ok = true;
    // only lane 0 draws from the queue; the other lanes' copies stay idle
    Segments sg(sk_ok, total, nkb_all, lane == 0 ? sk.queue : nullptr, (int)blockIdx.x,
                (int)gridDim.x);
    int sslot = 0;
    uint32_t sphase = 0;
    while (true) {
      int w = 0, kb0 = 0, kb1 = 0, have = 0;
      if (lane == 0 && ok) {
        have = sg.next(w, kb0, kb1) ? 1 : 0;
        // hand the segment to the MMA warp and the epilogue
        if (have) {
          if (mbar_wait(&bars->seg_empty[sslot], sphase ^ 1u, abort_flag, kWaitLimitNs)) {
            bars->seg[sslot] = make_int4(w, kb0, kb1, 0);
            mbar_arrive(&bars->seg_full[sslot]);
            if (++sslot == kSegRing) {
              sslot = 0;
              sphase ^= 1u;
            }
          } else {
            ok = false;
            have = 0;
          }
        }
      }
      have = __shfl_sync(0xffffffffu, have, 0);
      if (!have) break;
      w = __shfl_sync(0xffffffffu, w, 0);
      kb0 = __shfl_sync(0xffffffffu, kb0, 0);
      kb1 = __shfl_sync(0xffffffffu, kb1, 0);
      const Item it = decode_item<kBN>(w, n_mt, block_expert, block_off, offsets);
      const int n16 = (it.nrows + 15) & ~15;        // rows the MMA reads
      // this lane's token rows; rows past the block repeat its last row
      int tok[kRowsPerLane];
#pragma unroll
      for (int i = 0; i < kRowsPerLane; ++i) {
        const int r = min(lane * kRowsPerLane + i, it.nrows - 1);
        tok[i] = __ldg(gather_src + it.row0 + r) / gather_k;
      }
      const uint32_t bytes = kNumA * C::kABytes + (uint32_t)n16 * C::kRowBytes;
      const int f0 = it.mt * C::kFeatPerItem;
      const uint64_t pol_w = it.nb > 1 ? pol_shared : pol_once;
      for (int kb = kb0; kb < kb1; ++kb) {
        int free_ok = 1;
        if (lane == 0) {
          free_ok = mbar_wait(&bars->empty[stage], phase ^ 1u, abort_flag, kWaitLimitNs);
          if (free_ok) {
            uint64_t* fb = &bars->full[stage];
            uint8_t* sA = smem + stage * C::kStageBytes;
            const int k0 = kb * kBK;
            mbar_arrive_expect_tx(fb, bytes);
#pragma unroll
            for (int a = 0; a < kNumA; ++a) {
              const CUtensorMap* map = (kGLU && a == 1) ? &tmA1 : &tmA0;
              const int fa = f0 + (kGLU ? 0 : a * BM);
              if (a_atoms) {
                tma_load_4d(sA + a * C::kABytes, map, fb, 0, k0, fa >> 6, it.e, pol_w);
              } else {
                tma_load_3d(sA + a * C::kABytes, map, fb, fa, k0, it.e, pol_w);
                tma_load_3d(sA + a * C::kABytes + C::kAHalfBytes, map, fb, fa + 64, k0, it.e, pol_w);
              }
            }
          }
        }
        free_ok = __shfl_sync(0xffffffffu, free_ok, 0);
        if (!free_ok) {
          ok = false;
          break;
        }
        // the expected bytes are posted before any row lands
        uint64_t* fb = &bars->full[stage];
        uint8_t* sB = smem + stage * C::kStageBytes + kNumA * C::kABytes;
        const int k0 = kb * kBK;
#pragma unroll
        for (int g = 0; g < kRowsPerLane / 4; ++g) {
          const int r0 = lane * kRowsPerLane + 4 * g;
          if (r0 < n16)
            tma_gather4(sB + r0 * C::kRowBytes, xmap, fb, k0, tok[4 * g], tok[4 * g + 1],
                        tok[4 * g + 2], tok[4 * g + 3], pol_x);
        }
        ++issued;
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (!__all_sync(0xffffffffu, ok)) break;
    }
    if (lane == 0) {
      if (ok) {   // no more segments
        if (mbar_wait(&bars->seg_empty[sslot], sphase ^ 1u, abort_flag, kWaitLimitNs)) {
          bars->seg[sslot] = make_int4(-1, 0, 0, 0);
          mbar_arrive(&bars->seg_full[sslot]);
        } else {
          ok = false;
        }
      }
      if (!ok) {
        set_status(status, MOE_ERR_TIMEOUT, kWaitDetailProducer);
        raise_abort();
      }
      // No TMA write may land after the CTA exits: wait for the last loads.
      for (int i = issued > C::kStages ? issued - C::kStages : 0; i < issued; ++i)
        mbar_wait(&bars->full[i % C::kStages], (uint32_t)((i / C::kStages) & 1), nullptr,
                  kWaitLimitNs);
    }
  } else if (warp == 0) {
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
      // a pair takes its tiles in the fixed order (both ranks the same ones)
      Segments sg(sk_ok, total, nkb_all, kPair ? nullptr : sk.queue,
                  kPair ? (int)(blockIdx.x >> 1) : (int)blockIdx.x,
                  kPair ? (int)(gridDim.x >> 1) : (int)gridDim.x);
      int w, kb0, kb1;
      int sslot = 0;
      uint32_t sphase = 0;
      // hand a segment to the MMA warp and the epilogue (tile < 0: no more)
      auto publish = [&](int tile, int k0s, int k1s) {
        if (!mbar_wait(&bars->seg_empty[sslot], sphase ^ 1u, abort_flag, kWaitLimitNs))
          return false;
        bars->seg[sslot] = make_int4(tile, k0s, k1s, 0);
        mbar_arrive(&bars->seg_full[sslot]);
        if (++sslot == kSegRing) {
          sslot = 0;
          sphase ^= 1u;
        }
        return true;
      };
      while (ok && sg.next(w, kb0, kb1)) {
        if (!publish(w, kb0, kb1)) {
          ok = false;
          break;
        }
        const Item it = decode_item<kBN>(w, n_mt, block_expert, block_off, offsets);
        if (dep == kDepWait) {
          // the block's h rows: stored by every FC1 tile of the block
          if (!wait_count(blk_done + it.blk, blk_target, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          fence_async_global();   // the TMA loads below see what the acquire saw
        }
        // this CTA's token rows [rb0, rb0 + nr) of the block (pairs: its half)
        const int hb = kPair ? ((it.nrows + 31) & ~31) / 2 : 0;
        const int rb0 = kPair ? (int)rank * hb : 0;
        const int nr = kPair ? hb : it.nrows;
        const int nbox = (nr + kRowBox - 1) / kRowBox;
        const uint32_t bytes = kNumA * C::kABytes + nbox * C::kBBoxBytes;
        const int f0 = (kPair ? 2 * it.mt + (int)rank : it.mt) * C::kFeatPerItem;
        const uint64_t pol_w = it.nb > 1 ? pol_shared : pol_once;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&bars->empty[stage], phase ^ 1u, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          const bool second = kDualK && kb >= nkb;    // second K phase
          const int k0 = (second ? kb - nkb : kb) * kBK;
          uint8_t* sA = smem + stage * C::kStageBytes;
          uint8_t* sB = sA + kNumA * C::kABytes;
          uint64_t* fb = &bars->full[stage];
          if constexpr (kPair) {
            // rank 0's full barrier counts both ranks' bytes (equal halves)
            const uint32_t fbc = mapa_shared(smem_u32(fb), 0);
            if (rank == 0) mbar_arrive_expect_tx(fb, 2 * bytes);
#pragma unroll
            for (int a = 0; a < kNumA; ++a) {
              const CUtensorMap* map = (kGLU && a == 1) ? &tmA1 : &tmA0;
              const int fa = f0 + (kGLU ? 0 : a * BM);
              if (a_atoms) {
                tma_load_4d_pair(sA + a * C::kABytes, map, fbc, 0, k0, fa >> 6, it.e, pol_w);
              } else {
                tma_load_3d_pair(sA + a * C::kABytes, map, fbc, fa, k0, it.e, pol_w);
                tma_load_3d_pair(sA + a * C::kABytes + C::kAHalfBytes, map, fbc, fa + 64, k0,
                                 it.e, pol_w);
              }
            }
            for (int r = 0; r < nbox * kRowBox;) {
              const int rem = nbox * kRowBox - r;
              const int lg = (C::kBRows >= 128 && rem >= 128) ? 2 : rem >= 64 ? 1 : 0;
              tma_load_2d_pair(sB + r * C::kRowBytes, &rows.m[0][lg], fbc, k0,
                               it.row0 + rb0 + r, pol_x);
              r += kRowBox << lg;
            }
            ++issued;
            if (++stage == C::kStages) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          mbar_arrive_expect_tx(fb, bytes);
#pragma unroll
          for (int a = 0; a < kNumA; ++a) {
            const CUtensorMap* map = ((kGLU && a == 1) || second) ? &tmA1 : &tmA0;
            const int fa = f0 + (kGLU ? 0 : a * BM);
            if constexpr (kAKMajor) {
              // 128 weight rows x 64 K, K contiguous: one box
              tma_load_3d(sA + a * C::kABytes, map, fb, k0, fa, it.e, pol_w);
            } else if (a_atoms) {
              // 64 K rows x 128 features, features contiguous, as two 64-feature
              // atoms of a 4-D view: one box
              tma_load_4d(sA + a * C::kABytes, map, fb, 0, k0, fa >> 6, it.e, pol_w);
            } else {
              // 64 K rows x 64 features per box: two boxes
              tma_load_3d(sA + a * C::kABytes, map, fb, fa, k0, it.e, pol_w);
              tma_load_3d(sA + a * C::kABytes + C::kAHalfBytes, map, fb, fa + 64, k0, it.e, pol_w);
            }
          }
          // the block's rows, rounded up to 32, in boxes of 256, 128, 64 and 32 rows
          const CUtensorMap* bm = rows.m[second ? 1 : 0];
          for (int r = 0; r < nbox * kRowBox;) {
            const int rem = nbox * kRowBox - r;
            const int lg = (kBN >= 256 && rem >= 256) ? 3 : (kBN >= 128 && rem >= 128) ? 2
                                                                : rem >= 64             ? 1
                                                                                        : 0;
            tma_load_2d(sB + r * C::kRowBytes, &bm[lg], fb, k0, it.row0 + r, pol_x);
            r += kRowBox << lg;
          }
          ++issued;
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (ok) ok = publish(-1, 0, 0);
      if (!ok) {
        set_status(status, MOE_ERR_TIMEOUT, kWaitDetailProducer);
        raise_abort();
      }
      // No TMA write may land after the CTA exits: wait for the last loads
      // (pairs: rank 0's barriers count rank 1's loads too, and rank 1 does
      // not leave before rank 0 -- the cluster barrier at the end).
      if (!kPair || rank == 0)
        for (int i = issued > C::kStages ? issued - C::kStages : 0; i < issued; ++i)
          mbar_wait(&bars->full[i % C::kStages], (uint32_t)((i / C::kStages) & 1), nullptr,
                    kWaitLimitNs);
    }
  } else if (warp == 1 && kPair && rank != 0) {
    // ------------------------------------- pair rank 1: no MMAs of its own
    // It takes the segments (the producer's ring counts this warp) and waits
    // until rank 0's MMAs, which read its shared memory and write its tensor
    // memory, have drained.
    if (lane == 0) {
      bool ok = true;
      int sslot = 0;
      uint32_t sphase = 0;
      while (true) {
        if (!mbar_wait(&bars->seg_full[sslot], sphase, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        const int x = bars->seg[sslot].x;
        mbar_arrive(&bars->seg_empty[sslot]);
        if (++sslot == kSegRing) {
          sslot = 0;
          sphase ^= 1u;
        }
        if (x < 0) break;
      }
      if (!ok) {
        set_status(status, MOE_ERR_TIMEOUT, kWaitDetailMma);
        raise_abort();
      }
      if (!mbar_wait(&bars->drain, 0, nullptr, kWaitLimitNs))
        set_status(status, MOE_ERR_TIMEOUT, kWaitDetailDrain);
    }
  } else if (warp == 1) {
    // -------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t sbase = smem_u32(smem);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      int sslot = 0;
      uint32_t sphase = 0;
      while (ok) {
        if (!mbar_wait(&bars->seg_full[sslot], sphase, abort_flag, kWaitLimitNs)) {
          ok = false;
          break;
        }
        const int4 seg = bars->seg[sslot];
        mbar_arrive(&bars->seg_empty[sslot]);
        if (++sslot == kSegRing) {
          sslot = 0;
          sphase ^= 1u;
        }
        if (seg.x < 0) break;
        const int w = seg.x, kb0 = seg.y, kb1 = seg.z;
        const Item it = decode_item<kBN>(w, n_mt, block_expert, block_off, offsets);
        const int n = (it.nrows + 15) & ~15;
        const uint32_t idesc = idesc_bf16(BM, n, /*a_mn=*/!kAKMajor, /*b_mn=*/false);
        if constexpr (kAccBufs == 2) {
          if (!mbar_wait(&bars->acc_empty[acc], acc_phase ^ 1u, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
        }
        const uint32_t d0 = tmem_base + (uint32_t)(acc * C::kAccCols);
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!mbar_wait(&bars->full[stage], phase, abort_flag, kWaitLimitNs)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = sbase + (uint32_t)(stage * C::kStageBytes);
          const uint32_t b0 = a0 + (uint32_t)(kNumA * C::kABytes);
          if constexpr (kPair) {
            // one MMA per K step and weight tile over the whole block
            if (C::kRegions > 0 && kb == kb0) {   // the previous tile's epilogue is done
              for (int r = 0; ok && r < C::kRegions; ++r)
                ok = mbar_wait(&bars->acc_region[r], acc_phase ^ 1u, abort_flag, kWaitLimitNs);
              if (!ok) break;
              tc_fence_after();
            }
            const int np = (it.nrows + 31) & ~31;
            const uint32_t idesc_p = idesc_bf16(2 * BM, np, /*a_mn=*/true, /*b_mn=*/false);
#pragma unroll
            for (int kk = 0; kk < kBK / 16; ++kk) {
              const uint64_t db = sdesc_sw128(b0 + kk * 32, 16, 1024);
#pragma unroll
              for (int a = 0; a < kNumA; ++a) {
                const uint64_t da =
                    sdesc_sw128(a0 + a * C::kABytes + kk * 2048, C::kAHalfBytes, 1024);
                mma_bf16_ss_pair(d0 + (uint32_t)(a * kBN), da, db, idesc_p,
                                 (kb > kb0 || kk) ? 1u : 0u);
              }
            }
            if (!ok) break;
            mma_commit_pair(&bars->empty[stage], 0x3);
            if (++stage == C::kStages) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          if (C::kRegions > 0 && kb == kb0) {
            // First stage, one 64-token-column group at a time, each once the
            // epilogue has read it out of the previous tile.  Per accumulator
            // element the K order is the same as in the later stages.
            for (int r = 0; r < C::kRegions; ++r) {
              if (!mbar_wait(&bars->acc_region[r], acc_phase ^ 1u, abort_flag, kWaitLimitNs)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const int c = 64 * r;
              if (c >= n) continue;
              const int nr = n - c < 64 ? n - c : 64;
              const uint32_t idesc_r = idesc_bf16(BM, nr, /*a_mn=*/!kAKMajor, /*b_mn=*/false);
#pragma unroll
              for (int kk = 0; kk < kBK / 16; ++kk) {
                // token row c starts c * 128 bytes into the K-major N operand
                const uint64_t db = sdesc_sw128(b0 + c * C::kRowBytes + kk * 32, 16, 1024);
#pragma unroll
                for (int a = 0; a < kNumA; ++a) {
                  const uint64_t da =
                      kAKMajor ? sdesc_sw128(a0 + a * C::kABytes + kk * 32, 16, 1024)
                               : sdesc_sw128(a0 + a * C::kABytes + kk * 2048, C::kAHalfBytes, 1024);
                  mma_bf16_ss(d0 + (uint32_t)(a * kBN + c), da, db, idesc_r, kk ? 1u : 0u);
                }
              }
            }
            if (!ok) break;
          } else {
#pragma unroll
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint32_t accum = (kb > kb0 || kk) ? 1u : 0u;
            // N operand: K-major rows of 128 B; K step of 16 = 32 B inside the atom.
            const uint64_t db = sdesc_sw128(b0 + kk * 32, 16, 1024);
#pragma unroll
            for (int a = 0; a < kNumA; ++a) {
              // M operand.  MN-major: 64-feature atoms 8 KB apart (LBO), 8 K-rows
              // per 1 KB group (SBO), K step of 16 = 16 rows = 2 KB.  K-major:
              // rows of 128 B, 8-row groups 1 KB apart, K step of 16 = 32 B.
              const uint64_t da =
                  kAKMajor ? sdesc_sw128(a0 + a * C::kABytes + kk * 32, 16, 1024)
                           : sdesc_sw128(a0 + a * C::kABytes + kk * 2048, C::kAHalfBytes, 1024);
              mma_bf16_ss(d0 + (uint32_t)(a * kBN), da, db, idesc, accum);
            }
          }
          }
          mma_commit(&bars->empty[stage]);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        if constexpr (kPair) mma_commit_pair(&bars->acc_full[acc], 0x3);
        else mma_commit(&bars->acc_full[acc]);
        if (++acc == kAccBufs) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      if (!ok) {
        set_status(status, MOE_ERR_TIMEOUT, kWaitDetailMma);
        raise_abort();
      }
      // Every MMA issued so far completes before TMEM is released (pairs:
      // rank 1 waits for the same on its own drain barrier).
      if constexpr (kPair) mma_commit_pair(&bars->drain, 0x3);
      else mma_commit(&bars->drain);
      if (!mbar_wait(&bars->drain, 0, nullptr, kWaitLimitNs))
        set_status(status, MOE_ERR_TIMEOUT, kWaitDetailDrain);
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int q = warp & 3;            // TMEM lane quadrant this warp may read
    const int half = (warp - 2) >> 2;  // which alternate 16-column chunks it takes
    uint8_t* stg = smem + C::kStgOffset + (warp - 2) * C::kStgPerWarp;
    int slot = 0;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    int sk_n = 0;   // split tiles this CTA has taken part in (phase of the sk barriers)
    int sslot = 0;
    uint32_t sphase = 0;
    while (true) {
      const bool have = mbar_wait(&bars->seg_full[sslot], sphase, abort_flag, kWaitLimitNs);
      if (!__all_sync(0xffffffffu, have)) {
        ok = false;
        break;
      }
      const int4 seg = bars->seg[sslot];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->seg_empty[sslot]);
      if (++sslot == kSegRing) {
        sslot = 0;
        sphase ^= 1u;
      }
      if (seg.x < 0) break;
      const int w = seg.x, kb0 = seg.y, kb1 = seg.z;
      const Item it = decode_item<kBN>(w, n_mt, block_expert, block_off, offsets);
      const bool got = mbar_wait(&bars->acc_full[acc], acc_phase, abort_flag, kWaitLimitNs);
      if (!__all_sync(0xffffffffu, got)) {
        ok = false;
        break;
      }
      tc_fence_after();
      // the warp's first feature (pairs: rank r stores the r-th half of the tile)
      const int wfeat = (kPair ? 2 * it.mt + (int)rank : it.mt) * C::kFeatPerItem + q * 32;
      const int feat = wfeat + lane;
      const uint32_t tb = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * C::kAccCols);
      // A tile cut between two CTAs: store this part, count in at the boundary;
      // the second part to arrive adds the other's partial and stores the tile.
      const float* other = nullptr;   // the neighbour's partial to add
      bool store = true;
      if constexpr (kSKCapable) {
        if (kb0 > 0 || kb1 < nkb_all) {
          const bool head = kb0 == 0;   // the tile's first stages: this CTA's last part
          const int c = blockIdx.x;
          float* mine = sk.part + ((size_t)c * 2 + (head ? 1 : 0)) * kSlot;
          const float* theirs =
              sk.part + (head ? (size_t)(c + 1) * 2 : (size_t)(c - 1) * 2 + 1) * kSlot;
          int* cnt = sk.cnt + (head ? c : c - 1);
#pragma unroll
          for (int a = 0; a < kNumA; ++a)
            for (int c0 = 16 * half; c0 < it.nrows; c0 += 32) {
              uint32_t v[16];
              tmem_ld_32x32b_x16(tb + a * kBN + c0, v);
              tmem_ld_wait();
              float4* dst = reinterpret_cast<float4*>(
                  mine + ((size_t)a * BM + q * 32 + lane) * kBN + c0);
#pragma unroll
              for (int j = 0; j < 4; ++j)
                dst[j] = make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                     __uint_as_float(v[4 * j + 2]),
                                     __uint_as_float(v[4 * j + 3]));
            }
          __threadfence();   // this thread's partial is visible device-wide
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->sk_written);
          bool good = true;
          if (warp == 2 && lane == 0) {
            good = mbar_wait(&bars->sk_written, (uint32_t)(sk_n & 1), abort_flag, kWaitLimitNs);
            int last = 0;
            if (good) {
              __threadfence();
              last = atomicAdd(cnt, 1) == 1;
              if (last) *cnt = 0;   // both parts counted: zero for the next launch
            }
            bars->sk_last = last;
            mbar_arrive(&bars->sk_decided);
          }
          const bool dec =
              mbar_wait(&bars->sk_decided, (uint32_t)(sk_n & 1), abort_flag, kWaitLimitNs);
          ++sk_n;
          if (!__all_sync(0xffffffffu, good && dec)) {
            ok = false;
            break;
          }
          if (*reinterpret_cast<volatile int*>(&bars->sk_last)) {
            __threadfence();   // the neighbour's partial, published before its count
            other = theirs;
          } else {
            store = false;
          }
        }
      }
      // one 16-column chunk of the accumulator: TMEM -> registers -> epilogue
      // one 16-column chunk of the accumulator, already in registers (g: tile
      // 0 / gate, g2: tile 1 / up) -> epilogue -> global memory
      auto process = [&](int c0, uint32_t (&g)[16], uint32_t (&g2)[16]) {
        float pg[kNumA][16], pu[kNumA][16];
        if constexpr (kEpi == kEpiSwigluBwd) {
          // all saved g, u of the chunk are loaded first: a load placed after a
          // store to dg / du would otherwise wait for it (possible aliasing)
#pragma unroll
          for (int a = 0; a < kNumA; ++a)
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const bool in = c0 + c < it.nrows;
              const size_t i = (size_t)(it.row0 + c0 + c) * aux.ld + feat + a * BM;
              pg[a][c] = in ? __bfloat162float(aux.g[i]) : 0.f;
              pu[a][c] = in ? __bfloat162float(aux.u[i]) : 0.f;
            }
        }
        if constexpr (kSKCapable) {
          if (other != nullptr) {   // finish a cut tile: add the neighbour's part
#pragma unroll
            for (int a = 0; a < kNumA; ++a) {
              uint32_t* r = a == 0 ? g : g2;
              const float4* o4 = reinterpret_cast<const float4*>(
                  other + ((size_t)a * BM + q * 32 + lane) * kBN + c0);
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                const float4 t = __ldcg(o4 + j);
                r[4 * j] = __float_as_uint(__uint_as_float(r[4 * j]) + t.x);
                r[4 * j + 1] = __float_as_uint(__uint_as_float(r[4 * j + 1]) + t.y);
                r[4 * j + 2] = __float_as_uint(__uint_as_float(r[4 * j + 2]) + t.z);
                r[4 * j + 3] = __float_as_uint(__uint_as_float(r[4 * j + 3]) + t.w);
              }
            }
          }
        }
        if constexpr (C::kOuts > 0) {
          if (c0 + 16 <= it.nrows) {
            // a whole 16-row chunk: stage [row][feature] boxes, one TMA store each
            // this staging set's previous boxes have left shared memory
            if (lane == 0) bulk_wait_read<C::kStgSlots - 1>();
            __syncwarp();
            uint8_t* const set = stg + slot * C::kStgSet;
            slot = slot + 1 == C::kStgSlots ? 0 : slot + 1;
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              const float a0 = __uint_as_float(g[c]);
              float v[C::kOuts];
              if constexpr (kGLU) {
                const float a1 = __uint_as_float(g2[c]);
                v[0] = __fdividef(a0 * a1, 1.0f + __expf(-a0));
                if constexpr (kEpi == kEpiSwigluSave) {
                  v[1] = a0;
                  v[2] = a1;
                }
              } else if constexpr (kEpi == kEpiSwigluBwd) {
#pragma unroll
                for (int a = 0; a < kNumA; ++a) {
                  const float dh = a == 0 ? a0 : __uint_as_float(g2[c]);
                  const float gv = pg[a][c], uv = pu[a][c];
                  const float sg = __fdividef(1.0f, 1.0f + __expf(-gv));
                  v[2 * a] = dh * uv * sg * (1.0f + gv * (1.0f - sg));
                  v[2 * a + 1] = dh * gv * sg;
                }
              } else {
                v[0] = a0;
                if constexpr (kNumA == 2) v[1] = __uint_as_float(g2[c]);
              }
#pragma unroll
              for (int j = 0; j < C::kOuts; ++j)
                *reinterpret_cast<__nv_bfloat16*>(set + j * kStgBox + c * 64 + lane * 2) =
                    __float2bfloat16_rn(v[j]);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) {
              const int y = it.row0 + c0;
#pragma unroll
              for (int j = 0; j < C::kOuts; ++j) {
                // output j: which map, and its feature offset
                const int mi = kEpi == kEpiSwigluSave ? j : kEpi == kEpiSwigluBwd ? (j & 1) : 0;
                const int xo = kEpi == kEpiSwigluBwd ? (j >> 1) * BM
                             : kEpi == kEpiBf16 ? j * BM : 0;
                tma_store_2d(&outs.m[mi], set + j * kStgBox, wfeat + xo, y);
              }
              bulk_commit();
            }
            return;
          }
        }
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          if (c0 + c >= it.nrows) continue;
          const size_t row = (size_t)(it.row0 + c0 + c);
          const float a0 = __uint_as_float(g[c]);
          if constexpr (kEpi == kEpiF32) {
            // rows of a partial weight tile (feature >= m_valid) are zero padding
            if (feat < m_valid) static_cast<float*>(out_ptr)[row * ld_out + feat] = a0;
          } else if constexpr (kGLU) {
            const float a1 = __uint_as_float(g2[c]);
            const float hv = __fdividef(a0 * a1, 1.0f + __expf(-a0));
            static_cast<__nv_bfloat16*>(out_ptr)[row * ld_out + feat] = __float2bfloat16_rn(hv);
            if constexpr (kEpi == kEpiSwigluSave) {
              aux.g[row * aux.ld + feat] = __float2bfloat16_rn(a0);
              aux.u[row * aux.ld + feat] = __float2bfloat16_rn(a1);
            }
          } else if constexpr (kEpi == kEpiSwigluBwd) {
#pragma unroll
            for (int a = 0; a < kNumA; ++a) {
              const float dh = a == 0 ? a0 : __uint_as_float(g2[c]);
              const size_t i = row * aux.ld + feat + a * BM;
              const float gv = pg[a][c], uv = pu[a][c];
              const float sg = __fdividef(1.0f, 1.0f + __expf(-gv));
              aux.dg[i] = __float2bfloat16_rn(dh * uv * sg * (1.0f + gv * (1.0f - sg)));
              aux.du[i] = __float2bfloat16_rn(dh * gv * sg);
            }
          } else {
            __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out_ptr) + row * ld_out + feat;
            o[0] = __float2bfloat16_rn(a0);
            if constexpr (kNumA == 2) o[BM] = __float2bfloat16_rn(__uint_as_float(g2[c]));
          }
        }
      };
      auto load = [&](int c0, uint32_t (&g)[16], uint32_t (&g2)[16]) {
        tmem_ld_32x32b_x16(tb + c0, g);
        if constexpr (kNumA == 2) tmem_ld_32x32b_x16(tb + kBN + c0, g2);
      };
      if constexpr (C::kRegions > 0 && kEpi != kEpiSwigluBwd) {
        // One accumulator buffer: the next tile's MMAs wait for each 64-column
        // group.  Read this warp's two chunks of a group into registers, hand
        // the group back, then convert and store from registers, so the
        // tensor core waits only for the TMEM reads.
        for (int r = 0; r < C::kRegions; ++r) {
          const int c0 = 64 * r + 16 * half, c1 = c0 + 32;
          const bool l0 = store && c0 < it.nrows, l1 = store && c1 < it.nrows;
          uint32_t g0[16], h0[16], g1[16], h1[16];
          if (l0) load(c0, g0, h0);
          if (l1) load(c1, g1, h1);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {   // pairs: on rank 0's barrier
            if (kPair && rank != 0)
              mbar_arrive_cluster(mapa_shared(smem_u32(&bars->acc_region[r]), 0));
            else
              mbar_arrive(&bars->acc_region[r]);
          }
          if (l0) process(c0, g0, h0);
          if (l1) process(c1, g1, h1);
        }
      } else if constexpr (C::kRegions > 0) {
        // hand each 64-column group back as soon as this warp has read it
        for (int r = 0; r < C::kRegions; ++r) {
          for (int c0 = 64 * r + 16 * half; c0 < 64 * r + 64; c0 += 32)
            if (store && c0 < it.nrows) {
              uint32_t g[16], g2[16];
              load(c0, g, g2);
              tmem_ld_wait();
              process(c0, g, g2);
            }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&bars->acc_region[r]);
        }
      } else {
        if (store)
          for (int c0 = 16 * half; c0 < it.nrows; c0 += 32) {
            uint32_t g[16], g2[16];
            load(c0, g, g2);
            tmem_ld_wait();
            process(c0, g, g2);
          }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars->acc_empty[acc]);
      }
      if (dep == kDepSignal) {
        // this warp's part of the tile is in global memory: count it in
        __threadfence();   // the lanes' direct stores of a partial chunk
        __syncwarp();
        if (lane == 0) {
          if constexpr (C::kOuts > 0) bulk_wait_all();   // the TMA stores have completed
          fence_async_global();
          __threadfence();
          atomicAdd(blk_done + it.blk, 1);
        }
        __syncwarp();
      }

      if (++acc == kAccBufs) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (lane == 0) {
      if constexpr (C::kOuts > 0) bulk_wait_all();   // every staged box written
      if (!ok) {
        set_status(status, MOE_ERR_TIMEOUT, kWaitDetailEpilogue);
        raise_abort();
      }
    }
  }

  tc_fence_before();
  // pairs: neither rank leaves (or frees its tensor memory) while the other
  // may still read its shared memory, signal its barriers or write its TMEM
  if constexpr (kPair) cluster_sync(); else __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (kPair) tmem_dealloc_pair(tmem_base, C::kTmemCols);
    else tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

// ------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  // looked up once (thread-safe static initialisation)
  static const EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeTiledFn>(p);
    return nullptr;
  }();
  return fn;
}

// bf16 tensor map with a 128-byte swizzle; dims/strides innermost first.
bool make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
              const cuuint64_t* strides, const cuuint32_t* box,
              CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void*>(base), dims,
             strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// A bf16 output [rows, ld] (ld contiguous) as store boxes of 16 rows x 32
// features, unswizzled (the epilogue stages rows of 64 bytes).
bool map_out(CUtensorMap* m, const void* Y, int ld, int rows) {
  const cuuint64_t d[2] = {(cuuint64_t)ld, (cuuint64_t)rows};
  const cuuint64_t st[1] = {(cuuint64_t)ld * 2};
  const cuuint32_t box[2] = {32, 16};
  return make_map(m, Y, 2, d, st, box, CU_TENSOR_MAP_SWIZZLE_NONE);
}

}  // namespace

bool make_tensor_map_bf16(void* map, const void* base, int rank, const unsigned long long* dims,
                          const unsigned long long* strides, const unsigned int* box) {
  return make_map(static_cast<CUtensorMap*>(map), base, rank,
                  reinterpret_cast<const cuuint64_t*>(dims),
                  reinterpret_cast<const cuuint64_t*>(strides),
                  reinterpret_cast<const cuuint32_t*>(box));
}

namespace {

// A weight operand's tensor map; `atoms`: a 4-D view (64 features, K rows,
// 64-feature atoms, experts) whose one box covers a 128-feature tile.
struct WMap {
  CUtensorMap m;
  bool atoms;
};
// A token-row operand's tensor maps (boxes of 32, 64, 128, 256 rows).
struct RowMap4 {
  CUtensorMap h[4];
};

// Token rows gathered from x by the GEMM itself (see kGather).
struct Gather {
  const int32_t* sorted_src;   // row p of the expert groups is token sorted_src[p] / k
  int k;
};

// Clusters of two CTAs of `kern` that fit on the device at once (each CTA
// alone on its SM); 0 if the query fails.
template <typename Kern>
int pair_clusters(Kern kern, int smem) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * device_sm_count());
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return n;
}

// As launch_k, as clusters of two CTAs.
template <typename... KArgs, typename... Args>
cudaError_t launch_pair_k(void (*kern)(KArgs...), int grid, size_t smem, cudaStream_t s,
                          bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

template <int kNumA, int kEpi, int kBN, int kAccBufs, bool kAKMajor = false, bool kDualK = false,
          bool kGather = false, bool kPair = false>
cudaError_t launch_gemm(const WMap& a0, const WMap& a1, const RowMap4& b, const RowMap4& b1,
                        const int32_t* offsets, const int32_t* block_off,
                        const int32_t* num_blocks, const int32_t* block_expert, int M_total,
                        int K, long long nb_max, void* out, int ld_out, const EpiAux& aux,
                        const OutMaps& outs, int* status, cudaStream_t s,
                        StreamK sk = StreamK{nullptr, nullptr, 0, nullptr},
                        Gather gather = Gather{nullptr, 1}, int* blk_done = nullptr,
                        int blk_target = 0, int dep = kDepNone) {
  using C = Cfg<kNumA, kEpi, kBN, kAccBufs, kAKMajor, kDualK, kPair>;
  // one CTA per SM: a TMEM allocation never waits on another CTA of this or of
  // an overlapping launch
  static_assert(C::kSmemBytes > kSmemMax / 2, "one CTA per SM");
  auto kern = grouped_gemm_kernel<kNumA, kEpi, kBN, kAccBufs, kAKMajor, kDualK, kGather, kPair>;
  cudaError_t err =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (err != cudaSuccess) return err;
  if constexpr (kPair) {
    // a pair's tile covers 2 kFeatPerItem features (M_total a multiple of it);
    // one pair per two SMs, as many as are resident at once
    static const int clusters = pair_clusters(kern, C::kSmemBytes);
    if (clusters <= 0 || M_total % (2 * C::kFeatPerItem) != 0) return cudaErrorInvalidValue;
    const int n_mt = M_total / (2 * C::kFeatPerItem);
    const long long items = nb_max * n_mt;
    const int grid = 2 * (int)(items < clusters ? items : clusters);
    RowMaps rm;
    for (int j = 0; j < 4; ++j) rm.m[0][j] = rm.m[1][j] = b.h[j];
    const StreamK none{nullptr, nullptr, 0, nullptr};
    return launch_pair_k(kern, grid, C::kSmemBytes, s, dep == kDepWait, a0.m, a1.m, rm,
                         a0.atoms ? 1 : 0, offsets, block_off, num_blocks, block_expert, n_mt,
                         K, out, ld_out, M_total, aux, outs, none, gather.sorted_src, gather.k,
                         blk_done, blk_target, dep, status);
  }
  // a partial last feature tile (router with E not a multiple of 128) is
  // zero-filled by the TMA and not stored
  const int n_mt = (M_total + C::kFeatPerItem - 1) / C::kFeatPerItem;
  const long long items = nb_max * n_mt;
  const int grid = (int)(items < device_sm_count() ? items : device_sm_count());
  if (grid > kStreamKMaxCtas || (size_t)kNumA * BM * kBN * 4 > sk.slot_bytes) {
    sk.part = nullptr;
    sk.cnt = nullptr;
  }
  RowMaps rm;
  for (int j = 0; j < 4; ++j) {
    rm.m[0][j] = b.h[j];
    rm.m[1][j] = b1.h[j];
  }
  // a waiting launch starts early, on the SMs the previous one leaves
  return launch_k(kern, dim3(grid), dim3(kThreads), C::kSmemBytes, s, dep == kDepWait, a0.m,
                  a1.m, rm, a0.atoms ? 1 : 0, offsets, block_off, num_blocks, block_expert, n_mt,
                  K, out, ld_out, M_total, aux, outs, sk, gather.sorted_src, gather.k, blk_done,
                  blk_target, dep, status);
}

// With 256-row blocks FC2 pairs two adjacent W2 tiles whenever H allows it
// (measured faster than unpaired, double-buffered tiles on every large shape).
bool fc2_paired(int H) { return H % (2 * BM) == 0; }
// FC1 of the plain forward runs on CTA pairs (two SMs per tile, a four-stage
// ring) when the features split into pair tiles of 256 and the experts hold
// fewer than two 256-row blocks on average, where FC1 streams each weight
// tile once and is bound by HBM (measured: fine-grained layer 4.98 -> 4.88 ms).
// Where blocks share weight tiles FC1 is bound by the tensor core, and a pair
// MMA costs more than two single ones (DBRX-sized layer 3.83 -> 4.02 ms); FC2
// (32-stage tiles) gains nothing from the deeper ring either way.
bool ffn_paired_fc1(long long P, int E, int F) {
  return F % (2 * BM) == 0 && P < 2LL * kBlockRowsLarge * E;
}

struct PlanPtrs {
  const int32_t* offsets;
  const int32_t* block_off;
  const int32_t* num_blocks;
  const int32_t* block_expert;
};

// Weights as the MN-major M operand ([E, K, M] memory, M contiguous).  With M
// a multiple of 64: a 4-D view (64 features, K rows, M / 64 atoms, E) and
// boxes of two atoms x 64 K rows, one per 128-feature tile; otherwise (the
// router's narrow W_g) boxes of 64 features x 64 K rows, the features past M
// zero-filled.
bool map_weights_mn(WMap* m, const void* W, int K, int M, int E) {
  m->atoms = M % 64 == 0;
  if (m->atoms) {
    const cuuint64_t d[4] = {64, (cuuint64_t)K, (cuuint64_t)M / 64, (cuuint64_t)E};
    const cuuint64_t st[3] = {(cuuint64_t)M * 2, 128, (cuuint64_t)K * M * 2};
    const cuuint32_t box[4] = {64, (cuuint32_t)BK, 2, 1};
    return make_map(&m->m, W, 4, d, st, box);
  }
  const cuuint64_t d[3] = {(cuuint64_t)M, (cuuint64_t)K, (cuuint64_t)E};
  const cuuint64_t st[2] = {(cuuint64_t)M * 2, (cuuint64_t)K * M * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)BK, 1};
  return make_map(&m->m, W, 3, d, st, box);
}
// Weights as the K-major M operand ([E, M, K] memory, K contiguous): boxes of
// 128 rows x 64 K.
bool map_weights_k(WMap* m, const void* W, int M, int K, int E) {
  m->atoms = false;
  const cuuint64_t d[3] = {(cuuint64_t)K, (cuuint64_t)M, (cuuint64_t)E};
  const cuuint64_t st[2] = {(cuuint64_t)K * 2, (cuuint64_t)M * K * 2};
  const cuuint32_t box[3] = {(cuuint32_t)BK, (cuuint32_t)BM, 1};
  return make_map(&m->m, W, 3, d, st, box);
}
// Token rows [P, K] (K contiguous) as the N operand: boxes of 32, 64, 128 and
// 256 rows x 64 K.
bool map_rows(RowMap4* m, const void* X, int K, int P) {
  const cuuint64_t d[2] = {(cuuint64_t)K, (cuuint64_t)P};
  const cuuint64_t st[1] = {(cuuint64_t)K * 2};
  for (int j = 0; j < 4; ++j) {
    const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)(kRowBox << j)};
    if (!make_map(&m->h[j], X, 2, d, st, box)) return false;
  }
  return true;
}

// x [T, K] (K contiguous) as the source of gathered token rows: boxes of one
// row x 64 K (the only box height tile::gather4 takes), 128-byte swizzle.
bool map_gather_rows(RowMap4* m, const void* X, int K, int T) {
  const cuuint64_t d[2] = {(cuuint64_t)K, (cuuint64_t)T};
  const cuuint64_t st[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {(cuuint32_t)BK, 1};
  for (int j = 0; j < 4; ++j)
    if (!make_map(&m->h[j], X, 2, d, st, box)) return false;
  return true;
}

template <int kBN, int kBufs1>
cudaError_t launch_fc1(const WMap& mW1, const WMap& mW3, const RowMap4& mX,
                       const PlanPtrs& pl, int P, int H, int F, int E, __nv_bfloat16* h,
                       const EpiAux* save, int* status, cudaStream_t s, StreamK sk,
                       const Gather* gather, int* blk_done) {
  const long long nb_max = max_blocks(P, E, kBN);
  const int dep = blk_done != nullptr ? kDepSignal : kDepNone;
  OutMaps om;
  if (!map_out(&om.m[0], h, F, P)) return cudaErrorInvalidValue;
  if (gather != nullptr && save == nullptr)
    return launch_gemm<2, kEpiSwiglu, kBN, kBufs1, false, false, true>(
        mW1, mW3, mX, mX, pl.offsets, pl.block_off, pl.num_blocks, pl.block_expert, F, H, nb_max,
        h, F, EpiAux{}, om, status, s, sk, *gather, blk_done, 0, dep);
  if (save != nullptr) {
    if (!map_out(&om.m[1], save->g, save->ld, P) || !map_out(&om.m[2], save->u, save->ld, P))
      return cudaErrorInvalidValue;
    return launch_gemm<2, kEpiSwigluSave, kBN, kBufs1>(
        mW1, mW3, mX, mX, pl.offsets, pl.block_off, pl.num_blocks, pl.block_expert, F, H, nb_max,
        h, F, *save, om, status, s, sk);
  }
  if constexpr (kBN == kBlockRowsLarge && kBufs1 == 1) {
    if (ffn_paired_fc1(P, E, F))
      return launch_gemm<2, kEpiSwiglu, kBN, kBufs1, false, false, false, true>(
          mW1, mW3, mX, mX, pl.offsets, pl.block_off, pl.num_blocks, pl.block_expert, F, H,
          nb_max, h, F, EpiAux{}, om, status, s, sk, Gather{nullptr, 1}, blk_done, 0, dep);
  }
  return launch_gemm<2, kEpiSwiglu, kBN, kBufs1>(
      mW1, mW3, mX, mX, pl.offsets, pl.block_off, pl.num_blocks, pl.block_expert, F, H, nb_max, h,
      F, EpiAux{}, om, status, s, sk, Gather{nullptr, 1}, blk_done, 0, dep);
}

// blk_done: wait, per token block, for FC1's tiles of the block (FC1 of this
// forward ran with the same counters, F / 128 tiles per block).
template <int kNumA, int kBN, int kBufs>
cudaError_t launch_fc2(const WMap& mW2, const RowMap4& mH, const PlanPtrs& pl, int P,
                       int H, int F, int E, __nv_bfloat16* y, int* status, cudaStream_t s,
                       StreamK sk = StreamK{nullptr, nullptr, 0, nullptr},
                       int* blk_done = nullptr) {
  OutMaps om;
  if (!map_out(&om.m[0], y, H, P)) return cudaErrorInvalidValue;
  return launch_gemm<kNumA, kEpiBf16, kBN, kBufs>(
      mW2, mW2, mH, mH, pl.offsets, pl.block_off, pl.num_blocks, pl.block_expert, H, F,
      max_blocks(P, E, kBN), y, H, EpiAux{}, om, status, s, sk, Gather{nullptr, 1}, blk_done,
      (F / BM) * kEpiWarps, blk_done != nullptr ? kDepWait : kDepNone);
}

// kPairF / kPairH: pair adjacent weight tiles (single-buffered accumulators)
// in the dh / dx products; worth it for large blocks, whose long K keeps the
// unoverlapped epilogue a small share of a tile.
template <int kBN, bool kPairF, bool kPairH>
cudaError_t launch_dgrad_t(const WMap& mW2k, const RowMap4& mDY, const WMap& mW1k,
                           const WMap& mW3k, const RowMap4& mDG, const RowMap4& mDU,
                           const PlanPtrs& pl,
                           int P, int H, int F, int E, const EpiAux& aux,
                           __nv_bfloat16* dx_perm, int* status, cudaStream_t s,
                           StreamK sk = StreamK{nullptr, nullptr, 0, nullptr}) {
  const long long nb_max = max_blocks(P, E, kBN);
  constexpr int kAF = kPairF ? 2 : 1, kBufF = kPairF ? 1 : 2;
  constexpr int kAH = kPairH ? 2 : 1, kBufH = kPairH ? 1 : 2;
  // dh = dY W2[e]^T (M = F, K = H), then the SwiGLU derivative -> dg, du
  OutMaps oh, ox;
  if (!map_out(&oh.m[0], aux.dg, aux.ld, P) || !map_out(&oh.m[1], aux.du, aux.ld, P) ||
      !map_out(&ox.m[0], dx_perm, H, P))
    return cudaErrorInvalidValue;
  cudaError_t err = launch_gemm<kAF, kEpiSwigluBwd, kBN, kBufF, true>(
      mW2k, mW2k, mDY, mDY, pl.offsets, pl.block_off, pl.num_blocks, pl.block_expert, F, H,
      nb_max, nullptr, 0, aux, oh, status, s, sk);
  if (err != cudaSuccess) return err;
  // dx_perm = dg W1[e]^T + du W3[e]^T (M = H, K = F in two phases)
  return launch_gemm<kAH, kEpiBf16, kBN, kBufH, true, true>(
      mW1k, mW3k, mDG, mDU, pl.offsets, pl.block_off, pl.num_blocks, pl.block_expert, H, F,
      nb_max, dx_perm, H, EpiAux{}, ox, status, s, sk);
}

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
                               cudaStream_t s, cudaEvent_t after_fc1, const EpiAux* save,
                               const StreamKSpace* sks, const GatherRows* gather_rows,
                               int* blk_done) {
  if (P == 0) return cudaSuccess;
  // FC2 overlaps FC1 block by block (no event between them, plain forward)
  if (after_fc1 != nullptr || save != nullptr) blk_done = nullptr;
  const bool gathered = gather_rows != nullptr && save == nullptr;
  const FfnMode mode = ffn_mode(P, E);
  WMap mW1, mW3, mW2;
  RowMap4 mX, mH;
  if (!map_weights_mn(&mW1, W1, H, F, E) || !map_weights_mn(&mW3, W3, H, F, E) ||
      !map_weights_mn(&mW2, W2, F, H, E) || !map_rows(&mH, h, F, P))
    return cudaErrorInvalidValue;
  if (gathered ? !map_gather_rows(&mX, gather_rows->x, H, gather_rows->T)
               : !map_rows(&mX, x_perm, H, P))
    return cudaErrorInvalidValue;
  const Gather g{gathered ? gather_rows->sorted_src : nullptr, gathered ? gather_rows->k : 1};
  const Gather* gp = gathered ? &g : nullptr;
  const PlanPtrs pl{offsets, block_off, num_blocks, block_expert};
  // Balanced K split when the tiles do not fill the SMs evenly.  Tiles come
  // from the on-device queue when their costs differ: 256-row blocks with
  // fewer than two blocks per expert on average, where one expert's rows fill
  // a whole block and the next one's are cut into two smaller ones (measured:
  // fine-grained 1% faster with the queue; uniform blocks -- DBRX, decode --
  // 0.3-1.3% faster in the fixed order).
  const bool queue = mode == FfnMode::kLarge && (long long)P < 2LL * kBlockRowsLarge * E;
  // FC1 and FC2 draw from queue heads of their own (they may overlap)
  const StreamK sk =
      sks ? StreamK{sks->part, sks->cnt, sks->slot_bytes,
                    queue ? sks->cnt + kStreamKMaxCtas : nullptr}
          : StreamK{nullptr, nullptr, 0, nullptr};
  StreamK sk2 = sk;
  if (sk2.queue != nullptr) sk2.queue = sks->cnt + kStreamKMaxCtas + 1;
  cudaError_t err;
  if (mode == FfnMode::kTiny)
    err = launch_fc1<kBlockRowsTiny, 2>(mW1, mW3, mX, pl, P, H, F, E, h, save, status, s, sk, gp,
                                        blk_done);
  else if (mode == FfnMode::kSmall)
    err = launch_fc1<kBlockRows, 2>(mW1, mW3, mX, pl, P, H, F, E, h, save, status, s, sk, gp,
                                    blk_done);
  else
    err = launch_fc1<kBlockRowsLarge, 1>(mW1, mW3, mX, pl, P, H, F, E, h, save, status, s, sk,
                                         gp, blk_done);
  if (err != cudaSuccess) return err;
  if (after_fc1 != nullptr && (err = cudaEventRecord(after_fc1, s)) != cudaSuccess) return err;
  if (mode == FfnMode::kTiny)
    return launch_fc2<1, kBlockRowsTiny, 2>(mW2, mH, pl, P, H, F, E, y, status, s, sk2,
                                            blk_done);
  if (mode == FfnMode::kSmall)
    return launch_fc2<1, kBlockRows, 2>(mW2, mH, pl, P, H, F, E, y, status, s, sk2, blk_done);
  if (fc2_paired(H))
    return launch_fc2<2, kBlockRowsLarge, 1>(mW2, mH, pl, P, H, F, E, y, status, s, sk2,
                                             blk_done);
  return launch_fc2<1, kBlockRowsLarge, 2>(mW2, mH, pl, P, H, F, E, y, status, s, sk2,
                                           blk_done);
}

cudaError_t launch_dgrad(const __nv_bfloat16* dY, const __nv_bfloat16* g, const __nv_bfloat16* u,
                         const __nv_bfloat16* W1, const __nv_bfloat16* W3,
                         const __nv_bfloat16* W2, const int32_t* offsets,
                         const int32_t* block_off, const int32_t* num_blocks,
                         const int32_t* block_expert, int P, int H, int F, int E,
                         __nv_bfloat16* dg, __nv_bfloat16* du, __nv_bfloat16* dx_perm,
                         int* status, cudaStream_t s, const StreamKSpace* sks) {
  if (P == 0) return cudaSuccess;
  // fixed tile order (measured: the queue no faster for the backward products)
  const StreamK sk =
      sks ? StreamK{sks->part, sks->cnt, sks->slot_bytes, nullptr}
          : StreamK{nullptr, nullptr, 0, nullptr};
  WMap mW2k, mW1k, mW3k;
  RowMap4 mDY, mDG, mDU;
  if (!map_weights_k(&mW2k, W2, F, H, E) || !map_weights_k(&mW1k, W1, H, F, E) ||
      !map_weights_k(&mW3k, W3, H, F, E) || !map_rows(&mDY, dY, H, P) ||
      !map_rows(&mDG, dg, F, P) || !map_rows(&mDU, du, F, P))
    return cudaErrorInvalidValue;
  const PlanPtrs pl{offsets, block_off, num_blocks, block_expert};
  const EpiAux aux{const_cast<__nv_bfloat16*>(g), const_cast<__nv_bfloat16*>(u), dg, du, F};
  switch (ffn_mode(P, E)) {
    case FfnMode::kTiny:
      return launch_dgrad_t<kBlockRowsTiny, false, false>(mW2k, mDY, mW1k, mW3k, mDG, mDU, pl, P,
                                                          H, F, E, aux, dx_perm, status, s, sk);
    case FfnMode::kSmall:
      return launch_dgrad_t<kBlockRows, false, false>(mW2k, mDY, mW1k, mW3k, mDG, mDU, pl, P, H,
                                                      F, E, aux, dx_perm, status, s, sk);
    default: {
      const bool pf = F % (2 * BM) == 0, ph = H % (2 * BM) == 0;
      if (pf && ph)
        return launch_dgrad_t<kBlockRowsLarge, true, true>(mW2k, mDY, mW1k, mW3k, mDG, mDU, pl,
                                                           P, H, F, E, aux, dx_perm, status, s, sk);
      if (pf)
        return launch_dgrad_t<kBlockRowsLarge, true, false>(mW2k, mDY, mW1k, mW3k, mDG, mDU, pl,
                                                            P, H, F, E, aux, dx_perm, status, s, sk);
      if (ph)
        return launch_dgrad_t<kBlockRowsLarge, false, true>(mW2k, mDY, mW1k, mW3k, mDG, mDU, pl,
                                                            P, H, F, E, aux, dx_perm, status, s, sk);
      return launch_dgrad_t<kBlockRowsLarge, false, false>(mW2k, mDY, mW1k, mW3k, mDG, mDU, pl,
                                                           P, H, F, E, aux, dx_perm, status, s, sk);
    }
  }
}

cudaError_t launch_router_gemm(const __nv_bfloat16* x, const __nv_bfloat16* Wg, int T, int H,
                               int E, const int32_t* offsets, const int32_t* block_off,
                               const int32_t* num_blocks, const int32_t* block_expert,
                               float* logits, int* status, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  // logits^T = Wg^T x^T: one "expert" whose weight matrix is Wg [H, E]
  WMap mG;
  RowMap4 mX;
  if (!map_weights_mn(&mG, Wg, H, E, 1) || !map_rows(&mX, x, H, T)) return cudaErrorInvalidValue;
  const PlanPtrs pl{offsets, block_off, num_blocks, block_expert};
  switch (ffn_mode(T, 1)) {
    case FfnMode::kTiny:
      return launch_gemm<1, kEpiF32, kBlockRowsTiny, 2>(mG, mG, mX, mX, pl.offsets, pl.block_off,
                                                        pl.num_blocks, pl.block_expert, E, H,
                                                        max_blocks(T, 1, kBlockRowsTiny), logits,
                                                        E, EpiAux{}, OutMaps{}, status, s);
    case FfnMode::kSmall:
      return launch_gemm<1, kEpiF32, kBlockRows, 2>(mG, mG, mX, mX, pl.offsets, pl.block_off,
                                                    pl.num_blocks, pl.block_expert, E, H,
                                                    max_blocks(T, 1, kBlockRows), logits, E,
                                                    EpiAux{}, OutMaps{}, status, s);
    default:
      return launch_gemm<1, kEpiF32, kBlockRowsLarge, 2>(
          mG, mG, mX, mX, pl.offsets, pl.block_off, pl.num_blocks, pl.block_expert, E, H,
          max_blocks(T, 1, kBlockRowsLarge), logits, E, EpiAux{}, OutMaps{}, status, s);
  }
}

}  // namespace moe
