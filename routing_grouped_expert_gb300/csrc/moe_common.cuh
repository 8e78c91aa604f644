// Internal definitions shared by the libmoe translation units: tile sizes,
// workspace layout, device status word, small device helpers.
#pragma once

#include <utility>

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <stddef.h>

#include "../../include/moe.h"

namespace moe {

// ---------------------------------------------------------------- tiling
// Token block: at most beta routed rows of one expert (MegaFlux, §3.1).  The
// block is the N side of the expert GEMM tile; the M side is kTileM output
// features.  beta is 64 for decode batches (few rows per expert), 128 for
// moderate ones and 256 for large ones; block tables are sized for the
// smallest beta.
constexpr int kBlockRowsTiny = 64;
constexpr int kBlockRows = 128;
constexpr int kBlockRowsLarge = 256;
constexpr int kTileM = 128;
constexpr int kTileK = 64;           // one 128-byte swizzle atom of bf16
constexpr int kRowBox = 32;          // token rows per TMA box of the N operand
constexpr int kGroupBlocks = 16;     // blocks of one expert rastered together

// Upper bound of the number of token blocks over all experts.
inline __host__ __device__ long long max_blocks(long long P, int E, int beta = kBlockRows) {
  const long long nonempty = P < E ? P : E;
  return (P + beta - 1) / beta + nonempty;
}

// Tile configuration of the grouped FFN, a function of the routed rows P
// and the expert count E (mean rows per expert P/E):
//   tiny  (mean <= 40): 64-row blocks;
//   small (mean <= 80): 128-row blocks;
//   large            : 256-row blocks, two weight tiles per CTA tile.
// With uniform routing the largest expert stays within one block in the
// tiny and small modes.
enum class FfnMode { kTiny, kSmall, kLarge };
constexpr int kTinyModeMeanRows = 40;
constexpr int kSmallModeMeanRows = 80;
inline FfnMode ffn_mode(long long P, int E) {
  if (P <= (long long)kTinyModeMeanRows * E) return FfnMode::kTiny;
  if (P <= (long long)kSmallModeMeanRows * E) return FfnMode::kSmall;
  return FfnMode::kLarge;
}
inline int ffn_block_rows_of(long long P, int E) {
  switch (ffn_mode(P, E)) {
    case FfnMode::kTiny: return kBlockRowsTiny;
    case FfnMode::kSmall: return kBlockRows;
    default: return kBlockRowsLarge;
  }
}
// Permute chunking: one CTA handles the assignments of kChunkAssign / k
// consecutive tokens (at most kChunkAssign assignments).
constexpr int kChunkAssign = 512;
inline __host__ __device__ int tokens_per_chunk(int k) { return kChunkAssign / k; }
inline __host__ __device__ int num_chunks(int T, int k) {
  const int tpc = tokens_per_chunk(k);
  return (T + tpc - 1) / tpc;
}

// --------------------------------------------------------- device status
// ws[0]: first error code seen by any kernel (MOE_OK if none);
// ws[1]: a detail word (which wait timed out) for diagnostics.
enum : int { kWaitDetailProducer = 1, kWaitDetailMma = 2, kWaitDetailEpilogue = 3,
             kWaitDetailDrain = 4 };

__device__ __forceinline__ void set_status(int* status, int code, int detail = 0) {
  if (atomicCAS(status, 0, code) == 0 && detail) status[1] = detail;
}

// ------------------------------------------------------ workspace layout
// CTAs whose FC2 partial tiles the workspace has room for (a launch with a
// larger grid does not split tiles).
constexpr int kStreamKMaxCtas = 256;
// The split counters are followed by the grouped GEMM's tile-queue heads (FC1
// and FC2, one int each, padded to 128 bytes); all are zero between launches.
constexpr int kSkCntInts = kStreamKMaxCtas + 32;

struct WsLayout {
  size_t status;        // int32[64]
  size_t sk_cnt;        // int32[kSkCntInts]   split counters, then the tile-queue heads (cleared with status)
  size_t blk_done;      // int32[max_blocks]   FC1 tiles done per token block (cleared with status)
  size_t topk_idx;      // int32[P]
  size_t topk_w;        // f32[P]
  size_t counts;        // int32[E]
  size_t offsets;       // int32[E+1]
  size_t sorted_src;    // int32[P]
  size_t dest_of;       // int32[P]
  size_t chunk_base;    // int32[C*E]   per-chunk histograms, then bases
  size_t block_off;     // int32[E+1]
  size_t num_blocks;    // int32[1]
  size_t block_expert;  // int32[max_blocks]
  size_t x_perm;        // bf16[P*H]
  size_t h;             // bf16[P*F]
  size_t y;             // bf16[P*H]
  size_t sk_part;       // f32 [kStreamKMaxCtas][2] slots of sk_slot bytes: split partials
  size_t sk_slot;       // bytes of one slot: a 128-row accumulator of the layer's block size
  size_t stage_x;       // bf16[T*H]   device staging for moe_forward_host
  size_t stage_logits;  // f32[T*E]
  size_t stage_out;     // bf16[T*H]
  size_t total;
};

// Workspace of a training step (moe_forward_train, then moe_backward): the
// forward layout, whose routing, x_perm, h and y_sorted the backward reads,
// then the saved pre-activations and the backward's intermediates.
struct TrainLayout {
  WsLayout base;
  size_t g, u;          // bf16[P*F]
  size_t dY;            // bf16[P*H]
  size_t dg, du;        // bf16[P*F]
  size_t dx_perm;       // bf16[P*H]
  size_t total;
};

// Workspace of the layer from hidden states (router projection + routed
// experts + optional shared expert): the routed layout, then these regions.
struct GatedLayout {
  WsLayout base;
  size_t logits;        // f32[T*E]
  size_t s_offsets;     // int32[2]
  size_t s_block_off;   // int32[2]
  size_t s_num_blocks;  // int32[1]
  size_t s_block_expert;// int32[max_blocks(T, 1)]
  size_t s_h;           // bf16[T*Fs]
  size_t s_y;           // bf16[T*H]
  size_t total;
};

inline __host__ __device__ size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

inline WsLayout ws_layout(int T, int H, int F, int E, int k) {
  const size_t P = (size_t)T * k;
  const size_t C = (size_t)num_chunks(T, k);
  WsLayout L{};
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 1024); return at; };
  L.status = take(64 * 4);
  L.sk_cnt = take((size_t)kSkCntInts * 4);
  L.blk_done = take((size_t)max_blocks((long long)P, E, kBlockRowsTiny) * 4 + 4);
  L.chunk_base = take(C * E * 4);   // after status, sk_cnt, blk_done: one memset clears all
  L.topk_idx = take(P * 4);
  L.topk_w = take(P * 4);
  L.counts = take((size_t)E * 4);
  L.offsets = take((size_t)(E + 1) * 4);
  L.sorted_src = take(P * 4);
  L.dest_of = take(P * 4);
  L.block_off = take((size_t)(E + 1) * 4);
  L.num_blocks = take(4);
  L.block_expert = take((size_t)max_blocks((long long)P, E, kBlockRowsTiny) * 4 + 4);
  L.x_perm = take(P * H * 2);
  L.h = take(P * F * 2);
  L.y = take(P * H * 2);
  L.sk_slot = (size_t)kTileM * ffn_block_rows_of(P, E) * 4;
  L.sk_part = take((size_t)kStreamKMaxCtas * 2 * L.sk_slot);
  L.stage_x = take((size_t)T * H * 2);   // the host-buffer staging comes last
  L.stage_logits = take((size_t)T * E * 4);
  L.stage_out = take((size_t)T * H * 2);
  L.total = o;
  return L;
}

inline TrainLayout train_layout(int T, int H, int F, int E, int k) {
  TrainLayout R{};
  R.base = ws_layout(T, H, F, E, k);
  const size_t P = (size_t)T * k;
  size_t o = R.base.total;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 1024); return at; };
  R.g = take(P * F * 2);
  R.u = take(P * F * 2);
  R.dY = take(P * H * 2);
  R.dg = take(P * F * 2);
  R.du = take(P * F * 2);
  R.dx_perm = take(P * H * 2);
  R.total = o;
  return R;
}

inline GatedLayout gated_layout(int T, int H, int F, int Fs, int E, int k) {
  GatedLayout G{};
  G.base = ws_layout(T, H, F, E, k);
  size_t o = G.base.total;
  auto take = [&](size_t bytes) { size_t at = o; o = align_up(o + bytes, 1024); return at; };
  G.logits = take((size_t)T * E * 4);
  G.s_offsets = take(2 * 4);
  G.s_block_off = take(2 * 4);
  G.s_num_blocks = take(4);
  G.s_block_expert = take((size_t)max_blocks(T, 1, kBlockRowsTiny) * 4 + 4);
  G.s_h = take((size_t)T * (Fs > 0 ? Fs : 0) * 2);
  G.s_y = take((size_t)T * H * 2);
  G.total = o;
  return G;
}

template <typename Tp>
inline Tp* ws_ptr(void* ws, size_t off) { return reinterpret_cast<Tp*>((char*)ws + off); }

// -------------------------------------------- programmatic dependent launch
// The fused forward launches its chain of kernels with programmatic stream
// serialisation: a kernel may start while its predecessor on the stream still
// runs.  Such a kernel calls pdl_wait() before it touches memory that earlier
// kernels of the chain write, and pdl_trigger() only after that wait, so that
// when any kernel of the chain starts, every kernel before its direct
// predecessor has completed.  Without the launch attribute both are no-ops.
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                            cudaStream_t s, bool pdl, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? &attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ------------------------------------------------------------ launchers
// Each returns cudaSuccess or the launch error.  All enqueue on `s`; `pdl`
// launches with programmatic stream serialisation (see above).
cudaError_t launch_route(const float* logits, int T, int E, int k, int32_t* topk_idx,
                         float* topk_w, int32_t* chunk_hist, int* status, cudaStream_t s);
cudaError_t launch_count(const int32_t* topk_idx, int T, int E, int k, int32_t* chunk_hist,
                         int* status, cudaStream_t s);
cudaError_t launch_scan(int32_t* chunk_hist, int C, int E, int32_t* counts, int32_t* offsets,
                        int32_t* block_off, int32_t* num_blocks, int32_t* block_expert,
                        int beta, cudaStream_t s, bool pdl = false);
// Small batches: route, counts, scan, block plan and scatter in one launch
// instead of three, same results.  `ticket` is an int that holds zero
// between launches (the kernel leaves it zero).
constexpr int kSmallRouteAssign = 1024;
constexpr int kSmallRouteExperts = 256;
inline bool route_permute_small_ok(int T, int E, int k) {
  return (long long)T * k <= kSmallRouteAssign && E <= kSmallRouteExperts;
}
cudaError_t launch_route_permute_small(const float* logits, int T, int E, int k, int beta,
                                      int32_t* topk_idx, float* topk_w, int32_t* counts,
                                      int32_t* offsets, int32_t* block_off, int32_t* num_blocks,
                                      int32_t* block_expert, int32_t* sorted_src,
                                      int32_t* dest_of, int* ticket, int* status,
                                      cudaStream_t s);
// Out-of-range expert indices take no position: dest_of = -1 for them and
// sorted_src[offsets[E] .. T*k) = -1.
cudaError_t launch_scatter(const int32_t* topk_idx, int T, int E, int k,
                           const int32_t* chunk_base, const int32_t* offsets,
                           int32_t* sorted_src, int32_t* dest_of, cudaStream_t s,
                           bool pdl = false);
// Block plan of caller-supplied offsets of P rows; offsets that do not group
// P rows set MOE_ERR_INVALID_ARG in `status` and leave an empty plan.
cudaError_t launch_plan(const int32_t* offsets, int E, int P, int32_t* block_off,
                        int32_t* num_blocks, int32_t* block_expert, int beta, int* status,
                        cudaStream_t s);
// Token-block rows (beta) the grouped FFN uses for a layer of these sizes;
// the block plan must be built with the same value.
int ffn_block_rows(int P, int E, int H, int F);
// True when FC1 gathers its token rows from x itself (tile::gather4 loads,
// four rows per instruction) instead of reading an expert-ordered copy
// x_perm: only with small token blocks (the tiny mode, at most 64 rows), where
// a stage's gather instructions take less time than its MMAs.  Measured: with
// 256-row blocks the gather loads made the fine-grained FC1 2.6x slower.
inline bool ffn_gathers_rows(long long P, int E) { return ffn_mode(P, E) == FfnMode::kTiny; }
// x_perm[p] = x[sorted_src[p] / k] (positions holding -1 skipped).
cudaError_t launch_gather(const __nv_bfloat16* x, const int32_t* sorted_src, int P, int H, int k,
                          __nv_bfloat16* x_perm, cudaStream_t s, bool pdl = false);
// The same rows from the token side: x_perm[dest_of[t * k + j]] = x[t], each
// row of x read once.
cudaError_t launch_gather_tokens(const __nv_bfloat16* x, const int32_t* dest_of, int T, int H,
                                 int k, __nv_bfloat16* x_perm, cudaStream_t s, bool pdl = false);
// Extra tensors of the grouped-GEMM epilogues that read or write more than
// their main output.
struct EpiAux {
  __nv_bfloat16* g;    // [rows, ld]  gate pre-activation x W1
  __nv_bfloat16* u;    // [rows, ld]  up projection x W3
  __nv_bfloat16* dg;   // [rows, ld]  gradients of g and u (backward)
  __nv_bfloat16* du;
  int ld;
};
// Scratch of the grouped GEMM: partial tiles and boundary counters of the
// balanced K split, and the head of the tile queue.  The counters must be zero
// before a launch; every launch that completes leaves them zero.
struct StreamKSpace {
  float* part;         // [kStreamKMaxCtas][2] slots of slot_bytes (fp32 partial tiles)
  int* cnt;            // [kSkCntInts]: split counters, then the queue head at kStreamKMaxCtas
  size_t slot_bytes;
};
// Where FC1 takes its token rows from when it gathers them itself: row p of
// the expert groups is x[sorted_src[p] / k].
struct GatherRows {
  const __nv_bfloat16* x;      // [T, H]
  const int32_t* sorted_src;   // [T * k]
  int k, T;
};
// FC1 (+SwiGLU) and FC2 over the expert groups.  FC1's token rows are rows of
// x_perm (expert order), or, with `gather` (and no `save`), gathered from x
// by the GEMM's own loads.  With `save`, FC1 also keeps its pre-activations
// g = x W1, u = x W3 (bf16, [P, F]) for the backward.  With `blk_done` (one
// zeroed int per token block, no `after_fc1` event, no `save`) FC2 starts on
// the SMs FC1 leaves and waits, per token block, only for the FC1 tiles of
// that block.
cudaError_t launch_grouped_ffn(const __nv_bfloat16* x_perm, const int32_t* offsets,
                               const int32_t* block_off, const int32_t* num_blocks,
                               const int32_t* block_expert, const __nv_bfloat16* W1,
                               const __nv_bfloat16* W3, const __nv_bfloat16* W2, int P, int H,
                               int F, int E, __nv_bfloat16* h, __nv_bfloat16* y, int* status,
                               cudaStream_t s, cudaEvent_t after_fc1 = nullptr,
                               const EpiAux* save = nullptr,
                               const StreamKSpace* sks = nullptr,
                               const GatherRows* gather = nullptr,
                               int* blk_done = nullptr);
// Backward DGrad of both expert GEMMs: dh = dY W2^T -> dg, du (SwiGLU
// derivative from the saved g, u), dx_perm = dg W1^T + du W3^T.
cudaError_t launch_dgrad(const __nv_bfloat16* dY, const __nv_bfloat16* g, const __nv_bfloat16* u,
                         const __nv_bfloat16* W1, const __nv_bfloat16* W3,
                         const __nv_bfloat16* W2, const int32_t* offsets,
                         const int32_t* block_off, const int32_t* num_blocks,
                         const int32_t* block_expert, int P, int H, int F, int E,
                         __nv_bfloat16* dg, __nv_bfloat16* du, __nv_bfloat16* dx_perm,
                         int* status, cudaStream_t s, const StreamKSpace* sks = nullptr);
// out[t] = sum_j w[t,j] y_sorted[dest_of[t*k+j]] (+ y_shared[t] when given)
cudaError_t launch_combine(const __nv_bfloat16* y_sorted, const int32_t* dest_of,
                           const float* topk_w, int T, int H, int k, __nv_bfloat16* out,
                           cudaStream_t s, const __nv_bfloat16* y_shared = nullptr,
                           bool pdl = false);

// The same sum left in fp32 (no rounding), no shared expert.
cudaError_t launch_combine_f32(const __nv_bfloat16* y_sorted, const int32_t* dest_of,
                               const float* topk_w, int T, int H, int k, float* out,
                               cudaStream_t s, bool pdl = false);

// out[i] = bf16(in[i]) (round to nearest even).
cudaError_t launch_cast_bf16(const float* in, __nv_bfloat16* out, size_t n, cudaStream_t s);

// Block plan of one expert that takes every token in order (router GEMM,
// shared expert): offsets = {0, T}.
struct SingleExpertPlan {
  int32_t* offsets;       // [2]
  int32_t* block_off;     // [2]
  int32_t* num_blocks;    // [1]
  int32_t* block_expert;  // [max_blocks(T, 1)]
};
cudaError_t launch_single_expert_plan(int T, int beta, const SingleExpertPlan& plan,
                                      cudaStream_t s);
cudaError_t launch_router_gemm(const __nv_bfloat16* x, const __nv_bfloat16* Wg, int T, int H,
                               int E, const int32_t* offsets, const int32_t* block_off,
                               const int32_t* num_blocks, const int32_t* block_expert,
                               float* logits, int* status, cudaStream_t s);
// logits[T, E] fp32 = x[T, H] W_g[H, E]; E >= 64 on the tensor cores (the
// plan must then be built with ffn_block_rows(T, 1, .., ..)).
cudaError_t launch_router(const __nv_bfloat16* x, const __nv_bfloat16* Wg, int T, int H, int E,
                          const SingleExpertPlan& plan, float* logits, int* status,
                          cudaStream_t s);

// Backward steps (training).
cudaError_t launch_scale_gather(const __nv_bfloat16* dout, const int32_t* dest_of,
                                const float* topk_w, int T, int H, int k, __nv_bfloat16* dY,
                                cudaStream_t s);
cudaError_t launch_dw_dlogits(const __nv_bfloat16* dout, const __nv_bfloat16* y,
                              const int32_t* dest_of, const int32_t* topk_idx,
                              const float* logits, int T, int H, int E, int k, float* dlogits,
                              cudaStream_t s);
cudaError_t launch_wgrad(const __nv_bfloat16* x_perm, const __nv_bfloat16* h,
                         const __nv_bfloat16* dY, const __nv_bfloat16* dg,
                         const __nv_bfloat16* du, const int32_t* offsets, int P, int H, int F,
                         int E, __nv_bfloat16* dW1, __nv_bfloat16* dW3, __nv_bfloat16* dW2,
                         int* status, cudaStream_t s);

// The expert-replica planner (planner.cu): workspace bytes and launch.
// rounds = the searches' round limit (s + 2); lam < 0: no reduction penalty.
size_t plan_ws_bytes(int E, int G);
cudaError_t launch_plan_replicas(const int32_t* counts, int E, int G, int beta, int budget,
                                 int rounds, long long lam, void* ws, int32_t* n_out,
                                 int32_t* rows_out, int32_t* load_out, int32_t* info,
                                 cudaStream_t s);

// bf16 TMA tensor map with a 128-byte swizzle; dims/strides innermost first.
bool make_tensor_map_bf16(void* map /* CUtensorMap* */, const void* base, int rank,
                          const unsigned long long* dims, const unsigned long long* strides,
                          const unsigned int* box);

// Number of SMs of the current device (cached per device).
int device_sm_count();
// True when the current device is compute capability 10.3.
bool device_is_sm103();

}  // namespace moe
