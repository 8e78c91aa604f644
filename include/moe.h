/*
 * libmoe -- C ABI of the MoE expert-layer forward on one GPU (sm_103a).
 *
 * The layer:  out[t] = sum_{j<k} w[t,j] * FFN_{e[t,j]}(x[t]),
 *             FFN_e(x) = (silu(x W1[e]) * (x W3[e])) W2[e],
 * computed as four steps -- top-k gating, scatter into per-expert groups,
 * per-expert SwiGLU FFN, weighted return to token order -- following
 * "MegaScale-Infer: Serving Mixture-of-Experts at Scale with Disaggregated
 * Expert Parallelism" (§3.2 Big-Picture Architecture, steps (1)-(5);
 * §3.4 Supporting Implementation Details, Fused Kernels, steps (1)-(4)),
 * "MegaFlux: Skew-Resilient MoE Megakernels via Pipelined Expert
 * Replication" (§2.1, §3.1, §A.2) and "Piper: Efficient Large-Scale MoE
 * Training via Resource Modeling and Pipelined Hybrid Parallelism"
 * (§III-A, Table III).
 *
 * Conventions shared by every entry point
 *   - Tensor pointers are DEVICE pointers owned by the caller, row-major and
 *     contiguous, 16-byte aligned.  bf16 tensors are passed as void* and
 *     hold IEEE bfloat16 (__nv_bfloat16) values.  The library never
 *     allocates, frees or keeps a reference to caller memory beyond a call.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *     call only enqueues work on `stream` and returns; nothing synchronises
 *     except moe_get_device_status.
 *   - `ws` is a caller-owned device workspace of at least
 *     moe_workspace_size(T, H, F, E, k) bytes, 256-byte aligned.  It holds
 *     the intermediates (gathered rows, expert activations and outputs),
 *     8 to 32 MiB of partial tiles for the balanced K split of FC2, the
 *     head of the grouped GEMM's tile queue, and a device status word.  Its
 *     contents need no initialisation (each layer call clears the counters).  Calls that
 *     share one workspace must not overlap in time (use one stream per
 *     workspace).
 *   - Limits: 0 <= T, T*k < 2^31; 1 <= E <= MOE_MAX_EXPERTS;
 *     1 <= k <= min(E, MOE_MAX_TOPK); H and F positive multiples of 128.
 *     Violations are reported synchronously as MOE_ERR_INVALID_ARG and
 *     nothing is enqueued.  T == 0 is a valid no-op.
 *   - Conditions only the device can see (a non-finite router logit, a
 *     pipeline wait that ran out) are written to the status word in `ws`
 *     and read back with moe_get_device_status; the kernels never trap.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_MAX_EXPERTS 1024
#define MOE_MAX_TOPK 32

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* bad size, null or misaligned pointer       */
  MOE_ERR_NONFINITE = 2,    /* a router logit is NaN or +-inf (device)    */
  MOE_ERR_TIMEOUT = 3,      /* a bounded device wait ran out (device)     */
  MOE_ERR_WORKSPACE = 4,    /* ws is NULL, too small or misaligned        */
  MOE_ERR_CUDA = 5,         /* a CUDA runtime call or launch failed       */
  MOE_ERR_UNSUPPORTED = 6   /* no sm_103a device is current               */
} moe_status;

/* Bytes of workspace needed for a layer of these sizes (0 on bad sizes). */
size_t moe_workspace_size(int T, int H, int F, int E, int k);

/*
 * Step 1 -- top-k gating and weight normalisation
 * ("MegaScale-Infer", §3.4 Fused Kernels, steps (1) and (3)).
 *
 *   logits   [T, E] fp32 router output.
 *   topk_idx [T, k] int32 out: slot j is the j-th largest logit of the token;
 *            equal logits (also -0.0 vs +0.0) go to the lower expert index.
 *   topk_w   [T, k] fp32 out: softmax over the k selected logits (they sum
 *            to 1).
 * A NaN or infinite logit sets MOE_ERR_NONFINITE in the device status; the
 * outputs of that token are then unspecified.
 */
moe_status moe_route_topk(const float* logits, int T, int E, int k,
                          int32_t* topk_idx, float* topk_w,
                          void* ws, size_t ws_bytes, void* stream);

/*
 * Step 2 -- per-expert counts and the stable scatter into expert groups
 * ("MegaScale-Infer", §3.4 Fused Kernels, steps (2) and (4); order inside an
 * expert by token, then top-k position: "MegaFlux", §A.2).
 *
 * Assignment a = t*k + j.
 *   topk_idx   [T, k] int32 in, values in [0, E).
 *   counts     [E]    int32 out: assignments per expert (sum = T*k).
 *   offsets    [E+1]  int32 out: exclusive prefix sum of counts.
 *   sorted_src [T*k]  int32 out: sorted_src[p] = a, p ascending within each
 *              expert's range [offsets[e], offsets[e+1]) in ascending a.
 *   dest_of    [T*k]  int32 out: inverse map, sorted_src[dest_of[a]] == a.
 * Deterministic: bit-identical on every run.  An expert index outside
 * [0, E) sets MOE_ERR_INVALID_ARG in the device status; that assignment is
 * left out of the counts and takes no position: its dest_of is -1, and
 * sorted_src[offsets[E] .. T*k) holds -1.  The other assignments are grouped
 * as above.  moe_grouped_ffn and moe_combine skip positions and slots marked
 * -1, so a bad index never turns into a memory access.
 */
moe_status moe_permute(const int32_t* topk_idx, int T, int E, int k,
                       int32_t* counts, int32_t* offsets,
                       int32_t* sorted_src, int32_t* dest_of,
                       void* ws, size_t ws_bytes, void* stream);

/*
 * Step 3 -- per-expert SwiGLU FFN as a grouped GEMM over the expert groups
 * ("Piper", §III-A: W_gate, W_up in R^{d x dffn}, W_down in R^{dffn x d};
 * "MegaScale-Infer", §3.4 Performance Simulation Model: FFN Input and FFN
 * Output GEMMs; token blocks of at most beta rows per expert: "MegaFlux",
 * §3.1).  beta is 64, 128 or 256 rows, chosen from the mean rows per expert
 * (T*k/E at most 40, at most 80, above); an expert's rows are cut into
 * ceil(rows / beta) blocks of equal size (a multiple of 16 rows), so no block
 * is a near-empty tail.  The groups are unpadded: nothing is stored for rows
 * past offsets[E].
 *
 *   x          [T, H] bf16.
 *   sorted_src [T*k], offsets [E+1] as produced by moe_permute (positions
 *              holding -1 are skipped).  offsets that do not group T*k rows
 *              (offsets[0] != 0, a decrease, offsets[E] > T*k) set
 *              MOE_ERR_INVALID_ARG in the device status and nothing is
 *              computed.
 *   W1, W3     [E, H, F] bf16: gate (silu applied) and up projections.
 *   W2         [E, F, H] bf16: down projection.
 *   y_sorted   [T*k, H] bf16 out: y_sorted[p] = FFN_e(x[sorted_src[p]/k])
 *              for p in expert e's range.
 * bf16 operands, fp32 accumulation, SwiGLU applied to the fp32 accumulators;
 * the intermediate h = silu(g)*u is stored in bf16.
 */
moe_status moe_grouped_ffn(const void* x, const int32_t* sorted_src,
                           const int32_t* offsets,
                           const void* W1, const void* W3, const void* W2,
                           int T, int H, int F, int E, int k,
                           void* y_sorted, void* ws, size_t ws_bytes, void* stream);

/*
 * Step 4 -- weighted return to token order
 * ("MegaFlux", §2.1 final top-k sum; "MegaScale-Infer", §3.2 step (4)).
 *
 *   out[t] = sum_{j<k} topk_w[t,j] * y_sorted[dest_of[t*k+j]], summed in
 *   slot order in fp32 and rounded once to bf16.
 *   y_sorted [T*k, H] bf16, dest_of [T*k] int32, topk_w [T, k] fp32,
 *   out [T, H] bf16 out.  No workspace.  A slot whose dest_of is outside
 *   [0, T*k) (-1 from moe_permute for an out-of-range expert index) adds
 *   nothing.
 */
moe_status moe_combine(const void* y_sorted, const int32_t* dest_of,
                       const float* topk_w, int T, int H, int k,
                       void* out, void* stream);

/*
 * moe_permute for callers that cannot allocate device memory.  The pages
 * have no counterpart to this entry point; it exists for how the library is
 * called, not for what the layer computes.
 *
 * Who needs it: code whose device memory is wholly owned by another
 * allocator (a serving engine or host framework that reserves the GPU's
 * memory up front and hands out no extra buffers), and code on a hot path
 * that must not take cudaMalloc's implicit device synchronisation.  Such a
 * caller cannot provide the workspace moe_permute needs, so this variant
 * takes none and performs no allocation of any kind (no cudaMalloc, no
 * cudaFree, no allocating library routine).
 *
 * Arguments, outputs and ordering are those of moe_permute.  Its scratch
 * (per-chunk histograms, the token-block plan, a status word) is a fixed
 * device array of MOE_PERMUTE_NOALLOC_SCRATCH_BYTES inside the library;
 * every GPU on which the library's device code is loaded holds that array
 * until the process exits.  Sizes whose scratch would not fit return
 * MOE_ERR_WORKSPACE and enqueue nothing; they fit while
 *   4 * (64 + C*E + (E+1) + 64 + NB) <= MOE_PERMUTE_NOALLOC_SCRATCH_BYTES
 * (each term rounded up to 64), with C = ceil(T / floor(512 / k)) chunks
 * and NB = ceil(T*k / 128) + min(T*k, E) token blocks -- for example
 * T = 8192, k = 8, E = 256 needs about 136 KB.
 *
 * The first call in each CUDA context looks up the array's device address
 * (cudaGetSymbolAddress) with that context current, and caches it under the
 * context's ID; make that first call before any stream capture begins.  A
 * device reset (or a new context on the same device) loads the library's
 * device code afresh, at an address of its own: the next call sees a new
 * context ID and looks the address up again, so it never uses a stale one.
 * Every call shares the one array and it keeps the previous call's contents
 * (the status word is cleared by each call), so calls whose work overlaps on
 * the GPU -- on different streams, or from different threads -- race and
 * corrupt each other's results; serialise them.  Out-of-range expert indices
 * get the same -1 markers as in moe_permute (so the gather and the combine
 * skip them) but, unlike moe_permute, cannot be read back as a device status.
 */
#define MOE_PERMUTE_NOALLOC_SCRATCH_BYTES (1u << 20)
moe_status moe_permute_noalloc(const int32_t* topk_idx, int T, int E, int k,
                               int32_t* counts, int32_t* offsets,
                               int32_t* sorted_src, int32_t* dest_of,
                               void* stream);

/*
 * The whole layer: steps 1-4 on `stream`, intermediates in `ws`.
 *   x [T, H] bf16, router_logits [T, E] fp32, W1/W3 [E, H, F] bf16,
 *   W2 [E, F, H] bf16, out [T, H] bf16.
 * The device status word is cleared at the start of the call.
 */
moe_status moe_forward(const void* x, const float* router_logits,
                       const void* W1, const void* W3, const void* W2,
                       int T, int H, int F, int E, int k, void* out,
                       void* ws, size_t ws_bytes, void* stream);

/*
 * moe_forward captured once into a CUDA graph, for small batches whose
 * kernels are as short as the host's launches (measured: a 256-token,
 * 8-expert layer 42.6 -> 36.1 us per step, a 128-token decode layer 0.717 ->
 * 0.707 ms; large layers run slower from a graph, e.g. a 4096-token, 16-expert
 * prefill chunk 3.82 -> 4.08 ms).  moe_forward_graph_create records one
 * moe_forward with exactly these arguments on `stream` (a non-default
 * stream, not capturing; only the calling thread's work is recorded) and
 * instantiates it; nothing runs.
 * moe_graph_launch enqueues the whole layer on `stream`: it reads x and
 * router_logits and writes out, ws as they are at that time (same pointers,
 * same sizes, same weights), so a caller refills x and router_logits in place
 * between launches.  The graph holds no reference to the buffers: they must
 * outlive every launch.  Launches on one workspace must not overlap (order
 * them on one stream).  The handle is the caller's until moe_graph_destroy,
 * which waits for nothing: destroy only after the last launch has completed.
 * Errors: MOE_ERR_INVALID_ARG (as moe_forward; also a null stream or handle
 * pointer, a stream already capturing, T == 0), MOE_ERR_WORKSPACE,
 * MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA (capture or instantiation failed);
 * *graph is null on any error.
 */
typedef struct moe_graph_s* moe_graph;
moe_status moe_forward_graph_create(const void* x, const float* router_logits,
                                    const void* W1, const void* W3, const void* W2,
                                    int T, int H, int F, int E, int k, void* out,
                                    void* ws, size_t ws_bytes, void* stream,
                                    moe_graph* graph);
moe_status moe_graph_launch(moe_graph graph, void* stream);
moe_status moe_graph_destroy(moe_graph graph);

/*
 * moe_forward with the combine's fp32 sum left unrounded: out [T, H] fp32.
 * For a layer split over GPUs along the FFN features ("MegaScale-Infer",
 * §3.4 Performance Simulation Model: expert tensor parallelism, tpe), where
 * each GPU holds W1[:, :, Fg], W3[:, :, Fg] and W2[:, Fg, :] for its slice
 * Fg of the features, routes every token identically and computes this
 * partial output; the sum of the partials over the GPUs (one all-reduce or
 * reduce-scatter, in fp32) is the layer, since SwiGLU acts feature by
 * feature and the combine is linear.  Same arguments, workspace and status
 * as moe_forward; F is the slice's width (a multiple of 128).
 */
moe_status moe_forward_f32(const void* x, const float* router_logits,
                           const void* W1, const void* W3, const void* W2,
                           int T, int H, int F, int E, int k, float* out,
                           void* ws, size_t ws_bytes, void* stream);

/*
 * The routing a moe_forward (or moe_forward_f32 / moe_forward_host /
 * moe_forward_train) call on `ws` with these sizes computed: copies the
 * layer's own topk_idx [T, k], topk_w [T, k], counts [E], offsets [E+1],
 * sorted_src [T*k] and dest_of [T*k] (layouts as in moe_route_topk and
 * moe_permute) out of the workspace, stream-ordered after that call, for
 * inspecting and testing the fused path.
 */
moe_status moe_forward_routing(const void* ws, size_t ws_bytes, int T, int H, int F, int E,
                               int k, int32_t* topk_idx, float* topk_w, int32_t* counts,
                               int32_t* offsets, int32_t* sorted_src, int32_t* dest_of,
                               void* stream);

/* out[i] = bf16(in[i]) for i < n, round to nearest even: the layer's output
 * from the reduced fp32 partials of moe_forward_f32.  in fp32 [n], out bf16
 * [n], both 16-byte aligned device pointers; no workspace. */
moe_status moe_cast_bf16(const float* in, void* out, size_t n, void* stream);

/*
 * The whole layer with the per-step activations in HOST memory: takes
 * x_host [T, H] bf16 and logits_host [T, E] fp32, runs moe_forward and
 * returns the result in out_host [T, H] bf16.  The weights are device
 * pointers (resident model parameters).  A host buffer that is page-locked
 * and mapped into the device's address space (cudaHostAlloc, cudaHostRegister,
 * or a framework's pinned allocation) is used in place: the kernels read x and
 * the logits and write the result across the host-device link, each element
 * once, with no staging copy.  Any other host buffer is copied through a staging region of
 * `ws` (moe_workspace_size covers it) with cudaMemcpyAsync.  out_host is
 * valid once `stream` has been synchronised.
 */
moe_status moe_forward_host(const void* x_host, const float* logits_host,
                            const void* W1, const void* W3, const void* W2,
                            int T, int H, int F, int E, int k, void* out_host,
                            void* ws, size_t ws_bytes, void* stream);

/*
 * The steps either side of the routed path.
 *
 * Router projection ("MegaScale-Infer" §3.2, item 2: the gating network
 * decides each token's experts; "Piper" §II-A: a learned gating function):
 *   logits[T, E] fp32 = x[T, H] bf16 @ Wg[H, E] bf16, fp32 accumulation,
 *   no bias.  E < 64: any E; E >= 64: E a multiple of 8.  H a multiple of
 *   128.  ws: at least 512 + 4 * (ceil(T/128) + 2) bytes (256-byte aligned);
 *   moe_workspace_size_gated covers it.
 */
moe_status moe_router_logits(const void* x, const void* Wg, int T, int H, int E,
                             float* logits, void* ws, size_t ws_bytes, void* stream);

/* Workspace bytes for moe_forward_gated (Fs = 0 when there is no shared
 * expert); 0 on bad sizes. */
size_t moe_workspace_size_gated(int T, int H, int F, int Fs, int E, int k);

/*
 * The layer from hidden states: router projection, then moe_forward's four
 * steps, plus an optional always-active shared expert ("Piper", Table I:
 * "R + S" = routed + shared experts per token) applied to every token and
 * added with weight one after the routed slots:
 *   out[t] = sum_j w[t,j] FFN_{e[t,j]}(x[t]) + FFN_s(x[t]).
 *   Wg [H, E] bf16; W1/W3 [E, H, F], W2 [E, F, H] bf16;
 *   Ws1/Ws3 [H, Fs], Ws2 [Fs, H] bf16, all three NULL for no shared expert;
 *   Fs a multiple of 128 when present.  Routing is decided on the fp32
 *   router logits.  ws: moe_workspace_size_gated bytes.
 */
moe_status moe_forward_gated(const void* x, const void* Wg,
                             const void* W1, const void* W3, const void* W2,
                             const void* Ws1, const void* Ws3, const void* Ws2,
                             int T, int H, int F, int Fs, int E, int k, void* out,
                             void* ws, size_t ws_bytes, void* stream);

/*
 * Training: the layer's backward ("MegaFlux" §2.1 and §3.2: the backward
 * streams token blocks through DGrad and WGrad grouped GEMMs; the final
 * top-k sum's gradient gives each routing weight's gradient).
 *
 * moe_forward_train is moe_forward that also keeps, in `ws`, what the
 * backward needs (routing, gathered x rows, the gate and up pre-activations
 * g = x W1 and u = x W3 in bf16, h and the expert outputs); ws must hold
 * moe_workspace_size_train bytes.  moe_backward then takes dout = dL/dout
 * [T, H] bf16 and the same logits and weights, and writes
 *   dx      [T, H] bf16,
 *   dlogits [T, E] fp32 (softmax Jacobian over the k selected logits;
 *           zero for unselected experts),
 *   dW1, dW3 [E, H, F] bf16, dW2 [E, F, H] bf16 (fp32 accumulation; zero
 *           for experts that received no token).
 * The two calls must use the same ws, sizes, logits and weights, with no
 * other call on that ws in between; moe_backward leaves the saved state
 * intact, so it may be repeated (e.g. for another dout).
 */
size_t moe_workspace_size_train(int T, int H, int F, int E, int k);
moe_status moe_forward_train(const void* x, const float* router_logits,
                             const void* W1, const void* W3, const void* W2,
                             int T, int H, int F, int E, int k, void* out,
                             void* ws, size_t ws_bytes, void* stream);
moe_status moe_backward(const void* dout, const float* router_logits,
                        const void* W1, const void* W3, const void* W2,
                        int T, int H, int F, int E, int k,
                        void* dx, float* dlogits, void* dW1, void* dW3, void* dW2,
                        void* ws, size_t ws_bytes, void* stream);

/*
 * moe_forward with timing marks: records events[0] on `stream` before the
 * first kernel and events[i] after stage i, for the MOE_FORWARD_STAGES
 * stages route, scan, scatter, gather, fc1, fc2, combine (in that order; the
 * gather stage is empty when the token blocks are small -- T*k <= 40 E -- and
 * FC1 gathers the rows of x it needs itself; the scan and scatter stages are
 * empty for small batches -- T*k <= 1024 and E <= 256 -- where one kernel
 * routes, counts, scans and scatters).
 * `events` points to MOE_FORWARD_STAGES + 1 cudaEvent_t created by the
 * caller.  Same arguments, work and results as moe_forward.
 */
#define MOE_FORWARD_STAGES 7
moe_status moe_forward_events(const void* x, const float* router_logits,
                              const void* W1, const void* W3, const void* W2,
                              int T, int H, int F, int E, int k, void* out,
                              void* ws, size_t ws_bytes, void* const* events,
                              void* stream);

/* Name of timing stage i of moe_forward_events (NULL if out of range). */
const char* moe_forward_stage_name(int i);

/*
 * Expert-replica planning for expert-parallel execution on G GPUs
 * ("MegaFlux: Skew-Resilient MoE Megakernels via Pipelined Expert
 * Replication", §3.1 Planner: replica placement and token-block assignment;
 * §A.1 Greedy placement and refinement; §A.2 Reduction-aware planning).
 * Runs on the device, from the per-expert row counts of a routing (e.g. the
 * `counts` of moe_permute), so no host round trip sits between routing and
 * the plan; it changes no routed assignment, only which GPU computes which
 * token blocks of an expert.
 *
 * GPU g owns experts [ceil(g E / G), ceil((g+1) E / G)), i.e. expert e is owned
 * by floor(e G / E).  Each expert's rows are cut into ceil(c_e / beta) blocks
 * (the last one partial); block counts are the load.  Starting from the
 * no-replica plan, four bounded greedy searches move blocks from GPUs above
 * tau = ceil(total blocks / G) to GPUs below it that hold the expert, or to a
 * new replica there (at most `budget` replicas per GPU), for at most s + 2
 * rounds (s = `rounds`, or the budget when `rounds` is -1); the plan with the
 * smallest maximum load (then fewest replicas) is refined -- redundant
 * replicas pruned, single blocks moved between holders of an expert -- and,
 * when lambda >= 0 (backward plans, lambda = 12 in the pages), pruned with a
 * penalty of lambda blocks per remote replica charged to the expert's owner,
 * falling back to the no-replica plan unless that lowers the penalised
 * maximum load.  Ties go to the lower GPU, then the lower expert: the plan is
 * a deterministic function of the counts.
 *
 *   counts         [E] int32 device in: routed rows per expert (>= 0).
 *   blocks_per_gpu [E, G] int32 out: blocks of expert e computed on GPU g
 *                  (row sums = ceil(c_e / beta)).
 *   row_ranges     [E, G, 2] int32 out: [lo, hi) of expert e's rows (offsets
 *                  inside its group, routed order) that GPU g computes; the
 *                  holders take consecutive ranges in ascending GPU order.
 *   gpu_load       [G] int32 out: blocks per GPU.
 *   info           [4] int32 out: the winning search (0-3: donor priority by
 *                  GPU load / by block count x one / several new replicas
 *                  per round; 4: the no-replica plan), tau, the number of
 *                  replicas, the maximum load.
 *   ws             moe_plan_workspace_size(E, G) bytes, 256-byte aligned.
 * Limits: 1 <= G <= min(E, MOE_PLAN_MAX_GPUS), E <= MOE_MAX_EXPERTS,
 * beta >= 1, 0 <= budget <= E, rounds >= -1, lambda >= -1; otherwise
 * MOE_ERR_INVALID_ARG with nothing enqueued.  One CTA of 128 threads; its
 * time grows with E * G and with the number of single-block moves.
 */
#define MOE_PLAN_MAX_GPUS 64
size_t moe_plan_workspace_size(int E, int G);
moe_status moe_plan_replicas(const int32_t* counts, int E, int G, int beta, int budget,
                             int rounds, int lambda, int32_t* blocks_per_gpu,
                             int32_t* row_ranges, int32_t* gpu_load, int32_t* info,
                             void* ws, size_t ws_bytes, void* stream);

/*
 * Synchronises `stream` and returns the device status word of `ws`
 * (MOE_OK, MOE_ERR_NONFINITE, MOE_ERR_TIMEOUT or MOE_ERR_INVALID_ARG), or
 * MOE_ERR_CUDA if the synchronisation itself failed.
 */
moe_status moe_get_device_status(const void* ws, void* stream);

/*
 * Diagnostic (no counterpart on the pages): runs the bounded wait that
 * every pipeline wait of the grouped GEMM uses on a barrier that nothing
 * arrives on.  After `limit_ns` (1 ms .. 2 s, else MOE_ERR_INVALID_ARG) the
 * wait gives up and MOE_ERR_TIMEOUT is written to the status word of `ws`,
 * which moe_get_device_status then returns; the CUDA context stays usable.
 * It lets a test check the timeout path without faulting or hanging a GPU.
 */
moe_status moe_diag_wait_timeout(void* ws, size_t ws_bytes, long long limit_ns,
                                 void* stream);

/*
 * Diagnostic (no counterpart on the pages): the same for the bounded counter
 * wait with which FC2 waits for a token block's FC1 tiles when the two
 * overlap, on a counter in `ws` that nothing increments.  Same arguments and
 * results as moe_diag_wait_timeout.
 */
moe_status moe_diag_count_wait_timeout(void* ws, size_t ws_bytes, long long limit_ns,
                                       void* stream);

/* Static, NUL-terminated description of a status code. */
const char* moe_status_string(moe_status s);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
