// The extern "C" boundary of libmoe: argument checks, workspace carving and
// the launch sequence of each entry point.  See include/moe.h for the
// contract of every call.
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include <new>

#include "moe_common.cuh"

namespace moe {

namespace {
// Per-device attributes, read once; callers may run on several host threads.
constexpr int kMaxDevices = 64;
std::atomic<int> g_sm_count[kMaxDevices];
std::atomic<int> g_is_sm103[kMaxDevices];   // 0 unknown, 1 yes, 2 no
}  // namespace

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 1;
  int v = g_sm_count[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    v = n > 0 ? n : 1;
    g_sm_count[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

bool device_is_sm103() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  int v = g_is_sm103[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    v = (major == 10 && minor == 3) ? 1 : 2;
    g_is_sm103[dev].store(v, std::memory_order_relaxed);
  }
  return v == 1;
}

}  // namespace moe

using namespace moe;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool ok_ptr(const void* p) { return p != nullptr && aligned16(p); }

bool ok_route_sizes(int T, int E, int k) {
  return T >= 0 && E >= 1 && E <= MOE_MAX_EXPERTS && k >= 1 && k <= E && k <= MOE_MAX_TOPK &&
         (long long)T * k < (1LL << 31) && (long long)T * E < (1LL << 40);
}

bool ok_sizes(int T, int H, int F, int E, int k) {
  return ok_route_sizes(T, E, k) && H >= kTileM && F >= kTileM && H % kTileM == 0 &&
         F % kTileM == 0 && (long long)H * F * E < (1LL << 40);
}

moe_status check_ws(void* ws, size_t ws_bytes, size_t need) {
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < need)
    return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

#define MOE_TRY(expr)                                    \
  do {                                                   \
    cudaError_t _e = (expr);                             \
    if (_e != cudaSuccess) return MOE_ERR_CUDA;          \
  } while (0)

const char* const kStageNames[MOE_FORWARD_STAGES] = {"route", "scan", "scatter", "gather",
                                                     "fc1", "fc2", "combine"};

// An always-active expert run over every token in order.
struct SharedExpert {
  const void* W1;
  const void* W3;
  const void* W2;
  int Fs;
  SingleExpertPlan plan;
  __nv_bfloat16* h;   // [T, Fs]
  __nv_bfloat16* y;   // [T, H]
};

// The launch sequence of the whole layer on device buffers.  With `ev`
// non-null, ev[0] is recorded first and ev[i] after stage i.  With
// `clear` false the caller has already zeroed the status word and the chunk
// table.  With `sh` the shared expert's output is added in the combine.
moe_status forward_device(const void* x, const float* logits, const void* W1, const void* W3,
                          const void* W2, int T, int H, int F, int E, int k, void* out,
                          void* ws, const WsLayout& L, cudaStream_t s,
                          const cudaEvent_t* ev = nullptr, bool clear = true,
                          const SharedExpert* sh = nullptr, const EpiAux* save = nullptr,
                          bool out_f32 = false) {
  const int P = T * k;
  const int C = num_chunks(T, k);
  int* status = ws_ptr<int>(ws, L.status);
  int32_t* topk_idx = ws_ptr<int32_t>(ws, L.topk_idx);
  float* topk_w = ws_ptr<float>(ws, L.topk_w);
  int32_t* counts = ws_ptr<int32_t>(ws, L.counts);
  int32_t* offsets = ws_ptr<int32_t>(ws, L.offsets);
  int32_t* sorted_src = ws_ptr<int32_t>(ws, L.sorted_src);
  int32_t* dest_of = ws_ptr<int32_t>(ws, L.dest_of);
  int32_t* chunk = ws_ptr<int32_t>(ws, L.chunk_base);
  int32_t* block_off = ws_ptr<int32_t>(ws, L.block_off);
  int32_t* num_blocks = ws_ptr<int32_t>(ws, L.num_blocks);
  int32_t* block_expert = ws_ptr<int32_t>(ws, L.block_expert);
  __nv_bfloat16* x_perm = ws_ptr<__nv_bfloat16>(ws, L.x_perm);
  __nv_bfloat16* h = ws_ptr<__nv_bfloat16>(ws, L.h);
  __nv_bfloat16* y = ws_ptr<__nv_bfloat16>(ws, L.y);

  auto mark = [&](int i) { return ev ? cudaEventRecord(ev[i], s) : cudaSuccess; };
  // The plain layer chains its short kernels (scan, scatter, gather, combine)
  // by programmatic launch: each may start while its predecessor finishes (see
  // pdl_wait).  The two persistent GEMMs keep stream order: measured, their
  // statically scheduled CTAs gain nothing from starting early.  Stage events,
  // the shared expert or the backward's saves keep plain ordering throughout.
  const bool pdl = ev == nullptr && sh == nullptr && save == nullptr;
  // status word and the chunk histogram table (adjacent) start at zero
  if (clear)
    MOE_TRY(cudaMemsetAsync(status, 0,
                            L.chunk_base - L.status + (size_t)C * E * sizeof(int32_t), s));
  MOE_TRY(mark(0));
  if (route_permute_small_ok(T, E, k)) {
    // small batches: routing, counts, scan, block plan and scatter in one
    // launch (the scan and scatter stages are then empty); its ticket
    // counter is the first int of the zeroed chunk table
    MOE_TRY(launch_route_permute_small(logits, T, E, k, ffn_block_rows(P, E, H, F), topk_idx,
                                       topk_w, counts, offsets, block_off, num_blocks,
                                       block_expert, sorted_src, dest_of, chunk, status, s));
    MOE_TRY(mark(1));
    MOE_TRY(mark(2));
  } else {
    MOE_TRY(launch_route(logits, T, E, k, topk_idx, topk_w, chunk, status, s));
    MOE_TRY(mark(1));
    MOE_TRY(launch_scan(chunk, C, E, counts, offsets, block_off, num_blocks, block_expert,
                        ffn_block_rows(P, E, H, F), s, pdl));
    MOE_TRY(mark(2));
    MOE_TRY(launch_scatter(topk_idx, T, E, k, chunk, offsets, sorted_src, dest_of, s, pdl));
  }
  MOE_TRY(mark(3));
  // With small token blocks FC1 gathers its rows from x itself; otherwise (and
  // in the forward with saves, whose rows the backward's WGrad reads) they are
  // first copied into expert order (x_perm), each row of x read once.
  const bool gathers = save == nullptr && ffn_gathers_rows(P, E);
  if (!gathers)
    MOE_TRY(launch_gather_tokens(static_cast<const __nv_bfloat16*>(x), dest_of, T, H, k, x_perm,
                                 s, pdl));
  MOE_TRY(mark(4));
  const GatherRows gr{static_cast<const __nv_bfloat16*>(x), sorted_src, k, T};
  const StreamKSpace sks{ws_ptr<float>(ws, L.sk_part), ws_ptr<int>(ws, L.sk_cnt), L.sk_slot};
  MOE_TRY(launch_grouped_ffn(x_perm, offsets, block_off, num_blocks, block_expert,
                             static_cast<const __nv_bfloat16*>(W1),
                             static_cast<const __nv_bfloat16*>(W3),
                             static_cast<const __nv_bfloat16*>(W2), P, H, F, E, h, y, status, s,
                             ev ? ev[5] : nullptr, save, &sks, gathers ? &gr : nullptr,
                             pdl ? ws_ptr<int>(ws, L.blk_done) : nullptr));
  if (sh != nullptr)
    MOE_TRY(launch_grouped_ffn(static_cast<const __nv_bfloat16*>(x), sh->plan.offsets,
                               sh->plan.block_off, sh->plan.num_blocks, sh->plan.block_expert,
                               static_cast<const __nv_bfloat16*>(sh->W1),
                               static_cast<const __nv_bfloat16*>(sh->W3),
                               static_cast<const __nv_bfloat16*>(sh->W2), T, H, sh->Fs, 1, sh->h,
                               sh->y, status, s));   // its block size differs: no split
  MOE_TRY(mark(6));
  if (out_f32)
    MOE_TRY(launch_combine_f32(y, dest_of, topk_w, T, H, k, static_cast<float*>(out), s, pdl));
  else
    MOE_TRY(launch_combine(y, dest_of, topk_w, T, H, k, static_cast<__nv_bfloat16*>(out), s,
                           sh ? sh->y : nullptr, pdl));
  MOE_TRY(mark(7));
  return MOE_OK;
}

}  // namespace

extern "C" {

size_t moe_workspace_size(int T, int H, int F, int E, int k) {
  if (!ok_sizes(T, H, F, E, k)) return 0;
  return ws_layout(T, H, F, E, k).total;
}

moe_status moe_route_topk(const float* logits, int T, int E, int k, int32_t* topk_idx,
                          float* topk_w, void* ws, size_t ws_bytes, void* stream) {
  if (!ok_route_sizes(T, E, k)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!ok_ptr(logits) || !ok_ptr(topk_idx) || !ok_ptr(topk_w)) return MOE_ERR_INVALID_ARG;
  if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < 256)
    return MOE_ERR_WORKSPACE;
  if (!device_is_sm103()) return MOE_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* status = static_cast<int*>(ws);
  MOE_TRY(cudaMemsetAsync(status, 0, 2 * sizeof(int), s));
  return cuda_status(launch_route(logits, T, E, k, topk_idx, topk_w, nullptr, status, s));
}

moe_status moe_permute(const int32_t* topk_idx, int T, int E, int k, int32_t* counts,
                       int32_t* offsets, int32_t* sorted_src, int32_t* dest_of, void* ws,
                       size_t ws_bytes, void* stream) {
  if (!ok_route_sizes(T, E, k)) return MOE_ERR_INVALID_ARG;
  if (!ok_ptr(counts) || !ok_ptr(offsets)) return MOE_ERR_INVALID_ARG;
  if (T > 0 && (!ok_ptr(topk_idx) || !ok_ptr(sorted_src) || !ok_ptr(dest_of)))
    return MOE_ERR_INVALID_ARG;
  // Only the routing part of the layout is used; H = F = 128 keeps it small.
  const WsLayout L = ws_layout(T, kTileM, kTileM, E, k);
  if (check_ws(ws, ws_bytes, L.x_perm) != MOE_OK) return MOE_ERR_WORKSPACE;
  if (!device_is_sm103()) return MOE_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* status = ws_ptr<int>(ws, L.status);
  int32_t* chunk = ws_ptr<int32_t>(ws, L.chunk_base);
  MOE_TRY(cudaMemsetAsync(status, 0, 2 * sizeof(int), s));
  if (T == 0) {
    // Empty batch: all counts and offsets are zero.
    MOE_TRY(cudaMemsetAsync(counts, 0, (size_t)E * sizeof(int32_t), s));
    MOE_TRY(cudaMemsetAsync(offsets, 0, (size_t)(E + 1) * sizeof(int32_t), s));
    return MOE_OK;
  }
  const int C = num_chunks(T, k);
  MOE_TRY(launch_count(topk_idx, T, E, k, chunk, status, s));
  MOE_TRY(launch_scan(chunk, C, E, counts, offsets, ws_ptr<int32_t>(ws, L.block_off),
                      ws_ptr<int32_t>(ws, L.num_blocks), ws_ptr<int32_t>(ws, L.block_expert),
                      kBlockRows, s));
  MOE_TRY(launch_scatter(topk_idx, T, E, k, chunk, offsets, sorted_src, dest_of, s));
  return MOE_OK;
}

moe_status moe_grouped_ffn(const void* x, const int32_t* sorted_src, const int32_t* offsets,
                           const void* W1, const void* W3, const void* W2, int T, int H, int F,
                           int E, int k, void* y_sorted, void* ws, size_t ws_bytes,
                           void* stream) {
  if (!ok_sizes(T, H, F, E, k)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!ok_ptr(x) || !ok_ptr(sorted_src) || !ok_ptr(offsets) || !ok_ptr(W1) || !ok_ptr(W3) ||
      !ok_ptr(W2) || !ok_ptr(y_sorted))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(T, H, F, E, k);
  if (check_ws(ws, ws_bytes, L.stage_x) != MOE_OK) return MOE_ERR_WORKSPACE;
  if (!device_is_sm103()) return MOE_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int P = T * k;
  int* status = ws_ptr<int>(ws, L.status);
  int32_t* block_off = ws_ptr<int32_t>(ws, L.block_off);
  int32_t* num_blocks = ws_ptr<int32_t>(ws, L.num_blocks);
  int32_t* block_expert = ws_ptr<int32_t>(ws, L.block_expert);
  const StreamKSpace sks{ws_ptr<float>(ws, L.sk_part), ws_ptr<int>(ws, L.sk_cnt), L.sk_slot};
  // the status word, the split counters and queue heads, and the per-block
  // FC1 counters (adjacent) start at zero
  MOE_TRY(cudaMemsetAsync(status, 0, L.chunk_base - L.status, s));
  MOE_TRY(launch_plan(offsets, E, P, block_off, num_blocks, block_expert,
                      ffn_block_rows(P, E, H, F), status, s));
  // with small token blocks FC1 gathers the rows of x itself (row p = token
  // sorted_src[p] / k); otherwise they are copied into expert order first
  const bool gathers = ffn_gathers_rows(P, E);
  __nv_bfloat16* x_perm = ws_ptr<__nv_bfloat16>(ws, L.x_perm);
  if (!gathers)
    MOE_TRY(launch_gather(static_cast<const __nv_bfloat16*>(x), sorted_src, P, H, k, x_perm, s));
  const GatherRows gr{static_cast<const __nv_bfloat16*>(x), sorted_src, k, T};
  MOE_TRY(launch_grouped_ffn(x_perm, offsets, block_off, num_blocks, block_expert,
                             static_cast<const __nv_bfloat16*>(W1),
                             static_cast<const __nv_bfloat16*>(W3),
                             static_cast<const __nv_bfloat16*>(W2), P, H, F, E,
                             ws_ptr<__nv_bfloat16>(ws, L.h),
                             static_cast<__nv_bfloat16*>(y_sorted), status, s, nullptr, nullptr,
                             &sks, gathers ? &gr : nullptr, ws_ptr<int>(ws, L.blk_done)));
  return MOE_OK;
}

moe_status moe_combine(const void* y_sorted, const int32_t* dest_of, const float* topk_w, int T,
                       int H, int k, void* out, void* stream) {
  if (T < 0 || H < kTileM || H % kTileM != 0 || k < 1 || k > MOE_MAX_TOPK ||
      (long long)T * k >= (1LL << 31))
    return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!ok_ptr(y_sorted) || !ok_ptr(dest_of) || !ok_ptr(topk_w) || !ok_ptr(out))
    return MOE_ERR_INVALID_ARG;
  if (!device_is_sm103()) return MOE_ERR_UNSUPPORTED;
  return cuda_status(launch_combine(static_cast<const __nv_bfloat16*>(y_sorted), dest_of, topk_w,
                                    T, H, k, static_cast<__nv_bfloat16*>(out),
                                    static_cast<cudaStream_t>(stream)));
}

moe_status moe_forward(const void* x, const float* router_logits, const void* W1,
                       const void* W3, const void* W2, int T, int H, int F, int E, int k,
                       void* out, void* ws, size_t ws_bytes, void* stream) {
  if (!ok_sizes(T, H, F, E, k)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!ok_ptr(x) || !ok_ptr(router_logits) || !ok_ptr(W1) || !ok_ptr(W3) || !ok_ptr(W2) ||
      !ok_ptr(out))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(T, H, F, E, k);
  if (check_ws(ws, ws_bytes, L.total) != MOE_OK) return MOE_ERR_WORKSPACE;
  if (!device_is_sm103()) return MOE_ERR_UNSUPPORTED;
  return forward_device(x, router_logits, W1, W3, W2, T, H, F, E, k, out, ws, L,
                        static_cast<cudaStream_t>(stream));
}

// A captured moe_forward: the graph and its executable instance.
struct moe_graph_s {
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
};

moe_status moe_forward_graph_create(const void* x, const float* router_logits, const void* W1,
                                    const void* W3, const void* W2, int T, int H, int F, int E,
                                    int k, void* out, void* ws, size_t ws_bytes, void* stream,
                                    moe_graph* graph) {
  if (graph == nullptr) return MOE_ERR_INVALID_ARG;
  *graph = nullptr;
  if (!ok_sizes(T, H, F, E, k) || T == 0) return MOE_ERR_INVALID_ARG;
  if (!ok_ptr(x) || !ok_ptr(router_logits) || !ok_ptr(W1) || !ok_ptr(W3) || !ok_ptr(W2) ||
      !ok_ptr(out))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(T, H, F, E, k);
  if (check_ws(ws, ws_bytes, L.total) != MOE_OK) return MOE_ERR_WORKSPACE;
  if (!device_is_sm103()) return MOE_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (s == nullptr) return MOE_ERR_INVALID_ARG;   // the legacy stream cannot be captured
  cudaStreamCaptureStatus cs;
  if (cudaStreamIsCapturing(s, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone)
    return MOE_ERR_INVALID_ARG;
  // Only this thread's work on `s` is recorded; nothing runs until a launch.
  MOE_TRY(cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal));
  const moe_status st = forward_device(x, router_logits, W1, W3, W2, T, H, F, E, k, out, ws, L, s);
  cudaGraph_t g = nullptr;
  const cudaError_t end = cudaStreamEndCapture(s, &g);
  if (st != MOE_OK || end != cudaSuccess) {
    if (g != nullptr) cudaGraphDestroy(g);
    (void)cudaGetLastError();
    return st != MOE_OK ? st : MOE_ERR_CUDA;
  }
  cudaGraphExec_t exec = nullptr;
  if (cudaGraphInstantiate(&exec, g, 0) != cudaSuccess) {
    cudaGraphDestroy(g);
    (void)cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  moe_graph h = new (std::nothrow) moe_graph_s;
  if (h == nullptr) {
    cudaGraphExecDestroy(exec);
    cudaGraphDestroy(g);
    return MOE_ERR_CUDA;
  }
  h->graph = g;
  h->exec = exec;
  *graph = h;
  return MOE_OK;
}

moe_status moe_graph_launch(moe_graph graph, void* stream) {
  if (graph == nullptr) return MOE_ERR_INVALID_ARG;
  return cuda_status(cudaGraphLaunch(graph->exec, static_cast<cudaStream_t>(stream)));
}

moe_status moe_graph_destroy(moe_graph graph) {
  if (graph == nullptr) return MOE_OK;
  const cudaError_t a = cudaGraphExecDestroy(graph->exec);
  const cudaError_t b = cudaGraphDestroy(graph->graph);
  delete graph;
  return cuda_status(a != cudaSuccess ? a : b);
}

moe_status moe_forward_f32(const void* x, const float* router_logits, const void* W1,
                           const void* W3, const void* W2, int T, int H, int F, int E, int k,
                           float* out, void* ws, size_t ws_bytes, void* stream) {
  if (!ok_sizes(T, H, F, E, k)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!ok_ptr(x) || !ok_ptr(router_logits) || !ok_ptr(W1) || !ok_ptr(W3) || !ok_ptr(W2) ||
      !ok_ptr(out))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(T, H, F, E, k);
  if (check_ws(ws, ws_bytes, L.total) != MOE_OK) return MOE_ERR_WORKSPACE;
  if (!device_is_sm103()) return MOE_ERR_UNSUPPORTED;
  return forward_device(x, router_logits, W1, W3, W2, T, H, F, E, k, out, ws, L,
                        static_cast<cudaStream_t>(stream), nullptr, true, nullptr, nullptr,
                        /*out_f32=*/true);
}

moe_status moe_forward_routing(const void* ws, size_t ws_bytes, int T, int H, int F, int E,
                               int k, int32_t* topk_idx, float* topk_w, int32_t* counts,
                               int32_t* offsets, int32_t* sorted_src, int32_t* dest_of,
                               void* stream) {
  if (!ok_sizes(T, H, F, E, k)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!ok_ptr(topk_idx) || !ok_ptr(topk_w) || !ok_ptr(counts) || !ok_ptr(offsets) ||
      !ok_ptr(sorted_src) || !ok_ptr(dest_of))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(T, H, F, E, k);
  if (check_ws(const_cast<void*>(ws), ws_bytes, L.total) != MOE_OK) return MOE_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t P = (size_t)T * k;
  const char* w = static_cast<const char*>(ws);
  const cudaMemcpyKind d2d = cudaMemcpyDeviceToDevice;
  MOE_TRY(cudaMemcpyAsync(topk_idx, w + L.topk_idx, P * 4, d2d, s));
  MOE_TRY(cudaMemcpyAsync(topk_w, w + L.topk_w, P * 4, d2d, s));
  MOE_TRY(cudaMemcpyAsync(counts, w + L.counts, (size_t)E * 4, d2d, s));
  MOE_TRY(cudaMemcpyAsync(offsets, w + L.offsets, (size_t)(E + 1) * 4, d2d, s));
  MOE_TRY(cudaMemcpyAsync(sorted_src, w + L.sorted_src, P * 4, d2d, s));
  MOE_TRY(cudaMemcpyAsync(dest_of, w + L.dest_of, P * 4, d2d, s));
  return MOE_OK;
}

moe_status moe_cast_bf16(const float* in, void* out, size_t n, void* stream) {
  if (n == 0) return MOE_OK;
  if (!ok_ptr(in) || !ok_ptr(out) || n >= ((size_t)1 << 40)) return MOE_ERR_INVALID_ARG;
  if (!device_is_sm103()) return MOE_ERR_UNSUPPORTED;
  return cuda_status(launch_cast_bf16(in, static_cast<__nv_bfloat16*>(out), n,
                                      static_cast<cudaStream_t>(stream)));
}

moe_status moe_forward_events(const void* x, const float* router_logits, const void* W1,
                              const void* W3, const void* W2, int T, int H, int F, int E, int k,
                              void* out, void* ws, size_t ws_bytes, void* const* events,
                              void* stream) {
  if (!ok_sizes(T, H, F, E, k)) return MOE_ERR_INVALID_ARG;
  if (events == nullptr) return MOE_ERR_INVALID_ARG;
  for (int i = 0; i <= MOE_FORWARD_STAGES; ++i)
    if (events[i] == nullptr) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!ok_ptr(x) || !ok_ptr(router_logits) || !ok_ptr(W1) || !ok_ptr(W3) || !ok_ptr(W2) ||
      !ok_ptr(out))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(T, H, F, E, k);
  if (check_ws(ws, ws_bytes, L.total) != MOE_OK) return MOE_ERR_WORKSPACE;
  if (!device_is_sm103()) return MOE_ERR_UNSUPPORTED;
  return forward_device(x, router_logits, W1, W3, W2, T, H, F, E, k, out, ws, L,
                        static_cast<cudaStream_t>(stream),
                        reinterpret_cast<const cudaEvent_t*>(events));
}

const char* moe_forward_stage_name(int i) {
  return (i >= 0 && i < MOE_FORWARD_STAGES) ? kStageNames[i] : nullptr;
}

namespace {
// The device address of a host buffer that kernels may access directly
// (page-locked and mapped, 16-byte aligned), else nullptr.
void* mapped_host(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    (void)cudaGetLastError();   // not a CUDA-known pointer: clear the error
    return nullptr;
  }
  if (a.type != cudaMemoryTypeHost || a.devicePointer == nullptr ||
      (reinterpret_cast<uintptr_t>(a.devicePointer) & 15u) != 0)
    return nullptr;
  return a.devicePointer;
}
}  // namespace

moe_status moe_forward_host(const void* x_host, const float* logits_host, const void* W1,
                            const void* W3, const void* W2, int T, int H, int F, int E, int k,
                            void* out_host, void* ws, size_t ws_bytes, void* stream) {
  if (!ok_sizes(T, H, F, E, k)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (x_host == nullptr || logits_host == nullptr || out_host == nullptr || !ok_ptr(W1) ||
      !ok_ptr(W3) || !ok_ptr(W2))
    return MOE_ERR_INVALID_ARG;
  const WsLayout L = ws_layout(T, H, F, E, k);
  if (check_ws(ws, ws_bytes, L.total) != MOE_OK) return MOE_ERR_WORKSPACE;
  if (!device_is_sm103()) return MOE_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // A page-locked, mapped host buffer is used in place: the kernels load x
  // and the logits and store the result over the host link, each element
  // once, with no staging copy.  Any other host buffer goes through a staging
  // region of ws, and so does x when FC1 gathers its rows from x itself (it
  // would read each row once per feature tile).
  void* xm = ffn_gathers_rows((long long)T * k, E) ? nullptr : mapped_host(x_host);
  void* lm = mapped_host(logits_host);
  void* om = mapped_host(out_host);   // the combine writes each result row once
  void* dx = xm ? xm : ws_ptr<void>(ws, L.stage_x);
  float* dl = lm ? static_cast<float*>(lm) : ws_ptr<float>(ws, L.stage_logits);
  void* dout = om ? om : ws_ptr<void>(ws, L.stage_out);
  if (!xm) MOE_TRY(cudaMemcpyAsync(dx, x_host, (size_t)T * H * 2, cudaMemcpyHostToDevice, s));
  if (!lm)
    MOE_TRY(cudaMemcpyAsync(dl, logits_host, (size_t)T * E * 4, cudaMemcpyHostToDevice, s));
  const moe_status st = forward_device(dx, dl, W1, W3, W2, T, H, F, E, k, dout, ws, L, s);
  if (st != MOE_OK) return st;
  if (!om)
    MOE_TRY(cudaMemcpyAsync(out_host, dout, (size_t)T * H * 2, cudaMemcpyDeviceToHost, s));
  return MOE_OK;
}

size_t moe_workspace_size_gated(int T, int H, int F, int Fs, int E, int k) {
  if (!ok_sizes(T, H, F, E, k) || Fs < 0 || (Fs > 0 && (Fs % kTileM != 0)) ||
      (E >= 64 && E % 8 != 0))
    return 0;
  return gated_layout(T, H, F, Fs, E, k).total;
}

namespace {
// Router-only workspace: status word, then the single-expert plan.
constexpr size_t kRouterPlanOffset = 256;
size_t router_ws_bytes(int T) {
  return kRouterPlanOffset + 64 + 4 * ((size_t)max_blocks(T, 1, kBlockRowsTiny) + 1);
}
SingleExpertPlan router_plan(void* ws) {
  int32_t* p = ws_ptr<int32_t>(ws, kRouterPlanOffset);
  return SingleExpertPlan{p, p + 2, p + 4, p + 16};
}
bool ok_router_sizes(int T, int H, int E) {
  return T >= 0 && H >= kTileM && H % kTileM == 0 && E >= 1 && E <= MOE_MAX_EXPERTS &&
         (E < 64 || E % 8 == 0) && (long long)T * E < (1LL << 40);
}
}  // namespace

moe_status moe_router_logits(const void* x, const void* Wg, int T, int H, int E, float* logits,
                             void* ws, size_t ws_bytes, void* stream) {
  if (!ok_router_sizes(T, H, E)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!ok_ptr(x) || !ok_ptr(Wg) || !ok_ptr(logits)) return MOE_ERR_INVALID_ARG;
  if (check_ws(ws, ws_bytes, router_ws_bytes(T)) != MOE_OK) return MOE_ERR_WORKSPACE;
  if (!device_is_sm103()) return MOE_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int* status = static_cast<int*>(ws);
  const SingleExpertPlan plan = router_plan(ws);
  MOE_TRY(cudaMemsetAsync(status, 0, 2 * sizeof(int), s));
  if (E >= 64) MOE_TRY(launch_single_expert_plan(T, ffn_block_rows(T, 1, H, E), plan, s));
  MOE_TRY(launch_router(static_cast<const __nv_bfloat16*>(x),
                        static_cast<const __nv_bfloat16*>(Wg), T, H, E, plan, logits, status, s));
  return MOE_OK;
}

moe_status moe_forward_gated(const void* x, const void* Wg, const void* W1, const void* W3,
                             const void* W2, const void* Ws1, const void* Ws3, const void* Ws2,
                             int T, int H, int F, int Fs, int E, int k, void* out, void* ws,
                             size_t ws_bytes, void* stream) {
  const bool shared = Ws1 != nullptr || Ws3 != nullptr || Ws2 != nullptr;
  if (!ok_sizes(T, H, F, E, k) || !ok_router_sizes(T, H, E)) return MOE_ERR_INVALID_ARG;
  if (shared && (Fs < kTileM || Fs % kTileM != 0)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!ok_ptr(x) || !ok_ptr(Wg) || !ok_ptr(W1) || !ok_ptr(W3) || !ok_ptr(W2) || !ok_ptr(out))
    return MOE_ERR_INVALID_ARG;
  if (shared && (!ok_ptr(Ws1) || !ok_ptr(Ws3) || !ok_ptr(Ws2))) return MOE_ERR_INVALID_ARG;
  const GatedLayout G = gated_layout(T, H, F, shared ? Fs : 0, E, k);
  if (check_ws(ws, ws_bytes, G.total) != MOE_OK) return MOE_ERR_WORKSPACE;
  if (!device_is_sm103()) return MOE_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const WsLayout& L = G.base;
  int* status = ws_ptr<int>(ws, L.status);
  float* logits = ws_ptr<float>(ws, G.logits);
  const SingleExpertPlan plan{ws_ptr<int32_t>(ws, G.s_offsets), ws_ptr<int32_t>(ws, G.s_block_off),
                              ws_ptr<int32_t>(ws, G.s_num_blocks),
                              ws_ptr<int32_t>(ws, G.s_block_expert)};
  // status word and chunk table first: the router may report into it
  MOE_TRY(cudaMemsetAsync(status, 0,
                          L.chunk_base - L.status +
                              (size_t)num_chunks(T, k) * E * sizeof(int32_t), s));
  // the single-expert plan serves the tensor-core router and the shared expert
  if (E >= 64 || shared)
    MOE_TRY(launch_single_expert_plan(T, ffn_block_rows(T, 1, H, E), plan, s));
  MOE_TRY(launch_router(static_cast<const __nv_bfloat16*>(x),
                        static_cast<const __nv_bfloat16*>(Wg), T, H, E, plan, logits, status, s));
  SharedExpert sh{Ws1, Ws3, Ws2, Fs, plan, ws_ptr<__nv_bfloat16>(ws, G.s_h),
                  ws_ptr<__nv_bfloat16>(ws, G.s_y)};
  return forward_device(x, logits, W1, W3, W2, T, H, F, E, k, out, ws, L, s, nullptr,
                        /*clear=*/false, shared ? &sh : nullptr);
}

size_t moe_workspace_size_train(int T, int H, int F, int E, int k) {
  if (!ok_sizes(T, H, F, E, k)) return 0;
  return train_layout(T, H, F, E, k).total;
}

moe_status moe_forward_train(const void* x, const float* router_logits, const void* W1,
                             const void* W3, const void* W2, int T, int H, int F, int E, int k,
                             void* out, void* ws, size_t ws_bytes, void* stream) {
  if (!ok_sizes(T, H, F, E, k)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!ok_ptr(x) || !ok_ptr(router_logits) || !ok_ptr(W1) || !ok_ptr(W3) || !ok_ptr(W2) ||
      !ok_ptr(out))
    return MOE_ERR_INVALID_ARG;
  const TrainLayout R = train_layout(T, H, F, E, k);
  if (check_ws(ws, ws_bytes, R.total) != MOE_OK) return MOE_ERR_WORKSPACE;
  if (!device_is_sm103()) return MOE_ERR_UNSUPPORTED;
  const EpiAux save{ws_ptr<__nv_bfloat16>(ws, R.g), ws_ptr<__nv_bfloat16>(ws, R.u), nullptr,
                    nullptr, F};
  return forward_device(x, router_logits, W1, W3, W2, T, H, F, E, k, out, ws, R.base,
                        static_cast<cudaStream_t>(stream), nullptr, true, nullptr, &save);
}

moe_status moe_backward(const void* dout, const float* router_logits, const void* W1,
                        const void* W3, const void* W2, int T, int H, int F, int E, int k,
                        void* dx, float* dlogits, void* dW1, void* dW3, void* dW2, void* ws,
                        size_t ws_bytes, void* stream) {
  if (!ok_sizes(T, H, F, E, k)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  if (!ok_ptr(dout) || !ok_ptr(router_logits) || !ok_ptr(W1) || !ok_ptr(W3) || !ok_ptr(W2) ||
      !ok_ptr(dx) || !ok_ptr(dlogits) || !ok_ptr(dW1) || !ok_ptr(dW3) || !ok_ptr(dW2))
    return MOE_ERR_INVALID_ARG;
  const TrainLayout R = train_layout(T, H, F, E, k);
  if (check_ws(ws, ws_bytes, R.total) != MOE_OK) return MOE_ERR_WORKSPACE;
  if (!device_is_sm103()) return MOE_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const WsLayout& L = R.base;
  const int P = T * k;
  int* status = ws_ptr<int>(ws, L.status);
  const int32_t* topk_idx = ws_ptr<int32_t>(ws, L.topk_idx);
  const float* topk_w = ws_ptr<float>(ws, L.topk_w);
  const int32_t* offsets = ws_ptr<int32_t>(ws, L.offsets);
  const int32_t* dest_of = ws_ptr<int32_t>(ws, L.dest_of);
  const __nv_bfloat16* x_perm = ws_ptr<__nv_bfloat16>(ws, L.x_perm);
  const __nv_bfloat16* h = ws_ptr<__nv_bfloat16>(ws, L.h);
  const __nv_bfloat16* y = ws_ptr<__nv_bfloat16>(ws, L.y);
  __nv_bfloat16* dx_perm = ws_ptr<__nv_bfloat16>(ws, R.dx_perm);
  __nv_bfloat16* dY = ws_ptr<__nv_bfloat16>(ws, R.dY);
  __nv_bfloat16* dg = ws_ptr<__nv_bfloat16>(ws, R.dg);
  __nv_bfloat16* du = ws_ptr<__nv_bfloat16>(ws, R.du);
  const auto* dout_b = static_cast<const __nv_bfloat16*>(dout);
  const StreamKSpace sks{ws_ptr<float>(ws, L.sk_part), ws_ptr<int>(ws, L.sk_cnt), L.sk_slot};
  // the status word and the split counters of DGrad dx (adjacent) start at zero
  MOE_TRY(cudaMemsetAsync(status, 0, L.sk_cnt - L.status + kSkCntInts * sizeof(int), s));
  MOE_TRY(launch_scale_gather(dout_b, dest_of, topk_w, T, H, k, dY, s));
  MOE_TRY(launch_dw_dlogits(dout_b, y, dest_of, topk_idx, router_logits, T, H, E, k, dlogits, s));
  MOE_TRY(launch_dgrad(dY, ws_ptr<__nv_bfloat16>(ws, R.g), ws_ptr<__nv_bfloat16>(ws, R.u),
                       static_cast<const __nv_bfloat16*>(W1),
                       static_cast<const __nv_bfloat16*>(W3),
                       static_cast<const __nv_bfloat16*>(W2), offsets,
                       ws_ptr<int32_t>(ws, L.block_off), ws_ptr<int32_t>(ws, L.num_blocks),
                       ws_ptr<int32_t>(ws, L.block_expert), P, H, F, E, dg, du, dx_perm, status,
                       s, &sks));
  MOE_TRY(launch_combine(dx_perm, dest_of, nullptr, T, H, k, static_cast<__nv_bfloat16*>(dx), s));
  MOE_TRY(launch_wgrad(x_perm, h, dY, dg, du, offsets, P, H, F, E,
                       static_cast<__nv_bfloat16*>(dW1), static_cast<__nv_bfloat16*>(dW3),
                       static_cast<__nv_bfloat16*>(dW2), status, s));
  return MOE_OK;
}

size_t moe_plan_workspace_size(int E, int G) {
  if (E < 1 || E > MOE_MAX_EXPERTS || G < 1 || G > MOE_PLAN_MAX_GPUS || G > E) return 0;
  return plan_ws_bytes(E, G);
}

moe_status moe_plan_replicas(const int32_t* counts, int E, int G, int beta, int budget,
                             int rounds, int lambda, int32_t* blocks_per_gpu,
                             int32_t* row_ranges, int32_t* gpu_load, int32_t* info, void* ws,
                             size_t ws_bytes, void* stream) {
  if (E < 1 || E > MOE_MAX_EXPERTS || G < 1 || G > MOE_PLAN_MAX_GPUS || G > E || beta < 1 ||
      budget < 0 || budget > E || rounds < -1 || rounds > 1 << 20 || lambda < -1)
    return MOE_ERR_INVALID_ARG;
  if (!ok_ptr(counts) || !ok_ptr(blocks_per_gpu) || !ok_ptr(row_ranges) || !ok_ptr(gpu_load) ||
      !ok_ptr(info))
    return MOE_ERR_INVALID_ARG;
  if (check_ws(ws, ws_bytes, plan_ws_bytes(E, G)) != MOE_OK) return MOE_ERR_WORKSPACE;
  if (!device_is_sm103()) return MOE_ERR_UNSUPPORTED;
  const int s_rounds = rounds < 0 ? budget : rounds;
  return cuda_status(launch_plan_replicas(counts, E, G, beta, budget, s_rounds + 2, lambda, ws,
                                          blocks_per_gpu, row_ranges, gpu_load, info,
                                          static_cast<cudaStream_t>(stream)));
}

moe_status moe_get_device_status(const void* ws, void* stream) {
  if (ws == nullptr) return MOE_ERR_WORKSPACE;
  int word = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&word, ws, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  return static_cast<moe_status>(word);
}

const char* moe_status_string(moe_status st) {
  switch (st) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument (size, null or misaligned pointer, expert index)";
    case MOE_ERR_NONFINITE: return "a router logit is NaN or infinite";
    case MOE_ERR_TIMEOUT: return "a bounded device wait ran out";
    case MOE_ERR_WORKSPACE: return "workspace is null, misaligned or too small";
    case MOE_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
    case MOE_ERR_UNSUPPORTED: return "the current device is not an sm_103 GPU";
  }
  return "unknown status";
}

}  // extern "C"
