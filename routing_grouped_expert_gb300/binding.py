"""ctypes binding of libmoe.so: the same entry points as include/moe.h, taking
torch tensors.  This layer only checks shapes, dtypes and devices and passes
raw pointers, sizes and the current CUDA stream; all computation runs in the
library's kernels.  A missing or unloadable library raises MoeError: there is
no CPU or PyTorch fallback.
"""
from __future__ import annotations

import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmoe.so")

MOE_OK = 0
STATUS_NAMES = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_NONFINITE",
                3: "MOE_ERR_TIMEOUT", 4: "MOE_ERR_WORKSPACE", 5: "MOE_ERR_CUDA",
                6: "MOE_ERR_UNSUPPORTED"}

# Every symbol include/moe.h declares, with its ctypes signature.
_VP, _I, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "moe_workspace_size": (_SZ, [_I, _I, _I, _I, _I]),
    "moe_route_topk": (_I, [_VP, _I, _I, _I, _VP, _VP, _VP, _SZ, _VP]),
    "moe_permute": (_I, [_VP, _I, _I, _I, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]),
    "moe_permute_noalloc": (_I, [_VP, _I, _I, _I, _VP, _VP, _VP, _VP, _VP]),
    "moe_grouped_ffn": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _VP, _VP, _SZ,
                             _VP]),
    "moe_combine": (_I, [_VP, _VP, _VP, _I, _I, _I, _VP, _VP]),
    "moe_forward": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _VP, _VP, _SZ, _VP]),
    "moe_forward_host": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _VP, _VP, _SZ,
                              _VP]),
    "moe_forward_events": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _VP, _VP, _SZ,
                                _VP, _VP]),
    "moe_forward_stage_name": (ctypes.c_char_p, [_I]),
    "moe_get_device_status": (_I, [_VP, _VP]),
    "moe_status_string": (ctypes.c_char_p, [_I]),
    "moe_diag_wait_timeout": (_I, [_VP, _SZ, ctypes.c_longlong, _VP]),
    "moe_diag_count_wait_timeout": (_I, [_VP, _SZ, ctypes.c_longlong, _VP]),
    "moe_workspace_size_train": (_SZ, [_I, _I, _I, _I, _I]),
    "moe_forward_train": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _VP, _VP, _SZ, _VP]),
    "moe_backward": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _VP, _VP, _VP, _VP, _VP,
                          _VP, _SZ, _VP]),
    "moe_router_logits": (_I, [_VP, _VP, _I, _I, _I, _VP, _VP, _SZ, _VP]),
    "moe_workspace_size_gated": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "moe_forward_gated": (_I, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _I,
                               _VP, _VP, _SZ, _VP]),
    "moe_forward_f32": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _VP, _VP, _SZ, _VP]),
    "moe_forward_graph_create": (_I, [_VP, _VP, _VP, _VP, _VP, _I, _I, _I, _I, _I, _VP, _VP, _SZ,
                                      _VP, ctypes.POINTER(ctypes.c_void_p)]),
    "moe_graph_launch": (_I, [_VP, _VP]),
    "moe_graph_destroy": (_I, [_VP]),
    "moe_cast_bf16": (_I, [_VP, _VP, _SZ, _VP]),
    "moe_forward_routing": (_I, [_VP, _SZ, _I, _I, _I, _I, _I, _VP, _VP, _VP, _VP, _VP, _VP,
                                 _VP]),
    "moe_plan_workspace_size": (_SZ, [_I, _I]),
    "moe_plan_replicas": (_I, [_VP, _I, _I, _I, _I, _I, _I, _VP, _VP, _VP, _VP, _VP, _SZ, _VP]),
}


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        name = STATUS_NAMES.get(code, str(code))
        super().__init__(f"{what}: {name}")


_lib = None


def load_library(path: str | None = None):
    """Load libmoe.so once and declare its signatures."""
    global _lib
    if _lib is None:
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise MoeError(-1, f"libmoe.so is not built ({p}); run "
                               "`python -m routing_grouped_expert_gb300.build`")
        lib = ctypes.CDLL(p)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype, fn.argtypes = res, args
        _lib = lib
    return _lib


def _check(code: int, what: str):
    if code != MOE_OK:
        raise MoeError(code, what)


def _p(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _need(t: torch.Tensor, dtype, shape, name: str, cuda: bool = True):
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")
    if cuda and not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")


class Workspace:
    """A reusable device workspace (grows on demand, 256-byte aligned)."""

    def __init__(self, device=None):
        self.device = torch.device("cuda", torch.cuda.current_device()) if device is None \
            else torch.device(device)
        self.buf = torch.empty(0, dtype=torch.uint8, device=self.device)

    def ensure(self, nbytes: int) -> torch.Tensor:
        if self.buf.numel() < nbytes:
            self.buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.device)
        return self.buf

    @property
    def ptr(self):
        return ctypes.c_void_p(self.buf.data_ptr())

    @property
    def nbytes(self) -> int:
        return self.buf.numel()


_default_ws: dict = {}


def _ws(ws: Workspace | None, nbytes: int) -> Workspace:
    if ws is None:
        dev = torch.cuda.current_device()
        ws = _default_ws.setdefault(dev, Workspace(torch.device("cuda", dev)))
    ws.ensure(nbytes)
    return ws


# ------------------------------------------------------------ entry points
def moe_workspace_size(T: int, H: int, F: int, E: int, k: int) -> int:
    return int(load_library().moe_workspace_size(T, H, F, E, k))


def moe_status_string(code: int) -> str:
    return load_library().moe_status_string(code).decode()


def moe_get_device_status(ws: Workspace) -> int:
    """Synchronises the current stream; returns the device status word."""
    return int(load_library().moe_get_device_status(ws.ptr, _stream()))


def moe_diag_wait_timeout(ws: Workspace, limit_ns: int) -> None:
    """Make a bounded device wait run out (see include/moe.h)."""
    _check(load_library().moe_diag_wait_timeout(ws.ptr, ws.nbytes, limit_ns, _stream()),
           "moe_diag_wait_timeout")


def moe_diag_count_wait_timeout(ws: Workspace, limit_ns: int) -> None:
    """Make the bounded token-block counter wait run out (see include/moe.h)."""
    _check(load_library().moe_diag_count_wait_timeout(ws.ptr, ws.nbytes, limit_ns, _stream()),
           "moe_diag_count_wait_timeout")


def moe_route_topk(logits: torch.Tensor, k: int, topk_idx=None, topk_w=None,
                   ws: Workspace | None = None):
    T, E = logits.shape
    _need(logits, torch.float32, (T, E), "logits")
    topk_idx = torch.empty(T, k, dtype=torch.int32, device=logits.device) \
        if topk_idx is None else topk_idx
    topk_w = torch.empty(T, k, dtype=torch.float32, device=logits.device) \
        if topk_w is None else topk_w
    _need(topk_idx, torch.int32, (T, k), "topk_idx")
    _need(topk_w, torch.float32, (T, k), "topk_w")
    ws = _ws(ws, 256)
    _check(load_library().moe_route_topk(_p(logits), T, E, k, _p(topk_idx), _p(topk_w), ws.ptr,
                                         ws.nbytes, _stream()), "moe_route_topk")
    return topk_idx, topk_w


def moe_permute(topk_idx: torch.Tensor, E: int, ws: Workspace | None = None, out=None):
    T, k = topk_idx.shape
    _need(topk_idx, torch.int32, (T, k), "topk_idx")
    dev = topk_idx.device
    if out is None:
        out = (torch.empty(E, dtype=torch.int32, device=dev),
               torch.empty(E + 1, dtype=torch.int32, device=dev),
               torch.empty(T * k, dtype=torch.int32, device=dev),
               torch.empty(T * k, dtype=torch.int32, device=dev))
    counts, offsets, sorted_src, dest_of = out
    need = moe_workspace_size(T, 128, 128, E, k)
    ws = _ws(ws, need)
    _check(load_library().moe_permute(_p(topk_idx), T, E, k, _p(counts), _p(offsets),
                                      _p(sorted_src), _p(dest_of), ws.ptr, ws.nbytes, _stream()),
           "moe_permute")
    return counts, offsets, sorted_src, dest_of


def moe_grouped_ffn(x, sorted_src, offsets, W1, W3, W2, k: int, y_sorted=None,
                    ws: Workspace | None = None):
    T, H = x.shape
    E, _, F = W1.shape
    _need(x, torch.bfloat16, (T, H), "x")
    _need(W1, torch.bfloat16, (E, H, F), "W1")
    _need(W3, torch.bfloat16, (E, H, F), "W3")
    _need(W2, torch.bfloat16, (E, F, H), "W2")
    _need(sorted_src, torch.int32, (T * k,), "sorted_src")
    _need(offsets, torch.int32, (E + 1,), "offsets")
    y_sorted = torch.empty(T * k, H, dtype=torch.bfloat16, device=x.device) \
        if y_sorted is None else y_sorted
    _need(y_sorted, torch.bfloat16, (T * k, H), "y_sorted")
    ws = _ws(ws, moe_workspace_size(T, H, F, E, k))
    _check(load_library().moe_grouped_ffn(_p(x), _p(sorted_src), _p(offsets), _p(W1), _p(W3),
                                          _p(W2), T, H, F, E, k, _p(y_sorted), ws.ptr, ws.nbytes,
                                          _stream()), "moe_grouped_ffn")
    return y_sorted


def moe_combine(y_sorted, dest_of, topk_w, out=None):
    T, k = topk_w.shape
    H = y_sorted.shape[1]
    _need(y_sorted, torch.bfloat16, (y_sorted.shape[0], H), "y_sorted")
    _need(dest_of, torch.int32, (T * k,), "dest_of")
    _need(topk_w, torch.float32, (T, k), "topk_w")
    out = torch.empty(T, H, dtype=torch.bfloat16, device=y_sorted.device) if out is None else out
    _need(out, torch.bfloat16, (T, H), "out")
    _check(load_library().moe_combine(_p(y_sorted), _p(dest_of), _p(topk_w), T, H, k, _p(out),
                                      _stream()), "moe_combine")
    return out


def moe_forward(x, router_logits, W1, W3, W2, k: int, out=None, ws: Workspace | None = None):
    T, H = x.shape
    E, _, F = W1.shape
    _need(x, torch.bfloat16, (T, H), "x")
    _need(router_logits, torch.float32, (T, E), "router_logits")
    _need(W1, torch.bfloat16, (E, H, F), "W1")
    _need(W3, torch.bfloat16, (E, H, F), "W3")
    _need(W2, torch.bfloat16, (E, F, H), "W2")
    out = torch.empty(T, H, dtype=torch.bfloat16, device=x.device) if out is None else out
    _need(out, torch.bfloat16, (T, H), "out")
    ws = _ws(ws, moe_workspace_size(T, H, F, E, k))
    _check(load_library().moe_forward(_p(x), _p(router_logits), _p(W1), _p(W3), _p(W2), T, H, F,
                                      E, k, _p(out), ws.ptr, ws.nbytes, _stream()),
           "moe_forward")
    return out


FORWARD_STAGES = 7


class ForwardGraph:
    """moe_forward captured once into a CUDA graph on the current stream (which
    must not be the legacy default stream): launch() runs the whole layer on
    the current stream, reading x and router_logits and writing out as they
    are then.  The tensors given here, and the workspace memory captured (a
    private workspace unless one is given), are kept alive by this object;
    refill x and router_logits in place between launches."""

    def __init__(self, x, router_logits, W1, W3, W2, k: int, out=None,
                 ws: Workspace | None = None):
        T, H = x.shape
        E, _, F = W1.shape
        _need(x, torch.bfloat16, (T, H), "x")
        _need(router_logits, torch.float32, (T, E), "router_logits")
        _need(W1, torch.bfloat16, (E, H, F), "W1")
        _need(W3, torch.bfloat16, (E, H, F), "W3")
        _need(W2, torch.bfloat16, (E, F, H), "W2")
        out = torch.empty(T, H, dtype=torch.bfloat16, device=x.device) if out is None else out
        _need(out, torch.bfloat16, (T, H), "out")
        if ws is None:
            ws = Workspace(x.device)
        ws.ensure(moe_workspace_size(T, H, F, E, k))
        # the captured pointers: kept alive even if `ws` later grows elsewhere
        self.tensors = (x, router_logits, W1, W3, W2, out, ws.buf)
        self.ws, self.out = ws, out
        self._h = ctypes.c_void_p()
        _check(load_library().moe_forward_graph_create(
            _p(x), _p(router_logits), _p(W1), _p(W3), _p(W2), T, H, F, E, k, _p(out), ws.ptr,
            ws.nbytes, _stream(), ctypes.byref(self._h)), "moe_forward_graph_create")

    def launch(self):
        _check(load_library().moe_graph_launch(self._h, _stream()), "moe_graph_launch")
        return self.out

    def close(self):
        """Free the graph (after its last launch has completed)."""
        if self._h:
            _check(load_library().moe_graph_destroy(self._h), "moe_graph_destroy")
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def moe_forward_f32(x, router_logits, W1, W3, W2, k: int, out=None,
                    ws: Workspace | None = None):
    """The layer with its fp32 combine sum unrounded ([T, H] fp32): a partial
    output of a layer split over GPUs along the FFN features."""
    T, H = x.shape
    E, _, F = W1.shape
    _need(x, torch.bfloat16, (T, H), "x")
    _need(router_logits, torch.float32, (T, E), "router_logits")
    _need(W1, torch.bfloat16, (E, H, F), "W1")
    _need(W3, torch.bfloat16, (E, H, F), "W3")
    _need(W2, torch.bfloat16, (E, F, H), "W2")
    out = torch.empty(T, H, dtype=torch.float32, device=x.device) if out is None else out
    _need(out, torch.float32, (T, H), "out")
    ws = _ws(ws, moe_workspace_size(T, H, F, E, k))
    _check(load_library().moe_forward_f32(_p(x), _p(router_logits), _p(W1), _p(W3), _p(W2), T,
                                          H, F, E, k, _p(out), ws.ptr, ws.nbytes, _stream()),
           "moe_forward_f32")
    return out


def moe_forward_routing(ws: Workspace, T: int, H: int, F: int, E: int, k: int):
    """The routing the last layer call on `ws` computed: (topk_idx, topk_w,
    counts, offsets, sorted_src, dest_of) copied out of the workspace."""
    dev = ws.device
    outs = (torch.empty(T, k, dtype=torch.int32, device=dev),
            torch.empty(T, k, dtype=torch.float32, device=dev),
            torch.empty(E, dtype=torch.int32, device=dev),
            torch.empty(E + 1, dtype=torch.int32, device=dev),
            torch.empty(T * k, dtype=torch.int32, device=dev),
            torch.empty(T * k, dtype=torch.int32, device=dev))
    _check(load_library().moe_forward_routing(ws.ptr, ws.nbytes, T, H, F, E, k,
                                              *[_p(t) for t in outs], _stream()),
           "moe_forward_routing")
    return outs


def moe_cast_bf16(x: torch.Tensor, out=None):
    """bf16 copy of an fp32 tensor (round to nearest even), on the GPU."""
    _need(x, torch.float32, tuple(x.shape), "x")
    out = torch.empty(x.shape, dtype=torch.bfloat16, device=x.device) if out is None else out
    _need(out, torch.bfloat16, tuple(x.shape), "out")
    _check(load_library().moe_cast_bf16(_p(x), _p(out), x.numel(), _stream()), "moe_cast_bf16")
    return out


def moe_forward_stage_name(i: int) -> str:
    r = load_library().moe_forward_stage_name(i)
    return None if r is None else r.decode()


def moe_forward_events(x, router_logits, W1, W3, W2, k: int, events, out=None,
                       ws: Workspace | None = None):
    """moe_forward that records events[0] before the first kernel and
    events[i] after stage i (torch.cuda.Event objects with timing)."""
    T, H = x.shape
    E, _, F = W1.shape
    if len(events) != FORWARD_STAGES + 1:
        raise ValueError(f"need {FORWARD_STAGES + 1} events")
    out = torch.empty(T, H, dtype=torch.bfloat16, device=x.device) if out is None else out
    ws = _ws(ws, moe_workspace_size(T, H, F, E, k))
    for e in events:            # torch creates the CUDA event on its first record
        if e.cuda_event == 0:
            e.record()
    arr = (ctypes.c_void_p * (FORWARD_STAGES + 1))(*[e.cuda_event for e in events])
    _check(load_library().moe_forward_events(_p(x), _p(router_logits), _p(W1), _p(W3), _p(W2),
                                             T, H, F, E, k, _p(out), ws.ptr, ws.nbytes, arr,
                                             _stream()), "moe_forward_events")
    return out


def moe_forward_host(x_host, logits_host, W1, W3, W2, k: int, out_host=None,
                     ws: Workspace | None = None):
    """Host activations in (pinned CPU tensors), host result out; weights on
    the device.  The result is valid after the current stream synchronises."""
    T, H = x_host.shape
    E, _, F = W1.shape
    _need(x_host, torch.bfloat16, (T, H), "x_host", cuda=False)
    _need(logits_host, torch.float32, (T, E), "logits_host", cuda=False)
    _need(W1, torch.bfloat16, (E, H, F), "W1")
    _need(W3, torch.bfloat16, (E, H, F), "W3")
    _need(W2, torch.bfloat16, (E, F, H), "W2")
    out_host = torch.empty(T, H, dtype=torch.bfloat16, pin_memory=True) \
        if out_host is None else out_host
    _need(out_host, torch.bfloat16, (T, H), "out_host", cuda=False)
    ws = _ws(ws, moe_workspace_size(T, H, F, E, k))
    _check(load_library().moe_forward_host(_p(x_host), _p(logits_host), _p(W1), _p(W3), _p(W2),
                                           T, H, F, E, k, _p(out_host), ws.ptr, ws.nbytes,
                                           _stream()), "moe_forward_host")
    return out_host


# ------------------------------------------ either side of the routed path
def moe_workspace_size_gated(T: int, H: int, F: int, Fs: int, E: int, k: int) -> int:
    return int(load_library().moe_workspace_size_gated(T, H, F, Fs, E, k))


def moe_router_logits(x, Wg, logits=None, ws: Workspace | None = None):
    """logits [T, E] fp32 = x [T, H] @ Wg [H, E] (bf16 in)."""
    T, H = x.shape
    E = Wg.shape[1]
    _need(x, torch.bfloat16, (T, H), "x")
    _need(Wg, torch.bfloat16, (H, E), "Wg")
    logits = torch.empty(T, E, dtype=torch.float32, device=x.device) if logits is None \
        else logits
    _need(logits, torch.float32, (T, E), "logits")
    ws = _ws(ws, 1024 + 4 * (T // 128 + 4))
    _check(load_library().moe_router_logits(_p(x), _p(Wg), T, H, E, _p(logits), ws.ptr,
                                            ws.nbytes, _stream()), "moe_router_logits")
    return logits


def moe_forward_gated(x, Wg, W1, W3, W2, k: int, shared=None, out=None,
                      ws: Workspace | None = None):
    """Router projection + routed experts (+ `shared` = (Ws1, Ws3, Ws2))."""
    T, H = x.shape
    E, _, F = W1.shape
    _need(x, torch.bfloat16, (T, H), "x")
    _need(Wg, torch.bfloat16, (H, E), "Wg")
    _need(W1, torch.bfloat16, (E, H, F), "W1")
    _need(W3, torch.bfloat16, (E, H, F), "W3")
    _need(W2, torch.bfloat16, (E, F, H), "W2")
    Fs = 0
    if shared is not None:
        Ws1, Ws3, Ws2 = shared
        Fs = Ws1.shape[1]
        _need(Ws1, torch.bfloat16, (H, Fs), "Ws1")
        _need(Ws3, torch.bfloat16, (H, Fs), "Ws3")
        _need(Ws2, torch.bfloat16, (Fs, H), "Ws2")
    out = torch.empty(T, H, dtype=torch.bfloat16, device=x.device) if out is None else out
    _need(out, torch.bfloat16, (T, H), "out")
    ws = _ws(ws, moe_workspace_size_gated(T, H, F, Fs, E, k))
    sp = (None, None, None) if shared is None else tuple(_p(t) for t in shared)
    _check(load_library().moe_forward_gated(_p(x), _p(Wg), _p(W1), _p(W3), _p(W2), *sp, T, H,
                                            F, Fs, E, k, _p(out), ws.ptr, ws.nbytes, _stream()),
           "moe_forward_gated")
    return out


# ------------------------------------------------------------- training
def moe_workspace_size_train(T: int, H: int, F: int, E: int, k: int) -> int:
    return int(load_library().moe_workspace_size_train(T, H, F, E, k))


def moe_forward_train(x, router_logits, W1, W3, W2, k: int, ws: Workspace, out=None):
    """moe_forward that keeps in `ws` what moe_backward needs."""
    T, H = x.shape
    E, _, F = W1.shape
    _need(x, torch.bfloat16, (T, H), "x")
    _need(router_logits, torch.float32, (T, E), "router_logits")
    _need(W1, torch.bfloat16, (E, H, F), "W1")
    _need(W3, torch.bfloat16, (E, H, F), "W3")
    _need(W2, torch.bfloat16, (E, F, H), "W2")
    out = torch.empty(T, H, dtype=torch.bfloat16, device=x.device) if out is None else out
    ws.ensure(moe_workspace_size_train(T, H, F, E, k))
    _check(load_library().moe_forward_train(_p(x), _p(router_logits), _p(W1), _p(W3), _p(W2),
                                            T, H, F, E, k, _p(out), ws.ptr, ws.nbytes,
                                            _stream()), "moe_forward_train")
    return out


def moe_backward(dout, router_logits, W1, W3, W2, k: int, ws: Workspace):
    """Gradients after moe_forward_train on the same ws: (dx, dlogits, dW1,
    dW3, dW2)."""
    T, H = dout.shape
    E, _, F = W1.shape
    _need(dout, torch.bfloat16, (T, H), "dout")
    _need(router_logits, torch.float32, (T, E), "router_logits")
    dev = dout.device
    dx = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    dl = torch.empty(T, E, dtype=torch.float32, device=dev)
    dW1 = torch.empty(E, H, F, dtype=torch.bfloat16, device=dev)
    dW3 = torch.empty(E, H, F, dtype=torch.bfloat16, device=dev)
    dW2 = torch.empty(E, F, H, dtype=torch.bfloat16, device=dev)
    _check(load_library().moe_backward(_p(dout), _p(router_logits), _p(W1), _p(W3), _p(W2), T, H,
                                       F, E, k, _p(dx), _p(dl), _p(dW1), _p(dW3), _p(dW2),
                                       ws.ptr, ws.nbytes, _stream()), "moe_backward")
    return dx, dl, dW1, dW3, dW2


def moe_plan_workspace_size(E: int, G: int) -> int:
    return load_library().moe_plan_workspace_size(E, G)


def moe_plan_replicas(counts: torch.Tensor, G: int, beta: int, budget: int, rounds: int = -1,
                      lam: int = -1, ws: Workspace | None = None):
    """Replica plan of expert row counts [E] (int32, on the GPU) for G GPUs.
    Returns (blocks_per_gpu [E, G], row_ranges [E, G, 2], gpu_load [G], info [4]),
    int32 tensors on the counts' device; lam = -1: no reduction penalty."""
    E = counts.shape[0]
    _need(counts, torch.int32, (E,), "counts")
    dev = counts.device
    n = torch.empty(E, G, dtype=torch.int32, device=dev)
    rows = torch.empty(E, G, 2, dtype=torch.int32, device=dev)
    load = torch.empty(G, dtype=torch.int32, device=dev)
    info = torch.empty(4, dtype=torch.int32, device=dev)
    need = moe_plan_workspace_size(E, G)
    ws = _ws(ws, max(need, 256))
    _check(load_library().moe_plan_replicas(_p(counts), E, G, beta, budget, rounds, lam, _p(n),
                                            _p(rows), _p(load), _p(info), ws.ptr, ws.nbytes,
                                            _stream()), "moe_plan_replicas")
    return n, rows, load, info
