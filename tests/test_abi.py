"""The C-ABI library: it builds, loads, exports every symbol include/moe.h
declares, and rejects bad arguments on the host before touching a GPU.
No test here launches a kernel."""
import ctypes
import os
import re

import pytest

from routing_grouped_expert_gb300 import build as B
from routing_grouped_expert_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return ctypes.CDLL(B.LIB)


def test_library_exports_every_declared_symbol(lib):
    names = header_functions()
    assert len(names) >= 9, names
    for n in names:
        assert hasattr(lib, n), f"libmoe.so does not export {n}"
    assert set(names) == set(binding.SIGNATURES), "binding and header disagree"


def test_binding_loads_and_status_strings():
    binding.load_library()
    for code in range(7):
        s = binding.moe_status_string(code)
        assert isinstance(s, str) and s
    assert binding.moe_status_string(0) == "ok"


def test_workspace_size_rules():
    ws = binding.moe_workspace_size
    assert ws(256, 512, 1024, 8, 2) > 0
    assert ws(0, 512, 1024, 8, 2) > 0                  # empty batch is valid
    assert ws(256, 500, 1024, 8, 2) == 0               # H not a multiple of 128
    assert ws(256, 512, 1000, 8, 2) == 0               # F not a multiple of 128
    assert ws(256, 512, 1024, 8, 9) == 0               # k > E
    assert ws(256, 512, 1024, 8, 0) == 0               # k < 1
    assert ws(256, 512, 1024, 2000, 2) == 0            # E > MOE_MAX_EXPERTS
    assert ws(256, 512, 1024, 64, 33) == 0             # k > MOE_MAX_TOPK
    assert ws(-1, 512, 1024, 8, 2) == 0
    # grows with every dimension
    base = ws(256, 512, 1024, 8, 2)
    assert ws(512, 512, 1024, 8, 2) > base and ws(256, 512, 2048, 8, 2) > base


def test_host_validation_rejects_before_any_launch():
    lib = binding.load_library()
    p = ctypes.c_void_p(4096)          # never dereferenced: rejected first
    bad = ctypes.c_void_p(4097)        # misaligned
    # bad sizes -> MOE_ERR_INVALID_ARG
    assert lib.moe_forward(p, p, p, p, p, 16, 500, 1024, 8, 2, p, p, 1 << 30, None) == 1
    assert lib.moe_forward(p, p, p, p, p, 16, 512, 1024, 8, 9, p, p, 1 << 30, None) == 1
    assert lib.moe_route_topk(p, 16, 8, 0, p, p, p, 1 << 20, None) == 1
    # null / misaligned tensors -> MOE_ERR_INVALID_ARG
    assert lib.moe_forward(None, p, p, p, p, 16, 512, 1024, 8, 2, p, p, 1 << 30, None) == 1
    assert lib.moe_forward(bad, p, p, p, p, 16, 512, 1024, 8, 2, p, p, 1 << 30, None) == 1
    assert lib.moe_combine(p, p, p, 16, 512, 2, None, None) == 1
    # workspace too small / null / misaligned -> MOE_ERR_WORKSPACE
    assert lib.moe_forward(p, p, p, p, p, 16, 512, 1024, 8, 2, p, p, 100, None) == 4
    assert lib.moe_forward(p, p, p, p, p, 16, 512, 1024, 8, 2, p, None, 1 << 30, None) == 4
    assert lib.moe_forward(p, p, p, p, p, 16, 512, 1024, 8, 2, p, ctypes.c_void_p(4096 + 16),
                           1 << 30, None) == 4
    # empty batch is a no-op that touches nothing
    assert lib.moe_forward(None, None, p, p, p, 0, 512, 1024, 8, 2, None, None, 0, None) == 0
    assert lib.moe_combine(None, None, None, 0, 512, 2, None, None) == 0


def test_host_validation_of_the_other_entry_points():
    """Every entry point checks sizes, pointers and the workspace on the host,
    in that order, before anything is enqueued (nothing here needs a GPU)."""
    lib = binding.load_library()
    p = ctypes.c_void_p(4096)          # never dereferenced: rejected first
    big = 1 << 40
    INVALID, WS, OK = 1, 4, 0
    # permute: sizes, then the outputs (counts/offsets even for T = 0), then ws
    assert lib.moe_permute(p, 16, 8, 9, p, p, p, p, p, big, None) == INVALID      # k > E
    assert lib.moe_permute(p, 16, 8, 2, None, p, p, p, p, big, None) == INVALID   # counts
    assert lib.moe_permute(None, 16, 8, 2, p, p, p, p, p, big, None) == INVALID   # topk_idx
    assert lib.moe_permute(p, 16, 8, 2, p, p, p, p, p, 64, None) == WS
    assert lib.moe_permute(None, 0, 8, 2, p, p, None, None, None, 0, None) == WS  # T=0 needs ws
    # grouped FFN
    assert lib.moe_grouped_ffn(p, p, p, p, p, p, 16, 500, 1024, 8, 2, p, p, big, None) == INVALID
    assert lib.moe_grouped_ffn(p, p, p, p, p, p, 16, 512, 1024, 8, 2, None, p, big, None) == INVALID
    assert lib.moe_grouped_ffn(p, p, p, p, p, p, 16, 512, 1024, 8, 2, p, p, 64, None) == WS
    assert lib.moe_grouped_ffn(None, None, None, p, p, p, 0, 512, 1024, 8, 2, None, None, 0,
                               None) == OK
    # host-buffer forward
    assert lib.moe_forward_host(p, p, p, p, p, 16, 512, 1000, 8, 2, p, p, big, None) == INVALID
    assert lib.moe_forward_host(None, p, p, p, p, 16, 512, 1024, 8, 2, p, p, big, None) == INVALID
    assert lib.moe_forward_host(p, p, p, p, p, 16, 512, 1024, 8, 2, p, p, 64, None) == WS
    assert lib.moe_forward_host(None, None, p, p, p, 0, 512, 1024, 8, 2, None, None, 0,
                                None) == OK
    # router projection: H a multiple of 128, E within range (a multiple of 8 from 64 on)
    assert lib.moe_router_logits(p, p, 16, 500, 8, p, p, big, None) == INVALID
    assert lib.moe_router_logits(p, p, 16, 512, 100, p, p, big, None) == INVALID
    assert lib.moe_router_logits(p, None, 16, 512, 8, p, p, big, None) == INVALID
    assert lib.moe_router_logits(p, p, 16, 512, 8, p, p, 16, None) == WS
    assert lib.moe_router_logits(None, None, 0, 512, 8, None, None, 0, None) == OK
    # gated layer: the shared expert's three matrices come together or not at all
    wsg = binding.moe_workspace_size_gated
    assert wsg(16, 512, 1024, 256, 8, 2) > binding.moe_workspace_size(16, 512, 1024, 8, 2)
    assert wsg(16, 512, 1024, 200, 8, 2) == 0          # Fs not a multiple of 128
    assert wsg(16, 512, 1024, 0, 100, 2) == 0          # E >= 64 not a multiple of 8
    assert lib.moe_forward_gated(p, p, p, p, p, p, None, p, 16, 512, 1024, 256, 8, 2, p, p, big,
                                 None) == INVALID
    assert lib.moe_forward_gated(p, p, p, p, p, None, None, None, 16, 512, 1024, 0, 8, 2, p, p,
                                 64, None) == WS
    # training forward and backward
    wst = binding.moe_workspace_size_train
    assert wst(16, 512, 1024, 8, 2) > binding.moe_workspace_size(16, 512, 1024, 8, 2)
    assert wst(16, 512, 1024, 8, 9) == 0
    assert lib.moe_forward_train(p, p, p, p, p, 16, 512, 1024, 8, 2, p, p, 64, None) == WS
    assert lib.moe_forward_train(p, None, p, p, p, 16, 512, 1024, 8, 2, p, p, big,
                                 None) == INVALID
    assert lib.moe_backward(p, p, p, p, p, 16, 512, 1024, 8, 2, p, None, p, p, p, p, big,
                            None) == INVALID           # dlogits
    assert lib.moe_backward(p, p, p, p, p, 16, 512, 1024, 8, 2, p, p, p, p, p, p, 64,
                            None) == WS
    assert lib.moe_backward(None, None, p, p, p, 0, 512, 1024, 8, 2, None, None, None, None,
                            None, None, 0, None) == OK
    # stage names of the per-stage forward
    n = [lib.moe_forward_stage_name(i) for i in range(-1, 9)]
    assert n[0] is None and n[1] == b"route" and b"fc1" in n and b"combine" in n
    assert n[-1] is None
