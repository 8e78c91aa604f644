"""FLOP and byte accounting for the MoE expert-layer forward.

Used by the benchmark to turn measured times into roofline fractions.

* FLOPs are algorithmic: only routed tokens count, 2*T*k*3*H*F for the three
  expert GEMMs (FC1 gate and up: H->F each; FC2: F->H).  The expert FFN is the
  SwiGLU expert with three d x dffn matrices ("Piper", §III-A, Table III).
* Bytes are what the layer must move at least once: the weights of every
  expert that receives a token, plus x, the output and the router logits.
* util = min(topk/E * B/F * b, 1) is the utilisation model of the expert
  GEMMs for a batch of b tokens ("MegaScale-Infer", §2 Context and
  Motivation).  Its ridge b* = F/B is the batch at which a GEMM stops being
  bandwidth-bound.
"""
from __future__ import annotations

BF16 = 2
FP32 = 4
INT32 = 4


def ffn_flops(T: int, H: int, F: int, k: int) -> int:
    """Algorithmic FLOPs of the expert FFNs: 2 * T*k * 3*H*F."""
    return 2 * T * k * 3 * H * F


def expert_weight_bytes(H: int, F: int, n_experts: int, elem: int = BF16) -> int:
    """Bytes of n_experts SwiGLU experts (three H x F matrices each)."""
    return 3 * H * F * elem * n_experts


def layer_bytes(T: int, H: int, F: int, E: int, k: int, touched_experts: int) -> int:
    """Minimum HBM bytes of one layer forward: touched weights + x (bf16) +
    out (bf16) + logits (fp32)."""
    return (expert_weight_bytes(H, F, touched_experts) + T * H * BF16 + T * H * BF16
            + T * E * FP32)


def roofline_seconds(flops: float, nbytes: float, peak_flops: float, peak_bw: float):
    """(t_roof, bound) with t_roof = max(flops/peak_flops, bytes/peak_bw)."""
    tc, tm = flops / peak_flops, nbytes / peak_bw
    return (tc, "tensor") if tc >= tm else (tm, "hbm")


def ridge_tokens(peak_flops: float, peak_bw: float) -> float:
    """Batch size b* at which util reaches 1 for a dense GEMM: F/B."""
    return peak_flops / peak_bw


def util(topk: int, n_expert: int, peak_bw: float, peak_flops: float, b: float) -> float:
    """min(topk/#expert * B/F * b, 1)."""
    return min(topk / n_expert * peak_bw / peak_flops * b, 1.0)


# Per-kernel algorithmic bytes (one launch) ---------------------------------
def route_bytes(T: int, E: int, k: int) -> int:
    """logits read + topk_idx and topk_w written."""
    return T * E * FP32 + T * k * (INT32 + FP32)


def permute_bytes(T: int, k: int, H: int) -> int:
    """topk_idx read twice (count, scatter) + sorted_src, dest_of written +
    gather_bytes."""
    P = T * k
    return 2 * P * INT32 + 2 * P * INT32 + gather_bytes(T, k, H)


def gather_bytes(T: int, k: int, H: int) -> int:
    """Each row of x read once, written to its k places in expert order (plus
    dest_of read)."""
    return T * H * BF16 + T * k * H * BF16 + T * k * INT32


def ffn_gathers_rows(T: int, k: int, E: int) -> bool:
    """Whether FC1 gathers its token rows from x itself (the library does so
    when the mean rows per expert T*k/E is at most 40, its smallest block
    size); otherwise the gather kernel writes them in expert order first."""
    return T * k <= 40 * E


def forward_launches(T: int, k: int, E: int) -> int:
    """Kernels one moe_forward launches: routing (one kernel when T*k <= 1024
    and E <= 256, else route, scan and scatter), the gather unless FC1 gathers
    its rows itself, FC1, FC2 and the combine."""
    routing = 1 if (T * k <= 1024 and E <= 256) else 3
    return routing + (0 if ffn_gathers_rows(T, k, E) else 1) + 3


def fc1_bytes(H: int, F: int, touched: int, T: int, k: int, E: int) -> int:
    """W1 and W3 of touched experts + the token rows read + h written.  The
    rows are x itself (each of its T rows read once from HBM) when FC1
    gathers them, else the T*k rows of the expert-ordered copy."""
    rows = T if ffn_gathers_rows(T, k, E) else T * k
    return 2 * H * F * BF16 * touched + rows * H * BF16 + T * k * F * BF16


def fc2_bytes(H: int, F: int, touched: int, P: int) -> int:
    """W2 of touched experts + h read + y_sorted written."""
    return H * F * BF16 * touched + P * F * BF16 + P * H * BF16


def combine_bytes(T: int, H: int, k: int) -> int:
    """y_sorted rows read + out written + dest_of and topk_w read."""
    P = T * k
    return P * H * BF16 + T * H * BF16 + P * (INT32 + FP32)
