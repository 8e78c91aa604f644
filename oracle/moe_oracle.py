"""CPU oracle for the MoE expert-layer forward -- TEST INFRASTRUCTURE.

Only the test suite, the smoke check in the repository's graft entry module
and the CPU-baseline leg of the benchmark may import this module.  The
library's product path never does, and this module imports nothing from the
library package: the two share no code.

What it computes (the plain definition, in fp64):

    out[t] = sum_{j<k} w[t, j] * FFN_{e[t, j]}(x[t])
    FFN_e(x) = (silu(x @ W1[e]) * (x @ W3[e])) @ W2[e],  silu(z) = z / (1 + e^-z)

with e[t, :] the top-k experts of token t and w[t, :] the softmax of their
logits.  It is written twice:

  * forward_perm   -- the method's own order of steps: top-k gating,
    per-expert counts, weight normalisation, scatter into per-expert groups,
    per-expert FFN, weighted return to token order
    ("MegaScale-Infer", §3.4 Supporting Implementation Details: Fused Kernels,
    steps (1)-(4); §3.2 Big-Picture Architecture, steps (2)-(5));
  * forward_direct -- a per-token loop over the k slots with no permutation.

Sources for each step:
  top-k selection, counts, normalisation, scatter:
      "MegaScale-Infer", §3.4 Fused Kernels (steps 1-4).
  order of routed assignments inside an expert (by token, then top-k
  position) and retention of token id / top-k position / weight:
      "MegaFlux: Skew-Resilient MoE Megakernels via Pipelined Expert
      Replication", §A.2.
  SwiGLU expert with three matrices (gate, up: d x dffn; down: dffn x d):
      "Piper: Efficient Large-Scale MoE Training via Resource Modeling and
      Pipelined Hybrid Parallelism", §III-A and Table III.
  two expert GEMMs, "FFN Input" (b_e, h) x (h, h') and "FFN Output":
      "MegaScale-Infer", §3.4 Performance Simulation Model (Te).
  weighted top-k sum back to token order:
      "MegaFlux", §2.1; "MegaScale-Infer", §3.2 step (4)-(5).

Backward ("backward"): the gradients of the layer output with respect to x,
the router logits and the three expert matrices, given dout = dL/dout --
the DGrad/WGrad streams of the backward MoE pass ("MegaFlux", §2.1 and
§3.2 backward).  Written from the chain rule of the forward above:
  dY_p   = w[t,j] dout[t]                      (combine, p = dest_of[t*k+j])
  dw_tj  = <dout[t], y_p>                       (routing weight)
  dW2[e] = h_e^T dY_e,  dh = dY W2[e]^T        (FC2 WGrad / DGrad)
  dg = dh * u * s * (1 + g (1 - s)),  du = dh * g * s,  s = sigmoid(g)
  dW1[e] = x_e^T dg,  dW3[e] = x_e^T du,  dx_p = dg W1[e]^T + du W3[e]^T
  dx[t]  = sum_j dx_p                           (scatter back to tokens)
  dlogits[t, e_j] = w_j (dw_j - sum_i w_i dw_i), zero for unselected experts
                                                (softmax over the k selected).
The forward uses the fp32-rounded weights w; the logit gradient applies the
exact (fp64) softmax Jacobian, treating that rounding as the identity.

Either side of the routed path ("forward_gated"):
  router projection: the gating network that decides each token's experts
      ("MegaScale-Infer", §3.2 Big-Picture Architecture, item 2; "Piper",
      §II-A: a learned gating function), read as logits = x @ W_g;
  shared expert: an always-active expert next to the routed ones ("Piper",
      Table I, e.g. "8R + 1S" = 8 routed + 1 shared per token), read as a
      SwiGLU expert applied to every token and added with weight one.

Readings where the pages are silent (each is listed in the design notes):
  * experts are ranked on the raw fp32 logits; a larger value wins, equal
    values (including -0.0 == +0.0) go to the lower expert index;
  * the weights are the softmax over the k selected logits (softmax over all
    E and renormalising over the k is the same in exact arithmetic),
    computed in fp64 and rounded once to fp32;
  * W1 is the gate (silu applied), W3 the up projection, W2 the down
    projection;
  * non-finite logits are rejected;
  * no capacity limit: every routed assignment is computed (dropless);
  * the router has no bias; its logits are the layer's fp32 router output,
    so forward_gated rounds the fp64 product to fp32 before ranking.

Floating point: bf16 and fp32 inputs convert exactly to fp64; all sums are
fp64; no intermediate is rounded.  Matrix products use a library matmul
(torch, fp64, CPU) as a step; everything else is written out here.
"""
from __future__ import annotations

import numpy as np
import torch


class NonFiniteLogits(ValueError):
    """A router logit is NaN or infinite."""


def _f64(a) -> np.ndarray:
    """Exact conversion of a bf16/fp32/fp64 array (numpy or CPU torch) to fp64."""
    if isinstance(a, torch.Tensor):
        return a.detach().to("cpu", torch.float64).numpy()
    return np.asarray(a, dtype=np.float64)


def _mm(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """fp64 matrix product (library routine)."""
    return (torch.from_numpy(np.ascontiguousarray(a)) @
            torch.from_numpy(np.ascontiguousarray(b))).numpy()


# --------------------------------------------------------------------------
# Step 1 -- top-k gating and weight normalisation
# --------------------------------------------------------------------------
def route_topk(logits, k: int):
    """Top-k experts per token and their normalised weights.

    Slot j holds the j-th pick of a repeated arg-max over the experts not yet
    picked, so slots are in descending logit order; ties go to the lower
    expert index (numpy's argmax returns the first maximal index, and
    -0.0 == +0.0 compare equal).  Weights: softmax over the k selected logits
    in fp64, stored as fp32.

    Returns (topk_idx int32 [T, k], topk_w float32 [T, k]).
    """
    l = np.asarray(logits, dtype=np.float32)
    if l.ndim != 2:
        raise ValueError("logits must be [T, E]")
    T, E = l.shape
    if not 1 <= k <= E:
        raise ValueError(f"need 1 <= k <= E, got k={k}, E={E}")
    if not np.all(np.isfinite(l)):
        raise NonFiniteLogits("router logits contain NaN or inf")
    work = l.astype(np.float64)            # exact
    taken = np.zeros((T, E), dtype=bool)
    idx = np.empty((T, k), dtype=np.int32)
    rows = np.arange(T)
    for j in range(k):
        masked = np.where(taken, -np.inf, work)
        e = np.argmax(masked, axis=1) if T else np.zeros(0, dtype=np.int64)
        idx[:, j] = e
        taken[rows, e] = True
    sel = np.take_along_axis(work, idx.astype(np.int64), axis=1)   # [T, k]
    m = sel[:, :1] if T else sel
    ex = np.exp(sel - m)
    w = ex / ex.sum(axis=1, keepdims=True) if T else ex
    return idx, w.astype(np.float32)


# --------------------------------------------------------------------------
# Step 2 -- per-expert counts and the stable scatter into expert groups
# --------------------------------------------------------------------------
def permute(topk_idx, E: int):
    """Group routed assignments by expert.

    Assignment a = t*k + j (token t, top-k slot j).  counts[e] = number of
    assignments to e; offsets = exclusive prefix sum (length E+1).  Walking a
    in ascending order, each assignment takes the next free position of its
    expert, so inside an expert the order is by token, then top-k position.

    Returns (counts int32 [E], offsets int32 [E+1], sorted_src int32 [T*k],
    dest_of int32 [T*k]) with sorted_src[dest_of[a]] == a.
    """
    flat = np.asarray(topk_idx).reshape(-1).astype(np.int64)
    if flat.size and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("expert index out of range")
    counts = np.zeros(E, dtype=np.int64)
    for e in flat.tolist():
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    cursor = offsets[:-1].tolist()
    P = flat.size
    sorted_src = np.empty(P, dtype=np.int32)
    dest_of = np.empty(P, dtype=np.int32)
    for a, e in enumerate(flat.tolist()):
        p = cursor[e]
        cursor[e] = p + 1
        sorted_src[p] = a
        dest_of[a] = p
    return (counts.astype(np.int32), offsets.astype(np.int32), sorted_src, dest_of)


# --------------------------------------------------------------------------
# Step 3 -- the expert FFN (SwiGLU, three matrices)
# --------------------------------------------------------------------------
def silu(z: np.ndarray) -> np.ndarray:
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def expert_ffn(xrows, W1e, W3e, W2e) -> np.ndarray:
    """(silu(x W1e) * (x W3e)) W2e for the rows of x; fp64, nothing rounded."""
    x64 = _f64(xrows)
    g = _mm(x64, _f64(W1e))
    u = _mm(x64, _f64(W3e))
    return _mm(silu(g) * u, _f64(W2e))


def grouped_ffn(x, sorted_src, offsets, W1, W3, W2, k: int) -> np.ndarray:
    """y_sorted[p] = FFN_e(x[sorted_src[p] // k]) for p in expert e's range."""
    x64 = _f64(x)
    sorted_src = np.asarray(sorted_src)
    offsets = np.asarray(offsets)
    E = len(offsets) - 1
    P = int(offsets[-1])
    H = x64.shape[1]
    y = np.zeros((P, H), dtype=np.float64)
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if lo == hi:
            continue
        tok = sorted_src[lo:hi] // k
        y[lo:hi] = expert_ffn(x64[tok], W1[e], W3[e], W2[e])
    return y


# --------------------------------------------------------------------------
# Step 4 -- weighted return to token order
# --------------------------------------------------------------------------
def combine(y_sorted, dest_of, topk_w) -> np.ndarray:
    """out[t] = sum_j w[t, j] * y_sorted[dest_of[t*k + j]], slots in order."""
    w = np.asarray(topk_w, dtype=np.float64)
    T, k = w.shape
    y = np.asarray(y_sorted, dtype=np.float64)
    dest = np.asarray(dest_of).reshape(T, k)
    out = np.zeros((T, y.shape[1]), dtype=np.float64)
    for j in range(k):
        out += w[:, j:j + 1] * y[dest[:, j]]
    return out


# --------------------------------------------------------------------------
# The whole layer, two ways
# --------------------------------------------------------------------------
def forward_perm(x, logits, W1, W3, W2, k: int):
    """Route -> counts/scatter -> per-expert FFN -> weighted combine.

    Returns a dict with every intermediate (fp64 `out` [T, H])."""
    E = np.asarray(logits).shape[1]
    idx, w = route_topk(logits, k)
    counts, offsets, sorted_src, dest_of = permute(idx, E)
    y = grouped_ffn(x, sorted_src, offsets, W1, W3, W2, k)
    out = combine(y, dest_of, w)
    return dict(topk_idx=idx, topk_w=w, counts=counts, offsets=offsets,
                sorted_src=sorted_src, dest_of=dest_of, y_sorted=y, out=out)


def forward_direct(x, logits, W1, W3, W2, k: int, tokens=None) -> np.ndarray:
    """Per-token definition, no permutation: for each token t (all, or the
    listed ones) and slot j, y_tj = FFN_{e[t,j]}(x[t]); out[t] = sum_j w_tj y_tj.

    The FFN of one expert is evaluated once for all listed (t, j) pairs that
    chose it, which changes nothing in the arithmetic of any pair.  Returns
    fp64 [len(tokens), H]."""
    idx, w = route_topk(logits, k)
    tokens = np.arange(idx.shape[0]) if tokens is None else np.asarray(tokens)
    x64 = _f64(x)
    n, H = len(tokens), x64.shape[1]
    Y = np.zeros((n, k, H), dtype=np.float64)
    sel = idx[tokens]                                        # [n, k]
    for e in np.unique(sel).tolist():
        ii, jj = np.nonzero(sel == e)
        Y[ii, jj] = expert_ffn(x64[tokens[ii]], W1[e], W3[e], W2[e])
    out = np.zeros((n, H), dtype=np.float64)
    wt = w[tokens].astype(np.float64)
    for j in range(k):
        out += wt[:, j:j + 1] * Y[:, j]
    return out


# --------------------------------------------------------------------------
# Either side of the routed path: router projection and a shared expert
# --------------------------------------------------------------------------
def router_logits(x, Wg) -> np.ndarray:
    """logits[t, e] = sum_h x[t, h] * Wg[h, e], fp64 (Wg is [H, E])."""
    return _mm(_f64(x), _f64(Wg))


def forward_gated(x, Wg, W1, W3, W2, k: int, shared=None, logits=None):
    """The layer from hidden states.

    logits = x @ Wg rounded to fp32 (or the fp32 `logits` given, so a test can
    rank on another implementation's router output), the routed experts as in
    forward_perm, and -- when `shared` = (Ws1, Ws3, Ws2) -- the shared expert
    FFN_s(x[t]) added to every token's output with weight one."""
    l = (np.asarray(router_logits(x, Wg), dtype=np.float32) if logits is None
         else np.asarray(logits, dtype=np.float32))
    r = forward_perm(x, l, W1, W3, W2, k)
    r["logits"] = l
    if shared is not None:
        r["shared"] = expert_ffn(x, *shared)
        r["out"] = r["out"] + r["shared"]
    return r


# --------------------------------------------------------------------------
# Backward of the layer
# --------------------------------------------------------------------------
def backward(x, logits, W1, W3, W2, k: int, dout, magnitudes: bool = False):
    """Gradients of out = forward_perm(...)["out"] for the upstream gradient
    dout [T, H].  Returns dict with dx [T, H], dlogits [T, E], dW1, dW3
    [E, H, F], dW2 [E, F, H] and dw [T, k] (gradient of the routing
    weights), all fp64.

    With magnitudes=True it also returns, under "mag_<name>", the first-order
    size, in units of eps, of the change that rounding the stored operands
    (dY, g, u, h, y, dg, du and the per-assignment dx rows) by a relative eps
    makes to each gradient: sums over absolute values that follow each
    rounding through the chain rule, e.g. for dW1 the rounding of dY through
    dh, of u, of g through the SwiGLU derivative (whose factor crosses zero
    near g = -1.28), and of dg; for dW2 the rounding of h and of dY; for dx
    also the rounding of each assignment's row before the sum over slots; for
    the routing-weight gradient the rounding of h through y and of y.  For
    dW1, dW3, dW2 and dlogits this is the largest first-order change over all
    signs of the roundings; for dx it is an upper bound of it (the rounding of
    dY is followed through dh with the triangle inequality taken inside the
    sum over features)."""
    l = np.asarray(logits, dtype=np.float32)
    T, E = l.shape
    idx, w = route_topk(l, k)
    counts, offsets, sorted_src, dest_of = permute(idx, E)
    x64, d64 = _f64(x), _f64(dout)
    H = x64.shape[1]
    w64 = w.astype(np.float64)
    dx = np.zeros((T, H))
    dw = np.zeros((T, k))
    grads = {"dW1": [], "dW3": [], "dW2": []}
    mag = {"dW1": [], "dW3": [], "dW2": []}
    mdx = np.zeros((T, H))
    mdw = np.zeros((T, k))
    for e in range(E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if lo == hi:
            for name, like in (("dW1", W1[e]), ("dW3", W3[e]), ("dW2", W2[e])):
                grads[name].append(np.zeros(tuple(like.shape)))
                mag[name].append(np.zeros(tuple(like.shape)))
            continue
        W1e, W3e, W2e = _f64(W1[e]), _f64(W3[e]), _f64(W2[e])
        a = sorted_src[lo:hi]
        t, j = a // k, a % k
        X = x64[t]
        g, u = _mm(X, W1e), _mm(X, W3e)
        s = 1.0 / (1.0 + np.exp(-g))
        h = g * s * u
        Y = _mm(h, W2e)
        dY = w64[t, j][:, None] * d64[t]
        dw[t, j] = np.sum(d64[t] * Y, axis=1)
        grads["dW2"].append(_mm(h.T, dY))
        dh = _mm(dY, W2e.T)
        dg = dh * u * s * (1.0 + g * (1.0 - s))
        du = dh * g * s
        grads["dW1"].append(_mm(X.T, dg))
        grads["dW3"].append(_mm(X.T, du))
        np.add.at(dx, t, _mm(dg, W1e.T) + _mm(du, W3e.T))
        if magnitudes:
            # first-order sizes of what rounding each stored operand by a
            # relative eps does to each gradient, in units of eps
            aX, ah, adY = np.abs(X), np.abs(h), np.abs(dY)
            f = s * (1.0 + g * (1.0 - s))                       # d silu / d g
            fp = s * (1.0 - s) * (2.0 + g * (1.0 - 2.0 * s))    # its derivative
            gsp = s + g * s * (1.0 - s)                         # d (g s) / d g
            m_dh = _mm(adY, np.abs(W2e).T)                      # dY rounding -> dh
            m_dg = (m_dh * np.abs(u * f) + np.abs(dh * u) * (np.abs(f) + np.abs(g * fp))
                    + np.abs(dg))
            m_du = m_dh * np.abs(g * s) + np.abs(dh * g * gsp) + np.abs(du)
            mag["dW1"].append(_mm(aX.T, m_dg))
            mag["dW3"].append(_mm(aX.T, m_du))
            mag["dW2"].append(2.0 * _mm(ah.T, adY))             # h and dY rounded
            dxp = _mm(dg, W1e.T) + _mm(du, W3e.T)               # this expert's dx rows
            np.add.at(mdx, t, _mm(m_dg, np.abs(W1e).T) + _mm(m_du, np.abs(W3e).T)
                      + np.abs(dxp))
            # dw = <dout, y>: h rounded (through y = h W2) and y rounded
            mdw[t, j] = (np.sum(ah * np.abs(_mm(d64[t], W2e.T)), axis=1)
                         + np.sum(np.abs(d64[t] * Y), axis=1))
    # exact softmax of the selected logits for the Jacobian
    sel = np.take_along_axis(l.astype(np.float64), idx.astype(np.int64), axis=1)
    ex = np.exp(sel - sel[:, :1])
    p_exact = ex / ex.sum(axis=1, keepdims=True)
    dsel = p_exact * (dw - np.sum(p_exact * dw, axis=1, keepdims=True))
    dlogits = np.zeros((T, E))
    np.put_along_axis(dlogits, idx.astype(np.int64), dsel, axis=1)
    r = dict(dx=dx, dlogits=dlogits, dw=dw, dW1=np.stack(grads["dW1"]),
             dW3=np.stack(grads["dW3"]), dW2=np.stack(grads["dW2"]))
    if magnitudes:
        # dl_j = p_j ((1 - p_j) dw_j - sum_{i != j} p_i dw_i); each slot's dw
        # depends on roundings of its own rows only
        msel = p_exact * ((1.0 - 2.0 * p_exact) * mdw
                          + np.sum(p_exact * mdw, axis=1, keepdims=True))
        mdl = np.zeros((T, E))
        np.put_along_axis(mdl, idx.astype(np.int64), msel, axis=1)
        r.update(mag_dx=mdx, mag_dlogits=mdl, mag_dW1=np.stack(mag["dW1"]),
                 mag_dW3=np.stack(mag["dW3"]), mag_dW2=np.stack(mag["dW2"]))
    return r
