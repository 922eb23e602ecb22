"""Plain, slow CPU oracle for first-order MoE training (backward of the local
chain). TEST INFRASTRUCTURE, like ``moe_oracle``: nothing on the product path
imports it and it shares nothing with the CUDA library.

Follows the ruDNN user guide, section 12 "First-order MoE training":
  * selected_router_weights(logits, indices, options): FP32 [T, top_k] weights
    of a fixed selection, with softmax or sigmoid scoring, optional
    renormalize over the selected slots, then a finite positive scale;
  * selected_router_backward(logits, indices, grad_weights, options): the
    gradient of those weights with respect to the logits, [T, E] in the logits
    dtype. Only the continuous weights of the fixed selection are
    differentiated (not the top-k, the group choice or the correction bias).
    Repeated indices gather (each slot is its own term); an invalid index
    makes the whole row NaN;
  * combine_backward(expert_output, grad_output): dexpert (each dispatched
    row's share of grad_output, times its routing weight) and FP32 dweights;
  * cache.backward(dexpert): the dispatched rows' input gradient and FP32
    gradients of gate, up and down;
  * dispatch_backward(dinput): adds each token's dispatched rows back onto the
    token, without multiplying by the routing weight again.

Derivatives are the textbook ones written out, in f64: the softmax Jacobian
dP_i/dl_m = P_i (delta_im - P_m), the logistic derivative s (1 - s), the
quotient rule for renormalize, and SiLU'(g) = s(g) (1 + g (1 - s(g))).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from .moe_oracle import _exp32, round_to_dtype, widen


@dataclass
class RouterWeightOptions:
    """RouterWeightOptions (ruDNN user guide, section 12): RouterScoring
    Softmax or Sigmoid, renormalize of the selected weights, final scale."""
    scoring: str          # "softmax" | "sigmoid"
    renormalize: bool
    scale: float


def check_router_options(E: int, top_k: int, o: RouterWeightOptions):
    """1 <= top_k <= min(E, 64); a known scoring; scale finite and > 0."""
    if not (1 <= top_k <= min(E, 64)) or o.scoring not in ("softmax", "sigmoid") \
            or not np.isfinite(o.scale) or not o.scale > 0:
        raise ValueError(f"invalid router options for E={E}, top_k={top_k}: {o!r}")


def _invalid_rows(idx: np.ndarray, E: int) -> np.ndarray:
    return ((idx < 0) | (idx >= E)).any(axis=1)


def selected_router_weights(logits, indices, o: RouterWeightOptions):
    """FP32 weights of the given selection, and the same in f64.

    FP32 path: softmax as in the forward routing (max shift, exp rounded once,
    left-to-right FP32 sum over all E, p = e / s); sigmoid s = 1 / (1 + exp(-l));
    renormalize divides by the slot-ordered FP32 sum of the selected values;
    then the FP32 product with scale. Returns (w32 [T,k] float32, w64 [T,k])."""
    l32 = widen(logits).astype(np.float32)
    T, E = l32.shape
    idx = np.asarray(indices).astype(np.int64).reshape(T, -1)
    k = idx.shape[1]
    check_router_options(E, k, o)
    bad = _invalid_rows(idx, E)
    safe = np.where((idx >= 0) & (idx < E), idx, 0)
    one = np.float32(1.0)

    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        if o.scoring == "softmax":
            m = l32.max(axis=1)
            e = _exp32((l32 - m[:, None]).astype(np.float32))
            s = np.zeros(T, dtype=np.float32)
            for i in range(E):
                s = (s + e[:, i]).astype(np.float32)
            v = (np.take_along_axis(e, safe, axis=1) / s[:, None]).astype(np.float32)
        else:
            x = np.take_along_axis(l32, safe, axis=1)
            v = (one / (one + _exp32((-x).astype(np.float32)))).astype(np.float32)
        if o.renormalize:
            z = np.zeros(T, dtype=np.float32)
            for j in range(k):
                z = (z + v[:, j]).astype(np.float32)
            v = (v / z[:, None]).astype(np.float32)
        w32 = (v * np.float32(o.scale)).astype(np.float32)
    w32[bad] = np.nan

    l64 = l32.astype(np.float64)
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        if o.scoring == "softmax":
            e64 = np.exp(l64 - l64.max(axis=1, keepdims=True))
            v64 = np.take_along_axis(e64, safe, axis=1) / e64.sum(axis=1, keepdims=True)
        else:
            v64 = 1.0 / (1.0 + np.exp(-np.take_along_axis(l64, safe, axis=1)))
        if o.renormalize:
            v64 = v64 / v64.sum(axis=1, keepdims=True)
    w64 = v64 * float(o.scale)
    w64[bad] = np.nan
    return w32, w64


def router_jacobian(l64_row: np.ndarray, idx_row: np.ndarray, o: RouterWeightOptions) -> np.ndarray:
    """dw_j / dl_m for one row, [k, E], written out from the textbook
    derivatives (f64)."""
    E = l64_row.size
    k = idx_row.size
    onehot = np.zeros((k, E))
    onehot[np.arange(k), idx_row] = 1.0
    if o.scoring == "softmax":
        ex = np.exp(l64_row - l64_row.max())
        P = ex / ex.sum()
        dP = np.diag(P) - np.outer(P, P)            # dP_i / dl_m = P_i (delta_im - P_m)
        v = P[idx_row]
        dv = dP[idx_row, :]                          # [k, E]
    else:
        s = 1.0 / (1.0 + np.exp(-l64_row))
        v = s[idx_row]
        dv = onehot * (s * (1.0 - s))[idx_row][:, None]
    if o.renormalize:
        Z = v.sum()
        dZ = dv.sum(axis=0)                          # [E]
        J = (dv * Z - np.outer(v, dZ)) / (Z * Z)     # quotient rule
    else:
        J = dv
    return J * float(o.scale)


def selected_router_backward(logits, indices, grad_weights, o: RouterWeightOptions,
                             out_dtype: torch.dtype | None = None):
    """dL/dlogits = J^T grad_weights per row (f64), returned as f64 and as the
    value rounded to the logits dtype (through FP32). Rows with an invalid
    index, or whose weights are NaN, are NaN."""
    if out_dtype is None:
        out_dtype = logits.dtype if isinstance(logits, torch.Tensor) else torch.float32
    l64 = widen(logits).astype(np.float32).astype(np.float64)
    T, E = l64.shape
    idx = np.asarray(indices).astype(np.int64).reshape(T, -1)
    g = widen(grad_weights).astype(np.float32).astype(np.float64)
    k = idx.shape[1]
    check_router_options(E, k, o)
    bad = _invalid_rows(idx, E)
    out = np.full((T, E), np.nan)
    with np.errstate(over="ignore", invalid="ignore", divide="ignore"):
        for t in range(T):
            if bad[t]:
                continue
            J = router_jacobian(l64[t], idx[t], o)
            out[t] = J.T @ g[t]
    return out, round_to_dtype(out.astype(np.float32), out_dtype)


def combine_backward(y_dispatched, inv, weights, grad_out, T: int, top_k: int):
    """out[t] = sum_j w[t, j] y[inv[t, j]] differentiated (f64):
    dexpert[inv[t, j]] = w[t, j] grad_out[t]; dweights[t, j] = <grad_out[t], y[inv[t, j]]>.
    Rows of y no slot points at get zero; a slot whose inv is out of range
    gets a NaN dweight. The weights are the dtype-cast forward weights."""
    y = widen(y_dispatched)
    go = widen(grad_out)
    w = np.asarray(weights, dtype=np.float64).reshape(T, top_k)
    inv = np.asarray(inv, dtype=np.int64).reshape(T, top_k)
    n = y.shape[0]
    dexpert = np.zeros_like(y)
    dweights = np.full((T, top_k), np.nan)
    for t in range(T):
        for j in range(top_k):
            r = inv[t, j]
            if 0 <= r < n:
                dexpert[r] = w[t, j] * go[t]
                dweights[t, j] = float(go[t] @ y[r])
    return dexpert, dweights


def _silu(g):
    return g / (1.0 + np.exp(-g))


def _silu_grad(g):
    s = 1.0 / (1.0 + np.exp(-g))
    return s * (1.0 + g * (1.0 - s))


@dataclass
class ExpertGrads:
    dx_dispatched: np.ndarray  # [rows, H] f64
    dgate: np.ndarray          # [E, I, H]
    dup: np.ndarray            # [E, I, H]
    ddown: np.ndarray          # [E, H, I]
    # The same sums over |terms| carried through the chain (|dy| |W_down| for
    # dh, then |dh| |u| |SiLU'(g)|, ...): the scale a rounding error of each
    # entry is measured against.
    dx_abs: np.ndarray | None = None
    dgate_abs: np.ndarray | None = None
    dup_abs: np.ndarray | None = None
    ddown_abs: np.ndarray | None = None


def training_forward_cache(x_dispatched, gate, up, offsets):
    """The forward cache of the training forward (ruDNN user guide, section
    12, forward_dispatched_training): per dispatched row r of expert e, the
    pre-activations g = W_gate[e] x_r and u = W_up[e] x_r and the SwiGLU
    output h = SiLU(g) * u, in f64 from the dtype-rounded inputs with no
    intermediate rounding. Returns (g, u, h), each [rows, I]."""
    x, Wg, Wu = widen(x_dispatched), widen(gate), widen(up)
    E, I, _ = Wg.shape
    off = np.asarray(offsets, dtype=np.int64)
    g = np.zeros((x.shape[0], I))
    u = np.zeros((x.shape[0], I))
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi <= lo:
            continue
        g[lo:hi] = x[lo:hi] @ Wg[e].T
        u[lo:hi] = x[lo:hi] @ Wu[e].T
    with np.errstate(over="ignore"):
        h = _silu(g) * u
    return g, u, h


def experts_backward(x_dispatched, gate, up, down, offsets, dexpert, cache=None) -> ExpertGrads:
    """Backward of y_r = W_down[e] (SiLU(W_gate[e] x_r) * (W_up[e] x_r)) over the
    dispatched rows of each expert (f64 from the dtype-rounded inputs):
    dh = dy W_down, dW_down = dy^T h, dg = dh * u * SiLU'(g), du = dh * SiLU(g),
    dx = dg W_gate + du W_up, dW_gate = dg^T x, dW_up = du^T x.

    ``cache`` = (g, u, h) [rows, I] each: the forward cache the backward
    consumes (cache.backward of the pages); without it g, u and h come from
    training_forward_cache, in f64 from x."""
    x = widen(x_dispatched)
    if cache is None:
        cache = training_forward_cache(x, gate, up, offsets)
    cg, cu, ch = (widen(c) if isinstance(c, torch.Tensor) else np.asarray(c, dtype=np.float64) for c in cache)
    dy = widen(dexpert) if isinstance(dexpert, torch.Tensor) else np.asarray(dexpert, dtype=np.float64)
    Wg, Wu, Wd = widen(gate), widen(up), widen(down)
    E, I, H = Wg.shape
    off = np.asarray(offsets, dtype=np.int64)
    dx = np.zeros_like(x)
    dWg = np.zeros((E, I, H))
    dWu = np.zeros((E, I, H))
    dWd = np.zeros((E, H, I))
    ab = [np.zeros_like(x), np.zeros((E, I, H)), np.zeros((E, I, H)), np.zeros((E, H, I))]
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi <= lo:
            continue
        X, dY = x[lo:hi], dy[lo:hi]
        G, U, Hh = cg[lo:hi], cu[lo:hi], ch[lo:hi]
        dH = dY @ Wd[e]
        dWd[e] = dY.T @ Hh
        dG = dH * U * _silu_grad(G)
        dU = dH * _silu(G)
        dx[lo:hi] = dG @ Wg[e] + dU @ Wu[e]
        dWg[e] = dG.T @ X
        dWu[e] = dU.T @ X
        # |.| carried through the chain: each entry's sum of |terms|, with the
        # intermediate gradients replaced by their own |term| sums.
        dH_abs = np.abs(dY) @ np.abs(Wd[e])
        dG_abs = dH_abs * np.abs(U) * np.abs(_silu_grad(G))
        dU_abs = dH_abs * np.abs(_silu(G))
        ab[0][lo:hi] = dG_abs @ np.abs(Wg[e]) + dU_abs @ np.abs(Wu[e])
        ab[1][e] = dG_abs.T @ np.abs(X)
        ab[2][e] = dU_abs.T @ np.abs(X)
        ab[3][e] = np.abs(dY).T @ np.abs(Hh)
    return ExpertGrads(dx, dWg, dWu, dWd, *ab)


def dispatch_backward(dinput, inv, T: int, top_k: int):
    """dx[t] = sum over slots j of dinput[inv[t, j]], slot order, f64; no
    routing weight is applied. A token with an out-of-range inv gets a NaN row."""
    d = widen(dinput) if isinstance(dinput, torch.Tensor) else np.asarray(dinput, dtype=np.float64)
    inv = np.asarray(inv, dtype=np.int64).reshape(T, top_k)
    n, H = d.shape
    dx = np.zeros((T, H))
    for t in range(T):
        for j in range(top_k):
            r = inv[t, j]
            if 0 <= r < n:
                dx[t] += d[r]
            else:
                dx[t] = np.nan
    return dx
