"""First-order rounding-error bounds for the training path's expert cache and
gradients, derived from the roundings the kernels make (test infrastructure:
the bounds the GPU's results are held to, not reference values).

Model of the GPU computation (dtype D; u_D its unit roundoff: 2^-8 for BF16,
2^-11 for F16; F32 values are stored unrounded):
  * every contraction of n products accumulates in FP32: its error is at most
    n * 2^-23 of the sum of |terms| (products exact, one FP32 rounding per
    addition, the worst case of the tensor cores' and of FMA chains alike);
  * forward cache: g and u are the FP32 accumulators rounded once to D;
    h = SiLU(g_acc) * u_acc from the unrounded FP32 accumulators, rounded once
    to D; the 16-bit epilogue evaluates SiLU(g) = g (1/2 + tanh(g/2)/2) with
    tanh.approx (absolute error of the sigmoid below 2^-12), the F32 path with
    expf (a few FP32 ulps);
  * backward: dh = dy W_down stays FP32; dg = dh * u * SiLU'(g) and
    du = dh * SiLU(g) from the cached (rounded) g and u, with expf, rounded
    once to D; dx = dg W_gate + du W_up rounded once to D; the weight
    gradients dW_gate = dg^T x, dW_up = du^T x, dW_down = dy^T h are FP32.
Each bound adds, for one entry, every rounding above that reaches it,
carried linearly to first order through the formulas (|SiLU'| <= 1.1,
|SiLU''| <= 1/2 everywhere). The checks allow 1.25 times the bound: the
neglected second-order terms are a further u_D of it at most.
"""
from __future__ import annotations

import numpy as np
import torch

ACC = 2.0 ** -23                   # per-addition FP32 accumulation error (relative)
UNIT = {torch.float32: 0.0, torch.float16: 2.0 ** -11, torch.bfloat16: 2.0 ** -8}
SILU_SIGMOID_ABS = {torch.float32: 8 * 2.0 ** -24, torch.float16: 2.0 ** -12, torch.bfloat16: 2.0 ** -12}
FN32_REL = 16 * 2.0 ** -24          # expf-based SiLU / SiLU' in FP32 (backward epilogue)
SLACK = 1.25
DSILU_MAX = 1.1
D2SILU_MAX = 0.5


def _w(t):
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().cpu().to(torch.float64).numpy()


def _silu(g):
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def _dsilu(g):
    with np.errstate(over="ignore"):
        s = 1.0 / (1.0 + np.exp(-g))
    return s * (1.0 + g * (1.0 - s))


def expert_error_bounds(x_dispatched, gate, up, down, offsets, dexpert, dtype):
    """Bounds for the cache (g, u, h) [rows, I] and the gradients dx [rows, H],
    dgate/dup [E, I, H], ddown [E, H, I], given the exact (dtype-rounded)
    inputs. Returns a dict of arrays shaped like the quantities."""
    x, Wg, Wu, Wd, dy = (_w(a) for a in (x_dispatched, gate, up, down, dexpert))
    E, I, H = Wg.shape
    uD = UNIT[dtype]
    sig = SILU_SIGMOID_ABS[dtype]
    off = np.asarray(offsets, dtype=np.int64)
    rows = x.shape[0]
    b = {"g": np.zeros((rows, I)), "u": np.zeros((rows, I)), "h": np.zeros((rows, I)),
         "dx": np.zeros((rows, H)), "dgate": np.zeros((E, I, H)), "dup": np.zeros((E, I, H)),
         "ddown": np.zeros((E, H, I))}
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi <= lo:
            continue
        X, dY = x[lo:hi], dy[lo:hi]
        aX = np.abs(X)
        G, U = X @ Wg[e].T, X @ Wu[e].T
        S, dS = _silu(G), _dsilu(G)
        Hh = S * U
        # forward cache
        eg_acc = H * ACC * (aX @ np.abs(Wg[e]).T)
        eu_acc = H * ACC * (aX @ np.abs(Wu[e]).T)
        eg = uD * np.abs(G) + eg_acc
        eu = uD * np.abs(U) + eu_acc
        eh = (uD * np.abs(Hh) + np.abs(dS) * np.abs(U) * eg_acc + np.abs(S) * eu_acc
              + sig * np.abs(G) * np.abs(U) + 3 * 2.0 ** -24 * np.abs(Hh))
        b["g"][lo:hi], b["u"][lo:hi], b["h"][lo:hi] = eg, eu, eh
        # backward
        dH = dY @ Wd[e]
        adH = np.abs(dY) @ np.abs(Wd[e])
        edh = H * ACC * adH
        dG, dU = dH * U * dS, dH * S
        edg = (uD * np.abs(dG) + edh * np.abs(U) * np.abs(dS) + np.abs(dH) * eu * np.abs(dS)
               + np.abs(dH) * np.abs(U) * (D2SILU_MAX * eg + FN32_REL * (1.0 + np.abs(G))))
        edu = (uD * np.abs(dU) + edh * np.abs(S) + np.abs(dH) * (DSILU_MAX * eg + FN32_REL * np.abs(S)))
        DX = dG @ Wg[e] + dU @ Wu[e]
        b["dx"][lo:hi] = (uD * np.abs(DX) + edg @ np.abs(Wg[e]) + edu @ np.abs(Wu[e])
                          + 2 * I * ACC * (np.abs(dG) @ np.abs(Wg[e]) + np.abs(dU) @ np.abs(Wu[e])))
        n = hi - lo
        b["dgate"][e] = edg.T @ aX + n * ACC * (np.abs(dG).T @ aX)
        b["dup"][e] = edu.T @ aX + n * ACC * (np.abs(dU).T @ aX)
        b["ddown"][e] = np.abs(dY).T @ eh + n * ACC * (np.abs(dY).T @ np.abs(Hh))
    return b


def assert_within_bound(got, ref, bound, what):
    """|got - ref| <= SLACK * bound entry by entry, NaN positions equal."""
    got = _w(got)
    bad = np.isnan(got) != np.isnan(ref)
    assert not bad.any(), f"{what}: NaN positions differ at {np.argwhere(bad)[:5].tolist()}"
    fin = np.isfinite(ref)
    err = np.abs(got[fin] - ref[fin])
    lim = SLACK * bound[fin] + 1e-30
    if err.size == 0:
        return
    worst = int(np.argmax(err / lim))
    assert (err <= lim).all(), (f"{what}: error {err[worst]:.3e} above its rounding bound {lim[worst]:.3e} "
                                f"(reference {ref[fin][worst]:.3e}; {int((err > lim).sum())} entries over)")
