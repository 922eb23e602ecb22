"""Plain, slow CPU oracle for the local MoE forward chain.

TEST INFRASTRUCTURE. Nothing on the product path imports this module; it shares
no code, table or constant with the CUDA library. It exists so that the CUDA
path can be compared element by element with an implementation that a reader
can check against the pages by eye.

The chain (ruDNN user guide, section 3 "MoE workflow"):
    logits -> softmax/top-k routing -> compact dispatch -> SwiGLU experts -> weighted combine

Precision, as the oracle computes it:
  * inputs are the exact dtype-rounded bytes the GPU receives, widened exactly;
  * routing runs in FP32, every operation rounded to FP32 in a fixed sequential
    order, with exp computed in f64 and rounded once to FP32 (so the FP32 exp
    is correctly rounded up to double rounding); an f64 copy of the same
    softmax is kept for the self-checks;
  * expert projections, SiLU, the gate*up product, the down projection and the
    combine are f64 with no intermediate rounding.

Readings of the pages that the oracle fixes (each is also listed in the design
notes):
  R1  selection uses the FP32 logits (exactly the dtype values) ordered by value
      descending, ties to the lower expert id; softmax is strictly increasing,
      so this is "softmax, then top-k" without ties that exp rounding would add.
  R2  slot j = 0 holds the largest score; slots continue in that order.
  R3  a non-finite row (any NaN, any +inf, or every entry -inf) gets indices
      0..k-1 (all its probabilities are NaN, so all tie and the lower ids win)
      and NaN weights.
  R4  weights are cast to the logits dtype with round-to-nearest-even, with or
      without renormalize.
  R5  dispatch lists the (t, j) pairs of expert e in ascending t*k + j order.
  R6  h = SiLU(g) * u stays f64 (the GPU rounds h to the dtype).
  R7  combine uses the dtype-cast routing weights (what ``weights()`` returns).
  R10 p_i = e_i / s (a division), then w_j = p_j / sum of the selected p in
      slot order.
  R11 a -inf logit in an otherwise finite row has probability 0 and is
      selectable only when fewer than k finite entries exist (ties by id).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch


def widen(t) -> np.ndarray:
    """Exact f64 copy of a CPU tensor (bf16/f16/f32 all widen exactly)."""
    if isinstance(t, np.ndarray):
        return t.astype(np.float64)
    return t.detach().to("cpu").to(torch.float64).numpy()


def round_to_dtype(values32: np.ndarray, dtype: torch.dtype) -> np.ndarray:
    """Round FP32 values to ``dtype`` with round-to-nearest-even (torch's CPU
    cast) and return them widened to f64."""
    t = torch.from_numpy(np.ascontiguousarray(values32, dtype=np.float32))
    return t.to(dtype).to(torch.float64).numpy()


def _exp32(d32: np.ndarray) -> np.ndarray:
    """FP32 exponential: exp evaluated in f64, rounded once to FP32."""
    return np.exp(d32.astype(np.float64)).astype(np.float32)


@dataclass
class RouteResult:
    indices: np.ndarray     # [T, k] uint32
    weights32: np.ndarray   # [T, k] float32, before the cast to the logits dtype
    weights: np.ndarray     # [T, k] float64 holding the logits-dtype value
    weights64: np.ndarray   # [T, k] float64, the same softmax in f64
    bad: np.ndarray         # [T] bool, non-finite rows


def route(logits, top_k: int, renormalize: bool, out_dtype: torch.dtype | None = None) -> RouteResult:
    """Softmax over all E experts in FP32, then top-k with lower-id ties,
    optional renormalize, then cast to the logits dtype.

    Follows ruDNN user guide section 4 "Routing contract" (all three ruDNN
    pages state it), the max-shift softmax of "tiny-llm deep dive 5: ops.rs"
    (section on softmax) and the FP32 renormalize sum of "PyTorch general ops"
    (section "MoE routing: topk, scatter and masked_fill")."""
    if out_dtype is None:
        out_dtype = logits.dtype if isinstance(logits, torch.Tensor) else torch.float32
    l32 = widen(logits).astype(np.float32)          # exact: D values are FP32 values
    T, E = l32.shape
    if not 1 <= top_k <= E:
        raise ValueError("top_k must satisfy 1 <= top_k <= E")
    k = top_k

    # R3: rows holding a NaN or +inf, or only -inf, keep NaN weights.
    bad = np.isnan(l32).any(axis=1) | np.isposinf(l32).any(axis=1) | np.isneginf(l32).all(axis=1)

    # R1/R2: descending by logit, ties to the lower id (a stable sort keeps id order).
    order = np.argsort(-l32.astype(np.float64), axis=1, kind="stable")[:, :k]
    order[bad] = np.arange(k)
    indices = order.astype(np.uint32)

    weights32 = np.full((T, k), np.nan, dtype=np.float32)
    weights64 = np.full((T, k), np.nan, dtype=np.float64)
    good = np.nonzero(~bad)[0]
    if good.size:
        lg = l32[good]                                   # [G, E] float32
        m = lg.max(axis=1)                               # exact
        d = (lg - m[:, None]).astype(np.float32)         # l_i - m, FP32
        e = _exp32(d)                                    # FP32 exp
        s = np.zeros(good.size, dtype=np.float32)
        for i in range(E):                               # sequential FP32 sum over experts
            s = (s + e[:, i]).astype(np.float32)
        sel = order[good]
        p = (np.take_along_axis(e, sel, axis=1) / s[:, None]).astype(np.float32)
        if renormalize:
            z = np.zeros(good.size, dtype=np.float32)
            for j in range(k):                           # slot-order FP32 sum (R10)
                z = (z + p[:, j]).astype(np.float32)
            p = (p / z[:, None]).astype(np.float32)
        weights32[good] = p

        lg64 = lg.astype(np.float64)
        e64 = np.exp(lg64 - lg64.max(axis=1, keepdims=True))
        p64 = np.take_along_axis(e64, sel, axis=1) / e64.sum(axis=1, keepdims=True)
        if renormalize:
            p64 = p64 / p64.sum(axis=1, keepdims=True)
        weights64[good] = p64

    weights = round_to_dtype(weights32, out_dtype)
    return RouteResult(indices, weights32, weights, weights64, bad)


@dataclass
class GroupRoutingOptions:
    """GroupRoutingOptions of the grouped sigmoid routing (ruDNN user guide,
    section 10): top_k, groups, selected_groups, group_top_two, renormalize,
    scale."""
    top_k: int
    groups: int
    selected_groups: int
    group_top_two: bool
    renormalize: bool
    scale: float


def check_group_options(E: int, o: GroupRoutingOptions):
    """The ranges the guide states: experts 1..=1024, groups 1..=128, top_k
    1..=64; experts divisible by groups; selected groups valid; top_k at most
    the experts of the selected groups; two experts per group for
    group_top_two; scale finite and positive."""
    G = E // o.groups if o.groups else 0
    ok = (1 <= E <= 1024 and 1 <= o.groups <= 128 and 1 <= o.top_k <= 64 and E % o.groups == 0
          and 1 <= o.selected_groups <= o.groups and o.top_k <= o.selected_groups * G
          and (not o.group_top_two or G >= 2) and np.isfinite(o.scale) and o.scale > 0)
    if not ok:
        raise ValueError("invalid GroupRoutingOptions for E=%d: %r" % (E, o))


def route_sigmoid_grouped(logits, bias, o: GroupRoutingOptions,
                          out_dtype: torch.dtype | None = None) -> RouteResult:
    """Group-limited sigmoid routing with a selection-only correction bias
    (ruDNN user guide, section 10; the group-max, top-groups, mask, top-k
    steps of the DeepSeek-style routing in "PyTorch general ops", section
    "MoE routing: topk, scatter and masked_fill").

    In FP32: s_i = 1 / (1 + exp(-l_i)); corrected c_i = s_i + bias_i (bias
    only steers selection); group score = max of c over the group, or the
    sum of its two largest c with group_top_two; the selected_groups best
    groups (ties to the lower group id); among their experts the top_k
    largest c (ties to the lower id), slot 0 the largest; weights are the
    uncorrected s of the selected experts, divided by their slot-ordered sum
    when renormalize, then multiplied by scale, then cast to the logits dtype.
    Reading: a row holding a NaN (logit or bias) keeps NaN weights and
    indices 0..k-1, as the softmax contract does for non-finite rows."""
    if out_dtype is None:
        out_dtype = logits.dtype if isinstance(logits, torch.Tensor) else torch.float32
    l32 = widen(logits).astype(np.float32)
    T, E = l32.shape
    check_group_options(E, o)
    k, G = o.top_k, E // o.groups
    one = np.float32(1.0)
    e = _exp32((-l32).astype(np.float32))
    with np.errstate(over="ignore", divide="ignore"):
        s = (one / (one + e).astype(np.float32)).astype(np.float32)
    if bias is not None:
        b32 = widen(bias).astype(np.float32).reshape(1, E)
        c = (s + b32).astype(np.float32)
    else:
        c = s
    bad = np.isnan(c).any(axis=1)

    cg = c.reshape(T, o.groups, G).astype(np.float32)
    if o.group_top_two:
        srt = -np.sort(-cg.astype(np.float64), axis=2)             # descending, exact
        gs = (srt[:, :, 0].astype(np.float32) + srt[:, :, 1].astype(np.float32)).astype(np.float32)
    else:
        gs = cg.max(axis=2)
    gsel = np.argsort(-gs.astype(np.float64), axis=1, kind="stable")[:, :o.selected_groups]
    in_sel = np.zeros((T, o.groups), dtype=bool)
    np.put_along_axis(in_sel, gsel, True, axis=1)
    expert_ok = np.repeat(in_sel, G, axis=1)
    # Experts of the selected groups first (also one whose corrected score is
    # -inf), then by descending c, ties to the lower id.
    ids = np.broadcast_to(np.arange(E), (T, E))
    order = np.lexsort((ids, -c.astype(np.float64), ~expert_ok), axis=1)[:, :k]
    order[bad] = np.arange(k)
    indices = order.astype(np.uint32)

    w = np.take_along_axis(s, order, axis=1).astype(np.float32)
    if o.renormalize:
        z = np.zeros(T, dtype=np.float32)
        for j in range(k):
            z = (z + w[:, j]).astype(np.float32)
        w = (w / z[:, None]).astype(np.float32)
    w = (w * np.float32(o.scale)).astype(np.float32)
    w[bad] = np.nan

    s64 = 1.0 / (1.0 + np.exp(-l32.astype(np.float64)))
    w64 = np.take_along_axis(s64, order, axis=1)
    if o.renormalize:
        w64 = w64 / w64.sum(axis=1, keepdims=True)
    w64 = w64 * float(o.scale)
    w64[bad] = np.nan
    return RouteResult(indices, w, round_to_dtype(w, out_dtype), w64, bad)


@dataclass
class DispatchResult:
    counts: np.ndarray   # [E] uint32
    offsets: np.ndarray  # [E+1] uint32, exclusive prefix of counts
    row_src: np.ndarray  # [T*k] uint32, dispatched row r -> flat slot t*k + j
    inv: np.ndarray      # [T*k] uint32, flat slot t*k + j -> dispatched row r


def dispatch(indices: np.ndarray, E: int) -> DispatchResult:
    """Compact per-expert layout with no capacity dropping (ruDNN user guide,
    section 5 "Expert weights and dispatch"). Expert e's rows list its (t, j)
    pairs in ascending t*k + j (R5); the inverse map restores token order.
    Brute force: one pass over the flat slots per expert."""
    flat = np.asarray(indices, dtype=np.int64).reshape(-1)
    n = flat.size
    counts = np.zeros(E, dtype=np.uint32)
    row_src = np.zeros(n, dtype=np.uint32)
    inv = np.full(n, 0xFFFFFFFF, dtype=np.uint32)
    r = 0
    for e in range(E):
        members = np.nonzero(flat == e)[0]
        counts[e] = members.size
        row_src[r:r + members.size] = members
        inv[members] = np.arange(r, r + members.size, dtype=np.uint32)
        r += members.size
    offsets = np.zeros(E + 1, dtype=np.uint32)
    offsets[1:] = np.cumsum(counts, dtype=np.uint64).astype(np.uint32)
    return DispatchResult(counts, offsets, row_src[:r], inv)


def silu(g: np.ndarray) -> np.ndarray:
    """SiLU(x) = x / (1 + e^-x) ("tiny-llm deep dive 5: ops.rs", section on SiLU)."""
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


def _swiglu_rows(x_rows: np.ndarray, gate_e: np.ndarray, up_e: np.ndarray,
                 down_e: np.ndarray) -> np.ndarray:
    """W_down (SiLU(W_gate x) * W_up x) for each row x, bias free, in f64.
    gate_e, up_e: [I, H]; down_e: [H, I]; x_rows: [n, H] -> [n, H]."""
    g = x_rows @ gate_e.T
    u = x_rows @ up_e.T
    h = silu(g) * u
    return h @ down_e.T


def experts_forward_dispatched(x, gate, up, down, disp: DispatchResult, top_k: int) -> np.ndarray:
    """Expert outputs for every dispatched row, in dispatched order [T*k, H], f64.
    Row r of expert e is token row_src[r] // k (ruDNN user guide, section 6:
    forward_dispatched)."""
    x64 = widen(x)
    E = len(disp.counts)
    out = np.zeros((len(disp.row_src), x64.shape[1]), dtype=np.float64)
    for e in range(E):
        lo, hi = int(disp.offsets[e]), int(disp.offsets[e + 1])
        if hi == lo:
            continue
        tok = disp.row_src[lo:hi].astype(np.int64) // top_k
        out[lo:hi] = _swiglu_rows(x64[tok], widen(gate[e]), widen(up[e]), widen(down[e]))
    return out


def combine(y_dispatched: np.ndarray, inv: np.ndarray, weights: np.ndarray, T: int,
            top_k: int) -> np.ndarray:
    """out[t] = sum_j w[t, j] * y[inv[t*k + j]] in f64 (ruDNN user guide,
    section 6: combine restores token order and merges with the routing
    weights; R7: the weights are the dtype-cast ones). A NaN weight makes the
    row NaN."""
    H = y_dispatched.shape[1]
    out = np.zeros((T, H), dtype=np.float64)
    inv = np.asarray(inv, dtype=np.int64).reshape(T, top_k)
    for j in range(top_k):
        out += weights[:, j:j + 1] * y_dispatched[inv[:, j]]
    return out


@dataclass
class ForwardResult:
    route: RouteResult
    dispatch: DispatchResult
    y_dispatched: np.ndarray
    out: np.ndarray


def forward(x, logits, gate, up, down, top_k: int, renormalize: bool) -> ForwardResult:
    """The whole local chain: route, dispatch, SwiGLU experts, combine
    (ruDNN user guide, section 6, SwiGluExperts::forward)."""
    T = x.shape[0]
    E = logits.shape[1]
    rt = route(logits, top_k, renormalize)
    dp = dispatch(rt.indices, E)
    y = experts_forward_dispatched(x, gate, up, down, dp, top_k)
    out = combine(y, dp.inv, rt.weights, T, top_k)
    return ForwardResult(rt, dp, y, out)


def forward_with_routing(x, gate, up, down, rt: RouteResult) -> ForwardResult:
    """Dispatch, experts and combine for a given routing result (the same
    chain after any routing function)."""
    T, k = rt.indices.shape
    E = gate.shape[0]
    dp = dispatch(rt.indices, E)
    y = experts_forward_dispatched(x, gate, up, down, dp, k)
    out = combine(y, dp.inv, rt.weights, T, k)
    return ForwardResult(rt, dp, y, out)


def forward_tokens(x, logits, gate, up, down, top_k: int, renormalize: bool,
                   tokens: np.ndarray) -> np.ndarray:
    """The forward output for a subset of tokens only, [len(tokens), H] in f64.
    Routing and the expert MLP are per token, so each sampled token is routed
    on its own logits row and sent through its k experts."""
    tokens = np.asarray(tokens, dtype=np.int64)
    rt = route(logits[tokens], top_k, renormalize, out_dtype=logits.dtype)
    return forward_tokens_routed(x, gate, up, down, rt, tokens)


def forward_tokens_routed(x, gate, up, down, rt: RouteResult, tokens: np.ndarray) -> np.ndarray:
    """forward_tokens for a routing result already taken on the sampled rows
    (rt.indices[i] belongs to token tokens[i]), whatever routing made it."""
    tokens = np.asarray(tokens, dtype=np.int64)
    x64 = widen(x[tokens])
    out = np.zeros((tokens.size, x64.shape[1]), dtype=np.float64)
    for e in np.unique(rt.indices):
        sel = np.nonzero(rt.indices == e)            # (sample, slot) pairs routed to e
        y = _swiglu_rows(x64[sel[0]], widen(gate[int(e)]), widen(up[int(e)]), widen(down[int(e)]))
        np.add.at(out, sel[0], rt.weights[sel][:, None] * y)
    bad_rows = np.isnan(rt.weights).any(axis=1)
    out[bad_rows] = np.nan
    return out
